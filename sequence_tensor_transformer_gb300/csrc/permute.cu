// Neuron-permutation shard maps for Delayed TP ("Affinity-Aware Sharding for
// Delayed Tensor Parallelism", Abstract: the dense model is permuted before it
// is sharded, and under delayed partials which neurons share a device is a
// modelling decision).  Executing a permuted layout = renumbering each FFN's
// neurons once, then sharding contiguously: new neuron i of module l is old
// neuron perm[l][i]; W1g/W1u rows and W2 columns move together.
//
// HBM-bound gathers, every byte read and written once:
//   rows    W1g/W1u: one warp per output row, 16-byte coalesced copies
//   columns W2: one CTA per output row; the input row is staged in shared
//           memory and gathered into coalesced stores
// An index outside [0, F) is recorded in the status words and its output is
// written as zeros; no out-of-range address is formed.
#include <cuda_bf16.h>

#include "sptp.h"
#include "sptp_internal.h"

namespace sptp {

namespace {

__device__ void report_bad_index(DeviceStatus* st, int info) {
    if (st != nullptr && atomicCAS(&st->code, 0, SPTP_ERR_SHAPE) == 0) {
        st->where = kWherePermIndex;
        st->block = blockIdx.x;
        st->info = info;
    }
}

// out_rows[l][i][:] = in_rows[l][perm[l][i]][:] for two matrices at once
__global__ void __launch_bounds__(256) permute_rows_kernel(const uint8_t* in0, const uint8_t* in1, uint8_t* out0,
                                                           uint8_t* out1, const int* perm, int L, int F,
                                                           int row_bytes, DeviceStatus* st) {
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const int lane = threadIdx.x & 31;
    const long long total = static_cast<long long>(L) * F;
    for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total;
         w += warps) {
        const int l = static_cast<int>(w / F);
        const int src = perm[w];
        const bool ok = src >= 0 && src < F;
        if (!ok && lane == 0) report_bad_index(st, static_cast<int>(w));
        const long long mat = static_cast<long long>(l) * F * row_bytes;
        const long long dst_off = mat + (w - static_cast<long long>(l) * F) * row_bytes;
        const long long src_off = mat + static_cast<long long>(ok ? src : 0) * row_bytes;
        for (int c = lane * 16; c < row_bytes; c += 32 * 16) {
            uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
            if (ok) {
                a = __ldg(reinterpret_cast<const uint4*>(in0 + src_off + c));
                b = __ldg(reinterpret_cast<const uint4*>(in1 + src_off + c));
            }
            *reinterpret_cast<uint4*>(out0 + dst_off + c) = a;
            *reinterpret_cast<uint4*>(out1 + dst_off + c) = b;
        }
    }
}

// out[l][r][i] = in[l][r][perm[l][i]]; one CTA per (l, r) row, rows of F
// elements of `es` bytes staged in shared memory
template <typename T>
__global__ void __launch_bounds__(512) permute_cols_kernel(const T* in, T* out, const int* perm, int L, int R, int F,
                                                           DeviceStatus* st) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    T* row = reinterpret_cast<T*>(smem_raw);
    const long long rows = static_cast<long long>(L) * R;
    for (long long lr = blockIdx.x; lr < rows; lr += gridDim.x) {
        const int l = static_cast<int>(lr / R);
        const T* src = in + lr * F;
        T* dst = out + lr * F;
        const int* pl = perm + static_cast<long long>(l) * F;
        __syncthreads();  // previous row fully gathered
        for (int i = threadIdx.x; i < F; i += blockDim.x) row[i] = src[i];
        __syncthreads();
        for (int i = threadIdx.x; i < F; i += blockDim.x) {
            const int s = pl[i];
            const bool ok = s >= 0 && s < F;
            if (!ok && (lr % R) == 0) report_bad_index(st, i);
            dst[i] = ok ? row[s] : T(0);
        }
    }
}

}  // namespace

cudaError_t launch_permute_ffn(const void* W1g, const void* W1u, const void* W2, const int* perm, int L, int d,
                               int F, bool bf16, void* W1g_out, void* W1u_out, void* W2_out, DeviceStatus* st,
                               int num_sms, cudaStream_t s) {
    const int es = bf16 ? 2 : 4;
    const long long rows = static_cast<long long>(L) * F;
    if (rows == 0) return cudaSuccess;
    long long grid = (rows + 7) / 8;
    if (grid > static_cast<long long>(num_sms) * 8) grid = static_cast<long long>(num_sms) * 8;
    permute_rows_kernel<<<static_cast<int>(grid), 256, 0, s>>>(
        static_cast<const uint8_t*>(W1g), static_cast<const uint8_t*>(W1u), static_cast<uint8_t*>(W1g_out),
        static_cast<uint8_t*>(W1u_out), perm, L, F, d * es, st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = static_cast<size_t>(F) * es;
    long long grid2 = static_cast<long long>(L) * d;
    if (grid2 > static_cast<long long>(num_sms) * 4) grid2 = static_cast<long long>(num_sms) * 4;
    if (bf16) {
        e = cudaFuncSetAttribute(permute_cols_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        permute_cols_kernel<__nv_bfloat16><<<static_cast<int>(grid2), 512, smem, s>>>(
            static_cast<const __nv_bfloat16*>(W2), static_cast<__nv_bfloat16*>(W2_out), perm, L, d, F, st);
    } else {
        e = cudaFuncSetAttribute(permute_cols_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        permute_cols_kernel<float><<<static_cast<int>(grid2), 512, smem, s>>>(
            static_cast<const float*>(W2), static_cast<float*>(W2_out), perm, L, d, F, st);
    }
    return cudaGetLastError();
}

}  // namespace sptp
