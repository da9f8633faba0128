// Neuron-permutation shard maps for Delayed TP ("Affinity-Aware Sharding for
// Delayed Tensor Parallelism", Abstract: the dense model is permuted before it
// is sharded, and under delayed partials which neurons share a device is a
// modelling decision).  Executing a permuted layout = renumbering each FFN's
// neurons once, then sharding contiguously: new neuron i of module l is old
// neuron perm[l][i]; W1g/W1u rows and W2 columns move together.
//
// HBM-bound gathers, every byte read and written once:
//   rows    W1g/W1u: one warp per output row, 16-byte coalesced copies
//   columns W2: a CTA stages up to 8 whole rows in shared memory with
//           16-byte loads; each output column vector's indices are loaded
//           once and serve every staged row; 16-byte stores
// An index outside [0, F) is recorded in the status words and its output is
// written as zeros; no out-of-range address is formed.
#include <cuda_bf16.h>

#include "sptp.h"
#include "sptp_internal.h"
#include "sptp_ptx.cuh"

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
    const uint32_t warps = gridDim.x * (blockDim.x >> 5);
    const int lane = threadIdx.x & 31;
    const uint32_t total = static_cast<uint32_t>(L) * static_cast<uint32_t>(F);  // < 2^31, checked at launch
    for (uint32_t w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total; w += warps) {
        const int l = static_cast<int>(w / static_cast<uint32_t>(F));
        const int src = perm[w];
        const bool ok = src >= 0 && src < F;
        if (!ok && lane == 0) report_bad_index(st, static_cast<int>(w));
        const long long mat = static_cast<long long>(l) * F * row_bytes;
        const long long dst_off = mat + (w - static_cast<long long>(l) * F) * row_bytes;
        const long long src_off = mat + static_cast<long long>(ok ? src : 0) * row_bytes;
        const long long all_bytes = static_cast<long long>(total) * row_bytes;
        for (int c = lane * 16; c < row_bytes; c += 32 * 16) {
            // a checked build: both 16-byte vectors inside the [L][F] rows
            if (!checked_range(src_off + c, 16, all_bytes, st, nullptr, kWhereBoundsLoad) ||
                !checked_range(dst_off + c, 16, all_bytes, st, nullptr, kWhereBoundsStore))
                break;
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

// out[l][r][i] = in[l][r][perm[l][i]]: a CTA stages ROWS consecutive rows of
// one module in shared memory with 16-byte loads; then each thread takes
// output column vectors (16 bytes' worth of consecutive output elements),
// loads their indices once with 16-byte loads, and gathers and stores that
// vector for every staged row (F * sizeof(T) is a multiple of 16, and of 32
// for the index loads).
template <typename T, int ROWS>
__global__ void __launch_bounds__(512) permute_cols_kernel(const T* in, T* out, const int* perm, int L, int R, int F,
                                                           DeviceStatus* st) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    T* rows_s = reinterpret_cast<T*>(smem_raw);
    constexpr int E = 16 / sizeof(T);  // elements per 16-byte vector
    const int vec_per_row = F / E;
    const int gpl = (R + ROWS - 1) / ROWS;  // row groups per module
    const uint32_t groups = static_cast<uint32_t>(L) * static_cast<uint32_t>(gpl);
    for (uint32_t gi = blockIdx.x; gi < groups; gi += gridDim.x) {
        const int l = static_cast<int>(gi / static_cast<uint32_t>(gpl));
        const int r0 = static_cast<int>(gi - static_cast<uint32_t>(l) * gpl) * ROWS;
        const int nr = min(ROWS, R - r0);
        const T* src = in + (static_cast<long long>(l) * R + r0) * F;
        T* dst = out + (static_cast<long long>(l) * R + r0) * F;
        const int* pl = perm + static_cast<long long>(l) * F;
        __syncthreads();  // the previous group is fully gathered
        const int nvec = nr * vec_per_row;
#pragma unroll 4
        for (int v = threadIdx.x; v < nvec; v += blockDim.x)
            reinterpret_cast<uint4*>(rows_s)[v] = __ldg(reinterpret_cast<const uint4*>(src) + v);
        __syncthreads();
        for (int c = threadIdx.x; c < vec_per_row; c += blockDim.x) {
            int idx[E];
#pragma unroll
            for (int k = 0; k < E; k += 4) {
                const int4 q = __ldg(reinterpret_cast<const int4*>(pl + c * E + k));
                idx[k] = q.x, idx[k + 1] = q.y, idx[k + 2] = q.z, idx[k + 3] = q.w;
            }
#pragma unroll
            for (int k = 0; k < E; ++k) {
                const bool ok = idx[k] >= 0 && idx[k] < F;
                if (!ok) {
                    if (r0 == 0) report_bad_index(st, c * E + k);
                    idx[k] = -1;
                }
            }
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                if (r >= nr) break;
                const T* row_s = rows_s + static_cast<long long>(r) * F;
                union {
                    uint4 u;
                    T e[E];
                } pack;
#pragma unroll
                for (int k = 0; k < E; ++k) pack.e[k] = idx[k] >= 0 ? row_s[idx[k]] : T(0);
                // a checked build: the output vector inside the [L][R][F] matrix
                if (checked_range((static_cast<long long>(l) * R + r0 + r) * F + static_cast<long long>(c) * E, E,
                                  static_cast<long long>(L) * R * F, st, nullptr, kWhereBoundsStore))
                    reinterpret_cast<uint4*>(dst + static_cast<long long>(r) * F)[c] = pack.u;
            }
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
    if (rows >= (1ll << 31)) return cudaErrorInvalidValue;  // the kernels number rows with 32 bits
    long long grid = (rows + 7) / 8;
    if (grid > static_cast<long long>(num_sms) * 8) grid = static_cast<long long>(num_sms) * 8;
    permute_rows_kernel<<<static_cast<int>(grid), 256, 0, s>>>(
        static_cast<const uint8_t*>(W1g), static_cast<const uint8_t*>(W1u), static_cast<uint8_t*>(W1g_out),
        static_cast<uint8_t*>(W1u_out), perm, L, F, d * es, st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // as many whole rows per CTA as fit in ~96 KiB of shared memory (<= 8)
    int rpc = static_cast<int>((96u * 1024u) / (static_cast<size_t>(F) * es));
    rpc = rpc >= 8 ? 8 : (rpc >= 4 ? 4 : (rpc >= 2 ? 2 : 1));
    const size_t smem = static_cast<size_t>(rpc) * F * es;
    long long grid2 = static_cast<long long>(L) * ((d + rpc - 1) / rpc);
    if (grid2 > static_cast<long long>(num_sms) * 4) grid2 = static_cast<long long>(num_sms) * 4;
    auto launch = [&](auto kfn, auto tag) -> cudaError_t {
        using TT = decltype(tag);
        cudaError_t err =
            cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        kfn<<<static_cast<int>(grid2), 512, smem, s>>>(static_cast<const TT*>(W2), static_cast<TT*>(W2_out), perm, L,
                                                        d, F, st);
        return cudaGetLastError();
    };
    if (bf16) {
        switch (rpc) {
            case 8: return launch(permute_cols_kernel<__nv_bfloat16, 8>, __nv_bfloat16());
            case 4: return launch(permute_cols_kernel<__nv_bfloat16, 4>, __nv_bfloat16());
            case 2: return launch(permute_cols_kernel<__nv_bfloat16, 2>, __nv_bfloat16());
            default: return launch(permute_cols_kernel<__nv_bfloat16, 1>, __nv_bfloat16());
        }
    }
    switch (rpc) {
        case 8: return launch(permute_cols_kernel<float, 8>, float());
        case 4: return launch(permute_cols_kernel<float, 4>, float());
        case 2: return launch(permute_cols_kernel<float, 2>, float());
        default: return launch(permute_cols_kernel<float, 1>, float());
    }
}

}  // namespace sptp
