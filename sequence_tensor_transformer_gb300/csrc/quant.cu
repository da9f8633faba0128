// Row-wise E4M3 quantiser of the fp8 boundary variant: the linear layers of
// a tensor-parallel block run in fp8 ("[Feature] Async Tensor Parallelism
// for Archon Engine", "Additional Information": fp8 linear layers under TP).
// Each row r of a bf16 [R][K] operand (K the GEMM's reduction axis) gets a
// power-of-two scale 2^e_r, e_r the least integer >= -126 with
// max_k |a[r][k]| <= 448 * 2^e_r, and codes RNE_E4M3(a[r][k] * 2^-e_r).
// The product with 2^-e_r is exact, so the rounding decision is that of the
// bf16 value itself.
//
// HBM-bound: one CTA per row (grid-stride), 256 threads; each thread keeps
// up to kCached 16-byte vectors of its row in registers between the
// row-maximum pass and the quantise pass, so a row of up to 8192 elements is
// read once.  Longer rows re-read the rest (from L2).
#include "e4m3.cuh"
#include "sptp_internal.h"

namespace sptp {

namespace {

constexpr int kThreads = 256;
constexpr int kCached = 4;

__global__ void __launch_bounds__(kThreads) quantize_rows_e4m3_kernel(const uint4* __restrict__ a, long long R,
                                                                      int nvec, uint2* __restrict__ q,
                                                                      float* __restrict__ scale) {
    __shared__ float warp_max[kThreads / 32];
    for (long long r = blockIdx.x; r < R; r += gridDim.x) {
        const uint4* src = a + r * nvec;
        uint2* dst = q + r * nvec;
        uint4 v[kCached];
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < kCached; ++i) {
            const int idx = threadIdx.x + i * kThreads;
            if (idx < nvec) {
                v[i] = __ldcs(src + idx);
                amax = fmaxf(amax, absmax_bf16x8(v[i]));
            }
        }
        for (int idx = threadIdx.x + kCached * kThreads; idx < nvec; idx += kThreads)
            amax = fmaxf(amax, absmax_bf16x8(__ldg(src + idx)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
        __syncthreads();
        amax = warp_max[0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) amax = fmaxf(amax, warp_max[w]);
        __syncthreads();  // warp_max is reused by the next row
        const int e = e4m3_row_exponent(amax);
        const float inv = pow2f(-e);
        if (threadIdx.x == 0) scale[r] = pow2f(e);
#pragma unroll
        for (int i = 0; i < kCached; ++i) {
            const int idx = threadIdx.x + i * kThreads;
            if (idx < nvec) dst[idx] = e4m3_quant8(v[i], inv);
        }
        for (int idx = threadIdx.x + kCached * kThreads; idx < nvec; idx += kThreads)
            dst[idx] = e4m3_quant8(__ldg(src + idx), inv);
    }
}

}  // namespace

cudaError_t launch_quantize_rows_e4m3(const void* a, long long R, int K, void* q, float* scale, int num_sms,
                                      cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    long long grid = R;
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (grid > cap) grid = cap;
    quantize_rows_e4m3_kernel<<<static_cast<int>(grid), kThreads, 0, s>>>(static_cast<const uint4*>(a), R, K / 8,
                                                                          static_cast<uint2*>(q), scale);
    return cudaGetLastError();
}

}  // namespace sptp
