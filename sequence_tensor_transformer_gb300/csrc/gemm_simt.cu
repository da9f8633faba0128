// fp32 CUDA-core GEMMs for the fp32 boundary workloads (TF32 tensor cores
// cannot meet a 1e-5 relative error bound).  Same two shapes as the tcgen05
// path: gate/up with a SwiGLU epilogue and the per-shard down projection,
// C_g[m][n] = sum_k A_g[m][k] * B_g[n][k] with both operands K-contiguous.
// T x T tile per CTA (64, or 32 where 64-wide tiles would leave most SMs
// idle), 32-deep K slices staged in shared memory (the next slice's loads in
// flight in registers while the current one is multiplied), T/16 x T/16
// outputs per thread, fp32 FMA in ascending k: the same arithmetic per
// output for either tile.
#include "sptp_internal.h"

namespace sptp {

namespace {

constexpr int TK = 32;

template <Epi EPI, int T>
__global__ void __launch_bounds__(256) simt_gemm_nt(const __grid_constant__ SimtGemmParams p) {
    constexpr bool SWI = EPI == Epi::kSwiGLU;
    constexpr int TM = T, TN = T, R = T / 16;  // R x R outputs per thread
    constexpr int kLoads = TM * TK / 256;      // elements of each operand a thread stages per slice
    __shared__ float As[TK][TM + 4];
    __shared__ float Bs0[TK][TN + 4];
    __shared__ float Bs1[SWI ? TK : 1][SWI ? TN + 4 : 1];
    const int g = blockIdx.z;
    const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const float* A = p.A[g];
    const float* B0 = p.B0[g];
    const float* B1 = p.B1[g];
    float acc0[R][R] = {}, acc1[R][R] = {};
    // slice k0 of both operands into registers (zero past M, N or K)
    float ra[kLoads], rb0[kLoads], rb1[SWI ? kLoads : 1];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int i = 0; i < kLoads; ++i) {
            const int idx = threadIdx.x + i * 256;
            const int r = idx / TK, kk = idx % TK;
            const int k = k0 + kk;
            const int am = m0 + r, bn = n0 + r;
            ra[i] = (am < p.M && k < p.K) ? A[static_cast<long long>(am) * p.lda + k] : 0.f;
            rb0[i] = (bn < p.N && k < p.K) ? B0[static_cast<long long>(bn) * p.ldb + k] : 0.f;
            if (SWI) rb1[i] = (bn < p.N && k < p.K) ? B1[static_cast<long long>(bn) * p.ldb + k] : 0.f;
        }
    };
    fetch(0);
    for (int k0 = 0; k0 < p.K; k0 += TK) {
#pragma unroll
        for (int i = 0; i < kLoads; ++i) {
            const int idx = threadIdx.x + i * 256;
            const int r = idx / TK, kk = idx % TK;
            As[kk][r] = ra[i];
            Bs0[kk][r] = rb0[i];
            if (SWI) Bs1[kk][r] = rb1[i];
        }
        __syncthreads();
        if (k0 + TK < p.K) fetch(k0 + TK);  // in flight during this slice's FMAs
#pragma unroll
        for (int kk = 0; kk < TK; ++kk) {
            float a[R], b0[R], b1[R];
#pragma unroll
            for (int i = 0; i < R; ++i) a[i] = As[kk][ty * R + i];
#pragma unroll
            for (int j = 0; j < R; ++j) {
                b0[j] = Bs0[kk][tx * R + j];
                if (SWI) b1[j] = Bs1[kk][tx * R + j];
            }
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
                for (int j = 0; j < R; ++j) {
                    acc0[i][j] = fmaf(a[i], b0[j], acc0[i][j]);
                    if (SWI) acc1[i][j] = fmaf(a[i], b1[j], acc1[i][j]);
                }
        }
        __syncthreads();
    }
    float* C = p.C[g];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int m = m0 + ty * R + i;
        if (m >= p.M) continue;
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const int n = n0 + tx * R + j;
            if (n >= p.N) continue;
            float v = acc0[i][j];
            if (SWI) v = v / (1.0f + expf(-v)) * acc1[i][j];
            C[m * p.ldc + n] = v;
        }
    }
}

}  // namespace

cudaError_t launch_simt_gemm(const SimtGemmParams& p, Epi epi, cudaStream_t s) {
    if (p.M == 0 || p.N == 0 || p.G == 0) return cudaSuccess;
    // 64-wide tiles unless they would give fewer CTAs than half the SMs of
    // this GPU (152): then 32-wide ones, four times as many
    const long long tiles64 = static_cast<long long>((p.N + 63) / 64) * ((p.M + 63) / 64) * p.G;
    const int T = tiles64 < 76 ? 32 : 64;
    dim3 grid((p.N + T - 1) / T, (p.M + T - 1) / T, p.G);
    if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
    if (epi == Epi::kSwiGLU) {
        if (T == 32)
            simt_gemm_nt<Epi::kSwiGLU, 32><<<grid, 256, 0, s>>>(p);
        else
            simt_gemm_nt<Epi::kSwiGLU, 64><<<grid, 256, 0, s>>>(p);
    } else {
        if (T == 32)
            simt_gemm_nt<Epi::kStore, 32><<<grid, 256, 0, s>>>(p);
        else
            simt_gemm_nt<Epi::kStore, 64><<<grid, 256, 0, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace sptp
