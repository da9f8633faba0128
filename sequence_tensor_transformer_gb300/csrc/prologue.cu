// Boundary prologue: reduce-scatter arithmetic + residual add + RMSNorm
// ("[Feature] Async Tensor Parallelism for Archon Engine", "Potential
// Solution": the window between the reduce-scatter ending one sub-layer and
// the all-gather starting the next).  HBM-bound: every input byte is read
// once with 128-bit coalesced loads, every output byte written once.
//
// A group of threads per token row, one 16-byte column vector per thread and
// source, so every thread's loads are independent and in flight together; h
// stays in fp32 registers, so the row is read once.
// Summation order per element: r = ((0 + src_0) + src_1) + ... (fp32, list
// order; no sources gives r = 0),
// h = x + r; the norm uses the unrounded fp32 h.
#include <cuda_bf16.h>

#include "sptp_internal.h"

namespace sptp {

namespace {

template <typename T>
struct Vec;

template <>
struct Vec<__nv_bfloat16> {
    static constexpr int E = 8;
    __device__ static void load(const void* base, long long idx, float (&f)[8]) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + idx));
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 v = __bfloat1622float2(h2[i]);
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    }
    // streaming load (inputs read exactly once)
    __device__ static void load_stream(const void* base, long long idx, float (&f)[8]) {
        const uint4 u = __ldcs(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + idx));
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 v = __bfloat1622float2(h2[i]);
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    }
    __device__ static void store(void* base, long long idx, const float (&f)[8]) {
        uint4 u;
        __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) h2[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + idx) = u;
    }
};

template <>
struct Vec<float> {
    static constexpr int E = 4;
    __device__ static void load(const void* base, long long idx, float (&f)[4]) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx));
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
    __device__ static void load_stream(const void* base, long long idx, float (&f)[4]) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx));
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
    __device__ static void store(void* base, long long idx, const float (&f)[4]) {
        *reinterpret_cast<float4*>(static_cast<float*>(base) + idx) = make_float4(f[0], f[1], f[2], f[3]);
    }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One group of `tpr` threads (a multiple of 32) per token row, R rows per CTA;
// thread t of a group owns the 16-byte column vectors t, t+tpr, ... (VPT of
// them), so each thread issues its (sources + 1) x VPT loads back to back.
// The row's sum of squares is reduced with warp shuffles and, when a row
// spans several warps, through a double-buffered shared array (one
// __syncthreads per row).
template <typename T, int VPT>
__global__ void __launch_bounds__(1024) prologue_rows(const __grid_constant__ PrologueParams p, int tpr, int R) {
    using V = Vec<T>;
    constexpr int E = V::E;
    extern __shared__ float red[];  // [2][R][tpr / 32]
    const int grp = threadIdx.x / tpr;
    const int t = threadIdx.x - grp * tpr;
    const int lane = threadIdx.x & 31;
    const int wpr = tpr >> 5;
    const int wir = t >> 5;
    const long long total = static_cast<long long>(p.G) * p.M;
    const int d = p.d;
    int parity = 0;
    for (long long base = static_cast<long long>(blockIdx.x) * R; base < total;
         base += static_cast<long long>(gridDim.x) * R) {
        const long long gr = base + grp;
        const bool active = gr < total;
        const int g = active ? static_cast<int>(gr / p.M) : 0;
        const long long row = active ? gr - static_cast<long long>(g) * p.M : 0;
        const PrologueGroup& grpd = p.grp[g];
        const long long off = row * d;
        float h[VPT][E];
        float ss = 0.f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int col = (v * tpr + t) * E;
            if (active && col < d) {
                float r[E];
#pragma unroll
                for (int e = 0; e < E; ++e) r[e] = 0.f;
#pragma unroll 4
                for (int s = 0; s < grpd.n_src; ++s) {
                    float u[E];
                    V::load_stream(p.src[grpd.src_begin + s], off + col, u);
#pragma unroll
                    for (int e = 0; e < E; ++e) r[e] += u[e];
                }
                float xv[E];
                V::load_stream(grpd.x, off + col, xv);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    h[v][e] = xv[e] + r[e];
                    ss = fmaf(h[v][e], h[v][e], ss);
                }
            }
        }
        ss = warp_sum(ss);
        if (wpr > 1) {
            float* slot = red + (parity * R + grp) * wpr;
            if (lane == 0) slot[wir] = ss;
            __syncthreads();
            ss = 0.f;
            for (int w = 0; w < wpr; ++w) ss += slot[w];
            parity ^= 1;
        }
        if (!active) continue;
        const float inv = rsqrtf(ss / static_cast<float>(d) + p.eps);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int col = (v * tpr + t) * E;
            if (col < d) {
                if (grpd.h != nullptr) V::store(grpd.h, off + col, h[v]);
                if (grpd.y != nullptr) {
                    float gm[E];
                    V::load(p.gamma, col, gm);
#pragma unroll
                    for (int e = 0; e < E; ++e) gm[e] = h[v][e] * inv * gm[e];
                    V::store(grpd.y, off + col, gm);
                }
            }
        }
    }
}

template <typename T>
cudaError_t launch_typed(const PrologueParams& p, int num_sms, cudaStream_t s) {
    constexpr int E = Vec<T>::E;
    const long long rows = static_cast<long long>(p.G) * p.M;
    if (rows == 0) return cudaSuccess;
    const int nvec = (p.d + E - 1) / E;
    int vpt = 1;
    while ((nvec + vpt - 1) / vpt > 1024) vpt *= 2;
    if (vpt > 4) return cudaErrorInvalidValue;
    const int tpr = (((nvec + vpt - 1) / vpt) + 31) / 32 * 32;
    const int R = tpr >= 256 ? 1 : 256 / tpr;
    const int block = tpr * R;
    const size_t smem = static_cast<size_t>(2) * R * (tpr / 32) * sizeof(float);
    long long grid = (rows + R - 1) / R;
    const long long cap = static_cast<long long>(num_sms) * (2048 / block);
    if (grid > cap) grid = cap;
    const int g = static_cast<int>(grid);
    if (vpt == 1) prologue_rows<T, 1><<<g, block, smem, s>>>(p, tpr, R);
    else if (vpt == 2) prologue_rows<T, 2><<<g, block, smem, s>>>(p, tpr, R);
    else prologue_rows<T, 4><<<g, block, smem, s>>>(p, tpr, R);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prologue(const PrologueParams& p, bool bf16, int num_sms, cudaStream_t s) {
    return bf16 ? launch_typed<__nv_bfloat16>(p, num_sms, s) : launch_typed<float>(p, num_sms, s);
}

}  // namespace sptp
