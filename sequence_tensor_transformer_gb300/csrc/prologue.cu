// Boundary prologue: reduce-scatter arithmetic + residual add + RMSNorm
// ("[Feature] Async Tensor Parallelism for Archon Engine", "Potential
// Solution": the window between the reduce-scatter ending one sub-layer and
// the all-gather starting the next).  HBM-bound: every input byte is read
// once with 128-bit coalesced loads, every output byte written once.
//
// One warp per token row.  Lane l owns the 16-byte column vectors
// l, l+32, l+64, ... of the row and keeps h in fp32 registers, so the row
// is read once; the sum of squares is reduced with warp shuffles.
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

// Row fits in registers: NV vectors of E elements per lane.
template <typename T, int NV>
__global__ void __launch_bounds__(128) prologue_regs(const __grid_constant__ PrologueParams p) {
    using V = Vec<T>;
    constexpr int E = V::E;
    const int lane = threadIdx.x & 31;
    const long long warps_total = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const long long total_rows = static_cast<long long>(p.G) * p.M;
    const int d = p.d;
    for (long long gr = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); gr < total_rows;
         gr += warps_total) {
        const int g = static_cast<int>(gr / p.M);
        const long long row = gr - static_cast<long long>(g) * p.M;
        const PrologueGroup& grp = p.grp[g];
        const long long base = row * d;
        float h[NV][E];
        float ss = 0.f;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int col = (v * 32 + lane) * E;
            if (col < d) {
                float r[E];
#pragma unroll
                for (int e = 0; e < E; ++e) r[e] = 0.f;
                for (int s = 0; s < grp.n_src; ++s) {
                    float t[E];
                    V::load_stream(p.src[grp.src_begin + s], base + col, t);
#pragma unroll
                    for (int e = 0; e < E; ++e) r[e] += t[e];
                }
                float xv[E];
                V::load_stream(grp.x, base + col, xv);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    h[v][e] = xv[e] + r[e];
                    ss = fmaf(h[v][e], h[v][e], ss);
                }
            }
        }
        if (grp.h != nullptr) {
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int col = (v * 32 + lane) * E;
                if (col < d) V::store(grp.h, base + col, h[v]);
            }
        }
        if (grp.y != nullptr) {
            ss = warp_sum(ss);
            const float inv = rsqrtf(ss / static_cast<float>(d) + p.eps);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int col = (v * 32 + lane) * E;
                if (col < d) {
                    float gm[E];
                    V::load(p.gamma, col, gm);
#pragma unroll
                    for (int e = 0; e < E; ++e) gm[e] = h[v][e] * inv * gm[e];
                    V::store(grp.y, base + col, gm);
                }
            }
        }
    }
}

// Any d: two passes over the row (the second re-reads it from cache).
template <typename T>
__global__ void __launch_bounds__(128) prologue_two_pass(const __grid_constant__ PrologueParams p) {
    using V = Vec<T>;
    constexpr int E = V::E;
    const int lane = threadIdx.x & 31;
    const long long warps_total = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const long long total_rows = static_cast<long long>(p.G) * p.M;
    const int d = p.d;
    for (long long gr = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); gr < total_rows;
         gr += warps_total) {
        const int g = static_cast<int>(gr / p.M);
        const long long row = gr - static_cast<long long>(g) * p.M;
        const PrologueGroup& grp = p.grp[g];
        const long long base = row * d;
        float ss = 0.f;
        for (int pass = 0; pass < 2; ++pass) {
            float inv = 0.f;
            if (pass == 1) {
                if (grp.y == nullptr && grp.h == nullptr) break;
                ss = warp_sum(ss);
                inv = rsqrtf(ss / static_cast<float>(d) + p.eps);
            }
            for (int col = lane * E; col < d; col += 32 * E) {
                float r[E], h[E];
#pragma unroll
                for (int e = 0; e < E; ++e) r[e] = 0.f;
                for (int s = 0; s < grp.n_src; ++s) {
                    float t[E];
                    V::load(p.src[grp.src_begin + s], base + col, t);
#pragma unroll
                    for (int e = 0; e < E; ++e) r[e] += t[e];
                }
                float xv[E];
                V::load(grp.x, base + col, xv);
#pragma unroll
                for (int e = 0; e < E; ++e) h[e] = xv[e] + r[e];
                if (pass == 0) {
#pragma unroll
                    for (int e = 0; e < E; ++e) ss = fmaf(h[e], h[e], ss);
                } else {
                    // pass 1 reads x again, so h may alias x only after the
                    // read of this vector (it is: same lane, same column)
                    if (grp.y != nullptr) {
                        float gm[E];
                        V::load(p.gamma, col, gm);
#pragma unroll
                        for (int e = 0; e < E; ++e) gm[e] = h[e] * inv * gm[e];
                        V::store(grp.y, base + col, gm);
                    }
                    if (grp.h != nullptr) V::store(grp.h, base + col, h);
                }
            }
        }
    }
}

template <typename T, int NV>
cudaError_t launch_regs(const PrologueParams& p, int grid, cudaStream_t s) {
    prologue_regs<T, NV><<<grid, 128, 0, s>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const PrologueParams& p, int num_sms, cudaStream_t s) {
    constexpr int E = Vec<T>::E;
    const long long rows = static_cast<long long>(p.G) * p.M;
    if (rows == 0) return cudaSuccess;
    long long grid = (rows + 3) / 4;  // 4 warps (rows) per block
    const long long cap = static_cast<long long>(num_sms) * 16;
    if (grid > cap) grid = cap;
    const int nv = (p.d + 32 * E - 1) / (32 * E);
    const int g = static_cast<int>(grid);
    if (nv <= 1) return launch_regs<T, 1>(p, g, s);
    if (nv <= 2) return launch_regs<T, 2>(p, g, s);
    if (nv <= 4) return launch_regs<T, 4>(p, g, s);
    if (nv <= 8) return launch_regs<T, 8>(p, g, s);
    if (nv <= 12) return launch_regs<T, 12>(p, g, s);
    if (nv <= 16) return launch_regs<T, 16>(p, g, s);
    prologue_two_pass<T><<<g, 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prologue(const PrologueParams& p, bool bf16, int num_sms, cudaStream_t s) {
    return bf16 ? launch_typed<__nv_bfloat16>(p, num_sms, s) : launch_typed<float>(p, num_sms, s);
}

}  // namespace sptp
