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

#include "e4m3.cuh"
#include "sptp_ptx.cuh"

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
    __device__ static void load_smem(const uint8_t* base, int idx, float (&f)[8]) {
        const uint4 u = *reinterpret_cast<const uint4*>(base + static_cast<size_t>(idx) * 2);
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
    // evict-first store (final outputs nobody reads next)
    __device__ static void store_stream(void* base, long long idx, const float (&f)[8]) {
        uint4 u;
        __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) h2[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        __stcs(reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + idx), u);
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
    __device__ static void load_smem(const uint8_t* base, int idx, float (&f)[4]) {
        const float4 v = *reinterpret_cast<const float4*>(base + static_cast<size_t>(idx) * 4);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
    __device__ static void store(void* base, long long idx, const float (&f)[4]) {
        *reinterpret_cast<float4*>(static_cast<float*>(base) + idx) = make_float4(f[0], f[1], f[2], f[3]);
    }
    __device__ static void store_stream(void* base, long long idx, const float (&f)[4]) {
        __stcs(reinterpret_cast<float4*>(static_cast<float*>(base) + idx), make_float4(f[0], f[1], f[2], f[3]));
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
        // no division for one group; a 32-bit one otherwise (G * M < 2^31)
        const int g = gr < total && p.G > 1 ? static_cast<int>(static_cast<uint32_t>(gr) / static_cast<uint32_t>(p.M))
                                            : 0;
        const long long row = gr < total ? gr - static_cast<long long>(g) * p.M : 0;
        // a checked build: the (group, row) and the group's source list
        const bool active = gr < total &&
                            checked(g < p.G && row < p.M && p.grp[g].src_begin >= 0 &&
                                        p.grp[g].src_begin + p.grp[g].n_src <= kMaxSrc,
                                    p.status, nullptr, kWhereBoundsTile, gr);
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
                    for (int e = 0; e < E; ++e) gm[e] = (h[v][e] * gm[e]) * inv;
                    V::store(grpd.y, off + col, gm);
                }
            }
        }
    }
}

// Rows streamed through shared memory: thread 0 bulk-copies the (sources +
// 1) input rows of the CTA's next rows into an S-stage ring (one mbarrier per
// stage); the CTA's threads reduce the row from shared memory (VPT 16-byte
// vectors each, gamma held in registers) and store h and y with coalesced
// 16-byte stores (h, a final output, with evict-first hints; y stays in L2
// for the gate/up GEMM).  One __syncthreads per row: it completes the row's
// sum of squares and frees the row's stage, which thread 0 then refills with
// the row S ahead.  A CTA handles rows blockIdx.x, blockIdx.x + gridDim.x, ...
constexpr int kTmaMaxStages = 8;

struct TmaLayout {
    int S;              // stages
    int max_src;        // sources per stage slot (max over groups)
    uint32_t row_bytes; // d * sizeof(T)
};

//
// y_j = (h_j * gamma_j) * rsqrt(mean h^2 + eps), each product rounded to fp32.
// QUANT (bf16, one group): instead of y, write y's E4M3 codes and row scale
// (codes of y * 2^-e, e from the row maximum A of the bf16 y).  Rounding is
// monotone and sign-symmetric, so A = bf16(m * rsqrt) exactly, with
// m = max_j |h_j * gamma_j|: m joins the first block reduction and the row
// needs no second barrier.
template <typename T, int VPT, bool QUANT>
__global__ void __launch_bounds__(512) prologue_tma(const __grid_constant__ PrologueParams p, TmaLayout L) {
    using V = Vec<T>;
    constexpr int E = V::E;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    __shared__ uint64_t full[kTmaMaxStages];
    __shared__ __align__(16) float red[2][16];
    __shared__ __align__(16) float red_mg[2][16];
    __shared__ int abort_flag;
    const int nthr = blockDim.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
    const long long total = static_cast<long long>(p.G) * p.M;
    const int d = p.d;
    const uint32_t slot_bytes = L.row_bytes;
    const uint32_t stage_bytes = slot_bytes * static_cast<uint32_t>(L.max_src + 1);
    const long long first = blockIdx.x, stride = gridDim.x;
    const long long my_rows = first < total ? (total - first + stride - 1) / stride : 0;

    if (tid == 0) {
        for (int s = 0; s < L.S; ++s) mbar_init(&full[s], 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // (group, row) of global row gr: no division when there is one group;
    // otherwise a 32-bit one (G * M < 2^31 is checked at launch)
    auto locate = [&](long long gr, int& g, long long& row) {
        if (p.G == 1) {
            g = 0;
            row = gr;
        } else {
            const uint32_t q = static_cast<uint32_t>(gr) / static_cast<uint32_t>(p.M);
            g = static_cast<int>(q);
            row = gr - static_cast<long long>(q) * p.M;
        }
    };
    // thread 0: start the copies of this CTA's i-th row into stage s (= i % S)
    auto issue = [&](long long i, int s) {
        int g;
        long long row;
        locate(first + i * stride, g, row);
        const PrologueGroup& grp = p.grp[g];
        uint8_t* st = smem + static_cast<size_t>(s) * stage_bytes;
        // a checked build: the (group, row), the group's sources and the
        // stage; a failed check copies nothing, the row's wait gives up
        if (!checked(g < p.G && row < p.M && grp.src_begin >= 0 && grp.src_begin + grp.n_src <= kMaxSrc &&
                         grp.n_src <= L.max_src && s < L.S,
                     p.status, &abort_flag, kWhereBoundsLoad, row))
            return;
        mbar_arrive_expect_tx(&full[s], slot_bytes * static_cast<uint32_t>(grp.n_src + 1));
        const long long off = row * static_cast<long long>(slot_bytes);
        bulk_load(st, static_cast<const uint8_t*>(grp.x) + off, slot_bytes, &full[s]);
        for (int j = 0; j < grp.n_src; ++j)
            bulk_load(st + static_cast<size_t>(j + 1) * slot_bytes,
                      static_cast<const uint8_t*>(p.src[grp.src_begin + j]) + off, slot_bytes, &full[s]);
    };
    if (tid == 0)
        for (long long i = 0; i < L.S && i < my_rows; ++i) issue(i, static_cast<int>(i));

    float gm[VPT][E];
    if (p.gamma != nullptr) {
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int col = (v * nthr + tid) * E;
            if (col < d) V::load(p.gamma, col, gm[v]);
        }
    }

    WaitCtx wc{p.status, &abort_flag, p.wait_limit_ns};
    int parity = 0;
    int s = 0;           // stage of row i: i % S, kept by counting
    uint32_t phase = 0;  // (i / S) & 1
    long long i = 0;
    for (; i < my_rows; ++i) {
        const bool ok = mbar_wait(&full[s], phase, wc, kWherePrologueFull, static_cast<int>(i));
        int g;
        long long row;
        locate(first + i * stride, g, row);
        const PrologueGroup& grp = p.grp[g];
        const uint8_t* st = smem + static_cast<size_t>(s) * stage_bytes;
        const long long off = row * d;
        float hg[VPT][E];  // h * gamma; h itself is stored at once
        float ss = 0.f, mg = 0.f;
        if (ok) {
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int col = (v * nthr + tid) * E;
                if (col < d) {
                    float r[E];
#pragma unroll
                    for (int e = 0; e < E; ++e) r[e] = 0.f;
                    for (int j = 0; j < grp.n_src; ++j) {
                        float u[E];
                        V::load_smem(st + static_cast<size_t>(j + 1) * slot_bytes, col, u);
#pragma unroll
                        for (int e = 0; e < E; ++e) r[e] += u[e];
                    }
                    float hv[E];
                    V::load_smem(st, col, hv);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        hv[e] += r[e];
                        ss = fmaf(hv[e], hv[e], ss);
                        hg[v][e] = hv[e] * gm[v][e];
                        if constexpr (QUANT) mg = fmaxf(mg, fabsf(hg[v][e]));
                    }
                    // h (the new residual, a final output) needs no norm
                    if (grp.h != nullptr) V::store_stream(grp.h, off + col, hv);
                }
            }
        }
        ss = warp_sum(ss);
        if (lane == 0) red[parity][warp] = ss;
        if constexpr (QUANT) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, o));
            if (lane == 0) red_mg[parity][warp] = mg;
        }
        __syncthreads();
        if (abort_flag) break;  // uniform: written before the barrier
        if (tid == 0 && i + L.S < my_rows) {
            // every thread has read stage s; order those reads before the
            // copies that overwrite it
            fence_proxy_async_smem();
            issue(i + L.S, s);
        }
        // the per-warp values in ascending warp order (16-byte reads)
        ss = 0.f;
        if ((nwarps & 3) == 0) {
            for (int w = 0; w < nwarps; w += 4) {
                const float4 q4 = *reinterpret_cast<const float4*>(&red[parity][w]);
                ss = (((ss + q4.x) + q4.y) + q4.z) + q4.w;
                if constexpr (QUANT) {
                    const float4 m4 = *reinterpret_cast<const float4*>(&red_mg[parity][w]);
                    mg = fmaxf(mg, fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w)));
                }
            }
        } else {
            for (int w = 0; w < nwarps; ++w) {
                ss += red[parity][w];
                if constexpr (QUANT) mg = fmaxf(mg, red_mg[parity][w]);
            }
        }
        parity ^= 1;
        const float inv = rsqrtf(ss / static_cast<float>(d) + p.eps);
        if constexpr (!QUANT) {
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int col = (v * nthr + tid) * E;
                if (col < d) {
                    if (grp.y != nullptr) {
                        float yv[E];
#pragma unroll
                        for (int e = 0; e < E; ++e) yv[e] = hg[v][e] * inv;
                        V::store(grp.y, off + col, yv);
                    }
                }
            }
        } else {
            static_assert(E == 8, "bf16 rows only");
            // the bf16 activation y
            uint4 yb[VPT];
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int col = (v * nthr + tid) * E;
                if (col < d) {
                    __nv_bfloat162* b2 = reinterpret_cast<__nv_bfloat162*>(&yb[v]);
#pragma unroll
                    for (int e = 0; e < E / 2; ++e)
                        b2[e] = __floats2bfloat162_rn(hg[v][2 * e] * inv, hg[v][2 * e + 1] * inv);
                }
            }
            const int ex = e4m3_row_exponent(__bfloat162float(__float2bfloat16_rn(mg * inv)));
            const float qinv = pow2f(-ex);
            if (tid == 0) p.qscale[row] = pow2f(ex);
            uint8_t* qrow = static_cast<uint8_t*>(p.q) + off;
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int col = (v * nthr + tid) * E;
                if (col < d) *reinterpret_cast<uint2*>(qrow + col) = e4m3_quant8(yb[v], qinv);
            }
        }
        if (++s == L.S) {
            s = 0;
            phase ^= 1u;
        }
    }
    if (i < my_rows && tid == 0) {
        // left early: wait (bounded) for copies still in flight into the ring
        int local_abort = 0;
        WaitCtx drain{p.status, &local_abort, p.wait_limit_ns};
        for (long long j = i; j < my_rows && j < i + L.S; ++j)
            mbar_wait(&full[j % L.S], static_cast<uint32_t>((j / L.S) & 1), drain, kWhereDrain, -1);
    }
}

template <typename T, int VPT, bool QUANT = false>
cudaError_t launch_tma(const PrologueParams& p, const TmaLayout& L, int threads, int num_sms, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(L.S) * L.row_bytes * (L.max_src + 1) + 128;
    cudaError_t e = cudaFuncSetAttribute(prologue_tma<T, VPT, QUANT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const long long rows = static_cast<long long>(p.G) * p.M;
    int per_sm = static_cast<int>((200u * 1024u) / smem);
    const int by_threads = 2048 / threads;
    if (per_sm > by_threads) per_sm = by_threads;
    if (per_sm > 8) per_sm = 8;
    if (per_sm < 1) per_sm = 1;
    long long grid = static_cast<long long>(num_sms) * per_sm;
    if (grid > rows) grid = rows;
    prologue_tma<T, VPT, QUANT><<<static_cast<int>(grid), threads, smem, s>>>(p, L);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_typed(const PrologueParams& p, int num_sms, cudaStream_t s) {
    constexpr int E = Vec<T>::E;
    const long long rows = static_cast<long long>(p.G) * p.M;
    if (rows == 0) return cudaSuccess;
    if (p.G > 1 && rows >= (1ll << 31)) return cudaErrorInvalidValue;  // the kernels' 32-bit row split
    const int nvec = (p.d + E - 1) / E;

    // Shared-memory streaming path: rows of all sources staged by bulk copies.
    int max_src = 0;
    for (int g = 0; g < p.G; ++g) max_src = p.grp[g].n_src > max_src ? p.grp[g].n_src : max_src;
    const size_t stage_bytes = static_cast<size_t>(p.d) * sizeof(T) * (max_src + 1);
    int S = static_cast<int>((96u * 1024u) / stage_bytes);
    if (S > 4) S = 4;
    if (S < 2 && 2 * stage_bytes <= 200u * 1024u) S = 2;
    // up to 512 threads, one 16-byte vector each per source when it fits
    const int threads = nvec <= 512 ? (nvec + 31) / 32 * 32 : 512;
    const int vpt = (nvec + threads - 1) / threads;
    if (S >= 2 && vpt <= 8) {
        TmaLayout L{S, max_src, static_cast<uint32_t>(p.d * sizeof(T))};
        if constexpr (sizeof(T) == 2) {
            if (p.q != nullptr) {
                if (vpt <= 1) return launch_tma<T, 1, true>(p, L, threads, num_sms, s);
                if (vpt <= 2) return launch_tma<T, 2, true>(p, L, threads, num_sms, s);
                if (vpt <= 4) return launch_tma<T, 4, true>(p, L, threads, num_sms, s);
                return launch_tma<T, 8, true>(p, L, threads, num_sms, s);
            }
        }
        if (vpt <= 1) return launch_tma<T, 1>(p, L, threads, num_sms, s);
        if (vpt <= 2) return launch_tma<T, 2>(p, L, threads, num_sms, s);
        if (vpt <= 4) return launch_tma<T, 4>(p, L, threads, num_sms, s);
        return launch_tma<T, 8>(p, L, threads, num_sms, s);
    }

    // Register path (rows too wide for the shared-memory ring).
    int vptr = 1;
    while ((nvec + vptr - 1) / vptr > 1024) vptr *= 2;
    if (vptr > 4) return cudaErrorInvalidValue;
    const int tpr = (((nvec + vptr - 1) / vptr) + 31) / 32 * 32;
    const int R = tpr >= 256 ? 1 : 256 / tpr;
    const int block = tpr * R;
    const size_t smem = static_cast<size_t>(2) * R * (tpr / 32) * sizeof(float);
    long long grid = (rows + R - 1) / R;
    const long long cap = static_cast<long long>(num_sms) * (2048 / block);
    if (grid > cap) grid = cap;
    const int g = static_cast<int>(grid);
    if (vptr == 1) prologue_rows<T, 1><<<g, block, smem, s>>>(p, tpr, R);
    else if (vptr == 2) prologue_rows<T, 2><<<g, block, smem, s>>>(p, tpr, R);
    else prologue_rows<T, 4><<<g, block, smem, s>>>(p, tpr, R);
    cudaError_t e = cudaGetLastError();
    // rows too wide for the fused quantisation: quantise the stored y
    if (e == cudaSuccess && p.q != nullptr)
        e = launch_quantize_rows_e4m3(p.grp[0].y, p.M, p.d, p.q, p.qscale, num_sms, s);
    return e;
}

}  // namespace

cudaError_t launch_prologue(const PrologueParams& p, bool bf16, int num_sms, cudaStream_t s) {
    if (p.q != nullptr && (!bf16 || p.G != 1 || p.grp[0].y == nullptr || p.qscale == nullptr))
        return cudaErrorInvalidValue;
    return bf16 ? launch_typed<__nv_bfloat16>(p, num_sms, s) : launch_typed<float>(p, num_sms, s);
}

}  // namespace sptp
