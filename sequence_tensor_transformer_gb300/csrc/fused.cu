// Fused persistent SP-TP FFN boundary ("[Feature] Async Tensor Parallelism for
// Archon Engine", "Potential Solution": decompose all-gather + matmul into
// chunked pipelined operations, and overlap the sub-layer boundary's residual
// add + RMSNorm with the matmuls).
//
// One launch of CTA pairs (cta_group::2, one CTA per SM, all co-resident)
// computes the whole boundary:
//   warps 6..13  prologue: rows in sequence order: h = x + sum_p
//                partials[p], y = RMSNorm(h) * gamma; after each row a
//                release increment of its sequence chunk's counter (a chunk
//                is "gathered" once all its rows are produced)
//   warp 0       TMA producer: before a gate/up tile's first A load it waits
//                (bounded) until every sequence chunk its 256 rows overlap is
//                complete; before a down tile's, until every gate/up tile of
//                its (shard, rows) has been stored
//   warp 1       MMA issuer of the even CTA (M=256, N=256, K=16 UMMAs)
//   warps 2..5   epilogue: SwiGLU into s (then a release increment of the
//                (shard, 256-row block) counter) or the bf16 partials out
// The tile sequence is all gate/up tiles (raster bands of `band` 256-row
// tiles), then all down tiles; pair q takes tiles q, q + npairs, ...  Every
// dependency points to work earlier in that order or to prologue rows, which
// never wait, so with all CTAs resident every wait ends.
//
// With p.qkv set the same launch is the boundary in front of an attention
// sub-layer (the pages' 4 boundaries per block): the prologue rows feed a
// column-parallel store GEMM of each shard's Wqkv rows instead of gate/up,
// and there are no down tiles.
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "sptp_ptx.cuh"

namespace sptp {

namespace {

constexpr int BK = 64;
constexpr int PBM = 256, PBN = 256;
constexpr int STAGES = 6;
constexpr int A_BYTES = 128 * BK * 2;
constexpr int B_BYTES = 128 * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int PRO_WARPS = 8;
constexpr int THREADS = 32 * (6 + PRO_WARPS);
constexpr uint32_t IDESC = idesc_bf16_f32(PBM, PBN);

struct Bars {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Bars) <= BAR_BYTES, "barrier block too large");

struct Tile {
    bool down;
    int g, m, n;
};

// Tile t of the sequence.  Gate/up tiles: a first raster band of band0
// m-tiles (one sequence chunk, so the first wave waits only for that chunk's
// rows), then bands of `band`; down tiles: bands of `band`.  Inside a band the
// m-tile index runs fastest.
__device__ __forceinline__ Tile decode(const FusedParams& p, int t) {
    Tile r;
    r.down = t >= p.tiles_gu;
    const int nt = r.down ? p.nt_dn : p.nt_gu;
    int m0 = 0;
    if (r.down) {
        t -= p.tiles_gu;
    } else {
        const int first = p.band0 * p.P * nt;
        if (t < first) {
            r.m = t % p.band0;
            const int gn = t / p.band0;
            r.g = gn / nt;
            r.n = gn - r.g * nt;
            return r;
        }
        t -= first;
        m0 = p.band0;
    }
    const int per_band = p.band * p.P * nt;
    const int b = t / per_band;
    const int rr = t - b * per_band;
    m0 += b * p.band;
    const int bm = min(p.band, p.mt - m0);
    r.m = m0 + rr % bm;
    const int gn = rr / bm;
    r.g = gn / nt;
    r.n = gn - r.g * nt;
    return r;
}

// A checked build: the decoded tile lies in the launch's tile grid.
__device__ __forceinline__ bool tile_ok(const FusedParams& p, const Tile& tl, volatile int* abort_flag) {
    if constexpr (kBoundsChecked) {
        const int nt = tl.down ? p.nt_dn : p.nt_gu;
        const bool ok = tl.g >= 0 && tl.g < p.P && tl.m >= 0 && tl.m < p.mt && tl.n >= 0 && tl.n < nt;
        return checked(ok, p.status, abort_flag, kWhereBoundsTile, static_cast<long long>(tl.m) * 65536 + tl.n);
    }
    return true;
}

// silu with the fast divide (<= 2 ulp in fp32, below the bf16 output rounding)
__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// OR of `v` over the 128 epilogue threads (named barrier 1).
__device__ __forceinline__ bool epilogue_any(bool v) { return named_barrier_any<1, 128>(v); }

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&f)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 v = __bfloat1622float2(h2[i]);
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 u;
    __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h2[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return u;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// h = x + (0 + partial_0 + partial_1 + ...) for NV 8-column vectors of one
// row, 256 columns apart (vectors past d are left untouched).  The loads of
// kSrcBatch sources x NV vectors are issued together before any is used
// (8 16-byte loads in flight per lane), then added in source order.  (One
// source at a time, 2 x 4 and 5 x 2 measured: the attention-side boundary's
// rows 573 / 517 / 495 us, the FFN boundary 1646 / 1653 / 1623 TFLOP/s.)  h
// accumulates the partials first and x last (one IEEE addition per element,
// so h + x equals x + h bit for bit).
constexpr int kSrcBatch = 2;

template <int NV>
__device__ __forceinline__ void row_h(const FusedParams& p, long long row_off, int col0, float (&h)[NV][8]) {
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int e = 0; e < 8; ++e) h[v][e] = 0.f;
    for (int q0 = 0; q0 <= p.P; q0 += kSrcBatch) {
        uint4 u[kSrcBatch][NV];
#pragma unroll
        for (int b = 0; b < kSrcBatch; ++b) {
            const int q = q0 + b;
            if (q > p.P) break;
            const __nv_bfloat16* src = q < p.P ? static_cast<const __nv_bfloat16*>(p.partials[q])
                                               : static_cast<const __nv_bfloat16*>(p.x);
#pragma unroll
            for (int v = 0; v < NV; ++v)
                if (col0 + 256 * v < p.d)
                    u[b][v] = __ldg(reinterpret_cast<const uint4*>(src + row_off + col0 + 256 * v));
        }
#pragma unroll
        for (int b = 0; b < kSrcBatch; ++b) {
            if (q0 + b > p.P) break;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                if (col0 + 256 * v < p.d) {
                    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u[b][v]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f2 = __bfloat1622float2(h2[i]);
                        h[v][2 * i] += f2.x;
                        h[v][2 * i + 1] += f2.y;
                    }
                }
            }
        }
    }
}

// Block-row prologue (p.block_rows): the PRO_WARPS prologue warps of a CTA take
// one row together, rows blockIdx.x, blockIdx.x + gridDim.x, ...  Thread t
// owns the 16-byte column vectors t and t + 32 * PRO_WARPS; the loads of all
// sources (partials, then x) and both vectors are issued at once, so a row
// costs one round of loads; h stays in registers (one pass), its sum of
// squares meets through shared memory at one named barrier per row, and each
// warp publishes its part of the row (PRO_WARPS increments per row).  The sum
// of squares is reduced in the standalone prologue's order (one vector per
// thread, warps of 32 vectors, warp sums added in order), so h and y match
// it bit for bit: each thread keeps one partial sum per vector.
constexpr int kBrSrc = 5;  // sources held at once: P + 1 <= 5
constexpr int kBrVec = 2;  // vectors per thread: d <= 2 * 8 * 32 * PRO_WARPS

__device__ __forceinline__ void prologue_block_rows(const FusedParams& p, int tid, int wp, int lane,
                                                    volatile int* abort_flag) {
    constexpr int NT = 32 * PRO_WARPS;
    __shared__ float red[2][kBrVec * PRO_WARPS];
    const int d = p.d;
    const int nvec = d >> 3;
    float gm[kBrVec][8];
#pragma unroll
    for (int k = 0; k < kBrVec; ++k)
        if (tid + k * NT < nvec) load8(static_cast<const __nv_bfloat16*>(p.gamma) + (tid + k * NT) * 8, gm[k]);
    int par = 0;
    const long long md = static_cast<long long>(p.M) * d;
    for (long long row = blockIdx.x; row < p.M; row += gridDim.x) {
        const long long base = row * d;
        // a checked build: every vector of the row inside [M][d] (a failed
        // check leaves the whole row out, in every thread of the CTA alike)
        if (!checked_range(base, d, md, p.status, abort_flag, kWhereBoundsLoad)) break;
        uint4 u[kBrSrc][kBrVec];
#pragma unroll
        for (int q = 0; q < kBrSrc; ++q) {
            if (q > p.P) break;
            const __nv_bfloat16* src = q < p.P ? static_cast<const __nv_bfloat16*>(p.partials[q])
                                               : static_cast<const __nv_bfloat16*>(p.x);
#pragma unroll
            for (int k = 0; k < kBrVec; ++k)
                if (tid + k * NT < nvec)
                    u[q][k] = __ldg(reinterpret_cast<const uint4*>(src + base + (tid + k * NT) * 8));
        }
        // partials in order, then x (one IEEE addition: h + x == x + h)
        float h[kBrVec][8];
        float ssk[kBrVec];
#pragma unroll
        for (int k = 0; k < kBrVec; ++k) {
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) h[k][e] = 0.f;
#pragma unroll
            for (int q = 0; q < kBrSrc; ++q) {
                if (q > p.P || tid + k * NT >= nvec) break;
                const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u[q][k]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f2 = __bfloat1622float2(h2[i]);
                    h[k][2 * i] += f2.x;
                    h[k][2 * i + 1] += f2.y;
                }
            }
            if (tid + k * NT < nvec)
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(h[k][e], h[k][e], ss);
            ssk[k] = ss;
        }
        // vector k * NT + t belongs to "warp" k * PRO_WARPS + wp of 32 vectors
#pragma unroll
        for (int k = 0; k < kBrVec; ++k) {
            const float ws = warp_sum(ssk[k]);
            if (lane == 0) red[par][k * PRO_WARPS + wp] = ws;
        }
        named_barrier_sync<2, NT>();
        float ss = 0.f;
#pragma unroll
        for (int w = 0; w < kBrVec * PRO_WARPS; ++w) ss += red[par][w];
        par ^= 1;
        const float inv = rsqrtf(ss / static_cast<float>(d) + p.eps);
#pragma unroll
        for (int k = 0; k < kBrVec; ++k) {
            const int col = (tid + k * NT) * 8;
            if (col >= d) continue;
            if (p.h_out != nullptr)
                __stcs(reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.h_out) + base + col), pack8(h[k]));
            float yv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) yv[e] = (h[k][e] * gm[k][e]) * inv;
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.y) + base + col) = pack8(yv);
        }
        // make this warp's part of y visible to the TMA loads of other CTAs
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0 && checked_index(row / p.chunk_rows, p.chunks, p.status, abort_flag, kWhereBoundsCounter))
            red_release_add(&p.chunk_ready[row / p.chunk_rows], 1);
    }
}

__global__ void __launch_bounds__(THREADS, 1) boundary_fused_kernel(const __grid_constant__ FusedParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* a_tiles = smem;
    uint8_t* b_tiles = smem + STAGES * A_BYTES;
    Bars* bars = reinterpret_cast<Bars*>(smem + STAGES * STAGE_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&bars->acc_full[a], 1);
            mbar_init(&bars->acc_empty[a], 2 * 4 * 32);
        }
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        // a checked build: the launch is a cluster of two CTAs (every peer
        // address below maps into CTA 0 or 1 of it)
        checked(cluster_nctarank() == 2 && rank < 2, p.status, &bars->abort_flag, kWhereBoundsCluster, rank);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&p.mapY);
        for (int g = 0; g < p.P; ++g) {
            tma_prefetch_map(&p.mapW1g[g]);
            if (p.qkv) continue;  // the other maps are unset
            tma_prefetch_map(&p.mapW1u[g]);
            tma_prefetch_map(&p.mapS[g]);
            tma_prefetch_map(&p.mapW2[g]);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(&bars->tmem_base, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;

    WaitCtx wc{p.status, &bars->abort_flag, p.wait_limit_ns};
    volatile int* abort_flag = &bars->abort_flag;
    // false only in a checked build whose cluster check failed: no role runs
    const bool cta_ok = bars->abort_flag == 0;
    const int total = cta_ok ? p.tiles_gu + p.tiles_dn : 0;
    const int pair_id = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if ((warp >= 6 && p.pre_normed) || (warp >= 6 && !cta_ok)) {
        // y is already written: nothing for the prologue warps to do
    } else if (warp >= 6 && p.block_rows) {
        // ------------------------------------------------ prologue rows, one per CTA at a time
        prologue_block_rows(p, threadIdx.x - 6 * 32, warp - 6, lane, abort_flag);
    } else if (warp >= 6) {
        // ------------------------------------------------ prologue rows, one per warp
        const int W = gridDim.x * PRO_WARPS;
        const int d = p.d;
        for (long long row = static_cast<long long>(blockIdx.x) * PRO_WARPS + (warp - 6); row < p.M; row += W) {
            if (*wc.abort_flag) break;
            const long long base = row * d;
            if (!checked_range(base, d, static_cast<long long>(p.M) * d, p.status, abort_flag, kWhereBoundsLoad))
                break;
            constexpr int NV = 4;
            float ss = 0.f;
            for (int col0 = lane * 8; col0 < d; col0 += 256 * NV) {
                float h[NV][8];
                row_h<NV>(p, base, col0, h);
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    if (col0 + 256 * v < d)
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss = fmaf(h[v][e], h[v][e], ss);
            }
            ss = warp_sum(ss);
            const float inv = rsqrtf(ss / static_cast<float>(d) + p.eps);
            for (int col0 = lane * 8; col0 < d; col0 += 256 * NV) {
                float h[NV][8];
                row_h<NV>(p, base, col0, h);  // same inputs and order: the same h
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const int col = col0 + 256 * v;
                    if (col < d) {
                        float gm[8];
                        load8(static_cast<const __nv_bfloat16*>(p.gamma) + col, gm);
                        if (p.h_out != nullptr)
                            __stcs(reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.h_out) + base + col),
                                   pack8(h[v]));
#pragma unroll
                        for (int e = 0; e < 8; ++e) gm[e] = (h[v][e] * gm[e]) * inv;
                        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.y) + base + col) = pack8(gm);
                    }
                }
            }
            // make the row's y visible to the TMA loads of other CTAs
            fence_proxy_async_global();
            __syncwarp();
            if (lane == 0 && checked_index(row / p.chunk_rows, p.chunks, p.status, abort_flag, kWhereBoundsCounter))
                red_release_add(&p.chunk_ready[row / p.chunk_rows], 1);
        }
    } else if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        const uint32_t full0 = mapa_shared(smem_u32(&bars->full[0]), 0);
        int stage = 0;
        uint32_t phase = 0;
        int armed_parity[STAGES];
        for (int s = 0; s < STAGES; ++s) armed_parity[s] = -1;
        bool ok = true;
        for (int t = pair_id; ok && t < total; t += npairs) {
            const Tile tl = decode(p, t);
            if (!tile_ok(p, tl, abort_flag)) break;
            // dependency of this tile's A operand
            if (!tl.down) {
                if (!p.pre_normed) {
                    // every chunk the tile's rows overlap; a row counts once
                    // per publishing warp
                    const int need = p.chunk_rows * (p.block_rows ? PRO_WARPS : 1);
                    const int c1 = (min(p.M, (tl.m + 1) * PBM) - 1) / p.chunk_rows;
                    for (int c = tl.m * PBM / p.chunk_rows; ok && c <= c1; ++c)
                        ok = checked_index(c, p.chunks, p.status, abort_flag, kWhereBoundsCounter) &&
                             flag_wait_geq(&p.chunk_ready[c], need, wc, kWhereFusedRows, t);
                }
            } else {
                ok = checked_index(tl.g * p.mt + tl.m, p.P * p.mt, p.status, abort_flag, kWhereBoundsCounter) &&
                     flag_wait_geq(&p.gu_done[tl.g * p.mt + tl.m], 2 * p.nt_gu, wc, kWhereFusedGateUp, t);
            }
            if (!ok) break;
            fence_proxy_async_global();
            const int nk = tl.down ? p.nk_dn : p.nk_gu;
            const CUtensorMap* mA = tl.down ? &p.mapS[tl.g] : &p.mapY;
            // B: a gate/up tile's halves are gate and up rows; a down or QKV
            // tile's are rows n*256 + rank*128 of one matrix
            const bool split_b = tl.down || p.qkv;
            const CUtensorMap* mB =
                tl.down ? &p.mapW2[tl.g] : (p.qkv || rank == 0 ? &p.mapW1g[tl.g] : &p.mapW1u[tl.g]);
            const int brow = split_b ? tl.n * PBN + static_cast<int>(rank) * 128 : tl.n * 128;
            const int arow = tl.m * PBM + static_cast<int>(rank) * 128;
            // a checked build: the box origins of every k-block (A: y [M][d]
            // or s [M][f]; B: W1g/W1u/Wqkv rows [f][d] or W2 columns [d][f])
            const int ka = tl.down ? p.f : p.d;
            const int b_rows = tl.down ? p.nt_dn * PBN : (p.qkv ? p.nt_gu * PBN : p.nt_gu * 128);
            for (int kb = 0; kb < nk; ++kb) {
                if (!checked_tma(kb * BK, BK, ka, arow, static_cast<long long>(p.mt) * PBM, p.status, abort_flag) ||
                    !checked_tma(kb * BK, BK, ka, brow, b_rows, p.status, abort_flag)) {
                    ok = false;
                    break;
                }
                if (!mbar_wait(&bars->empty[stage], phase ^ 1u, wc, kWhereProducerEmpty, t)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    mbar_arrive_expect_tx(&bars->full[stage], 2 * STAGE_BYTES);
                    armed_parity[stage] = static_cast<int>(phase);
                }
                const uint32_t fb = full0 + static_cast<uint32_t>(stage * sizeof(uint64_t));
                tma_load_2d_pair(a_tiles + stage * A_BYTES, mA, fb, kb * BK, arow);
                tma_load_2d_pair(b_tiles + stage * B_BYTES, mB, fb, kb * BK, brow);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        WaitCtx drain{p.status, &bars->abort_flag, p.wait_limit_ns};
        int dummy_abort = 0;
        drain.abort_flag = &dummy_abort;
        if (leader) {
            for (int s = 0; s < STAGES; ++s)
                if (armed_parity[s] >= 0)
                    mbar_wait(&bars->full[s], static_cast<uint32_t>(armed_parity[s]), drain, kWhereDrain, s);
        } else if (!ok) {
            const unsigned long long t0 = global_timer_ns();
            while (global_timer_ns() - t0 < 200000ull) __nanosleep(1000);
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------------------------ MMA issuer (even CTA)
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        int local = 0;
        for (int t = pair_id; ok && t < total; t += npairs, ++local) {
            const Tile tl = decode(p, t);
            if (!tile_ok(p, tl, abort_flag)) break;
            const int nk = tl.down ? p.nk_dn : p.nk_gu;
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            if (!mbar_wait(&bars->acc_empty[acc], acc_phase ^ 1u, wc, kWhereMmaAccEmpty, t)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * PBN);
            for (int kb = 0; kb < nk; ++kb) {
                if (!mbar_wait(&bars->full[stage], phase, wc, kWhereMmaFull, t)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t adesc = smem_desc_kmajor_sw128(smem_u32(a_tiles + stage * A_BYTES));
                const uint64_t bdesc = smem_desc_kmajor_sw128(smem_u32(b_tiles + stage * B_BYTES));
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_bf16_pair(d_tmem, adesc + 2ull * k, bdesc + 2ull * k, IDESC, (kb | k) != 0 ? 1u : 0u);
                umma_commit_pair_multicast(&bars->empty[stage], 0x3);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit_pair_multicast(&bars->acc_full[acc], 0x3);
        }
        umma_commit_pair_multicast(&bars->drain, 0x1);
        WaitCtx drain{p.status, &bars->abort_flag, p.wait_limit_ns};
        int dummy_abort = 0;
        drain.abort_flag = &dummy_abort;
        mbar_wait(&bars->drain, 0, drain, kWhereDrain, -1);
    } else if (warp >= 2 && warp < 6) {
        // ------------------------------------------------ epilogue (both CTAs)
        const uint32_t acc_empty0 = mapa_shared(smem_u32(&bars->acc_empty[0]), 0);
        const int quarter = warp & 3;
        const int row_in_tile = static_cast<int>(rank) * 128 + quarter * 32 + lane;
        int local = 0;
        for (int t = pair_id; t < total; t += npairs, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            const bool ok = mbar_wait(&bars->acc_full[acc], acc_phase, wc, kWhereEpilogueAccFull, t);
            // the four epilogue warps leave together (they share barrier 1)
            if (epilogue_any(!ok)) break;
            tc_fence_after();
            const Tile tl = decode(p, t);
            // a checked build: a bad tile leaves it unstored (its readers
            // then give up through their bounded waits)
            const bool tile_good = tile_ok(p, tl, abort_flag);
            const int row = tl.m * PBM + row_in_tile;
            const bool row_ok = row < p.M && tile_good;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * PBN);
            if (!tl.down && !p.qkv) {
                __nv_bfloat16* out =
                    reinterpret_cast<__nv_bfloat16*>(p.s_out[tl.g]) + static_cast<long long>(row) * p.f;
#pragma unroll 1
                for (int c = 0; c < PBN / 2; c += 16) {
                    uint32_t gv[16], uv[16];
                    tmem_ld_16cols(taddr + c, gv);
                    tmem_ld_16cols(taddr + PBN / 2 + c, uv);
                    tmem_ld_wait();
                    uint32_t packed[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float a0 = __uint_as_float(gv[2 * j]), a1 = __uint_as_float(gv[2 * j + 1]);
                        const float b0 = __uint_as_float(uv[2 * j]), b1 = __uint_as_float(uv[2 * j + 1]);
                        packed[j] = pack_bf16x2(silu_f(a0) * b0, silu_f(a1) * b1);
                    }
                    const int col = tl.n * (PBN / 2) + c;
                    if (row_ok) {
#pragma unroll
                        for (int v = 0; v < 2; ++v)
                            if (col + 8 * v < p.f &&
                                checked_range(static_cast<long long>(row) * p.f + col + 8 * v, 8,
                                              static_cast<long long>(p.M) * p.f, p.status, abort_flag,
                                              kWhereBoundsStore))
                                *reinterpret_cast<uint4*>(out + col + 8 * v) =
                                    make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
                    }
                }
            } else {
                // down partials [M][d], or the shard's q, k, v columns [M][f]
                const int ncols = tl.down ? p.d : p.f;
                __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(tl.down ? p.out[tl.g] : p.s_out[tl.g]) +
                                     static_cast<long long>(row) * ncols;
#pragma unroll 1
                for (int c = 0; c < PBN; c += 16) {
                    uint32_t v16[16];
                    tmem_ld_16cols(taddr + c, v16);
                    tmem_ld_wait();
                    uint32_t packed[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        packed[j] = pack_bf16x2(__uint_as_float(v16[2 * j]), __uint_as_float(v16[2 * j + 1]));
                    const int col = tl.n * PBN + c;
                    if (row_ok) {
#pragma unroll
                        for (int v = 0; v < 2; ++v)
                            if (col + 8 * v < ncols &&
                                checked_range(static_cast<long long>(row) * ncols + col + 8 * v, 8,
                                              static_cast<long long>(p.M) * ncols, p.status, abort_flag,
                                              kWhereBoundsStore))
                                __stcs(reinterpret_cast<uint4*>(out + col + 8 * v),
                                       make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                                  packed[4 * v + 3]));
                    }
                }
            }
            // reads complete and fenced; outputs are published separately below
            tc_fence_before();
            mbar_arrive_cluster_relaxed(acc_empty0 + static_cast<uint32_t>(acc * sizeof(uint64_t)));
            if (!tl.down && !p.qkv) {
                // this CTA's 128 rows of the s tile are stored: publish them
                // to the down tiles' TMA loads
                fence_proxy_async_global();
                named_barrier_sync<1, 128>();
                if (warp == 2 && lane == 0 && tile_good &&
                    checked_index(tl.g * p.mt + tl.m, p.P * p.mt, p.status, abort_flag, kWhereBoundsCounter))
                    red_release_add(&p.gu_done[tl.g * p.mt + tl.m], 1);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

}  // namespace

// Number of co-resident CTA pairs of the fused kernel (0 if it cannot run).
int fused_max_pairs(int num_sms) {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const int slot = dev & 63;
    if (cached[slot] != 0) return cached[slot] < 0 ? 0 : cached[slot];
    if (cudaFuncSetAttribute(boundary_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
        cudaSuccess) {
        cached[slot] = -1;
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, boundary_fused_kernel, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        cached[slot] = -1;
        return 0;
    }
    cached[slot] = n;
    return n;
}

cudaError_t launch_boundary_fused(const FusedParams& p, int pairs, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(boundary_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // the CTAs wait on one another's work: all of them must be resident
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, boundary_fused_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sptp
