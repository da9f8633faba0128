// Fused persistent Delayed-TP stack ("Affinity-Aware Sharding for Delayed
// Tensor Parallelism", Abstract: every device adds its own partial at once and
// the other devices' partials delta modules later).
//
// One cooperative launch of CTA pairs runs all L modules of the stack:
//   warps 6..11   prologue: rows in the order (module step l = 0..L, 256-row
//                 block m, shard p, row); row r of shard p at step l waits
//                 (bounded) until step l-1's down tiles of block m are stored,
//                 then x_p[r] += own partial of module l-1 + the other shards'
//                 partials of module l-1-delta (+ every pending partial at the
//                 final step when flushing), and y_p[r] = RMSNorm_l(x_p[r]);
//                 each row is published on its block's readiness counter
//   warp 0        TMA producer: a gate/up tile (l, m, p, n) waits until every
//                 shard's rows of block m are normed for module l; a down tile
//                 (l, m, p, n) until all gate/up tiles of (l, p, m) are stored
//   warp 1        MMA issuer of the even CTA (M=256, N=256, K=16 UMMAs)
//   warps 2..5    epilogue: SwiGLU into s_p or the partial o_p^(l) into the
//                 pending ring (row segments staged through shared memory,
//                 store_staged.cuh), then a release increment of the tile's
//                 counter
// GEMM tiles run block by block over (module, 256-row block), each block's
// down tiles `lag` blocks after its gate/up tiles, so module l+1's first
// blocks start while module l's last ones finish.  Every dependency points to
// earlier work in that order or to prologue rows of the same or an earlier
// step, so with all CTAs resident every wait ends.  A pending-ring slot is
// rewritten by down(l, p, m) only after gate/up(l, *, m) saw every shard's
// step-l rows of block m normed, i.e. after every reader of the slot's old
// contents has read them.
//
// Weights, y, s and the ring are addressed through 3-D / 4-D tensor maps:
//   y    [P][M][d]      -> {d, M, P}
//   W1g  [L][P][f][d]   -> {d, f, L*P}   (W1u alike)
//   s    [P][M][f]      -> {f, M, P}
//   W2   [L][d][P][f]   -> {f, P, d, L}
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "sptp_ptx.cuh"
#include "store_staged.cuh"

namespace sptp {

namespace {

constexpr int BK = 64;
constexpr int PBM = 256, PBN = 256;
constexpr int STAGES = 6;
constexpr int A_BYTES = 128 * BK * 2;
constexpr int B_BYTES = 128 * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int BAR_BYTES = 256;
constexpr int TMEM_COLS = 512;
constexpr int EPI_WARPS = 4;
// pipeline stages, barriers, then one output staging buffer per epilogue warp
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES + EPI_WARPS * kOutWarpBytes;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
constexpr int PRO_WARPS = 6;
constexpr int PRO_WARP0 = 2 + EPI_WARPS;
constexpr int THREADS = 32 * (2 + EPI_WARPS + PRO_WARPS);
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
    int l, m, p, n;
};

// Tile t of the software-pipelined sequence over global blocks b = l*mt + m
// (module l, 256-row block m): slot s emits the gate/up tiles of block s (all
// shards), then the down tiles of block s - lag, so a down tile is picked up
// about `lag` blocks after the gate/up tiles it reads; every dependency stays
// earlier in the sequence (lag < mt).
__device__ __forceinline__ Tile decode(const DtpFusedParams& p, int t) {
    const int G = p.P * p.nt_gu, D = p.P * p.nt_dn;
    const int nb = p.L * p.mt;
    int b, q;
    bool down;
    if (t < p.lag * G) {
        b = t / G;
        q = t - b * G;
        down = false;
    } else {
        t -= p.lag * G;
        const int mid = (nb - p.lag) * (G + D);
        if (t < mid) {
            const int s = p.lag + t / (G + D);
            q = t % (G + D);
            down = q >= G;
            if (down) q -= G;
            b = down ? s - p.lag : s;
        } else {
            t -= mid;
            b = nb - p.lag + t / D;
            q = t % D;
            down = true;
        }
    }
    Tile r;
    r.down = down;
    r.l = b / p.mt;
    r.m = b - r.l * p.mt;
    const int nt = down ? p.nt_dn : p.nt_gu;
    r.p = q / nt;
    r.n = q - r.p * nt;
    return r;
}

// A checked build: the decoded tile lies in the launch's tile grid.
__device__ __forceinline__ bool tile_ok(const DtpFusedParams& p, const Tile& tl, volatile int* abort_flag) {
    if constexpr (kBoundsChecked) {
        const int nt = tl.down ? p.nt_dn : p.nt_gu;
        const bool ok = tl.l >= 0 && tl.l < p.L && tl.m >= 0 && tl.m < p.mt && tl.p >= 0 && tl.p < p.P && tl.n >= 0 &&
                        tl.n < nt;
        return checked(ok, p.status, abort_flag, kWhereBoundsTile, static_cast<long long>(tl.m) * 65536 + tl.n);
    }
    return true;
}

__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void add8(const __nv_bfloat16* ptr, float (&r)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(ptr);
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 v = __bfloat1622float2(h2[i]);
        r[2 * i] += v.x;
        r[2 * i + 1] += v.y;
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

// Columns of one row handled per batch: lane l owns the 16-byte vectors at
// columns base + 8*l + 256*v, v < kRowVec, i.e. 1024 columns per batch.
constexpr int kRowVec = 4;

// Number of partial sources added into shard sh's stream at step l, and
// the j-th of them, in the canonical order: own partial of module l-1; the
// other shards' partials of module l-1-delta (ascending shard); at the final
// flushing step the still-pending ones (module-major, ascending shard).
__device__ __forceinline__ int n_sources(const DtpFusedParams& p, int l) {
    int n = l >= 1 ? 1 : 0;
    if (l - 1 - p.delta >= 0) n += p.P - 1;
    if (l == p.L && p.flush) n += (p.P - 1) * (p.L - (p.L - p.delta > 0 ? p.L - p.delta : 0));
    return n;
}

__device__ __forceinline__ const __nv_bfloat16* source_j(const DtpFusedParams& p, int l, int sh, int j,
                                                         volatile int* abort_flag) {
    const long long act = static_cast<long long>(p.M) * p.d;
    const __nv_bfloat16* ring = static_cast<const __nv_bfloat16*>(p.ring);
    int module, q;
    if (l >= 1 && j == 0) {
        module = l - 1;
        q = sh;
    } else {
        if (l >= 1) --j;
        const int n_oth = (l - 1 - p.delta >= 0) ? p.P - 1 : 0;
        int idx;
        if (j < n_oth) {
            module = l - 1 - p.delta;
            idx = j;
        } else {
            j -= n_oth;
            module = (p.L - p.delta > 0 ? p.L - p.delta : 0) + j / (p.P - 1);
            idx = j % (p.P - 1);
        }
        q = idx < sh ? idx : idx + 1;
    }
    // a checked build: a module that has run, one of the P shards, and the
    // ring slot it lives in
    if (!checked_index(module, p.L, p.status, abort_flag, kWhereBoundsRing) ||
        !checked_index(q, p.P, p.status, abort_flag, kWhereBoundsRing) ||
        !checked_index(module % p.S, p.S, p.status, abort_flag, kWhereBoundsRing))
        return nullptr;
    return ring + (static_cast<long long>(module % p.S) * p.P + q) * act;
}

// h for one batch of a row of shard `sh` at step l: x + (0 + s_0 + s_1 +
// ...), the sources in the order above -- the three-launch path's order.
// Loads are issued three sources (x counting as the last one) at a time, so a
// row with up to two partial sources costs one round of loads.
constexpr int kSrcBatch = 3;

__device__ __forceinline__ void step_h(const DtpFusedParams& p, int l, int sh, long long row, int base, int lane,
                                       float (&h)[kRowVec][8], volatile int* abort_flag) {
    const long long act = static_cast<long long>(p.M) * p.d;
    const long long off = row * p.d + base + lane * 8;
    const int col0 = base + lane * 8;
    const int ns = n_sources(p, l);
#pragma unroll
    for (int v = 0; v < kRowVec; ++v)
#pragma unroll
        for (int e = 0; e < 8; ++e) h[v][e] = 0.f;
    for (int j0 = 0; j0 <= ns; j0 += kSrcBatch) {
        uint4 u[kSrcBatch][kRowVec];
#pragma unroll
        for (int jj = 0; jj < kSrcBatch; ++jj) {
            const int j = j0 + jj;
            if (j <= ns) {
                const __nv_bfloat16* s0 =
                    j == ns ? static_cast<const __nv_bfloat16*>(p.x) + sh * act : source_j(p, l, sh, j, abort_flag);
#pragma unroll
                for (int v = 0; v < kRowVec; ++v) {
                    u[jj][v] = make_uint4(0u, 0u, 0u, 0u);
                    if (col0 + 256 * v < p.d && s0 != nullptr &&
                        checked_range(off + 256 * v, 8, act, p.status, abort_flag, kWhereBoundsLoad))
                        u[jj][v] = *reinterpret_cast<const uint4*>(s0 + off + 256 * v);
                }
            }
        }
        // in order: the sources, then x (one IEEE addition each, so h + x ==
        // x + h bit for bit)
#pragma unroll
        for (int jj = 0; jj < kSrcBatch; ++jj) {
            if (j0 + jj <= ns) {
#pragma unroll
                for (int v = 0; v < kRowVec; ++v) {
                    if (col0 + 256 * v < p.d) {
                        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u[jj][v]);
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
}

// Writes one batch of the row: x_p <- h, and y_p <- h * inv * gamma_l (l < L).
__device__ __forceinline__ void step_store(const DtpFusedParams& p, int l, int sh, long long row, int base, int lane,
                                           const float (&h)[kRowVec][8], float inv, volatile int* abort_flag) {
    const long long act = static_cast<long long>(p.M) * p.d;
    __nv_bfloat16* xr = static_cast<__nv_bfloat16*>(p.x) + sh * act + row * p.d;
    __nv_bfloat16* yr = static_cast<__nv_bfloat16*>(p.y) + sh * act + row * p.d;
    const __nv_bfloat16* gl = static_cast<const __nv_bfloat16*>(p.gamma) + static_cast<long long>(l) * p.d;
#pragma unroll
    for (int v = 0; v < kRowVec; ++v) {
        const int col = base + lane * 8 + 256 * v;
        // a checked build: x_p and y_p are [P][M][d]
        if (col < p.d && checked_range(sh * act + row * p.d + col, 8, p.P * act, p.status, abort_flag,
                                       kWhereBoundsStore)) {
            if (l < p.L) {
                float gm[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) gm[e] = 0.f;
                add8(gl + col, gm);
#pragma unroll
                for (int e = 0; e < 8; ++e) gm[e] = h[v][e] * inv * gm[e];
                *reinterpret_cast<uint4*>(yr + col) = pack8(gm);
            }
            *reinterpret_cast<uint4*>(xr + col) = pack8(h[v]);
        }
    }
}

__global__ void __launch_bounds__(THREADS, 1) dtp_fused_kernel(const __grid_constant__ DtpFusedParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* a_tiles = smem;
    uint8_t* b_tiles = smem + STAGES * A_BYTES;
    Bars* bars = reinterpret_cast<Bars*>(smem + STAGES * STAGE_BYTES);
    uint8_t* out_stage = smem + STAGES * STAGE_BYTES + BAR_BYTES;

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
            mbar_init(&bars->acc_empty[a], 2 * EPI_WARPS * 32);
        }
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        // a checked build: the launch is a cluster of two CTAs
        checked(cluster_nctarank() == 2 && rank < 2, p.status, &bars->abort_flag, kWhereBoundsCluster, rank);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&p.mapY);
        tma_prefetch_map(&p.mapW1g);
        tma_prefetch_map(&p.mapW1u);
        tma_prefetch_map(&p.mapS);
        tma_prefetch_map(&p.mapW2);
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
    const int total = cta_ok ? p.total_tiles : 0;
    const int pair_id = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (warp >= PRO_WARP0 && cta_ok) {
        // ------------------------------------------------ prologue rows, all steps
        // 32-bit row numbering (P * M * (L + 1) < 2^31, checked at launch):
        // 64-bit divisions per row would cost the warps more than the row
        const uint32_t W = gridDim.x * PRO_WARPS;
        const uint32_t per_step = static_cast<uint32_t>(p.P) * static_cast<uint32_t>(p.M);
        const uint32_t all = per_step * static_cast<uint32_t>(p.L + 1);
        const uint32_t per_block = static_cast<uint32_t>(p.P) * PBM;
        const int d = p.d;
        for (uint32_t i = blockIdx.x * PRO_WARPS + (warp - PRO_WARP0); i < all; i += W) {
            if (*wc.abort_flag) break;
            const int l = static_cast<int>(i / per_step);
            const uint32_t rem = i - static_cast<uint32_t>(l) * per_step;
            // order inside a step: block m, then shard, then the block's rows
            const int m = static_cast<int>(rem / per_block);
            const int rows_m = min(PBM, p.M - m * PBM);
            const uint32_t idx = rem - static_cast<uint32_t>(m) * per_block;
            const int sh = static_cast<int>(rows_m == PBM ? idx / PBM : idx / static_cast<uint32_t>(rows_m));
            const long long row = static_cast<long long>(m) * PBM + (idx - static_cast<uint32_t>(sh) * rows_m);
            // a checked build: the row's (step, block, shard, row) and its counters
            if (!checked(l <= p.L && m < p.mt && sh < p.P && row < p.M, p.status, abort_flag, kWhereBoundsTile, i) ||
                !checked_index(l * p.mt + m, (p.L + 1) * p.mt, p.status, abort_flag, kWhereBoundsCounter))
                break;
            if (l >= 1 &&
                !warp_flag_wait_geq(&p.dn_done[(l - 1) * p.mt + m], 2 * p.P * p.nt_dn, wc, kWhereFusedRows,
                                    static_cast<int>(i)))
                break;
            float ss = 0.f;
            float h[kRowVec][8];
            for (int base = 0; base < d; base += 256 * kRowVec) {
                step_h(p, l, sh, row, base, lane, h, abort_flag);
#pragma unroll
                for (int v = 0; v < kRowVec; ++v)
                    if (base + lane * 8 + 256 * v < d)
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss = fmaf(h[v][e], h[v][e], ss);
            }
            ss = warp_sum(ss);
            const float inv = rsqrtf(ss / static_cast<float>(d) + p.eps);
            __syncwarp();  // every lane has read x_p[row] before it is rewritten
            if (d <= 256 * kRowVec) {
                step_store(p, l, sh, row, 0, lane, h, inv, abort_flag);  // one batch: h is still in registers
            } else {
                for (int base = 0; base < d; base += 256 * kRowVec) {
                    step_h(p, l, sh, row, base, lane, h, abort_flag);  // same inputs and order: the same h
                    step_store(p, l, sh, row, base, lane, h, inv, abort_flag);
                }
            }
            if (l < p.L) {
                // publish the row's y to the gate/up tiles' TMA loads
                fence_proxy_async_global();
                __syncwarp();
                if (lane == 0) red_release_add(&p.rb_ready[l * p.mt + m], 1);
            }
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
            if (!tl.down) {
                const int need = p.P * min(PBM, p.M - tl.m * PBM);
                ok = checked_index(tl.l * p.mt + tl.m, p.L * p.mt, p.status, abort_flag, kWhereBoundsCounter) &&
                     flag_wait_geq(&p.rb_ready[tl.l * p.mt + tl.m], need, wc, kWhereFusedRows, t);
            } else {
                const int gi = (tl.l * p.P + tl.p) * p.mt + tl.m;
                ok = checked_index(gi, p.L * p.P * p.mt, p.status, abort_flag, kWhereBoundsCounter) &&
                     flag_wait_geq(&p.gu_done[gi], 2 * p.nt_gu, wc, kWhereFusedGateUp, t);
            }
            if (!ok) break;
            fence_proxy_async_global();
            const int nk = tl.down ? p.nk_dn : p.nk_gu;
            const int arow = tl.m * PBM + static_cast<int>(rank) * 128;
            // B rows: gate/up tiles n * 128 of [f] rows; down tiles n * 256 +
            // rank * 128 of [d] rows
            const int brow = tl.down ? tl.n * PBN + static_cast<int>(rank) * 128 : tl.n * 128;
            const int b_rows = tl.down ? p.nt_dn * PBN : p.nt_gu * 128;
            const int ka = tl.down ? p.f : p.d;
            for (int kb = 0; kb < nk; ++kb) {
                // a checked build: the box origins (the trailing coordinates,
                // shard and module, are checked with the tile)
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
                uint8_t* at = a_tiles + stage * A_BYTES;
                uint8_t* bt = b_tiles + stage * B_BYTES;
                if (!tl.down) {
                    tma_load_3d_pair(at, &p.mapY, fb, kb * BK, arow, tl.p);
                    tma_load_3d_pair(bt, rank == 0 ? &p.mapW1g : &p.mapW1u, fb, kb * BK, brow, tl.l * p.P + tl.p);
                } else {
                    tma_load_3d_pair(at, &p.mapS, fb, kb * BK, arow, tl.p);
                    tma_load_4d_pair(bt, &p.mapW2, fb, kb * BK, tl.p, brow, tl.l);
                }
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
    } else if (warp >= 2 && warp < 2 + EPI_WARPS) {
        // ------------------------------------------------ epilogue (both CTAs)
        const uint32_t acc_empty0 = mapa_shared(smem_u32(&bars->acc_empty[0]), 0);
        const int quarter = warp & 3;
        // warp w reads TMEM lanes [32*(w%4), +32); with more than four
        // epilogue warps the tile's columns are split between them
        constexpr int kSplits = EPI_WARPS / 4;
        const int split = (warp - 2) / 4;
        const long long act = static_cast<long long>(p.M) * p.d;
        int local = 0;
        for (int t = pair_id; t < total; t += npairs, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            const bool ok = mbar_wait(&bars->acc_full[acc], acc_phase, wc, kWhereEpilogueAccFull, t);
            if (named_barrier_any<1, 32 * EPI_WARPS>(!ok)) break;
            tc_fence_after();
            const Tile tl = decode(p, t);
            // a checked build: a bad tile or ring slot is not stored (its
            // readers then give up through their bounded waits)
            const bool tile_good = tile_ok(p, tl, abort_flag) &&
                                   checked_index(tl.l % p.S, p.S, p.status, abort_flag, kWhereBoundsRing);
            const int row0 = tile_good ? tl.m * PBM + static_cast<int>(rank) * 128 + quarter * 32
                                       : p.M;  // the warp's first row
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * PBN);
            uint8_t* wbuf = out_stage + (warp - 2) * kOutWarpBytes;
            if (!tl.down) {
                // s [M][f] of shard p, in blocks of 64 SwiGLU columns
                __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.s) + static_cast<long long>(tl.p) * p.M * p.f;
#pragma unroll 1
                for (int c0 = split * (PBN / 2 / kSplits); c0 < (split + 1) * (PBN / 2 / kSplits); c0 += 64) {
                    uint32_t packed[32];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t gv[16], uv[16];
                        tmem_ld_16cols(taddr + c0 + 16 * q, gv);
                        tmem_ld_16cols(taddr + PBN / 2 + c0 + 16 * q, uv);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float a0 = __uint_as_float(gv[2 * j]), a1 = __uint_as_float(gv[2 * j + 1]);
                            const float b0 = __uint_as_float(uv[2 * j]), b1 = __uint_as_float(uv[2 * j + 1]);
                            packed[8 * q + j] = pack_bf16x2(silu_f(a0) * b0, silu_f(a1) * b1);
                        }
                    }
                    store_block_staged<false>(wbuf, packed, lane, out, p.f, nullptr, 0, 0, row0, p.M,
                                              tl.n * (PBN / 2) + c0, p.f, static_cast<long long>(p.M) * p.f,
                                              p.status, abort_flag);
                }
            } else {
                // the partial [M][d] in ring slot l mod S, shard p, in blocks of 64 columns
                __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.ring) +
                                     (static_cast<long long>(tl.l % p.S) * p.P + tl.p) * act;
#pragma unroll 1
                for (int c0 = split * (PBN / kSplits); c0 < (split + 1) * (PBN / kSplits); c0 += 64) {
                    uint32_t packed[32];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t v16[16];
                        tmem_ld_16cols(taddr + c0 + 16 * q, v16);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            packed[8 * q + j] =
                                pack_bf16x2(__uint_as_float(v16[2 * j]), __uint_as_float(v16[2 * j + 1]));
                    }
                    store_block_staged<false>(wbuf, packed, lane, out, p.d, nullptr, 0, 0, row0, p.M,
                                              tl.n * PBN + c0, p.d, act, p.status, abort_flag);
                }
            }
            // reads complete and fenced; outputs are published separately below
            tc_fence_before();
            mbar_arrive_cluster_relaxed(acc_empty0 + static_cast<uint32_t>(acc * sizeof(uint64_t)));
            // this CTA's half of the tile is stored: publish it (s to the down
            // tiles' TMA loads, which needs the proxy fence; the partial to the
            // next steps' prologue rows, plain loads: release/acquire suffices)
            if (!tl.down) fence_proxy_async_global();
            named_barrier_sync<1, 32 * EPI_WARPS>();
            if (warp == 2 && lane == 0 && tile_good) {
                if (!tl.down) {
                    const int gi = (tl.l * p.P + tl.p) * p.mt + tl.m;
                    if (checked_index(gi, p.L * p.P * p.mt, p.status, abort_flag, kWhereBoundsCounter))
                        red_release_add(&p.gu_done[gi], 1);
                } else if (checked_index(tl.l * p.mt + tl.m, p.L * p.mt, p.status, abort_flag, kWhereBoundsCounter)) {
                    red_release_add(&p.dn_done[tl.l * p.mt + tl.m], 1);
                }
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

int dtp_fused_max_pairs(int num_sms) {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const int slot = dev & 63;
    if (cached[slot] != 0) return cached[slot] < 0 ? 0 : cached[slot];
    if (cudaFuncSetAttribute(dtp_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
        cudaSuccess) {
        cudaGetLastError();
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
    if (cudaOccupancyMaxActiveClusters(&n, dtp_fused_kernel, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        cached[slot] = -1;
        return 0;
    }
    cached[slot] = n;
    return n;
}

cudaError_t launch_dtp_fused(const DtpFusedParams& p, int pairs, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(dtp_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeCooperative;  // all CTAs resident: they wait on one another
    attr[1].val.cooperative = 1;
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, dtp_fused_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace sptp
