// Persistent tcgen05 GEMM for sm_103a on CTA pairs (cta_group::2), with a
// TMA-fed shared-memory pipeline and TMEM accumulators, used for the
// column-parallel gate/up projection (with a fused SwiGLU epilogue) and the
// row-parallel down projection (with a bf16 partial-store epilogue) of the
// SP-TP FFN boundary ("[Feature] Async Tensor Parallelism for Archon Engine",
// "Potential Solution").
//
// A cluster of two CTAs, one per SM, computes 256 x 256 tiles; each CTA
// stages its own 128 rows of A and of B in six 32 KiB stages:
//   warp 0      TMA producer (both CTAs)
//   warp 1      MMA issuer of the even CTA: 4 x tcgen05.mma (M=256, N=256,
//               K=16) per stage into one of two TMEM accumulators of 256
//               fp32 columns
//   warps 2..5  epilogue (both CTAs): tcgen05.ld of the accumulator, SwiGLU
//               or bf16 convert, global stores; overlaps the next tile's MMAs
// Tiles are walked in raster bands of `band` m-tiles (4096 rows) so that
// concurrently running pairs share A and B tiles in L2.  The kernel runs on
// bf16 operands (kind::f16, 64 elements per 128-byte row) or on E4M3
// operands (kind::f8f6f4, 128 per row) for the fp8 linear layers ("[Feature]
// Async Tensor Parallelism for Archon Engine", "Additional Information"),
// whose epilogue multiplies the fp32 accumulator by the token row's and the
// output column's power-of-two scales.  Its plain (store) epilogue stages each
// warp's 32 x 64 output block in shared memory and writes whole 128-byte row
// segments (store_staged.cuh); the SwiGLU epilogue stores from registers.
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "sptp_ptx.cuh"
#include "store_staged.cuh"

namespace sptp {

namespace {

constexpr int BK = 64;               // K elements per stage (one 128-byte swizzle row of bf16)
constexpr int TMEM_COLS = 512;       // two accumulators of 256 fp32 columns
constexpr int BAR_BYTES = 256;

__device__ __forceinline__ void decode_tile(const TcGemmParams& p, int t, int& g, int& m, int& n) {
    const int per_band = p.band * p.G * p.nt;
    const int b = t / per_band;
    const int r = t - b * per_band;
    const int m0 = b * p.band;
    const int bm = min(p.band, p.mt - m0);
    m = m0 + r % bm;
    const int gn = r / bm;
    g = gn / p.nt;
    n = gn - g * p.nt;
}

// silu(a) = a / (1 + e^-a) with the fast divide (<= 2 ulp in fp32, far below
// the bf16 rounding of the output); for a < -87 the divisor overflows and the
// result is 0, the correctly rounded bf16 value there.
__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------------------
// The CTA-pair kernel (cta_group::2, cluster of 2): the pair computes a
// 256 x 256 tile.  Each CTA stages its own 128 A rows and one half of the B
// tile (SwiGLU: CTA 0 the 128 gate rows, CTA 1 the 128 up rows; plain: the
// two 128-row halves), so a stage is 32 KiB per CTA and 6 stages fit.  The
// even CTA issues the UMMAs (M=256, N=256, K=16); both CTAs' TMA loads
// complete on the even CTA's full barrier; commits are multicast to both
// CTAs' empty / accumulator-full barriers; both CTAs' epilogues release the
// accumulator on the even CTA's accumulator-empty barrier.
namespace pair {

constexpr int PBM = 256;                     // tile rows (128 per CTA)
constexpr int PBN = 256;                     // UMMA N
constexpr int kMaxPStages = 6;
constexpr int A_BYTES = 128 * BK * 2;        // 16 KiB
constexpr int B_BYTES = 128 * BK * 2;        // 16 KiB (half of the B tile)
constexpr int PSTAGE_BYTES = A_BYTES + B_BYTES;
// The plain epilogue stages its output blocks (store_staged.cuh): one
// kOutWarpBytes buffer per epilogue warp after the barrier block.
template <Epi EPI, int ST, int EW>
constexpr int psmem_bytes() {
    return 1024 + ST * PSTAGE_BYTES + BAR_BYTES + (EPI == Epi::kStore ? EW * kOutWarpBytes : 0);
}
static_assert(psmem_bytes<Epi::kStore, kMaxPStages, 4>() <= 227 * 1024, "pipeline does not fit in shared memory");
// A stage holds 128-byte K slices of each operand row: 64 bf16 or 128 E4M3
// elements.  Either way 4 UMMAs of 32 bytes per row consume it.
template <bool E4M3>
__host__ __device__ constexpr int k_elems() { return E4M3 ? 128 : 64; }
template <bool E4M3>
__host__ __device__ constexpr uint32_t pair_idesc() {
    return E4M3 ? idesc_e4m3_f32(PBM, PBN) : idesc_bf16_f32(PBM, PBN);
}
// Epilogue warps EW: 4 (one per TMEM lane quarter) or 8 (two per quarter,
// each taking half of the tile's columns).
template <int EW>
constexpr int pair_threads() { return 32 * (2 + EW); }

// Column scales of 32 consecutive output columns from col; columns past N
// read none (their products are discarded).  Every lane reads the same
// addresses: one broadcast transaction per load.
__device__ __forceinline__ void load_col_scales(const float* sg, const float* su, int col, int N, float* cg,
                                                float* cu) {
    if (col + 32 <= N) {
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(sg + col) + v);
            const float4 b = __ldg(reinterpret_cast<const float4*>(su + col) + v);
            cg[4 * v] = a.x, cg[4 * v + 1] = a.y, cg[4 * v + 2] = a.z, cg[4 * v + 3] = a.w;
            cu[4 * v] = b.x, cu[4 * v + 1] = b.y, cu[4 * v + 2] = b.z, cu[4 * v + 3] = b.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            cg[j] = col + j < N ? __ldg(sg + col + j) : 0.0f;
            cu[j] = col + j < N ? __ldg(su + col + j) : 0.0f;
        }
    }
}

__device__ __forceinline__ void load_col_scales_strided(const float* sc, int stride, int col, int N, float* cs) {
#pragma unroll
    for (int j = 0; j < 32; ++j) cs[j] = col + j < N ? __ldg(sc + static_cast<long long>(col + j) * stride) : 0.0f;
}

// A checked build: the decoded tile lies in the launch's tile grid.
__device__ __forceinline__ bool tile_ok(const TcGemmParams& p, int g, int m, int n, volatile int* abort_flag) {
    if constexpr (kBoundsChecked) {
        const bool ok = g >= 0 && g < p.G && m >= 0 && m < p.mt && n >= 0 && n < p.nt;
        return checked(ok, p.status, abort_flag, kWhereBoundsTile, static_cast<long long>(m) * 65536 + n);
    }
    return true;
}

struct Bars {
    uint64_t full[kMaxPStages];
    uint64_t empty[kMaxPStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Bars) <= BAR_BYTES, "barrier block too large");

template <Epi EPI, int EW, bool E4M3, int PSTAGES>
__global__ void __launch_bounds__(pair_threads<EW>(), 1) tc_gemm_pair_kernel(const __grid_constant__ TcGemmParams p) {
    constexpr int KE = k_elems<E4M3>();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* a_tiles = smem;
    uint8_t* b_tiles = smem + PSTAGES * A_BYTES;
    Bars* bars = reinterpret_cast<Bars*>(smem + PSTAGES * PSTAGE_BYTES);
    uint8_t* out_stage = smem + PSTAGES * PSTAGE_BYTES + BAR_BYTES;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < PSTAGES; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&bars->acc_full[a], 1);
            mbar_init(&bars->acc_empty[a], 2 * EW * 32);
        }
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        // a checked build: the launch is a cluster of two CTAs
        checked(cluster_nctarank() == 2 && rank < 2, p.status, &bars->abort_flag, kWhereBoundsCluster, rank);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int g = 0; g < p.G; ++g) {
            tma_prefetch_map(&p.mapA[g]);
            tma_prefetch_map(&p.mapB0[g]);
            if (EPI == Epi::kSwiGLU) tma_prefetch_map(&p.mapB1[g]);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(&bars->tmem_base, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // peer barriers initialised and peer TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;

    WaitCtx wc{p.status, &bars->abort_flag, p.wait_limit_ns};
    volatile int* abort_flag = &bars->abort_flag;
    // zero only in a checked build whose cluster check failed: no role runs
    const int total = bars->abort_flag == 0 ? p.G * p.mt * p.nt : 0;
    const int pair_id = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        const uint32_t full0 = mapa_shared(smem_u32(&bars->full[0]), 0);
        int stage = 0;
        uint32_t phase = 0;
        int armed_parity[PSTAGES];
        for (int s = 0; s < PSTAGES; ++s) armed_parity[s] = -1;
        bool ok = true;
        for (int t = pair_id; ok && t < total; t += npairs) {
            int g, m, n;
            decode_tile(p, t, g, m, n);
            if (!tile_ok(p, g, m, n, abort_flag)) break;
            const int arow = m * PBM + static_cast<int>(rank) * 128;
            const int brow = EPI == Epi::kSwiGLU ? n * 128 : n * PBN + static_cast<int>(rank) * 128;
            const int b_rows = EPI == Epi::kSwiGLU ? p.nt * 128 : p.nt * PBN;
            for (int kb = 0; kb < p.nk; ++kb) {
                // a checked build: the box origins of both operands
                if (!checked_tma(kb * KE, KE, p.K, arow, static_cast<long long>(p.mt) * PBM, p.status, abort_flag) ||
                    !checked_tma(kb * KE, KE, p.K, brow, b_rows, p.status, abort_flag)) {
                    ok = false;
                    break;
                }
                if (!mbar_wait(&bars->empty[stage], phase ^ 1u, wc, kWhereProducerEmpty, t)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    mbar_arrive_expect_tx(&bars->full[stage], 2 * PSTAGE_BYTES);
                    armed_parity[stage] = static_cast<int>(phase);
                }
                const uint32_t fb = full0 + static_cast<uint32_t>(stage * sizeof(uint64_t));
                tma_load_2d_pair(a_tiles + stage * A_BYTES, &p.mapA[g], fb, kb * KE, arow);
                uint8_t* bt = b_tiles + stage * B_BYTES;
                if (EPI == Epi::kSwiGLU) {
                    tma_load_2d_pair(bt, rank == 0 ? &p.mapB0[g] : &p.mapB1[g], fb, kb * KE, brow);
                } else {
                    tma_load_2d_pair(bt, &p.mapB0[g], fb, kb * KE, brow);
                }
                if (++stage == PSTAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        WaitCtx drain{p.status, &bars->abort_flag, p.wait_limit_ns};
        int dummy_abort = 0;
        drain.abort_flag = &dummy_abort;
        if (leader) {
            // both CTAs' copies complete on the leader's full barriers
            for (int s = 0; s < PSTAGES; ++s)
                if (armed_parity[s] >= 0)
                    mbar_wait(&bars->full[s], static_cast<uint32_t>(armed_parity[s]), drain, kWhereDrain, s);
        } else if (!ok) {
            // give copies this CTA may still have in flight time to land
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
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            if (!mbar_wait(&bars->acc_empty[acc], acc_phase ^ 1u, wc, kWhereMmaAccEmpty, t)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * PBN);
            for (int kb = 0; kb < p.nk; ++kb) {
                if (!mbar_wait(&bars->full[stage], phase, wc, kWhereMmaFull, t)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t adesc = smem_desc_kmajor_sw128(smem_u32(a_tiles + stage * A_BYTES));
                const uint64_t bdesc = smem_desc_kmajor_sw128(smem_u32(b_tiles + stage * B_BYTES));
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if constexpr (E4M3)
                        umma_e4m3_pair(d_tmem, adesc + 2ull * k, bdesc + 2ull * k, pair_idesc<E4M3>(),
                                       (kb | k) != 0 ? 1u : 0u);
                    else
                        umma_bf16_pair(d_tmem, adesc + 2ull * k, bdesc + 2ull * k, pair_idesc<E4M3>(),
                                       (kb | k) != 0 ? 1u : 0u);
                }
                umma_commit_pair_multicast(&bars->empty[stage], 0x3);
                if (++stage == PSTAGES) {
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
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue (both CTAs)
        // warp w reads TMEM lanes [32*(w%4), +32); with 8 epilogue warps,
        // warps 2..5 take the first half of the tile's columns, 6..9 the second
        constexpr int kSplits = EW / 4;
        const uint32_t acc_empty0 = mapa_shared(smem_u32(&bars->acc_empty[0]), 0);
        const int quarter = warp & 3;
        const int half = (warp - 2) / 4;
        int local = 0;
        for (int t = pair_id; t < total; t += npairs, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            const bool ok = mbar_wait(&bars->acc_full[acc], acc_phase, wc, kWhereEpilogueAccFull, t);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            int g, m, n;
            decode_tile(p, t, g, m, n);
            // a checked build: a bad tile is not stored
            const bool tile_good = tile_ok(p, g, m, n, abort_flag);
            if (!tile_good) g = 0;
            const int row0 = tile_good ? m * PBM + static_cast<int>(rank) * 128 + quarter * 32 : p.M;
            const int row = row0 + lane;
            const bool row_ok = row < p.M;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * PBN);
            __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out[g]);
            // E4M3: the token row's scale (power of two; rows past M read none)
            float rs = 1.0f;
            if constexpr (E4M3) rs = row_ok ? __ldg(p.row_scale[g] + row) : 0.0f;
            if (EPI == Epi::kSwiGLU) {
                // each lane stores its own row: 64 bytes per 32 columns (the
                // stores are half the plain epilogue's per tile, and gate/up
                // K is long, so staging them measured no faster)
                __nv_bfloat16* orow = out + static_cast<long long>(row) * p.ldo;
#pragma unroll 1
                for (int c = half * (PBN / 2 / kSplits); c < (half + 1) * (PBN / 2 / kSplits); c += 32) {
                    uint32_t gv[32], uv[32];
                    tmem_ld_32cols(taddr + c, gv);
                    tmem_ld_32cols(taddr + PBN / 2 + c, uv);
                    const int col = n * (PBN / 2) + c;
                    float cg[32], cu[32];
                    if constexpr (E4M3) load_col_scales(p.col_scale0[g], p.col_scale1[g], col, p.N, cg, cu);
                    tmem_ld_wait();
                    uint32_t packed[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        float a0 = __uint_as_float(gv[2 * j]), a1 = __uint_as_float(gv[2 * j + 1]);
                        float b0 = __uint_as_float(uv[2 * j]), b1 = __uint_as_float(uv[2 * j + 1]);
                        if constexpr (E4M3) {
                            a0 = a0 * rs * cg[2 * j];
                            a1 = a1 * rs * cg[2 * j + 1];
                            b0 = b0 * rs * cu[2 * j];
                            b1 = b1 * rs * cu[2 * j + 1];
                        }
                        packed[j] = pack_bf16x2(silu_f(a0) * b0, silu_f(a1) * b1);
                    }
                    if (row_ok) {
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            if (col + 8 * v < p.N &&
                                checked_range(static_cast<long long>(row) * p.ldo + col + 8 * v, 8,
                                              static_cast<long long>(p.M) * p.ldo, p.status, abort_flag,
                                              kWhereBoundsStore))
                                *reinterpret_cast<uint4*>(orow + col + 8 * v) =
                                    make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
                    }
                }
            } else {
                __nv_bfloat16* split_out = reinterpret_cast<__nv_bfloat16*>(p.out[0]);
                uint8_t* wbuf = out_stage + (warp - 2) * kOutWarpBytes;
#pragma unroll 1
                for (int c0 = half * (PBN / kSplits); c0 < (half + 1) * (PBN / kSplits); c0 += 64) {
                    uint32_t packed[32];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int c = c0 + 32 * hh;
                        uint32_t v32[32];
                        tmem_ld_32cols(taddr + c, v32);
                        const int col = n * PBN + c;
                        float cs[32];
                        if constexpr (E4M3) load_col_scales_strided(p.col_scale0[g], p.col_scale_stride, col, p.N, cs);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            float v0 = __uint_as_float(v32[2 * j]), v1 = __uint_as_float(v32[2 * j + 1]);
                            if constexpr (E4M3) {
                                v0 = v0 * rs * cs[2 * j];
                                v1 = v1 * rs * cs[2 * j + 1];
                            }
                            packed[16 * hh + j] = pack_bf16x2(v0, v1);
                        }
                    }
                    // the outputs are final: evict-first stores
                    const long long limit = p.split_w > 0 ? static_cast<long long>(p.N / p.split_w) * p.split_stride
                                                          : static_cast<long long>(p.M) * p.ldo;
                    store_block_staged<true>(wbuf, packed, lane, out, p.ldo, split_out, p.split_w, p.split_stride,
                                             row0, p.M, n * PBN + c0, p.N, limit, p.status, abort_flag);
                }
            }
            // The accumulator's reads are complete (tcgen05.wait::ld) and
            // ordered before this signal by the fence; nothing else hangs on
            // it, so it need not wait for this thread's output stores to
            // drain, as a release arrive would (with 14-k-block tiles that
            // drain cost 9 % of the attention out-projection: 333 vs 305 us).
            tc_fence_before();
            mbar_arrive_cluster_relaxed(acc_empty0 + static_cast<uint32_t>(acc * sizeof(uint64_t)));
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still touch its memory
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

}  // namespace pair

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

}  // namespace

bool encode_map_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = get_encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_map_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                   uint32_t box_inner, uint32_t box_outer) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = get_encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_map_bf16_nd(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                        const uint64_t* strides_bytes, const uint32_t* box) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = get_encode_fn();
    if (fn == nullptr || rank < 2 || rank > 5) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) gs[i] = strides_bytes[i];
    }
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gd,
                    gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

template <Epi EPI, int EW, bool E4M3 = false, int ST = 6>
cudaError_t launch_pair_typed(const TcGemmParams& p, int num_sms, cudaStream_t s) {
    auto* kfn = pair::tc_gemm_pair_kernel<EPI, EW, E4M3, ST>;
    constexpr int PSMEM_BYTES = pair::psmem_bytes<EPI, ST, EW>();
    static_assert(PSMEM_BYTES <= 227 * 1024, "pipeline and output staging do not fit in shared memory");
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, PSMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(pair::pair_threads<EW>(), 1, 1);
    cfg.dynamicSmemBytes = PSMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // as many co-resident pairs as the GPU holds (one CTA per SM)
    static int max_clusters[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const int slot = (dev & 63);
    if (max_clusters[slot] == 0) {
        cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, kfn, &cfg);
        if (e != cudaSuccess || n <= 0) return e != cudaSuccess ? e : cudaErrorInvalidConfiguration;
        max_clusters[slot] = n;
    }
    const int total = p.G * p.mt * p.nt;
    const int pairs = total < max_clusters[slot] ? total : max_clusters[slot];
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    e = cudaLaunchKernelEx(&cfg, kfn, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_gemm_pair(const TcGemmParams& p, Epi epi, int num_sms, cudaStream_t s) {
    if (p.G * p.mt * p.nt == 0) return cudaSuccess;
    // Four epilogue warps: measured faster than eight on every workload here
    // (8192x4096x14336 boundary 1681 vs 1669 TFLOP/s, attention boundary 1250
    // vs 1209, per-module Delayed-TP stack 856 vs 825).
    return epi == Epi::kSwiGLU ? launch_pair_typed<Epi::kSwiGLU, 4>(p, num_sms, s)
                               : launch_pair_typed<Epi::kStore, 4>(p, num_sms, s);
}

cudaError_t launch_tc_gemm_pair_e4m3(const TcGemmParams& p, Epi epi, int num_sms, cudaStream_t s) {
    if (p.G * p.mt * p.nt == 0) return cudaSuccess;
    // six stages and four epilogue warps, as for bf16: a seventh stage
    // measured no faster (8192 x 4096 x 14336: E4M3 step 2824 vs 2824
    // TFLOP/s), eight epilogue warps slower (E4M3 gate/up 604-608 vs 590 us)
    return epi == Epi::kSwiGLU ? launch_pair_typed<Epi::kSwiGLU, 4, true>(p, num_sms, s)
                               : launch_pair_typed<Epi::kStore, 4, true>(p, num_sms, s);
}

}  // namespace sptp
