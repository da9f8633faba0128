// Neuron-permutation shard maps for Delayed TP ("Affinity-Aware Sharding for
// Delayed Tensor Parallelism", Abstract: the dense model is permuted before it
// is sharded, and under delayed partials which neurons share a device is a
// modelling decision).  Executing a permuted layout = renumbering each FFN's
// neurons once, then sharding contiguously: new neuron i of module l is old
// neuron perm[l][i]; W1g/W1u rows and W2 columns move together.
//
// HBM-bound gathers, every byte read and written once.  One persistent
// launch does all three matrices through a bulk-copy pipeline (pipe::
// below) when a W1 row of each matrix, and a W2 row, fit a 32 KiB stage;
// otherwise two launches:
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

// ---------------------------------------------------------------------------
// One persistent launch for all three matrices: per CTA a ring of
// shared-memory stages that warp 0 fills with bulk copies, up to NS units
// ahead, while the other warps drain them with 16-byte coalesced stores (two
// CTAs per SM).  The work is cut into units, dealt round-robin to the CTAs:
//   A: RA consecutive output rows i0.. of module l of W1g and W1u: each source
//      row perm[l][i] is bulk-copied into the stage, and the warps store the
//      stage's rows to the (contiguous) output rows;
//   B: RB consecutive rows r0.. of module l of W2, contiguous: one bulk load;
//      the warps gather each row's permuted columns from the stage and store
//      them.
// An index outside [0, F) is reported and its output written as zeros.
namespace pipe {

constexpr int NS = 3;                // stages
constexpr int STAGE = 32 * 1024;     // bytes per stage
constexpr int THREADS = 512;
constexpr int CONSUMERS = THREADS - 32;  // warps 1..: stores
constexpr int MAX_RA = 16;           // W1 rows per unit (warp 0 lanes index them)
constexpr int CTAS_PER_SM = 2;
constexpr int SMEM = 1024 + NS * STAGE + 256;
static_assert(CTAS_PER_SM * (SMEM + 1024) <= 228 * 1024, "shared memory budget");

struct Params {
    const uint8_t* w1g;
    const uint8_t* w1u;
    const uint8_t* w2;
    uint8_t* w1g_out;
    uint8_t* w1u_out;
    uint8_t* w2_out;
    const int* perm;
    int L, d, F, es;
    int RA, RB;              // rows per unit of kind A / B
    int ua_per_l, ub_per_l;  // units per module
    int units_a, units;
    DeviceStatus* st;
    unsigned long long wait_limit_ns;
};

struct Bars {
    uint64_t full[NS];   // loads landed (transaction bytes)
    uint64_t empty[NS];  // the consumers have read the stage
    uint32_t valid[NS];  // kind A: bit r set when row r's index is in range
    int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct Unit {
    bool a;
    int l, first, n;  // module, first row, rows
};

__device__ __forceinline__ Unit unit_at(const Params& p, int u) {
    Unit x;
    x.a = u < p.units_a;
    const int v = x.a ? u : u - p.units_a;
    const int per = x.a ? p.ua_per_l : p.ub_per_l;
    const int rows = x.a ? p.RA : p.RB;
    x.l = v / per;
    x.first = (v - x.l * per) * rows;
    x.n = min(rows, (x.a ? p.F : p.d) - x.first);
    return x;
}

// Lane r's source index for kind-A unit x (row first + r), or -1.
__device__ __forceinline__ int unit_index(const Params& p, const Unit& x, int lane) {
    return x.a && lane < x.n ? p.perm[static_cast<long long>(x.l) * p.F + x.first + lane] : -1;
}

// Warp 0: arms stage s and issues unit x's loads into it.  idx: this lane's
// unit_index, loaded ahead so that its latency overlaps the previous units'
// issue.
__device__ __forceinline__ void issue_loads(const Params& p, const Unit& x, int idx, uint8_t* stage, Bars* bars,
                                            int s, int lane, volatile int* abort_flag) {
    const long long row_bytes = static_cast<long long>(p.d) * p.es;
    if (x.a) {
        const bool ok = lane < x.n && idx >= 0 && idx < p.F;
        if (lane < x.n && !ok) report_bad_index(p.st, x.first + lane);
        const uint32_t mask = __ballot_sync(0xffffffffu, ok);
        if (lane == 0) {
            bars->valid[s] = mask;
            mbar_arrive_expect_tx(&bars->full[s], static_cast<uint32_t>(2 * __popc(mask) * row_bytes));
        }
        __syncwarp();
        if (ok) {
            const long long src = (static_cast<long long>(x.l) * p.F + idx) * row_bytes;
            const long long all = static_cast<long long>(p.L) * p.F * row_bytes;
            // a checked build: the source row inside [L][F] rows
            if (checked_range(src, row_bytes, all, p.st, abort_flag, kWhereBoundsLoad)) {
                bulk_load(stage + lane * row_bytes, p.w1g + src, static_cast<uint32_t>(row_bytes), &bars->full[s]);
                bulk_load(stage + (p.RA + lane) * row_bytes, p.w1u + src, static_cast<uint32_t>(row_bytes),
                          &bars->full[s]);
            }
        }
    } else if (lane == 0) {
        const long long row_bytes2 = static_cast<long long>(p.F) * p.es;
        const long long src = (static_cast<long long>(x.l) * p.d + x.first) * row_bytes2;
        const uint32_t bytes = static_cast<uint32_t>(x.n * row_bytes2);
        mbar_arrive_expect_tx(&bars->full[s], bytes);
        if (checked_range(src, x.n * row_bytes2, static_cast<long long>(p.L) * p.d * row_bytes2, p.st, abort_flag,
                          kWhereBoundsLoad))
            bulk_load(stage, p.w2 + src, bytes, &bars->full[s]);
    }
}

template <typename T>
__global__ void __launch_bounds__(THREADS, CTAS_PER_SM) permute_pipe_kernel(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* stages = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    Bars* bars = reinterpret_cast<Bars*>(stages + NS * STAGE);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], CONSUMERS);
        }
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    WaitCtx wc{p.st, &bars->abort_flag, p.wait_limit_ns};
    volatile int* abort_flag = &bars->abort_flag;
    constexpr int E = 16 / sizeof(T);
    const long long row_bytes = static_cast<long long>(p.d) * p.es;
    // this CTA's units: blockIdx.x + k * gridDim.x
    const int mine = p.units > static_cast<int>(blockIdx.x)
                         ? (p.units - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                         : 0;
    auto unit_of = [&](int k) { return unit_at(p, static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x)); };
    int armed_parity[NS];  // warp 0: the last phase armed on each full barrier
    for (int s = 0; s < NS; ++s) armed_parity[s] = -1;

    if (warp == 0) {
        // ------------------------------------------------ loads
        // the source indices of the next two units are loaded a unit ahead
        int idx0 = mine > 0 ? unit_index(p, unit_of(0), lane) : -1;
        int idx1 = mine > 1 ? unit_index(p, unit_of(1), lane) : -1;
        for (int k = 0; k < mine; ++k) {
            const int s = k % NS;
            const int idx2 = k + 2 < mine ? unit_index(p, unit_of(k + 2), lane) : -1;
            if (k >= NS && !mbar_wait(&bars->empty[s], static_cast<uint32_t>((k / NS - 1) & 1), wc,
                                      kWherePermStage, k))
                break;
            issue_loads(p, unit_of(k), idx0, stages + s * STAGE, bars, s, lane, abort_flag);
            armed_parity[s] = (k / NS) & 1;
            idx0 = idx1;
            idx1 = idx2;
        }
    } else {
        // ------------------------------------------------ stores
        const int ct = tid - 32;
        for (int k = 0; k < mine; ++k) {
            const int s = k % NS;
            const uint8_t* stage = stages + s * STAGE;
            const Unit x = unit_of(k);
            if (!mbar_wait(&bars->full[s], static_cast<uint32_t>((k / NS) & 1), wc, kWherePermStage, k)) break;
            if (x.a) {
                // output rows first.. of both matrices, 16 bytes per thread
                const uint32_t valid = bars->valid[s];
                const int vec_per_row = static_cast<int>(row_bytes / 16);
                const int nvec = x.n * vec_per_row;
                const long long dst = (static_cast<long long>(x.l) * p.F + x.first) * row_bytes;
                for (int v = ct; v < 2 * nvec; v += CONSUMERS) {
                    const int m = v >= nvec ? 1 : 0;
                    const int w = v - m * nvec;
                    const int r = w / vec_per_row;
                    uint4 val = make_uint4(0u, 0u, 0u, 0u);
                    if ((valid >> r) & 1u)
                        val = reinterpret_cast<const uint4*>(stage + (m * p.RA + r) * row_bytes)[w - r * vec_per_row];
                    // a checked build: the 16 bytes inside their matrix
                    if (checked_range(dst + 16ll * w, 16, static_cast<long long>(p.L) * p.F * row_bytes, p.st,
                                      abort_flag, kWhereBoundsStore))
                        *reinterpret_cast<uint4*>((m ? p.w1u_out : p.w1g_out) + dst + 16ll * w) = val;
                }
            } else {
                const T* in_s = reinterpret_cast<const T*>(stage);
                const int* pl = p.perm + static_cast<long long>(x.l) * p.F;
                T* out = reinterpret_cast<T*>(p.w2_out) + (static_cast<long long>(x.l) * p.d + x.first) * p.F;
                for (int c = ct; c < p.F / E; c += CONSUMERS) {
                    int idx[E];
#pragma unroll
                    for (int q = 0; q < E; q += 4) {
                        const int4 v = __ldg(reinterpret_cast<const int4*>(pl + c * E + q));
                        idx[q] = v.x, idx[q + 1] = v.y, idx[q + 2] = v.z, idx[q + 3] = v.w;
                    }
#pragma unroll
                    for (int q = 0; q < E; ++q) {
                        if (idx[q] < 0 || idx[q] >= p.F) {
                            if (x.first == 0) report_bad_index(p.st, c * E + q);
                            idx[q] = -1;
                        }
                    }
                    for (int r = 0; r < x.n; ++r) {
                        const T* row = in_s + static_cast<long long>(r) * p.F;
                        union {
                            uint4 u;
                            T e[E];
                        } pack;
#pragma unroll
                        for (int q = 0; q < E; ++q) pack.e[q] = idx[q] >= 0 ? row[idx[q]] : T(0);
                        const long long off = static_cast<long long>(r) * p.F + static_cast<long long>(c) * E;
                        // a checked build: the output vector inside W2_out
                        if (checked_range((static_cast<long long>(x.l) * p.d + x.first) * p.F + off, E,
                                          static_cast<long long>(p.L) * p.d * p.F, p.st, abort_flag,
                                          kWhereBoundsStore))
                            *reinterpret_cast<uint4*>(out + off) = pack.u;
                    }
                }
            }
            mbar_arrive(&bars->empty[s]);  // this thread has read the stage
        }
    }
    __syncthreads();
    if (tid == 0) {
        // loads issued but not consumed (a role gave up) land before the CTA exits
        WaitCtx drain{p.st, &bars->abort_flag, p.wait_limit_ns};
        int dummy = 0;
        drain.abort_flag = &dummy;
        for (int s = 0; s < NS; ++s)
            if (armed_parity[s] >= 0)
                mbar_wait(&bars->full[s], static_cast<uint32_t>(armed_parity[s]), drain, kWhereDrain, s);
    }
}

}  // namespace pipe

}  // namespace

cudaError_t launch_permute_ffn(const void* W1g, const void* W1u, const void* W2, const int* perm, int L, int d,
                               int F, bool bf16, void* W1g_out, void* W1u_out, void* W2_out, DeviceStatus* st,
                               int num_sms, cudaStream_t s) {
    const int es = bf16 ? 2 : 4;
    const long long rows = static_cast<long long>(L) * F;
    if (rows == 0) return cudaSuccess;
    if (rows >= (1ll << 31)) return cudaErrorInvalidValue;  // the kernels number rows with 32 bits
    // the pipelined kernel, when one W1 row of each matrix, and one W2 row,
    // fit a stage
    {
        pipe::Params p;
        p.w1g = static_cast<const uint8_t*>(W1g);
        p.w1u = static_cast<const uint8_t*>(W1u);
        p.w2 = static_cast<const uint8_t*>(W2);
        p.w1g_out = static_cast<uint8_t*>(W1g_out);
        p.w1u_out = static_cast<uint8_t*>(W1u_out);
        p.w2_out = static_cast<uint8_t*>(W2_out);
        p.perm = perm;
        p.L = L;
        p.d = d;
        p.F = F;
        p.es = es;
        const long long ra = pipe::STAGE / (2ll * d * es), rb = pipe::STAGE / (1ll * F * es);
        p.RA = static_cast<int>(ra < pipe::MAX_RA ? ra : pipe::MAX_RA);
        p.RB = static_cast<int>(rb < 1024 ? rb : 1024);
        if (p.RA >= 1 && p.RB >= 1) {
            p.ua_per_l = (F + p.RA - 1) / p.RA;
            p.ub_per_l = (d + p.RB - 1) / p.RB;
            const long long ua = static_cast<long long>(L) * p.ua_per_l, ub = static_cast<long long>(L) * p.ub_per_l;
            if (ua + ub < (1ll << 31)) {
                p.units_a = static_cast<int>(ua);
                p.units = static_cast<int>(ua + ub);
                p.st = st;
                p.wait_limit_ns = kWaitLimitNs;
                const int grid = p.units < pipe::CTAS_PER_SM * num_sms ? p.units : pipe::CTAS_PER_SM * num_sms;
                auto kfn = bf16 ? pipe::permute_pipe_kernel<__nv_bfloat16> : pipe::permute_pipe_kernel<float>;
                cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, pipe::SMEM);
                if (e != cudaSuccess) return e;
                kfn<<<grid, pipe::THREADS, pipe::SMEM, s>>>(p);
                return cudaGetLastError();
            }
        }
    }
    // otherwise two launches: the W1 rows, then the W2 columns
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
