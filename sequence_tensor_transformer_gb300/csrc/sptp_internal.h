// Internal declarations shared by the library's translation units:
// kernel parameter blocks and host-side launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sptp {

constexpr int kMaxGroups = 8;          // shards per launch (P <= 8)
constexpr int kMaxSrcPerGroup = 64;    // partial sources summed into one stream
constexpr int kMaxSrc = kMaxGroups * kMaxSrcPerGroup;

// Device status words at the start of every workspace.
struct DeviceStatus {
    int code;       // 0 or SPTP_ERR_TIMEOUT
    int where;      // which wait gave up (kWhere*)
    int block;      // blockIdx.x of the first CTA that gave up
    int info;       // role-specific detail (tile index)
    int flag;       // test flag for the wait self-test
};

enum : int {
    kWhereProducerEmpty = 1,
    kWhereMmaFull = 2,
    kWhereMmaAccEmpty = 3,
    kWhereEpilogueAccFull = 4,
    kWhereDrain = 5,
    kWhereSelftestFlag = 6,
    kWhereSelftestBarrier = 7,
    kWherePrologueFull = 8,
    kWherePrologueEmpty = 9,
    kWhereFusedRows = 10,
    kWhereFusedGateUp = 11,
    kWherePermIndex = 12,
    kWherePermStage = 13,
    // bounds-checked builds (SPTP_BOUNDS_CHECK): what failed its check
    kWhereBoundsTile = 20,     // a decoded tile or row index outside its range
    kWhereBoundsCounter = 21,  // a readiness-counter index
    kWhereBoundsRing = 22,     // a pending-ring slot, module or source shard
    kWhereBoundsCluster = 23,  // the cluster shape or a CTA's rank in it
    kWhereBoundsTma = 24,      // a TMA box origin (alignment or range)
    kWhereBoundsStore = 25,    // a global store outside its buffer
    kWhereBoundsLoad = 26,     // a global load or bulk copy outside its buffer
};

// Default limit of every bounded device-side wait (ns). A legitimate wait in
// these kernels lasts microseconds.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// ---------------------------------------------------------------- prologue
struct PrologueGroup {
    const void* x;   // [M][d]
    void* h;         // [M][d] or nullptr
    void* y;         // [M][d] or nullptr (accumulate only, no norm)
    int src_begin;   // first index into PrologueParams::src
    int n_src;       // number of partial sources summed into this group
};

struct PrologueParams {
    PrologueGroup grp[kMaxGroups];
    const void* src[kMaxSrc];
    const void* gamma;   // [d]
    int G, M, d;
    float eps;
    DeviceStatus* status;            // may be null (no status words)
    unsigned long long wait_limit_ns;
    // bf16, G == 1 only: when q != nullptr the bf16 y is also quantised row-wise
    // to E4M3 codes q [M][d] with power-of-two scales qscale [M] (grp[0].y
    // must still be given: rows too wide for the fused path are written there
    // and quantised by a second launch)
    void* q;
    float* qscale;
};

// Launches the partial-sum + residual + RMSNorm kernel over G groups of M rows.
cudaError_t launch_prologue(const PrologueParams& p, bool bf16, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------- tcgen05 GEMM
// out_g[m][n] = epilogue( sum_k A_g[m][k] * B_g[n][k] ) for every group g.
// SwiGLU mode: B_g is the gate block (mapB0) stacked on the up block (mapB1),
// 128 rows each, and out = silu(gate) * up; plain mode: B_g has 256 rows per
// tile (mapB0) and out = the bf16-rounded accumulator.
struct TcGemmParams {
    CUtensorMap mapA[kMaxGroups];
    CUtensorMap mapB0[kMaxGroups];
    CUtensorMap mapB1[kMaxGroups];
    void* out[kMaxGroups];
    long long ldo;         // output row stride (elements)
    int M, N, K;           // rows, output columns, reduction length (per group)
    int G, mt, nt, nk;     // groups, m-tiles, n-tiles, k-blocks
    int band;              // m-tiles per raster band
    DeviceStatus* status;
    unsigned long long wait_limit_ns;
    // E4M3 operands only: power-of-two dequantisation scales, applied in the
    // epilogue as acc * row_scale[row] * col_scale[col * col_scale_stride]
    const float* row_scale[kMaxGroups];   // per A row (token)
    const float* col_scale0[kMaxGroups];  // per output column (B0 row)
    const float* col_scale1[kMaxGroups];  // per SwiGLU up column (B1 row)
    int col_scale_stride;
    // kStore with split_w > 0: the output columns belong to consecutive
    // blocks of split_w columns, block j stored at out[0] + j * split_stride
    // as a [M][split_w] matrix (column-parallel shards computed as one GEMM)
    int split_w;
    long long split_stride;
};

enum class Epi { kSwiGLU, kStore };

// CTA-pair (cta_group::2) GEMM: tiles of 256 rows (mt counts 256-row tiles)
// and 256 B rows; tensor maps with boxes of 64 x 128.
cudaError_t launch_tc_gemm_pair(const TcGemmParams& p, Epi epi, int num_sms, cudaStream_t s);
// The same CTA-pair GEMM on E4M3 operands (tcgen05 kind::f8f6f4; tensor maps
// of bytes with boxes of 128 x 128), dequantised in the epilogue.
cudaError_t launch_tc_gemm_pair_e4m3(const TcGemmParams& p, Epi epi, int num_sms, cudaStream_t s);

// Encodes a 2-D byte (E4M3) tensor map with 128-byte swizzle.
bool encode_map_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                   uint32_t box_inner, uint32_t box_outer);

// Row-wise E4M3 quantiser: q[r][k] = RNE_E4M3(a[r][k] * 2^-e_r), scale[r] =
// 2^e_r with e_r the least integer >= -126 such that max_k |a[r][k]| <=
// 448 * 2^e_r.  a bf16 [R][K], K % 8 == 0.
cudaError_t launch_quantize_rows_e4m3(const void* a, long long R, int K, void* q, float* scale, int num_sms,
                                      cudaStream_t s);

// Encodes a 2-D bf16 tensor map (inner = contiguous dim) with 128-byte swizzle.
bool encode_map_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

// ---------------------------------------------------------------- fused boundary
// One persistent CTA-pair launch: prologue rows, gate/up + SwiGLU tiles and
// down tiles with bounded-wait readiness counters between them (bf16).
struct FusedParams {
    CUtensorMap mapY;                  // y [M][d], box 64 x 128
    CUtensorMap mapW1g[kMaxGroups];    // W1g rows F_g [f][d], box 64 x 128
    CUtensorMap mapW1u[kMaxGroups];    // W1u rows F_g
    CUtensorMap mapS[kMaxGroups];      // s_g [M][f], box 64 x 128
    CUtensorMap mapW2[kMaxGroups];     // W2 columns F_g [d][f] (row stride F), box 64 x 128
    void* s_out[kMaxGroups];           // s_g
    void* out[kMaxGroups];             // out[g] [M][d]
    const void* x;                     // [M][d]
    const void* partials[kMaxGroups];  // [M][d] each
    const void* gamma;                 // [d]
    void* h_out;                       // [M][d] or nullptr
    void* y;                           // [M][d] (workspace)
    float eps;
    int M, d, P, f;
    int mt, nt_gu, nt_dn, nk_gu, nk_dn;   // 256-row tiles
    int band0, band;                      // m-tiles of the first gate/up band, of the others
    int tiles_gu, tiles_dn;
    // qkv != 0: the boundary in front of attention.  The first tile phase is
    // a column-parallel store GEMM (B = mapW1g[g], shard g's Wqkv rows [f][d];
    // output s_out[g] [M][f]) and there is no down phase (tiles_dn == 0).
    int qkv;
    // block_rows != 0: the CTA's prologue warps take one row together (needs
    // P + 1 <= 5 sources and d <= 4096); each of them publishes its part, so a
    // row adds PRO_WARPS to its chunk's counter
    int block_rows;
    // pre_normed != 0: y was written by a preceding prologue launch (stream
    // order); the prologue warps idle and gate/up tiles do not wait for rows
    int pre_normed;
    // The sequence chunks of the (identity) all-gather: chunk c is rows
    // [c * chunk_rows, (c + 1) * chunk_rows); a gate/up tile reads its rows of
    // y once every chunk they overlap is complete.
    int chunks, chunk_rows;
    int* chunk_ready;                  // [chunks] prologue rows published per chunk
    int* gu_done;                      // [P][mt] gate/up tile halves stored
    DeviceStatus* status;
    unsigned long long wait_limit_ns;
};

int fused_max_pairs(int num_sms);
cudaError_t launch_boundary_fused(const FusedParams& p, int pairs, cudaStream_t s);

// ---------------------------------------------------------------- fused Delayed-TP stack
struct DtpFusedParams {
    CUtensorMap mapY;    // y [P][M][d] as {d, M, P}, box {64, 128, 1}
    CUtensorMap mapW1g;  // W1g [L][P][f][d] as {d, f, L*P}, box {64, 128, 1}
    CUtensorMap mapW1u;
    CUtensorMap mapS;    // s [P][M][f] as {f, M, P}, box {64, 128, 1}
    CUtensorMap mapW2;   // W2 [L][d][P][f] as {f, P, d, L}, box {64, 1, 128, 1}
    void* x;             // x_shards [P][M][d], updated in place
    const void* gamma;   // [L][d]
    void* y;             // [P][M][d]
    void* s;             // [P][M][f]
    void* ring;          // pending partials [S][P][M][d]
    float eps;
    int M, d, P, f, L, delta, flush, S;
    int mt, nt_gu, nt_dn, nk_gu, nk_dn;
    int tiles_per_lm, total_tiles;
    int lag;             // blocks between a block's gate/up and down tiles (< mt)
    int* rb_ready;       // [L][mt]   prologue rows normed (all shards)
    int* gu_done;        // [L][P][mt] gate/up tile halves stored
    int* dn_done;        // [L][mt]   down tile halves stored (all shards)
    DeviceStatus* status;
    unsigned long long wait_limit_ns;
};

int dtp_fused_max_pairs(int num_sms);
cudaError_t launch_dtp_fused(const DtpFusedParams& p, int pairs, cudaStream_t s);

// Encodes a rank-N bf16 tensor map (dims innermost first, strides in bytes
// for dims 1..N-1) with 128-byte swizzle.
bool encode_map_bf16_nd(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                        const uint64_t* strides_bytes, const uint32_t* box);

// ---------------------------------------------------------------- fp32 SIMT GEMM
struct SimtGemmParams {
    const float* A[kMaxGroups];
    const float* B0[kMaxGroups];
    const float* B1[kMaxGroups];
    float* C[kMaxGroups];
    long long lda, ldb, ldc;
    int M, N, K, G;
};

cudaError_t launch_simt_gemm(const SimtGemmParams& p, Epi epi, cudaStream_t s);

// ---------------------------------------------------------------- neuron permutation
cudaError_t launch_permute_ffn(const void* W1g, const void* W1u, const void* W2, const int* perm, int L, int d,
                               int F, bool bf16, void* W1g_out, void* W1u_out, void* W2_out, DeviceStatus* st,
                               int num_sms, cudaStream_t s);

// ---------------------------------------------------------------- argument checks (api.cu)
// Every argument check of sptp_ffn_forward_ex, with no CUDA call.
int check_ffn_forward_args(const void* x, const void* partials, const void* gamma, const void* W1g,
                           const void* W1u, const void* W2, int M, int d, int F, int P, int chunks, float eps,
                           int dtype, const void* out, const void* resid_out, const void* workspace,
                           size_t ws_bytes, int variant);
// SPTP_OK, SPTP_ERR_DEVICE (not compute capability 10.3) or SPTP_ERR_CUDA.
int current_device_ok();

// ---------------------------------------------------------------- self-test
cudaError_t launch_wait_selftest(DeviceStatus* st, unsigned long long limit_ns, cudaStream_t s);

}  // namespace sptp
