/*
 * sptp.h -- C ABI of the GB300 (sm_103a) SP-TP FFN boundary library (libsptp.so).
 *
 * The library computes the sequence-parallel tensor-parallel (SP-TP) FFN
 * sub-layer boundary of a Megatron-style transformer with the P tensor-parallel
 * shards held as P buffers on ONE GPU, and a Delayed-TP stack of FFN sub-layers.
 *
 * Sources (web pages, by title and section):
 *   [A] "[Feature] Async Tensor Parallelism for Archon Engine",
 *       "TP Communication Is on Activations, Not Weights" and "Potential
 *       Solution" (chunked all-gather + matmul; the boundary reduce-scatter ->
 *       residual add + RMSNorm -> all-gather; norm(all_gather(x)) ==
 *       all_gather(norm(x))).
 *   [B] "Affinity-Aware Sharding for Delayed Tensor Parallelism", Abstract
 *       (Delayed TP; contiguous neuron sharding).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers on the current CUDA device,
 *     row-major and densely packed unless stated.  The caller owns every
 *     buffer; the library allocates no memory and keeps no data between calls.
 *   - Element type is given by `dtype` (sptp_dtype): SPTP_BF16 (compute in
 *     fp32, store bf16; tcgen05 tensor-core GEMMs) or SPTP_FP32 (fp32
 *     throughout; CUDA-core GEMMs).  `gamma` and all weights use the same type.
 *   - Weights use the [out][in] layout: W1g, W1u are [F][d], W2 is [d][F].
 *     Shard p owns neurons F_p = [p*F/P, (p+1)*F/P): rows F_p of W1g/W1u and
 *     columns F_p of W2 ([B], contiguous layout).
 *   - Work is enqueued asynchronously on `cuda_stream` (a cudaStream_t; NULL
 *     is the legacy default stream).  Nothing is synchronised.
 *   - Errors are returned as negative sptp_status codes; argument errors are
 *     detected before any CUDA call, so an error leaves all buffers untouched.
 *     SPTP_ERR_CUDA reports a launch failure.  A device-side wait that runs
 *     out (see sptp_read_device_status) is reported through the workspace.
 *   - Shape rules: M >= 0 (M == 0 is a no-op that returns SPTP_OK; the
 *     activation pointers may then be NULL), d >= 8,
 *     d % 8 == 0, d <= 16384; F > 0, F % P == 0, (F/P) % 8 == 0;
 *     1 <= P <= 8.  (Multiples of 8 keep every row 16-byte aligned.)
 *   - Pointers must be 16-byte aligned.
 */
#ifndef SPTP_H
#define SPTP_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* In C++ the enums get int as their underlying type, so that every int a C
 * caller passes is a valid value (and is rejected by the checks below rather
 * than being undefined). */
#ifdef __cplusplus
#define SPTP_ENUM_INT : int
#else
#define SPTP_ENUM_INT
#endif

/* Element type of activations, gamma and weights. */
typedef enum sptp_dtype_e SPTP_ENUM_INT { SPTP_BF16 = 0, SPTP_FP32 = 1 } sptp_dtype;

typedef enum sptp_status_e SPTP_ENUM_INT {
    SPTP_OK = 0,
    SPTP_ERR_NULL = -1,          /* a required pointer is NULL */
    SPTP_ERR_SHAPE = -2,         /* a size or divisibility rule is violated */
    SPTP_ERR_DTYPE = -3,         /* dtype is not an sptp_dtype */
    SPTP_ERR_WORKSPACE = -4,     /* ws_bytes smaller than the *_workspace_size query */
    SPTP_ERR_CUDA = -5,          /* a CUDA runtime call or kernel launch failed */
    SPTP_ERR_TIMEOUT = -6,       /* a bounded device-side wait ran out */
    SPTP_ERR_UNIMPLEMENTED = -7, /* the requested variant does not exist for this entry point and
                                    dtype, or this device cannot run its launch */
    SPTP_ERR_ALIAS = -8,         /* an output overlaps an input it must not overlap */
    SPTP_ERR_TOO_LARGE = -9,     /* the problem needs more scratch than the library's static array */
    SPTP_ERR_DEVICE = -10,       /* current device is not compute capability 10.3 */
    SPTP_ERR_BOUNDS = -11        /* bounds-checked builds only: a kernel computed an index or address
                                    outside its buffer and skipped the access */
} sptp_status;

/*
 * sptp_variant -- how a boundary call is split into launches.  Every
 * variant computes the same outputs; they differ in how the partial sum +
 * residual + RMSNorm rows reach the GEMMs.  SPTP_VARIANT_AUTO is the
 * library's default for the entry point and dtype; any other value runs
 * exactly that variant or returns SPTP_ERR_UNIMPLEMENTED (nothing enqueued)
 * where it does not exist or this device cannot co-schedule its launch.
 *   PAIR    (sptp_ffn_forward, sptp_attn_qkv_forward; bf16 and fp32) the
 *           prologue kernel over all M rows, then the GEMM launches (bf16:
 *           tcgen05 CTA-pair GEMMs; fp32: CUDA-core GEMMs).  The default.
 *   CHAIN   (sptp_ffn_forward, bf16) the prologue kernel, then ONE persistent
 *           launch running every gate/up tile and then every down tile; a
 *           down tile starts as soon as the gate/up tiles of its rows are
 *           stored.
 *   FUSED   (sptp_ffn_forward, sptp_attn_qkv_forward, dtp_ffn_stack_forward;
 *           bf16) ONE persistent launch: prologue warps produce the normed
 *           rows in sequence order, 256-row block by block, and the GEMM tiles
 *           consume each block as soon as it is published (the chunked
 *           all-gather + matmul of [A] "Potential Solution", literally).  The
 *           default of dtp_ffn_stack_forward for bf16.
 *   LAYERS  (dtp_ffn_stack_forward) a prologue launch and two GEMM launches
 *           per module.  The default for fp32, and for bf16 where FUSED
 *           cannot be launched.
 */
typedef enum sptp_variant_e SPTP_ENUM_INT {
    SPTP_VARIANT_AUTO = 0,
    SPTP_VARIANT_PAIR = 1,
    SPTP_VARIANT_CHAIN = 2,
    SPTP_VARIANT_FUSED = 3,
    SPTP_VARIANT_LAYERS = 4
} sptp_variant;

/* Bytes at the start of every workspace holding the device status words. */
#define SPTP_WS_HEADER_BYTES 4096

/* Workspace bytes needed by sptp_ffn_forward for these sizes (0 on bad args).
 * Layout: header | y [M][d] normed activations | s [P][M][F/P] SwiGLU output. */
size_t sptp_ffn_workspace_size(int M, int d, int F, int P, int chunks, sptp_dtype dtype);

/*
 * sptp_ffn_forward -- one SP-TP FFN sub-layer boundary ([A] "Potential
 * Solution", sub-layer boundary overlap; intra-layer chunked all-gather +
 * matmul).  For every token row t:
 *     r       = sum_{p=0}^{P-1} partials[p][t]      (reduce-scatter arithmetic)
 *     h       = x[t] + r                            (residual add)
 *     y       = h * gamma / sqrt(mean_j h_j^2 + eps) (RMSNorm)
 *   and for every shard p (chunk c of y, rows [c*M/chunks, (c+1)*M/chunks),
 *   is gathered to all shards; on one GPU the gather is the identity):
 *     s_p     = silu(y W1g[F_p]^T) * (y W1u[F_p]^T)  (column-parallel, SwiGLU)
 *     out[p]  = s_p W2[:, F_p]^T                    (row-parallel partial)
 *
 *   x         [M][d]    residual stream in
 *   partials  [P][M][d] the previous sub-layer's row-parallel partials
 *   gamma     [d]       RMSNorm scale
 *   W1g, W1u  [F][d]    gate / up projections;  W2 [d][F] down projection
 *   chunks    number of sequence chunks of the all-gather; M % chunks == 0,
 *             chunks % P == 0.  Chunk c is rows [c*M/chunks, (c+1)*M/chunks)
 *             and belongs to shard floor(c*P/chunks).  With
 *             SPTP_VARIANT_FUSED the gate/up tiles read a chunk's rows of y as
 *             soon as every row of the chunk is produced; the PAIR and CHAIN
 *             variants produce every chunk before the GEMMs start, so for
 *             them chunks changes nothing but the validation.
 *   out       [P][M][d] the next sub-layer's P partials (not reduced).  Must
 *             not overlap any input or the workspace.
 *   resid_out [M][d]    h, the new residual stream; may be NULL (not written)
 *             and may be exactly x (in place).
 *   workspace at least sptp_ffn_workspace_size(...) bytes, 256-byte aligned.
 * Numerics (bf16): sums, norm and SwiGLU in fp32; h, y, s and out are each
 * rounded once to bf16 (round to nearest even).  Every variant gives the same
 * bits.
 * sptp_ffn_forward runs SPTP_VARIANT_AUTO; sptp_ffn_forward_ex runs the
 * variant it is given (PAIR, CHAIN or FUSED; see sptp_variant).
 */
int sptp_ffn_forward(const void* x, const void* partials, const void* gamma,
                     const void* W1g, const void* W1u, const void* W2,
                     int M, int d, int F, int P, int chunks, float eps, sptp_dtype dtype,
                     void* out, void* resid_out,
                     void* workspace, size_t ws_bytes, void* cuda_stream);
int sptp_ffn_forward_ex(const void* x, const void* partials, const void* gamma,
                        const void* W1g, const void* W1u, const void* W2,
                        int M, int d, int F, int P, int chunks, float eps, sptp_dtype dtype,
                        void* out, void* resid_out,
                        void* workspace, size_t ws_bytes, void* cuda_stream, sptp_variant variant);

/* Workspace bytes needed by dtp_ffn_stack_forward (0 on bad args).
 * Layout: header | y [P][M][d] | s [P][M][F/P] | pending ring [S][P][M][d],
 * S = min(delta + 1, L). */
size_t dtp_ffn_stack_workspace_size(int M, int d, int F, int P, int L, int delta, sptp_dtype dtype);

/*
 * dtp_ffn_stack_forward -- a Delayed-TP stack of L FFN sub-layers ([B],
 * Abstract).  Shard p keeps its own residual stream x_p = x_shards[p].
 * Module l on shard p computes o_p^(l) = FFN_l,p(RMSNorm_l(x_p)) with shard
 * p's neurons; shard p adds o_p^(l) to x_p at once, and another shard q's
 * o_q^(l) reaches x_p `delta` modules later (before module l + 1 + delta).
 * delta == 0 is standard TP.  After module L-1 each shard adds its own last
 * partial and the partials arriving then; `flush` != 0 also adds every
 * other-shard partial still pending.
 *
 *   x_shards [P][M][d]  in/out residual streams (updated in place)
 *   gamma    [L][d];  W1g, W1u [L][F][d];  W2 [L][d][F]
 *   delta >= 0; L >= 1; 1 + (P-1)*min(L, delta+1) <= 64.
 * Numerics (bf16): each stream update is summed in fp32 (own partial first,
 * then other shards in ascending shard order, then x_p) and rounded to bf16.
 * dtp_ffn_stack_forward runs SPTP_VARIANT_AUTO (FUSED for bf16 where the
 * device can run it, else LAYERS); dtp_ffn_stack_forward_ex runs the variant
 * it is given (FUSED or LAYERS).
 */
int dtp_ffn_stack_forward(void* x_shards, const void* gamma,
                          const void* W1g, const void* W1u, const void* W2,
                          int M, int d, int F, int P, int L, int delta, int flush,
                          float eps, sptp_dtype dtype,
                          void* workspace, size_t ws_bytes, void* cuda_stream);
int dtp_ffn_stack_forward_ex(void* x_shards, const void* gamma,
                             const void* W1g, const void* W1u, const void* W2,
                             int M, int d, int F, int P, int L, int delta, int flush,
                             float eps, sptp_dtype dtype,
                             void* workspace, size_t ws_bytes, void* cuda_stream, sptp_variant variant);

/* ---- Step-level entry points (the same kernels the two calls above use). ---- */

/*
 * sptp_prologue -- steps 1-3 of the boundary ([A] "Potential Solution"):
 * h = x + sum_p partials[p]; y = RMSNorm(h) * gamma.  h_out may be NULL or x.
 * y_out [M][d] must not overlap the inputs.
 */
int sptp_prologue(const void* x, const void* partials, const void* gamma,
                  int M, int d, int P, float eps, sptp_dtype dtype,
                  void* h_out, void* y_out, void* cuda_stream);

/*
 * sptp_gateup_swiglu -- column-parallel gate/up GEMM with the SwiGLU epilogue
 * for every shard ([A] "Potential Solution"): s[p] = silu(y W1g[F_p]^T) *
 * (y W1u[F_p]^T), s_out laid out [P][M][F/P].  workspace: at least
 * SPTP_WS_HEADER_BYTES (status words).
 */
int sptp_gateup_swiglu(const void* y, const void* W1g, const void* W1u,
                       int M, int d, int F, int P, sptp_dtype dtype, void* s_out,
                       void* workspace, size_t ws_bytes, void* cuda_stream);

/*
 * sptp_down_proj -- row-parallel down GEMM per shard ([A] "Potential
 * Solution"): out[p] = s[p] W2[:, F_p]^T with s [P][M][F/P], out [P][M][d].
 * Also the row-parallel output projection of an attention sub-layer (s = the
 * per-shard attention output, W2 = Wo [d][F]).  workspace: at least
 * SPTP_WS_HEADER_BYTES.
 */
int sptp_down_proj(const void* s, const void* W2, int M, int d, int F, int P, sptp_dtype dtype,
                   void* out, void* workspace, size_t ws_bytes, void* cuda_stream);

/* Workspace bytes needed by sptp_attn_qkv_forward (0 on bad args).
 * Layout: header | y [M][d]. */
size_t sptp_attn_qkv_workspace_size(int M, int d, int N, int P, int chunks, sptp_dtype dtype);

/*
 * sptp_attn_qkv_forward -- the sub-layer boundary in front of an attention
 * sub-layer ([A] "Potential Solution": 4 boundaries per block, between the
 * attention and FFN sub-layers both ways).  Steps 1-3 as in
 * sptp_ffn_forward (partial sum, residual add, RMSNorm), the (identity)
 * chunked gather, then each shard's column-parallel QKV projection:
 *     qkv_out[p] = y Wqkv[p*N/P .. (p+1)*N/P)^T
 *   Wqkv      [N][d]: shard p owns rows [p*N/P, (p+1)*N/P) (its heads' q, k
 *             and v rows, arranged by the caller); N % P == 0, (N/P) % 8 == 0
 *   qkv_out   [P][M][N/P]; resid_out, chunks, eps, dtype, workspace and the
 *   shape rules as in sptp_ffn_forward.
 * The row-parallel output projection after attention, which yields the next
 * P partials, is sptp_down_proj with F = the attention width (attn [P][M][F/P],
 * Wo [d][F]).
 * sptp_attn_qkv_forward runs SPTP_VARIANT_AUTO (PAIR); sptp_attn_qkv_forward_ex
 * runs the variant it is given (PAIR, or FUSED for bf16).
 */
int sptp_attn_qkv_forward(const void* x, const void* partials, const void* gamma, const void* Wqkv,
                          int M, int d, int N, int P, int chunks, float eps, sptp_dtype dtype,
                          void* qkv_out, void* resid_out,
                          void* workspace, size_t ws_bytes, void* cuda_stream);
int sptp_attn_qkv_forward_ex(const void* x, const void* partials, const void* gamma, const void* Wqkv,
                             int M, int d, int N, int P, int chunks, float eps, sptp_dtype dtype,
                             void* qkv_out, void* resid_out,
                             void* workspace, size_t ws_bytes, void* cuda_stream, sptp_variant variant);

/*
 * sptp_permute_ffn_neurons -- executes a neuron-permutation shard map for
 * Delayed TP ([B], Abstract: the dense model is permuted before it is
 * sharded; with delayed partials, which neurons share a device changes the
 * model).  For every module l and new neuron i, new neuron i is old neuron
 * perm[l][i]:
 *     W1g_out[l][i][:] = W1g[l][perm[l][i]][:],  W1u_out likewise,
 *     W2_out[l][:][i]  = W2[l][:][perm[l][i]].
 * Contiguous sharding of the outputs (dtp_ffn_stack_forward) then gives
 * shard p the old neurons perm[l][F_p].
 *   W1g, W1u [L][F][d];  W2 [L][d][F];  perm: DEVICE int32 [L][F], meant to
 *   be a permutation of 0..F-1 per module.  An entry outside [0, F) is
 *   recorded as SPTP_ERR_SHAPE in the workspace status words (see
 *   sptp_read_device_status) and its outputs are zero-filled.
 *   Outputs must not overlap the inputs or each other.  F*sizeof(dtype) <=
 *   200 KiB.  workspace: at least SPTP_WS_HEADER_BYTES.
 */
int sptp_permute_ffn_neurons(const void* W1g, const void* W1u, const void* W2, const int* perm,
                             int L, int d, int F, sptp_dtype dtype,
                             void* W1g_out, void* W1u_out, void* W2_out,
                             void* workspace, size_t ws_bytes, void* cuda_stream);

/* ---- fp8 (E4M3) linear layers ------------------------------------------------
 * [A] "Additional Information" names fp8 (MXFP8) linear layers inside
 * tensor-parallel blocks; the pages fix no scaling recipe.  This library's
 * reading: every linear quantises its bf16 input row-wise (rows along the
 * GEMM's reduction axis) to OCP E4M3 with a power-of-two scale, and its GEMM
 * accumulates in fp32 on tcgen05 (kind::f8f6f4) and dequantises in the
 * epilogue.  A power-of-two scale makes a * 2^-e exact, so the codes depend on
 * the bf16 values alone.
 */

/*
 * sptp_quantize_rows_e4m3 -- row-wise E4M3 quantisation of a bf16 [R][K]:
 *     e_r      = least integer >= -126 with max_k |a[r][k]| <= 448 * 2^e_r
 *     q[r][k]  = RNE_E4M3(a[r][k] * 2^-e_r)       (E4M3 bytes, [R][K])
 *     scale[r] = 2^e_r                            (fp32, [R])
 * The weights of sptp_ffn_forward_fp8 are quantised with it once: W1g and
 * W1u as [F][d] (R = F, K = d: one scale per neuron) and W2 as [d*P][F/P]
 * (R = d*P, K = F/P: one scale per output feature n and shard p, at index
 * n*P + p -- shard p quantises its own slice).
 *   R >= 0 (0 is a no-op), K > 0, K % 16 == 0; a and q 16-byte aligned,
 *   scale 4-byte aligned; q and scale must not overlap a or each other.
 *   Inputs must be finite (non-finite values are outside the contract).
 */
int sptp_quantize_rows_e4m3(const void* a, long long R, int K, void* q, float* scale,
                            void* cuda_stream);

/* Workspace bytes needed by sptp_ffn_forward_fp8 (0 on bad args).  Layout:
 * header | y bf16 [M][d] | qy [M][d] | sy [M] | s bf16 [P][M][F/P] |
 * qs [P][M][F/P] | ss [P][M], each part 256-byte aligned. */
size_t sptp_ffn_fp8_workspace_size(int M, int d, int F, int P, int chunks);

/*
 * sptp_ffn_forward_fp8 -- sptp_ffn_forward with fp8 linear layers (bf16
 * activations in and out).  Steps 1-3 as there (fp32 partial sum, residual
 * add, RMSNorm); y is the bf16 activation; then for every shard p:
 *     qy, sy = quantize_rows(y)                    (over d, one scale per token)
 *     a      = (qy qW1g[F_p]^T) * sy[t] * sW1g[n]   b likewise with W1u
 *     s_p    = bf16(silu(a) * b)
 *     qs, ss = quantize_rows(s_p)                  (over F/P, per token and shard)
 *     out[p] = bf16((qs qW2[:, F_p]^T) * ss[p][t] * sW2[n*P + p])
 *   x, partials, gamma, out, resid_out, chunks, eps: as in sptp_ffn_forward
 *   (bf16).  qW1g, qW1u [F][d] E4M3 with sW1g, sW1u [F] fp32; qW2 [d][F]
 *   E4M3 with sW2 [d][P] fp32: the outputs of sptp_quantize_rows_e4m3 above.
 *   Shape rules of sptp_ffn_forward plus d % 16 == 0 and (F/P) % 16 == 0.
 */
int sptp_ffn_forward_fp8(const void* x, const void* partials, const void* gamma,
                         const void* qW1g, const float* sW1g, const void* qW1u, const float* sW1u,
                         const void* qW2, const float* sW2,
                         int M, int d, int F, int P, int chunks, float eps,
                         void* out, void* resid_out,
                         void* workspace, size_t ws_bytes, void* cuda_stream);

/*
 * sptp_prologue_e4m3 -- steps 1-3 with the gate/up linear's quantisation of y
 * fused (one launch where a row's sources fit the kernel's shared-memory
 * ring; otherwise y is stored to y_work and quantised by a second launch):
 * h = x + sum_p partials[p]; y = bf16(RMSNorm(h) * gamma); q_out [M][d] and
 * scale_out [M] as sptp_quantize_rows_e4m3(y).  bf16 only; h_out may be NULL
 * or x; y_work [M][d] bf16 scratch (contents undefined afterwards); d % 16 == 0.
 */
int sptp_prologue_e4m3(const void* x, const void* partials, const void* gamma,
                       int M, int d, int P, float eps,
                       void* h_out, void* y_work, void* q_out, float* scale_out, void* cuda_stream);

/* The two fp8 GEMMs of sptp_ffn_forward_fp8 as separate launches:
 *   sptp_gateup_swiglu_e4m3: s_out [P][M][F/P] bf16 from qy [M][d], sy [M].
 *   sptp_down_proj_e4m3: out [P][M][d] bf16 from qs [P][M][F/P], ss [P][M].
 * Weights and scales as in sptp_ffn_forward_fp8; workspace: at least
 * SPTP_WS_HEADER_BYTES (status words). */
int sptp_gateup_swiglu_e4m3(const void* qy, const float* sy, const void* qW1g, const float* sW1g,
                            const void* qW1u, const float* sW1u, int M, int d, int F, int P,
                            void* s_out, void* workspace, size_t ws_bytes, void* cuda_stream);
int sptp_down_proj_e4m3(const void* qs, const float* ss, const void* qW2, const float* sW2,
                        int M, int d, int F, int P, void* out,
                        void* workspace, size_t ws_bytes, void* cuda_stream);

/*
 * sptp_read_device_status -- synchronises `cuda_stream` and returns the
 * status the kernels recorded in the workspace header since the last call
 * that reset it (every entry point above resets it when it starts):
 * SPTP_OK; SPTP_ERR_TIMEOUT if a bounded device-side wait ran out (the
 * kernels then stop early and their outputs are undefined); or
 * SPTP_ERR_SHAPE if sptp_permute_ffn_neurons met an index outside [0, F).  No counterpart
 * on the pages: this is the library's own failure detection.
 */
int sptp_read_device_status(const void* workspace, void* cuda_stream);

/*
 * sptp_wait_selftest -- enqueues a one-CTA kernel that waits on a flag in the
 * workspace header that nothing sets and on an mbarrier that never completes,
 * each with the bounded wait the GEMM kernels use and a limit of `limit_ns`
 * nanoseconds; both waits give up and record SPTP_ERR_TIMEOUT.  If
 * `preset_flag` != 0 the flag is set first and the flag wait succeeds.  Used to
 * test failure detection without hanging the GPU.  No counterpart on the pages.
 */
int sptp_wait_selftest(void* workspace, size_t ws_bytes, unsigned long long limit_ns,
                       int preset_flag, void* cuda_stream);

/* Bytes of the static device scratch array used by sptp_ffn_forward_noalloc. */
#define SPTP_NOALLOC_SCRATCH_BYTES (64u << 20)

/*
 * sptp_ffn_forward_noalloc -- sptp_ffn_forward for callers that cannot
 * allocate device memory (for example a plugin inside a host framework that
 * owns every device allocation, or a serving loop that must not call
 * cudaMalloc because it can synchronise the device).  The pages describe no
 * such entry point; it exists for those callers.
 *   - Arguments, results and errors are those of sptp_ffn_forward (variant
 *     AUTO), without the workspace.  The caller still passes every input and
 *     output.  The arguments are checked first, in the same order and with
 *     the same codes; then the size limit; then the device.
 *   - Scratch is a library-owned 256-byte aligned __device__ array of
 *     SPTP_NOALLOC_SCRATCH_BYTES (64 MiB) that every GPU loading the library
 *     holds until the process exits.  Problems whose
 *     sptp_ffn_workspace_size(...) exceeds it return SPTP_ERR_TOO_LARGE
 *     before any CUDA call (bf16, d=4096, F=14336: up to about 1800 tokens).
 *   - No cudaMalloc, cudaFree or other allocating call is made.  The array's
 *     device address is looked up (cudaGetSymbolAddress) on the first call in
 *     each device context, with that device current; make that first call
 *     before any stream capture.
 *   - Every call shares the one array, so calls whose work overlaps on the
 *     GPU (different streams, or different host threads) race and give wrong
 *     results; serialise them.  The array keeps the last call's contents; the
 *     status words are cleared at the start of each call.
 */
int sptp_ffn_forward_noalloc(const void* x, const void* partials, const void* gamma,
                             const void* W1g, const void* W1u, const void* W2,
                             int M, int d, int F, int P, int chunks, float eps, sptp_dtype dtype,
                             void* out, void* resid_out, void* cuda_stream);

/*
 * Failure detection of the no-allocation forward, whose status words live in
 * the library's static array rather than in a caller workspace.
 *   sptp_noalloc_read_device_status: as sptp_read_device_status, for the
 *     last sptp_ffn_forward_noalloc on the current device (synchronises
 *     `cuda_stream`).
 *   sptp_noalloc_wait_selftest: as sptp_wait_selftest, with the static
 *     array's status words.
 * No counterpart on the pages.
 */
int sptp_noalloc_read_device_status(void* cuda_stream);
int sptp_noalloc_wait_selftest(unsigned long long limit_ns, int preset_flag, void* cuda_stream);

/* Human-readable text of a status code (static storage). */
const char* sptp_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPTP_H */
