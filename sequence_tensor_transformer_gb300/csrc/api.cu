// C ABI of libsptp.so: argument validation, workspace layout and the launch
// sequence of every entry point.  Every step of the computation runs in the
// library's own kernels; this file only checks arguments, lays out the
// caller's workspace and enqueues launches (the grouped GEMM launches are in
// launch.cu).
#include <cuda_bf16.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "launch.h"
#include "sptp.h"
#include "sptp_internal.h"

using namespace sptp;

namespace {

constexpr int kMaxD = 16384;
constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }


bool dtype_ok(int dtype) { return dtype == SPTP_BF16 || dtype == SPTP_FP32; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    if (a == nullptr || b == nullptr || an == 0 || bn == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

// Sizes common to both entry points.
int check_common(int M, int d, int F, int P, int dtype) {
    if (!dtype_ok(dtype)) return SPTP_ERR_DTYPE;
    if (M < 0 || d < 8 || d % 8 != 0 || d > kMaxD) return SPTP_ERR_SHAPE;
    if (P < 1 || P > kMaxGroups) return SPTP_ERR_SHAPE;
    if (F <= 0 || F % P != 0 || (F / P) % 8 != 0) return SPTP_ERR_SHAPE;
    if (static_cast<long long>(M) * F >= (1ll << 40)) return SPTP_ERR_SHAPE;
    return SPTP_OK;
}


// Per-device SM count and compute capability, queried once per device.
int device_info(DevInfo* out) {
    static std::mutex mu;
    static DevInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPTP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        DevInfo di;
        if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return SPTP_ERR_CUDA;
        cache[dev] = di;
        have[dev] = true;
    }
    *out = cache[dev];
    if (out->major != 10 || out->minor != 3) return SPTP_ERR_DEVICE;
    return SPTP_OK;
}

DeviceStatus* ws_status(void* ws) { return reinterpret_cast<DeviceStatus*>(ws); }

int reset_status(void* ws, cudaStream_t s) {
    return cudaMemsetAsync(ws, 0, sizeof(DeviceStatus), s) == cudaSuccess ? SPTP_OK : SPTP_ERR_CUDA;
}

// Readiness counters of the fused Delayed-TP stack: per module, rows normed
// and down halves stored per 256-row block; gate/up halves per (shard, block).
size_t dtp_counter_bytes(int M, int P, int L) {
    const size_t mt = (static_cast<size_t>(M) + 255) / 256;
    return static_cast<size_t>(L) * mt * (2 + static_cast<size_t>(P)) * sizeof(int);
}

// A variant value the header defines (sptp_variant).
bool variant_known(int v) { return v >= SPTP_VARIANT_AUTO && v <= SPTP_VARIANT_LAYERS; }

// A cooperative launch the runtime refuses to start enqueues nothing; the
// caller may take another path (SPTP_VARIANT_AUTO) or report it.
bool launch_rejected(cudaError_t e) {
    return e == cudaErrorCooperativeLaunchTooLarge || e == cudaErrorInvalidValue || e == cudaErrorNotSupported ||
           e == cudaErrorInvalidConfiguration;
}

// Readiness counters of the fused boundary: per sequence chunk, prologue rows
// published; per (shard, 256-row block), gate/up tile halves stored.
size_t fused_counter_bytes(int M, int P, int chunks) {
    const size_t mt = (static_cast<size_t>(M) + 255) / 256;
    return (static_cast<size_t>(chunks) + static_cast<size_t>(P) * mt) * sizeof(int);
}

// Whether the persistent launches can run here: 0 if every CTA pair of the
// launch cannot be resident at once (the CTAs wait on one another).
bool fused_runs(const DevInfo& di, int M, int chunks) {
    // a chunk's counter reaches rows x prologue warps (32-bit)
    return static_cast<long long>(M / chunks) * 8 < (1ll << 31) && fused_max_pairs(di.sms) > 0;
}
bool dtp_fused_runs(const DevInfo& di, int M, int P, int L) {
    // the kernel numbers prologue rows with 32 bits
    return static_cast<long long>(P) * M * (L + 1) < (1ll << 31) && dtp_fused_max_pairs(di.sms) > 0;
}

constexpr int kFirstBandRows = 2048;

// ------------------------------------------------------------ fp8 (E4M3)


int check_fp8(int M, int d, int F, int P) {
    const int rc = check_common(M, d, F, P, SPTP_BF16);
    if (rc != SPTP_OK) return rc;
    if (d % 16 != 0 || (F / P) % 16 != 0) return SPTP_ERR_SHAPE;
    return SPTP_OK;
}


struct Fp8Layout {
    size_t y, qy, sy, s, qs, ss, total;
};

Fp8Layout fp8_layout(int M, int d, int F, int P) {
    Fp8Layout L;
    const size_t md = static_cast<size_t>(M) * d, mf = static_cast<size_t>(M) * F;
    L.y = SPTP_WS_HEADER_BYTES;
    L.qy = L.y + align_up(md * 2);
    L.sy = L.qy + align_up(md);
    L.s = L.sy + align_up(static_cast<size_t>(M) * 4);
    L.qs = L.s + align_up(mf * 2);
    L.ss = L.qs + align_up(mf);
    L.total = L.ss + align_up(static_cast<size_t>(M) * P * 4);
    return L;
}

// The whole bf16 boundary as one persistent launch (fused.cu), or with
// pre_normed its GEMM tiles alone after a prologue launch (the CHAIN
// variant).  The caller has checked fused_runs().  Returns SPTP_OK, or
// SPTP_ERR_UNIMPLEMENTED if the runtime refused the launch (nothing but the
// counter reset enqueued), or SPTP_ERR_CUDA.
int fused_forward(const void* x, const void* partials, const void* gamma, const void* W1g, const void* W1u,
                  const void* W2, int M, int d, int F, int P, int chunks, float eps, void* out, void* resid_out,
                  void* y, void* sbuf, int* counters, DeviceStatus* st, int band, const DevInfo& di,
                  cudaStream_t s, bool pre_normed = false) {
    const int max_pairs = fused_max_pairs(di.sms);
    const size_t es = 2;
    const int f = F / P;
    const size_t act = static_cast<size_t>(M) * d * es;
    FusedParams p;
    std::memset(&p, 0, sizeof(p));
    bool ok = encode_map_bf16(&p.mapY, y, d, M, static_cast<uint64_t>(d) * es, kBK, kBM);
    for (int g = 0; g < P && ok; ++g) {
        const size_t woff = static_cast<size_t>(g) * f * d * es;
        ok = encode_map_bf16(&p.mapW1g[g], cptr(W1g, woff), d, f, static_cast<uint64_t>(d) * es, kBK, kBM) &&
             encode_map_bf16(&p.mapW1u[g], cptr(W1u, woff), d, f, static_cast<uint64_t>(d) * es, kBK, kBM) &&
             encode_map_bf16(&p.mapS[g], mptr(sbuf, static_cast<size_t>(g) * M * f * es), f, M,
                             static_cast<uint64_t>(f) * es, kBK, kBM) &&
             encode_map_bf16(&p.mapW2[g], cptr(W2, static_cast<size_t>(g) * f * es), f, d,
                             static_cast<uint64_t>(F) * es, kBK, kBM);
        p.s_out[g] = mptr(sbuf, static_cast<size_t>(g) * M * f * es);
        p.out[g] = mptr(out, static_cast<size_t>(g) * act);
        p.partials[g] = cptr(partials, static_cast<size_t>(g) * act);
    }
    if (!ok) return SPTP_ERR_CUDA;
    p.x = x;
    p.gamma = gamma;
    p.h_out = resid_out;
    p.y = y;
    p.eps = eps;
    p.M = M;
    p.d = d;
    p.P = P;
    p.f = f;
    p.mt = (M + 255) / 256;
    p.nt_gu = (f + kBNSwiGLU - 1) / kBNSwiGLU;
    p.nt_dn = (d + kBNStore - 1) / kBNStore;
    p.nk_gu = (d + kBK - 1) / kBK;
    p.nk_dn = (f + kBK - 1) / kBK;
    const int pband = (band + 1) / 2;
    p.band = pband < 1 ? 1 : (pband > p.mt ? p.mt : pband);
    // First gate/up band: 2048 rows, or one sequence chunk if taller.  The
    // first wave waits for these rows from the prologue warps; a shorter band
    // starts sooner but streams the weights once more.  (Measured on the
    // 8192 x 4096 x 14336 boundary: first bands of 2048 / 4096 rows gave
    // 1670-1675 / 1638-1639 TFLOP/s.)
    const int chunk_rows = M / chunks;
    const int first_rows = chunk_rows > kFirstBandRows ? chunk_rows : kFirstBandRows;
    const int first_tiles = first_rows / 256;
    p.band0 = first_tiles < 1 ? 1 : (first_tiles > p.band ? p.band : first_tiles);
    p.tiles_gu = P * p.mt * p.nt_gu;
    p.tiles_dn = P * p.mt * p.nt_dn;
    p.block_rows = P + 1 <= 5 && d <= 4096 ? 1 : 0;
    p.pre_normed = pre_normed ? 1 : 0;
    p.chunks = chunks;
    p.chunk_rows = chunk_rows;
    p.chunk_ready = counters;
    p.gu_done = counters + chunks;
    p.status = st;
    p.wait_limit_ns = kWaitLimitNs;
    const int total = p.tiles_gu + p.tiles_dn;
    const int pairs = total < max_pairs ? total : max_pairs;
    if (cudaMemsetAsync(counters, 0, fused_counter_bytes(M, P, chunks), s) != cudaSuccess) return SPTP_ERR_CUDA;
    const cudaError_t e = launch_boundary_fused(p, pairs, s);
    if (e == cudaSuccess) return SPTP_OK;
    cudaGetLastError();
    return launch_rejected(e) ? SPTP_ERR_UNIMPLEMENTED : SPTP_ERR_CUDA;
}

// The bf16 boundary in front of attention as one persistent launch
// (fused.cu with qkv set: prologue rows feed each shard's column-parallel QKV
// GEMM).  The caller has checked fused_runs(); returns as fused_forward.
int fused_attn_forward(const void* x, const void* partials, const void* gamma, const void* Wqkv, int M, int d,
                       int N, int P, int chunks, float eps, void* qkv_out, void* resid_out, void* y, int* counters,
                       DeviceStatus* st, int band, const DevInfo& di, cudaStream_t s) {
    const int max_pairs = fused_max_pairs(di.sms);
    const size_t es = 2;
    const int n = N / P;
    const size_t act = static_cast<size_t>(M) * d * es;
    FusedParams p;
    std::memset(&p, 0, sizeof(p));
    bool ok = encode_map_bf16(&p.mapY, y, d, M, static_cast<uint64_t>(d) * es, kBK, kBM);
    for (int g = 0; g < P && ok; ++g) {
        ok = encode_map_bf16(&p.mapW1g[g], cptr(Wqkv, static_cast<size_t>(g) * n * d * es), d, n,
                             static_cast<uint64_t>(d) * es, kBK, kBM);
        p.s_out[g] = mptr(qkv_out, static_cast<size_t>(g) * M * n * es);
        p.partials[g] = cptr(partials, static_cast<size_t>(g) * act);
    }
    if (!ok) return SPTP_ERR_CUDA;
    p.x = x;
    p.gamma = gamma;
    p.h_out = resid_out;
    p.y = y;
    p.eps = eps;
    p.M = M;
    p.d = d;
    p.P = P;
    p.f = n;
    p.qkv = 1;
    p.mt = (M + 255) / 256;
    p.nt_gu = (n + kBNStore - 1) / kBNStore;
    p.nk_gu = (d + kBK - 1) / kBK;
    const int pband = (band + 1) / 2;
    p.band = pband < 1 ? 1 : (pband > p.mt ? p.mt : pband);
    const int chunk_rows = M / chunks;
    const int first_rows = chunk_rows > kFirstBandRows ? chunk_rows : kFirstBandRows;
    const int first_tiles = first_rows / 256;
    p.band0 = first_tiles < 1 ? 1 : (first_tiles > p.band ? p.band : first_tiles);
    p.tiles_gu = P * p.mt * p.nt_gu;
    p.tiles_dn = 0;
    p.block_rows = P + 1 <= 5 && d <= 4096 ? 1 : 0;
    p.chunks = chunks;
    p.chunk_rows = chunk_rows;
    p.chunk_ready = counters;
    p.gu_done = nullptr;  // no down tiles
    p.status = st;
    p.wait_limit_ns = kWaitLimitNs;
    const int pairs = p.tiles_gu < max_pairs ? p.tiles_gu : max_pairs;
    if (cudaMemsetAsync(counters, 0, static_cast<size_t>(chunks) * sizeof(int), s) != cudaSuccess)
        return SPTP_ERR_CUDA;
    const cudaError_t e = launch_boundary_fused(p, pairs, s);
    if (e == cudaSuccess) return SPTP_OK;
    cudaGetLastError();
    return launch_rejected(e) ? SPTP_ERR_UNIMPLEMENTED : SPTP_ERR_CUDA;
}

// The whole bf16 Delayed-TP stack as one persistent launch (fused_dtp.cu).
// The caller has checked dtp_fused_runs(); returns as fused_forward.
int dtp_fused_forward(void* x_shards, const void* gamma, const void* W1g, const void* W1u, const void* W2, int M,
                      int d, int F, int P, int L, int delta, int flush, float eps, void* ybase, void* sbuf,
                      void* ring, int S, int* counters, DeviceStatus* st, const DevInfo& di, cudaStream_t s) {
    const int max_pairs = dtp_fused_max_pairs(di.sms);
    const int f = F / P;
    const uint64_t es = 2;
    DtpFusedParams p;
    std::memset(&p, 0, sizeof(p));
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(M), static_cast<uint64_t>(P)};
        const uint64_t str[2] = {d * es, static_cast<uint64_t>(M) * d * es};
        const uint32_t box[3] = {kBK, kBM, 1};
        if (!encode_map_bf16_nd(&p.mapY, ybase, 3, dims, str, box)) return SPTP_ERR_CUDA;
    }
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(f),
                                  static_cast<uint64_t>(L) * P};
        const uint64_t str[2] = {d * es, static_cast<uint64_t>(f) * d * es};
        const uint32_t box[3] = {kBK, kBM, 1};
        if (!encode_map_bf16_nd(&p.mapW1g, W1g, 3, dims, str, box) ||
            !encode_map_bf16_nd(&p.mapW1u, W1u, 3, dims, str, box))
            return SPTP_ERR_CUDA;
    }
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(f), static_cast<uint64_t>(M), static_cast<uint64_t>(P)};
        const uint64_t str[2] = {f * es, static_cast<uint64_t>(M) * f * es};
        const uint32_t box[3] = {kBK, kBM, 1};
        if (!encode_map_bf16_nd(&p.mapS, sbuf, 3, dims, str, box)) return SPTP_ERR_CUDA;
    }
    {
        const uint64_t dims[4] = {static_cast<uint64_t>(f), static_cast<uint64_t>(P), static_cast<uint64_t>(d),
                                  static_cast<uint64_t>(L)};
        const uint64_t str[3] = {f * es, static_cast<uint64_t>(F) * es, static_cast<uint64_t>(d) * F * es};
        const uint32_t box[4] = {kBK, 1, kBM, 1};
        if (!encode_map_bf16_nd(&p.mapW2, W2, 4, dims, str, box)) return SPTP_ERR_CUDA;
    }
    p.x = x_shards;
    p.gamma = gamma;
    p.y = ybase;
    p.s = sbuf;
    p.ring = ring;
    p.eps = eps;
    p.M = M;
    p.d = d;
    p.P = P;
    p.f = f;
    p.L = L;
    p.delta = delta;
    p.flush = flush ? 1 : 0;
    p.S = S;
    p.mt = (M + 255) / 256;
    p.nt_gu = (f + kBNSwiGLU - 1) / kBNSwiGLU;
    p.nt_dn = (d + kBNStore - 1) / kBNStore;
    p.nk_gu = (d + kBK - 1) / kBK;
    p.nk_dn = (f + kBK - 1) / kBK;
    p.tiles_per_lm = P * (p.nt_gu + p.nt_dn);
    p.total_tiles = L * p.mt * p.tiles_per_lm;
    p.rb_ready = counters;
    p.gu_done = counters + static_cast<size_t>(L) * p.mt;
    p.dn_done = p.gu_done + static_cast<size_t>(L) * P * p.mt;
    p.status = st;
    p.wait_limit_ns = kWaitLimitNs;
    const int pairs = p.total_tiles < max_pairs ? p.total_tiles : max_pairs;
    // a block's down tiles come about one wave of tiles after its gate/up
    // tiles; the lag stays below the blocks of one module (and of the stack)
    int lag = (pairs + p.tiles_per_lm - 1) / p.tiles_per_lm + 1;
    if (lag > p.mt - 1) lag = p.mt - 1;
    if (lag > L * p.mt - 1) lag = L * p.mt - 1;
    p.lag = lag < 0 ? 0 : lag;
    if (cudaMemsetAsync(counters, 0, dtp_counter_bytes(M, P, L), s) != cudaSuccess) return SPTP_ERR_CUDA;
    const cudaError_t e = launch_dtp_fused(p, pairs, s);
    if (e == cudaSuccess) return SPTP_OK;
    cudaGetLastError();
    return launch_rejected(e) ? SPTP_ERR_UNIMPLEMENTED : SPTP_ERR_CUDA;
}

}  // namespace

namespace sptp {

// Every argument check of sptp_ffn_forward_ex, in order, with no CUDA call;
// also used by the no-allocation entry point before it touches its scratch.
int check_ffn_forward_args(const void* x, const void* partials, const void* gamma, const void* W1g,
                           const void* W1u, const void* W2, int M, int d, int F, int P, int chunks, float eps,
                           int dtype, const void* out, const void* resid_out, const void* workspace,
                           size_t ws_bytes, int variant) {
    // activations of an empty sequence (M == 0) may be NULL
    if (!gamma || !W1g || !W1u || !W2 || !workspace || (M != 0 && (!x || !partials || !out)))
        return SPTP_ERR_NULL;
    const int rc = check_common(M, d, F, P, dtype);
    if (rc != SPTP_OK) return rc;
    if (chunks < 1 || chunks % P != 0 || (M > 0 && M % chunks != 0)) return SPTP_ERR_SHAPE;
    // the launch plan: AUTO is PAIR; CHAIN and FUSED are bf16 only
    const int v = variant == SPTP_VARIANT_AUTO ? SPTP_VARIANT_PAIR : variant;
    if (!variant_known(variant) || v == SPTP_VARIANT_LAYERS || (dtype != SPTP_BF16 && v != SPTP_VARIANT_PAIR))
        return SPTP_ERR_UNIMPLEMENTED;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return SPTP_ERR_SHAPE;
    const void* ptrs[] = {x, partials, gamma, W1g, W1u, W2, out, resid_out, workspace};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SPTP_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return SPTP_ERR_SHAPE;
    const size_t need = sptp_ffn_workspace_size(M, d, F, P, chunks, static_cast<sptp_dtype>(dtype));
    if (ws_bytes < need) return SPTP_ERR_WORKSPACE;
    const size_t es = esize(dtype);
    const size_t act = static_cast<size_t>(M) * d * es;
    const size_t out_bytes = act * P;
    const size_t wg = static_cast<size_t>(F) * d * es;
    // out must not overlap anything it is computed from or the workspace
    const void* ins[] = {x, partials, gamma, W1g, W1u, W2, workspace, resid_out};
    const size_t insz[] = {act, out_bytes, d * es, wg, wg, wg, need, resid_out ? act : 0};
    for (int i = 0; i < 8; ++i)
        if (overlaps(out, out_bytes, ins[i], insz[i])) return SPTP_ERR_ALIAS;
    const void* wins[] = {x, partials, gamma, W1g, W1u, W2};
    const size_t wsz[] = {act, out_bytes, d * es, wg, wg, wg};
    for (int i = 0; i < 6; ++i)
        if (overlaps(workspace, need, wins[i], wsz[i])) return SPTP_ERR_ALIAS;
    if (resid_out && resid_out != x) {
        const void* rins[] = {x, partials, gamma, W1g, W1u, W2, workspace};
        const size_t rsz[] = {act, out_bytes, d * es, wg, wg, wg, need};
        for (int i = 0; i < 7; ++i)
            if (overlaps(resid_out, act, rins[i], rsz[i])) return SPTP_ERR_ALIAS;
    }
    return SPTP_OK;
}

// SPTP_OK if the current device is the one the kernels are built for.
int current_device_ok() {
    DevInfo di;
    return device_info(&di);
}

}  // namespace sptp

extern "C" {

const char* sptp_status_string(int status) {
    switch (status) {
        case SPTP_OK: return "ok";
        case SPTP_ERR_NULL: return "a required pointer is NULL";
        case SPTP_ERR_SHAPE: return "a size or divisibility rule is violated";
        case SPTP_ERR_DTYPE: return "unknown dtype";
        case SPTP_ERR_WORKSPACE: return "workspace too small";
        case SPTP_ERR_CUDA: return "CUDA runtime call or kernel launch failed";
        case SPTP_ERR_TIMEOUT: return "a bounded device-side wait ran out";
        case SPTP_ERR_UNIMPLEMENTED:
            return "the requested variant does not exist for this entry point and dtype, or cannot launch here";
        case SPTP_ERR_ALIAS: return "an output overlaps an input";
        case SPTP_ERR_TOO_LARGE: return "problem needs more scratch than the static no-allocation array holds";
        case SPTP_ERR_DEVICE: return "current device is not compute capability 10.3 (sm_103a)";
        case SPTP_ERR_BOUNDS: return "a bounds check of the checked build failed (the access was skipped)";
        default: return "unknown status";
    }
}

size_t sptp_ffn_workspace_size(int M, int d, int F, int P, int chunks, sptp_dtype dtype) {
    if (check_common(M, d, F, P, dtype) != SPTP_OK || chunks < 1) return 0;
    const size_t es = esize(dtype);
    return SPTP_WS_HEADER_BYTES + align_up(static_cast<size_t>(M) * d * es) +
           align_up(static_cast<size_t>(M) * F * es) + align_up(fused_counter_bytes(M, P, chunks));
}

int sptp_ffn_forward(const void* x, const void* partials, const void* gamma, const void* W1g, const void* W1u,
                     const void* W2, int M, int d, int F, int P, int chunks, float eps, sptp_dtype dtype, void* out,
                     void* resid_out, void* workspace, size_t ws_bytes, void* cuda_stream) {
    return sptp_ffn_forward_ex(x, partials, gamma, W1g, W1u, W2, M, d, F, P, chunks, eps, dtype, out, resid_out,
                               workspace, ws_bytes, cuda_stream, SPTP_VARIANT_AUTO);
}

int sptp_ffn_forward_ex(const void* x, const void* partials, const void* gamma, const void* W1g, const void* W1u,
                        const void* W2, int M, int d, int F, int P, int chunks, float eps, sptp_dtype dtype,
                        void* out, void* resid_out, void* workspace, size_t ws_bytes, void* cuda_stream,
                        sptp_variant variant) {
    int rc = check_ffn_forward_args(x, partials, gamma, W1g, W1u, W2, M, d, F, P, chunks, eps, dtype, out,
                                    resid_out, workspace, ws_bytes, variant);
    if (rc != SPTP_OK) return rc;
    const int v = variant == SPTP_VARIANT_AUTO ? SPTP_VARIANT_PAIR : variant;
    const size_t es = esize(dtype);
    const size_t act = static_cast<size_t>(M) * d * es;
    if (M == 0) return SPTP_OK;
    DevInfo di;
    if ((rc = device_info(&di)) != SPTP_OK) return rc;
    if ((v == SPTP_VARIANT_FUSED || v == SPTP_VARIANT_CHAIN) && !fused_runs(di, M, chunks))
        return SPTP_ERR_UNIMPLEMENTED;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if ((rc = reset_status(workspace, s)) != SPTP_OK) return rc;

    void* y = mptr(workspace, SPTP_WS_HEADER_BYTES);
    void* sbuf = mptr(workspace, SPTP_WS_HEADER_BYTES + align_up(act));
    int* counters = reinterpret_cast<int*>(
        mptr(workspace, SPTP_WS_HEADER_BYTES + align_up(act) + align_up(static_cast<size_t>(M) * F * es)));
    const int band = raster_band();

    if (v == SPTP_VARIANT_FUSED)
        return fused_forward(x, partials, gamma, W1g, W1u, W2, M, d, F, P, chunks, eps, out, resid_out, y, sbuf,
                             counters, ws_status(workspace), band, di, s);

    // 1-3: reduce-scatter arithmetic, residual add, RMSNorm (every chunk)
    PrologueParams pp;
    std::memset(&pp, 0, sizeof(pp));
    pp.G = 1;
    pp.M = M;
    pp.d = d;
    pp.eps = eps;
    pp.gamma = gamma;
    pp.grp[0] = PrologueGroup{x, resid_out, y, 0, P};
    for (int p = 0; p < P; ++p) pp.src[p] = cptr(partials, static_cast<size_t>(p) * act);
    pp.status = ws_status(workspace);
    pp.wait_limit_ns = kWaitLimitNs;
    if ((rc = cuda_status(launch_prologue(pp, dtype == SPTP_BF16, di.sms, s))) != SPTP_OK) return rc;

    if (v == SPTP_VARIANT_CHAIN) {
        // 4-7 as one persistent launch: gate/up and down tiles in one sequence
        // (the prologue above has run: a refused launch is a launch failure)
        rc = fused_forward(x, partials, gamma, W1g, W1u, W2, M, d, F, P, chunks, eps, out, resid_out, y, sbuf,
                           counters, ws_status(workspace), band, di, s, true);
        return rc == SPTP_ERR_UNIMPLEMENTED ? SPTP_ERR_CUDA : rc;
    }

    // 4-6: chunked gather (identity) + column-parallel gate/up + SwiGLU,
    // tiles walked chunk by chunk
    const void* A[kMaxGroups];
    for (int g = 0; g < P; ++g) A[g] = y;
    if ((rc = gateup(A, W1g, W1u, M, d, F, P, dtype, sbuf, ws_status(workspace), band, di, s)) != SPTP_OK)
        return rc;

    // 7: row-parallel down projection, one partial per shard
    void* outs[kMaxGroups];
    for (int g = 0; g < P; ++g) outs[g] = mptr(out, static_cast<size_t>(g) * act);
    return down(sbuf, W2, M, d, F, P, dtype, outs, ws_status(workspace), down_raster_band(), di, s);
}

size_t dtp_ffn_stack_workspace_size(int M, int d, int F, int P, int L, int delta, sptp_dtype dtype) {
    if (check_common(M, d, F, P, dtype) != SPTP_OK || L < 1 || delta < 0) return 0;
    const size_t es = esize(dtype);
    const size_t S = static_cast<size_t>(delta + 1 < L ? delta + 1 : L);
    const size_t act = static_cast<size_t>(M) * d * es;
    return SPTP_WS_HEADER_BYTES + align_up(act * P) + align_up(static_cast<size_t>(M) * F * es) +
           align_up(S * P * act) + align_up(dtp_counter_bytes(M, P, L));
}

int dtp_ffn_stack_forward(void* x_shards, const void* gamma, const void* W1g, const void* W1u, const void* W2,
                          int M, int d, int F, int P, int L, int delta, int flush, float eps, sptp_dtype dtype,
                          void* workspace, size_t ws_bytes, void* cuda_stream) {
    return dtp_ffn_stack_forward_ex(x_shards, gamma, W1g, W1u, W2, M, d, F, P, L, delta, flush, eps, dtype,
                                    workspace, ws_bytes, cuda_stream, SPTP_VARIANT_AUTO);
}

int dtp_ffn_stack_forward_ex(void* x_shards, const void* gamma, const void* W1g, const void* W1u, const void* W2,
                             int M, int d, int F, int P, int L, int delta, int flush, float eps, sptp_dtype dtype,
                             void* workspace, size_t ws_bytes, void* cuda_stream, sptp_variant variant) {
    if (!gamma || !W1g || !W1u || !W2 || !workspace || (M != 0 && !x_shards)) return SPTP_ERR_NULL;
    int rc = check_common(M, d, F, P, dtype);
    if (rc != SPTP_OK) return rc;
    // AUTO: the fused stack for bf16 where it can run, else per-module launches
    if (!variant_known(variant) || variant == SPTP_VARIANT_PAIR || variant == SPTP_VARIANT_CHAIN ||
        (dtype != SPTP_BF16 && variant == SPTP_VARIANT_FUSED))
        return SPTP_ERR_UNIMPLEMENTED;
    if (L < 1 || delta < 0) return SPTP_ERR_SHAPE;
    const int S = delta + 1 < L ? delta + 1 : L;
    if (1 + (P - 1) * S > kMaxSrcPerGroup) return SPTP_ERR_SHAPE;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return SPTP_ERR_SHAPE;
    const void* ptrs[] = {x_shards, gamma, W1g, W1u, W2, workspace};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SPTP_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return SPTP_ERR_SHAPE;
    const size_t need = dtp_ffn_stack_workspace_size(M, d, F, P, L, delta, dtype);
    if (ws_bytes < need) return SPTP_ERR_WORKSPACE;
    const size_t es = esize(dtype);
    const size_t act = static_cast<size_t>(M) * d * es;
    const size_t wg = static_cast<size_t>(L) * F * d * es;
    const void* ins[] = {gamma, W1g, W1u, W2, workspace};
    const size_t insz[] = {static_cast<size_t>(L) * d * es, wg, wg, wg, need};
    for (int i = 0; i < 5; ++i)
        if (overlaps(x_shards, act * P, ins[i], insz[i])) return SPTP_ERR_ALIAS;
    if (M == 0) return SPTP_OK;
    DevInfo di;
    if ((rc = device_info(&di)) != SPTP_OK) return rc;
    const bool fused_ok = dtype == SPTP_BF16 && dtp_fused_runs(di, M, P, L);
    if (variant == SPTP_VARIANT_FUSED && !fused_ok) return SPTP_ERR_UNIMPLEMENTED;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if ((rc = reset_status(workspace, s)) != SPTP_OK) return rc;

    const int f = F / P;
    char* ybase = mptr(workspace, SPTP_WS_HEADER_BYTES);
    char* sbuf = ybase + align_up(act * P);
    char* ring = sbuf + align_up(static_cast<size_t>(M) * F * es);
    int* counters = reinterpret_cast<int*>(ring + align_up(static_cast<size_t>(S) * P * act));
    if (fused_ok && variant != SPTP_VARIANT_LAYERS) {
        rc = dtp_fused_forward(x_shards, gamma, W1g, W1u, W2, M, d, F, P, L, delta, flush, eps, ybase, sbuf, ring, S,
                               counters, ws_status(workspace), di, s);
        // a launch the runtime refused enqueued nothing: AUTO takes the
        // per-module launches below
        if (rc != SPTP_ERR_UNIMPLEMENTED || variant == SPTP_VARIANT_FUSED) return rc;
    }
    auto xs = [&](int p) { return mptr(x_shards, static_cast<size_t>(p) * act); };
    auto yp = [&](int p) { return ybase + static_cast<size_t>(p) * act; };
    auto o = [&](int l, int p) { return ring + (static_cast<size_t>(l % S) * P + p) * act; };

    const void* A[kMaxGroups];
    void* outs[kMaxGroups];
    for (int l = 0; l <= L; ++l) {
        // stream update before module l (or the final one at l == L):
        // own partial of module l-1, other shards' partials of module l-1-delta
        // and, at the end with flush, every other-shard partial still pending
        PrologueParams pp;
        std::memset(&pp, 0, sizeof(pp));
        pp.G = P;
        pp.M = M;
        pp.d = d;
        pp.eps = eps;
        pp.gamma = l < L ? cptr(gamma, static_cast<size_t>(l) * d * es) : gamma;
        int ns = 0;
        for (int p = 0; p < P; ++p) {
            const int begin = ns;
            if (l >= 1) pp.src[ns++] = o(l - 1, p);
            const int k = l - 1 - delta;
            if (k >= 0)
                for (int q = 0; q < P; ++q)
                    if (q != p) pp.src[ns++] = o(k, q);
            if (l == L && flush)
                for (int kk = (L - delta > 0 ? L - delta : 0); kk < L; ++kk)
                    for (int q = 0; q < P; ++q)
                        if (q != p) pp.src[ns++] = o(kk, q);
            pp.grp[p] = PrologueGroup{xs(p), xs(p), l < L ? yp(p) : nullptr, begin, ns - begin};
        }
        pp.status = ws_status(workspace);
        pp.wait_limit_ns = kWaitLimitNs;
        if ((rc = cuda_status(launch_prologue(pp, dtype == SPTP_BF16, di.sms, s))) != SPTP_OK) return rc;
        if (l == L) break;

        const size_t woff = static_cast<size_t>(l) * F * d * es;
        for (int p = 0; p < P; ++p) A[p] = yp(p);
        if ((rc = gateup(A, cptr(W1g, woff), cptr(W1u, woff), M, d, F, P, dtype, sbuf, ws_status(workspace),
                         raster_band(), di, s)) != SPTP_OK)
            return rc;
        for (int p = 0; p < P; ++p) outs[p] = o(l, p);
        if ((rc = down(sbuf, cptr(W2, woff), M, d, F, P, dtype, outs, ws_status(workspace), down_raster_band(),
                       di, s)) != SPTP_OK)
            return rc;
        (void)f;
    }
    return SPTP_OK;
}

int sptp_prologue(const void* x, const void* partials, const void* gamma, int M, int d, int P, float eps,
                  sptp_dtype dtype, void* h_out, void* y_out, void* cuda_stream) {
    if (!gamma || (M != 0 && (!x || !partials || !y_out))) return SPTP_ERR_NULL;
    int rc = check_common(M, d, 8 * P, P, dtype);
    if (rc != SPTP_OK) return rc;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return SPTP_ERR_SHAPE;
    const void* ptrs[] = {x, partials, gamma, h_out, y_out};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SPTP_ERR_SHAPE;
    const size_t es = esize(dtype);
    const size_t act = static_cast<size_t>(M) * d * es;
    const void* ins[] = {x, partials, gamma, h_out};
    const size_t insz[] = {act, act * P, d * es, h_out ? act : 0};
    for (int i = 0; i < 4; ++i)
        if (overlaps(y_out, act, ins[i], insz[i])) return SPTP_ERR_ALIAS;
    if (h_out && h_out != x && (overlaps(h_out, act, partials, act * P) || overlaps(h_out, act, x, act)))
        return SPTP_ERR_ALIAS;
    if (M == 0) return SPTP_OK;
    DevInfo di;
    if ((rc = device_info(&di)) != SPTP_OK) return rc;
    PrologueParams pp;
    std::memset(&pp, 0, sizeof(pp));
    pp.G = 1;
    pp.M = M;
    pp.d = d;
    pp.eps = eps;
    pp.gamma = gamma;
    pp.grp[0] = PrologueGroup{x, h_out, y_out, 0, P};
    for (int p = 0; p < P; ++p) pp.src[p] = cptr(partials, static_cast<size_t>(p) * act);
    pp.status = nullptr;  // no workspace: a timed-out wait only stops the CTA
    pp.wait_limit_ns = kWaitLimitNs;
    return cuda_status(launch_prologue(pp, dtype == SPTP_BF16, di.sms, static_cast<cudaStream_t>(cuda_stream)));
}

int sptp_gateup_swiglu(const void* y, const void* W1g, const void* W1u, int M, int d, int F, int P, sptp_dtype dtype,
                       void* s_out, void* workspace, size_t ws_bytes, void* cuda_stream) {
    if (!W1g || !W1u || !workspace || (M != 0 && (!y || !s_out))) return SPTP_ERR_NULL;
    int rc = check_common(M, d, F, P, dtype);
    if (rc != SPTP_OK) return rc;
    const void* ptrs[] = {y, W1g, W1u, s_out, workspace};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SPTP_ERR_SHAPE;
    if (ws_bytes < SPTP_WS_HEADER_BYTES) return SPTP_ERR_WORKSPACE;
    const size_t es = esize(dtype);
    const size_t sb = static_cast<size_t>(M) * F * es, wg = static_cast<size_t>(F) * d * es;
    if (overlaps(s_out, sb, y, static_cast<size_t>(M) * d * es) || overlaps(s_out, sb, W1g, wg) ||
        overlaps(s_out, sb, W1u, wg) || overlaps(s_out, sb, workspace, SPTP_WS_HEADER_BYTES))
        return SPTP_ERR_ALIAS;
    if (M == 0) return SPTP_OK;
    DevInfo di;
    if ((rc = device_info(&di)) != SPTP_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if ((rc = reset_status(workspace, s)) != SPTP_OK) return rc;
    const void* A[kMaxGroups];
    for (int g = 0; g < P; ++g) A[g] = y;
    return gateup(A, W1g, W1u, M, d, F, P, dtype, s_out, ws_status(workspace), raster_band(), di, s);
}

int sptp_down_proj(const void* s_in, const void* W2, int M, int d, int F, int P, sptp_dtype dtype, void* out,
                   void* workspace, size_t ws_bytes, void* cuda_stream) {
    if (!W2 || !workspace || (M != 0 && (!s_in || !out))) return SPTP_ERR_NULL;
    int rc = check_common(M, d, F, P, dtype);
    if (rc != SPTP_OK) return rc;
    const void* ptrs[] = {s_in, W2, out, workspace};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SPTP_ERR_SHAPE;
    if (ws_bytes < SPTP_WS_HEADER_BYTES) return SPTP_ERR_WORKSPACE;
    const size_t es = esize(dtype);
    const size_t ob = static_cast<size_t>(P) * M * d * es;
    if (overlaps(out, ob, s_in, static_cast<size_t>(M) * F * es) ||
        overlaps(out, ob, W2, static_cast<size_t>(F) * d * es) ||
        overlaps(out, ob, workspace, SPTP_WS_HEADER_BYTES))
        return SPTP_ERR_ALIAS;
    if (M == 0) return SPTP_OK;
    DevInfo di;
    if ((rc = device_info(&di)) != SPTP_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if ((rc = reset_status(workspace, s)) != SPTP_OK) return rc;
    void* outs[kMaxGroups];
    for (int g = 0; g < P; ++g) outs[g] = mptr(out, static_cast<size_t>(g) * M * d * es);
    return down(s_in, W2, M, d, F, P, dtype, outs, ws_status(workspace), down_raster_band(), di, s);
}

size_t sptp_attn_qkv_workspace_size(int M, int d, int N, int P, int chunks, sptp_dtype dtype) {
    if (check_common(M, d, N, P, dtype) != SPTP_OK || chunks < 1) return 0;
    return SPTP_WS_HEADER_BYTES + align_up(static_cast<size_t>(M) * d * esize(dtype)) +
           align_up(static_cast<size_t>(chunks) * sizeof(int));
}

int sptp_attn_qkv_forward(const void* x, const void* partials, const void* gamma, const void* Wqkv, int M, int d,
                          int N, int P, int chunks, float eps, sptp_dtype dtype, void* qkv_out, void* resid_out,
                          void* workspace, size_t ws_bytes, void* cuda_stream) {
    return sptp_attn_qkv_forward_ex(x, partials, gamma, Wqkv, M, d, N, P, chunks, eps, dtype, qkv_out, resid_out,
                                    workspace, ws_bytes, cuda_stream, SPTP_VARIANT_AUTO);
}

int sptp_attn_qkv_forward_ex(const void* x, const void* partials, const void* gamma, const void* Wqkv, int M,
                             int d, int N, int P, int chunks, float eps, sptp_dtype dtype, void* qkv_out,
                             void* resid_out, void* workspace, size_t ws_bytes, void* cuda_stream,
                             sptp_variant variant) {
    if (!gamma || !Wqkv || !workspace || (M != 0 && (!x || !partials || !qkv_out))) return SPTP_ERR_NULL;
    int rc = check_common(M, d, N, P, dtype);
    if (rc != SPTP_OK) return rc;
    if (chunks < 1 || chunks % P != 0 || (M > 0 && M % chunks != 0)) return SPTP_ERR_SHAPE;
    // the launch plan: AUTO is PAIR (prologue + one column-parallel GEMM);
    // FUSED is bf16 only; there is no CHAIN or LAYERS form
    const int v = variant == SPTP_VARIANT_AUTO ? SPTP_VARIANT_PAIR : variant;
    if (!variant_known(variant) || (v != SPTP_VARIANT_PAIR && v != SPTP_VARIANT_FUSED) ||
        (dtype != SPTP_BF16 && v == SPTP_VARIANT_FUSED))
        return SPTP_ERR_UNIMPLEMENTED;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return SPTP_ERR_SHAPE;
    const void* ptrs[] = {x, partials, gamma, Wqkv, qkv_out, resid_out, workspace};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SPTP_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return SPTP_ERR_SHAPE;
    const size_t need = sptp_attn_qkv_workspace_size(M, d, N, P, chunks, dtype);
    if (ws_bytes < need) return SPTP_ERR_WORKSPACE;
    const size_t es = esize(dtype);
    const size_t act = static_cast<size_t>(M) * d * es;
    const size_t qb = static_cast<size_t>(M) * N * es, wb = static_cast<size_t>(N) * d * es;
    const void* ins[] = {x, partials, gamma, Wqkv, workspace, resid_out};
    const size_t insz[] = {act, act * P, d * es, wb, need, resid_out ? act : 0};
    for (int i = 0; i < 6; ++i)
        if (overlaps(qkv_out, qb, ins[i], insz[i])) return SPTP_ERR_ALIAS;
    const void* wins[] = {x, partials, gamma, Wqkv};
    const size_t wsz[] = {act, act * P, d * es, wb};
    for (int i = 0; i < 4; ++i)
        if (overlaps(workspace, need, wins[i], wsz[i])) return SPTP_ERR_ALIAS;
    if (resid_out && resid_out != x) {
        const void* rins[] = {x, partials, gamma, Wqkv, workspace};
        const size_t rsz[] = {act, act * P, d * es, wb, need};
        for (int i = 0; i < 5; ++i)
            if (overlaps(resid_out, act, rins[i], rsz[i])) return SPTP_ERR_ALIAS;
    }
    if (M == 0) return SPTP_OK;
    DevInfo di;
    if ((rc = device_info(&di)) != SPTP_OK) return rc;
    if (v == SPTP_VARIANT_FUSED && !fused_runs(di, M, chunks)) return SPTP_ERR_UNIMPLEMENTED;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if ((rc = reset_status(workspace, s)) != SPTP_OK) return rc;
    void* y = mptr(workspace, SPTP_WS_HEADER_BYTES);
    int* counters = reinterpret_cast<int*>(mptr(workspace, SPTP_WS_HEADER_BYTES + align_up(act)));
    if (v == SPTP_VARIANT_FUSED)
        return fused_attn_forward(x, partials, gamma, Wqkv, M, d, N, P, chunks, eps, qkv_out, resid_out, y,
                                  counters, ws_status(workspace), raster_band(), di, s);
    PrologueParams pp;
    std::memset(&pp, 0, sizeof(pp));
    pp.G = 1;
    pp.M = M;
    pp.d = d;
    pp.eps = eps;
    pp.gamma = gamma;
    pp.grp[0] = PrologueGroup{x, resid_out, y, 0, P};
    for (int p = 0; p < P; ++p) pp.src[p] = cptr(partials, static_cast<size_t>(p) * act);
    pp.status = ws_status(workspace);
    pp.wait_limit_ns = kWaitLimitNs;
    if ((rc = cuda_status(launch_prologue(pp, dtype == SPTP_BF16, di.sms, s))) != SPTP_OK) return rc;
    return colpar_store(y, Wqkv, M, d, N, P, dtype, qkv_out, ws_status(workspace), raster_band(), di,
                        s);
}

int sptp_permute_ffn_neurons(const void* W1g, const void* W1u, const void* W2, const int* perm, int L, int d,
                             int F, sptp_dtype dtype, void* W1g_out, void* W1u_out, void* W2_out, void* workspace,
                             size_t ws_bytes, void* cuda_stream) {
    if (!W1g || !W1u || !W2 || !perm || !W1g_out || !W1u_out || !W2_out || !workspace) return SPTP_ERR_NULL;
    int rc = check_common(8, d, F, 1, dtype);
    if (rc != SPTP_OK) return rc;
    if (L < 1) return SPTP_ERR_SHAPE;
    const size_t es = esize(dtype);
    if (static_cast<size_t>(F) * es > 200u * 1024u) return SPTP_ERR_SHAPE;  // one W2 row in shared memory
    if (ws_bytes < SPTP_WS_HEADER_BYTES) return SPTP_ERR_WORKSPACE;
    const void* ptrs[] = {W1g, W1u, W2, perm, W1g_out, W1u_out, W2_out, workspace};
    for (const void* q : ptrs)
        if (!aligned16(q)) return SPTP_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(perm) & 3u) != 0) return SPTP_ERR_SHAPE;
    const size_t wb = static_cast<size_t>(L) * F * d * es;
    const void* outs[] = {W1g_out, W1u_out, W2_out};
    const void* ins[] = {W1g, W1u, W2, perm, workspace};
    const size_t insz[] = {wb, wb, wb, static_cast<size_t>(L) * F * sizeof(int), SPTP_WS_HEADER_BYTES};
    for (const void* o : outs) {
        for (int i = 0; i < 5; ++i)
            if (overlaps(o, wb, ins[i], insz[i])) return SPTP_ERR_ALIAS;
        for (const void* o2 : outs)
            if (o2 != o && overlaps(o, wb, o2, wb)) return SPTP_ERR_ALIAS;
    }
    DevInfo di;
    if ((rc = device_info(&di)) != SPTP_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if ((rc = reset_status(workspace, s)) != SPTP_OK) return rc;
    return cuda_status(launch_permute_ffn(W1g, W1u, W2, perm, L, d, F, dtype == SPTP_BF16, W1g_out, W1u_out, W2_out,
                                          ws_status(workspace), di.sms, s));
}

int sptp_read_device_status(const void* workspace, void* cuda_stream) {
    if (!workspace) return SPTP_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return SPTP_ERR_CUDA;
    DeviceStatus st;
    if (cudaMemcpy(&st, workspace, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return SPTP_ERR_CUDA;
    return st.code;
}

int sptp_wait_selftest(void* workspace, size_t ws_bytes, unsigned long long limit_ns, int preset_flag,
                       void* cuda_stream) {
    if (!workspace) return SPTP_ERR_NULL;
    if (ws_bytes < SPTP_WS_HEADER_BYTES) return SPTP_ERR_WORKSPACE;
    if (limit_ns == 0 || limit_ns > 10000000000ull) return SPTP_ERR_SHAPE;
    DevInfo di;
    int rc = device_info(&di);
    if (rc != SPTP_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if ((rc = reset_status(workspace, s)) != SPTP_OK) return rc;
    if (preset_flag) {
        static const int one = 1;
        if (cudaMemcpyAsync(&ws_status(workspace)->flag, &one, sizeof(int), cudaMemcpyHostToDevice, s) !=
            cudaSuccess)
            return SPTP_ERR_CUDA;
    }
    return cuda_status(launch_wait_selftest(ws_status(workspace), limit_ns, s));
}

int sptp_quantize_rows_e4m3(const void* a, long long R, int K, void* q, float* scale, void* cuda_stream) {
    if (R < 0 || K <= 0 || K % 16 != 0 || R > (1ll << 40) / K) return SPTP_ERR_SHAPE;
    if (R == 0) return SPTP_OK;
    if (!a || !q || !scale) return SPTP_ERR_NULL;
    if (!aligned16(a) || !aligned16(q) || (reinterpret_cast<uintptr_t>(scale) & 3u) != 0) return SPTP_ERR_SHAPE;
    const size_t ab = static_cast<size_t>(R) * K * 2, qb = static_cast<size_t>(R) * K, sb = static_cast<size_t>(R) * 4;
    if (overlaps(q, qb, a, ab) || overlaps(scale, sb, a, ab) || overlaps(scale, sb, q, qb)) return SPTP_ERR_ALIAS;
    DevInfo di;
    const int rc = device_info(&di);
    if (rc != SPTP_OK) return rc;
    return cuda_status(launch_quantize_rows_e4m3(a, R, K, q, scale, di.sms, static_cast<cudaStream_t>(cuda_stream)));
}

size_t sptp_ffn_fp8_workspace_size(int M, int d, int F, int P, int chunks) {
    if (check_fp8(M, d, F, P) != SPTP_OK || chunks < 1) return 0;
    return fp8_layout(M, d, F, P).total;
}

int sptp_ffn_forward_fp8(const void* x, const void* partials, const void* gamma, const void* qW1g, const float* sW1g,
                         const void* qW1u, const float* sW1u, const void* qW2, const float* sW2, int M, int d, int F,
                         int P, int chunks, float eps, void* out, void* resid_out, void* workspace, size_t ws_bytes,
                         void* cuda_stream) {
    if (!gamma || !qW1g || !sW1g || !qW1u || !sW1u || !qW2 || !sW2 || !workspace ||
        (M != 0 && (!x || !partials || !out)))
        return SPTP_ERR_NULL;
    int rc = check_fp8(M, d, F, P);
    if (rc != SPTP_OK) return rc;
    if (chunks < 1 || chunks % P != 0 || (M > 0 && M % chunks != 0)) return SPTP_ERR_SHAPE;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return SPTP_ERR_SHAPE;
    const void* ptrs[] = {x, partials, gamma, qW1g, qW1u, qW2, out, resid_out, workspace};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SPTP_ERR_SHAPE;
    const void* sc[] = {sW1g, sW1u, sW2};
    for (const void* q : sc)
        if ((reinterpret_cast<uintptr_t>(q) & 15u) != 0) return SPTP_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return SPTP_ERR_SHAPE;
    const Fp8Layout lay = fp8_layout(M, d, F, P);
    if (ws_bytes < lay.total) return SPTP_ERR_WORKSPACE;
    const size_t act = static_cast<size_t>(M) * d * 2;
    const size_t out_bytes = act * P;
    const size_t wq = static_cast<size_t>(F) * d;
    const void* ins[] = {x, partials, gamma, qW1g, sW1g, qW1u, sW1u, qW2, sW2, workspace, resid_out};
    const size_t insz[] = {act, out_bytes, static_cast<size_t>(d) * 2, wq, static_cast<size_t>(F) * 4, wq,
                           static_cast<size_t>(F) * 4, wq, static_cast<size_t>(d) * P * 4, lay.total,
                           resid_out ? act : 0};
    for (int i = 0; i < 11; ++i)
        if (overlaps(out, out_bytes, ins[i], insz[i])) return SPTP_ERR_ALIAS;
    for (int i = 0; i < 9; ++i)
        if (overlaps(workspace, lay.total, ins[i], insz[i])) return SPTP_ERR_ALIAS;
    if (resid_out && resid_out != x) {
        for (int i = 0; i < 10; ++i)
            if (i != 0 && overlaps(resid_out, act, ins[i], insz[i])) return SPTP_ERR_ALIAS;
        if (overlaps(resid_out, act, x, act)) return SPTP_ERR_ALIAS;
    }
    if (M == 0) return SPTP_OK;
    DevInfo di;
    if ((rc = device_info(&di)) != SPTP_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if ((rc = reset_status(workspace, s)) != SPTP_OK) return rc;
    DeviceStatus* st = ws_status(workspace);
    void* y = mptr(workspace, lay.y);
    void* qy = mptr(workspace, lay.qy);
    float* sy = reinterpret_cast<float*>(mptr(workspace, lay.sy));
    void* sbuf = mptr(workspace, lay.s);
    void* qs = mptr(workspace, lay.qs);
    float* ss = reinterpret_cast<float*>(mptr(workspace, lay.ss));
    const int band = raster_band();
    const int f = F / P;

    // 1-3: partial sum, residual add, RMSNorm -> the bf16 activation y ...
    PrologueParams pp;
    std::memset(&pp, 0, sizeof(pp));
    pp.G = 1;
    pp.M = M;
    pp.d = d;
    pp.eps = eps;
    pp.gamma = gamma;
    pp.grp[0] = PrologueGroup{x, resid_out, y, 0, P};
    for (int p = 0; p < P; ++p) pp.src[p] = cptr(partials, static_cast<size_t>(p) * act);
    pp.status = st;
    pp.wait_limit_ns = kWaitLimitNs;
    // ... and the gate/up linear's quantisation of y per token, fused
    pp.q = qy;
    pp.qscale = sy;
    if ((rc = cuda_status(launch_prologue(pp, true, di.sms, s))) != SPTP_OK) return rc;
    // 4-6: (identity) gather + column-parallel E4M3 gate/up + SwiGLU
    if ((rc = gateup_e4m3(qy, sy, qW1g, sW1g, qW1u, sW1u, M, d, F, P, sbuf, st, band, di, s)) != SPTP_OK) return rc;
    // the down linear quantises s per token within each shard
    if ((rc = cuda_status(launch_quantize_rows_e4m3(sbuf, static_cast<long long>(P) * M, f, qs, ss, di.sms, s))) !=
        SPTP_OK)
        return rc;
    // 7: row-parallel E4M3 down projection, one partial per shard
    void* outs[kMaxGroups];
    for (int g = 0; g < P; ++g) outs[g] = mptr(out, static_cast<size_t>(g) * act);
    return down_e4m3(qs, ss, qW2, sW2, M, d, F, P, outs, st, band, di, s);
}

int sptp_prologue_e4m3(const void* x, const void* partials, const void* gamma, int M, int d, int P, float eps,
                       void* h_out, void* y_work, void* q_out, float* scale_out, void* cuda_stream) {
    if (!gamma || (M != 0 && (!x || !partials || !y_work || !q_out || !scale_out))) return SPTP_ERR_NULL;
    int rc = check_common(M, d, 8 * P, P, SPTP_BF16);
    if (rc != SPTP_OK) return rc;
    if (d % 16 != 0 || !(eps >= 0.f) || !std::isfinite(eps)) return SPTP_ERR_SHAPE;
    const void* ptrs[] = {x, partials, gamma, h_out, y_work, q_out, scale_out};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SPTP_ERR_SHAPE;
    const size_t act = static_cast<size_t>(M) * d * 2;
    const void* ins[] = {x, partials, gamma, h_out};
    const size_t insz[] = {act, act * P, static_cast<size_t>(d) * 2, h_out ? act : 0};
    void* outs[] = {y_work, q_out, scale_out};
    const size_t osz[] = {act, act / 2, static_cast<size_t>(M) * 4};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 4; ++i)
            if (overlaps(outs[o], osz[o], ins[i], insz[i])) return SPTP_ERR_ALIAS;
        for (int j = o + 1; j < 3; ++j)
            if (overlaps(outs[o], osz[o], outs[j], osz[j])) return SPTP_ERR_ALIAS;
    }
    if (h_out && h_out != x && (overlaps(h_out, act, partials, act * P) || overlaps(h_out, act, x, act)))
        return SPTP_ERR_ALIAS;
    if (M == 0) return SPTP_OK;
    DevInfo di;
    if ((rc = device_info(&di)) != SPTP_OK) return rc;
    PrologueParams pp;
    std::memset(&pp, 0, sizeof(pp));
    pp.G = 1;
    pp.M = M;
    pp.d = d;
    pp.eps = eps;
    pp.gamma = gamma;
    pp.grp[0] = PrologueGroup{x, h_out, y_work, 0, P};
    for (int p = 0; p < P; ++p) pp.src[p] = cptr(partials, static_cast<size_t>(p) * act);
    pp.status = nullptr;
    pp.wait_limit_ns = kWaitLimitNs;
    pp.q = q_out;
    pp.qscale = scale_out;
    return cuda_status(launch_prologue(pp, true, di.sms, static_cast<cudaStream_t>(cuda_stream)));
}

int sptp_gateup_swiglu_e4m3(const void* qy, const float* sy, const void* qW1g, const float* sW1g, const void* qW1u,
                            const float* sW1u, int M, int d, int F, int P, void* s_out, void* workspace,
                            size_t ws_bytes, void* cuda_stream) {
    if (!qW1g || !sW1g || !qW1u || !sW1u || !workspace || (M != 0 && (!qy || !sy || !s_out))) return SPTP_ERR_NULL;
    int rc = check_fp8(M, d, F, P);
    if (rc != SPTP_OK) return rc;
    const void* ptrs[] = {qy, sy, qW1g, sW1g, qW1u, sW1u, s_out, workspace};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SPTP_ERR_SHAPE;
    if (ws_bytes < SPTP_WS_HEADER_BYTES) return SPTP_ERR_WORKSPACE;
    const size_t sb = static_cast<size_t>(M) * F * 2, wq = static_cast<size_t>(F) * d;
    const void* ins[] = {qy, sy, qW1g, sW1g, qW1u, sW1u, workspace};
    const size_t insz[] = {static_cast<size_t>(M) * d, static_cast<size_t>(M) * 4, wq, static_cast<size_t>(F) * 4,
                           wq, static_cast<size_t>(F) * 4, SPTP_WS_HEADER_BYTES};
    for (int i = 0; i < 7; ++i)
        if (overlaps(s_out, sb, ins[i], insz[i])) return SPTP_ERR_ALIAS;
    if (M == 0) return SPTP_OK;
    DevInfo di;
    if ((rc = device_info(&di)) != SPTP_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if ((rc = reset_status(workspace, s)) != SPTP_OK) return rc;
    return gateup_e4m3(qy, sy, qW1g, sW1g, qW1u, sW1u, M, d, F, P, s_out, ws_status(workspace),
                       raster_band(), di, s);
}

int sptp_down_proj_e4m3(const void* qs, const float* ss, const void* qW2, const float* sW2, int M, int d, int F,
                        int P, void* out, void* workspace, size_t ws_bytes, void* cuda_stream) {
    if (!qW2 || !sW2 || !workspace || (M != 0 && (!qs || !ss || !out))) return SPTP_ERR_NULL;
    int rc = check_fp8(M, d, F, P);
    if (rc != SPTP_OK) return rc;
    const void* ptrs[] = {qs, ss, qW2, sW2, out, workspace};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return SPTP_ERR_SHAPE;
    if (ws_bytes < SPTP_WS_HEADER_BYTES) return SPTP_ERR_WORKSPACE;
    const size_t ob = static_cast<size_t>(P) * M * d * 2;
    const void* ins[] = {qs, ss, qW2, sW2, workspace};
    const size_t insz[] = {static_cast<size_t>(M) * F, static_cast<size_t>(M) * P * 4, static_cast<size_t>(F) * d,
                           static_cast<size_t>(d) * P * 4, SPTP_WS_HEADER_BYTES};
    for (int i = 0; i < 5; ++i)
        if (overlaps(out, ob, ins[i], insz[i])) return SPTP_ERR_ALIAS;
    if (M == 0) return SPTP_OK;
    DevInfo di;
    if ((rc = device_info(&di)) != SPTP_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if ((rc = reset_status(workspace, s)) != SPTP_OK) return rc;
    void* outs[kMaxGroups];
    for (int g = 0; g < P; ++g) outs[g] = mptr(out, static_cast<size_t>(g) * M * d * 2);
    return down_e4m3(qs, ss, qW2, sW2, M, d, F, P, outs, ws_status(workspace), raster_band(), di, s);
}

}  // extern "C"
