// GEMM launches shared by the C-ABI entry points: the tensor maps, tile
// counts and raster band of each grouped GEMM (gate/up + SwiGLU, down,
// column-parallel store, and their E4M3 forms).  The kernels are in
// gemm_tc.cu (tcgen05 CTA pairs, bf16 and E4M3) and gemm_simt.cu (fp32).
#include <cstring>

#include "launch.h"

namespace sptp {

// Raster band: the GEMMs walk the m-tiles of 4096 rows against each B panel
// before moving to the next panel, so the band's A tiles stay in L2 while the
// weights are streamed about M/4096 times.  (Measured on the 8192 x 4096 x
// 14336 boundary, end to end: bands of 1024 / 2048 / 4096 / 8192 rows gave
// 1589 / 1644 / 1658 / 1602 TFLOP/s; at M=65536 with 8192-row chunks, a band
// of one chunk gave 1576-1582 and 4096 rows 1599-1601.)  The band does not
// follow the sequence chunks: in the multi-launch paths every chunk's rows
// are ready before the GEMM starts.
constexpr int kBandRows = 4096;

int raster_band() { return kBandRows / kBM; }

// Raster band of the down GEMM (rows).  A build option (-DSPTP_DOWN_BAND_ROWS)
// for measuring the effect of the band on the down GEMM's DRAM traffic.
#ifndef SPTP_DOWN_BAND_ROWS
#define SPTP_DOWN_BAND_ROWS 4096
#endif

int down_raster_band() { return SPTP_DOWN_BAND_ROWS / kBM; }

// Gate/up + SwiGLU for P groups: s_g = silu(A_g W1g[F_g]^T) * (A_g W1u[F_g]^T).
int gateup(const void* const* A, const void* W1g, const void* W1u, int M, int d, int F, int P, int dtype,
           void* s_out, DeviceStatus* st, int band, const DevInfo& di, cudaStream_t s) {
    const int f = F / P;
    const size_t es = esize(dtype);
    if (M == 0) return SPTP_OK;
    if (dtype == SPTP_BF16) {
        TcGemmParams p;
        std::memset(&p, 0, sizeof(p));
        for (int g = 0; g < P; ++g) {
            const size_t woff = static_cast<size_t>(g) * f * d * es;
            if (!encode_map_bf16(&p.mapA[g], A[g], d, M, static_cast<uint64_t>(d) * es, kBK, kBM) ||
                !encode_map_bf16(&p.mapB0[g], cptr(W1g, woff), d, f, static_cast<uint64_t>(d) * es, kBK,
                                 kBNSwiGLU) ||
                !encode_map_bf16(&p.mapB1[g], cptr(W1u, woff), d, f, static_cast<uint64_t>(d) * es, kBK,
                                 kBNSwiGLU))
                return SPTP_ERR_CUDA;
            p.out[g] = mptr(s_out, static_cast<size_t>(g) * M * f * es);
        }
        p.ldo = f;
        p.M = M;
        p.N = f;
        p.K = d;
        p.G = P;
        p.mt = (M + 2 * kBM - 1) / (2 * kBM);
        p.nt = (f + kBNSwiGLU - 1) / kBNSwiGLU;
        p.nk = (d + kBK - 1) / kBK;
        band = (band + 1) / 2;
        p.band = band < 1 ? 1 : (band > p.mt ? p.mt : band);
        p.status = st;
        p.wait_limit_ns = kWaitLimitNs;
        return cuda_status(launch_tc_gemm_pair(p, Epi::kSwiGLU, di.sms, s));
    }
    SimtGemmParams p;
    std::memset(&p, 0, sizeof(p));
    for (int g = 0; g < P; ++g) {
        const size_t woff = static_cast<size_t>(g) * f * d;
        p.A[g] = static_cast<const float*>(A[g]);
        p.B0[g] = static_cast<const float*>(W1g) + woff;
        p.B1[g] = static_cast<const float*>(W1u) + woff;
        p.C[g] = static_cast<float*>(s_out) + static_cast<size_t>(g) * M * f;
    }
    p.lda = d;
    p.ldb = d;
    p.ldc = f;
    p.M = M;
    p.N = f;
    p.K = d;
    p.G = P;
    return cuda_status(launch_simt_gemm(p, Epi::kSwiGLU, s));
}

// Down projection for P groups: out_g = s_g W2[:, F_g]^T.
int down(const void* s_in, const void* W2, int M, int d, int F, int P, int dtype, void* const* out,
         DeviceStatus* st, int band, const DevInfo& di, cudaStream_t s) {
    const int f = F / P;
    const size_t es = esize(dtype);
    if (M == 0) return SPTP_OK;
    if (dtype == SPTP_BF16) {
        // a CTA pair stages each B tile as two 128-row halves
        const uint32_t bbox = kBNStore / 2;
        TcGemmParams p;
        std::memset(&p, 0, sizeof(p));
        for (int g = 0; g < P; ++g) {
            if (!encode_map_bf16(&p.mapA[g], cptr(s_in, static_cast<size_t>(g) * M * f * es), f, M,
                                 static_cast<uint64_t>(f) * es, kBK, kBM) ||
                !encode_map_bf16(&p.mapB0[g], cptr(W2, static_cast<size_t>(g) * f * es), f, d,
                                 static_cast<uint64_t>(F) * es, kBK, bbox))
                return SPTP_ERR_CUDA;
            p.out[g] = out[g];
        }
        p.ldo = d;
        p.M = M;
        p.N = d;
        p.K = f;
        p.G = P;
        p.mt = (M + 2 * kBM - 1) / (2 * kBM);
        p.nt = (d + kBNStore - 1) / kBNStore;
        p.nk = (f + kBK - 1) / kBK;
        band = (band + 1) / 2;
        p.band = band < 1 ? 1 : (band > p.mt ? p.mt : band);
        p.status = st;
        p.wait_limit_ns = kWaitLimitNs;
        return cuda_status(launch_tc_gemm_pair(p, Epi::kStore, di.sms, s));
    }
    SimtGemmParams p;
    std::memset(&p, 0, sizeof(p));
    for (int g = 0; g < P; ++g) {
        p.A[g] = static_cast<const float*>(s_in) + static_cast<size_t>(g) * M * f;
        p.B0[g] = static_cast<const float*>(W2) + static_cast<size_t>(g) * f;
        p.B1[g] = nullptr;
        p.C[g] = static_cast<float*>(out[g]);
    }
    p.lda = f;
    p.ldb = F;
    p.ldc = d;
    p.M = M;
    p.N = d;
    p.K = f;
    p.G = P;
    return cuda_status(launch_simt_gemm(p, Epi::kStore, s));
}

// Column-parallel projection for P groups with a plain bf16/fp32 store:
// out_g [M][N/P] = A W[g*N/P .. (g+1)*N/P)^T, W [N][K] row-major.
int colpar_store(const void* A, const void* W, int M, int K, int N, int P, int dtype, void* out, DeviceStatus* st,
                 int band, const DevInfo& di, cudaStream_t s) {
    const int n = N / P;
    const size_t es = esize(dtype);
    if (M == 0) return SPTP_OK;
    if (dtype == SPTP_BF16) {
        const int bm = 2 * kBM;
        const uint32_t bbox = kBNStore / 2;
        TcGemmParams p;
        std::memset(&p, 0, sizeof(p));
        if (P > 1 && n % kBNStore != 0) {
            // Every shard reads the same A, so the P shards run as one GEMM
            // over all N rows of W, each 8-column vector stored to its
            // shard's [M][N/P] block: no half-empty last tile per shard
            // (N/P = 1152 fills 4.5 tiles of 256).
            if (!encode_map_bf16(&p.mapA[0], A, K, M, static_cast<uint64_t>(K) * es, kBK, kBM) ||
                !encode_map_bf16(&p.mapB0[0], W, K, N, static_cast<uint64_t>(K) * es, kBK, bbox))
                return SPTP_ERR_CUDA;
            p.out[0] = out;
            p.split_w = n;
            p.split_stride = static_cast<long long>(M) * n;
            p.ldo = n;
            p.M = M;
            p.N = N;
            p.K = K;
            p.G = 1;
            p.mt = (M + bm - 1) / bm;
            p.nt = (N + kBNStore - 1) / kBNStore;
            p.nk = (K + kBK - 1) / kBK;
            band = (band + 1) / 2;
            p.band = band < 1 ? 1 : (band > p.mt ? p.mt : band);
            p.status = st;
            p.wait_limit_ns = kWaitLimitNs;
            return cuda_status(launch_tc_gemm_pair(p, Epi::kStore, di.sms, s));
        }
        for (int g = 0; g < P; ++g) {
            if (!encode_map_bf16(&p.mapA[g], A, K, M, static_cast<uint64_t>(K) * es, kBK, kBM) ||
                !encode_map_bf16(&p.mapB0[g], cptr(W, static_cast<size_t>(g) * n * K * es), K, n,
                                 static_cast<uint64_t>(K) * es, kBK, bbox))
                return SPTP_ERR_CUDA;
            p.out[g] = mptr(out, static_cast<size_t>(g) * M * n * es);
        }
        p.ldo = n;
        p.M = M;
        p.N = n;
        p.K = K;
        p.G = P;
        p.mt = (M + bm - 1) / bm;
        p.nt = (n + kBNStore - 1) / kBNStore;
        p.nk = (K + kBK - 1) / kBK;
        band = (band + 1) / 2;
        p.band = band < 1 ? 1 : (band > p.mt ? p.mt : band);
        p.status = st;
        p.wait_limit_ns = kWaitLimitNs;
        return cuda_status(launch_tc_gemm_pair(p, Epi::kStore, di.sms, s));
    }
    SimtGemmParams p;
    std::memset(&p, 0, sizeof(p));
    for (int g = 0; g < P; ++g) {
        p.A[g] = static_cast<const float*>(A);
        p.B0[g] = static_cast<const float*>(W) + static_cast<size_t>(g) * n * K;
        p.B1[g] = nullptr;
        p.C[g] = static_cast<float*>(out) + static_cast<size_t>(g) * M * n;
    }
    p.lda = K;
    p.ldb = K;
    p.ldc = n;
    p.M = M;
    p.N = n;
    p.K = K;
    p.G = P;
    return cuda_status(launch_simt_gemm(p, Epi::kStore, s));
}

// E4M3 gate/up + SwiGLU for P groups on the CTA-pair tcgen05 GEMM.
int gateup_e4m3(const void* qy, const float* sy, const void* qW1g, const float* sW1g, const void* qW1u,
                const float* sW1u, int M, int d, int F, int P, void* s_out, DeviceStatus* st, int band,
                const DevInfo& di, cudaStream_t s) {
    const int f = F / P;
    if (M == 0) return SPTP_OK;
    TcGemmParams p;
    std::memset(&p, 0, sizeof(p));
    for (int g = 0; g < P; ++g) {
        const size_t woff = static_cast<size_t>(g) * f * d;
        if (!encode_map_u8(&p.mapA[g], qy, d, M, d, kBK8, kBM) ||
            !encode_map_u8(&p.mapB0[g], cptr(qW1g, woff), d, f, d, kBK8, kBNSwiGLU) ||
            !encode_map_u8(&p.mapB1[g], cptr(qW1u, woff), d, f, d, kBK8, kBNSwiGLU))
            return SPTP_ERR_CUDA;
        p.out[g] = mptr(s_out, static_cast<size_t>(g) * M * f * 2);
        p.row_scale[g] = sy;
        p.col_scale0[g] = sW1g + static_cast<size_t>(g) * f;
        p.col_scale1[g] = sW1u + static_cast<size_t>(g) * f;
    }
    p.col_scale_stride = 1;
    p.ldo = f;
    p.M = M;
    p.N = f;
    p.K = d;
    p.G = P;
    p.mt = (M + 2 * kBM - 1) / (2 * kBM);
    p.nt = (f + kBNSwiGLU - 1) / kBNSwiGLU;
    p.nk = (d + kBK8 - 1) / kBK8;
    band = (band + 1) / 2;
    p.band = band < 1 ? 1 : (band > p.mt ? p.mt : band);
    p.status = st;
    p.wait_limit_ns = kWaitLimitNs;
    return cuda_status(launch_tc_gemm_pair_e4m3(p, Epi::kSwiGLU, di.sms, s));
}

// E4M3 down projection for P groups: out_g = (qs_g qW2[:, F_g]^T) ss_g sW2[:, g].
int down_e4m3(const void* qs, const float* ss, const void* qW2, const float* sW2, int M, int d, int F, int P,
              void* const* out, DeviceStatus* st, int band, const DevInfo& di, cudaStream_t s) {
    const int f = F / P;
    if (M == 0) return SPTP_OK;
    TcGemmParams p;
    std::memset(&p, 0, sizeof(p));
    for (int g = 0; g < P; ++g) {
        if (!encode_map_u8(&p.mapA[g], cptr(qs, static_cast<size_t>(g) * M * f), f, M, f, kBK8, kBM) ||
            !encode_map_u8(&p.mapB0[g], cptr(qW2, static_cast<size_t>(g) * f), f, d, F, kBK8, kBNStore / 2))
            return SPTP_ERR_CUDA;
        p.out[g] = out[g];
        p.row_scale[g] = ss + static_cast<size_t>(g) * M;
        p.col_scale0[g] = sW2 + g;
    }
    p.col_scale_stride = P;
    p.ldo = d;
    p.M = M;
    p.N = d;
    p.K = f;
    p.G = P;
    p.mt = (M + 2 * kBM - 1) / (2 * kBM);
    p.nt = (d + kBNStore - 1) / kBNStore;
    p.nk = (f + kBK8 - 1) / kBK8;
    band = (band + 1) / 2;
    p.band = band < 1 ? 1 : (band > p.mt ? p.mt : band);
    p.status = st;
    p.wait_limit_ns = kWaitLimitNs;
    return cuda_status(launch_tc_gemm_pair_e4m3(p, Epi::kStore, di.sms, s));
}

}  // namespace sptp
