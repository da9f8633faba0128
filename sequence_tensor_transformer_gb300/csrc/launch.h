// GEMM launch helpers shared by the C-ABI entry points (launch.cu): tile
// shapes, the raster band and the grouped GEMM launches of the boundary.
// Sizes are validated by the callers.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "sptp.h"
#include "sptp_internal.h"

namespace sptp {

constexpr int kBM = 128, kBNSwiGLU = 128, kBNStore = 256, kBK = 64;
constexpr int kBK8 = 128;  // E4M3 elements per 128-byte swizzle row

struct DevInfo {
    int sms = 0;
    int major = 0, minor = 0;
};

inline size_t esize(int dtype) { return dtype == SPTP_BF16 ? 2 : 4; }
inline const char* cptr(const void* base, size_t off_bytes) { return static_cast<const char*>(base) + off_bytes; }
inline char* mptr(void* base, size_t off_bytes) { return static_cast<char*>(base) + off_bytes; }
inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? SPTP_OK : SPTP_ERR_CUDA; }

// m-tiles (128 rows) per raster band, of the gate/up and of the down GEMM
int raster_band();
int down_raster_band();

// Gate/up + SwiGLU for P groups: s_g = silu(A_g W1g[F_g]^T) * (A_g W1u[F_g]^T);
// s_out [P][M][F/P].
int gateup(const void* const* A, const void* W1g, const void* W1u, int M, int d, int F, int P, int dtype,
           void* s_out, DeviceStatus* st, int band, const DevInfo& di, cudaStream_t s);
// Down projection for P groups: out_g = s_g W2[:, F_g]^T.
int down(const void* s_in, const void* W2, int M, int d, int F, int P, int dtype, void* const* out,
         DeviceStatus* st, int band, const DevInfo& di, cudaStream_t s);
// Column-parallel store GEMM: out_g [M][N/P] = A W[g N/P .. (g+1) N/P)^T.
int colpar_store(const void* A, const void* W, int M, int K, int N, int P, int dtype, void* out, DeviceStatus* st,
                 int band, const DevInfo& di, cudaStream_t s);
// The E4M3 forms of gate/up and down (row scales of A, column scales of B).
int gateup_e4m3(const void* qy, const float* sy, const void* qW1g, const float* sW1g, const void* qW1u,
                const float* sW1u, int M, int d, int F, int P, void* s_out, DeviceStatus* st, int band,
                const DevInfo& di, cudaStream_t s);
int down_e4m3(const void* qs, const float* ss, const void* qW2, const float* sW2, int M, int d, int F, int P,
              void* const* out, DeviceStatus* st, int band, const DevInfo& di, cudaStream_t s);

}  // namespace sptp
