// Coalesced output stores for the GEMM epilogues.  An epilogue warp reads
// TMEM lanes: each lane owns one output row, so a direct 16-byte store per
// lane touches 32 different rows (32 L2 requests of half a sector each).  The
// warp instead writes its 32 x 64 block (bf16) to a shared-memory buffer,
// one row per lane, and stores it back with eight lanes per 128-byte row
// segment: four whole rows per store instruction, an eighth of the L2
// requests.  Short-K tiles, whose epilogue is close to their MMA time, are
// where this pays.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "sptp_ptx.cuh"

namespace sptp {

// 32 rows of 128 bytes at a 144-byte pitch: with the 16-byte pad both the
// row-per-lane writes and the segment-per-lane reads are conflict-free.
constexpr int kOutPitch = 144;
constexpr int kOutWarpBytes = 32 * kOutPitch;

// Stores the warp's block: lane l holds row (row0 + l)'s 64 packed columns
// [col0, col0 + 64) in pk.  out points at element [0][0] of a matrix with
// row pitch ldo (elements); rows at or past M and columns at or past N are
// not stored.  With split_w > 0 column c goes instead to split_out +
// (c / split_w) * split_stride as a [M][split_w] matrix (split_w a multiple
// of 8, so a 16-byte vector never straddles two blocks).  STREAM selects
// evict-first stores for outputs nothing in the same launch reads.
// limit: elements of the destination buffer from out (split_out with
// split_w > 0); a checked build stores nothing outside it.
template <bool STREAM>
__device__ __forceinline__ void store_block_staged(uint8_t* wbuf, const uint32_t (&pk)[32], int lane,
                                                   __nv_bfloat16* out, long long ldo, __nv_bfloat16* split_out,
                                                   int split_w, long long split_stride, int row0, int M, int col0,
                                                   int N, long long limit, DeviceStatus* st,
                                                   volatile int* abort_flag) {
    uint8_t* mine = wbuf + lane * kOutPitch;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(mine + 16 * j) = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    __syncwarp();
    const int seg = lane & 7;
    const int col = col0 + 8 * seg;
    long long first = col;  // element offset of the lane's column in row 0
    long long pitch = ldo;
    __nv_bfloat16* ref = out;
    if (split_w > 0) {
        const int blk = col / split_w;
        first = blk * split_stride + (col - blk * split_w);
        pitch = split_w;
        ref = split_out;
    }
    __nv_bfloat16* base = ref + first;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 4 * i + (lane >> 3);
        const uint4 v = *reinterpret_cast<const uint4*>(wbuf + r * kOutPitch + 16 * seg);
        const int row = row0 + r;
        if (row < M && col < N &&
            checked_range(first + static_cast<long long>(row) * pitch, 8, limit, st, abort_flag, kWhereBoundsStore)) {
            uint4* dst = reinterpret_cast<uint4*>(base + static_cast<long long>(row) * pitch);
            if constexpr (STREAM)
                __stcs(dst, v);
            else
                *dst = v;
        }
    }
    __syncwarp();  // every lane has read the block before the buffer is rewritten
}

}  // namespace sptp
