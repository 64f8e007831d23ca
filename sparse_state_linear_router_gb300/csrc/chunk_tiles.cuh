// chunk_tiles.cuh -- helpers of the chunked tensor-core kernels that stage
// 128-row bf16 operand tiles (128-byte swizzle, two 64-column atoms per
// 8-row group) and write per-row results through a warp's shared patch.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "sse_internal.cuh"
#include "umma.cuh"

namespace sse {
namespace tiles {

using umma::smem_u32;
using umma::sw128_offset;

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
// byte offset of element (row, col) of a 128-row bf16 tile of up to 128
// columns: two 64-column atoms per 8-row group, 128-byte swizzle
__device__ __forceinline__ uint32_t toff(int row, int col) { return sw128_offset(row, col, 2); }

// 16-byte asynchronous copies into shared memory (zero-filled when !valid:
// nothing is read there); the caller waits with cp_async_wait_all().
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// The 128 rows tok[0..127] of NT [T * H, W] bf16 tensors (W = 64 or 128) into
// their swizzled tiles by 16-byte asynchronous copies, zero-filled for token
// -1, by a CTA of exactly 256 threads; the caller waits with
// cp_async_wait_all().  Thread x copies piece x % (W / 8) of rows
// x / (W / 8) + (256 / (W / 8)) i: one token lookup per row serves all NT
// tensors, and the tile offsets of a thread's rows step by whole 8-row groups
// (the swizzle of row r depends on r % 8 only), so the pass is a few
// instructions per copy.
template <int W, int NT>
__device__ __forceinline__ void stage_rows_n(unsigned char *const (&tiles)[NT], const __nv_bfloat16 *const (&srcs)[NT],
                                             const int *tok, int H, int h) {
    static_assert(W == 64 || W == 128, "row width");
    constexpr int kPieces = W / 8, kRowsPerPass = 256 / kPieces, kPasses = kChunkRows / kRowsPerPass;
    constexpr uint32_t kStep = (kRowsPerPass / 8) * 2048;  // bytes between a thread's rows
    const int r0 = threadIdx.x / kPieces, c8 = threadIdx.x % kPieces;
    const uint32_t o0 = toff(r0, c8 * 8);
    int64_t src[kPasses];
    bool ok[kPasses];
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
        const int t = tok[r0 + kRowsPerPass * i];
        ok[i] = t >= 0;
        src[i] = ok[i] ? ((int64_t)t * H + h) * W + c8 * 8 : 0;
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const uint32_t d = smem_u32(tiles[n]) + o0;
#pragma unroll
        for (int i = 0; i < kPasses; ++i) cp_async16(d + kStep * i, srcs[n] + src[i], ok[i]);
    }
}

constexpr int kPatchStride = 20;  // floats per row of a warp's store patch (16 used; rows stay 16-byte aligned)

// A 32-row x 16-column block of fp32 values, one row per lane, goes out through
// the warp's shared patch: each store instruction then writes 8 rows x 64
// contiguous bytes instead of 32 rows x 16.  Row (lane / 4 + 8 kk) of the block
// lands at base + sr[kk] * width + col0 (skipped when sr[kk] < 0).
__device__ __forceinline__ void warp_put16(float *patch, int lane, const float (&v)[16], float *base, int width,
                                           int col0, const int64_t (&sr)[4]) {
    float4 *pr = reinterpret_cast<float4 *>(patch + lane * kPatchStride);
#pragma unroll
    for (int i = 0; i < 4; ++i) pr[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    __syncwarp();
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int rr = (lane >> 2) + 8 * kk, qd = lane & 3;
        if (sr[kk] >= 0)
            *reinterpret_cast<float4 *>(base + sr[kk] * width + col0 + 4 * qd) =
                *reinterpret_cast<const float4 *>(patch + rr * kPatchStride + 4 * qd);
    }
    __syncwarp();
}

// A 32-row x 32-column block of bf16 values, one row per lane (16 packed
// words), goes out through the same patch: 64 contiguous bytes per row, and
// each store instruction writes 8 rows.  Row (lane / 4 + 8 kk) of the block
// lands at base + sr[kk] * width + col0 (skipped when sr[kk] < 0).
__device__ __forceinline__ void warp_put32_bf16(float *patch, int lane, const uint32_t (&w)[16], __nv_bfloat16 *base,
                                                int width, int col0, const int64_t (&sr)[4]) {
    uint4 *pr = reinterpret_cast<uint4 *>(patch + lane * kPatchStride);
#pragma unroll
    for (int i = 0; i < 4; ++i) pr[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    __syncwarp();
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int rr = (lane >> 2) + 8 * kk, qd = lane & 3;
        if (sr[kk] >= 0)
            *reinterpret_cast<uint4 *>(base + sr[kk] * width + col0 + 8 * qd) =
                *reinterpret_cast<const uint4 *>(patch + rr * kPatchStride + 4 * qd);
    }
    __syncwarp();
}

}  // namespace tiles
}  // namespace sse
