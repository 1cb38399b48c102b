// attn_common.cuh — tile geometry and operand descriptors shared by the
// attention kernels.
//
// Layout in HBM: Q, K, V, out, dout, dQ, dK, dV are [B, H, T, d_h] bf16,
// row-major; a tile is 128 consecutive rows of one (b, h), so the kernels view
// each tensor as a 2-D array [B*H*T, d_h] and address tile (b, h, X) at row
// (b*H + h)*T + 128*X.
//
// Layout in shared memory (all written by TMA or by the kernels themselves):
// a [128 x d_h] bf16 tile is stored as d_h/CHUNK column chunks of [128 x CHUNK]
// elements, each row of a chunk one swizzle span (128 B for d_h >= 64, 64 B for
// d_h = 32), in the canonical swizzled form the tcgen05 descriptors expect.
// Square [128 x 128] operand tiles the kernels write themselves (P, dS, G) use
// two 64-column chunks with the 128-byte swizzle.  Such a tile serves both as
// a K-major operand (rows = M or N, columns = K) and as an MN-major operand
// (columns = M or N, rows = K).
#pragma once

#include "ptx.cuh"

namespace saf {

template <int D>
struct TileGeom {
  static_assert(D == 32 || D == 64 || D == 128, "d_h must be 32, 64 or 128");
  static constexpr int ROWS = 128;
  static constexpr int SWZ = (D >= 64) ? 128 : 64;     // bytes per swizzled row
  static constexpr int CHUNK = SWZ / 2;                // bf16 columns per chunk
  static constexpr int NCHUNK = D / CHUNK;             // 1 or 2
  static constexpr int CHUNK_BYTES = ROWS * SWZ;
  static constexpr int TILE_BYTES = ROWS * D * 2;
  static constexpr uint32_t LAYOUT = swizzle_layout_code(SWZ);
  static constexpr int KSTEPS = D / 16;                // MMA k-steps over d_h

  // K-major operand over d_h (Q, K, dO as [rows x d_h]): k-step kk of 16.
  __device__ static __forceinline__ uint64_t kmajor_desc(uint32_t tile_saddr, int kk) {
    constexpr int per_chunk = CHUNK / 16;
    const uint32_t a = tile_saddr + (uint32_t)(kk / per_chunk) * CHUNK_BYTES +
                       (uint32_t)(kk % per_chunk) * 32u;
    return sdesc(a, 16u, 8u * SWZ, LAYOUT);
  }
  // MN-major operand: a [128 rows (K) x d_h (N)] tile (V, dO, Q, K used as
  // the N side of a product over rows): k-step kk covers rows 16kk..16kk+15.
  __device__ static __forceinline__ uint64_t mnmajor_desc(uint32_t tile_saddr, int kk) {
    const uint32_t a = tile_saddr + (uint32_t)kk * 16u * SWZ;
    return sdesc(a, (uint32_t)CHUNK_BYTES, 8u * SWZ, LAYOUT);
  }
};

// Square [128 x 128] bf16 tile written by the kernels (two 64-col chunks,
// 128-byte swizzle).
struct SqTile {
  static constexpr int BYTES = 128 * 128 * 2;
  static constexpr int CHUNK_BYTES = 128 * 128;
  // As K-major operand (rows = M/N, cols = K): k-step kk of 16 columns.
  __device__ static __forceinline__ uint64_t kmajor_desc(uint32_t saddr, int kk) {
    const uint32_t a = saddr + (uint32_t)(kk >> 2) * CHUNK_BYTES + (uint32_t)(kk & 3) * 32u;
    return sdesc(a, 16u, 1024u, kLayoutSw128);
  }
  // As MN-major operand (cols = M/N, rows = K): k-step kk covers rows 16kk..
  __device__ static __forceinline__ uint64_t mnmajor_desc(uint32_t saddr, int kk) {
    const uint32_t a = saddr + (uint32_t)kk * 16u * 128u;
    return sdesc(a, (uint32_t)CHUNK_BYTES, 1024u, kLayoutSw128);
  }
  // Shared address of 16-byte unit u (0..15) of row r.
  __device__ static __forceinline__ uint32_t unit_addr(uint32_t saddr, uint32_t r, uint32_t u) {
    return saddr + (u >> 3) * CHUNK_BYTES + sw128_offset(r, u & 7u);
  }
};

// Item of round k for CTA `cta` of a persistent grid of `grid` CTAs: even
// rounds run forwards, odd rounds backwards, so that with items sorted
// longest first the CTA that drew one of the longest items in one round
// draws one of the shortest in the next.  Once an index is past the end,
// every later round's is too.
__device__ __forceinline__ int snake_item(int k, int cta, int grid) {
  return (k & 1) ? (k + 1) * grid - 1 - cta : k * grid + cta;
}

}  // namespace saf
