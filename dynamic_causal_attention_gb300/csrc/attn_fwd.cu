// attn_fwd.cu — forward of the SAF hybrid causal attention layer, and the
// static-head engine that the backward reuses for dV.
//
// Method ("When Can Attention Heads Be Statically Defined?", close-reading
// notes): a dynamic head computes softmax_causal(Q K^T / sqrt(d_h)) V (§1); a
// frozen head mixes V with P(i,j) = exp(alpha(j) + rho(i-j)) / Z(i), j <= i
// (Eq. (3)), which the fused kernel rebuilds tile by tile from alpha, rho and
// Z and multiplies by V, without any Q/K work (§3.3, App. D.2, Fig. 2).
//
// Kernels
//   static_prep_kernel  (K1) per static head: the generator tables and
//                       log Z(i).  Because alpha/rho are shared by the batch,
//                       this runs once per head, not once per sequence.
//   hybrid_fwd_kernel   (K2) one persistent launch, one CTA per SM, over a
//                       longest-first list of work items:
//     dynamic item (b, h, I): Q tile I against key tiles J = 0..I; S = Q K^T
//       and O += P V run on tcgen05 with fp32 accumulators in TMEM; online
//       softmax in registers, one query row per thread.
//     static item (h, I, batch group): for J = 0..I a generated tile G[I,J]
//       (bf16, in shared memory) feeds one MMA per sequence of the group, so
//       one generated tile serves the whole batch.
//
// Factored static generator.  With a(j) = exp(alpha(j) - max alpha) and
// r(d) = exp(rho(d) - max rho), P(i,j) = a(j) r(i-j) / Z'(i) where
// Z'(i) = sum_{k<=i} a(k) r(i-k): the shift cancels between numerator and
// Z.  A tile element is then two multiplies, no exponential.  When
// range(alpha) + range(rho) > 80 the products could underflow in fp32, and
// the head falls back to the exact form exp2(alpha2(j) + rho2(i-j) - log2 Z(i)).
//
// Warp roles in K2 (384 threads): warp 0 issues TMA copies, warp 1 issues
// the S = Q K^T MMAs and warp 3 the P V MMAs (one lane each), warp 2 owns the
// TMEM allocation, warps 4..11 are two compute warpgroups (softmax / tile generation / epilogue):
// each tile row belongs to one thread of each, which split its 128 key
// columns and exchange row maxima and sums through shared memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attn_common.cuh"
#include "attn_kernels.h"
#include "internal.h"

namespace saf {

// ============================================================ K1: static prep
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kMaxFactoredRange = 80.0f;

__device__ __forceinline__ void block_minmax(float& mx, float& mn, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  __syncthreads();
  if (lane == 0) {
    red[warp] = mx;
    red[32 + warp] = mn;
  }
  __syncthreads();
  mx = red[0];
  mn = red[32];
  for (int w = 1; w < nw; ++w) {
    mx = fmaxf(mx, red[w]);
    mn = fminf(mn, red[32 + w]);
  }
}

// grid (T / kPrepRows, n_static), 256 threads (8 warps), dynamic smem 2 * T + 8
// floats.  Each block scans alpha/rho for their finite ranges and picks the
// mode.  Factored heads: the block writes its kPrepRows entries of the tables and,
// block 0, the head's shift max alpha + max rho.  Exact heads: each warp
// also forms log Z of kPrepRows / 8 rows by an online log-sum-exp, its 32 lanes
// splitting the causal sum, merged across lanes in a fixed order.
constexpr int kPrepRows = 128;  // rows of a head per block (T is a multiple of 128)

__global__ void __launch_bounds__(256) static_prep_kernel(StaticPrep p) {
  extern __shared__ float sh[];
  __shared__ float red[64];
  const int T = p.T, hs = blockIdx.y, h = p.heads[hs];
  const int row0 = blockIdx.x * kPrepRows;
  const int nload = row0 + kPrepRows;  // entries 0 .. row0 + kPrepRows - 1 are needed
  float* sa = sh;
  float* sr = sh + T + 8;  // sr[-8 .. -1] = 0: the last stride reads past d = 0
  const float* alpha = p.alpha + (size_t)h * T;
  const float* rho = p.rho + (size_t)h * T;
  // finite max/min of alpha and rho over the whole head (every block agrees)
  float amax = -INFINITY, amin = INFINITY, rmax = -INFINITY, rmin = INFINITY;
  // 16-byte loads, four per thread in flight (T is a multiple of 128)
  const float4* alpha4 = reinterpret_cast<const float4*>(alpha);
  const float4* rho4 = reinterpret_cast<const float4*>(rho);
#pragma unroll 4
  for (int t4 = threadIdx.x; t4 < T / 4; t4 += blockDim.x) {
    const float4 a4 = alpha4[t4], r4 = rho4[t4];
    const float av[4] = {a4.x, a4.y, a4.z, a4.w};
    const float rv[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int t = 4 * t4 + e;
      if (t < nload) {
        sa[t] = av[e];
        sr[t] = rv[e];
      }
      if (isfinite(av[e])) { amax = fmaxf(amax, av[e]); amin = fminf(amin, av[e]); }
      if (isfinite(rv[e])) { rmax = fmaxf(rmax, rv[e]); rmin = fminf(rmin, rv[e]); }
    }
  }
  block_minmax(amax, amin, red);
  block_minmax(rmax, rmin, red);
  const bool all_masked = !(amax > -INFINITY) || !(rmax > -INFINITY);
  const bool exact = !all_masked && ((amax - amin) + (rmax - rmin) > kMaxFactoredRange);
  float* a_tab = p.a_tab + (size_t)hs * T;
  float* r_tab = p.r_tab + (size_t)hs * (T + 128);
  float* row_tab = p.row_tab + (size_t)hs * T;
  float* logZ = p.logZ + (size_t)hs * T;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    p.mode[hs] = exact ? 1 : 0;
    p.shift[hs] = (exact || all_masked) ? 0.f : amax + rmax;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  if (!exact) {
    // a = exp(alpha - max), r = exp(rho - max) for this block's kPrepRows entries.
    // Z'(i) is not formed here: the forward sums it from its own tiles and
    // the backward reads it back from the forward's lse.
    __syncthreads();
    for (int t = threadIdx.x; t < kPrepRows; t += blockDim.x) {
      a_tab[row0 + t] = all_masked ? 0.f : expf(sa[row0 + t] - amax);
      r_tab[127 + row0 + t] = all_masked ? 0.f : expf(sr[row0 + t] - rmax);
    }
    if (blockIdx.x == 0 && threadIdx.x < 127) r_tab[threadIdx.x] = 0.f;
    if (blockIdx.x == 0 && threadIdx.x == 127) r_tab[T + 127] = 0.f;
  } else {
    __syncthreads();
    for (int m = 0; m < kPrepRows / 8; ++m) {
      const int i = row0 + warp * (kPrepRows / 8) + m;
      // per-lane online log-sum-exp, then a fixed-order merge across lanes
      float mx = -INFINITY, sm = 0.f;
      for (int k = lane; k <= i; k += 32) {
        const float t = sa[k] + sr[i - k];
        if (t > mx) {
          sm = sm * expf(mx - t) + 1.f;
          mx = t;
        } else if (t > -INFINITY) {
          sm += expf(t - mx);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, mx, o);
        const float so = __shfl_xor_sync(0xffffffffu, sm, o);
        const float mn = fmaxf(mx, mo);
        if (mn > -INFINITY) {
          sm = sm * expf(mx - mn) + so * expf(mo - mn);
          mx = mn;
        }
      }
      if (lane == 0) {
        const float lz = (mx > -INFINITY) ? mx + logf(sm) : -INFINITY;
        logZ[i] = lz;
        row_tab[i] = (mx > -INFINITY) ? -lz * kLog2e : -INFINITY;
      }
    }
    for (int t = threadIdx.x; t < kPrepRows; t += blockDim.x) {
      a_tab[row0 + t] = sa[row0 + t] * kLog2e;
      r_tab[127 + row0 + t] = sr[row0 + t] * kLog2e;
    }
    if (blockIdx.x == 0 && threadIdx.x < 127) r_tab[threadIdx.x] = -INFINITY;
    if (blockIdx.x == 0 && threadIdx.x == 127) r_tab[T + 127] = -INFINITY;
  }
}

__global__ void zero_u32_kernel(uint32_t* dst, size_t n) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    dst[i] = 0u;
}

int elementwise_blocks(size_t n) {
  size_t b = (n + 1023) / 1024;
  if (b < 1) b = 1;
  if (b > 4096) b = 4096;
  return (int)b;
}

}  // namespace

cudaError_t launch_static_prep(const StaticPrep& p, cudaStream_t s) {
  if (p.n_static == 0) return cudaSuccess;
  const size_t smem = (2 * (size_t)p.T + 8) * sizeof(float);
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(static_prep_kernel),
                                       160 * 1024);
  if (e != cudaSuccess) return e;
  trace_begin(s);
  static_prep_kernel<<<dim3(p.T / kPrepRows, p.n_static), 256, smem, s>>>(p);
  trace_end(s, "static_prep");
  return cudaGetLastError();
}

cudaError_t launch_zero_u32(void* dst, size_t n_words, cudaStream_t s) {
  trace_begin(s);
  zero_u32_kernel<<<elementwise_blocks(n_words / 4), 256, 0, s>>>(static_cast<uint32_t*>(dst),
                                                                  n_words);
  trace_end(s, "zero");
  return cudaGetLastError();
}

// ============================================================ K2: fused kernel
namespace {

template <int D>
struct FwdSmem {
  using G = TileGeom<D>;
  // TMEM S/P buffers: three for d_h <= 64 (then S of tile j + 1 only waits for
  // P V of tile j - 2), two for d_h = 128 (the O accumulator needs the rest).
  // Three 128-column S/P buffers; the rest holds O (128 columns: one
  // sequence of a static group at d_h = 128, two at 64).  The transposed
  // engine at d_h = 128 keeps two buffers so that O holds two sequences.
  static constexpr int NBUF = 3;
  static constexpr int NBUF_T = (D == 128) ? 2 : 3;
  // K ring; d_h <= 64 forward: two rings of two, one per MMA issuer
  static constexpr int KST = (D == 128) ? 2 : 4;
  static constexpr int VST = (D == 128) ? 3 : 4;  // V ring (consumed a step after K)
  // d_h = 64: a static step's two V tiles in an even-aligned slot pair are one
  // N = 128 operand (a tile is one 128-byte-swizzled chunk, so the slot
  // stride equals the chunk stride of a [128 x 128] MN-major operand).
  static constexpr bool PAIR_V = (D == 64) && (VST % 2 == 0);
  // Q tiles: two slots for d_h <= 64 (the next item's Q lands while this
  // item's score tiles are issued), one for d_h = 128 (shared memory budget)
  static constexpr int QST = (D == 128) ? 1 : 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QST * G::TILE_BYTES;
  static constexpr int OFF_V = OFF_K + KST * G::TILE_BYTES;
  // d_h = 64: a dynamic item's output tile is staged here (128-byte swizzled,
  // as the tensor map expects) and written with one tensor store.
  static constexpr bool OSTAGE = (D == 64);
  static constexpr int OFF_OS = OFF_V + VST * G::TILE_BYTES;
  static constexpr int OFF_X = OFF_OS + (OSTAGE ? G::TILE_BYTES : 0);  // row max / sum exchange
  // a static step's generator tables (a ring of its own, read only by the
  // compute warps)
  static constexpr int AST = 4;
  static constexpr int AUX_SLOT = 2048;
  static constexpr int OFF_AUX = OFF_X + 3 * 2 * 128 * 4;
  static constexpr int OFF_BAR = OFF_AUX + AST * AUX_SLOT;
  static constexpr int NBAR = 2 * QST + 2 * KST + 2 * VST + 3 * NBUF + 2 + 2 + 2 * AST + 2;  // NBUF >= NBUF_T
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int ALLOC = BYTES + 1024;  // slack to align the base to 1024 B
  static_assert(ALLOC <= 232448, "shared memory budget exceeded");
  // a table slot (static items): 128 column values then a 256-entry distance
  // window.
  static constexpr int AUX_COL = 0;
  static constexpr int AUX_WIN = 512;
  static constexpr int AUX_BYTES = 512 + 1024;
};

// One thread's 64 columns of a generated tile, written as packed bf16 to
// TMEM columns tdst .. tdst + 31.  colv_s: shared address of the half's 64
// column values; win_s: the distance window (centre at entry 127); rc = the
// row minus the half's first column.  Forward element (i = row, j = col):
// distance rc - cl; transposed (j = row, i = col): distance cl - rc.
// Factored: colv * r(distance) * rowv; exact: exp2(colv + r(distance) + rowv).
// With SUMS (factored forward) adds the row sums of the fp32 values and of
// their bf16 roundings to zsum and zrnd.
template <bool TRANSPOSED, bool EXACT, bool SUMS>
__device__ __forceinline__ void gen_tile(uint32_t colv_s, uint32_t win_s, int rc, uint64_t row2,
                                         uint32_t tdst, float& zsum, float& zrnd) {
  // SUMS: the fp32 sum of this thread's 64 values, and the sum of the same
  // values after rounding to bf16 (what the MMA actually weighs V with)
  uint64_t sum2 = 0, rnd2 = 0;
  // address of window entry 127 + distance for column 0 of the half
  const uint32_t w0 = win_s + 4u * (uint32_t)(127 + (TRANSPOSED ? -rc : rc));
#pragma unroll
  for (int q0 = 0; q0 < 32; q0 += 16) {
    uint32_t pk[16];
#pragma unroll
    for (int qq = 0; qq < 16; ++qq) {
      const int cl = 2 * (q0 + qq);
      const uint64_t cv = lds_f32x2(colv_s + 4u * cl);
      const float wa = lds_f32(TRANSPOSED ? w0 + 4u * cl : w0 - 4u * cl);
      const float wb = lds_f32(TRANSPOSED ? w0 + 4u * (cl + 1) : w0 - 4u * (cl + 1));
      const uint64_t wv = f2_pack(wa, wb);
      if (EXACT) {
        float x0, x1;
        f2_unpack(f2_add(f2_add(cv, wv), row2), x0, x1);
        pk[qq] = pack_bf16x2(fast_exp2(x0), fast_exp2(x1));
      } else {
        // the forward's factored row factor is 1 (Z' divides in the epilogue)
        const uint64_t g = SUMS ? f2_mul(cv, wv) : f2_mul(f2_mul(cv, wv), row2);
        pk[qq] = pack_bf16x2_f2(g);
        if (SUMS) {
          sum2 = f2_add(sum2, g);
          rnd2 = f2_add(rnd2, f2_pack(__uint_as_float(pk[qq] << 16),
                                      __uint_as_float(pk[qq] & 0xffff0000u)));
        }
      }
    }
    tmem_st_x16(tdst + q0, pk);
  }
  if (SUMS) {
    float lo, hi;
    f2_unpack(sum2, lo, hi);
    zsum += lo + hi;
    f2_unpack(rnd2, lo, hi);
    zrnd += lo + hi;
  }
}

// TMEM columns (d_h = 128, and the transposed engine): NBUF 128-column
// buffers from 0 hold S (fp32).  Each compute half (key columns 0..63 or
// 64..127 of the tile) writes its P, as packed bf16, over the first 32
// columns of its own S half, so P k-steps 0..3 sit at buffer + 0.. and 4..7
// at buffer + 64..; static items keep their generated tiles in the same
// places.  The O accumulator follows the buffers (d_h columns for a dynamic
// item, group * d_h for a static item).  The forward at d_h <= 64 lays the
// columns out differently (see SPLIT in the kernel).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;
__device__ __forceinline__ uint32_t p_col(int kk) {
  return (uint32_t)((kk < 4) ? kk * 8 : 64 + (kk - 4) * 8);
}

enum : int {
  kSiteProdQ = 1, kSiteProdK, kSiteProdV, kSiteMmaQ, kSiteMmaK, kSiteMmaS, kSiteMmaV,
  kSiteMmaP, kSiteMmaO, kSiteCmpS, kSiteCmpP, kSiteCmpPV, kSiteCmpO, kSiteCmpAux
};

struct Item {
  bool is_static;
  int b;       // dynamic: sequence; static: first sequence of the group
  int nb;      // static: sequences in the group
  int h;       // head id
  int hs;      // static: index into the static tables
  int X;       // output tile index (I forward, J transposed)
  int nsteps;  // inner tiles
};

// Longest first: forward items in descending query tile; for each tile the
// static items (each worth a group of sequences) come before the dynamic ones.
// Transposed (static dV) items in ascending key tile.
template <bool TRANSPOSED>
__device__ __forceinline__ Item decode_item(const FwdParams& p, int it) {
  Item r;
  const int n_st_items = p.n_static * p.n_groups;
  const int per_x = n_st_items + (TRANSPOSED ? 0 : p.B * p.n_dynamic);
  const int q = it / per_x, rem = it - q * per_x;
  r.X = TRANSPOSED ? q : (p.nI - 1 - q);
  r.nsteps = TRANSPOSED ? (p.nI - r.X) : (r.X + 1);
  if (rem < n_st_items) {
    r.is_static = true;
    r.hs = rem / p.n_groups;
    const int g = rem - r.hs * p.n_groups;
    r.h = p.static_heads[r.hs];
    r.b = g * p.group;
    r.nb = min(p.group, p.B - r.b);
  } else {
    const int d = rem - n_st_items;
    r.is_static = false;
    r.b = d / p.n_dynamic;
    r.h = p.dynamic_heads[d - r.b * p.n_dynamic];
    r.hs = -1;
    r.nb = 1;
  }
  return r;
}

// Store 16 packed bf16x2 values of one tile row from fp32 pairs.
__device__ __forceinline__ void store_row16(__nv_bfloat16* dst, const uint32_t (&o)[16], float s) {
  uint4 v0, v1;
  v0.x = pack_bf16x2(__uint_as_float(o[0]) * s, __uint_as_float(o[1]) * s);
  v0.y = pack_bf16x2(__uint_as_float(o[2]) * s, __uint_as_float(o[3]) * s);
  v0.z = pack_bf16x2(__uint_as_float(o[4]) * s, __uint_as_float(o[5]) * s);
  v0.w = pack_bf16x2(__uint_as_float(o[6]) * s, __uint_as_float(o[7]) * s);
  v1.x = pack_bf16x2(__uint_as_float(o[8]) * s, __uint_as_float(o[9]) * s);
  v1.y = pack_bf16x2(__uint_as_float(o[10]) * s, __uint_as_float(o[11]) * s);
  v1.z = pack_bf16x2(__uint_as_float(o[12]) * s, __uint_as_float(o[13]) * s);
  v1.w = pack_bf16x2(__uint_as_float(o[14]) * s, __uint_as_float(o[15]) * s);
  *reinterpret_cast<uint4*>(dst) = v0;
  *reinterpret_cast<uint4*>(dst + 8) = v1;
}

// Threads: warp 0 TMA producer (Q, K, static tables), warp 2 TMEM owner and V
// producer, warps 1 and 3 MMA issuers, warps 4..11 two compute halves.
// d_h = 128 and transposed: warp 1 issues S, warp 3 P V; warps 4..7 take key
// columns 0..63 and warps 8..11 key columns 64..127 of each tile (a row per
// thread, two threads per row).  Forward at d_h <= 64 (SPLIT): half g takes
// the key tiles j = g, g + 2, ... of a dynamic item, whole rows, and warp 1
// (g = 0) or 3 (g = 1) issues that half's S and P V.
template <int D, bool TRANSPOSED>
__global__ void __launch_bounds__(384, 1)
    hybrid_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  using G = TileGeom<D>;
  using L = FwdSmem<D>;
  constexpr int DH = D / 2;  // output columns per compute half
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = q_full + L::QST;
  uint64_t* k_full = q_empty + L::QST;
  uint64_t* k_empty = k_full + L::KST;
  uint64_t* v_full = k_empty + L::KST;
  uint64_t* v_empty = v_full + L::VST;
  constexpr int NB = TRANSPOSED ? L::NBUF_T : L::NBUF;
  constexpr uint32_t kTmemO = NB * 128;
  // d_h <= 64, forward: the two compute halves take alternate key tiles of a
  // dynamic item, each with its own running max, sum and O accumulator (O_0
  // at kTmemO, O_1 after it), merged once per item
  constexpr bool SPLIT = (D <= 64) && !TRANSPOSED;
  // With SPLIT the TMEM holds two S buffers (columns 0..255, buffer g for
  // compute half g and its issuer, so each has one producer and one
  // consumer), two P buffers of packed bf16 (256..383: a dynamic tile's P or
  // a static step's generated tile) and O (384..511).  An S buffer is free
  // once the softmax has read it, a P buffer once its P V products are done,
  // so the next score tile never waits for a P V product.  K tiles likewise
  // go to a ring per issuer (slots 2g, 2g + 1).
  constexpr uint32_t kTmemP = 256;
  static_assert(!SPLIT || kTmemO + 2 * D <= kTmemCols, "TMEM: two O accumulators");
  static_assert(!SPLIT || kTmemP + 128 <= kTmemO, "TMEM: two P buffers");
  // S ready (MMA -> compute); without SPLIT also a static use of the buffer
  // granted (warp 1 -> compute)
  uint64_t* s_full = v_empty + L::VST;
  // buffer free again: its P V MMAs done (MMA -> all); with SPLIT: the
  // softmax has read the S buffer (compute -> S issuer, 128 arrivals)
  uint64_t* s_empty = s_full + NB;
  uint64_t* p_full = s_empty + NB;       // P / G written, O rescaled (compute -> MMA)
  uint64_t* o_full = p_full + NB;
  uint64_t* o_empty = o_full + 1;
  uint64_t* p_empty = o_empty + 1;       // SPLIT: P buffer's P V products done (two)
  uint64_t* aux_full = p_empty + 2;      // static tables landed (TMA -> compute)
  uint64_t* aux_empty = aux_full + L::AST;  // static tables read (every compute thread -> producer)
  // per MMA-issuing warp (1, 3): all its products done, before TMEM is freed
  uint64_t* mma_drained = aux_empty + L::AST;
  float* xmax = reinterpret_cast<float*>(smem + L::OFF_X);  // [2 parity][2 halves][128]
  float* xsum = xmax + 2 * 2 * 128;                         // [2 halves][128]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  const WaitCtl wc{abort_flag, p.status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    // with SPLIT both MMA issuers release a Q slot and both complete O
    for (int s = 0; s < L::QST; ++s) { mbar_init(q_full + s, 1); mbar_init(q_empty + s, SPLIT ? 2 : 1); }
    for (int s = 0; s < L::KST; ++s) { mbar_init(k_full + s, 1); mbar_init(k_empty + s, 1); }
    for (int s = 0; s < L::VST; ++s) { mbar_init(v_full + s, 1); mbar_init(v_empty + s, 1); }
    for (int s = 0; s < NB; ++s) {
      mbar_init(s_full + s, 1);
      mbar_init(s_empty + s, SPLIT ? 128 : 1);
      mbar_init(p_full + s, 256);
    }
    mbar_init(p_empty, 1);
    mbar_init(p_empty + 1, 1);
    for (int s = 0; s < L::AST; ++s) { mbar_init(aux_full + s, 1); mbar_init(aux_empty + s, 256); }
    mbar_init(o_full, SPLIT ? 2 : 1);
    mbar_init(mma_drained, 1);
    mbar_init(mma_drained + 1, 1);
    mbar_init(o_empty, 256);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sK = smem_u32(smem + L::OFF_K);
  const uint32_t sV = smem_u32(smem + L::OFF_V);
  const int H = p.H, T = p.T;

  if (warp == 0 || warp == 2) {
    // ---------------------------------------------------------- producers
    // warp 0: Q, K (and a static step's tables); warp 2 (after the TMEM
    // allocation): V, so that neither ring waits behind the other
    const bool kprod = (warp == 0);
    if (lane == 0) {
      uint32_t qc = 0, kc = 0, vc = 0, ac = 0;
      uint32_t kn0 = 0, kn1 = 0;  // SPLIT: uses of each issuer's K ring
      bool held_q = false;        // the first Q tile was withheld (testing)
      for (int kr = 0, it = snake_item(0, blockIdx.x, gridDim.x); it < p.n_items;
         it = snake_item(++kr, blockIdx.x, gridDim.x)) {
        const Item w = decode_item<TRANSPOSED>(p, it);
        if (!w.is_static) {
          const int row0 = (w.b * H + w.h) * T;                           // Q rows
          const int kv0 = (w.b * p.H_kv + w.h / p.group_kv) * T;          // K/V rows
          if (kprod) {
            const int qs = qc % L::QST;
            mbar_wait(q_empty + qs, ((qc / L::QST) & 1) ^ 1, wc, kSiteProdQ);
            // failure-path testing: CTA 0 withholds its first Q tile, so that
            // the waits on it run out (it is then not drained either)
            const bool hold = p.hold_first_q && blockIdx.x == 0 && qc == 0;
            held_q |= hold;
            ++qc;
            if (!hold) {
              mbar_arrive_expect_tx(q_full + qs, G::TILE_BYTES);
              for (int c = 0; c < G::NCHUNK; ++c)
                tma_load_2d(smem + L::OFF_Q + qs * G::TILE_BYTES + c * G::CHUNK_BYTES, &tm_q,
                            q_full + qs, c * G::CHUNK, row0 + w.X * 128);
            }
            for (int j = 0; j < w.nsteps; ++j) {
              int ks;
              uint32_t kpar;
              if (SPLIT) {
                const uint32_t n = (j & 1) ? kn1++ : kn0++;
                ks = 2 * (j & 1) + (int)(n & 1);
                kpar = ((n >> 1) & 1) ^ 1;
              } else {
                ks = kc % L::KST;
                kpar = ((kc / L::KST) & 1) ^ 1;
                ++kc;
              }
              mbar_wait(k_empty + ks, kpar, wc, kSiteProdK);
              mbar_arrive_expect_tx(k_full + ks, G::TILE_BYTES);
              for (int c = 0; c < G::NCHUNK; ++c)
                tma_load_2d(smem + L::OFF_K + ks * G::TILE_BYTES + c * G::CHUNK_BYTES, &tm_k,
                            k_full + ks, c * G::CHUNK, kv0 + j * 128);
            }
          } else {
            for (int j = 0; j < w.nsteps; ++j) {
              const int vs = vc % L::VST;
              mbar_wait(v_empty + vs, ((vc / L::VST) & 1) ^ 1, wc, kSiteProdV);
              ++vc;
              mbar_arrive_expect_tx(v_full + vs, G::TILE_BYTES);
              for (int c = 0; c < G::NCHUNK; ++c)
                tma_load_2d(smem + L::OFF_V + vs * G::TILE_BYTES + c * G::CHUNK_BYTES, &tm_v,
                            v_full + vs, c * G::CHUNK, kv0 + j * 128);
            }
          }
        } else {
          // A static step's tables go into the table ring (warp 0), its V
          // tiles into the V ring (warp 2).
          auto load_aux = [&](int step) {
            // inner tile Y: J (forward) or I (transposed)
            const int Y = TRANSPOSED ? (w.X + step) : step;
            const int dist0 = TRANSPOSED ? (Y - w.X) : (w.X - Y);  // (I - J) in tiles
            const int as = ac % L::AST;
            mbar_wait(aux_empty + as, ((ac / L::AST) & 1) ^ 1, wc, kSiteProdK);
            ++ac;
            mbar_arrive_expect_tx(aux_full + as, L::AUX_BYTES);
            uint8_t* aux = smem + L::OFF_AUX + as * L::AUX_SLOT;
            // column values: a(j) for j in tile J (forward) or row values of
            // tile I (transposed)
            const float* col_src = TRANSPOSED ? (p.row_tab + (size_t)w.hs * T + Y * 128)
                                              : (p.a_tab + (size_t)w.hs * T + Y * 128);
            bulk_load(aux + L::AUX_COL, col_src, 512, aux_full + as);
            bulk_load(aux + L::AUX_WIN, p.r_tab + (size_t)w.hs * (T + 128) + dist0 * 128, 1024,
                      aux_full + as);
          };
          if (kprod) {
            for (int step = 0; step < w.nsteps; ++step) load_aux(step);
          } else {
            for (int step = 0; step < w.nsteps; ++step) {
              const int Y = TRANSPOSED ? (w.X + step) : step;
              if (L::PAIR_V && w.nb == 2 && (vc & 1)) {
                // the pair must start at an even slot: one slot carries nothing
                const int vs = vc % L::VST;
                mbar_wait(v_empty + vs, ((vc / L::VST) & 1) ^ 1, wc, kSiteProdV);
                ++vc;
                mbar_arrive(v_full + vs);
              }
              for (int bb = 0; bb < w.nb; ++bb) {
                const int vs = vc % L::VST;
                mbar_wait(v_empty + vs, ((vc / L::VST) & 1) ^ 1, wc, kSiteProdV);
                ++vc;
                mbar_arrive_expect_tx(v_full + vs, G::TILE_BYTES);
                // forward: V of the head's K/V group; transposed: dO of the head
                const int row0 = TRANSPOSED ? ((w.b + bb) * H + w.h) * T
                                            : ((w.b + bb) * p.H_kv + w.h / p.group_kv) * T;
                for (int c = 0; c < G::NCHUNK; ++c)
                  tma_load_2d(smem + L::OFF_V + vs * G::TILE_BYTES + c * G::CHUNK_BYTES, &tm_v,
                              v_full + vs, c * G::CHUNK, row0 + Y * 128);
              }
            }
          }
        }
      }
      // Drain: every copy issued must have landed before the CTA exits (a
      // withheld Q tile, use 0 of slot 0, was never issued).
      for (int s = 0; s < L::QST; ++s)
        if (qc > (uint32_t)s && !(held_q && s == 0 && (qc - 1) / L::QST == 0))
          mbar_drain(q_full + s, ((qc - 1 - s) / L::QST) & 1);
      if (SPLIT) {
        for (int g = 0; g < 2; ++g) {
          const uint32_t n = g ? kn1 : kn0;
          for (uint32_t i = 0; i < 2; ++i)
            if (n > i) {
              const uint32_t m = n - 1 - i;  // the last use of slot 2g + (m & 1)
              mbar_drain(k_full + 2 * g + (int)(m & 1), (m >> 1) & 1);
            }
        }
      } else {
        for (int s = 0; s < L::KST; ++s)
          if (kc > (uint32_t)s) mbar_drain(k_full + s, ((kc - 1 - s) / L::KST) & 1);
      }
      for (int s = 0; s < L::AST; ++s)
        if (ac > (uint32_t)s) mbar_drain(aux_full + s, ((ac - 1 - s) / L::AST) & 1);
      for (int s = 0; s < L::VST; ++s)
        if (vc > (uint32_t)s) mbar_drain(v_full + s, ((vc - 1 - s) / L::VST) & 1);
    }
  } else if (SPLIT && (warp == 1 || warp == 3)) {
    // ---------------------------------------------------------- MMA issuers
    // Issuer g (warp 1: g = 0, warp 3: g = 1) issues S and P V of the key
    // tiles j = g, g + 2, ... of a dynamic item, i.e. of compute half g, so
    // that one half's products never queue behind the other half's softmax.
    // Static items: issuer 0 issues every step (one accumulation chain),
    // issuer 1 only keeps its ring counts.
    if (lane == 0) {
      const int g = (warp == 1) ? 0 : 1;
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, false, true);
      constexpr uint32_t idesc_pair = idesc_bf16(128, 2 * D, false, true);
      uint32_t qc = 0, vc = 0, sc = 0, oc = 0;
      uint32_t kn = 0, sn = 0;  // uses of this issuer's K ring and of S buffer g
      for (int kr = 0, it = snake_item(0, blockIdx.x, gridDim.x); it < p.n_items;
           it = snake_item(++kr, blockIdx.x, gridDim.x)) {
        const Item w = decode_item<TRANSPOSED>(p, it);
        // before the first product into O: the previous item's O has been
        // read out (an issuer without products waits too, so that its
        // o_full arrival falls into this item's phase)
        bool o_ready = false;
        auto wait_o = [&]() {
          if (!o_ready) mbar_wait(o_empty, (oc & 1) ^ 1, wc, kSiteMmaO);
          o_ready = true;
        };
        if (!w.is_static) {
          const int qs = qc % L::QST;
          const uint32_t sQ = smem_u32(smem + L::OFF_Q + qs * G::TILE_BYTES);
          mbar_wait(q_full + qs, (qc / L::QST) & 1, wc, kSiteMmaQ);
          ++qc;
          // S of this half's tiles, in order (j = g, g + 2, ...)
          auto issue_s = [&]() {
            const int ks = 2 * g + (int)(kn & 1);
            mbar_wait(k_full + ks, (kn >> 1) & 1, wc, kSiteMmaK);
            mbar_wait(s_empty + g, (sn & 1) ^ 1, wc, kSiteMmaS);
            tc_fence_after();
            const uint32_t kt = sK + ks * G::TILE_BYTES;
#pragma unroll
            for (int kk = 0; kk < G::KSTEPS; ++kk)
              mma_bf16_ss(tmem + kTmemS + (uint32_t)g * 128, G::kmajor_desc(sQ, kk),
                          G::kmajor_desc(kt, kk), idesc_s, kk > 0);
            mma_commit(k_empty + ks);
            mma_commit(s_full + g);
            ++kn;
            ++sn;
          };
          auto issue_pv = [&](int j) {
            const uint32_t u = sc + j, pb = u & 1;
            const uint32_t vq = vc + j;
            const int vs = vq % L::VST;
            mbar_wait(v_full + vs, (vq / L::VST) & 1, wc, kSiteMmaV);
            mbar_wait(p_full + pb, (u >> 1) & 1, wc, kSiteMmaP);
            tc_fence_after();
            const uint32_t vt = sV + vs * G::TILE_BYTES;
            const uint32_t pa = tmem + kTmemP + pb * 64;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16_ts(tmem + kTmemO + (uint32_t)g * D, pa + 8 * kk, G::mnmajor_desc(vt, kk),
                          idesc_pv, (j > 1 || kk > 0));
            mma_commit(v_empty + vs);
            mma_commit(p_empty + pb);
          };
          // S of the half's next tile goes out as soon as the half has read
          // the previous one; its P V once the P is written
          if (g < w.nsteps) issue_s();
          for (int j = g; j < w.nsteps; j += 2) {
            if (j + 2 < w.nsteps) issue_s();
            wait_o();
            issue_pv(j);
          }
          mma_commit(q_empty + qs);
          vc += w.nsteps;
        } else {
          for (int step = 0; step < w.nsteps; ++step) {
            const uint32_t u = sc + step, pb = u & 1;
            if (g == 1) {
              // the V ring positions issuer 0 consumes for this step
              if (L::PAIR_V && w.nb == 2 && (vc & 1)) ++vc;
              vc += w.nb;
              continue;
            }
            // the previous item's P buffers are all written and read once its
            // O has been read out, so this parity wait cannot match an older use
            wait_o();
            mbar_wait(p_full + pb, (u >> 1) & 1, wc, kSiteMmaP);
            const uint32_t ga = tmem + kTmemP + pb * 64;
            if (L::PAIR_V && w.nb == 2) {
              // Two sequences' V tiles in adjacent slots form one [128 x 2 d_h]
              // MN-major operand (the slot stride is the chunk stride), so one
              // N = 2 d_h product fills O_b0 | O_b1.
              if (vc & 1) {
                const int vs = vc % L::VST;
                mbar_wait(v_full + vs, (vc / L::VST) & 1, wc, kSiteMmaV);
                mma_commit(v_empty + vs);
                ++vc;
              }
              const int vs = vc % L::VST;
              mbar_wait(v_full + vs, (vc / L::VST) & 1, wc, kSiteMmaV);
              mbar_wait(v_full + vs + 1, ((vc + 1) / L::VST) & 1, wc, kSiteMmaV);
              tc_fence_after();
              const uint32_t vt = sV + vs * G::TILE_BYTES;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_bf16_ts(tmem + kTmemO, ga + 8 * kk, G::mnmajor_desc(vt, kk), idesc_pair,
                            (step > 0 || kk > 0));
              mma_commit(v_empty + vs);
              mma_commit(v_empty + vs + 1);
              vc += 2;
            } else {
              for (int bb = 0; bb < w.nb; ++bb) {
                const int vs = vc % L::VST;
                mbar_wait(v_full + vs, (vc / L::VST) & 1, wc, kSiteMmaV);
                tc_fence_after();
                const uint32_t vt = sV + vs * G::TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                  mma_bf16_ts(tmem + kTmemO + bb * D, ga + 8 * kk, G::mnmajor_desc(vt, kk),
                              idesc_pv, (step > 0 || kk > 0));
                mma_commit(v_empty + vs);
                ++vc;
              }
            }
            mma_commit(p_empty + pb);
          }
        }
        sc += w.nsteps;
        wait_o();
        mma_commit(o_full);  // (with no products pending this arrives at once)
        ++oc;
      }
      // every product of this warp has completed before TMEM is freed (after
      // an abort no later wait guarantees it)
      mma_commit(mma_drained + g);
      mbar_drain(mma_drained + g, 0);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- S issuer
    // S = Q K^T of every dynamic step.  A second warp issues the P V
    // products, so that a score MMA never queues behind a wait for the
    // softmax: each issuing thread blocks while its MMAs are accepted.
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      uint32_t qc = 0, kc = 0, sc = 0;
      for (int kr = 0, it = snake_item(0, blockIdx.x, gridDim.x); it < p.n_items;
         it = snake_item(++kr, blockIdx.x, gridDim.x)) {
        const Item w = decode_item<TRANSPOSED>(p, it);
        const uint32_t sc0 = sc;
        if (!w.is_static) {
          const int qs = qc % L::QST;
          const uint32_t sQ = smem_u32(smem + L::OFF_Q + qs * G::TILE_BYTES);
          mbar_wait(q_full + qs, (qc / L::QST) & 1, wc, kSiteMmaQ);
          ++qc;
          for (int j = 0; j < w.nsteps; ++j) {
            const uint32_t u = sc0 + j;
            const int ks = kc % L::KST;
            mbar_wait(k_full + ks, (kc / L::KST) & 1, wc, kSiteMmaK);
            const uint32_t b = u % NB;
            mbar_wait(s_empty + b, ((u / NB) & 1) ^ 1, wc, kSiteMmaS);
            tc_fence_after();
            const uint32_t kt = sK + ks * G::TILE_BYTES;
#pragma unroll
            for (int kk = 0; kk < G::KSTEPS; ++kk)
              mma_bf16_ss(tmem + kTmemS + b * 128, G::kmajor_desc(sQ, kk), G::kmajor_desc(kt, kk),
                          idesc_s, kk > 0);
            mma_commit(k_empty + ks);
            mma_commit(s_full + b);
            if (j == w.nsteps - 1) mma_commit(q_empty + qs);
            ++kc;
          }
        } else {
          // A static step's buffer is granted here too, once its previous
          // use is done: this warp takes part in every use of every buffer,
          // so its parity waits never meet a phase two uses away.
          for (int step = 0; step < w.nsteps; ++step) {
            const uint32_t u = sc0 + step, b = u % NB;
            mbar_wait(s_empty + b, ((u / NB) & 1) ^ 1, wc, kSiteMmaS);
            mbar_arrive(s_full + b);
          }
        }
        sc = sc0 + w.nsteps;
      }
      mma_commit(mma_drained);  // every product of this warp done before TMEM is freed
      mbar_drain(mma_drained, 0);
    }
  } else if (warp == 3) {
    // ---------------------------------------------------------- P V issuer
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, false, true);
      constexpr uint32_t idesc_pair = idesc_bf16(128, 2 * D, false, true);
      uint32_t vc = 0, sc = 0, oc = 0;
      for (int kr = 0, it = snake_item(0, blockIdx.x, gridDim.x); it < p.n_items;
         it = snake_item(++kr, blockIdx.x, gridDim.x)) {
        const Item w = decode_item<TRANSPOSED>(p, it);
        const uint32_t sc0 = sc;
        if (!w.is_static) {
          for (int j = 0; j < w.nsteps; ++j) {
            const uint32_t u = sc0 + j;
            const int vs = vc % L::VST;
            mbar_wait(v_full + vs, (vc / L::VST) & 1, wc, kSiteMmaV);
            const uint32_t pb = u % NB;
            mbar_wait(p_full + pb, (u / NB) & 1, wc, kSiteMmaP);
            if (j == 0) mbar_wait(o_empty, (oc & 1) ^ 1, wc, kSiteMmaO);
            tc_fence_after();
            const uint32_t vt = sV + vs * G::TILE_BYTES;
            const uint32_t pa = tmem + kTmemS + pb * 128;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16_ts(tmem + kTmemO, pa + p_col(kk), G::mnmajor_desc(vt, kk), idesc_pv,
                          (j > 0 || kk > 0));
            mma_commit(v_empty + vs);
            mma_commit(s_empty + pb);
            ++vc;
          }
          mma_commit(o_full);
          ++oc;
        } else {
          for (int step = 0; step < w.nsteps; ++step) {
            const uint32_t u = sc0 + step;
            const uint32_t pb = u % NB;
            mbar_wait(p_full + pb, (u / NB) & 1, wc, kSiteMmaP);
            if (step == 0) mbar_wait(o_empty, (oc & 1) ^ 1, wc, kSiteMmaO);
            const uint32_t ga = tmem + kTmemS + pb * 128;
            if (L::PAIR_V && w.nb == 2) {
              // Two sequences' V tiles in adjacent slots form one [128 x 2 d_h]
              // MN-major operand (the slot stride is the chunk stride), so one
              // N = 2 d_h product fills O_b0 | O_b1.
              if (vc & 1) {
                const int vs = vc % L::VST;
                mbar_wait(v_full + vs, (vc / L::VST) & 1, wc, kSiteMmaV);
                mma_commit(v_empty + vs);
                ++vc;
              }
              const int vs = vc % L::VST;
              mbar_wait(v_full + vs, (vc / L::VST) & 1, wc, kSiteMmaV);
              mbar_wait(v_full + vs + 1, ((vc + 1) / L::VST) & 1, wc, kSiteMmaV);
              tc_fence_after();
              const uint32_t vt = sV + vs * G::TILE_BYTES;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_bf16_ts(tmem + kTmemO, ga + p_col(kk), G::mnmajor_desc(vt, kk), idesc_pair,
                            (step > 0 || kk > 0));
              mma_commit(v_empty + vs);
              mma_commit(v_empty + vs + 1);
              vc += 2;
            } else {
              for (int bb = 0; bb < w.nb; ++bb) {
                const int vs = vc % L::VST;
                mbar_wait(v_full + vs, (vc / L::VST) & 1, wc, kSiteMmaV);
                tc_fence_after();
                const uint32_t vt = sV + vs * G::TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                  mma_bf16_ts(tmem + kTmemO + bb * D, ga + p_col(kk), G::mnmajor_desc(vt, kk),
                              idesc_pv, (step > 0 || kk > 0));
                mma_commit(v_empty + vs);
                ++vc;
              }
            }
            // the use ends here (warp 1 granted it through s_full)
            mma_commit(s_empty + pb);
          }
          mma_commit(o_full);
          ++oc;
        }
        sc = sc0 + w.nsteps;
      }
      mma_commit(mma_drained + 1);  // every product of this warp done before TMEM is freed
      mbar_drain(mma_drained + 1, 0);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------- compute halves
    const int hf = (warp - 4) >> 2;              // key columns 64*hf .. 64*hf + 63
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;                // tile row == TMEM lane
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    const int pair_bar = 2 + q4;                 // the two warps that share these rows
    uint32_t ac = 0, sc = 0, oc = 0;  // static tables, P ring uses (all steps), items
    uint32_t sn = 0;  // SPLIT: this half's dynamic tiles (uses of S buffer hf)
    for (int kr = 0, it = snake_item(0, blockIdx.x, gridDim.x); it < p.n_items;
         it = snake_item(++kr, blockIdx.x, gridDim.x)) {
      const Item w = decode_item<TRANSPOSED>(p, it);
      const uint32_t sc0 = sc;
      if (!w.is_static && SPLIT) {
        // this half's key tiles: j = hf, hf + 2, ...; a thread holds a whole
        // row of each of its tiles
        float m_run = -INFINITY, l_run = 0.f;
        for (int j = hf; j < w.nsteps; j += 2) {
          const uint32_t u = sc0 + j;   // P ring use
          const uint32_t sb = (uint32_t)hf, pb = u & 1;
          const uint32_t sbase = trow + kTmemS + sb * 128;
          const uint32_t pbase = trow + kTmemP + pb * 64;
          mbar_wait(s_full + sb, sn & 1, wc, kSiteCmpS);
          ++sn;
          tc_fence_after();
          uint32_t sr[128];
          {
            uint32_t (&a0)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr);
            uint32_t (&a1)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr + 32);
            uint32_t (&a2)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr + 64);
            uint32_t (&a3)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr + 96);
            tmem_ld_x32(sbase, a0);
            tmem_ld_x32(sbase + 32, a1);
            tmem_ld_x32(sbase + 64, a2);
            tmem_ld_x32(sbase + 96, a3);
            tmem_wait_ld(a0);
            tmem_wait_ld(a1);
            tmem_wait_ld(a2);
            tmem_wait_ld(a3);
          }
          // the S buffer may take the next score tile
          tc_fence_before();
          mbar_arrive(s_empty + sb);
          // causal mask on the diagonal tile: key column c > row r
          if (j == w.X) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c > r) sr[c] = 0xff800000u;  // -inf
          }
          float mx[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mx[k] = fmaxf(__uint_as_float(sr[k]), __uint_as_float(sr[k + 8]));
#pragma unroll
          for (int c = 16; c < 128; c += 16)
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mx[k] = fmax3(mx[k], __uint_as_float(sr[c + k]), __uint_as_float(sr[c + 8 + k]));
          const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                 fmaxf(mx[6], mx[7])) * p.scale_log2;
          const float m_new = fmaxf(m_run, mt);
          const bool need = m_new > m_run + 8.0f;
          const float m_use = need ? m_new : m_run;
          const float corr = need ? fast_exp2(m_run - m_new) : 1.0f;
          const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
          const uint64_t nm2 = f2_pack(-m_use, -m_use);
          uint64_t acc[2] = {0ull, 0ull};
          // the P buffer is free once the P V products of two uses back are
          // done (for j >= 2 those are this half's previous tile, so O_hf is
          // also final for a rescale)
          mbar_wait(p_empty + pb, ((u >> 1) & 1) ^ 1, wc, kSiteCmpPV);
          tc_fence_after();
          // P as packed bf16 pairs, 8 columns at a time (few registers live
          // beside the row's 128 scores)
#pragma unroll
          for (int q0 = 0; q0 < 64; q0 += 8) {
            uint32_t pk[8];
#pragma unroll
            for (int qq = 0; qq < 8; ++qq) {
              const int q = q0 + qq;
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * q]), __uint_as_float(sr[2 * q + 1])),
                               sc2, nm2),
                        x0, x1);
              const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
              acc[qq & 1] = f2_add(acc[qq & 1], f2_pack(e0, e1));
              pk[qq] = pack_bf16x2(e0, e1);
            }
            tmem_st_x8(pbase + q0, pk);
          }
          float rs;
          {
            const uint64_t t = f2_add(acc[0], acc[1]);
            float lo, hi;
            f2_unpack(t, lo, hi);
            rs = lo + hi;
          }
          // Rescale this half's O when some row of the warp moved its max
          // (its previous P V has finished: the P buffer wait above).
          if (j > 1 && __any_sync(0xffffffffu, need)) {
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 16) {
              uint32_t o[16];
              const uint32_t ta = trow + kTmemO + hf * D + c0;
              tmem_ld_x16(ta, o);
              tmem_wait_ld(o);
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
              tmem_st_x16(ta, o);
            }
          }
          tmem_wait_st();
          l_run = l_run * corr + rs;
          m_run = m_use;
          tc_fence_before();
          mbar_arrive_cnt(p_full + pb, 2);  // the other half does not touch this tile
        }
        sc = sc0 + w.nsteps;
        // merge the halves' (max, sum) of each row; a half without tiles (a
        // one-tile item) has sum 0 and weight 0
        xmax[hf * 128 + r] = m_run;
        xsum[hf * 128 + r] = l_run;
        named_bar_sync(pair_bar, 64);
        const float m_oth = xmax[(1 - hf) * 128 + r], l_oth = xsum[(1 - hf) * 128 + r];
        named_bar_sync(pair_bar, 64);  // xsum / xmax may be rewritten by the next item
        const bool has1 = w.nsteps > 1;
        const float m0 = hf == 0 ? m_run : m_oth, l0 = hf == 0 ? l_run : l_oth;
        const float m1 = hf == 0 ? m_oth : m_run, l1 = hf == 0 ? l_oth : l_run;
        const float mm = has1 ? fmaxf(m0, m1) : m0;
        const float c0 = fast_exp2(m0 - mm);
        const float c1 = has1 ? fast_exp2(m1 - mm) : 0.f;
        const float l_tot = l0 * c0 + l1 * c1;
        const float inv_l = 1.0f / l_tot;
        const float w0 = c0 * inv_l, w1 = c1 * inv_l;
        mbar_wait(o_full, oc & 1, wc, kSiteCmpO);
        tc_fence_after();
        // this half writes output columns hf * d_h / 2 .. + d_h / 2 - 1
        uint32_t o[DH / 16][16];
#pragma unroll
        for (int c = 0; c < DH / 16; ++c) tmem_ld_x16(trow + kTmemO + hf * DH + 16 * c, o[c]);
#pragma unroll
        for (int c = 0; c < DH / 16; ++c) tmem_wait_ld(o[c]);
#pragma unroll
        for (int c = 0; c < DH / 16; ++c)
#pragma unroll
          for (int e = 0; e < 16; ++e) o[c][e] = __float_as_uint(__uint_as_float(o[c][e]) * w0);
        if (has1) {
#pragma unroll
          for (int c = 0; c < DH / 16; ++c) {
            uint32_t o1[16];
            tmem_ld_x16(trow + kTmemO + D + hf * DH + 16 * c, o1);
            tmem_wait_ld(o1);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              o[c][e] = __float_as_uint(fmaf(__uint_as_float(o1[e]), w1, __uint_as_float(o[c][e])));
          }
        }
        const size_t orow = ((size_t)(w.b * H + w.h) * T + (size_t)w.X * 128 + r);
        if constexpr (L::OSTAGE) {
          // bf16 into the staging tile, then one tensor store
          if (warp == 4 && lane == 0) bulk_wait_group_read0();
          named_bar_sync(1, 256);
          const uint32_t stg = smem_u32(smem + L::OFF_OS);
#pragma unroll
          for (int c = 0; c < DH / 16; ++c) {
            uint32_t v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              v[e] = pack_bf16x2(__uint_as_float(o[c][2 * e]), __uint_as_float(o[c][2 * e + 1]));
            const uint32_t u = (uint32_t)(hf * (DH / 8) + 2 * c);
            st_shared_v4(stg + sw128_offset(r, u), v[0], v[1], v[2], v[3]);
            st_shared_v4(stg + sw128_offset(r, u + 1), v[4], v[5], v[6], v[7]);
          }
          fence_proxy_async_smem();
          named_bar_sync(1, 256);
          if (warp == 4 && lane == 0) {
            tma_store_2d(&tm_o, smem + L::OFF_OS, 0, (w.b * H + w.h) * T + w.X * 128);
            bulk_commit_group();
          }
        } else {
#pragma unroll
          for (int c = 0; c < DH / 16; ++c)
            store_row16(p.out + orow * D + hf * DH + 16 * c, o[c], 1.0f);
        }
        if (hf == 0 && p.lse) p.lse[orow] = (mm + log2f(l_tot)) * kLn2;
        tc_fence_before();
        mbar_arrive(o_empty);
        ++oc;
      } else if (!w.is_static) {
        float m_run = -INFINITY, l_run = 0.f;
        for (int j = 0; j < w.nsteps; ++j) {
          const uint32_t u = sc0 + j;
          const uint32_t sb = u % NB;
          const uint32_t sbase = trow + kTmemS + sb * 128 + 64 * hf;
          mbar_wait(s_full + sb, (u / NB) & 1, wc, kSiteCmpS);
          tc_fence_after();
          uint32_t sr[64];
          {
            uint32_t (&a0)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr);
            uint32_t (&a1)[32] = *reinterpret_cast<uint32_t(*)[32]>(sr + 32);
            tmem_ld_x32(sbase, a0);
            tmem_ld_x32(sbase + 32, a1);
            tmem_wait_ld(a0);
            tmem_wait_ld(a1);
          }
          // Causal mask on the diagonal tile: key column 64*hf + c > row r.
          if (j == w.X) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (64 * hf + c > r) sr[c] = 0xff800000u;  // -inf
          }
          // Partial row max over this half (eight short chains), then the
          // other half's through shared memory.
          float mx[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mx[k] = fmaxf(__uint_as_float(sr[k]), __uint_as_float(sr[k + 8]));
#pragma unroll
          for (int c = 16; c < 64; c += 16)
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mx[k] = fmax3(mx[k], __uint_as_float(sr[c + k]), __uint_as_float(sr[c + 8 + k]));
          const float mh = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                 fmaxf(mx[6], mx[7]));
          float* xm = xmax + (u & 1) * 256;
          xm[hf * 128 + r] = mh;
          named_bar_sync(pair_bar, 64);
          const float mt = fmaxf(mh, xm[(1 - hf) * 128 + r]) * p.scale_log2;
          const float m_new = fmaxf(m_run, mt);
          const bool need = m_new > m_run + 8.0f;
          const float m_use = need ? m_new : m_run;
          const float corr = need ? fast_exp2(m_run - m_new) : 1.0f;
          // p = exp2(s * scale_log2 - m_use): one packed FMA per pair, two
          // exponentials, a packed add into four partial sums; P goes over the
          // first 32 columns of this half (already read), 16 at a time.
          const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
          const uint64_t nm2 = f2_pack(-m_use, -m_use);
          uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int q0 = 0; q0 < 32; q0 += 16) {
            uint32_t pk[16];
#pragma unroll
            for (int qq = 0; qq < 16; ++qq) {
              const int q = q0 + qq;
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * q]), __uint_as_float(sr[2 * q + 1])),
                               sc2, nm2),
                        x0, x1);
              const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
              acc[qq & 3] = f2_add(acc[qq & 3], f2_pack(e0, e1));
              pk[qq] = pack_bf16x2(e0, e1);
            }
            tmem_st_x16(sbase + q0, pk);
          }
          float rs;
          {
            const uint64_t t = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
            float lo, hi;
            f2_unpack(t, lo, hi);
            rs = lo + hi;
          }
          // Rescale this half's O columns when some row of the warp moved its
          // max: the previous tile's P V must have finished first.
          if (j > 0 && __any_sync(0xffffffffu, need)) {
            const uint32_t up = u - 1;
            mbar_wait(s_empty + (up % NB), (up / NB) & 1, wc, kSiteCmpPV);
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < DH; c0 += 16) {
              uint32_t o[16];
              const uint32_t ta = trow + kTmemO + hf * DH + c0;
              tmem_ld_x16(ta, o);
              tmem_wait_ld(o);
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
              tmem_st_x16(ta, o);
            }
          }
          tmem_wait_st();
          l_run = l_run * corr + rs;
          m_run = m_use;
          tc_fence_before();
          mbar_arrive(p_full + sb);
        }
        sc = sc0 + w.nsteps;
        // epilogue: O / l -> out (each half its d_h / 2 columns), lse
        xsum[hf * 128 + r] = l_run;
        named_bar_sync(pair_bar, 64);
        const float l_tot = l_run + xsum[(1 - hf) * 128 + r];
        named_bar_sync(pair_bar, 64);  // xsum may be rewritten by the next item
        mbar_wait(o_full, oc & 1, wc, kSiteCmpO);
        tc_fence_after();
        const float inv_l = 1.0f / l_tot;
        const size_t orow = ((size_t)(w.b * H + w.h) * T + (size_t)w.X * 128 + r);
        if constexpr (L::OSTAGE && !TRANSPOSED) {
          // O / l as bf16 into the staging tile, then one tensor store
          uint32_t o[2][16];
          tmem_ld_x16(trow + kTmemO + hf * DH, o[0]);
          tmem_ld_x16(trow + kTmemO + hf * DH + 16, o[1]);
          tmem_wait_ld(o[0]);
          tmem_wait_ld(o[1]);
          // the previous item's tensor store has read the staging tile
          if (warp == 4 && lane == 0) bulk_wait_group_read0();
          named_bar_sync(1, 256);
          const uint32_t stg = smem_u32(smem + L::OFF_OS);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              v[e] = pack_bf16x2(__uint_as_float(o[h2][2 * e]) * inv_l,
                                 __uint_as_float(o[h2][2 * e + 1]) * inv_l);
            const uint32_t u = (uint32_t)(hf * 4 + 2 * h2);
            st_shared_v4(stg + sw128_offset(r, u), v[0], v[1], v[2], v[3]);
            st_shared_v4(stg + sw128_offset(r, u + 1), v[4], v[5], v[6], v[7]);
          }
          fence_proxy_async_smem();
          named_bar_sync(1, 256);
          if (warp == 4 && lane == 0) {
            tma_store_2d(&tm_o, smem + L::OFF_OS, 0, (w.b * H + w.h) * T + w.X * 128);
            bulk_commit_group();
          }
        } else {
          __nv_bfloat16* dst = p.out + orow * D + hf * DH;
#pragma unroll
          for (int c0 = 0; c0 < DH; c0 += 16) {
            uint32_t o[16];
            tmem_ld_x16(trow + kTmemO + hf * DH + c0, o);
            tmem_wait_ld(o);
            store_row16(dst + c0, o, inv_l);
          }
        }
        if (hf == 0 && p.lse) p.lse[orow] = (m_run + log2f(l_tot)) * kLn2;
        tc_fence_before();
        mbar_arrive(o_empty);
        ++oc;
      } else {
        // static item: generate G (or G^T) tiles into TMEM, then the epilogue
        const bool exact = p.mode[w.hs] != 0;
        // per-row value: transposed a(j); forward exact -log2 Z(i); forward
        // factored 1: the tiles hold a(j) r(i-j), whose row sums give Z'(i),
        // and the epilogue divides by it
        const float rowv = TRANSPOSED ? p.a_tab[(size_t)w.hs * T + w.X * 128 + r]
                           : exact    ? p.row_tab[(size_t)w.hs * T + w.X * 128 + r]
                                      : 1.0f;
        const uint64_t row2 = f2_pack(rowv, rowv);
        // this half's share of Z'(i) (forward, factored): exact, and of the
        // bf16 weights the products use
        float zpart = 0.f, zround = 0.f;
        for (int step = 0; step < w.nsteps; ++step) {
          const uint32_t u = sc0 + step;
          const int as = ac % L::AST;
          mbar_wait(aux_full + as, (ac / L::AST) & 1, wc, kSiteCmpAux);
          const float* aux = reinterpret_cast<const float*>(smem + L::OFF_AUX + as * L::AUX_SLOT);
          const float* colv = aux + 64 * hf;       // this half's 64 column values
          const float* win = aux + L::AUX_WIN / 4; // window, centre at 127
          // the buffer must be free: SPLIT, the P V products of two uses back
          // are done; otherwise warp 1 has granted it
          if (SPLIT)
            mbar_wait(p_empty + (u & 1), ((u >> 1) & 1) ^ 1, wc, kSiteCmpP);
          else
            mbar_wait(s_full + (u % NB), (u / NB) & 1, wc, kSiteCmpP);  // warp 1's grant
          tc_fence_after();
          // this half's 64 keys as 32 packed columns
          const uint32_t gdst = SPLIT ? trow + kTmemP + (u & 1) * 64 + 32 * hf
                                      : trow + kTmemS + (u % NB) * 128 + 64 * hf;
          if (exact)
            gen_tile<TRANSPOSED, true, false>(smem_u32(colv), smem_u32(win), r - 64 * hf, row2,
                                              gdst, zpart, zround);
          else
            gen_tile<TRANSPOSED, false, !TRANSPOSED>(smem_u32(colv), smem_u32(win), r - 64 * hf,
                                                     row2, gdst, zpart, zround);
          // this thread has read the table slot
          mbar_arrive(aux_empty + as);
          ++ac;
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(p_full + (SPLIT ? (u & 1) : (u % NB)));
        }
        sc = sc0 + w.nsteps;
        // forward, factored: Z'(i) = both halves' sums.  out = O divided by
        // the sum of the bf16 weights the products used (so each row of the
        // pattern that V is mixed with sums to one exactly: the identity
        // pattern copies V), lse = log Z' (exact sum) + the head's shift
        float oscale = 1.0f, lse_i = 0.f;
        if (!TRANSPOSED && !exact) {
          xsum[hf * 128 + r] = zpart;
          xmax[hf * 128 + r] = zround;
          named_bar_sync(pair_bar, 64);
          const float z = zpart + xsum[(1 - hf) * 128 + r];
          const float zr = zround + xmax[(1 - hf) * 128 + r];
          named_bar_sync(pair_bar, 64);  // xsum may be rewritten by the next item
          oscale = zr > 0.f ? 1.0f / zr : 0.f;
          lse_i = z > 0.f ? logf(z) + p.shift[w.hs] : -INFINITY;
        }
        mbar_wait(o_full, oc & 1, wc, kSiteCmpO);
        tc_fence_after();
        const int trow_i = w.X * 128 + r;
        for (int bb = 0; bb < w.nb; ++bb) {
          const size_t orow = ((size_t)((w.b + bb) * H + w.h) * T + trow_i);
          if (TRANSPOSED && p.out_acc) {
            // grouped K/V: several query heads add into one K/V head's dV
            const size_t arow =
                ((size_t)((w.b + bb) * p.H_kv + w.h / p.group_kv) * T + trow_i);
            float* dst = p.out_acc + arow * D + hf * DH;
#pragma unroll
            for (int c0 = 0; c0 < DH; c0 += 16) {
              uint32_t o[16];
              tmem_ld_x16(trow + kTmemO + bb * D + hf * DH + c0, o);
              tmem_wait_ld(o);
#pragma unroll
              for (int e = 0; e < 16; e += 4)
                atomicAdd(reinterpret_cast<float4*>(dst + c0 + e),
                          make_float4(__uint_as_float(o[e]), __uint_as_float(o[e + 1]),
                                      __uint_as_float(o[e + 2]), __uint_as_float(o[e + 3])));
            }
            continue;
          }
          __nv_bfloat16* dst = p.out + orow * D + hf * DH;
#pragma unroll
          for (int c0 = 0; c0 < DH; c0 += 16) {
            uint32_t o[16];
            tmem_ld_x16(trow + kTmemO + bb * D + hf * DH + c0, o);
            tmem_wait_ld(o);
            store_row16(dst + c0, o, oscale);
          }
          if (!TRANSPOSED && hf == 0 && p.lse)
            p.lse[orow] = exact ? p.logZ[(size_t)w.hs * T + trow_i] : lse_i;
        }
        tc_fence_before();
        mbar_arrive(o_empty);
        ++oc;
      }
    }
  }

  // ------------------------------------------------------------ teardown
  // every tensor store issued must have completed before the CTA exits
  if (L::OSTAGE && !TRANSPOSED && warp == 4 && lane == 0) bulk_wait_group0();
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool TRANSPOSED>
cudaError_t launch_fused(const FwdLaunch& L, cudaStream_t s) {
  using S = FwdSmem<D>;
  auto kern = hybrid_fwd_kernel<D, TRANSPOSED>;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), S::ALLOC);
  if (e != cudaSuccess) return e;
  if (L.p.n_items == 0) return cudaSuccess;
  const int grid = L.p.n_items < L.num_sms ? L.p.n_items : L.num_sms;
  trace_begin(s);
  kern<<<grid, 384, S::ALLOC, s>>>(L.tm_q, L.tm_k, L.tm_v, L.tm_o, L.p);
  trace_end(s, TRANSPOSED ? "static_dv" : "hybrid_fwd");
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_hybrid_fwd(const FwdLaunch& L, cudaStream_t s) {
  switch (L.d_h) {
    case 32: return L.transposed ? launch_fused<32, true>(L, s) : launch_fused<32, false>(L, s);
    case 64: return L.transposed ? launch_fused<64, true>(L, s) : launch_fused<64, false>(L, s);
    case 128:
      return L.transposed ? launch_fused<128, true>(L, s) : launch_fused<128, false>(L, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace saf
