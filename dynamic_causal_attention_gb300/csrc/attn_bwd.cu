// attn_bwd.cu — backward of the SAF hybrid layer: dynamic heads, and the
// alpha/rho gradients of frozen heads.
//
// ("When Can Attention Heads Be Statically Defined?", close-reading notes:
// dynamic heads keep the ordinary attention backward; a frozen head's
// attention backward is only dV = P^T dZ, §3.3 / App. D.2 — that part reuses
// the forward's static engine, transposed.  The alpha/rho gradients are an
// extension: the chain rule through Eq. (3).)
//
// bwd_dynamic_kernel (K4): one persistent launch over items (b, h, J), J a
// 128-row key tile, longest first.  Per item K_J and V_J stay in shared
// memory and dK_J, dV_J accumulate in TMEM while the query tiles I = J..nI-1
// stream through:
//     S^T  = K_J Q_I^T,  dP^T = V_J dO_I^T           (tcgen05, fp32 in TMEM)
//     P^T  = exp2(S^T * log2e/sqrt(d) - lse2(i)),   dS^T = P^T * (dP^T - D(i))
//                                                   (compute warps, 1 row/thread)
//     dV_J += P^T dO_I,  dK_J += dS^T Q_I           (tcgen05, A operand in TMEM)
//     dQ_I  = dS K_J                                (tcgen05, dS^T tile in smem
//                                                    read as an MN-major A)
// d_h <= 64: P^T goes, as packed bf16, to spare TMEM columns (dV is a TS MMA)
// and dS^T to one of two swizzled shared-memory tiles (dK and dQ are SS MMAs).
// d_h = 128: TMEM has no spare columns, so P^T and dS^T are written, packed,
// over the S^T columns just read (dV and dK are TS MMAs), dS^T also goes to
// shared memory for dQ, and dQ goes over the dP^T columns.  dQ_I is read from
// TMEM by a second warpgroup and added into an fp32 accumulator (zeroed by the
// pre-pass) with one TMA tensor reduce-add per 32 columns: staged in a tile of
// its own for d_h <= 64, in the step's own Q_I/dO_I stage (once dV and dK have
// read it) for d_h = 128.  A post-pass scales it by 1/sqrt(d) and converts it.
//
// param_grad_kernel (K5): items (h_static, J), handed out in snake order.
// For I = J..nI-1 the batch-summed dP^T(j, i) = sum_b V_b(j) . dO_b(i) is one
// MMA chain with K = B*d; eight compute warps (a 32-row group x a 64-column
// half each) form dl = P(i,j) (dP - sum_b D_b(i)) with P(i,j) rebuilt from the
// static tables and keep the row sums (alpha) in registers.  For the diagonal
// sums (rho) each warp writes its 32 x 32 block of dl to shared memory by
// diagonal, so that lane q adds up diagonals q and q + 32 with vector loads,
// and adds its three distance sums of the tile to global with atomics (no
// barrier across the warps per tile).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn_common.cuh"
#include "attn_kernels.h"
#include "internal.h"

namespace saf {
namespace {

constexpr uint32_t kTmemCols = 512;

template <int D>
struct BwdSmem {
  using G = TileGeom<D>;
  // d_h = 128 leaves no free TMEM columns: dQ goes over the dP^T columns once
  // the compute has read them, and P^T and dS^T over the S^T columns.
  static constexpr bool DQ_ALIAS = (256 + 3 * D > 512);
  // d_h <= 64: P^T goes to spare TMEM columns (TS MMA for dV) and dS^T to
  // shared memory (SS MMAs for dK, dQ), so the S^T/dP^T columns are free as
  // soon as the compute warps have loaded them and the next step's scores
  // overlap this step's softmax.  d_h = 128 writes P^T and dS^T packed over
  // the S^T columns (TS MMAs for dV, dK); dS^T also goes to shared memory.
  static constexpr bool PS = !DQ_ALIAS;
  // Q_I, dO_I stages; d_h = 128 keeps two stages by dropping the alignment
  // slack (the dynamic shared base is checked at run time instead).
  static constexpr int QST = (D == 128) ? 2 : 3;
  static constexpr int STAGE = 2 * G::TILE_BYTES + 1024;  // Q_I, dO_I, -lse2[128], -D[128]
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + G::TILE_BYTES;
  static constexpr int OFF_Q = OFF_V + G::TILE_BYTES;
  static constexpr int OFF_DST = OFF_Q + QST * STAGE;
  // dQ staging for the tensor reduce-add (d_h <= 64): one [128 rows x 128 B]
  // chunk (32 fp32 columns), 128-byte swizzled, reused for each chunk of the
  // row.  d_h = 128 stages dQ (64 KB) in its step's own Q_I/dO_I stage, whose
  // 64 KB of tiles are free once dK and dV have read them.
  static constexpr bool DQ_TMA = (D <= 64);
  static constexpr int DQS_BYTES = DQ_TMA ? 128 * 32 * 4 : 0;
  // PS: two dS^T tiles, used by alternate steps
  static constexpr int DST_BUFS = PS ? 2 : 1;
  static constexpr int OFF_DQS = OFF_DST + DST_BUFS * SqTile::BYTES;
  static constexpr int OFF_BAR = OFF_DQS + DQS_BYTES;
  static constexpr int NBAR = 2 + 2 * QST + 16;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int SLACK = (BYTES + 1024 <= 232448) ? 1024 : 0;
  static constexpr int ALLOC = BYTES + SLACK;
  static_assert(ALLOC <= 232448, "shared memory budget exceeded");
  // TMEM columns.  S^T (fp32) at 0, dP^T at 128, then dV and dK.
  // d_h = 128: compute half hf reads the groups of 32 query columns
  // 32hf..32hf+31 and 64+32hf..64+32hf+31 of S^T and dP^T; into each S^T
  // group, once read, it writes the group's P^T packed as bf16 pairs (16
  // columns) and then its dS^T (the other 16).  The whole dP^T region is then
  // free, and dQ (one N = 128 product) goes there.
  static constexpr uint32_t T_S = 0, T_DP = 128;
  static constexpr uint32_t T_DV = 256, T_DK = 256 + D;
  static constexpr uint32_t T_DQ = (D == 128) ? T_DP : 256 + 2 * D;
  // PS: P^T as packed bf16 (query columns 2c, 2c+1 in column T_PT + c), the
  // TMEM A operand of dV; 64 columns, free for d_h <= 64.
  static constexpr uint32_t T_PT = 256 + 3 * D;
  static_assert(!PS || T_PT + 64 <= 512, "P^T does not fit in TMEM");
  // d_h = 128: packed P^T column of the k-step kk (query columns
  // 16kk..16kk+15), in the S^T group of 32 columns that holds them (half
  // (kk >> 1) & 1, group kk >> 2); dS^T of the same k-step 16 columns on.
  __device__ static __forceinline__ uint32_t a_col(int kk) {
    return (uint32_t)(32 * ((kk >> 1) & 1) + 64 * (kk >> 2) + 8 * (kk & 1));
  }
  static constexpr uint32_t DS_OFF = 16;
};

enum : int {
  kSiteBProdKV = 101, kSiteBProdQ, kSiteBMmaKV, kSiteBMmaQ, kSiteBMmaS, kSiteBMmaP, kSiteBMmaKD,
  kSiteBMmaDQ, kSiteBCmpQ, kSiteBCmpS, kSiteBCmpP, kSiteBCmpKD, kSiteBDq, kSiteBMmaTS,
  kSiteBAlign
};

// Item (b, K/V head kv, key tile J): the query tiles I = J..nI-1 of every
// dynamic query head that K/V head serves, head by head; dK_J and dV_J
// collect all of them.
struct BItem {
  int b, kv, J, span, db, nsteps;  // span = nI - J query tiles per head
};

// Items come in groups of p.pairs_per_group (sequence, K/V head) pairs, the
// groups one after another and, inside a group, key tile by key tile
// (longest first).  The CTAs running at any time then add into the dQ rows of
// a few groups only, a working set that stays in L2 (the TMA reduce-adds run
// at about half speed once their target falls out of L2); across the whole
// list the item lengths still cycle from long to short for the snake order.
__device__ __forceinline__ BItem decode_bwd(const BwdParams& p, int it) {
  BItem r;
  const int n_pairs = p.B * p.n_kv;
  const int G = p.pairs_per_group;
  const int full = n_pairs / G;                          // complete groups
  const int per_full = G * p.nI;
  int pair;
  if (it < full * per_full) {
    const int g = it / per_full, w = it - g * per_full;
    r.J = w / G;
    pair = g * G + (w - r.J * G);
  } else {
    const int gs = n_pairs - full * G;                   // the last, smaller group
    const int w = it - full * per_full;
    r.J = w / gs;
    pair = full * G + (w - r.J * gs);
  }
  r.b = pair / p.n_kv;
  r.kv = p.kv_list[pair - r.b * p.n_kv];
  r.span = p.nI - r.J;
  r.db = p.dyn_begin[r.kv];
  r.nsteps = p.dyn_count[r.kv] * r.span;
  return r;
}

// Query head and query tile of step t of an item.
__device__ __forceinline__ void step_of(const BwdParams& p, const BItem& w, int t, int& hq,
                                        int& I) {
  const int q = t / w.span;
  hq = p.dyn_by_kv[w.db + q];
  I = w.J + (t - q * w.span);
}

// Threads: warp 0 TMA producer, warp 1 MMA issuer (for d_h <= 64 only the
// S^T/dP^T products; warp 3 issues dV, dK and dQ), warp 2 TMEM owner,
// warps 4..11 two compute halves (query columns 0..63 and 64..127 of every
// key row; a row per thread), warps 12..15 the dQ warps.
template <int D>
__global__ void __launch_bounds__(512, 1)
    bwd_dynamic_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using G = TileGeom<D>;
  using L = BwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  if (L::SLACK == 0 && smem != smem_raw) {
    // no room to realign: report and leave without touching anything
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kSiteBAlign);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* q_full = bars + 2;
  uint64_t* q_empty = q_full + L::QST;
  uint64_t* s_full = q_empty + L::QST;   // S^T, dP^T ready
  uint64_t* p_full = s_full + 1;         // P^T, dS^T written (TMEM + smem)
  uint64_t* p_empty = p_full + 1;        // the dS^T smem tile is free again
  uint64_t* dq_full = p_empty + 1;
  uint64_t* dq_empty = dq_full + 1;
  uint64_t* kd_full = dq_empty + 1;
  uint64_t* kd_empty = kd_full + 1;
  uint64_t* s_free = kd_empty + 1;       // S^T, dP^T loaded by the compute warps (PS)
  uint64_t* pt_empty = s_free + 1;       // the P^T columns are free again (PS)
  uint64_t* p_empty2 = pt_empty + 1;     // PS: dS^T tile 1 free again (tile 0: p_empty)
  uint64_t* dp_full = p_empty2 + 1;      // DQ_ALIAS: dP^T ready (s_full: S^T ready)
  // DQ_ALIAS: the step's dV has read P^T and dO (dk_done: dK, dS^T and Q)
  uint64_t* dv_done = dp_full + 1;
  uint64_t* dk_done = dv_done + 1;
  // DQ_ALIAS: p_full is the first group of query columns of both compute
  // halves done (P^T and dS^T in TMEM), p_full1 the second (and the dS^T tile)
  uint64_t* p_full1 = dk_done + 1;
  // per MMA-issuing warp (1, 3): all its products done, before TMEM is freed
  uint64_t* mma_drained = p_full1 + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  const WaitCtl wc{abort_flag, p.status};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int s = 0; s < L::QST; ++s) { mbar_init(q_full + s, 1); mbar_init(q_empty + s, 1); }
    mbar_init(s_full, 1);
    mbar_init(p_full, 256);
    mbar_init(p_empty, 1);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128);
    mbar_init(kd_full, 1);
    mbar_init(kd_empty, 256);
    mbar_init(s_free, 256);
    mbar_init(pt_empty, 1);
    mbar_init(p_empty2, 1);
    mbar_init(dp_full, 1);
    mbar_init(dv_done, 1);
    mbar_init(dk_done, 1);
    mbar_init(p_full1, 256);
    mbar_init(mma_drained, 1);
    mbar_init(mma_drained + 1, 1);
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
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sK = smem_u32(smem + L::OFF_K);
  const uint32_t sV = smem_u32(smem + L::OFF_V);
  const uint32_t sDST = smem_u32(smem + L::OFF_DST);
  const int H = p.H, T = p.T;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    // Lane 0 waits for the buffer and posts the expected bytes; then one lane
    // per tile chunk issues its copy (one issuing thread moves about 29 bytes
    // per clock from L2, four about 74) and two more the -lse/-D vectors.
    uint32_t kvc = 0, qc = 0;
    for (int kr = 0, it = snake_item(0, blockIdx.x, gridDim.x); it < p.n_items;
         it = snake_item(++kr, blockIdx.x, gridDim.x)) {
      const BItem w = decode_bwd(p, it);
      const int kvrow0 = (w.b * p.H_kv + w.kv) * T;
      if (lane == 0) {
        mbar_wait(kv_empty, (kvc & 1) ^ 1, wc, kSiteBProdKV);
        mbar_arrive_expect_tx(kv_full, 2 * G::TILE_BYTES);
      }
      __syncwarp();
      ++kvc;
      if (lane < 2 * G::NCHUNK) {
        const int c = lane >> 1;
        if (lane & 1)
          tma_load_2d(smem + L::OFF_V + c * G::CHUNK_BYTES, &tm_v, kv_full, c * G::CHUNK,
                      kvrow0 + w.J * 128);
        else
          tma_load_2d(smem + L::OFF_K + c * G::CHUNK_BYTES, &tm_k, kv_full, c * G::CHUNK,
                      kvrow0 + w.J * 128);
      }
      for (int t = 0; t < w.nsteps; ++t) {
        int hq, I;
        step_of(p, w, t, hq, I);
        const int row0 = (w.b * H + hq) * T;
        const int qs = qc % L::QST;
        if (lane == 0) {
          mbar_wait(q_empty + qs, ((qc / L::QST) & 1) ^ 1, wc, kSiteBProdQ);
          mbar_arrive_expect_tx(q_full + qs, 2 * G::TILE_BYTES + 1024);
        }
        __syncwarp();
        ++qc;
        uint8_t* st = smem + L::OFF_Q + qs * L::STAGE;
        if (lane < 2 * G::NCHUNK) {
          const int c = lane >> 1;
          if (lane & 1)
            tma_load_2d(st + G::TILE_BYTES + c * G::CHUNK_BYTES, &tm_do, q_full + qs,
                        c * G::CHUNK, row0 + I * 128);
          else
            tma_load_2d(st + c * G::CHUNK_BYTES, &tm_q, q_full + qs, c * G::CHUNK,
                        row0 + I * 128);
        } else if (lane == 2 * G::NCHUNK) {
          bulk_load(st + 2 * G::TILE_BYTES, p.lse2 + row0 + I * 128, 512, q_full + qs);
        } else if (lane == 2 * G::NCHUNK + 1) {
          bulk_load(st + 2 * G::TILE_BYTES + 512, p.Dvec + row0 + I * 128, 512, q_full + qs);
        }
      }
    }
    if (lane == 0) {
      if (kvc > 0) mbar_drain(kv_full, (kvc - 1) & 1);
      for (int s = 0; s < L::QST; ++s)
        if (qc > (uint32_t)s) mbar_drain(q_full + s, ((qc - 1 - s) / L::QST) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t id_acc = idesc_bf16(128, D, false, true);
      uint32_t kvc = 0, qc = 0, pc = 0, dqc = 0, kdc = 0;
      // S^T and dP^T of the step whose Q/dO sit in stage `qs_of`.
      auto issue_s = [&](uint32_t qcount) {
        const int qs = qcount % L::QST;
        mbar_wait(q_full + qs, (qcount / L::QST) & 1, wc, kSiteBMmaQ);
        tc_fence_after();
        const uint32_t sQ = smem_u32(smem + L::OFF_Q + qs * L::STAGE);
        const uint32_t sDO = sQ + G::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < G::KSTEPS; ++kk)
          mma_bf16_ss(tmem + L::T_S, G::kmajor_desc(sK, kk), G::kmajor_desc(sQ, kk), id_s,
                      kk > 0);
#pragma unroll
        for (int kk = 0; kk < G::KSTEPS; ++kk)
          mma_bf16_ss(tmem + L::T_DP, G::kmajor_desc(sV, kk), G::kmajor_desc(sDO, kk), id_s,
                      kk > 0);
        mma_commit(s_full);
      };
      // DQ_ALIAS: S^T and dP^T issued separately (same stage).
      auto issue_st = [&](uint32_t qcount) {
        const int qs = qcount % L::QST;
        mbar_wait(q_full + qs, (qcount / L::QST) & 1, wc, kSiteBMmaQ);
        tc_fence_after();
        const uint32_t sQ = smem_u32(smem + L::OFF_Q + qs * L::STAGE);
#pragma unroll
        for (int kk = 0; kk < G::KSTEPS; ++kk)
          mma_bf16_ss(tmem + L::T_S, G::kmajor_desc(sK, kk), G::kmajor_desc(sQ, kk), id_s,
                      kk > 0);
        mma_commit(s_full);
      };
      auto issue_dpt = [&](uint32_t qcount) {
        const int qs = qcount % L::QST;
        mbar_wait(q_full + qs, (qcount / L::QST) & 1, wc, kSiteBMmaQ);
        tc_fence_after();
        const uint32_t sDO = smem_u32(smem + L::OFF_Q + qs * L::STAGE) + G::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < G::KSTEPS; ++kk)
          mma_bf16_ss(tmem + L::T_DP, G::kmajor_desc(sV, kk), G::kmajor_desc(sDO, kk), id_s,
                      kk > 0);
        mma_commit(dp_full);
      };
      uint32_t sfc = 0;
      if constexpr (L::PS) {
        // S^T and dP^T only; warp 3 issues dV, dK and dQ.
        for (int kr = 0, it = snake_item(0, blockIdx.x, gridDim.x); it < p.n_items;
         it = snake_item(++kr, blockIdx.x, gridDim.x)) {
          const BItem w = decode_bwd(p, it);
          mbar_wait(kv_full, kvc & 1, wc, kSiteBMmaKV);
          ++kvc;
          // the previous item's last S^T/dP^T must have been loaded
          if (it != (int)blockIdx.x) {
            mbar_wait(s_free, sfc & 1, wc, kSiteBMmaS);
            ++sfc;
          }
          issue_s(qc);
          ++qc;
          for (int t = 0; t + 1 < w.nsteps; ++t) {
            // next step's scores as soon as this step's are in registers
            mbar_wait(s_free, sfc & 1, wc, kSiteBMmaS);
            ++sfc;
            issue_s(qc);
            ++qc;
          }
        }
      }
      // d_h = 128, per step: once the compute's first group of query columns
      // is in TMEM, dV and dK over its k-steps; once the second is, dQ (one
      // N = 128 product into the dP^T columns the compute has read) and the
      // rest of dV and dK.  The next step's S^T goes out once
      // dK has completed (dV and dK read P^T and dS^T from the S^T columns;
      // this warp's products complete in issue order, so the wait only makes
      // the order explicit), its dP^T once the dQ warps have taken dQ out of
      // TMEM; the reduce-adds of dQ then run while the next step computes.
      constexpr uint32_t id_dq = idesc_bf16(128, 128, true, true);
      uint32_t dkc = 0;
      for (int kr = 0, it = snake_item(0, blockIdx.x, gridDim.x); !L::PS && it < p.n_items;
           it = snake_item(++kr, blockIdx.x, gridDim.x)) {
        const BItem w = decode_bwd(p, it);
        mbar_wait(kv_full, kvc & 1, wc, kSiteBMmaKV);
        ++kvc;
        if (dkc > 0) mbar_wait(dk_done, (dkc - 1) & 1, wc, kSiteBMmaTS);
        issue_st(qc);
        if (dqc > 0) mbar_wait(dq_empty, (dqc - 1) & 1, wc, kSiteBMmaDQ);
        issue_dpt(qc);
        for (int t = 0; t < w.nsteps; ++t) {
          const int qs = qc % L::QST;
          const uint32_t sQ = smem_u32(smem + L::OFF_Q + qs * L::STAGE);
          const uint32_t sDO = sQ + G::TILE_BYTES;
          // dV and dK over the k-steps of the first group of query columns
          // (0..63) while the compute works on the second
          mbar_wait(p_full, pc & 1, wc, kSiteBMmaP);
          if (t == 0) mbar_wait(kd_empty, (kdc & 1) ^ 1, wc, kSiteBMmaKD);
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ts(tmem + L::T_DV, tmem + L::T_S + L::a_col(kk), G::mnmajor_desc(sDO, kk),
                        id_acc, (t > 0 || kk > 0));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ts(tmem + L::T_DK, tmem + L::T_S + L::a_col(kk) + L::DS_OFF,
                        G::mnmajor_desc(sQ, kk), id_acc, (t > 0 || kk > 0));
          mbar_wait(p_full1, pc & 1, wc, kSiteBMmaP);
          tc_fence_after();
          // dQ_I = dS K_J: A the dS^T tile (MN-major), B K_J (MN-major)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ss(tmem + L::T_DQ, SqTile::mnmajor_desc(sDST, kk), G::mnmajor_desc(sK, kk),
                        id_dq, kk > 0);
          mma_commit(dq_full);
          ++dqc;
#pragma unroll
          for (int kk = 4; kk < 8; ++kk)
            mma_bf16_ts(tmem + L::T_DV, tmem + L::T_S + L::a_col(kk), G::mnmajor_desc(sDO, kk),
                        id_acc, true);
          mma_commit(dv_done);
#pragma unroll
          for (int kk = 4; kk < 8; ++kk)
            mma_bf16_ts(tmem + L::T_DK, tmem + L::T_S + L::a_col(kk) + L::DS_OFF,
                        G::mnmajor_desc(sQ, kk), id_acc, true);
          mma_commit(dk_done);
          ++dkc;
          // (the dQ warps stage dQ in this stage and then release it)
          ++qc;
          ++pc;
          if (t + 1 < w.nsteps) {
            mbar_wait(dk_done, (dkc - 1) & 1, wc, kSiteBMmaTS);      // P^T, dS^T read
            issue_st(qc);
            mbar_wait(dq_empty, (dqc - 1) & 1, wc, kSiteBMmaDQ);     // dQ out of TMEM
            issue_dpt(qc);
          }
        }
        mma_commit(kd_full);
        mma_commit(kv_empty);
        ++kdc;
      }
      // every product of this warp has completed before TMEM is freed (after
      // an abort no later wait guarantees it)
      mma_commit(mma_drained);
      mbar_drain(mma_drained, 0);
    }
  } else if (warp == 3) {
    // ---------------------------------------------------------- dV/dK/dQ issuer (PS)
    if (L::PS && lane == 0) {
      constexpr uint32_t id_acc = idesc_bf16(128, D, false, true);
      constexpr uint32_t id_dq = idesc_bf16(128, D, true, true);
      uint32_t kvc = 0, qc = 0, pc = 0, dqc = 0, kdc = 0;
      for (int kr = 0, it = snake_item(0, blockIdx.x, gridDim.x); it < p.n_items;
         it = snake_item(++kr, blockIdx.x, gridDim.x)) {
        const BItem w = decode_bwd(p, it);
        mbar_wait(kv_full, kvc & 1, wc, kSiteBMmaKV);  // K_J is the B operand of dQ
        ++kvc;
        for (int t = 0; t < w.nsteps; ++t) {
          const int qs = qc % L::QST;
          const uint32_t sQ = smem_u32(smem + L::OFF_Q + qs * L::STAGE);
          const uint32_t sDO = sQ + G::TILE_BYTES;
          const uint32_t sDSTb = sDST + (pc & 1) * SqTile::BYTES;  // this step's dS^T tile
          mbar_wait(p_full, pc & 1, wc, kSiteBMmaP);
          if (t == 0) mbar_wait(kd_empty, (kdc & 1) ^ 1, wc, kSiteBMmaKD);
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ts(tmem + L::T_DV, tmem + L::T_PT + 8 * kk, G::mnmajor_desc(sDO, kk),
                        id_acc, (t > 0 || kk > 0));
          mma_commit(pt_empty);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ss(tmem + L::T_DK, SqTile::kmajor_desc(sDSTb, kk), G::mnmajor_desc(sQ, kk),
                        id_acc, (t > 0 || kk > 0));
          mma_commit(q_empty + qs);  // S^T/dP^T of this stage completed before p_full
          ++qc;
          mbar_wait(dq_empty, (dqc & 1) ^ 1, wc, kSiteBMmaDQ);
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ss(tmem + L::T_DQ, SqTile::mnmajor_desc(sDSTb, kk), G::mnmajor_desc(sK, kk),
                        id_dq, kk > 0);
          mma_commit((pc & 1) ? p_empty2 : p_empty);
          ++pc;
          mma_commit(dq_full);
          ++dqc;
        }
        mma_commit(kd_full);
        mma_commit(kv_empty);  // the item's S^T/dP^T all completed before its last p_full
        ++kdc;
      }
      mma_commit(mma_drained + 1);  // every product of this warp done before TMEM is freed
      mbar_drain(mma_drained + 1, 0);
    }
  } else if (warp >= 4 && warp < 12) {
    // ---------------------------------------------------------- compute halves
    const int hf = (warp - 4) >> 2;          // query columns 64*hf .. 64*hf + 63
    const int r = (warp & 3) * 32 + lane;    // key row j within the tile == TMEM lane
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
    uint32_t qc = 0, sc = 0, pc = 0, kdc = 0;
    for (int kr = 0, it = snake_item(0, blockIdx.x, gridDim.x); it < p.n_items;
         it = snake_item(++kr, blockIdx.x, gridDim.x)) {
      const BItem w = decode_bwd(p, it);
      for (int t = 0; t < w.nsteps; ++t) {
        const int qs = qc % L::QST;
        mbar_wait(q_full + qs, (qc / L::QST) & 1, wc, kSiteBCmpQ);
        const float* nl_s = reinterpret_cast<const float*>(smem + L::OFF_Q + qs * L::STAGE +
                                                           2 * G::TILE_BYTES) + 64 * hf;
        const uint32_t nl_a = smem_u32(nl_s);  // -lse2 at +0, -D at +512 bytes
        mbar_wait(s_full, sc & 1, wc, kSiteBCmpS);
        tc_fence_after();
        const bool diag = (t % w.span == 0);  // I == J: the causal diagonal
        if constexpr (L::PS) {
          // Four 16-column chunks; the TMEM loads of chunk k + 1 are issued
          // right after chunk k's have landed, so they fly while chunk k is
          // computed (tcgen05.wait::ld waits for every load in flight).
          uint32_t sv[2][16], dv[2][16];
          const uint32_t sDSTb = sDST + (pc & 1) * SqTile::BYTES;  // this step's dS^T tile
          tmem_ld_x16(trow + L::T_S + 64 * hf, sv[0]);
          tmem_ld_x16(trow + L::T_DP + 64 * hf, dv[0]);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int b = k & 1;
            const int col = 64 * hf + 16 * k;  // first query column of this chunk
            tmem_wait_ld(sv[b]);
            tmem_wait_ld(dv[b]);
            if (k + 1 < 4) {
              tmem_ld_x16(trow + L::T_S + col + 16, sv[b ^ 1]);
              tmem_ld_x16(trow + L::T_DP + col + 16, dv[b ^ 1]);
            } else {
              // every S^T/dP^T column this thread reads is in registers
              tc_fence_before();
              mbar_arrive(s_free);
            }
            if (diag) {
              // causal mask of the diagonal tile: query column < key row
#pragma unroll
              for (int e = 0; e < 16; ++e)
                if (col + e < r) sv[b][e] = 0xff800000u;  // -inf: P = 0, dS = 0
            }
            uint32_t pk[8], dk[8];
#pragma unroll
            for (int k4 = 0; k4 < 16; k4 += 4) {
              const float4 nl = lds_f32x4(nl_a + 4u * (16 * k + k4));
              const float4 nd = lds_f32x4(nl_a + 512u + 4u * (16 * k + k4));
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                const int e = k4 + 2 * h2;
                const float l0 = h2 ? nl.z : nl.x, l1 = h2 ? nl.w : nl.y;
                const float e0 = h2 ? nd.z : nd.x, e1 = h2 ? nd.w : nd.y;
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[b][e]), __uint_as_float(sv[b][e + 1])),
                                 sc2, f2_pack(l0, l1)),
                          x0, x1);
                const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                const uint64_t g2 = f2_mul(
                    f2_pack(p0, p1),
                    f2_add(f2_pack(__uint_as_float(dv[b][e]), __uint_as_float(dv[b][e + 1])),
                           f2_pack(e0, e1)));
                pk[e >> 1] = pack_bf16x2(p0, p1);
                dk[e >> 1] = pack_bf16x2_f2(g2);
              }
            }
            if (k == 0) {
              // P^T goes to TMEM, read there by the previous step's dV first;
              // this dS^T tile was last read by dK and dQ two steps back
              mbar_wait(pt_empty, (pc & 1) ^ 1, wc, kSiteBCmpP);
              mbar_wait((pc & 1) ? p_empty2 : p_empty, ((pc >> 1) & 1) ^ 1, wc, kSiteBCmpP);
              tc_fence_after();
            }
            tmem_st_x8(trow + L::T_PT + (uint32_t)(col >> 1), pk);
#pragma unroll
            for (int u = 0; u < 2; ++u)
              st_shared_v4(SqTile::unit_addr(sDSTb, r, (uint32_t)(col >> 3) + u), dk[4 * u],
                           dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
          }
          tmem_wait_st();
        }
#pragma unroll 1
        for (int c0 = 0; !L::PS && c0 < 64; c0 += 32) {
          // this half's query columns: 32hf..32hf+31, then 64+32hf..64+32hf+31
          const int col = 32 * hf + 2 * c0;  // first query column of this chunk
          const float* nlc = nl_s - 64 * hf + col;   // -lse2 of these columns
          const float* ndc = nlc + 128;               // -D of these columns
          // P from S^T first (dP^T may still be on its way), then dS
          uint32_t sv[32], pk[16], dk[16];
          tmem_ld_x32(trow + L::T_S + col, sv);
          tmem_wait_ld(sv);
#pragma unroll
          for (int k4 = 0; k4 < 32; k4 += 4) {
            const float4 nl = *reinterpret_cast<const float4*>(nlc + k4);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int k = k4 + 2 * h2;
              const float l0 = h2 ? nl.z : nl.x, l1 = h2 ? nl.w : nl.y;
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[k]), __uint_as_float(sv[k + 1])), sc2,
                               f2_pack(l0, l1)),
                        x0, x1);
              float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              if (diag) {
                if (col + k < r) p0 = 0.f;
                if (col + k + 1 < r) p1 = 0.f;
              }
              sv[k] = __float_as_uint(p0);  // P kept in fp32 for dS
              sv[k + 1] = __float_as_uint(p1);
              pk[k >> 1] = pack_bf16x2(p0, p1);
            }
          }
          // P^T over the first 16 of the S^T columns just read (TMEM A
          // operand of dV)
          tmem_st_x16(trow + L::T_S + col, pk);
          if (c0 == 0 && L::DQ_ALIAS) {
            mbar_wait(dp_full, sc & 1, wc, kSiteBCmpS);
            tc_fence_after();
          }
          uint32_t dv[32];
          tmem_ld_x32(trow + L::T_DP + col, dv);
          tmem_wait_ld(dv);
#pragma unroll
          for (int k4 = 0; k4 < 32; k4 += 4) {
            const float4 nd = *reinterpret_cast<const float4*>(ndc + k4);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int k = k4 + 2 * h2;
              const float e0 = h2 ? nd.z : nd.x, e1 = h2 ? nd.w : nd.y;
              const uint64_t g2 = f2_mul(
                  f2_pack(__uint_as_float(sv[k]), __uint_as_float(sv[k + 1])),
                  f2_add(f2_pack(__uint_as_float(dv[k]), __uint_as_float(dv[k + 1])),
                         f2_pack(e0, e1)));
              dk[k >> 1] = pack_bf16x2_f2(g2);
            }
          }
          // dS^T over the other 16 of them (A operand of dK), and into
          // shared memory for dQ
          tmem_st_x16(trow + L::T_S + col + L::DS_OFF, dk);
          // the dS^T tile in shared memory was read by the previous step's
          // dQ, which completed before this step's S^T (one issuing thread,
          // so s_full's commit covers it)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t unit = (uint32_t)(col >> 3) + u;
            st_shared_v4(SqTile::unit_addr(sDST, r, unit), dk[4 * u], dk[4 * u + 1],
                         dk[4 * u + 2], dk[4 * u + 3]);
          }
          if (c0 == 0) {
            // the first group's P^T and dS^T are in TMEM: dV and dK take
            // their k-steps 0..3 while this thread does the second group
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(p_full);
          }
        }
        if constexpr (!L::PS) tmem_wait_st();
        tc_fence_before();
        fence_proxy_async_smem();
        mbar_arrive(L::PS ? p_full : p_full1);
        ++qc;
        ++sc;
        ++pc;
      }
      // epilogue: half 0 writes dV_J, half 1 writes dK_J (scaled)
      mbar_wait(kd_full, kdc & 1, wc, kSiteBCmpKD);
      tc_fence_after();
      const size_t orow = (size_t)(w.b * p.H_kv + w.kv) * T + (size_t)w.J * 128 + r;
      __nv_bfloat16* dst = (hf == 0 ? p.dV : p.dK) + orow * D;
      // frozen query heads of this K/V head added their dV in fp32 beforehand
      const float* addv =
          (hf == 0 && p.dv_acc && p.kv_has_static[w.kv]) ? p.dv_acc + orow * D : nullptr;
      const float sc_out = hf == 0 ? 1.0f : p.scale;
      const uint32_t colb = hf == 0 ? L::T_DV : L::T_DK;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 16) {
        uint32_t o[16];
        tmem_ld_x16(trow + colb + c0, o);
        tmem_wait_ld(o);
        if (addv) {
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            const float4 a = *reinterpret_cast<const float4*>(addv + c0 + e);
            o[e] = __float_as_uint(__uint_as_float(o[e]) + a.x);
            o[e + 1] = __float_as_uint(__uint_as_float(o[e + 1]) + a.y);
            o[e + 2] = __float_as_uint(__uint_as_float(o[e + 2]) + a.z);
            o[e + 3] = __float_as_uint(__uint_as_float(o[e + 3]) + a.w);
          }
        }
        uint4 v0, v1;
        v0.x = pack_bf16x2(__uint_as_float(o[0]) * sc_out, __uint_as_float(o[1]) * sc_out);
        v0.y = pack_bf16x2(__uint_as_float(o[2]) * sc_out, __uint_as_float(o[3]) * sc_out);
        v0.z = pack_bf16x2(__uint_as_float(o[4]) * sc_out, __uint_as_float(o[5]) * sc_out);
        v0.w = pack_bf16x2(__uint_as_float(o[6]) * sc_out, __uint_as_float(o[7]) * sc_out);
        v1.x = pack_bf16x2(__uint_as_float(o[8]) * sc_out, __uint_as_float(o[9]) * sc_out);
        v1.y = pack_bf16x2(__uint_as_float(o[10]) * sc_out, __uint_as_float(o[11]) * sc_out);
        v1.z = pack_bf16x2(__uint_as_float(o[12]) * sc_out, __uint_as_float(o[13]) * sc_out);
        v1.w = pack_bf16x2(__uint_as_float(o[14]) * sc_out, __uint_as_float(o[15]) * sc_out);
        *reinterpret_cast<uint4*>(dst + c0) = v0;
        *reinterpret_cast<uint4*>(dst + c0 + 8) = v1;
      }
      tc_fence_before();
      mbar_arrive(kd_empty);
      ++kdc;
    }
  } else if (warp >= 12) {
    // ---------------------------------------------------------- dQ warps
    const int r = (warp & 3) * 32 + lane;  // query row i within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    uint32_t dqc = 0;
    for (int kr = 0, it = snake_item(0, blockIdx.x, gridDim.x); it < p.n_items;
         it = snake_item(++kr, blockIdx.x, gridDim.x)) {
      const BItem w = decode_bwd(p, it);
      for (int t = 0; t < w.nsteps; ++t) {
        int hq, I;
        step_of(p, w, t, hq, I);
        mbar_wait(dq_full, dqc & 1, wc, kSiteBDq);
        tc_fence_after();
        if constexpr (L::DQ_TMA) {
          // TMEM -> registers -> swizzled staging tile -> one tensor
          // reduce-add per 32-column chunk, issued by one thread.
          uint32_t o[D];
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 16)
            tmem_ld_x16(tmem + lane_base + L::T_DQ + c0,
                        *reinterpret_cast<uint32_t(*)[16]>(o + c0));
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 16)
            tmem_wait_ld(*reinterpret_cast<uint32_t(*)[16]>(o + c0));
          tc_fence_before();
          mbar_arrive(dq_empty);
          const uint32_t stg = smem_u32(smem + L::OFF_DQS);
          const int row = (w.b * H + hq) * T + I * 128;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            if (r == 0) bulk_wait_group_read0();  // the staging chunk has been read
            named_bar_sync(6, 128);
#pragma unroll
            for (int u = 0; u < 8; ++u)
              st_shared_v4(stg + sw128_offset(r, (uint32_t)u), o[32 * c + 4 * u],
                           o[32 * c + 4 * u + 1], o[32 * c + 4 * u + 2], o[32 * c + 4 * u + 3]);
            fence_proxy_async_smem();
            named_bar_sync(6, 128);
            if (r == 0) {
              tma_reduce_add_2d(&tm_dq, smem + L::OFF_DQS, c * 32, row);
              bulk_commit_group();
            }
          }
        } else {
          // d_h = 128: dQ is loaded 64 columns at a time and staged in this
          // step's Q_I/dO_I stage, the low half over dO_I once dV has read it
          // and the high half over Q_I once dK has, with one tensor
          // reduce-add per 32-column chunk.  The TMEM columns (the next
          // step's dP^T goes there) are released once both halves are out;
          // waiting for dK first also keeps dk_done (and dv_done) from
          // running two phases ahead of these waits, since the next step's
          // dP^T waits for the release.  The stage goes back to the producer
          // once the reduce-adds have read it.
          const int qs = (int)(dqc % (uint32_t)L::QST);
          const int row = (w.b * H + hq) * T + I * 128;
          const int stage_off = L::OFF_Q + qs * L::STAGE;
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t o[64];
            {
              uint32_t (&o0)[32] = *reinterpret_cast<uint32_t(*)[32]>(o);
              uint32_t (&o1)[32] = *reinterpret_cast<uint32_t(*)[32]>(o + 32);
              const uint32_t src = tmem + lane_base + L::T_DQ + 64u * (uint32_t)hh;
              tmem_ld_x32(src, o0);
              tmem_ld_x32(src + 32, o1);
              tmem_wait_ld(o0);
              tmem_wait_ld(o1);
            }
            mbar_wait(hh ? dk_done : dv_done, dqc & 1, wc, kSiteBDq);
            if (hh) {
              tc_fence_before();
              mbar_arrive(dq_empty);  // all of dQ is out of TMEM
            }
            // low half: dO_I's two 16 KB chunks; high half: Q_I's
            const int half_off = stage_off + (hh ? 0 : G::TILE_BYTES);
            const uint32_t sh = smem_u32(smem + half_off);
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int u = 0; u < 8; ++u)
                st_shared_v4(sh + (uint32_t)c * 16384u + sw128_offset(r, (uint32_t)u),
                             o[32 * c + 4 * u], o[32 * c + 4 * u + 1], o[32 * c + 4 * u + 2],
                             o[32 * c + 4 * u + 3]);
            fence_proxy_async_smem();
            named_bar_sync(6, 128);
            if (r == 0) {
              tma_reduce_add_2d(&tm_dq, smem + half_off, 64 * hh, row);
              tma_reduce_add_2d(&tm_dq, smem + half_off + 16384, 64 * hh + 32, row);
              bulk_commit_group();
            }
          }
          if (r == 0) {
            bulk_wait_group_read0();  // the producer may load the stage again
            mbar_arrive(q_empty + qs);
          }
        }
        ++dqc;
      }
    }
    // every reduction issued must have completed before the CTA exits
    if (r == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ============================================================ K5: dalpha/drho
template <int D>
struct PgSmem {
  using G = TileGeom<D>;
  static constexpr int ST = (D == 128) ? 2 : (D == 64 ? 3 : 4);  // (V_b[J], dO_b[I]) pairs
  static constexpr int STAGE = 2 * G::TILE_BYTES;
  static constexpr int AUX = 2048;                     // col values, D sums, r window
  // Per compute warp, its 32 x 32 block of dl laid out by diagonal: row
  // e = k - rr + 32 (k column, rr row of the block), 36 floats a row.
  static constexpr int SKW_ROW = 36;
  static constexpr int SKW = 64 * SKW_ROW * 4;
  static constexpr int OFF_ST = 0;
  static constexpr int OFF_AUX = OFF_ST + ST * STAGE;
  static constexpr int OFF_SKW = OFF_AUX + 2 * AUX;
  static constexpr int OFF_BAR = OFF_SKW + 8 * SKW;
  static constexpr int NBAR = 2 * ST + 4 + 4 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int ALLOC = OFF_MISC + 16 + 1024;
  static_assert(ALLOC <= 232448, "shared memory budget exceeded");
};

enum : int { kSitePgProd = 201, kSitePgProdAux, kSitePgMma, kSitePgMmaAcc, kSitePgAux, kSitePgAcc };


template <int D>
__global__ void __launch_bounds__(384, 1)
    param_grad_kernel(const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_do, const ParamGradParams p) {
  using G = TileGeom<D>;
  using L = PgSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* st_full = bars;
  uint64_t* st_empty = st_full + L::ST;
  uint64_t* aux_full = st_empty + L::ST;
  uint64_t* aux_empty = aux_full + 2;
  uint64_t* acc_full = aux_empty + 2;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_drained = acc_empty + 2;  // the issuer's products all done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  const WaitCtl wc{abort_flag, p.status};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::ST; ++s) { mbar_init(st_full + s, 1); mbar_init(st_empty + s, 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(aux_full + s, 1);
      mbar_init(aux_empty + s, 8);  // every compute warp has read the slot
      mbar_init(acc_full + s, 1);
      mbar_init(acc_empty + s, 256);
    }
    mbar_init(mma_drained, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  // Cells of the diagonal blocks that no (row, column) pair maps to are read
  // as zeros, and nothing ever writes them.
  {
    float4* z = reinterpret_cast<float4*>(smem + L::OFF_SKW);
    for (int t = threadIdx.x; t < 8 * L::SKW / 16; t += blockDim.x)
      z[t] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int H = p.H, T = p.T, B = p.B;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t sc = 0, ac = 0;
      for (int k = 0;; ++k) {
        const int it = snake_item(k, blockIdx.x, gridDim.x);
        if (it >= p.n_items) break;
        const int J = it / p.n_static, hs = it - J * p.n_static, h = p.static_heads[hs];
        for (int I = J; I < p.nI; ++I) {
          const int as = ac & 1;
          mbar_wait(aux_empty + as, ((ac >> 1) & 1) ^ 1, wc, kSitePgProdAux);
          ++ac;
          uint8_t* aux = smem + L::OFF_AUX + as * L::AUX;
          mbar_arrive_expect_tx(aux_full + as, 2048);
          bulk_load(aux, p.row_tab + (size_t)hs * T + I * 128, 512, aux_full + as);
          bulk_load(aux + 512, p.Dsum + (size_t)hs * T + I * 128, 512, aux_full + as);
          bulk_load(aux + 1024, p.r_tab + (size_t)hs * (T + 128) + (I - J) * 128, 1024,
                    aux_full + as);
          for (int b = 0; b < B; ++b) {
            const int s = sc % L::ST;
            mbar_wait(st_empty + s, ((sc / L::ST) & 1) ^ 1, wc, kSitePgProd);
            ++sc;
            uint8_t* st = smem + L::OFF_ST + s * L::STAGE;
            const int row0 = (b * H + h) * T;                          // dO rows
            const int vrow0 = (b * p.H_kv + h / p.group_kv) * T;      // V rows
            mbar_arrive_expect_tx(st_full + s, 2 * G::TILE_BYTES);
            for (int c = 0; c < G::NCHUNK; ++c) {
              tma_load_2d(st + c * G::CHUNK_BYTES, &tm_v, st_full + s, c * G::CHUNK,
                          vrow0 + J * 128);
              tma_load_2d(st + G::TILE_BYTES + c * G::CHUNK_BYTES, &tm_do, st_full + s,
                          c * G::CHUNK, row0 + I * 128);
            }
          }
        }
      }
      for (int s = 0; s < L::ST; ++s)
        if (sc > (uint32_t)s) mbar_drain(st_full + s, ((sc - 1 - s) / L::ST) & 1);
      for (int s = 0; s < 2; ++s)
        if (ac > (uint32_t)s) mbar_drain(aux_full + s, ((ac - 1 - s) >> 1) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id = idesc_bf16(128, 128, false, false);
      uint32_t sc = 0, cc = 0;
      for (int k = 0;; ++k) {
        const int it = snake_item(k, blockIdx.x, gridDim.x);
        if (it >= p.n_items) break;
        const int J = it / p.n_static;
        for (int I = J; I < p.nI; ++I) {
          const int ab = cc & 1;
          mbar_wait(acc_empty + ab, ((cc >> 1) & 1) ^ 1, wc, kSitePgMmaAcc);
          tc_fence_after();
          for (int b = 0; b < B; ++b) {
            const int s = sc % L::ST;
            mbar_wait(st_full + s, (sc / L::ST) & 1, wc, kSitePgMma);
            tc_fence_after();
            const uint32_t sv = smem_u32(smem + L::OFF_ST + s * L::STAGE);
#pragma unroll
            for (int kk = 0; kk < G::KSTEPS; ++kk)
              mma_bf16_ss(tmem + ab * 128, G::kmajor_desc(sv, kk),
                          G::kmajor_desc(sv + G::TILE_BYTES, kk), id, (b > 0 || kk > 0));
            mma_commit(st_empty + s);
            ++sc;
          }
          mma_commit(acc_full + ab);
          ++cc;
        }
      }
      // every product has completed before TMEM is freed (after an abort no
      // later wait guarantees it)
      mma_commit(mma_drained);
      mbar_drain(mma_drained, 0);
    }
  } else if (warp >= 4) {
    // Warp (rg, hf): key rows r = 32 rg + lane of tile J, query columns
    // 64 hf .. 64 hf + 63 of tile I.
    const int rg = warp & 3, hf = (warp - 4) >> 2, w8 = warp - 4;
    const int r = rg * 32 + lane;
    const uint32_t lane_base = (uint32_t)(rg * 32) << 16;
    float* skw = reinterpret_cast<float*>(smem + L::OFF_SKW + w8 * L::SKW);
    // row lane writes block column k to skw[(k - lane + 32) * 36 + lane]
    float* skw_w = skw + (32 - lane) * L::SKW_ROW + lane;
    // lane q sums the block diagonals e = q and e = q + 32
    const float4* skw_lo = reinterpret_cast<const float4*>(skw + lane * L::SKW_ROW);
    const float4* skw_hi = reinterpret_cast<const float4*>(skw + (lane + 32) * L::SKW_ROW);
    const uint64_t m1 = f2_pack(-1.f, -1.f);
    uint32_t ac = 0, cc = 0;
    for (int k = 0;; ++k) {
      const int it = snake_item(k, blockIdx.x, gridDim.x);
      if (it >= p.n_items) break;
      const int J = it / p.n_static, hs = it - J * p.n_static, h = p.static_heads[hs];
      const bool exact = p.mode[hs] != 0;
      const float rowv = p.a_tab[(size_t)hs * T + J * 128 + r];
      const uint64_t row2 = f2_pack(rowv, rowv);
      uint64_t dal2 = 0;
      for (int I = J; I < p.nI; ++I) {
        const int as = ac & 1;
        mbar_wait(aux_full + as, (ac >> 1) & 1, wc, kSitePgAux);
        const float* aux = reinterpret_cast<const float*>(smem + L::OFF_AUX + as * L::AUX);
        const float* colv = aux + 64 * hf;        // 1/Z'(i) or -log2 Z(i)
        const float* dsum = aux + 128 + 64 * hf;  // sum_b D_b(i)
        const float* rwin = aux + 256 + 127 + 64 * hf - r;  // r(i - j), i - j = c - r
        const int ab = cc & 1;
        mbar_wait(acc_full + ab, (cc >> 1) & 1, wc, kSitePgAcc);
        tc_fence_after();
        // diagonal sums of this warp: d = 127 + 64 hf - 32 rg - 32 + 32 m + lane
        float dg0 = 0.f, dg1 = 0.f, dg2 = 0.f;
#pragma unroll 1
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t v[32];
          tmem_ld_x32(tmem + lane_base + ab * 128 + 64 * hf + 32 * ch, v);
          tmem_wait_ld(v);
#pragma unroll
          for (int k4 = 0; k4 < 32; k4 += 4) {
            const int c = 32 * ch + k4;
            const float4 cv = *reinterpret_cast<const float4*>(colv + c);
            const float4 ds = *reinterpret_cast<const float4*>(dsum + c);
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
              const float w0 = rwin[c + e], w1 = rwin[c + e + 1];
              const uint64_t cv2 = e ? f2_pack(cv.z, cv.w) : f2_pack(cv.x, cv.y);
              const uint64_t ds2 = e ? f2_pack(ds.z, ds.w) : f2_pack(ds.x, ds.y);
              uint64_t p2;
              if (exact) {
                float a0, a1;
                f2_unpack(f2_add(f2_add(f2_pack(w0, w1), cv2), row2), a0, a1);
                p2 = f2_pack(fast_exp2(a0), fast_exp2(a1));
              } else {
                p2 = f2_mul(f2_mul(f2_pack(w0, w1), cv2), row2);
              }
              const uint64_t x2 = f2_fma(ds2, m1, f2_pack(__uint_as_float(v[k4 + e]),
                                                          __uint_as_float(v[k4 + e + 1])));
              const uint64_t dl2 = f2_mul(p2, x2);
              dal2 = f2_add(dal2, dl2);
              float d0, d1;
              f2_unpack(dl2, d0, d1);
              skw_w[(k4 + e) * L::SKW_ROW] = d0;
              skw_w[(k4 + e + 1) * L::SKW_ROW] = d1;
            }
          }
          __syncwarp();
          uint64_t lo_a = 0, lo_b = 0, hi_a = 0, hi_b = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 x = skw_lo[j];
            const float4 y = skw_hi[j];
            lo_a = f2_add(lo_a, f2_pack(x.x, x.y));
            lo_b = f2_add(lo_b, f2_pack(x.z, x.w));
            hi_a = f2_add(hi_a, f2_pack(y.x, y.y));
            hi_b = f2_add(hi_b, f2_pack(y.z, y.w));
          }
          __syncwarp();
          float t0, t1, t2, t3;
          f2_unpack(f2_add(lo_a, lo_b), t0, t1);
          f2_unpack(f2_add(hi_a, hi_b), t2, t3);
          const float elo = t0 + t1, ehi = t2 + t3;  // block diagonals lane, lane + 32
          if (ch == 0) { dg0 += elo; dg1 += ehi; } else { dg1 += elo; dg2 += ehi; }
        }
        tc_fence_before();
        mbar_arrive(acc_empty + ab);
        ++cc;
        __syncwarp();
        if (lane == 0) mbar_arrive(aux_empty + as);  // this warp has read the table slot
        ++ac;
        // This warp's diagonal sums go straight to drho (no step-wide barrier
        // to combine the eight warps first): lane's sums dg0..dg2 are the
        // block diagonals o = lane, lane + 32, lane + 64, i.e. tile diagonal
        // t = c - r + 127 = o + 95 + 64 hf - 32 rg, global distance
        // (I - J) * 128 - 127 + t.
        const int t0 = lane + 95 + 64 * hf - 32 * rg;
        const int d0 = (I - J) * 128 - 127 + t0;
        const float dgs[3] = {dg0, dg1, dg2};
#pragma unroll
        for (int m = 0; m < 3; ++m) {
          const int delta = d0 + 32 * m;
          if (delta >= 0 && delta < T && dgs[m] != 0.f)
            atomicAdd(&p.drho[(size_t)h * T + delta], dgs[m]);
        }
      }
      float da0, da1;
      f2_unpack(dal2, da0, da1);
      // the two column halves of row r add into a zeroed entry: 0 + a + b is
      // the same in either order
      atomicAdd(&p.dalpha[(size_t)h * T + J * 128 + r], da0 + da1);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

template <int D>
cudaError_t launch_dyn(const BwdLaunch& L, cudaStream_t s) {
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(bwd_dynamic_kernel<D>),
                                       BwdSmem<D>::ALLOC);
  if (e != cudaSuccess) return e;
  if (L.p.n_items == 0) return cudaSuccess;
  const int grid = L.p.n_items < L.num_sms ? L.p.n_items : L.num_sms;
  trace_begin(s);
  bwd_dynamic_kernel<D><<<grid, 512, BwdSmem<D>::ALLOC, s>>>(L.tm_q, L.tm_k, L.tm_v, L.tm_do,
                                                              L.tm_dq, L.p);
  trace_end(s, "bwd_dynamic");
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_pg(const ParamGradLaunch& L, cudaStream_t s) {
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(param_grad_kernel<D>),
                                       PgSmem<D>::ALLOC);
  if (e != cudaSuccess) return e;
  if (L.p.n_items == 0) return cudaSuccess;
  const int grid = L.p.n_items < L.num_sms ? L.p.n_items : L.num_sms;
  trace_begin(s);
  param_grad_kernel<D><<<grid, 384, PgSmem<D>::ALLOC, s>>>(L.tm_v, L.tm_do, L.p);
  trace_end(s, "param_grad");
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dynamic(const BwdLaunch& L, cudaStream_t s) {
  switch (L.d_h) {
    case 32: return launch_dyn<32>(L, s);
    case 64: return launch_dyn<64>(L, s);
    case 128: return launch_dyn<128>(L, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_param_grads(const ParamGradLaunch& L, cudaStream_t s) {
  switch (L.d_h) {
    case 32: return launch_pg<32>(L, s);
    case 64: return launch_pg<64>(L, s);
    case 128: return launch_pg<128>(L, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace saf
