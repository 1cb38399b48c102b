// attn_kernels.h — launch descriptors of the attention kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace saf {

// Parameters of the fused forward kernel (and of its transposed static-only
// form, which computes dV = P^T dO for the frozen heads).
struct FwdParams {
  int B, H, T, nI;            // nI = T / 128
  int H_kv, group_kv;         // K/V heads; query heads per K/V head (1: one each)
  int n_static, n_dynamic;    // head counts
  int group, n_groups;        // sequences per static item, groups per head
  int n_items;
  float scale_log2;           // log2(e) / sqrt(d_h)
  uint8_t static_heads[kMaxHeads];
  uint8_t dynamic_heads[kMaxHeads];
  const float* a_tab;         // [n_static, T]
  const float* r_tab;         // [n_static, T + 128]
  const float* row_tab;       // [n_static, T]
  const float* logZ;          // [n_static, T]
  const int* mode;            // [n_static]
  const float* shift;         // [n_static] log Z = log Z' + shift (factored heads)
  __nv_bfloat16* out;         // forward: out; transposed: dV
  float* out_acc;             // transposed with group_kv > 1: fp32 dV [B, H_kv, T, d_h],
                              // added to with atomics (out is then unused)
  float* lse;                 // forward only (nullable)
  int* status;                // device status word
  // Failure-path testing only (0 otherwise): CTA 0 withholds its first Q tile
  // so that the waits on it run out and the CTA takes the abort path.
  int hold_first_q;
};

// Sequences per static work item: the TMEM columns left for the O
// accumulator (512 minus the S/P buffers) divided by d_h.  Three buffers
// leave 128 columns; the transposed engine at d_h = 128 keeps two (256).
inline int static_group(int d_h, int B, bool transposed = false) {
  const int cols = (transposed && d_h == 128) ? 256 : 128;
  const int g = cols / d_h;
  return g < B ? g : B;
}

struct FwdLaunch {
  // bf16 views [B*H*T, d_h] (Q) and [B*H_kv*T, d_h] (K, V); tm_v = dO
  // ([B*H*T, d_h]) when transposed
  CUtensorMap tm_q, tm_k, tm_v;
  CUtensorMap tm_o;  // out [B*H*T, d_h] bf16 (forward, d_h = 64: tiled output stores)
  FwdParams p;
  int d_h;
  bool transposed;
  int num_sms;
};
cudaError_t launch_hybrid_fwd(const FwdLaunch& L, cudaStream_t s);

// Backward pre-pass: D(b,h,i) = sum_d dO * O for every row, the log2-scaled
// lse copy for dynamic heads, and the batch sums of D for static heads.
struct BwdPre {
  int B, H, T, d_h;
  const __nv_bfloat16* out;
  const __nv_bfloat16* dout;
  const float* lse;
  float* Dvec;        // [B, H, T]  -D
  float* lse2;        // [B, H, T]  -lse * log2(e)
  float* Dsum;        // [n_static, T] (nullable): sum over b of D
  float* dq_acc;      // [B, H, T, d_h] fp32 zeroed here (nullable)
  int n_static;
  uint8_t static_heads[kMaxHeads];
  // Per-row table of the frozen heads from the forward's lse (sequence 0):
  // factored 1/Z'(i) = exp(shift - lse), exact -lse * log2(e).  Nullable.
  float* row_tab;     // [n_static, T]
  const int* mode;
  const float* shift;
  uint8_t static_slot[kMaxHeads];  // head -> index among the frozen heads, 255 if dynamic
};
cudaError_t launch_bwd_pre(const BwdPre& p, cudaStream_t s);

// Dynamic-head backward (KV-tile parallel).
struct BwdParams {
  int B, H, T, nI;
  int H_kv;                   // K/V heads (H: one per query head)
  int n_kv, n_items;          // K/V heads that serve a dynamic query head; items
  int pairs_per_group;        // (sequence, K/V head) pairs per group of items
  float scale_log2;           // log2(e) / sqrt(d_h)
  float scale;                // 1 / sqrt(d_h)
  // The dynamic query heads grouped by K/V head: K/V head kv_list[i] serves
  // dyn_by_kv[dyn_begin[kv] .. dyn_begin[kv] + dyn_count[kv] - 1].
  uint8_t kv_list[kMaxHeads];
  uint16_t dyn_begin[kMaxHeads], dyn_count[kMaxHeads];
  uint8_t dyn_by_kv[kMaxHeads];
  uint8_t kv_has_static[kMaxHeads];
  const float* dv_acc;        // [B, H_kv, T, d_h] fp32 dV of the frozen heads, added to
                              // the dV of K/V heads with kv_has_static (nullable)
  const float* lse2;          // [B, H, T]  -lse * log2(e)
  const float* Dvec;          // [B, H, T]  -D
  float* dq_acc;              // [B, H, T, d_h] fp32, zeroed
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  int* status;
};
struct BwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  CUtensorMap tm_dq;             // fp32 [B*H*T, d_h] view of dq_acc (d_h <= 64)
  BwdParams p;
  int d_h;
  int num_sms;
};
cudaError_t launch_bwd_dynamic(const BwdLaunch& L, cudaStream_t s);

// Static-head alpha/rho gradients.
struct ParamGradParams {
  int B, H, T, nI;
  int H_kv, group_kv;         // V rows of query head h: K/V head h / group_kv
  int n_static, n_items;
  uint8_t static_heads[kMaxHeads];
  const float* a_tab;
  const float* r_tab;
  const float* row_tab;
  const int* mode;
  const float* Dsum;          // [n_static, T]
  float* dalpha;              // [H, T]
  float* drho;                // [H, T]
  int* status;
};
struct ParamGradLaunch {
  CUtensorMap tm_v, tm_do;
  ParamGradParams p;
  int d_h;
  int num_sms;
};
cudaError_t launch_param_grads(const ParamGradLaunch& L, cudaStream_t s);

// dQ: fp32 accumulator -> output dtype (scaled); zero dQ rows of static
// heads and dK rows of K/V heads that serve no dynamic head; dV of those K/V
// heads from the fp32 static accumulator when there is one.
struct BwdPost {
  int B, H, T, d_h, H_kv;
  const float* dq_acc;
  __nv_bfloat16* dQ;
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  const float* dv_acc;        // nullable
  uint8_t is_static[kMaxHeads];
  uint8_t kv_no_dyn[kMaxHeads];
};
cudaError_t launch_bwd_post(const BwdPost& p, cudaStream_t s);

}  // namespace saf
