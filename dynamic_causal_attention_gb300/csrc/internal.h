// internal.h — declarations shared by the host API (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/saf.h"

namespace saf {

// Launch bookkeeping (per host thread): trace_begin() before and trace_end()
// after every kernel launch.  trace_end counts the launch for
// saf_last_launch_count(); when the kernel trace is enabled the pair also
// records two CUDA events on the launch stream around the kernel.
void trace_begin(cudaStream_t s);
void trace_end(cudaStream_t s, const char* kernel);
// Start counting launches for a new entry-point call.
void launch_count_reset();

// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device.  cudaFuncSetAttribute applies to the current device only, so this
// is done once per (kernel, device); safe to call from several host threads.
cudaError_t set_max_dynamic_smem(const void* kernel, int bytes);

// ------------------------------------------------------------ calibration
struct CalibLaunch {
  const float* A;     // [n, head_count, T, T]
  int n;
  int head_begin;
  int head_count;
  int T;
  int count0;         // samples already merged into these heads
  float* mean;        // [num_heads, T, T]
  float* m2;          // [num_heads, T, T]
  float* ent;         // [num_heads, T, T] sum_n x log x, or null (not tracked)
};
cudaError_t launch_calib_accumulate(const CalibLaunch& p, cudaStream_t s);

struct CalibFinalize {
  int num_heads;
  int T;
  int N;
  int k;
  const float* mean;
  const float* m2;
  double* row_partials;  // [num_heads, T]
  float* A_hat;          // nullable
  float* s_var;
  int32_t* selected;     // nullable when k == 0
  const float* ent;      // KL score only: sum_n x log x state
};
cudaError_t launch_calib_finalize(const CalibFinalize& p, cudaStream_t s);
// Forward-KL score per head (into p.s_var) and its exact top-k.
cudaError_t launch_calib_finalize_kl(const CalibFinalize& p, cudaStream_t s);
// Sharp-mean pattern: causal softmax of each row of the running mean.
cudaError_t launch_calib_sharp(const float* mean, int num_heads, int T, float* out,
                               cudaStream_t s);

// ------------------------------------------------------------ compact fit
struct FitParams {
  const float* A_hat;        // [num_heads, T, T]
  int T;
  const int32_t* candidates; // [n_candidates] head indices, priority order
  int n_candidates;
  int k;
  float kl_max;
  int steps;
  float lr, beta1, beta2, eps;
  float* alpha;              // [n_candidates, T]
  float* rho;                // [n_candidates, T]
  float* kl;                 // [n_candidates]
  int32_t* selected;         // [k] (nullable when k == 0)
  int32_t* n_selected;       // [1]
};
size_t fit_smem_bytes(int T);
cudaError_t launch_fit(const FitParams& p, cudaStream_t s);

// ------------------------------------------------------------ attention
constexpr int kMaxHeads = 256;

// Static-head pre-pass (alpha/rho -> generator tables and log Z).
struct StaticPrep {
  int T;
  int n_static;
  const uint8_t* heads_dev;  // unused (heads passed by value below)
  uint8_t heads[kMaxHeads];  // static head ids
  const float* alpha;        // [H, T]
  const float* rho;          // [H, T]
  float* a_tab;              // [n_static, T]
  float* r_tab;              // [n_static, T + 128] (127 leading pads)
  float* row_tab;            // [n_static, T] : -log2 Z (exact heads only)
  float* logZ;               // [n_static, T] natural log (exact heads only)
  int* mode;                 // [n_static] 0 factored, 1 exact
  float* shift;              // [n_static] factored: max alpha + max rho (0 if all masked)
};
cudaError_t launch_static_prep(const StaticPrep& p, cudaStream_t s);

// Elementwise helpers.
cudaError_t launch_zero_u32(void* dst, size_t n_words, cudaStream_t s);
// [n_slabs, T_src, d] rows (bf16 or fp32) into [n_slabs, T_dst, d] (bf16 or
// fp32): rows t >= T_src of the destination are zero (padding), rows of the
// source past T_dst are dropped (cropping).  d % 4 == 0.
cudaError_t launch_restage_rows(const void* src, bool src_f32, void* dst, bool dst_f32,
                                size_t n_slabs, int T_src, int T_dst, int d, cudaStream_t s);
// [n_rows, T_src] fp32 into [n_rows, T_dst], entries t >= T_src set to `fill`.
cudaError_t launch_restage_vec(const float* src, float* dst, size_t n_rows, int T_src, int T_dst,
                               float fill, cudaStream_t s);

}  // namespace saf
