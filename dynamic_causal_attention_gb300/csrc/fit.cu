// fit.cu — the compact pattern fit of SAF ("When Can Attention Heads Be
// Statically Defined?", §3 Eq. (3)/(4), App. A.2): for each candidate head
// the mean pattern A_hat is compressed into alpha (absolute key position) and
// rho (distance) by 400 Adam steps on the row-averaged cross-entropy; a head
// whose fitted pattern has mean row KL(A_hat || P_hat) above 0.2 nat is
// skipped and the next head in variance order is tried.
//
// The gradient only needs the target's column and diagonal sums (Eq. (4):
// they are sufficient statistics) and the same two sums of the current
// P_hat:  d/dalpha(j) = (colsum_P(j) - colsum_A(j)) / T,
//         d/drho(d)   = (diagsum_P(d) - diagsum_A(d)) / T.
//
// fit_kernel: one CTA per candidate head; alpha, rho, the Adam moments, the
// target marginals, log Z and the gradients live in shared memory (11 T
// floats).  Per step:
//   log Z(i)       two passes over k <= i (max, then the shifted sum of exps);
//   colsum_P(j)    sum_{i>=j} exp(alpha(j) + rho(i-j) - log Z(i));
//   diagsum_P(d)   sum_{i>=d} exp(alpha(i-d) + rho(d) - log Z(i));
// every exponent is <= 0 (log Z(i) bounds each of its terms), so nothing
// overflows in fp32.  Rows, columns and diagonals of lengths n and T + 1 - n
// are paired on one thread so that every thread does the same work.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace saf {
namespace {

constexpr int kFitThreads = 512;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
  return t;
}

// Row max then log-sum-exp of alpha(k) + rho(i - k), k <= i.
__device__ __forceinline__ float row_logz(const float* al, const float* rh, int i) {
  float m = -INFINITY;
  for (int k = 0; k <= i; ++k) m = fmaxf(m, al[k] + rh[i - k]);
  if (!(m > -INFINITY)) return -INFINITY;
  float s = 0.f;
  for (int k = 0; k <= i; ++k) s += __expf(al[k] + rh[i - k] - m);
  return m + __logf(s);
}

__global__ void __launch_bounds__(kFitThreads) fit_kernel(FitParams p) {
  extern __shared__ float sh[];
  __shared__ float red[32];
  const int T = p.T;
  float* al = sh;           // alpha
  float* rh = al + T;       // rho
  float* ma = rh + T;       // Adam moments
  float* va = ma + T;
  float* mr = va + T;
  float* vr = mr + T;
  float* ca = vr + T;       // target column sums
  float* da = ca + T;       // target diagonal sums
  float* lz = da + T;       // log Z
  float* ga = lz + T;       // gradients
  float* gr = ga + T;
  const int cand = blockIdx.x;
  const int head = p.candidates[cand];
  const float* A = p.A_hat + (size_t)head * T * T;

  // target marginals: column sums over rows i >= j, diagonal sums over i - j = d
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    float c = 0.f, d = 0.f;
    for (int i = t; i < T; ++i) {
      c += A[(size_t)i * T + t];
      d += A[(size_t)i * T + (i - t)];
    }
    ca[t] = c;
    da[t] = d;
    const float n = (float)(T - t);
    al[t] = __logf(fmaxf(c / n, 1e-30f));
    rh[t] = __logf(fmaxf(d / n, 1e-30f));
    ma[t] = va[t] = mr[t] = vr[t] = 0.f;
  }
  __syncthreads();

  const float inv_T = 1.0f / (float)T;
  float b1t = 1.f, b2t = 1.f;
  for (int step = 1; step <= p.steps; ++step) {
    // log Z of rows t and T-1-t
    for (int t = threadIdx.x; t < (T + 1) / 2; t += blockDim.x) {
      lz[t] = row_logz(al, rh, t);
      if (T - 1 - t != t) lz[T - 1 - t] = row_logz(al, rh, T - 1 - t);
    }
    __syncthreads();
    // gradients of column j and diagonal d, for j, d in {t, T-1-t}
    for (int t = threadIdx.x; t < (T + 1) / 2; t += blockDim.x) {
      for (int q = 0; q < (T - 1 - t != t ? 2 : 1); ++q) {
        const int j = q ? T - 1 - t : t;
        float c = 0.f, d = 0.f;
        for (int i = j; i < T; ++i) {
          c += __expf(al[j] + rh[i - j] - lz[i]);
          d += __expf(al[i - j] + rh[j] - lz[i]);
        }
        ga[j] = (c - ca[j]) * inv_T;
        gr[j] = (d - da[j]) * inv_T;
      }
    }
    __syncthreads();  // every read of alpha/rho for this step is done
    b1t *= p.beta1;
    b2t *= p.beta2;
    const float c1 = 1.f - b1t, c2 = 1.f - b2t;
    for (int j = threadIdx.x; j < T; j += blockDim.x) {
      const float g = ga[j], h = gr[j];
      ma[j] = p.beta1 * ma[j] + (1.f - p.beta1) * g;
      va[j] = p.beta2 * va[j] + (1.f - p.beta2) * g * g;
      mr[j] = p.beta1 * mr[j] + (1.f - p.beta1) * h;
      vr[j] = p.beta2 * vr[j] + (1.f - p.beta2) * h * h;
      al[j] -= p.lr * (ma[j] / c1) / (sqrtf(va[j] / c2) + p.eps);
      rh[j] -= p.lr * (mr[j] / c1) / (sqrtf(vr[j] / c2) + p.eps);
    }
    __syncthreads();
  }

  // final log Z and mean row KL(A_hat || P_hat)
  for (int t = threadIdx.x; t < (T + 1) / 2; t += blockDim.x) {
    lz[t] = row_logz(al, rh, t);
    if (T - 1 - t != t) lz[T - 1 - t] = row_logz(al, rh, T - 1 - t);
  }
  __syncthreads();
  float kl = 0.f;
  for (int i = 0; i < T; ++i) {
    for (int j = threadIdx.x; j <= i; j += blockDim.x) {
      const float a = A[(size_t)i * T + j];
      if (a > 0.f) kl += a * (__logf(a) - (al[j] + rh[i - j] - lz[i]));
    }
  }
  kl = block_sum(kl, red) * inv_T;
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    p.alpha[(size_t)cand * T + t] = al[t];
    p.rho[(size_t)cand * T + t] = rh[t];
  }
  if (threadIdx.x == 0) p.kl[cand] = kl;
}

// Walk the candidates in order and keep the first k whose KL passes.
__global__ void fit_select_kernel(FitParams p) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  int n = 0;
  for (int c = 0; c < p.n_candidates && n < p.k; ++c)
    if (p.kl[c] <= p.kl_max) p.selected[n++] = p.candidates[c];
  *p.n_selected = n;
}

}  // namespace

size_t fit_smem_bytes(int T) { return (size_t)11 * T * sizeof(float); }

cudaError_t launch_fit(const FitParams& p, cudaStream_t s) {
  const size_t smem = fit_smem_bytes(p.T);
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(fit_kernel), 200 * 1024);
  if (e != cudaSuccess) return e;
  trace_begin(s);
  fit_kernel<<<p.n_candidates, kFitThreads, smem, s>>>(p);
  trace_end(s, "fit");
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  trace_begin(s);
  fit_select_kernel<<<1, 32, 0, s>>>(p);
  trace_end(s, "fit_select");
  return cudaGetLastError();
}

}  // namespace saf
