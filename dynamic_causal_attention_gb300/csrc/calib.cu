// calib.cu — the calibration reduction of SAF ("When Can Attention Heads Be
// Statically Defined?", §3.1): per-head mean pattern A_hat over N sequences,
// the variance score s_var of Eq. (1), and the global ascending top-k with
// k = round(r L H).
//
// The work is a streaming reduction over the n axis of A [n, heads, T, T]:
// HBM-bound, so the kernels read each lower-triangle float4 of A exactly once
// with streaming (evict-first) 16-byte loads, keep eight samples per element
// in flight, and touch the upper triangle never.
//
// Per element the state holds mean and M2 (sum of squared deviations) in
// fp32.  Each batch of up to 8 samples is reduced two-pass in registers and
// merged into the state with the pairwise update of Chan, Golub and LeVeque
// (1979):  n = na + nb,  delta = mean_b - mean_a,
//          mean = mean_a + delta * nb / n,
//          M2   = M2_a + M2_b + delta^2 * na * nb / n.
// s_var sums M2 over the triangle in fp64 with a fixed reduction order, so
// results are deterministic run to run.
//
// Optionally the state also keeps sum_n x log x per element, from which the
// row-wise forward-KL selector (the alternative to s_var that the notes
// compare, App. B.2) follows without a second pass over A.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace saf {
namespace {

constexpr int kBatch = 8;
// 128-thread blocks: at the accumulate kernel's ~90 registers a thread, five
// of them fit an SM (20 warps), against two of 256 threads (16 warps).
constexpr int kAccThreads = 128;

// Lower-triangle float4 units of a T x T matrix (T % 4 == 0): rows 4q..4q+3
// each have q + 1 units; the group of rows 4q..4q+3 starts at unit 2 q (q+1).
__device__ __forceinline__ void unit_to_row_col(uint32_t u, int& row, int& c4) {
  int q = (int)((sqrtf(1.0f + 2.0f * (float)u) - 1.0f) * 0.5f);
  while (2u * (uint32_t)q * (uint32_t)(q + 1) > u) --q;
  while (2u * (uint32_t)(q + 1) * (uint32_t)(q + 2) <= u) ++q;
  const uint32_t rel = u - 2u * (uint32_t)q * (uint32_t)(q + 1);
  row = 4 * q + (int)(rel / (uint32_t)(q + 1));
  c4 = (int)(rel % (uint32_t)(q + 1));
}

__device__ __forceinline__ float4 masked(float4 v, int row, int col0) {
  // Entries above the diagonal (col > row) are treated as zero.
  if (col0 + 0 > row) v.x = 0.f;
  if (col0 + 1 > row) v.y = 0.f;
  if (col0 + 2 > row) v.z = 0.f;
  if (col0 + 3 > row) v.w = 0.f;
  return v;
}

// x log2 x with the limit 0 at x = 0: the argument is clamped to 1e-30 (for
// x below it the term is under 1e-28, far below what the sums resolve), so
// no branch is needed.  The entropy sums are kept in log2 units; the score
// rows convert to nats once per row.
constexpr float kLn2f = 0.6931471805599453f;
__device__ __forceinline__ float xlog2x(float x) { return x * __log2f(fmaxf(x, 1e-30f)); }

template <bool KL>
__global__ void __launch_bounds__(kAccThreads) calib_accumulate_kernel(CalibLaunch p) {
  const int T = p.T;
  const uint32_t units_per_head = 2u * (uint32_t)(T / 4) * (uint32_t)(T / 4 + 1);
  const uint64_t total = (uint64_t)units_per_head * (uint64_t)p.head_count;
  const size_t sample_stride = (size_t)p.head_count * (size_t)T * (size_t)T;
  for (uint64_t g = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (uint64_t)gridDim.x * blockDim.x) {
    const int hl = (int)(g / units_per_head);
    int row, c4;
    unit_to_row_col((uint32_t)(g - (uint64_t)hl * units_per_head), row, c4);
    const int col0 = c4 * 4;
    const size_t in_off = ((size_t)hl * T + row) * (size_t)T + col0;
    const size_t st_off = ((size_t)(p.head_begin + hl) * T + row) * (size_t)T + col0;

    float4 mean = make_float4(0.f, 0.f, 0.f, 0.f), m2 = mean, ent = mean;
    if (p.count0 > 0) {
      mean = *reinterpret_cast<const float4*>(p.mean + st_off);
      m2 = *reinterpret_cast<const float4*>(p.m2 + st_off);
      if (KL) ent = *reinterpret_cast<const float4*>(p.ent + st_off);
    }
    int cnt = p.count0;
    const float* src = p.A + in_off;
    for (int s = 0; s < p.n; s += kBatch) {
      const int m = min(kBatch, p.n - s);
      float4 x[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (k < m) x[k] = __ldcs(reinterpret_cast<const float4*>(src + (size_t)(s + k) * sample_stride));
      const float inv_m = 1.0f / (float)m;
      float4 mb = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (k < m) {
          x[k] = masked(x[k], row, col0);
          mb.x += x[k].x; mb.y += x[k].y; mb.z += x[k].z; mb.w += x[k].w;
          if (KL) {
            ent.x = fmaf(x[k].x, __log2f(fmaxf(x[k].x, 1e-30f)), ent.x);
            ent.y = fmaf(x[k].y, __log2f(fmaxf(x[k].y, 1e-30f)), ent.y);
            ent.z = fmaf(x[k].z, __log2f(fmaxf(x[k].z, 1e-30f)), ent.z);
            ent.w = fmaf(x[k].w, __log2f(fmaxf(x[k].w, 1e-30f)), ent.w);
          }
        }
      mb.x *= inv_m; mb.y *= inv_m; mb.z *= inv_m; mb.w *= inv_m;
      float4 qb = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (k < m) {
          const float dx = x[k].x - mb.x, dy = x[k].y - mb.y, dz = x[k].z - mb.z,
                      dw = x[k].w - mb.w;
          qb.x += dx * dx; qb.y += dy * dy; qb.z += dz * dz; qb.w += dw * dw;
        }
      if (cnt == 0) {
        mean = mb;
        m2 = qb;
      } else {
        const float n_tot = (float)(cnt + m);
        const float wb = (float)m / n_tot;
        const float wab = (float)cnt * (float)m / n_tot;
        const float dx = mb.x - mean.x, dy = mb.y - mean.y, dz = mb.z - mean.z, dw = mb.w - mean.w;
        mean.x += dx * wb; mean.y += dy * wb; mean.z += dz * wb; mean.w += dw * wb;
        m2.x += qb.x + dx * dx * wab; m2.y += qb.y + dy * dy * wab;
        m2.z += qb.z + dz * dz * wab; m2.w += qb.w + dw * dw * wab;
      }
      cnt += m;
    }
    *reinterpret_cast<float4*>(p.mean + st_off) = mean;
    *reinterpret_cast<float4*>(p.m2 + st_off) = m2;
    if (KL) *reinterpret_cast<float4*>(p.ent + st_off) = ent;
  }
}

// Row kernels: one warp per (row, head), kRowsPerBlock rows per block, 16-byte
// loads.  Each lane sums its terms in fp32; the lanes' sums are combined by a
// fixed-order shuffle tree (deterministic) and the row's total leaves as one
// double.  (Per-element fp64 additions would run on this GPU's few fp64
// units and bound the kernels; fp32 partial sums of non-negative M2 terms, or
// of the score's per-element terms, carry no cancellation at this length.)
constexpr int kRowsPerBlock = 8;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// KL score rows: sum_j (sum_n x log2 x - N A_hat log2 A_hat) over the lower
// part of one row, times ln 2 (sum_n KL(A_n,i || A_hat_i) = that difference,
// because sum_n A_n = N A_hat).
__global__ void __launch_bounds__(32 * kRowsPerBlock) calib_kl_rows_kernel(CalibFinalize p) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5), h = blockIdx.y, T = p.T;
  if (row >= T) return;  // a whole warp
  const size_t base = ((size_t)h * T + row) * (size_t)T;
  const float N = (float)p.N;
  float acc = 0.f;
  for (int c4 = lane; c4 * 4 <= row; c4 += 32) {
    const int col0 = c4 * 4;
    const float4 mu = masked(*reinterpret_cast<const float4*>(p.mean + base + col0), row, col0);
    const float4 e = masked(*reinterpret_cast<const float4*>(p.ent + base + col0), row, col0);
    acc += ((e.x - N * xlog2x(mu.x)) + (e.y - N * xlog2x(mu.y))) +
           ((e.z - N * xlog2x(mu.z)) + (e.w - N * xlog2x(mu.w)));
  }
  acc = warp_sum(acc);
  if (lane == 0) p.row_partials[(size_t)h * T + row] = (double)acc * (double)kLn2f;
}

// Writes the full row of A_hat (zeros above the diagonal) and the row's sum
// of M2 over its lower part.
__global__ void __launch_bounds__(32 * kRowsPerBlock) calib_rows_kernel(CalibFinalize p) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5), h = blockIdx.y, T = p.T;
  if (row >= T) return;  // a whole warp
  const size_t base = ((size_t)h * T + row) * (size_t)T;
  float acc = 0.f;
  for (int c4 = lane; c4 < T / 4; c4 += 32) {
    const int col0 = c4 * 4;
    float4 mu = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col0 <= row) {
      mu = masked(*reinterpret_cast<const float4*>(p.mean + base + col0), row, col0);
      const float4 q = masked(*reinterpret_cast<const float4*>(p.m2 + base + col0), row, col0);
      acc += (q.x + q.y) + (q.z + q.w);
    }
    if (p.A_hat) __stcs(reinterpret_cast<float4*>(p.A_hat + base + col0), mu);
  }
  acc = warp_sum(acc);
  if (lane == 0) p.row_partials[(size_t)h * T + row] = (double)acc;
}

// Per head: the sum of its T row totals (fp64, one warp per head, fixed
// order), divided by `denom`.
__global__ void __launch_bounds__(256) calib_head_sums_kernel(CalibFinalize p, double denom) {
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (h >= p.num_heads) return;
  double acc = 0.0;
  for (int r = lane; r < p.T; r += 32) acc += p.row_partials[(size_t)h * p.T + r];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) p.s_var[h] = (float)(acc / denom);
}

// Sharp-mean pattern: one warp per (row, head) applies a causal softmax to
// the row of the running mean of the accumulated logits and writes the
// normalised row with exact zeros above the diagonal.  Rows of up to
// 128 * NC columns are held in registers (NC float4 per lane): one read of
// the row, one exponential per entry, fp32 lane sums and a fixed-order
// shuffle tree.  Longer rows take three passes over the row (the row stays
// in L1 between them): the maximum, the sum of exponentials (fp32 per 4
// columns, fp64 across them and across the warp, in a fixed order), then the
// normalised row.
constexpr int kSharpRows = 8;  // rows (warps) per block

__device__ __forceinline__ float4 causal_row4(const float4* src, int c4, int row) {
  float4 a = src[c4];
  const int c = 4 * c4;
  if (c + 1 > row) a.y = -INFINITY;
  if (c + 2 > row) a.z = -INFINITY;
  if (c + 3 > row) a.w = -INFINITY;
  return a;
}

template <int NC>
__global__ void __launch_bounds__(32 * kSharpRows) calib_sharp_rows_reg_kernel(
    const float* __restrict__ mean, int T, float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kSharpRows + (threadIdx.x >> 5), h = blockIdx.y;
  if (row >= T) return;  // a whole warp
  const size_t base = ((size_t)h * T + row) * (size_t)T;
  const float4* src = reinterpret_cast<const float4*>(mean + base);
  const int n4 = T / 4, last4 = row / 4;
  float4 a[NC];
  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    const int c4 = lane + 32 * j;
    a[j] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (c4 <= last4) a[j] = causal_row4(src, c4, row);
    mx = fmaxf(mx, fmaxf(fmaxf(a[j].x, a[j].y), fmaxf(a[j].z, a[j].w)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  // column 0 is in every row, so mx is finite; exp(-inf - mx) is an exact 0
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    a[j] = make_float4(expf(a[j].x - mx), expf(a[j].y - mx), expf(a[j].z - mx), expf(a[j].w - mx));
    sum += (a[j].x + a[j].y) + (a[j].z + a[j].w);
  }
  const float inv = 1.0f / warp_sum(sum);
  float4* dst = reinterpret_cast<float4*>(out + base);
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    const int c4 = lane + 32 * j;
    if (c4 < n4) __stcs(dst + c4, make_float4(a[j].x * inv, a[j].y * inv, a[j].z * inv, a[j].w * inv));
  }
}

__global__ void __launch_bounds__(32 * kSharpRows) calib_sharp_rows_kernel(
    const float* __restrict__ mean, int T, float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kSharpRows + (threadIdx.x >> 5), h = blockIdx.y;
  if (row >= T) return;  // a whole warp
  const size_t base = ((size_t)h * T + row) * (size_t)T;
  const float4* src = reinterpret_cast<const float4*>(mean + base);
  const int n4 = T / 4, last4 = row / 4;
  float mx = -INFINITY;
  for (int c4 = lane; c4 <= last4; c4 += 32) {
    const float4 a = causal_row4(src, c4, row);
    mx = fmaxf(mx, fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  double sum = 0.0;
  for (int c4 = lane; c4 <= last4; c4 += 32) {
    const float4 a = causal_row4(src, c4, row);
    sum += (double)((expf(a.x - mx) + expf(a.y - mx)) + (expf(a.z - mx) + expf(a.w - mx)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float inv = (float)(1.0 / sum);
  float4* dst = reinterpret_cast<float4*>(out + base);
  for (int c4 = lane; c4 < n4; c4 += 32) {
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c4 <= last4) {
      const float4 a = causal_row4(src, c4, row);
      o = make_float4(expf(a.x - mx) * inv, expf(a.y - mx) * inv, expf(a.z - mx) * inv,
                      expf(a.w - mx) * inv);
    }
    __stcs(dst + c4, o);
  }
}

// One block: the exact top-k of the per-head scores by rank over the unique
// 64-bit keys (bits(score) << 32 | index).
constexpr int kMaxCalibHeads = 8192;

__global__ void __launch_bounds__(1024) calib_select_kernel(CalibFinalize p) {
  __shared__ float sv[kMaxCalibHeads];
  for (int h = threadIdx.x; h < p.num_heads; h += blockDim.x) sv[h] = p.s_var[h];
  __syncthreads();
  for (int h = threadIdx.x; h < p.num_heads; h += blockDim.x) {
    const uint64_t kh = ((uint64_t)__float_as_uint(sv[h]) << 32) | (uint32_t)h;
    int rank = 0;
    for (int g = 0; g < p.num_heads; ++g) {
      const uint64_t kg = ((uint64_t)__float_as_uint(sv[g]) << 32) | (uint32_t)g;
      rank += (kg < kh) ? 1 : 0;
    }
    if (rank < p.k) p.selected[rank] = h;
  }
}

}  // namespace

cudaError_t launch_calib_accumulate(const CalibLaunch& p, cudaStream_t s) {
  const uint64_t units = 2ull * (uint64_t)(p.T / 4) * (uint64_t)(p.T / 4 + 1) * (uint64_t)p.head_count;
  const uint64_t want = (units + kAccThreads - 1) / kAccThreads;
  const int blocks = (int)(want < (1u << 30) ? want : (1u << 30));
  trace_begin(s);
  if (p.ent)
    calib_accumulate_kernel<true><<<blocks, kAccThreads, 0, s>>>(p);
  else
    calib_accumulate_kernel<false><<<blocks, kAccThreads, 0, s>>>(p);
  trace_end(s, "calib_accumulate");
  return cudaGetLastError();
}

cudaError_t launch_head_sums_and_select(const CalibFinalize& p, double denom, cudaStream_t s) {
  trace_begin(s);
  calib_head_sums_kernel<<<(p.num_heads + 7) / 8, 256, 0, s>>>(p, denom);
  trace_end(s, "calib_head_sums");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.k == 0) return e;
  trace_begin(s);
  calib_select_kernel<<<1, 1024, 0, s>>>(p);
  trace_end(s, "calib_select");
  return cudaGetLastError();
}

cudaError_t launch_calib_finalize(const CalibFinalize& p, cudaStream_t s) {
  if (p.num_heads > kMaxCalibHeads) return cudaErrorInvalidValue;
  trace_begin(s);
  calib_rows_kernel<<<dim3((p.T + kRowsPerBlock - 1) / kRowsPerBlock, p.num_heads),
                      32 * kRowsPerBlock, 0, s>>>(p);
  trace_end(s, "calib_rows");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_head_sums_and_select(p, (double)(p.N - 1) * (double)p.T * (double)p.T, s);
}

cudaError_t launch_calib_finalize_kl(const CalibFinalize& p, cudaStream_t s) {
  if (p.num_heads > kMaxCalibHeads || p.ent == nullptr) return cudaErrorInvalidValue;
  trace_begin(s);
  calib_kl_rows_kernel<<<dim3((p.T + kRowsPerBlock - 1) / kRowsPerBlock, p.num_heads),
                         32 * kRowsPerBlock, 0, s>>>(p);
  trace_end(s, "calib_kl_rows");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_head_sums_and_select(p, (double)p.N * (double)p.T, s);
}

cudaError_t launch_calib_sharp(const float* mean, int num_heads, int T, float* out,
                               cudaStream_t s) {
  if (T % 4 != 0) return cudaErrorInvalidValue;
  trace_begin(s);
  const dim3 grid((T + kSharpRows - 1) / kSharpRows, num_heads);
  const int n4 = T / 4;
  if (n4 <= 32 * 2)
    calib_sharp_rows_reg_kernel<2><<<grid, 32 * kSharpRows, 0, s>>>(mean, T, out);
  else if (n4 <= 32 * 4)
    calib_sharp_rows_reg_kernel<4><<<grid, 32 * kSharpRows, 0, s>>>(mean, T, out);
  else if (n4 <= 32 * 8)
    calib_sharp_rows_reg_kernel<8><<<grid, 32 * kSharpRows, 0, s>>>(mean, T, out);
  else
    calib_sharp_rows_kernel<<<grid, 32 * kSharpRows, 0, s>>>(mean, T, out);
  trace_end(s, "calib_sharp_rows");
  return cudaGetLastError();
}

}  // namespace saf
