// attn_bwd_aux.cu — the small bandwidth-bound passes around the backward
// kernels of the hybrid layer:
//   bwd_pre   D(b,h,i) = sum_d dO(b,h,i,d) * out(b,h,i,d) (the softmax
//             backward's row term), stored negated, and -lse * log2(e) (the
//             dynamic backward adds both), plus for frozen heads the batch
//             sums of D that the alpha/rho gradients need; it also zeroes the
//             fp32 dQ accumulator, and rebuilds the frozen heads' per-row table
//             from the forward's lse (log Z);
//   bwd_post  dQ = (1/sqrt(d_h)) * fp32 accumulator -> bf16, and zeros for the
//             dQ/dK rows of frozen heads (they have no query/key path).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn_kernels.h"
#include "internal.h"
#include "ptx.cuh"

namespace saf {
namespace {

// Blocks walk (b, h) slabs of T rows (blockIdx.y) so that the per-head
// choices are uniform; one group of D/8 lanes per row, each lane reads 8 bf16
// of dO and of out.  A frozen head's D is only formed when its batch sums
// are wanted (alpha/rho gradients); its per-row table needs only the lse.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(BwdPre p) {
  constexpr int LPR = D / 8;  // lanes per row
  const int n_bh = p.B * p.H;
  for (int bh = blockIdx.y; bh < n_bh; bh += gridDim.y) {
    const int h = bh % p.H;
    const int hs = p.static_slot[h];
    const bool need_d = (hs == 255) || (p.Dsum != nullptr);
    for (uint32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < (uint32_t)p.T * LPR;
         t += gridDim.x * blockDim.x) {
      const int i = (int)(t / LPR), sub = (int)(t % LPR);
      const size_t row = (size_t)bh * p.T + i;
      float acc = 0.f;
      if (need_d) {
        const uint4 a = *reinterpret_cast<const uint4*>(p.out + row * D + sub * 8);
        const uint4 b = *reinterpret_cast<const uint4*>(p.dout + row * D + sub * 8);
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 x = __bfloat1622float2(a2[k]), y = __bfloat1622float2(b2[k]);
          acc = fmaf(x.x, y.x, acc);
          acc = fmaf(x.y, y.y, acc);
        }
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      }
      // the accumulator rows of frozen heads are never added to or read
      if (hs == 255 && p.dq_acc) {
        float4* z = reinterpret_cast<float4*>(p.dq_acc + row * D + sub * 8);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (sub == 0) {
        const float l = p.lse[row];
        if (need_d) {
          p.Dvec[row] = -acc;
          p.lse2[row] = -l * 1.4426950408889634f;
        }
        if (hs != 255 && p.row_tab && bh < p.H) {  // sequence 0: rows (h, i)
          float v;
          if (p.mode[hs]) v = -l * 1.4426950408889634f;
          else v = (l > -INFINITY) ? expf(p.shift[hs] - l) : 0.f;
          p.row_tab[(size_t)hs * p.T + i] = v;
        }
      }
    }
  }
}

__global__ void dsum_kernel(BwdPre p) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x, hs = blockIdx.y;
  if (i >= p.T) return;
  const int h = p.static_heads[hs];
  float s = 0.f;
  for (int b = 0; b < p.B; ++b) s -= p.Dvec[((size_t)b * p.H + h) * p.T + i];
  p.Dsum[(size_t)hs * p.T + i] = s;
}

// Blocks walk (b, h) slabs (blockIdx.y), 16-byte units within a slab.
template <int D>
__global__ void __launch_bounds__(256) bwd_post_kernel(BwdPost p, float scale) {
  const uint32_t units = (uint32_t)p.T * (D / 8);
  const int n_bh = p.B * p.H, n_bkv = p.B * p.H_kv;
  for (int bh = blockIdx.y; bh < n_bh; bh += gridDim.y) {
    const bool st = p.is_static[bh % p.H];
    // the [B, H_kv, T, d_h] tensors: slab bh is (b, kv) while in range
    const bool kv_zero = bh < n_bkv && p.kv_no_dyn[bh % p.H_kv];
    const size_t base = (size_t)bh * p.T * D;
    for (uint32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < units;
         u += gridDim.x * blockDim.x) {
      const size_t e = base + (size_t)u * 8;
      if (kv_zero) {
        *reinterpret_cast<uint4*>(p.dK + e) = make_uint4(0u, 0u, 0u, 0u);
        if (p.dv_acc) {
          const float4 a = *reinterpret_cast<const float4*>(p.dv_acc + e);
          const float4 b = *reinterpret_cast<const float4*>(p.dv_acc + e + 4);
          uint4 v;
          v.x = pack_bf16x2(a.x, a.y);
          v.y = pack_bf16x2(a.z, a.w);
          v.z = pack_bf16x2(b.x, b.y);
          v.w = pack_bf16x2(b.z, b.w);
          *reinterpret_cast<uint4*>(p.dV + e) = v;
        }
      }
      uint4 q;
      if (st) {
        q = make_uint4(0u, 0u, 0u, 0u);
      } else {
        const float4 a = *reinterpret_cast<const float4*>(p.dq_acc + e);
        const float4 b = *reinterpret_cast<const float4*>(p.dq_acc + e + 4);
        q.x = pack_bf16x2(a.x * scale, a.y * scale);
        q.y = pack_bf16x2(a.z * scale, a.w * scale);
        q.z = pack_bf16x2(b.x * scale, b.y * scale);
        q.w = pack_bf16x2(b.z * scale, b.w * scale);
      }
      *reinterpret_cast<uint4*>(p.dQ + e) = q;
    }
  }
}

// Grid over (b, h) slabs: x covers one slab's threads in about four rounds.
dim3 slab_grid(size_t slab_threads, int n_bh) {
  size_t gx = (slab_threads + 1023) / 1024;
  if (gx < 1) gx = 1;
  if (gx > 1024) gx = 1024;
  return dim3((unsigned)gx, (unsigned)(n_bh < 65535 ? n_bh : 65535));
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdPre& p, cudaStream_t s) {
  const dim3 blocks = slab_grid((size_t)p.T * (p.d_h / 8), p.B * p.H);
  trace_begin(s);
  switch (p.d_h) {
    case 32: bwd_pre_kernel<32><<<blocks, 256, 0, s>>>(p); break;
    case 64: bwd_pre_kernel<64><<<blocks, 256, 0, s>>>(p); break;
    case 128: bwd_pre_kernel<128><<<blocks, 256, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  trace_end(s, "bwd_pre");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.Dsum == nullptr || p.n_static == 0) return e;
  trace_begin(s);
  dsum_kernel<<<dim3((p.T + 255) / 256, p.n_static), 256, 0, s>>>(p);
  trace_end(s, "bwd_dsum");
  return cudaGetLastError();
}

cudaError_t launch_bwd_post(const BwdPost& p, cudaStream_t s) {
  const float scale = 1.0f / sqrtf((float)p.d_h);
  const dim3 blocks = slab_grid((size_t)p.T * p.d_h / 8, p.B * p.H);
  trace_begin(s);
  switch (p.d_h) {
    case 32: bwd_post_kernel<32><<<blocks, 256, 0, s>>>(p, scale); break;
    case 64: bwd_post_kernel<64><<<blocks, 256, 0, s>>>(p, scale); break;
    case 128: bwd_post_kernel<128><<<blocks, 256, 0, s>>>(p, scale); break;
    default: return cudaErrorInvalidValue;
  }
  trace_end(s, "bwd_post");
  return cudaGetLastError();
}

}  // namespace saf
