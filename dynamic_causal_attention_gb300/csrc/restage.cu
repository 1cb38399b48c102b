// restage.cu — copies between the caller's tensors and the kernels' staging
// buffers: bf16 <-> fp32 conversion, and the padding of a sequence length
// that is not a multiple of 128 (the attention kernels work on whole
// 128-row tiles).
//
// Rows: [n_slabs, T_src, d] -> [n_slabs, T_dst, d], one (sequence, head) per
// slab.  Padding (T_dst > T_src) writes zero rows t >= T_src; cropping
// (T_dst < T_src) drops them.  Vectors: [n_rows, T_src] -> [n_rows, T_dst]
// fp32 with a fill value for the padded entries.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace saf {
namespace {

__device__ __forceinline__ float4 load4(const void* base, size_t off, bool f32) {
  if (f32) return *reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
  const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + off);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
  return make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
}

__device__ __forceinline__ void store4(void* base, size_t off, bool f32, float4 v) {
  if (f32) {
    *reinterpret_cast<float4*>(static_cast<float*>(base) + off) = v;
    return;
  }
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 o;
  o.x = *reinterpret_cast<const uint32_t*>(&a);
  o.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(base) + off) = o;
}

// four consecutive elements of the destination per thread (d % 4 == 0)
__global__ void restage_rows_kernel(const void* __restrict__ src, bool src_f32,
                                    void* __restrict__ dst, bool dst_f32, size_t n_slabs,
                                    int T_src, int T_dst, int d) {
  const int d4 = d / 4;
  const size_t per_slab = (size_t)T_dst * d4;
  const size_t n4 = n_slabs * per_slab;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t slab = i / per_slab;
    const size_t rem = i - slab * per_slab;
    const int t = (int)(rem / d4), c4 = (int)(rem - (size_t)t * d4);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < T_src) v = load4(src, (slab * T_src + t) * d + 4 * c4, src_f32);
    store4(dst, (slab * T_dst + t) * d + 4 * c4, dst_f32, v);
  }
}

__global__ void restage_vec_kernel(const float* __restrict__ src, float* __restrict__ dst,
                                   size_t n_rows, int T_src, int T_dst, float fill) {
  const size_t n = n_rows * (size_t)T_dst;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t row = i / T_dst;
    const int t = (int)(i - row * T_dst);
    dst[i] = t < T_src ? src[row * T_src + t] : fill;
  }
}

int blocks_for(size_t n) {
  size_t b = (n + 255) / 256;
  if (b < 1) b = 1;
  if (b > 8192) b = 8192;
  return (int)b;
}

}  // namespace

cudaError_t launch_restage_rows(const void* src, bool src_f32, void* dst, bool dst_f32,
                                size_t n_slabs, int T_src, int T_dst, int d, cudaStream_t s) {
  if (d % 4 != 0) return cudaErrorInvalidValue;
  trace_begin(s);
  restage_rows_kernel<<<blocks_for(n_slabs * (size_t)T_dst * (d / 4)), 256, 0, s>>>(
      src, src_f32, dst, dst_f32, n_slabs, T_src, T_dst, d);
  trace_end(s, "restage");
  return cudaGetLastError();
}

cudaError_t launch_restage_vec(const float* src, float* dst, size_t n_rows, int T_src, int T_dst,
                               float fill, cudaStream_t s) {
  trace_begin(s);
  restage_vec_kernel<<<blocks_for(n_rows * (size_t)T_dst), 256, 0, s>>>(src, dst, n_rows, T_src,
                                                                        T_dst, fill);
  trace_end(s, "restage_vec");
  return cudaGetLastError();
}

}  // namespace saf
