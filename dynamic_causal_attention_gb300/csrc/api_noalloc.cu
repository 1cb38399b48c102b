// api_noalloc.cu — saf_hybrid_attn_fwd_noalloc, a forward entry point that
// allocates nothing.
//
// saf_hybrid_attn_fwd needs a caller-provided workspace for its scratch (the
// frozen heads' generator tables, log Z and a status word).  Some callers
// cannot provide one: an inference-engine plugin whose enqueue step must not
// allocate (the engine owns every byte of device memory and plans it ahead),
// or code that only ever receives input and output pointers.  For them this
// file keeps that scratch in one file-scope __device__ array of fixed size,
// which every GPU that loads the library holds until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/saf.h"
#include "attn_kernels.h"
#include "internal.h"

namespace saf {
namespace {

// Largest scratch the no-allocation forward may use: 4 MiB, enough for
// n_static * (4 T + 128) floats plus 1 KiB (e.g. 16 frozen heads at T = 16384).
constexpr size_t kNoAllocScratchBytes = 4u << 20;

static __device__ __align__(256) unsigned char g_fwd_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_fwd_scratch on the current device, looked up once per
// device (the host-side name of the array is not a device address).
saf_status scratch_on_current_device(uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SAF_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_scratch) != cudaSuccess || p == nullptr)
      return SAF_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = static_cast<uint8_t*>(g_scratch_ptr[dev]);
  return SAF_OK;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct ScratchLayout {
  size_t status, a_tab, r_tab, row_tab, logZ, mode, total;
};

ScratchLayout scratch_layout(int n_static, int T) {
  ScratchLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const size_t hs = (size_t)n_static, t = (size_t)T;
  L.status = take(256);
  L.a_tab = take(hs * t * 4);
  L.r_tab = take(hs * (t + 128) * 4);
  L.row_tab = take(hs * t * 4);
  L.logZ = take(hs * t * 4);
  L.mode = take(hs * 8);  // n_static ints of mode, then n_static floats of shift
  L.total = off;
  return L;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool encode_rows_na(CUtensorMap* m, const void* base, uint64_t rows, int d) {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!fn) return false;
  const int swz = d >= 64 ? 128 : 64;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {(cuuint32_t)(swz / 2), 128u};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace saf

using namespace saf;

extern "C" saf_status saf_hybrid_attn_fwd_noalloc(const saf_attn_dims* dims, const void* Q,
                                                  const void* K, const void* V,
                                                  const float* alpha, const float* rho,
                                                  const uint8_t* head_is_static, void* out,
                                                  float* lse, void* stream) {
  if (!dims || !head_is_static || !V || !out) return SAF_ERR_INVALID_ARG;
  const saf_attn_dims d = *dims;
  if (d.B < 1 || d.H < 1 || d.T < 1 || d.d_h < 1) return SAF_ERR_INVALID_ARG;
  if (d.dtype != SAF_BF16) return SAF_ERR_UNSUPPORTED;  // fp32 I/O needs staging buffers
  if (d.H > kMaxHeads || d.T % 128 != 0 || d.T > 16384) return SAF_ERR_UNSUPPORTED;
  if (d.d_h != 32 && d.d_h != 64 && d.d_h != 128) return SAF_ERR_UNSUPPORTED;
  if ((uint64_t)d.B * d.H * d.T >= (1ull << 31)) return SAF_ERR_UNSUPPORTED;
  if (d.H_kv < 0 || (d.H_kv > 0 && d.H % d.H_kv != 0)) return SAF_ERR_INVALID_ARG;
  const int Hkv = d.H_kv > 0 ? d.H_kv : d.H;
  int n_static = 0, n_dynamic = 0;
  uint8_t st[kMaxHeads], dy[kMaxHeads];
  for (int h = 0; h < d.H; ++h) {
    if (head_is_static[h]) st[n_static++] = (uint8_t)h;
    else dy[n_dynamic++] = (uint8_t)h;
  }
  if (n_dynamic > 0 && (!Q || !K)) return SAF_ERR_INVALID_ARG;
  if (n_static > 0 && (!alpha || !rho)) return SAF_ERR_INVALID_ARG;
  if ((Q && !aligned16(Q)) || (K && !aligned16(K)) || !aligned16(V) || !aligned16(out) ||
      (lse && !aligned16(lse)) || (alpha && !aligned16(alpha)) || (rho && !aligned16(rho)))
    return SAF_ERR_INVALID_ARG;
  // The scratch is a fixed-size array: shapes whose tables do not fit are
  // rejected before anything is launched.
  const ScratchLayout L = scratch_layout(n_static, d.T);
  if (L.total > kNoAllocScratchBytes) return SAF_ERR_UNSUPPORTED;
  uint8_t* ws = nullptr;
  const saf_status ss = scratch_on_current_device(&ws);
  if (ss != SAF_OK) return ss;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the status word must start
  // at zero; the tables are fully rewritten by the pre-pass.
  if (cudaMemsetAsync(ws + L.status, 0, sizeof(int), s) != cudaSuccess) return SAF_ERR_CUDA;

  if (n_static > 0) {
    StaticPrep sp;
    memset(&sp, 0, sizeof(sp));
    sp.T = d.T;
    sp.n_static = n_static;
    memcpy(sp.heads, st, (size_t)n_static);
    sp.alpha = alpha;
    sp.rho = rho;
    sp.a_tab = reinterpret_cast<float*>(ws + L.a_tab);
    sp.r_tab = reinterpret_cast<float*>(ws + L.r_tab);
    sp.row_tab = reinterpret_cast<float*>(ws + L.row_tab);
    sp.logZ = reinterpret_cast<float*>(ws + L.logZ);
    sp.mode = reinterpret_cast<int*>(ws + L.mode);
    sp.shift = reinterpret_cast<float*>(ws + L.mode) + n_static;
    if (launch_static_prep(sp, s) != cudaSuccess) return SAF_ERR_CUDA;
  }

  FwdLaunch fl;
  memset(&fl, 0, sizeof(fl));
  FwdParams& p = fl.p;
  p.B = d.B;
  p.H = d.H;
  p.T = d.T;
  p.nI = d.T / 128;
  p.H_kv = Hkv;
  p.group_kv = d.H / Hkv;
  p.n_static = n_static;
  p.n_dynamic = n_dynamic;
  p.group = static_group(d.d_h, d.B);
  p.n_groups = (d.B + p.group - 1) / p.group;
  p.n_items = p.nI * (n_static * p.n_groups + d.B * n_dynamic);
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)d.d_h);
  memcpy(p.static_heads, st, (size_t)n_static);
  memcpy(p.dynamic_heads, dy, (size_t)n_dynamic);
  p.a_tab = reinterpret_cast<const float*>(ws + L.a_tab);
  p.r_tab = reinterpret_cast<const float*>(ws + L.r_tab);
  p.row_tab = reinterpret_cast<const float*>(ws + L.row_tab);
  p.logZ = reinterpret_cast<const float*>(ws + L.logZ);
  p.mode = reinterpret_cast<const int*>(ws + L.mode);
  p.shift = reinterpret_cast<const float*>(ws + L.mode) + n_static;
  p.status = reinterpret_cast<int*>(ws + L.status);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  const uint64_t rows = (uint64_t)d.B * d.H * d.T;
  const uint64_t rows_kv = (uint64_t)d.B * Hkv * d.T;
  const void* qb = Q ? Q : out;
  const void* kb = K ? K : V;
  if (!encode_rows_na(&fl.tm_q, qb, rows, d.d_h) || !encode_rows_na(&fl.tm_k, kb, rows_kv, d.d_h) ||
      !encode_rows_na(&fl.tm_v, V, rows_kv, d.d_h) || !encode_rows_na(&fl.tm_o, out, rows, d.d_h))
    return SAF_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SAF_ERR_CUDA;
  fl.d_h = d.d_h;
  fl.transposed = false;
  fl.num_sms = sms;
  if (launch_hybrid_fwd(fl, s) != cudaSuccess) return SAF_ERR_CUDA;
  return SAF_OK;
}
