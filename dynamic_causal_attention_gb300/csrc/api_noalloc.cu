// api_noalloc.cu — saf_hybrid_attn_fwd_noalloc, a forward entry point that
// allocates nothing.
//
// saf_hybrid_attn_fwd needs a caller-provided workspace for its scratch (the
// frozen heads' generator tables, log Z and a status word).  Some callers
// cannot provide one: an inference-engine plugin whose enqueue step must not
// allocate (the engine owns every byte of device memory and plans it ahead),
// or code that only ever receives input and output pointers.  For them this
// file keeps that scratch in one file-scope __device__ array of fixed size,
// which every GPU that loads the library holds until the process exits.  The
// argument checks, the launch parameters and the kernels are those of
// saf_hybrid_attn_fwd; only where the scratch lives differs.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/saf.h"
#include "attn_kernels.h"
#include "host_common.h"
#include "internal.h"

namespace saf {
namespace {

// Largest scratch the no-allocation forward may use: 4 MiB.  The frozen
// heads' tables take n_static * (4 T + 130) * 4 bytes plus at most 1.5 KiB of
// status word and alignment, e.g. 15 frozen heads at T = 16384 or 16 at
// T = 16256 (16 at T = 16384 does not fit).
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

// The scratch holds one table slot per frozen head (not per head, as the
// workspace of saf_hybrid_attn_fwd does).
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

StaticTables scratch_tables(uint8_t* ws, const ScratchLayout& L, int n_static) {
  StaticTables t;
  t.a_tab = reinterpret_cast<float*>(ws + L.a_tab);
  t.r_tab = reinterpret_cast<float*>(ws + L.r_tab);
  t.row_tab = reinterpret_cast<float*>(ws + L.row_tab);
  t.logZ = reinterpret_cast<float*>(ws + L.logZ);
  t.mode = reinterpret_cast<int*>(ws + L.mode);
  t.shift = reinterpret_cast<float*>(ws + L.mode) + n_static;
  t.status = reinterpret_cast<int*>(ws + L.status);
  return t;
}

}  // namespace
}  // namespace saf

using namespace saf;

extern "C" saf_status saf_hybrid_attn_fwd_noalloc(const saf_attn_dims* dims, const void* Q,
                                                  const void* K, const void* V,
                                                  const float* alpha, const float* rho,
                                                  const uint8_t* head_is_static, void* out,
                                                  float* lse, void* stream) {
  launch_count_reset();
  const saf_status ds = check_dims(dims);
  if (ds != SAF_OK) return ds;
  if (empty_dims(*dims)) return SAF_OK;  // nothing to compute
  const saf_attn_dims d = *dims;
  // fp32 I/O and lengths that are not a multiple of 128 need staging buffers
  if (d.dtype != SAF_BF16 || d.T % 128 != 0) return SAF_ERR_UNSUPPORTED;
  if (!head_is_static || !V || !out) return SAF_ERR_INVALID_ARG;
  const HeadSplit hs = split_heads(head_is_static, d.H);
  if (hs.n_dynamic > 0 && (!Q || !K)) return SAF_ERR_INVALID_ARG;
  if (hs.n_static > 0 && (!alpha || !rho)) return SAF_ERR_INVALID_ARG;
  if ((Q && !aligned16(Q)) || (K && !aligned16(K)) || !aligned16(V) || !aligned16(out) ||
      (lse && !aligned16(lse)) || (alpha && !aligned16(alpha)) || (rho && !aligned16(rho)))
    return SAF_ERR_INVALID_ARG;
  // The scratch is a fixed-size array: shapes whose tables do not fit are
  // rejected before anything is launched.
  const ScratchLayout L = scratch_layout(hs.n_static, d.T);
  if (L.total > kNoAllocScratchBytes) return SAF_ERR_UNSUPPORTED;
  uint8_t* ws = nullptr;
  const saf_status ss = scratch_on_current_device(&ws);
  if (ss != SAF_OK) return ss;
  const StaticTables tabs = scratch_tables(ws, L, hs.n_static);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: the status word must start
  // at zero; the tables are fully rewritten by the pre-pass.
  if (cudaMemsetAsync(tabs.status, 0, sizeof(int), s) != cudaSuccess) return SAF_ERR_CUDA;
  if (hs.n_static > 0 && launch_static_prep(make_prep(d, hs, alpha, rho, tabs), s) != cudaSuccess)
    return SAF_ERR_CUDA;

  FwdLaunch fl;
  memset(&fl, 0, sizeof(fl));
  fill_fwd_params(fl.p, d, hs, tabs, false);
  fl.p.out = static_cast<__nv_bfloat16*>(out);
  fl.p.lse = lse;
  const uint64_t rows = (uint64_t)d.B * d.H * d.T;
  const uint64_t rows_kv = (uint64_t)d.B * kv_heads(d) * d.T;
  // Q/K maps must be valid descriptors even when only static heads exist.
  const void* qb = Q ? Q : out;
  const void* kb = K ? K : V;
  if (!encode_rows(&fl.tm_q, qb, rows, d.d_h) || !encode_rows(&fl.tm_k, kb, rows_kv, d.d_h) ||
      !encode_rows(&fl.tm_v, V, rows_kv, d.d_h) || !encode_rows(&fl.tm_o, out, rows, d.d_h))
    return SAF_ERR_CUDA;
  fl.d_h = d.d_h;
  fl.transposed = false;
  fl.num_sms = sm_count();
  if (launch_hybrid_fwd(fl, s) != cudaSuccess) return SAF_ERR_CUDA;
  return SAF_OK;
}
