// api.cu — host side of the libsaf C ABI: argument checks, workspace carving,
// TMA descriptor encoding, head lists and the launch sequence of each call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/saf.h"
#include "attn_kernels.h"
#include "host_common.h"
#include "internal.h"

namespace saf {

static thread_local int g_launches = 0;

// Kernel trace: a per-thread list of (kernel, start event, end event).
struct TraceRec {
  const char* name;
  cudaEvent_t ev[2];
};
struct TraceState {
  bool on = false;
  std::vector<TraceRec> recs;   // recorded this trace
  std::vector<cudaEvent_t> pool;
  size_t next_event = 0;
  cudaEvent_t take() {
    if (next_event == pool.size()) {
      cudaEvent_t e = nullptr;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      pool.push_back(e);
    }
    return pool[next_event++];
  }
};
static thread_local TraceState g_trace;
static thread_local cudaEvent_t g_pending = nullptr;
constexpr size_t kMaxTraceRecords = 1u << 16;

void trace_begin(cudaStream_t s) {
  g_pending = nullptr;
  if (!g_trace.on || g_trace.recs.size() >= kMaxTraceRecords) return;
  g_pending = g_trace.take();
  if (g_pending) cudaEventRecord(g_pending, s);
}

void trace_end(cudaStream_t s, const char* kernel) {
  ++g_launches;
  if (!g_pending) return;
  cudaEvent_t e = g_trace.take();
  if (!e) return;
  cudaEventRecord(e, s);
  g_trace.recs.push_back(TraceRec{kernel, {g_pending, e}});
  g_pending = nullptr;
}

void launch_count_reset() { g_launches = 0; }

// Failure-path testing (saf_debug_forward_hold): read by every forward launch.
static std::atomic<int> g_dbg_hold{0};

cudaError_t set_max_dynamic_smem(const void* kernel, int bytes) {
  struct Done {
    const void* kernel;
    int device, bytes;
  };
  static std::mutex mu;
  static std::vector<Done> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const Done& d : done)
    if (d.kernel == kernel && d.device == dev && d.bytes == bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.push_back(Done{kernel, dev, bytes});
  return e;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

namespace {
EncodeTiledFn encode_fn() {
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
  return fn;
}
}  // namespace

// 2-D view [rows, d] of a bf16 tensor, box of 128 rows x one swizzle chunk.
bool encode_rows(CUtensorMap* m, const void* base, uint64_t rows, int d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int swz = d >= 64 ? 128 : 64;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {(cuuint32_t)(swz / 2), 128u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {
// 2-D view [rows, d] of an fp32 tensor, box of 128 rows x 32 columns (128 B,
// 128-byte swizzle): the staging layout of the backward's dQ reduction.
bool encode_rows_f32(CUtensorMap* m, const void* base, uint64_t rows, int d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 4};
  const cuuint32_t box[2] = {32u, 128u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------ workspace
struct WsLayout {
  size_t status, a_tab, r_tab, row_tab, logZ, mode;
  size_t q16, k16, v16, o16, do16, dq16, dk16, dv16;
  size_t Dvec, lse2, Dsum, dq_acc, dv_acc;
  size_t lse_p, ap, rp, dap, drp;  // padded copies (sequence length not a multiple of 128)
  size_t total;
};

}  // namespace

int kv_heads(const saf_attn_dims& d) { return d.H_kv > 0 ? d.H_kv : d.H; }

// The kernels work on whole 128-row tiles: a sequence length that is not a
// multiple of 128 runs on copies padded to the next multiple (zero rows of Q,
// K, V, dO; -inf entries of alpha and rho), cropped afterwards.  Padded keys
// lie above the causal diagonal of every real row, and padded rows carry
// dO = 0, so they change no output or gradient of the real rows.
saf_attn_dims padded_dims(const saf_attn_dims& d) {
  saf_attn_dims p = d;
  p.T = (d.T + 127) / 128 * 128;
  return p;
}

namespace {
WsLayout ws_layout(const saf_attn_dims& du) {
  WsLayout L;
  const saf_attn_dims d = padded_dims(du);
  const bool ragged = d.T != du.T;
  const size_t B = d.B, H = d.H, T = d.T, D = d.d_h;
  const size_t Hkv = (size_t)kv_heads(d);
  const size_t elems = B * H * T * D;
  const size_t elems_kv = B * Hkv * T * D;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L.status = take(256);
  L.a_tab = take(H * T * 4);
  L.r_tab = take(H * (T + 128) * 4);
  L.row_tab = take(H * T * 4);
  L.logZ = take(H * T * 4);
  L.mode = take(H * 8);  // H ints of mode, then H floats of shift
  const bool staged = d.dtype == SAF_F32 || ragged;
  const size_t stage = staged ? elems * 2 : 0;
  const size_t stage_kv = staged ? elems_kv * 2 : 0;
  L.q16 = take(stage);
  L.k16 = take(stage_kv);
  L.v16 = take(stage_kv);
  L.o16 = take(stage);
  L.do16 = take(stage);
  L.dq16 = take(stage);
  L.dk16 = take(stage_kv);
  L.dv16 = take(stage_kv);
  L.Dvec = take(B * H * T * 4);
  L.lse2 = take(B * H * T * 4);
  L.Dsum = take(H * T * 4);
  L.dq_acc = take(elems * 4);
  // grouped K/V: the frozen query heads' dV, summed per K/V head in fp32
  L.dv_acc = take(Hkv < H ? elems_kv * 4 : 0);
  L.lse_p = take(ragged ? B * H * T * 4 : 0);
  L.ap = take(ragged ? H * T * 4 : 0);
  L.rp = take(ragged ? H * T * 4 : 0);
  L.dap = take(ragged ? H * T * 4 : 0);
  L.drp = take(ragged ? H * T * 4 : 0);
  L.total = off;
  return L;
}

// The static tables of the workspace (every head has a slot).
StaticTables ws_tables(uint8_t* ws, const WsLayout& L, int H) {
  StaticTables t;
  t.a_tab = reinterpret_cast<float*>(ws + L.a_tab);
  t.r_tab = reinterpret_cast<float*>(ws + L.r_tab);
  t.row_tab = reinterpret_cast<float*>(ws + L.row_tab);
  t.logZ = reinterpret_cast<float*>(ws + L.logZ);
  t.mode = reinterpret_cast<int*>(ws + L.mode);
  t.shift = reinterpret_cast<float*>(ws + L.mode) + H;
  t.status = reinterpret_cast<int*>(ws + L.status);
  return t;
}
}  // namespace

saf_status check_dims(const saf_attn_dims* d) {
  if (!d) return SAF_ERR_INVALID_ARG;
  if (d->B < 0 || d->H < 0 || d->T < 0 || d->d_h < 1) return SAF_ERR_INVALID_ARG;
  if (d->dtype != SAF_BF16 && d->dtype != SAF_F32) return SAF_ERR_INVALID_ARG;
  if (d->H_kv < 0 || (d->H_kv > 0 && d->H % d->H_kv != 0)) return SAF_ERR_INVALID_ARG;
  if (d->H > kMaxHeads) return SAF_ERR_UNSUPPORTED;
  if (d->T > kMaxT) return SAF_ERR_UNSUPPORTED;
  if (d->d_h != 32 && d->d_h != 64 && d->d_h != 128) return SAF_ERR_UNSUPPORTED;
  const uint64_t t_pad = ((uint64_t)d->T + 127) / 128 * 128;
  if ((uint64_t)d->B * d->H * t_pad >= (1ull << 31)) return SAF_ERR_UNSUPPORTED;
  return SAF_OK;
}

HeadSplit split_heads(const uint8_t* head_is_static, int H) {
  HeadSplit s;
  memset(s.is_static, 0, sizeof(s.is_static));
  for (int h = 0; h < H; ++h) {
    if (head_is_static[h]) {
      s.st[s.n_static++] = (uint8_t)h;
      s.is_static[h] = 1;
    } else {
      s.dy[s.n_dynamic++] = (uint8_t)h;
    }
  }
  return s;
}

namespace {
saf_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SAF_OK : SAF_ERR_CUDA; }
}  // namespace

#define SAF_TRY(expr)                           \
  do {                                          \
    cudaError_t e_ = (expr);                    \
    if (e_ != cudaSuccess) return SAF_ERR_CUDA; \
  } while (0)

StaticPrep make_prep(const saf_attn_dims& d, const HeadSplit& hs, const float* alpha,
                     const float* rho, const StaticTables& t) {
  StaticPrep sp;
  memset(&sp, 0, sizeof(sp));
  sp.T = d.T;
  sp.n_static = hs.n_static;
  memcpy(sp.heads, hs.st, sizeof(sp.heads));
  sp.alpha = alpha;
  sp.rho = rho;
  sp.a_tab = t.a_tab;
  sp.r_tab = t.r_tab;
  sp.row_tab = t.row_tab;
  sp.logZ = t.logZ;
  sp.mode = t.mode;
  sp.shift = t.shift;
  return sp;
}

void fill_fwd_params(FwdParams& p, const saf_attn_dims& d, const HeadSplit& hs,
                     const StaticTables& t, bool transposed) {
  memset(&p, 0, sizeof(p));
  p.B = d.B;
  p.H = d.H;
  p.T = d.T;
  p.nI = d.T / 128;
  p.H_kv = kv_heads(d);
  p.group_kv = d.H / p.H_kv;
  p.n_static = hs.n_static;
  p.n_dynamic = transposed ? 0 : hs.n_dynamic;
  p.group = static_group(d.d_h, d.B, transposed);
  p.n_groups = (d.B + p.group - 1) / p.group;
  p.n_items = p.nI * (p.n_static * p.n_groups + (transposed ? 0 : d.B * hs.n_dynamic));
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)d.d_h);
  memcpy(p.static_heads, hs.st, sizeof(p.static_heads));
  memcpy(p.dynamic_heads, hs.dy, sizeof(p.dynamic_heads));
  p.a_tab = t.a_tab;
  p.r_tab = t.r_tab;
  p.row_tab = t.row_tab;
  p.logZ = t.logZ;
  p.mode = t.mode;
  p.shift = t.shift;
  p.status = t.status;
  if (!transposed) p.hold_first_q = g_dbg_hold.load();
}

}  // namespace saf

using namespace saf;

extern "C" {

const char* saf_status_string(saf_status s) {
  switch (s) {
    case SAF_OK: return "SAF_OK";
    case SAF_ERR_INVALID_ARG: return "SAF_ERR_INVALID_ARG";
    case SAF_ERR_UNSUPPORTED: return "SAF_ERR_UNSUPPORTED";
    case SAF_ERR_CUDA: return "SAF_ERR_CUDA";
    case SAF_ERR_STATE: return "SAF_ERR_STATE";
    case SAF_ERR_TIMEOUT: return "SAF_ERR_TIMEOUT";
  }
  return "SAF_ERR_UNKNOWN";
}

int saf_last_launch_count(void) { return g_launches; }

saf_status saf_debug_forward_hold(int hold) {
  g_dbg_hold.store(hold != 0);
  return SAF_OK;
}

saf_status saf_trace_enable(int enable) {
  g_trace.on = enable != 0;
  g_trace.recs.clear();
  g_trace.next_event = 0;
  return SAF_OK;
}

int saf_trace_count(void) { return (int)g_trace.recs.size(); }

saf_status saf_trace_get(int index, const char** kernel, float* ms) {
  if (index < 0 || index >= (int)g_trace.recs.size() || !kernel || !ms) return SAF_ERR_INVALID_ARG;
  const TraceRec& r = g_trace.recs[index];
  if (cudaEventSynchronize(r.ev[1]) != cudaSuccess) return SAF_ERR_CUDA;
  if (cudaEventElapsedTime(ms, r.ev[0], r.ev[1]) != cudaSuccess) return SAF_ERR_CUDA;
  *kernel = r.name;
  return SAF_OK;
}

size_t saf_hybrid_attn_workspace_size(const saf_attn_dims* dims, int want_param_grads) {
  (void)want_param_grads;  // the parameter-gradient pass needs no extra scratch
  if (check_dims(dims) != SAF_OK || empty_dims(*dims)) return 0;
  return ws_layout(*dims).total;
}

saf_status saf_hybrid_attn_fwd(const saf_attn_dims* dims, const void* Q, const void* K,
                               const void* V, const float* alpha, const float* rho,
                               const uint8_t* head_is_static, void* out, float* lse,
                               void* workspace, size_t ws_bytes, void* stream) {
  g_launches = 0;
  const saf_status ds = check_dims(dims);
  if (ds != SAF_OK) return ds;
  if (empty_dims(*dims)) return SAF_OK;  // nothing to compute
  const saf_attn_dims du = *dims;                 // the caller's shape
  const saf_attn_dims d = padded_dims(du);       // the kernels' shape
  const bool ragged = d.T != du.T;
  if (!head_is_static || !V || !out || !workspace) return SAF_ERR_INVALID_ARG;
  const HeadSplit hs = split_heads(head_is_static, d.H);
  if (hs.n_dynamic > 0 && (!Q || !K)) return SAF_ERR_INVALID_ARG;
  if (hs.n_static > 0 && (!alpha || !rho)) return SAF_ERR_INVALID_ARG;
  if ((Q && !aligned16(Q)) || (K && !aligned16(K)) || !aligned16(V) || !aligned16(out) ||
      (lse && !aligned16(lse)) || (alpha && !aligned16(alpha)) || (rho && !aligned16(rho)))
    return SAF_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SAF_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(du);
  if (ws_bytes < L.total) return SAF_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t slabs = (size_t)d.B * d.H, slabs_kv = (size_t)d.B * kv_heads(d);
  SAF_TRY(cudaMemsetAsync(ws + L.status, 0, sizeof(int), s));

  // fp32 I/O and ragged lengths run on bf16 copies of whole tiles
  const bool f32 = d.dtype == SAF_F32;
  const bool staged = f32 || ragged;
  const void *q16 = Q, *k16 = K, *v16 = V;
  void* o16 = out;
  if (staged) {
    if (hs.n_dynamic > 0) {
      SAF_TRY(launch_restage_rows(Q, f32, ws + L.q16, false, slabs, du.T, d.T, d.d_h, s));
      SAF_TRY(launch_restage_rows(K, f32, ws + L.k16, false, slabs_kv, du.T, d.T, d.d_h, s));
    }
    SAF_TRY(launch_restage_rows(V, f32, ws + L.v16, false, slabs_kv, du.T, d.T, d.d_h, s));
    q16 = ws + L.q16;
    k16 = ws + L.k16;
    v16 = ws + L.v16;
    o16 = ws + L.o16;
  }
  const float *alpha_k = alpha, *rho_k = rho;
  if (ragged && hs.n_static > 0) {
    float* ap = reinterpret_cast<float*>(ws + L.ap);
    float* rp = reinterpret_cast<float*>(ws + L.rp);
    SAF_TRY(launch_restage_vec(alpha, ap, d.H, du.T, d.T, -INFINITY, s));
    SAF_TRY(launch_restage_vec(rho, rp, d.H, du.T, d.T, -INFINITY, s));
    alpha_k = ap;
    rho_k = rp;
  }
  float* lse_k = (ragged && lse) ? reinterpret_cast<float*>(ws + L.lse_p) : lse;
  if (hs.n_static > 0)
    SAF_TRY(launch_static_prep(make_prep(d, hs, alpha_k, rho_k, ws_tables(ws, L, d.H)), s));

  FwdLaunch fl;
  memset(&fl, 0, sizeof(fl));
  fill_fwd_params(fl.p, d, hs, ws_tables(ws, L, d.H), false);
  fl.p.out = static_cast<__nv_bfloat16*>(o16);
  fl.p.lse = lse_k;
  const uint64_t rows = (uint64_t)d.B * d.H * d.T;
  const uint64_t rows_kv = (uint64_t)d.B * kv_heads(d) * d.T;
  // Q/K maps must be valid descriptors even when only static heads exist.
  const void* qb = q16 ? q16 : o16;
  const void* kb = k16 ? k16 : v16;
  if (!encode_rows(&fl.tm_q, qb, rows, d.d_h) || !encode_rows(&fl.tm_k, kb, rows_kv, d.d_h) ||
      !encode_rows(&fl.tm_v, v16, rows_kv, d.d_h) || !encode_rows(&fl.tm_o, o16, rows, d.d_h))
    return SAF_ERR_CUDA;
  fl.d_h = d.d_h;
  fl.transposed = false;
  fl.num_sms = sm_count();
  SAF_TRY(launch_hybrid_fwd(fl, s));
  if (staged) SAF_TRY(launch_restage_rows(o16, false, out, f32, slabs, d.T, du.T, d.d_h, s));
  if (ragged && lse) SAF_TRY(launch_restage_vec(lse_k, lse, slabs, d.T, du.T, 0.f, s));
  return SAF_OK;
}

saf_status saf_hybrid_attn_bwd(const saf_attn_dims* dims, const void* Q, const void* K,
                               const void* V, const void* out, const float* lse,
                               const void* dout, const float* alpha, const float* rho,
                               const uint8_t* head_is_static, void* dQ, void* dK, void* dV,
                               float* dalpha, float* drho, void* workspace, size_t ws_bytes,
                               void* stream) {
  g_launches = 0;
  const saf_status ds = check_dims(dims);
  if (ds != SAF_OK) return ds;
  if (empty_dims(*dims)) return SAF_OK;  // nothing to compute
  const saf_attn_dims du = *dims;                 // the caller's shape
  const saf_attn_dims d = padded_dims(du);       // the kernels' shape
  const bool ragged = d.T != du.T;
  if (!head_is_static || !V || !out || !lse || !dout || !dQ || !dK || !dV || !workspace)
    return SAF_ERR_INVALID_ARG;
  if ((dalpha == nullptr) != (drho == nullptr)) return SAF_ERR_INVALID_ARG;
  const HeadSplit hs = split_heads(head_is_static, d.H);
  if (hs.n_dynamic > 0 && (!Q || !K)) return SAF_ERR_INVALID_ARG;
  if (hs.n_static > 0 && (!alpha || !rho)) return SAF_ERR_INVALID_ARG;
  const void* ptrs[] = {V, out, lse, dout, dQ, dK, dV};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SAF_ERR_INVALID_ARG;
  if ((Q && !aligned16(Q)) || (K && !aligned16(K)) || (alpha && !aligned16(alpha)) ||
      (rho && !aligned16(rho)) || (dalpha && !aligned16(dalpha)) || (drho && !aligned16(drho)))
    return SAF_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SAF_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(du);
  if (ws_bytes < L.total) return SAF_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int Hkv = kv_heads(d), gkv = d.H / Hkv;
  const size_t elems_kv = (size_t)d.B * Hkv * d.T * d.d_h;
  const size_t slabs = (size_t)d.B * d.H, slabs_kv = (size_t)d.B * Hkv;
  const uint64_t rows = (uint64_t)d.B * d.H * d.T;
  const uint64_t rows_kv = (uint64_t)d.B * Hkv * d.T;
  SAF_TRY(cudaMemsetAsync(ws + L.status, 0, sizeof(int), s));

  // K/V heads: which serve dynamic query heads, which serve frozen ones
  uint8_t kv_has_dyn[kMaxHeads], kv_has_static[kMaxHeads];
  memset(kv_has_dyn, 0, sizeof(kv_has_dyn));
  memset(kv_has_static, 0, sizeof(kv_has_static));
  for (int h = 0; h < d.H; ++h) (hs.is_static[h] ? kv_has_static : kv_has_dyn)[h / gkv] = 1;
  float* dv_acc = (gkv > 1 && hs.n_static > 0) ? reinterpret_cast<float*>(ws + L.dv_acc) : nullptr;

  // fp32 I/O and ragged lengths run on bf16 copies of whole tiles
  const bool f32 = d.dtype == SAF_F32;
  const bool staged = f32 || ragged;
  const void *q16 = Q, *k16 = K, *v16 = V, *o16 = out, *do16 = dout;
  void *dq16 = dQ, *dk16 = dK, *dv16 = dV;
  if (staged) {
    if (hs.n_dynamic > 0) {
      SAF_TRY(launch_restage_rows(Q, f32, ws + L.q16, false, slabs, du.T, d.T, d.d_h, s));
      SAF_TRY(launch_restage_rows(K, f32, ws + L.k16, false, slabs_kv, du.T, d.T, d.d_h, s));
    }
    SAF_TRY(launch_restage_rows(V, f32, ws + L.v16, false, slabs_kv, du.T, d.T, d.d_h, s));
    SAF_TRY(launch_restage_rows(out, f32, ws + L.o16, false, slabs, du.T, d.T, d.d_h, s));
    SAF_TRY(launch_restage_rows(dout, f32, ws + L.do16, false, slabs, du.T, d.T, d.d_h, s));
    q16 = ws + L.q16;
    k16 = ws + L.k16;
    v16 = ws + L.v16;
    o16 = ws + L.o16;
    do16 = ws + L.do16;
    dq16 = ws + L.dq16;
    dk16 = ws + L.dk16;
    dv16 = ws + L.dv16;
  }
  // ragged lengths: lse of the padded rows 0 (their dO is 0, so P there
  // is finite and contributes nothing), alpha/rho padded with -inf, and
  // dalpha/drho formed over the padded length, then cropped
  const float *alpha_k = alpha, *rho_k = rho, *lse_k = lse;
  float *dalpha_k = dalpha, *drho_k = drho;
  if (ragged) {
    float* lp = reinterpret_cast<float*>(ws + L.lse_p);
    SAF_TRY(launch_restage_vec(lse, lp, slabs, du.T, d.T, 0.f, s));
    lse_k = lp;
    if (hs.n_static > 0) {
      float* ap = reinterpret_cast<float*>(ws + L.ap);
      float* rp = reinterpret_cast<float*>(ws + L.rp);
      SAF_TRY(launch_restage_vec(alpha, ap, d.H, du.T, d.T, -INFINITY, s));
      SAF_TRY(launch_restage_vec(rho, rp, d.H, du.T, d.T, -INFINITY, s));
      alpha_k = ap;
      rho_k = rp;
    }
    if (dalpha) {
      dalpha_k = reinterpret_cast<float*>(ws + L.dap);
      drho_k = reinterpret_cast<float*>(ws + L.drp);
    }
  }
  if (hs.n_static > 0)
    SAF_TRY(launch_static_prep(make_prep(d, hs, alpha_k, rho_k, ws_tables(ws, L, d.H)), s));

  // pre-pass: D, lse2, per-head batch sums of D for static heads
  BwdPre pre;
  memset(&pre, 0, sizeof(pre));
  pre.B = d.B; pre.H = d.H; pre.T = d.T; pre.d_h = d.d_h;
  pre.out = static_cast<const __nv_bfloat16*>(o16);
  pre.dout = static_cast<const __nv_bfloat16*>(do16);
  pre.lse = lse_k;
  pre.Dvec = reinterpret_cast<float*>(ws + L.Dvec);
  pre.lse2 = reinterpret_cast<float*>(ws + L.lse2);
  pre.Dsum = dalpha_k ? reinterpret_cast<float*>(ws + L.Dsum) : nullptr;
  pre.n_static = hs.n_static;
  memset(pre.static_slot, 255, sizeof(pre.static_slot));
  for (int i = 0; i < hs.n_static; ++i) pre.static_slot[hs.st[i]] = (uint8_t)i;
  if (hs.n_static > 0) {
    pre.row_tab = reinterpret_cast<float*>(ws + L.row_tab);
    pre.mode = reinterpret_cast<const int*>(ws + L.mode);
    pre.shift = reinterpret_cast<const float*>(ws + L.mode) + d.H;
  }
  memcpy(pre.static_heads, hs.st, sizeof(pre.static_heads));
  float* dq_acc = reinterpret_cast<float*>(ws + L.dq_acc);
  pre.dq_acc = hs.n_dynamic > 0 ? dq_acc : nullptr;
  SAF_TRY(launch_bwd_pre(pre, s));

  if (hs.n_static > 0) {
    // dV = P^T dO for the frozen heads: the forward's static engine,
    // transposed.  With grouped K/V it adds into an fp32 sum per K/V head,
    // which the dynamic pass (or the post-pass) folds into dV.
    if (dv_acc) SAF_TRY(cudaMemsetAsync(dv_acc, 0, elems_kv * sizeof(float), s));
    FwdLaunch fl;
    memset(&fl, 0, sizeof(fl));
    fill_fwd_params(fl.p, d, hs, ws_tables(ws, L, d.H), true);
    fl.p.out = static_cast<__nv_bfloat16*>(dv16);
    fl.p.out_acc = dv_acc;
    fl.p.lse = nullptr;
    if (!encode_rows(&fl.tm_q, do16, rows, d.d_h) || !encode_rows(&fl.tm_k, do16, rows, d.d_h) ||
        !encode_rows(&fl.tm_v, do16, rows, d.d_h))
      return SAF_ERR_CUDA;
    fl.d_h = d.d_h;
    fl.transposed = true;
    fl.num_sms = sm_count();
    SAF_TRY(launch_hybrid_fwd(fl, s));
  }
  if (hs.n_dynamic > 0) {
    BwdLaunch bl;
    memset(&bl, 0, sizeof(bl));
    BwdParams& p = bl.p;
    p.B = d.B; p.H = d.H; p.T = d.T; p.nI = d.T / 128;
    p.H_kv = Hkv;
    int nd = 0;
    for (int kv = 0; kv < Hkv; ++kv) {
      p.dyn_begin[kv] = (uint16_t)nd;
      for (int h = kv * gkv; h < (kv + 1) * gkv; ++h)
        if (!hs.is_static[h]) p.dyn_by_kv[nd++] = (uint8_t)h;
      p.dyn_count[kv] = (uint16_t)(nd - p.dyn_begin[kv]);
      if (p.dyn_count[kv] > 0) p.kv_list[p.n_kv++] = (uint8_t)kv;
      p.kv_has_static[kv] = kv_has_static[kv];
    }
    p.n_items = p.nI * d.B * p.n_kv;
    {
      // Items in groups of (sequence, K/V head) pairs when the dQ accumulator,
      // Q and dO of all pairs exceed half of L2: about five rounds of the
      // grid per group keeps the group's working set in L2 (a third to a
      // quarter of the DRAM traffic measured on the 124M and 1B layers) at
      // no cost in time; smaller groups leave long items for the tail.
      const int n_pairs = d.B * p.n_kv;
      int max_dyn = 1;
      for (int i = 0; i < p.n_kv; ++i)
        max_dyn = p.dyn_count[p.kv_list[i]] > max_dyn ? p.dyn_count[p.kv_list[i]] : max_dyn;
      const double ws = (double)n_pairs * max_dyn * d.T * d.d_h * 8.0;
      const int sms = sm_count();
      int G = (int)((5.0 * sms) / p.nI + 0.5);
      if (ws <= 64.0 * 1024 * 1024 || G >= n_pairs) G = n_pairs;
      p.pairs_per_group = G < 1 ? 1 : G;
    }
    p.scale = 1.0f / sqrtf((float)d.d_h);
    p.scale_log2 = 1.4426950408889634f * p.scale;
    p.dv_acc = dv_acc;
    p.lse2 = pre.lse2;
    p.Dvec = pre.Dvec;
    p.dq_acc = dq_acc;
    p.dK = static_cast<__nv_bfloat16*>(dk16);
    p.dV = static_cast<__nv_bfloat16*>(dv16);
    p.status = reinterpret_cast<int*>(ws + L.status);
    if (!encode_rows(&bl.tm_q, q16, rows, d.d_h) || !encode_rows(&bl.tm_k, k16, rows_kv, d.d_h) ||
        !encode_rows(&bl.tm_v, v16, rows_kv, d.d_h) || !encode_rows(&bl.tm_do, do16, rows, d.d_h) ||
        !encode_rows_f32(&bl.tm_dq, dq_acc, rows, d.d_h))
      return SAF_ERR_CUDA;
    bl.d_h = d.d_h;
    bl.num_sms = sm_count();
    SAF_TRY(launch_bwd_dynamic(bl, s));
  }
  if (dalpha_k) {
    SAF_TRY(launch_zero_u32(dalpha_k, (size_t)d.H * d.T, s));
    SAF_TRY(launch_zero_u32(drho_k, (size_t)d.H * d.T, s));
    if (hs.n_static > 0) {
      ParamGradLaunch gl;
      memset(&gl, 0, sizeof(gl));
      ParamGradParams& p = gl.p;
      p.B = d.B; p.H = d.H; p.T = d.T; p.nI = d.T / 128;
      p.H_kv = Hkv;
      p.group_kv = gkv;
      p.n_static = hs.n_static;
      p.n_items = hs.n_static * p.nI;
      memcpy(p.static_heads, hs.st, sizeof(p.static_heads));
      p.a_tab = reinterpret_cast<const float*>(ws + L.a_tab);
      p.r_tab = reinterpret_cast<const float*>(ws + L.r_tab);
      p.row_tab = reinterpret_cast<const float*>(ws + L.row_tab);
      p.mode = reinterpret_cast<const int*>(ws + L.mode);
      p.Dsum = pre.Dsum;
      p.dalpha = dalpha_k;
      p.drho = drho_k;
      p.status = reinterpret_cast<int*>(ws + L.status);
      if (!encode_rows(&gl.tm_v, v16, rows_kv, d.d_h) || !encode_rows(&gl.tm_do, do16, rows, d.d_h))
        return SAF_ERR_CUDA;
      gl.d_h = d.d_h;
      gl.num_sms = sm_count();
      SAF_TRY(launch_param_grads(gl, s));
    }
  }
  BwdPost post;
  memset(&post, 0, sizeof(post));
  post.B = d.B; post.H = d.H; post.T = d.T; post.d_h = d.d_h; post.H_kv = Hkv;
  post.dq_acc = dq_acc;
  post.dQ = static_cast<__nv_bfloat16*>(dq16);
  post.dK = static_cast<__nv_bfloat16*>(dk16);
  post.dV = static_cast<__nv_bfloat16*>(dv16);
  post.dv_acc = dv_acc;
  memcpy(post.is_static, hs.is_static, sizeof(post.is_static));
  for (int kv = 0; kv < Hkv; ++kv) post.kv_no_dyn[kv] = kv_has_dyn[kv] ? 0 : 1;
  SAF_TRY(launch_bwd_post(post, s));
  if (staged) {
    SAF_TRY(launch_restage_rows(dq16, false, dQ, f32, slabs, d.T, du.T, d.d_h, s));
    SAF_TRY(launch_restage_rows(dk16, false, dK, f32, slabs_kv, d.T, du.T, d.d_h, s));
    SAF_TRY(launch_restage_rows(dv16, false, dV, f32, slabs_kv, d.T, du.T, d.d_h, s));
  }
  if (ragged && dalpha) {
    SAF_TRY(launch_restage_vec(dalpha_k, dalpha, d.H, d.T, du.T, 0.f, s));
    SAF_TRY(launch_restage_vec(drho_k, drho, d.H, d.T, du.T, 0.f, s));
  }
  return SAF_OK;
}

// ------------------------------------------------------------ calibration
namespace {
struct CalibHandle {
  int num_heads = 0, T = 0;
  float* mean = nullptr;
  float* m2 = nullptr;
  float* ent = nullptr;  // sum_n x log x (only with SAF_CALIB_TRACK_KL)
  double* partials = nullptr;
  int* status = nullptr;
  std::vector<int> counts;
};
}  // namespace

saf_status saf_calib_create_ex(void** handle, int num_heads, int T, unsigned flags) {
  g_launches = 0;
  if (!handle) return SAF_ERR_INVALID_ARG;
  *handle = nullptr;
  if (num_heads < 1 || T < 4 || T % 4 != 0) return SAF_ERR_INVALID_ARG;
  if ((flags & ~(unsigned)SAF_CALIB_TRACK_KL) != 0) return SAF_ERR_INVALID_ARG;
  if (T > kMaxT || num_heads > 8192) return SAF_ERR_UNSUPPORTED;
  CalibHandle* h = new CalibHandle();
  h->num_heads = num_heads;
  h->T = T;
  h->counts.assign(num_heads, 0);
  const size_t n = (size_t)num_heads * T * T;
  const bool kl = (flags & SAF_CALIB_TRACK_KL) != 0;
  if (cudaMalloc(&h->mean, n * 4) != cudaSuccess || cudaMalloc(&h->m2, n * 4) != cudaSuccess ||
      (kl && cudaMalloc(&h->ent, n * 4) != cudaSuccess) ||
      cudaMalloc(&h->partials, (size_t)num_heads * T * 8) != cudaSuccess ||
      cudaMalloc(&h->status, 256) != cudaSuccess || cudaMemset(h->status, 0, 256) != cudaSuccess) {
    cudaFree(h->mean);
    cudaFree(h->m2);
    cudaFree(h->ent);
    cudaFree(h->partials);
    cudaFree(h->status);
    delete h;
    return SAF_ERR_CUDA;
  }
  *handle = h;
  return SAF_OK;
}

saf_status saf_calib_create(void** handle, int num_heads, int T) {
  return saf_calib_create_ex(handle, num_heads, T, 0u);
}

saf_status saf_calib_accumulate(void* handle, const float* A, int n, int head_begin,
                                int head_count, void* stream) {
  g_launches = 0;
  CalibHandle* h = static_cast<CalibHandle*>(handle);
  if (!h || n < 0 || head_count < 0 || head_begin < 0 || head_begin + head_count > h->num_heads)
    return SAF_ERR_INVALID_ARG;
  if (n == 0 || head_count == 0) return SAF_OK;  // no samples: nothing changes
  if (!A || !aligned16(A)) return SAF_ERR_INVALID_ARG;
  const int c0 = h->counts[head_begin];
  for (int i = head_begin; i < head_begin + head_count; ++i)
    if (h->counts[i] != c0) return SAF_ERR_STATE;
  CalibLaunch p;
  p.A = A;
  p.n = n;
  p.head_begin = head_begin;
  p.head_count = head_count;
  p.T = h->T;
  p.count0 = c0;
  p.mean = h->mean;
  p.m2 = h->m2;
  p.ent = h->ent;
  const cudaError_t e = launch_calib_accumulate(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return SAF_ERR_CUDA;
  for (int i = head_begin; i < head_begin + head_count; ++i) h->counts[i] += n;
  return SAF_OK;
}

int saf_calib_num_select(double r, int num_heads) {
  const double x = r * (double)num_heads;
  return (int)nearbyint(x);  // default rounding mode: ties to even
}

saf_status saf_calib_finalize(void* handle, int k, float* A_hat, float* s_var, int32_t* selected,
                              void* stream) {
  g_launches = 0;
  CalibHandle* h = static_cast<CalibHandle*>(handle);
  if (!h || !s_var || !aligned16(s_var) || (A_hat && !aligned16(A_hat))) return SAF_ERR_INVALID_ARG;
  if (k < 0 || k > h->num_heads || (k > 0 && !selected)) return SAF_ERR_INVALID_ARG;
  const int N = h->counts[0];
  for (int c : h->counts)
    if (c != N) return SAF_ERR_STATE;
  if (N < 2) return SAF_ERR_STATE;
  CalibFinalize p;
  p.num_heads = h->num_heads;
  p.T = h->T;
  p.N = N;
  p.k = k;
  p.mean = h->mean;
  p.m2 = h->m2;
  p.row_partials = h->partials;
  p.A_hat = A_hat;
  p.s_var = s_var;
  p.selected = selected;
  p.ent = nullptr;
  return cuda_status(launch_calib_finalize(p, static_cast<cudaStream_t>(stream)));
}

saf_status saf_calib_finalize_kl(void* handle, int k, float* s_kl, int32_t* selected,
                                 void* stream) {
  g_launches = 0;
  CalibHandle* h = static_cast<CalibHandle*>(handle);
  if (!h || !s_kl || !aligned16(s_kl)) return SAF_ERR_INVALID_ARG;
  if (k < 0 || k > h->num_heads || (k > 0 && !selected)) return SAF_ERR_INVALID_ARG;
  if (!h->ent) return SAF_ERR_STATE;
  const int N = h->counts[0];
  for (int c : h->counts)
    if (c != N) return SAF_ERR_STATE;
  if (N < 1) return SAF_ERR_STATE;
  CalibFinalize p;
  p.num_heads = h->num_heads;
  p.T = h->T;
  p.N = N;
  p.k = k;
  p.mean = h->mean;
  p.m2 = h->m2;
  p.row_partials = h->partials;
  p.A_hat = nullptr;
  p.s_var = s_kl;
  p.selected = selected;
  p.ent = h->ent;
  return cuda_status(launch_calib_finalize_kl(p, static_cast<cudaStream_t>(stream)));
}

saf_status saf_calib_finalize_sharp(void* handle, float* pattern, void* stream) {
  g_launches = 0;
  CalibHandle* h = static_cast<CalibHandle*>(handle);
  if (!h || !pattern) return SAF_ERR_INVALID_ARG;
  const int N = h->counts[0];
  for (int c : h->counts)
    if (c != N) return SAF_ERR_STATE;
  if (N < 1) return SAF_ERR_STATE;
  return cuda_status(
      launch_calib_sharp(h->mean, h->num_heads, h->T, pattern, static_cast<cudaStream_t>(stream)));
}

saf_status saf_fit_compact(const float* A_hat, int num_heads, int T, const int32_t* candidates,
                           int n_candidates, int k, float kl_max, int steps, float lr,
                           float* alpha, float* rho, float* kl, int32_t* selected,
                           int32_t* n_selected, void* stream) {
  g_launches = 0;
  if (!A_hat || !candidates || !alpha || !rho || !kl || !n_selected) return SAF_ERR_INVALID_ARG;
  if (num_heads < 1 || T < 1 || n_candidates < 1 || steps < 0 || k < 0 || k > n_candidates)
    return SAF_ERR_INVALID_ARG;
  if (k > 0 && !selected) return SAF_ERR_INVALID_ARG;
  if (!(lr > 0.f) || !(kl_max >= 0.f)) return SAF_ERR_INVALID_ARG;
  if (T > 4096) return SAF_ERR_UNSUPPORTED;
  if (!aligned16(A_hat) || !aligned16(alpha) || !aligned16(rho)) return SAF_ERR_INVALID_ARG;
  FitParams p;
  p.A_hat = A_hat;
  p.T = T;
  p.candidates = candidates;
  p.n_candidates = n_candidates;
  p.k = k;
  p.kl_max = kl_max;
  p.steps = steps;
  p.lr = lr;
  p.beta1 = 0.9f;
  p.beta2 = 0.999f;
  p.eps = 1e-8f;
  p.alpha = alpha;
  p.rho = rho;
  p.kl = kl;
  p.selected = selected;
  p.n_selected = n_selected;
  return cuda_status(launch_fit(p, static_cast<cudaStream_t>(stream)));
}

saf_status saf_calib_reset(void* handle) {
  CalibHandle* h = static_cast<CalibHandle*>(handle);
  if (!h) return SAF_ERR_INVALID_ARG;
  for (int& c : h->counts) c = 0;
  return SAF_OK;
}

saf_status saf_calib_destroy(void* handle) {
  CalibHandle* h = static_cast<CalibHandle*>(handle);
  if (!h) return SAF_OK;
  cudaDeviceSynchronize();
  cudaFree(h->mean);
  cudaFree(h->m2);
  cudaFree(h->ent);
  cudaFree(h->partials);
  cudaFree(h->status);
  delete h;
  return SAF_OK;
}

saf_status saf_get_device_status(void* workspace_or_handle, int is_calib_handle, int* site,
                                 void* stream) {
  if (site) *site = 0;
  if (!workspace_or_handle) return SAF_ERR_INVALID_ARG;
  int* word = is_calib_handle ? static_cast<CalibHandle*>(workspace_or_handle)->status
                              : static_cast<int*>(workspace_or_handle);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, word, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(word, 0, sizeof(int), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return SAF_ERR_CUDA;
  if (site) *site = v;
  return v == 0 ? SAF_OK : SAF_ERR_TIMEOUT;
}

}  // extern "C"
