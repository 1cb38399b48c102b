// host_common.h — host-side helpers shared by the attention entry points
// (api.cu and api_noalloc.cu): argument checks, the split of heads into
// frozen and dynamic ones, the launch parameters of the fused forward and
// the TMA tensor maps of the [rows, d_h] bf16 views.  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/saf.h"
#include "attn_kernels.h"

namespace saf {

constexpr int kMaxT = 16384;  // longest sequence the attention calls accept

bool aligned16(const void* p);
size_t align256(size_t x);
int sm_count();  // of the current device
int kv_heads(const saf_attn_dims& d);

// SAF_OK, or the status an attention call returns for these dimensions.
saf_status check_dims(const saf_attn_dims* d);
// B, H or T zero: a layer with nothing to compute (valid; the calls return
// SAF_OK at once, touching no pointer).
inline bool empty_dims(const saf_attn_dims& d) { return d.B == 0 || d.H == 0 || d.T == 0; }

struct HeadSplit {
  int n_static = 0, n_dynamic = 0;
  uint8_t st[kMaxHeads], dy[kMaxHeads], is_static[kMaxHeads];
};
HeadSplit split_heads(const uint8_t* head_is_static, int H);

// Device scratch of the frozen heads' pre-pass, wherever the caller keeps it.
struct StaticTables {
  float* a_tab;    // [slots, T]
  float* r_tab;    // [slots, T + 128]
  float* row_tab;  // [slots, T]
  float* logZ;     // [slots, T]
  int* mode;       // [slots]
  float* shift;    // [slots]
  int* status;     // device status word
};
StaticPrep make_prep(const saf_attn_dims& d, const HeadSplit& hs, const float* alpha,
                     const float* rho, const StaticTables& t);
void fill_fwd_params(FwdParams& p, const saf_attn_dims& d, const HeadSplit& hs,
                     const StaticTables& t, bool transposed);

// 2-D view [rows, d] of a bf16 tensor, box of 128 rows x one swizzle chunk.
bool encode_rows(CUtensorMap* m, const void* base, uint64_t rows, int d);

}  // namespace saf
