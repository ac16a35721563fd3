// kda_internal.cuh -- shared device/host helpers of the KDA CUDA library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Workspace header: the device status word and scheduler counters live in the
// first 256 bytes; per-path scratch follows at kWsPayload.
struct WsHeader {
  uint32_t status;        // KDA_DEVICE_* bits
  uint32_t next_item;     // dynamic work counter of the persistent prefill
  uint32_t num_entries;   // work-list entries written by the planning kernel
  uint32_t num_splits;    // sequences the planning kernel cut in two
  uint32_t reserved[60];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");
constexpr size_t kWsPayload = 256;

__device__ __forceinline__ void raise_status(uint32_t* status, uint32_t bit) {
  atomicOr(status, bit);
}

// Bounds checks of computed indices in the debug build (compiled with -DKDA_DEBUG): a failed
// check records itself in a per-file device flag and the access it guards is skipped (never a
// trap); each kernel folds the flag into KDA_DEVICE_DEBUG_BOUNDS of its status word before it
// returns.  In the normal build KDA_CHECK(c) is the constant true and costs nothing.
#ifdef KDA_DEBUG
#define KDA_DEBUG_FLAG_DEFINE() static __device__ unsigned int g_kda_bounds = 0
#define KDA_CHECK(c) ((c) ? true : (atomicOr(&g_kda_bounds, 1u), false))
#define KDA_DEBUG_FOLD(status) \
  do { if (*(volatile unsigned int*)&g_kda_bounds) atomicOr((status), KDA_DEVICE_DEBUG_BOUNDS); } while (0)
#else
#define KDA_DEBUG_FLAG_DEFINE() static_assert(true, "")
#define KDA_CHECK(c) (true || (c))  // never evaluated; keeps the operands referenced
#define KDA_DEBUG_FOLD(status) do { } while (0)
#endif

// ---- element conversions ----------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);  // round to nearest even
}

// Resolved per-sequence state slot: index -1 -> sentinel (num_slots - 1);
// returns -1 for an index outside [-1, num_slots).
__device__ __forceinline__ int64_t resolve_slot(const int32_t* idx, int n, int64_t num_slots) {
  const int32_t s = idx[n];
  if (s < -1 || (int64_t)s >= num_slots) return -1;
  return s < 0 ? num_slots - 1 : (int64_t)s;
}

// Sequence bounds with validation against [0, T]; returns false if invalid.
__device__ __forceinline__ bool seq_bounds(const int32_t* cu, int n, int64_t T, int64_t* bos,
                                           int64_t* eos) {
  const int64_t a = cu[n], b = cu[n + 1];
  if (a < 0 || b < a || b > T) return false;
  *bos = a;
  *eos = b;
  return true;
}

}  // namespace kda

// Internal launchers (C++ linkage, defined in the .cu files).
namespace kda {
// In-kernel gate activation.  When `a` is set the log-decay is not read from g but
// computed per (token, v-head, channel) as
//   g = max(-exp(A_log[h]) * softplus(a + dt_bias[h][c]), lb)
// (the gate form of the KDA / GDN tests in the sglang PR 27488 and PR 30169 digests).
struct GateAct {
  const void* a;         // [T, Hv, K], qkv dtype; null: g is given
  const float* A_log;    // [Hv]
  const float* dt_bias;  // [Hv, K] or null
  float lb;              // lower bound of g; -inf: none
};
// softplus(x) = log(1 + e^x), evaluated without overflow
__device__ __forceinline__ float softplus_f32(float x) { return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))); }

struct PrefillArgs {
  kda_desc_t d;
  float scale;
  int64_t slot_stride;
  const void *q, *k, *v;
  const float *g, *beta;
  GateAct act;               // act.a null: g is given
  int gate_k;                // gate values per (token, v-head): K, or 1 (scalar gate)
  bool l2norm;               // normalise q and k rows in the kernel
  bool state_vk;             // states stored [V][K] per head (KDA_FLAG_STATE_VK)
  const int32_t* cu;
  const void* state_in;      // pool, dense h0 or null
  const int32_t* idx;        // null in dense mode
  void* state_out;           // pool (== state_in), dense ht, or null
  void* o;
  uint32_t* status;
  uint8_t* ws;               // workspace base
  size_t ws_bytes;
};
// Bound of the tensor-core prefill's pipeline waits for launches from now on
// (kda_set_pipeline_wait_limit; 2 s by default).
uint64_t pipeline_wait_limit_ns();
cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t st);
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t st);
size_t prefill_tc_workspace(const kda_desc_t& d);      // beyond the header, with splitting
size_t prefill_tc_min_workspace(const kda_desc_t& d);  // beyond the header, no splitting
bool prefill_tc_supported(const kda_desc_t& d);

struct DecodeArgs {
  kda_desc_t d;
  float scale;
  int64_t slot_stride;
  const void *q, *k, *v;
  const float *g, *beta;
  int gate_k;                // K, or 1 (scalar gate)
  bool l2norm;               // normalise q and k rows in the kernel
  bool state_vk;             // states stored [V][K] per head (KDA_FLAG_STATE_VK)
  void* pool;
  const int32_t* idx;
  void* o;
  uint32_t* status;
  // draft steps (kda_decode_draft); plain decode: cu null, cache null, update_pool true
  const int32_t* cu;
  void* cache;
  int64_t cache_pitch;
  int max_steps;
  bool update_pool;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);
}  // namespace kda
