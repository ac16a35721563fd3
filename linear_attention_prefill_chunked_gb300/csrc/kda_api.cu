// kda_api.cu -- the extern "C" boundary: argument validation, workspace sizing,
// dispatch to the tensor-core or CUDA-core prefill, decode, status readback.
#include <atomic>
#include <cmath>

#include "kda_internal.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {
std::atomic<uint64_t> g_wait_limit_ns{tc::kWaitLimitNs};
}  // namespace
uint64_t pipeline_wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
}  // namespace kda

namespace {

using kda::kWsPayload;

bool dims_ok(const kda_desc_t* d) {
  if (!d) return false;
  if (d->num_seqs < 0 || d->total_tokens < 0) return false;
  if (d->num_k_heads <= 0 || d->num_v_heads <= 0) return false;
  if (d->num_v_heads % d->num_k_heads != 0) return false;
  if (d->chunk_size != 64) return false;
  if ((d->flags & ~(KDA_FLAG_CUDA_CORE_PATH | KDA_FLAG_SCALAR_GATE | KDA_FLAG_QK_L2NORM |
                    KDA_FLAG_STATE_VK)) != 0)
    return false;
  if (!(d->qkv_dtype == KDA_BF16 || d->qkv_dtype == KDA_F32)) return false;
  if (!(d->state_dtype == KDA_BF16 || d->state_dtype == KDA_F32)) return false;
  if (!std::isfinite(d->scale)) return false;
  return true;
}

bool heads_supported(const kda_desc_t* d) {
  const int K = d->head_k_dim, V = d->head_v_dim;
  return (K == 64 || K == 128) && (V == 64 || V == 128);
}

int64_t slot_pitch(const kda_desc_t* d) {
  const int64_t dense = (int64_t)d->num_v_heads * d->head_k_dim * d->head_v_dim;
  return d->slot_stride_elems == 0 ? dense : d->slot_stride_elems;
}

bool pitch_ok(const kda_desc_t* d) {
  const int64_t dense = (int64_t)d->num_v_heads * d->head_k_dim * d->head_v_dim;
  const int64_t p = slot_pitch(d);
  return p >= dense && p % 8 == 0;  // 8 elements keeps every row 16-byte aligned
}

float eff_scale(const kda_desc_t* d) {
  return d->scale > 0.f ? d->scale : 1.0f / std::sqrt((float)d->head_k_dim);
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

extern "C" {

const char* kda_status_string(kda_status_t s) {
  switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported configuration";
    case KDA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case KDA_ERR_CUDA: return "CUDA error";
    case KDA_ERR_DEVICE_DATA: return "invalid device data (see status bits)";
  }
  return "unknown status";
}

int kda_chunk_prefill_path(const kda_desc_t* d) {
  if (!dims_ok(d) || !heads_supported(d)) return -1;
  return kda::prefill_tc_supported(*d) ? 1 : 0;
}

size_t kda_chunk_prefill_workspace_size(const kda_desc_t* d) {
  if (!dims_ok(d) || !heads_supported(d)) return 0;
  size_t extra = kda::prefill_tc_supported(*d) ? kda::prefill_tc_workspace(*d) : 0;
  return kWsPayload + round_up(extra, 256);
}

size_t kda_chunk_prefill_min_workspace_size(const kda_desc_t* d) {
  if (!dims_ok(d) || !heads_supported(d)) return 0;
  size_t extra = kda::prefill_tc_supported(*d) ? kda::prefill_tc_min_workspace(*d) : 0;
  return kWsPayload + round_up(extra, 256);
}

size_t kda_decode_workspace_size(const kda_desc_t* d) {
  if (!dims_ok(d) || !heads_supported(d)) return 0;
  return kWsPayload;
}

namespace {
// Shared by kda_chunk_prefill (g given) and kda_chunk_prefill_act (g from a).
kda_status_t prefill_common(const kda_desc_t* d, const void* q, const void* k, const void* v,
                            const float* g, const kda::GateAct& act, const float* beta,
                            const int32_t* cu_seqlens, void* state, const int32_t* state_indices,
                            void* final_state, void* o, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  if (!dims_ok(d)) return KDA_ERR_INVALID_ARGUMENT;
  if (!heads_supported(d)) return KDA_ERR_UNSUPPORTED;
  if (d->num_v_heads > 65535) return KDA_ERR_UNSUPPORTED;  // grid.y limit
  if (!cu_seqlens || !workspace || !aligned(workspace, 256)) return KDA_ERR_INVALID_ARGUMENT;
  const bool has_gate = act.a ? (act.A_log != nullptr) : (g != nullptr);
  if (d->total_tokens > 0 && (!q || !k || !v || !has_gate || !beta || !o))
    return KDA_ERR_INVALID_ARGUMENT;
  const bool pool = state_indices != nullptr;
  if (pool) {
    if (!state || d->num_slots <= 0 || !pitch_ok(d)) return KDA_ERR_INVALID_ARGUMENT;
    if (final_state != nullptr && final_state != state) return KDA_ERR_INVALID_ARGUMENT;
  }
  {
    const void* ptrs[] = {q, k, v, g, act.a, o, state, final_state};
    for (const void* p : ptrs)
      if (p && !aligned(p, 16)) return KDA_ERR_INVALID_ARGUMENT;
  }
  if (workspace_bytes < kda_chunk_prefill_min_workspace_size(d)) return KDA_ERR_WORKSPACE_TOO_SMALL;

  kda::PrefillArgs a;
  a.d = *d;
  a.scale = eff_scale(d);
  a.slot_stride = pool ? slot_pitch(d) : (int64_t)d->num_v_heads * d->head_k_dim * d->head_v_dim;
  a.q = q; a.k = k; a.v = v; a.g = g; a.act = act; a.beta = beta; a.cu = cu_seqlens;
  a.gate_k = (d->flags & KDA_FLAG_SCALAR_GATE) ? 1 : d->head_k_dim;
  a.l2norm = (d->flags & KDA_FLAG_QK_L2NORM) != 0;
  a.state_vk = (d->flags & KDA_FLAG_STATE_VK) != 0;
  a.state_in = state;
  a.idx = state_indices;
  a.state_out = pool ? state : final_state;
  a.o = o;
  a.ws = static_cast<uint8_t*>(workspace);
  a.ws_bytes = workspace_bytes;
  a.status = &reinterpret_cast<kda::WsHeader*>(workspace)->status;

  // An error left by earlier, unrelated work is cleared here, so that the launch checks
  // below report failures of this call's own launches only.
  (void)cudaGetLastError();
  // The header (status word, scheduler counter) starts every call at zero.
  if (cudaMemsetAsync(workspace, 0, sizeof(kda::WsHeader), stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (d->num_seqs == 0) return KDA_OK;
  cudaError_t err = kda::prefill_tc_supported(*d) ? kda::launch_prefill_tc(a, stream)
                                                  : kda::launch_prefill_simt(a, stream);
  return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
}  // namespace

kda_status_t kda_chunk_prefill(const kda_desc_t* d, const void* q, const void* k, const void* v,
                               const float* g, const float* beta, const int32_t* cu_seqlens,
                               void* state, const int32_t* state_indices, void* final_state,
                               void* o, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
  const kda::GateAct none{nullptr, nullptr, nullptr, -INFINITY};
  return prefill_common(d, q, k, v, g, none, beta, cu_seqlens, state, state_indices, final_state,
                        o, workspace, workspace_bytes, stream);
}

kda_status_t kda_chunk_prefill_act(const kda_desc_t* d, const void* q, const void* k,
                                   const void* v, const void* a, const float* A_log,
                                   const float* dt_bias, float lower_bound, const float* beta,
                                   const int32_t* cu_seqlens, void* state,
                                   const int32_t* state_indices, void* final_state, void* o,
                                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (d && d->total_tokens > 0 && (!a || !A_log)) return KDA_ERR_INVALID_ARGUMENT;
  if (lower_bound != lower_bound || lower_bound > 0.f) return KDA_ERR_INVALID_ARGUMENT;  // NaN or > 0
  const kda::GateAct act{a, A_log, dt_bias, lower_bound};
  return prefill_common(d, q, k, v, nullptr, act, beta, cu_seqlens, state, state_indices,
                        final_state, o, workspace, workspace_bytes, stream);
}

kda_status_t kda_decode(const kda_desc_t* d, const void* q, const void* k, const void* v,
                        const float* g, const float* beta, void* state_pool,
                        const int32_t* state_indices, void* o, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  if (!dims_ok(d)) return KDA_ERR_INVALID_ARGUMENT;
  if (!heads_supported(d)) return KDA_ERR_UNSUPPORTED;
  if (d->total_tokens != d->num_seqs) return KDA_ERR_INVALID_ARGUMENT;
  if (d->num_v_heads > 65535) return KDA_ERR_UNSUPPORTED;  // grid.y limit
  if (!workspace || !aligned(workspace, 256)) return KDA_ERR_INVALID_ARGUMENT;
  if (d->num_seqs > 0 && (!q || !k || !v || !g || !beta || !o || !state_pool))
    return KDA_ERR_INVALID_ARGUMENT;
  if (d->num_slots <= 0 || !pitch_ok(d)) return KDA_ERR_INVALID_ARGUMENT;
  {
    const void* ptrs[] = {q, k, v, g, o, state_pool};
    for (const void* p : ptrs)
      if (p && !aligned(p, 16)) return KDA_ERR_INVALID_ARGUMENT;
  }
  if (workspace_bytes < kda_decode_workspace_size(d)) return KDA_ERR_WORKSPACE_TOO_SMALL;

  kda::DecodeArgs a;
  a.d = *d;
  a.scale = eff_scale(d);
  a.slot_stride = slot_pitch(d);
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.gate_k = (d->flags & KDA_FLAG_SCALAR_GATE) ? 1 : d->head_k_dim;
  a.l2norm = (d->flags & KDA_FLAG_QK_L2NORM) != 0;
  a.state_vk = (d->flags & KDA_FLAG_STATE_VK) != 0;
  a.pool = state_pool;
  a.idx = state_indices;
  a.o = o;
  a.status = &reinterpret_cast<kda::WsHeader*>(workspace)->status;
  a.cu = nullptr;
  a.cache = nullptr;
  a.cache_pitch = 0;
  a.max_steps = 1;
  a.update_pool = true;
  (void)cudaGetLastError();  // report this call's own launch errors only
  if (cudaMemsetAsync(workspace, 0, sizeof(kda::WsHeader), stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  return kda::launch_decode(a, stream) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_decode_draft(const kda_desc_t* d, const void* q, const void* k, const void* v,
                              const float* g, const float* beta, const int32_t* cu_seqlens,
                              void* state_pool, const int32_t* state_indices, void* step_cache,
                              int64_t cache_pitch_elems, int32_t max_steps, int update_pool,
                              void* o, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
  if (!dims_ok(d)) return KDA_ERR_INVALID_ARGUMENT;
  if (!heads_supported(d)) return KDA_ERR_UNSUPPORTED;
  if (d->num_v_heads > 65535) return KDA_ERR_UNSUPPORTED;  // grid.y limit
  if (!workspace || !aligned(workspace, 256) || !cu_seqlens) return KDA_ERR_INVALID_ARGUMENT;
  if (d->total_tokens > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARGUMENT;
  if (d->num_seqs > 0 && !state_pool) return KDA_ERR_INVALID_ARGUMENT;
  if (d->num_slots <= 0 || !pitch_ok(d) || max_steps < 1) return KDA_ERR_INVALID_ARGUMENT;
  const int64_t hkv = (int64_t)d->num_v_heads * d->head_k_dim * d->head_v_dim;
  if (step_cache && (cache_pitch_elems < (int64_t)max_steps * hkv || cache_pitch_elems % 8 != 0))
    return KDA_ERR_INVALID_ARGUMENT;
  {
    const void* ptrs[] = {q, k, v, g, o, state_pool, step_cache};
    for (const void* p : ptrs)
      if (p && !aligned(p, 16)) return KDA_ERR_INVALID_ARGUMENT;
  }
  if (workspace_bytes < kda_decode_workspace_size(d)) return KDA_ERR_WORKSPACE_TOO_SMALL;

  kda::DecodeArgs a;
  a.d = *d;
  a.scale = eff_scale(d);
  a.slot_stride = slot_pitch(d);
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.gate_k = (d->flags & KDA_FLAG_SCALAR_GATE) ? 1 : d->head_k_dim;
  a.l2norm = (d->flags & KDA_FLAG_QK_L2NORM) != 0;
  a.state_vk = (d->flags & KDA_FLAG_STATE_VK) != 0;
  a.pool = state_pool;
  a.idx = state_indices;
  a.o = o;
  a.status = &reinterpret_cast<kda::WsHeader*>(workspace)->status;
  a.cu = cu_seqlens;
  a.cache = step_cache;
  a.cache_pitch = cache_pitch_elems;
  a.max_steps = max_steps;
  a.update_pool = update_pool != 0;
  (void)cudaGetLastError();  // report this call's own launch errors only
  if (cudaMemsetAsync(workspace, 0, sizeof(kda::WsHeader), stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  return kda::launch_decode(a, stream) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_set_pipeline_wait_limit(uint64_t nanoseconds) {
  if (nanoseconds > kda::tc::kWaitLimitNs) return KDA_ERR_INVALID_ARGUMENT;
  kda::g_wait_limit_ns.store(nanoseconds == 0 ? kda::tc::kWaitLimitNs : nanoseconds,
                             std::memory_order_relaxed);
  return KDA_OK;
}

kda_status_t kda_read_device_status(const void* workspace, uint32_t* bits_out,
                                    cudaStream_t stream) {
  if (!workspace) return KDA_ERR_INVALID_ARGUMENT;
  uint32_t bits = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KDA_ERR_CUDA;
  if (cudaMemcpy(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (bits_out) *bits_out = bits;
  return bits ? KDA_ERR_DEVICE_DATA : KDA_OK;
}

}  // extern "C"
