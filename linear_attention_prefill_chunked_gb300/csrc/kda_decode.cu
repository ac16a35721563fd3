// kda_decode.cu -- one-token-per-row KDA decode on a state pool, in place.
//
// Per row n and v-head h (slot s = idx[n], -1 -> sentinel num_slots-1):
//   S <- Diag(exp g) S;  u = beta (v - S^T k);  S <- S + k u^T;  o = scale S^T q
// which is one step of the recurrence the prefill evaluates in chunks.
//
// Grid (N, Hv, V / VT): rows on grid.x (limit 2^31-1), heads on grid.y, value
// tiles on grid.z -- rows and heads are never folded into one axis, the rule of
// the sglang PR 37317 digest "FLA/MoE grid split" (实现拆解 item 1, 风险与影响
// item 5), which fixed launches failing once N*Hv exceeded 65535.
//
// The kernel is bound by HBM: it streams each state tile (K x VT fp32) in and
// out exactly once.  A CTA of 256 threads holds the tile in registers: 32 (or
// VT/4) threads cover one row with 16-byte vector accesses, the 8 row groups
// split the K rows, and the two channel reductions (S^T k and S^T q) go through
// shared memory.
#include "kda_internal.cuh"

namespace kda {
namespace {

KDA_DEBUG_FLAG_DEFINE();

constexpr int kDecThreads = 256;

template <typename ST> struct Vec4;
template <> struct Vec4<float> {
  __device__ static void load(const float* p, float r[4]) {
    const float4 x = *reinterpret_cast<const float4*>(p);
    r[0] = x.x; r[1] = x.y; r[2] = x.z; r[3] = x.w;
  }
  __device__ static void store(float* p, const float r[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(r[0], r[1], r[2], r[3]);
  }
};
template <> struct Vec4<__nv_bfloat16> {
  __device__ static void load(const __nv_bfloat16* p, float r[4]) {
    const uint2 x = *reinterpret_cast<const uint2*>(p);
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&x.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&x.y);
    r[0] = __low2float(a); r[1] = __high2float(a); r[2] = __low2float(b); r[3] = __high2float(b);
  }
  __device__ static void store(__nv_bfloat16* p, const float r[4]) {
    __nv_bfloat162 a = __floats2bfloat162_rn(r[0], r[1]);
    __nv_bfloat162 b = __floats2bfloat162_rn(r[2], r[3]);
    uint2 x;
    x.x = *reinterpret_cast<uint32_t*>(&a);
    x.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = x;
  }
};

// Draft steps (speculative decoding): with `cu` set, row n is a request whose tokens
// cu[n] .. cu[n+1]-1 run one after another from the same state; the state after step j
// is written to cache + n * cache_pitch + j * Hv*K*V (per-request pitch passed in, not
// inferred from a buffer shape: PR 37317 digest, 实现拆解 item 2), and the pool row is
// written only if update_pool.  Without `cu` each row is one token and the pool is updated.
struct DraftArgs {
  const int32_t* cu;   // [N+1] or null
  void* cache;         // null: no per-step states
  int64_t cache_pitch;
  int max_steps;
  bool update_pool;
};

template <typename QT, typename ST, int K, int VT>
__global__ void __launch_bounds__(kDecThreads, 2)
kda_decode_kernel(const QT* __restrict__ q, const QT* __restrict__ k, const QT* __restrict__ v,
                  const float* __restrict__ g, const float* __restrict__ beta,
                  ST* __restrict__ pool, const int32_t* __restrict__ idx, QT* __restrict__ o,
                  uint32_t* __restrict__ status, int Hk, int Hv, int V, int64_t num_slots,
                  int64_t slot_stride, float scale, int gk, bool l2norm, DraftArgs dr, int64_t T) {
  constexpr int TPR = VT / 4;               // threads per row
  constexpr int RG = kDecThreads / TPR;     // row groups
  constexpr int RPT = K / RG;               // rows per thread
  static_assert(K % RG == 0, "K must split over the row groups");

  const int n = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * VT;
  const int tid = threadIdx.x, rg = tid / TPR, col = (tid % TPR) * 4;

  int64_t bos = n, eos = n + 1;
  if (dr.cu != nullptr) {
    if (!seq_bounds(dr.cu, n, T, &bos, &eos) || eos - bos > dr.max_steps) {
      if (tid == 0 && blockIdx.z == 0 && h == 0) raise_status(status, KDA_DEVICE_BAD_SEQLENS);
      return;
    }
  }
  int64_t slot = n;
  if (idx != nullptr) {
    slot = resolve_slot(idx, n, num_slots);
    if (slot < 0) {
      if (tid == 0 && blockIdx.z == 0) raise_status(status, KDA_DEVICE_BAD_SLOT);
      return;
    }
  } else if (slot >= num_slots) {
    if (tid == 0 && blockIdx.z == 0) raise_status(status, KDA_DEVICE_BAD_SLOT);
    return;
  }

  __shared__ float red_w[RG][VT];
  __shared__ float red_o[RG][VT];
  __shared__ float red_n[2][kDecThreads / 32];
  __shared__ float kq_s[3][K];  // k, q and exp(g) of the current token, shared by the block

  const int kh = h / (Hv / Hk);
  ST* S = pool + slot * slot_stride + (size_t)h * K * V + v0 + col;
  float s[RPT][4];
  // Issue every state load first (the tile is the whole cost of the kernel).
#pragma unroll
  for (int j = 0; j < RPT; ++j) Vec4<ST>::load(S + (size_t)(rg + j * RG) * V, s[j]);

  for (int64_t t = bos; t < eos; ++t) {
    if (t > bos) __syncthreads();
    if (!KDA_CHECK(t >= 0 && t < T && t - bos < dr.max_steps)) break;  // uniform  // the previous step's readers of the shared arrays are done
    // k, q, exp(g) of token t into shared memory (registers stay with the state tile);
    // with l2norm the two norms are reduced over the block first
    float kv = 0.f, qv = 0.f;
    if (tid < K) {
      kv = to_f32(k[((size_t)t * Hk + kh) * K + tid]);
      qv = to_f32(q[((size_t)t * Hk + kh) * K + tid]);
      kq_s[2][tid] = expf(g[((size_t)t * Hv + h) * gk + (gk > 1 ? tid : 0)]);
    }
    float ik = 1.f, iq = 1.f;
    if (l2norm) {
      float sk = kv * kv, sq = qv * qv;
#pragma unroll
      for (int o2 = 16; o2; o2 >>= 1) {
        sk += __shfl_xor_sync(0xffffffffu, sk, o2);
        sq += __shfl_xor_sync(0xffffffffu, sq, o2);
      }
      if ((tid & 31) == 0) {
        red_n[0][tid >> 5] = sk;
        red_n[1][tid >> 5] = sq;
      }
      __syncthreads();
      float tk = 0.f, tq = 0.f;
#pragma unroll
      for (int r = 0; r < K / 32; ++r) {
        tk += red_n[0][r];
        tq += red_n[1][r];
      }
      ik = 1.f / fmaxf(sqrtf(tk), 1e-12f);
      iq = 1.f / fmaxf(sqrtf(tq), 1e-12f);
    }
    if (tid < K) {
      kq_s[0][tid] = kv * ik;
      kq_s[1][tid] = qv * iq;
    }
    __syncthreads();
    float w[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const int c = rg + j * RG;
      const float e = kq_s[2][c], kr = kq_s[0][c];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        s[j][i] *= e;                    // decay first
        w[i] = fmaf(kr, s[j][i], w[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) red_w[rg][col + i] = w[i];
    __syncthreads();
    const float b = beta[(size_t)t * Hv + h];
    float u[4];
    {
      float vin[4];
      const QT* vn = v + ((size_t)t * Hv + h) * V + v0 + col;
#pragma unroll
      for (int i = 0; i < 4; ++i) vin[i] = to_f32(vn[i]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int r = 0; r < RG; ++r) acc += red_w[r][col + i];
        u[i] = b * (vin[i] - acc);
      }
    }
    ST* C = dr.cache ? static_cast<ST*>(dr.cache) + n * dr.cache_pitch +
                           (t - bos) * ((int64_t)Hv * K * V) + (size_t)h * K * V + v0 + col
                     : nullptr;
    float ov[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const int c = rg + j * RG;
      const float kr = kq_s[0][c], qr = kq_s[1][c];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        s[j][i] = fmaf(kr, u[i], s[j][i]);
        ov[i] = fmaf(qr, s[j][i], ov[i]);
      }
      if (C) Vec4<ST>::store(C + (size_t)(rg + j * RG) * V, s[j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) red_o[rg][col + i] = ov[i];
    __syncthreads();
    if (rg == 0) {
      QT* on = o + ((size_t)t * Hv + h) * V + v0 + col;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int r = 0; r < RG; ++r) acc += red_o[r][col + i];
        on[i] = from_f32<QT>(scale * acc);
      }
    }
  }
  if (tid == 0) KDA_DEBUG_FOLD(status);
  if (dr.update_pool) {
#pragma unroll
    for (int j = 0; j < RPT; ++j) Vec4<ST>::store(S + (size_t)(rg + j * RG) * V, s[j]);
  }
}

// The same step on states stored transposed (KDA_FLAG_STATE_VK: row v of a head's state
// holds S[:, v], K contiguous values -- the layout of the pages' GDN pool test).  A CTA holds
// VT state rows (value channels v0 ..) with all K key channels: TPR = K/4 threads cover one
// row with 16-byte accesses, so both reductions over the key channels (S^T k, S^T q) are
// shuffles within the row's threads, and u needs no exchange at all.
template <typename QT, typename ST, int K, int VT>
__global__ void __launch_bounds__(kDecThreads, 2)
kda_decode_vk_kernel(const QT* __restrict__ q, const QT* __restrict__ k, const QT* __restrict__ v,
                     const float* __restrict__ g, const float* __restrict__ beta,
                     ST* __restrict__ pool, const int32_t* __restrict__ idx, QT* __restrict__ o,
                     uint32_t* __restrict__ status, int Hk, int Hv, int V, int64_t num_slots,
                     int64_t slot_stride, float scale, int gk, bool l2norm, DraftArgs dr, int64_t T) {
  constexpr int TPR = K / 4;                // threads per row (16 or 32: within one warp)
  constexpr int RG = kDecThreads / TPR;     // row groups
  constexpr int RPT = VT / RG;              // rows per thread
  static_assert(VT % RG == 0, "VT must split over the row groups");

  const int n = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * VT;
  const int tid = threadIdx.x, rg = tid / TPR, col = (tid % TPR) * 4;

  int64_t bos = n, eos = n + 1;
  if (dr.cu != nullptr) {
    if (!seq_bounds(dr.cu, n, T, &bos, &eos) || eos - bos > dr.max_steps) {
      if (tid == 0 && blockIdx.z == 0 && h == 0) raise_status(status, KDA_DEVICE_BAD_SEQLENS);
      return;
    }
  }
  int64_t slot = n;
  if (idx != nullptr) {
    slot = resolve_slot(idx, n, num_slots);
    if (slot < 0) {
      if (tid == 0 && blockIdx.z == 0) raise_status(status, KDA_DEVICE_BAD_SLOT);
      return;
    }
  } else if (slot >= num_slots) {
    if (tid == 0 && blockIdx.z == 0) raise_status(status, KDA_DEVICE_BAD_SLOT);
    return;
  }

  __shared__ float red_n[2][kDecThreads / 32];
  __shared__ float kq_s[3][K];

  const int kh = h / (Hv / Hk);
  ST* S = pool + slot * slot_stride + (size_t)h * K * V + (size_t)v0 * K + col;
  float s[RPT][4];
#pragma unroll
  for (int j = 0; j < RPT; ++j) Vec4<ST>::load(S + (size_t)(rg + j * RG) * K, s[j]);

  for (int64_t t = bos; t < eos; ++t) {
    if (t > bos) __syncthreads();
    if (!KDA_CHECK(t >= 0 && t < T && t - bos < dr.max_steps)) break;  // uniform
    float kv = 0.f, qv = 0.f;
    if (tid < K) {
      kv = to_f32(k[((size_t)t * Hk + kh) * K + tid]);
      qv = to_f32(q[((size_t)t * Hk + kh) * K + tid]);
      kq_s[2][tid] = expf(g[((size_t)t * Hv + h) * gk + (gk > 1 ? tid : 0)]);
    }
    float ik = 1.f, iq = 1.f;
    if (l2norm) {
      float sk = kv * kv, sq = qv * qv;
#pragma unroll
      for (int o2 = 16; o2; o2 >>= 1) {
        sk += __shfl_xor_sync(0xffffffffu, sk, o2);
        sq += __shfl_xor_sync(0xffffffffu, sq, o2);
      }
      if ((tid & 31) == 0) {
        red_n[0][tid >> 5] = sk;
        red_n[1][tid >> 5] = sq;
      }
      __syncthreads();
      float tk = 0.f, tq = 0.f;
#pragma unroll
      for (int r = 0; r < K / 32; ++r) {
        tk += red_n[0][r];
        tq += red_n[1][r];
      }
      ik = 1.f / fmaxf(sqrtf(tk), 1e-12f);
      iq = 1.f / fmaxf(sqrtf(tq), 1e-12f);
    }
    if (tid < K) {
      kq_s[0][tid] = kv * ik;
      kq_s[1][tid] = qv * iq;
    }
    __syncthreads();
    float kr[4], qr[4], er[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      kr[i] = kq_s[0][col + i];
      qr[i] = kq_s[1][col + i];
      er[i] = kq_s[2][col + i];
    }
    const float b = beta[(size_t)t * Hv + h];
    const QT* vn = v + ((size_t)t * Hv + h) * V + v0;
    ST* C = dr.cache ? static_cast<ST*>(dr.cache) + n * dr.cache_pitch +
                           (t - bos) * ((int64_t)Hv * K * V) + (size_t)h * K * V + (size_t)v0 * K + col
                     : nullptr;
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const int row = rg + j * RG;
      float w = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        s[j][i] *= er[i];  // decay first
        w = fmaf(kr[i], s[j][i], w);
      }
#pragma unroll
      for (int o2 = TPR / 2; o2; o2 >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o2);
      const float u = b * (to_f32(vn[row]) - w);
      float ov = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        s[j][i] = fmaf(kr[i], u, s[j][i]);
        ov = fmaf(qr[i], s[j][i], ov);
      }
#pragma unroll
      for (int o2 = TPR / 2; o2; o2 >>= 1) ov += __shfl_xor_sync(0xffffffffu, ov, o2);
      if (col == 0) o[((size_t)t * Hv + h) * V + v0 + row] = from_f32<QT>(scale * ov);
      if (C) Vec4<ST>::store(C + (size_t)row * K, s[j]);
    }
  }
  if (tid == 0) KDA_DEBUG_FOLD(status);
  if (dr.update_pool) {
#pragma unroll
    for (int j = 0; j < RPT; ++j) Vec4<ST>::store(S + (size_t)(rg + j * RG) * K, s[j]);
  }
}

template <typename QT, typename ST, int K>
cudaError_t launch_typed(const DecodeArgs& a, cudaStream_t st) {
  const int V = a.d.head_v_dim;
  const int VT = V >= 128 ? 128 : 64;
  dim3 grid((unsigned)a.d.num_seqs, (unsigned)a.d.num_v_heads, (unsigned)(V / VT));
  const DraftArgs dr{a.cu, a.cache, a.cache_pitch, a.max_steps, a.update_pool};
  if (a.state_vk) {
    if (VT == 128)
      kda_decode_vk_kernel<QT, ST, K, 128><<<grid, kDecThreads, 0, st>>>(
          (const QT*)a.q, (const QT*)a.k, (const QT*)a.v, a.g, a.beta, (ST*)a.pool, a.idx,
          (QT*)a.o, a.status, a.d.num_k_heads, a.d.num_v_heads, V, a.d.num_slots, a.slot_stride,
          a.scale, a.gate_k, a.l2norm, dr, a.d.total_tokens);
    else
      kda_decode_vk_kernel<QT, ST, K, 64><<<grid, kDecThreads, 0, st>>>(
          (const QT*)a.q, (const QT*)a.k, (const QT*)a.v, a.g, a.beta, (ST*)a.pool, a.idx,
          (QT*)a.o, a.status, a.d.num_k_heads, a.d.num_v_heads, V, a.d.num_slots, a.slot_stride,
          a.scale, a.gate_k, a.l2norm, dr, a.d.total_tokens);
    return cudaGetLastError();
  }
  if (VT == 128)
    kda_decode_kernel<QT, ST, K, 128><<<grid, kDecThreads, 0, st>>>(
        (const QT*)a.q, (const QT*)a.k, (const QT*)a.v, a.g, a.beta, (ST*)a.pool, a.idx,
        (QT*)a.o, a.status, a.d.num_k_heads, a.d.num_v_heads, V, a.d.num_slots, a.slot_stride,
        a.scale, a.gate_k, a.l2norm, DraftArgs{a.cu, a.cache, a.cache_pitch, a.max_steps,
                                                 a.update_pool}, a.d.total_tokens);
  else
    kda_decode_kernel<QT, ST, K, 64><<<grid, kDecThreads, 0, st>>>(
        (const QT*)a.q, (const QT*)a.k, (const QT*)a.v, a.g, a.beta, (ST*)a.pool, a.idx,
        (QT*)a.o, a.status, a.d.num_k_heads, a.d.num_v_heads, V, a.d.num_slots, a.slot_stride,
        a.scale, a.gate_k, a.l2norm, DraftArgs{a.cu, a.cache, a.cache_pitch, a.max_steps,
                                                 a.update_pool}, a.d.total_tokens);
  return cudaGetLastError();
}

template <typename QT, typename ST>
cudaError_t launch_k(const DecodeArgs& a, cudaStream_t st) {
  return a.d.head_k_dim == 128 ? launch_typed<QT, ST, 128>(a, st) : launch_typed<QT, ST, 64>(a, st);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  if (a.d.num_seqs == 0) return cudaSuccess;
  const bool qb = a.d.qkv_dtype == KDA_BF16, sb = a.d.state_dtype == KDA_BF16;
  if (qb && sb) return launch_k<__nv_bfloat16, __nv_bfloat16>(a, st);
  if (qb) return launch_k<__nv_bfloat16, float>(a, st);
  if (sb) return launch_k<float, __nv_bfloat16>(a, st);
  return launch_k<float, float>(a, st);
}

}  // namespace kda
