// kda_prefill_simt.cu -- chunked KDA prefill on CUDA cores in fp32.
//
// This is the path for fp32 inputs (and for head dims the tensor-core kernel
// does not cover).  It evaluates the same chunked form as the tensor-core path,
// the pipeline of the sglang PR 27488 digest "KDA SM100 CuteDSL prefill"
// (关键文件: gate prologue, KKT inverse + U/W, h kernel, output kernel), in
// fp32 throughout.  One CTA owns one (sequence, v-head) and walks its chunks:
//
//   Gamma  = inclusive per-channel cumsum of g inside the chunk
//   A[r,i] = beta_r sum_c k_r k_i exp(Gamma_r - Gamma_i)   (i < r)
//   B[r,i] = scale  sum_c q_r k_i exp(Gamma_r - Gamma_i)   (i <= r)
//   Tm     = (I + A)^-1 Diag(beta)
//   KG = k exp(Gamma), QG = scale q exp(Gamma), KR = k exp(Gamma_last - Gamma)
//   U  = Tm (V - KG S);  O = QG S + B U;  S <- Diag(exp Gamma_last) S + KR^T U
//
// Every exponent above is <= 0 for g <= 0, so nothing overflows however large
// the per-chunk decay (the fp32 exp overflow the pages report for realistic
// gates, PR 27488 digest 功能与动机, cannot occur); the pairwise exponentials
// cost more SFU work than the tensor-core path's factorised form, which does
// not matter here.
#include "kda_internal.cuh"

namespace kda {
namespace {

KDA_DEBUG_FLAG_DEFINE();

constexpr int kC = 64;          // chunk size
constexpr int kSimtThreads = 256;

template <int K, int V>
struct SimtSmem {
  static constexpr int KP = K + 1;                      // padded pitches (bank spread)
  static constexpr int DP = (K > V ? K : V) + 1;
  static constexpr int VP = V + 1;
  static constexpr size_t kb = 0;                                   // [64][DP]  k -> KG -> U
  static constexpr size_t qb = kb + (size_t)kC * DP;                // [64][KP]  q -> QG
  static constexpr size_t gb = qb + (size_t)kC * KP;                // [64][KP]  g -> Gamma -> KR
  static constexpr size_t vb = gb + (size_t)kC * KP;                // [64][VP]  v -> V - KG S
  static constexpr size_t am = vb + (size_t)kC * VP;                // [64][65]  A -> Tm
  static constexpr size_t bm = am + (size_t)kC * (kC + 1);          // [64][65]  B
  static constexpr size_t sm = bm + (size_t)kC * (kC + 1);          // [K][V]    state
  static constexpr size_t gl = sm + (size_t)K * V;                  // [K]       Gamma_last
  static constexpr size_t be = gl + K;                              // [64]      beta
  static constexpr size_t rb = be + kC;                             // [64]      row buffer
  static constexpr size_t total_floats = rb + kC;
  static constexpr size_t bytes = total_floats * sizeof(float);
};

template <typename QT, typename ST, int K, int V>
__global__ void __launch_bounds__(kSimtThreads)
kda_prefill_simt_kernel(const QT* __restrict__ q, const QT* __restrict__ k,
                        const QT* __restrict__ v, const float* __restrict__ g,
                        const float* __restrict__ beta, const int32_t* __restrict__ cu,
                        const ST* state_in, const int32_t* __restrict__ idx, ST* state_out,
                        QT* __restrict__ o, uint32_t* __restrict__ status, int Hk, int Hv,
                        int64_t T, int64_t num_slots, int64_t slot_stride, float scale,
                        GateAct act, int gk, bool l2norm, bool state_vk) {
  using L = SimtSmem<K, V>;
  extern __shared__ float smem[];
  float* Kb = smem + L::kb;
  float* Qb = smem + L::qb;
  float* Gb = smem + L::gb;
  float* Vb = smem + L::vb;
  float* Am = smem + L::am;
  float* Bm = smem + L::bm;
  float* S = smem + L::sm;
  float* Gl = smem + L::gl;
  float* Be = smem + L::be;
  float* Rb = smem + L::rb;
  constexpr int DP = L::DP, KP = L::KP, VP = L::VP, AP = kC + 1;

  const int n = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  int64_t bos, eos;
  if (!seq_bounds(cu, n, T, &bos, &eos)) {
    if (tid == 0 && h == 0) raise_status(status, KDA_DEVICE_BAD_SEQLENS);
    return;
  }
  const ST* src = nullptr;
  ST* dst = nullptr;
  if (idx != nullptr) {
    const int64_t slot = resolve_slot(idx, n, num_slots);
    if (slot < 0) {
      if (tid == 0 && h == 0) raise_status(status, KDA_DEVICE_BAD_SLOT);
      return;
    }
    src = state_in + slot * slot_stride + (size_t)h * K * V;
    dst = state_out + slot * slot_stride + (size_t)h * K * V;
  } else {
    if (state_in) src = state_in + ((size_t)n * Hv + h) * K * V;
    if (state_out) dst = state_out + ((size_t)n * Hv + h) * K * V;
  }
  // S is [K][V] in shared memory; a transposed state buffer ([V][K]) is read across
  for (int e = tid; e < K * V; e += kSimtThreads)
    S[e] = src ? to_f32(src[state_vk ? (e % V) * K + e / V : e]) : 0.f;

  const int kh = h / (Hv / Hk);
  const QT* ga = static_cast<const QT*>(act.a);
  const float Ah = ga ? expf(act.A_log[h]) : 0.f;
  for (int64_t t0 = bos; t0 < eos; t0 += kC) {
    const int c = (int)((eos - t0) < kC ? (eos - t0) : kC);
    __syncthreads();  // previous chunk's readers of every buffer are done
    // ---- load the chunk (rows past the sequence end: k = q = v = g = beta = 0)
    for (int e = tid; e < kC * K; e += kSimtThreads) {
      const int r = e / K, ch = e % K;
      const bool ok = r < c;
      const size_t qk = ((size_t)(t0 + r) * Hk + kh) * K + ch;
      Kb[r * DP + ch] = ok ? to_f32(k[qk]) : 0.f;
      Qb[r * KP + ch] = ok ? to_f32(q[qk]) : 0.f;
      float gv = 0.f;
      if (ok) {
        const int gc = gk > 1 ? ch : 0;  // scalar gate: one value per (token, head)
        const size_t gi = ((size_t)(t0 + r) * Hv + h) * gk + gc;
        if (ga) {
          const float x = to_f32(ga[gi]) + (act.dt_bias ? act.dt_bias[(size_t)h * gk + gc] : 0.f);
          gv = fmaxf(-Ah * softplus_f32(x), act.lb);
        } else {
          gv = g[gi];
        }
      }
      Gb[r * KP + ch] = gv;
    }
    for (int e = tid; e < kC * V; e += kSimtThreads) {
      const int r = e / V, j = e % V;
      Vb[r * VP + j] = r < c ? to_f32(v[((size_t)(t0 + r) * Hv + h) * V + j]) : 0.f;
    }
    if (tid < kC) Be[tid] = tid < c ? beta[(size_t)(t0 + tid) * Hv + h] : 0.f;
    __syncthreads();
    if (l2norm) {  // q and k rows -> x / max(||x||, 1e-12), one warp per row
      const int wp = tid >> 5, ln = tid & 31;
      for (int r = wp; r < 2 * kC; r += kSimtThreads / 32) {
        float* row = r < kC ? Kb + r * DP : Qb + (r - kC) * KP;
        float ss = 0.f;
        for (int ch = ln; ch < K; ch += 32) ss = fmaf(row[ch], row[ch], ss);
#pragma unroll
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = 1.f / fmaxf(sqrtf(ss), 1e-12f);
        for (int ch = ln; ch < K; ch += 32) row[ch] *= inv;
      }
      __syncthreads();
    }
    // ---- Gamma: inclusive cumsum per channel
    for (int ch = tid; ch < K; ch += kSimtThreads) {
      float acc = 0.f;
      for (int r = 0; r < kC; ++r) {
        acc += Gb[r * KP + ch];
        Gb[r * KP + ch] = acc;
      }
      Gl[ch] = acc;
    }
    __syncthreads();
    // ---- A (strictly lower, beta-row-scaled) and B (lower, scaled)
    for (int e = tid; e < kC * kC; e += kSimtThreads) {
      const int r = e / kC, i = e % kC;
      float a = 0.f, b = 0.f;
      if (i <= r) {
        for (int ch = 0; ch < K; ++ch) {
          const float f = expf(Gb[r * KP + ch] - Gb[i * KP + ch]) * Kb[i * DP + ch];
          a = fmaf(Kb[r * DP + ch], f, a);
          b = fmaf(Qb[r * KP + ch], f, b);
        }
      }
      Am[r * AP + i] = i < r ? Be[r] * a : 0.f;
      Bm[r * AP + i] = i <= r ? scale * b : 0.f;
    }
    __syncthreads();
    // ---- (I + A)^-1 in place, row by row: X_r = e_r - sum_{i<r} A[r,i] X_i
    for (int r = 1; r < kC; ++r) {
      if (tid < kC) Rb[tid] = Am[r * AP + tid];
      __syncthreads();
      if (tid < r) {  // column tid of row r (columns >= r are 0 / identity)
        float x = -Rb[tid];
        for (int i = tid + 1; i < r; ++i) x = fmaf(-Rb[i], Am[i * AP + tid], x);
        Am[r * AP + tid] = x;
      }
      __syncthreads();
    }
    // Tm = X Diag(beta) (X has a unit diagonal), and the pre-scaled operands.
    for (int e = tid; e < kC * kC; e += kSimtThreads) {
      const int r = e / kC, i = e % kC;
      const float x = i < r ? Am[r * AP + i] : (i == r ? 1.f : 0.f);
      Am[r * AP + i] = x * Be[i];
    }
    for (int e = tid; e < kC * K; e += kSimtThreads) {
      const int r = e / K, ch = e % K;
      const float G = Gb[r * KP + ch];
      const float kk = Kb[r * DP + ch];
      Kb[r * DP + ch] = kk * expf(G);                      // KG
      Gb[r * KP + ch] = kk * expf(Gl[ch] - G);             // KR
      Qb[r * KP + ch] = scale * Qb[r * KP + ch] * expf(G); // QG
    }
    __syncthreads();
    // ---- Y = V - KG S (in place in Vb)
    for (int e = tid; e < kC * V; e += kSimtThreads) {
      const int r = e / V, j = e % V;
      float acc = Vb[r * VP + j];
      for (int ch = 0; ch < K; ++ch) acc = fmaf(-Kb[r * DP + ch], S[ch * V + j], acc);
      Vb[r * VP + j] = acc;
    }
    __syncthreads();
    // ---- U = Tm Y  (into Kb; KG is dead)
    for (int e = tid; e < kC * V; e += kSimtThreads) {
      const int r = e / V, j = e % V;
      float acc = 0.f;
      for (int i = 0; i <= r; ++i) acc = fmaf(Am[r * AP + i], Vb[i * VP + j], acc);
      Kb[r * DP + j] = acc;
    }
    __syncthreads();
    // ---- O = QG S + B U
    for (int e = tid; e < c * V; e += kSimtThreads) {
      const int r = e / V, j = e % V;
      float acc = 0.f;
      for (int ch = 0; ch < K; ++ch) acc = fmaf(Qb[r * KP + ch], S[ch * V + j], acc);
      for (int i = 0; i <= r; ++i) acc = fmaf(Bm[r * AP + i], Kb[i * DP + j], acc);
      if (KDA_CHECK(t0 + r < T)) o[((size_t)(t0 + r) * Hv + h) * V + j] = from_f32<QT>(acc);
    }
    __syncthreads();
    // ---- S <- Diag(exp Gamma_last) S + KR^T U
    for (int e = tid; e < K * V; e += kSimtThreads) {
      const int ch = e / V, j = e % V;
      float acc = expf(Gl[ch]) * S[e];
      for (int r = 0; r < c; ++r) acc = fmaf(Gb[r * KP + ch], Kb[r * DP + j], acc);
      S[e] = acc;
    }
  }
  __syncthreads();
  if (dst)
    for (int e = tid; e < K * V; e += kSimtThreads)
      dst[state_vk ? (e % V) * K + e / V : e] = from_f32<ST>(S[e]);
  if (tid == 0) KDA_DEBUG_FOLD(status);
}

template <typename QT, typename ST, int K, int V>
cudaError_t launch_typed(const PrefillArgs& a, cudaStream_t st) {
  using L = SimtSmem<K, V>;
  auto kern = kda_prefill_simt_kernel<QT, ST, K, V>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::bytes);
  if (err != cudaSuccess) return err;
  dim3 grid((unsigned)a.d.num_seqs, (unsigned)a.d.num_v_heads);
  kern<<<grid, kSimtThreads, L::bytes, st>>>(
      (const QT*)a.q, (const QT*)a.k, (const QT*)a.v, a.g, a.beta, a.cu,
      (const ST*)a.state_in, a.idx, (ST*)a.state_out, (QT*)a.o, a.status, a.d.num_k_heads,
      a.d.num_v_heads, a.d.total_tokens, a.d.num_slots, a.slot_stride, a.scale, a.act, a.gate_k,
      a.l2norm, a.state_vk);
  return cudaGetLastError();
}

template <typename QT, typename ST>
cudaError_t launch_kv(const PrefillArgs& a, cudaStream_t st) {
  const int K = a.d.head_k_dim, V = a.d.head_v_dim;
  if (K == 128 && V == 128) return launch_typed<QT, ST, 128, 128>(a, st);
  if (K == 128 && V == 64) return launch_typed<QT, ST, 128, 64>(a, st);
  if (K == 64 && V == 128) return launch_typed<QT, ST, 64, 128>(a, st);
  return launch_typed<QT, ST, 64, 64>(a, st);
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs& a, cudaStream_t st) {
  if (a.d.num_seqs == 0) return cudaSuccess;
  const bool qb = a.d.qkv_dtype == KDA_BF16, sb = a.d.state_dtype == KDA_BF16;
  if (qb && sb) return launch_kv<__nv_bfloat16, __nv_bfloat16>(a, st);
  if (qb) return launch_kv<__nv_bfloat16, float>(a, st);
  if (sb) return launch_kv<float, __nv_bfloat16>(a, st);
  return launch_kv<float, float>(a, st);
}

}  // namespace kda
