// kda_prefill_tc.cu -- fused tensor-core (tcgen05 + TMEM + TMA) chunked KDA
// prefill for bf16 q/k/v and 128x128 heads on sm_103a.
//
// Method (per v-head, chunks of C = 64 tokens aligned to each sequence start;
// the chunked pipeline of the sglang PR 27488 digest "KDA SM100 CuteDSL
// prefill": gate prologue, KKT inverse + U/W, h kernel, output kernel -- here
// fused into one persistent kernel so that only q/k/v/g/beta, o and the pool
// rows touch HBM):
//
//   e_r = exp(g_r); per 16-token sub-chunk s: rho_r (inclusive cumulative
//   product from the sub-chunk start), kap_r (exclusive product to its end),
//   pi_s (sub-chunk product); E_s / F_s = products of pi before / after s.
//   Every factor is a product of numbers <= 1, so no exponent is ever positive
//   (the fix the pages describe for the fp32 overflow at per-chunk log-decay
//   sums of ~-6e4: PR 27488 digest, 功能与动机 and 实现拆解 item 1).
//
//   A[r,i] = beta_r sum_c k_r k_i prod_{j=i+1..r} e_j    (i < r)
//   B[r,i] = scale  sum_c q_r k_i prod_{j=i+1..r} e_j    (i <= r)
//   computed by ONE MMA  [k rho; q rho] (128 x 128) x CB^T (128 x 192) where
//   CB holds the column tokens pre-scaled for each sub-chunk reference:
//     block 0: k kap                  (adjacent sub-chunk pairs)
//     block 1: k kap pi_1, k kap pi_1 pi_2, k kap pi_2, 0   (distance 2 and 3)
//     block 2: k kap / pi_s = k / rho (diagonal sub-chunks) on channels whose
//              sub-chunk product pi_s >= 2^-64; the remaining ("unsafe")
//              channels get their diagonal terms from an exact pairwise loop.
//   Tm = (I + A)^-1 Diag(beta)   (fp32 blocked inverse on CUDA cores)
//   U~^T = V^T Tm^T,  W^T = KG^T Tm^T                     (MMA, KG = k rho E)
//   per chunk, sequentially (state S^T fp32 in TMEM, lanes = value channel):
//     U^T = U~^T - S^T W^T          (MMA accumulating onto U~)
//     O^T = S^T QG^T + U^T B^T      (QG = scale q rho E)
//     S^T = S^T Diag(gamma) + U^T KR   (KR = k kap F, gamma = prod e)
//
// CTA = 9 warps, one CTA per SM, persistent over (sequence, head) items sorted
// longest first and fetched from a global counter:
//   warp 0     producer: item scheduling, TMA loads of q/k/v, L2 prefetch
//   warps 1-4  intra group (S-independent work of chunk c+1)
//   warps 5-8  recurrence group (state update and output of chunk c)
// Pool I/O (sglang PR 30169 digest, 实现拆解 items 1-3) is fused: the
// recurrence group reads h0 from pool[state_indices[n]] (-1 -> last slot) and
// writes the final state back to the same row.
#include <cudaTypedefs.h>

#include "kda_internal.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int kC = 64;
constexpr int kK = 128;
constexpr int kV = 128;
constexpr int kThreads = 288;
constexpr int kRing = 4;
constexpr float kSafeMin = 5.421010862427522e-20f;  // 2^-64

// ---- shared memory map (offsets from a 1024-aligned base) -------------------------
constexpr uint32_t OFF_QK = 0;        // [2 K-atoms][128 rows: k 0-63 | q 64-127][128 B]
constexpr uint32_t OFF_VB = 32768;    // [2 v-blocks][64 tokens][128 B]        (MN-major A)
constexpr uint32_t OFF_CB = 49152;    // [3 blocks][128 ch][128 B]             (MN-major B)
constexpr uint32_t OFF_KG = 98304;    // [128 ch][64 tokens]                   (K-major A)
constexpr uint32_t OFF_TM = 114688;   // [64 r][64 i]                          (K-major B)
constexpr uint32_t OFF_WB = 122880;   // [128 ch][64 tokens]  -W              (MN-major B)
constexpr uint32_t OFF_QG = 139264;   // [128 ch][64 tokens]  QG              (MN-major B)
constexpr uint32_t OFF_BB = 155648;   // [64 r][64 i]         B               (K-major B)
constexpr uint32_t OFF_KR = 163840;   // [128 ch][64 tokens]  KR              (K-major B)
constexpr uint32_t OFF_ST = 180224;   // [2 K-atoms][128 v][128 B]  S^T bf16   (K-major A)
constexpr uint32_t OFF_UT = 212992;   // [128 v][64 tokens]   U^T bf16        (K-major A)
constexpr uint32_t OFF_SMALL = 229376;
// fp32 scratch of the inverse, aliased on CB blocks 1 and 2 (dead after MMA-AB)
constexpr uint32_t OFF_AS = OFF_CB + 16384;  // A (and B before it is packed), 64x64 fp32
constexpr uint32_t OFF_XS = OFF_CB + 32768;  // B rows, then X = (I + A)^-1, 64x64 fp32

// ---- TMEM columns ------------------------------------------------------------------
constexpr uint32_t TM_U = 0;     // U~ -> U (64)
constexpr uint32_t TM_O = 64;    // O double buffer (2 x 64)
constexpr uint32_t TM_S = 192;   // S^T fp32 (128)
constexpr uint32_t TM_AB = 320;  // A/B result (192), later W^T (64)

enum Bar {
  B_QK_FULL, B_V_FULL, B_QK_FREE, B_VB_FREE, B_AB_DONE, B_UW_DONE, B_GAMMA0, B_GAMMA1,
  B_REC_READY, B_M1A, B_M1B, B_M3A, B_M3B, B_E1, B_DRAIN_IG, B_DRAIN_RG,
  B_ITEM_FULL, B_ITEM_EMPTY = B_ITEM_FULL + kRing, B_COUNT = B_ITEM_EMPTY + kRing
};

struct ItemInfo {
  int32_t n, h, kh, nchunks;
  int64_t bos, eos, slot;  // slot: pool row, or -1 in dense mode
  int32_t done, pad;
};

struct Small {
  uint64_t bar[B_COUNT];
  ItemInfo ring[kRing];
  float beta[kC];
  float gamma[2][kK];
  uint32_t unsafe[4][4];  // [sub-chunk][channel word]
  uint32_t tmem_base;
  uint32_t abort;
};
constexpr uint32_t kSmemBytes = OFF_SMALL + sizeof(Small) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");

struct TcParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_g;
  const __nv_bfloat16 *q, *k;
  const float *g, *beta;
  const int32_t *cu, *idx, *order;
  const void* state_in;
  void* state_out;
  __nv_bfloat16* o;
  uint32_t* status;
  uint32_t* next_item;
  int32_t N, Hk, Hv, num_items;
  int64_t T, num_slots, slot_stride;
  float scale;
};

// ---- small helpers -----------------------------------------------------------------
__device__ __forceinline__ float bf_bits(uint32_t b16) { return __uint_as_float(b16 << 16); }
__device__ __forceinline__ uint16_t to_bf_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
// Element (row, ch) of a K-major operand with 128 channels in two 64-wide atoms.
__device__ __forceinline__ uint32_t kmaj_elem(uint32_t row, uint32_t ch, uint32_t rows_per_atom) {
  return (ch >> 6) * rows_per_atom * 128u + sw128_off(row, (ch & 63u) >> 3) + (ch & 7u) * 2u;
}
__device__ __forceinline__ void st_chunk(uint8_t* sm, uint32_t off, uint32_t a, uint32_t b,
                                         uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4*>(sm + off) = make_uint4(a, b, c, d);
}
__device__ __forceinline__ int sidx(int r, int i) { return r * 64 + (i ^ ((r & 7) << 2)); }

__device__ __forceinline__ void fail(const TcParams& p, Small* s) {
  if (atomicExch(&s->abort, 1u) == 0u) raise_status(p.status, KDA_DEVICE_PIPE_TIMEOUT);
}
__device__ __forceinline__ bool aborted(Small* s) {
  return *reinterpret_cast<volatile uint32_t*>(&s->abort) != 0u;
}
// Bounded wait.  A timeout marks the CTA aborted and every later wait fails at
// once; callers never branch on the result inside a chunk (control flow stays
// uniform so every named barrier is reached), they leave at chunk boundaries.
__device__ __forceinline__ bool wait_bar(const TcParams& p, Small* s, int b, uint32_t parity) {
  if (mbar_try_wait(&s->bar[b], parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(&s->bar[b], parity)) return true;
    if (aborted(s)) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      fail(p, s);
      return false;
    }
  }
}

// ======================================================================================
// Producer (warp 0, lane 0): items and TMA loads.
// ======================================================================================
__device__ void run_producer(const TcParams& p, uint8_t* sm, Small* s) {
  uint32_t gc = 0, n_qk = 0, n_v = 0;
  for (int k = 0;; ++k) {
    const int slot = k % kRing;
    if (k >= kRing && !wait_bar(p, s, B_ITEM_EMPTY + slot, ((k / kRing) - 1) & 1)) break;
    ItemInfo info{};
    // fetch the next valid item
    for (;;) {
      const uint32_t it = aborted(s) ? (uint32_t)p.num_items : atomicAdd(p.next_item, 1u);
      if (it >= (uint32_t)p.num_items) { info.done = 1; break; }
      const int n = p.order[it / p.Hv], h = it % p.Hv;
      int64_t bos, eos;
      if (!seq_bounds(p.cu, n, p.T, &bos, &eos)) { raise_status(p.status, KDA_DEVICE_BAD_SEQLENS); continue; }
      int64_t sl = -1;
      if (p.idx) {
        sl = resolve_slot(p.idx, n, p.num_slots);
        if (sl < 0) { raise_status(p.status, KDA_DEVICE_BAD_SLOT); continue; }
      }
      info.n = n; info.h = h; info.kh = h / (p.Hv / p.Hk);
      info.bos = bos; info.eos = eos; info.slot = sl;
      info.nchunks = (int)((eos - bos + kC - 1) / kC);
      info.done = 0;
      break;
    }
    s->ring[slot] = info;
    mbar_arrive(&s->bar[B_ITEM_FULL + slot]);
    if (info.done) break;
    bool stop = false;
    for (int lc = 0; lc < info.nchunks; ++lc, ++gc) {
      const int t0 = (int)(info.bos + (int64_t)lc * kC);
      if (gc > 0 && !wait_bar(p, s, B_QK_FREE, (gc - 1) & 1)) { stop = true; break; }
      mbar_expect_tx(&s->bar[B_QK_FULL], 32768);
      ++n_qk;
      tma_load_3d(sm + OFF_QK + 0, &p.tm_k, &s->bar[B_QK_FULL], 0, info.kh, t0);
      tma_load_3d(sm + OFF_QK + 16384, &p.tm_k, &s->bar[B_QK_FULL], 64, info.kh, t0);
      tma_load_3d(sm + OFF_QK + 8192, &p.tm_q, &s->bar[B_QK_FULL], 0, info.kh, t0);
      tma_load_3d(sm + OFF_QK + 24576, &p.tm_q, &s->bar[B_QK_FULL], 64, info.kh, t0);
      tma_prefetch_3d(&p.tm_g, 0, info.h, t0);
      if (lc + 1 < info.nchunks) {
        tma_prefetch_3d(&p.tm_k, 0, info.kh, t0 + kC);
        tma_prefetch_3d(&p.tm_k, 64, info.kh, t0 + kC);
        tma_prefetch_3d(&p.tm_q, 0, info.kh, t0 + kC);
        tma_prefetch_3d(&p.tm_q, 64, info.kh, t0 + kC);
        tma_prefetch_3d(&p.tm_g, 0, info.h, t0 + kC);
      }
      if (gc > 0 && !wait_bar(p, s, B_VB_FREE, (gc - 1) & 1)) { stop = true; break; }
      mbar_expect_tx(&s->bar[B_V_FULL], 16384);
      ++n_v;
      tma_load_3d(sm + OFF_VB + 0, &p.tm_v, &s->bar[B_V_FULL], 0, info.h, t0);
      tma_load_3d(sm + OFF_VB + 8192, &p.tm_v, &s->bar[B_V_FULL], 64, info.h, t0);
      if (lc + 1 < info.nchunks) {
        tma_prefetch_3d(&p.tm_v, 0, info.h, t0 + kC);
        tma_prefetch_3d(&p.tm_v, 64, info.h, t0 + kC);
      }
    }
    if (stop) break;
  }
  // Let the last loads land before the CTA can exit (bounded, ignores abort).
  if (n_qk > 0) mbar_wait(&s->bar[B_QK_FULL], (n_qk - 1) & 1);
  if (n_v > 0) mbar_wait(&s->bar[B_V_FULL], (n_v - 1) & 1);
}

// Reads the next item descriptor (whole group); returns it.  The group leader
// releases the ring slot once every thread of the group has read it.
__device__ __forceinline__ ItemInfo next_item(const TcParams& p, Small* s, int k, bool leader,
                                              uint32_t bar_id, bool& ok) {
  const int slot = k % kRing;
  ok = wait_bar(p, s, B_ITEM_FULL + slot, (k / kRing) & 1);
  ItemInfo info = s->ring[slot];
  const bool stop = named_bar_any(bar_id, 128, !ok || info.done != 0 || aborted(s));
  if (leader && ok) mbar_arrive(&s->bar[B_ITEM_EMPTY + slot]);
  info.done = stop ? 1 : 0;
  return info;
}

// ======================================================================================
// Intra group (warps 1-4): S-independent work of each chunk.
// ======================================================================================
__device__ void run_intra(const TcParams& p, uint8_t* sm, Small* s, uint32_t tbase) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int tl = quad * 32 + lane;  // TMEM lane of this thread / channel of the prologue
  const int it = threadIdx.x - 32;  // 0..127 within the group
  const bool leader_warp = (warp == 1);
  const uint32_t taddr_q = tbase + ((uint32_t)(quad * 32) << 16);
  const uint32_t sbase = smem_u32(sm);
  float* As = reinterpret_cast<float*>(sm + OFF_AS);
  float* Xs = reinterpret_cast<float*>(sm + OFF_XS);
  uint32_t gc = 0;

  for (int k = 0;; ++k) {
    bool ok;
    const ItemInfo info = next_item(p, s, k, it == 0, 1, ok);
    if (info.done) break;
    const int h = info.h, kh = info.kh;
    bool stop = false;
    for (int lc = 0; lc < info.nchunks; ++lc, ++gc) {
      if (named_bar_any(1, 128, aborted(s))) { stop = true; break; }
      const int64_t t0 = info.bos + (int64_t)lc * kC;
      const int cv = (int)min((int64_t)kC, info.eos - t0);
      // ------------------------------------------------------------- prologue
      const int ch = tl;
      float e[kC];
      {
        const float* gp = p.g + ((size_t)t0 * p.Hv + h) * kK + ch;
#pragma unroll
        for (int r = 0; r < kC; ++r) e[r] = (r < cv) ? gp[(size_t)r * p.Hv * kK] : 0.f;
#pragma unroll
        for (int r = 0; r < kC; ++r) e[r] = __expf(e[r]);  // g = 0 on padded rows -> 1
      }
      if (tl < kC) s->beta[tl] = (tl < cv) ? p.beta[(size_t)(t0 + tl) * p.Hv + h] : 0.f;
      float pi[4];
#pragma unroll
      for (int sc = 0; sc < 4; ++sc) {
        float a = 1.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) a *= e[sc * 16 + j];
        pi[sc] = a;
      }
      const float E1v = pi[0], E2v = pi[0] * pi[1], E3v = pi[0] * pi[1] * pi[2];
      const float Es[4] = {1.f, E1v, E2v, E3v};
      const float Fs[4] = {pi[1] * pi[2] * pi[3], pi[2] * pi[3], pi[3], 1.f};
      bool safe[4];
#pragma unroll
      for (int sc = 0; sc < 4; ++sc) {
        safe[sc] = pi[sc] >= kSafeMin;
        const uint32_t m = __ballot_sync(0xffffffffu, !safe[sc]);
        if (lane == 0) s->unsafe[sc][quad] = m;
      }
      wait_bar(p, s, B_QK_FULL, gc & 1);
      // QG buffer and this gamma buffer are free once MMA-1b of the previous chunk ran
      if (gc > 0) wait_bar(p, s, B_M1B, (gc - 1) & 1);
      s->gamma[gc & 1][ch] = E3v * pi[3];
#pragma unroll
      for (int sc = 0; sc < 4; ++sc) {
        float kap[16];
        {
          float a = 1.f;
#pragma unroll
          for (int j = 15; j >= 0; --j) { kap[j] = a; a *= e[sc * 16 + j]; }
        }
        const float inv_pi = safe[sc] ? 1.f / pi[sc] : 0.f;
        uint32_t w_cb0[8], w_dg[8], w_kg[8], w_qg[8], w_m1[8], w_m12[8], w_m2[8];
        float rho = 1.f;
        const float qscale = p.scale * Es[sc];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          float kk[2], dg[2], kg[2], qg[2], m1[2], m12[2], m2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int r = sc * 16 + j + u;
            rho *= e[r];
            const uint32_t ka = kmaj_elem(r, ch, 128), qa = kmaj_elem(64 + r, ch, 128);
            uint16_t* kp = reinterpret_cast<uint16_t*>(sm + OFF_QK + ka);
            uint16_t* qp = reinterpret_cast<uint16_t*>(sm + OFF_QK + qa);
            const float kv = (r < cv) ? bf_bits(*kp) : 0.f;
            const float qv = (r < cv) ? bf_bits(*qp) : 0.f;
            *kp = to_bf_bits(kv * rho);
            *qp = to_bf_bits(qv * rho);
            kk[u] = kv * kap[j + u];
            dg[u] = kk[u] * inv_pi;
            kg[u] = kv * rho * Es[sc];
            qg[u] = qv * rho * qscale;
            m1[u] = kk[u] * pi[1];
            m12[u] = kk[u] * pi[1] * pi[2];
            m2[u] = kk[u] * pi[2];
          }
          w_cb0[j / 2] = pack_bf16x2(kk[0], kk[1]);
          w_dg[j / 2] = pack_bf16x2(dg[0], dg[1]);
          w_kg[j / 2] = pack_bf16x2(kg[0], kg[1]);
          w_qg[j / 2] = pack_bf16x2(qg[0], qg[1]);
          w_m1[j / 2] = pack_bf16x2(m1[0], m1[1]);
          w_m12[j / 2] = pack_bf16x2(m12[0], m12[1]);
          w_m2[j / 2] = pack_bf16x2(m2[0], m2[1]);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t cj = sc * 2 + hh, o = hh * 4;
          st_chunk(sm, OFF_CB + 0 + sw128_off(ch, cj), w_cb0[o], w_cb0[o + 1], w_cb0[o + 2], w_cb0[o + 3]);
          st_chunk(sm, OFF_CB + 32768 + sw128_off(ch, cj), w_dg[o], w_dg[o + 1], w_dg[o + 2], w_dg[o + 3]);
          st_chunk(sm, OFF_KG + sw128_off(ch, cj), w_kg[o], w_kg[o + 1], w_kg[o + 2], w_kg[o + 3]);
          st_chunk(sm, OFF_QG + sw128_off(ch, cj), w_qg[o], w_qg[o + 1], w_qg[o + 2], w_qg[o + 3]);
          if (sc == 0) {
            st_chunk(sm, OFF_CB + 16384 + sw128_off(ch, 0 + hh), w_m1[o], w_m1[o + 1], w_m1[o + 2], w_m1[o + 3]);
            st_chunk(sm, OFF_CB + 16384 + sw128_off(ch, 2 + hh), w_m12[o], w_m12[o + 1], w_m12[o + 2], w_m12[o + 3]);
          } else if (sc == 1) {
            st_chunk(sm, OFF_CB + 16384 + sw128_off(ch, 4 + hh), w_m2[o], w_m2[o + 1], w_m2[o + 2], w_m2[o + 3]);
          } else if (sc == 3) {
            st_chunk(sm, OFF_CB + 16384 + sw128_off(ch, 6 + hh), 0u, 0u, 0u, 0u);
          }
        }
      }
      fence_async_smem();
      named_bar(1, 128);
      if (it == 0) mbar_arrive(&s->bar[B_GAMMA0 + (gc & 1)]);
      if (leader_warp) {
        if (lane == 0) {
          tc_fence_after();
          const uint32_t idesc = idesc_bf16(128, 192, 0, 1);
#pragma unroll
          for (int st = 0; st < 8; ++st) {
            const uint64_t a = sdesc_sw128(sbase + OFF_QK + (st >> 2) * 16384 + (st & 3) * 32, 16, 1024);
            const uint64_t b = sdesc_sw128(sbase + OFF_CB + st * 2048, 16384, 1024);
            mma_bf16(tbase + TM_AB, a, b, idesc, st > 0 ? 1u : 0u);
          }
          mma_commit(&s->bar[B_AB_DONE]);
          mma_commit(&s->bar[B_QK_FREE]);
        }
        __syncwarp();
      }
      // ------------------------------------------------------------- A / B rows
      wait_bar(p, s, B_AB_DONE, gc & 1);
      tc_fence_after();
      {
        const int L = tl, r = L & 63, a = r >> 4;
        const bool isB = L >= 64;
        const int a0 = (r >> 5) * 2;  // the two sub-chunks of this warp: a0, a0 + 1
        float x[kC];
#pragma unroll
        for (int i = 0; i < kC; ++i) x[i] = 0.f;
        // column of TMEM (relative to TM_AB) holding block (row sub-chunk aa, column block b)
        auto colof = [](int aa, int b) -> int {
          if (b == aa) return 128 + 16 * aa;
          if (b == aa - 1) return 16 * b;
          if (b == aa - 2) return aa == 2 ? 64 : 96;
          if (b == aa - 3) return 80;
          return -1;
        };
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          float v0[16], v1[16];
          const int c0 = (b <= a0) ? colof(a0, b) : -1;
          const int c1 = (b <= a0 + 1) ? colof(a0 + 1, b) : -1;
          if (c0 >= 0) tmem_ld16(taddr_q + TM_AB + c0, v0);
          if (c1 >= 0) tmem_ld16(taddr_q + TM_AB + c1, v1);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float val = 0.f;
            if (a == a0 && c0 >= 0) val = v0[j];
            if (a == a0 + 1 && c1 >= 0) val = v1[j];
            x[16 * b + j] = val;
          }
        }
        tc_fence_before();
        float* row = (isB ? Xs : As);
#pragma unroll
        for (int i = 0; i < kC; ++i) row[sidx(r, i)] = x[i];
      }
      named_bar(1, 128);
      // exact pairwise terms of the diagonal sub-chunk blocks on "unsafe" channels
      {
        const int L = tl, r = L & 63, a = r >> 4;
        const bool isB = L >= 64;
        uint32_t any = 0;
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) any |= s->unsafe[a][wd];
        if (any != 0u && r < cv) {
          float* row = (isB ? Xs : As);
          const __nv_bfloat16* xsrc = isB ? p.q : p.k;
          for (int wd = 0; wd < 4; ++wd) {
            uint32_t m = s->unsafe[a][wd];
            while (m) {
              const int c = wd * 32 + (__ffs(m) - 1);
              m &= m - 1;
              const float xr = __bfloat162float(xsrc[((size_t)(t0 + r) * p.Hk + kh) * kK + c]);
              float pr = 1.f;
              for (int i = r; i >= a * 16; --i) {
                const float ki = __bfloat162float(p.k[((size_t)(t0 + i) * p.Hk + kh) * kK + c]);
                row[sidx(r, i)] += xr * ki * pr;
                pr *= __expf(p.g[((size_t)(t0 + i) * p.Hv + h) * kK + c]);
                if (pr == 0.f) break;
              }
            }
          }
        }
      }
      named_bar(1, 128);
      // A: mask + beta_r (in place); B: mask + scale -> bf16 -> BB
      {
        const int L = tl, r = L & 63;
        if (L < 64) {
          const float br = s->beta[r];
#pragma unroll
          for (int i = 0; i < kC; ++i) {
            const float v = As[sidx(r, i)];
            As[sidx(r, i)] = (i < r) ? br * v : 0.f;
          }
        } else {
          if (gc > 0) wait_bar(p, s, B_M3A, (gc - 1) & 1);  // BB free
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int i0 = j * 8 + u * 2;
              const float v0 = (i0 <= r) ? p.scale * Xs[sidx(r, i0)] : 0.f;
              const float v1 = (i0 + 1 <= r) ? p.scale * Xs[sidx(r, i0 + 1)] : 0.f;
              w[u] = pack_bf16x2(v0, v1);
            }
            st_chunk(sm, OFF_BB + sw128_off(r, j), w[0], w[1], w[2], w[3]);
          }
        }
      }
      named_bar(1, 128);
      // ------------------------------------------------------------- inverse
      // (1) 16x16 diagonal blocks by forward substitution: thread (blk, col j)
      if (it < 64) {
        const int blk = it >> 4, j = it & 15, o = blk * 16;
        float xv[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) xv[rr] = (rr == j) ? 1.f : 0.f;
#pragma unroll
        for (int rr = 1; rr < 16; ++rr) {
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < rr; ++i) acc = fmaf(As[sidx(o + rr, o + i)], xv[i], acc);
          if (rr > j) xv[rr] = -acc;
        }
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) Xs[sidx(o + rr, o + j)] = xv[rr];
      } else {
        // zero the blocks of X above the diagonal blocks' rows that merges do not write
        const int t2 = it - 64;  // 0..63: clear row t2's strictly-upper 16-blocks
        const int rb = t2 >> 4;
#pragma unroll
        for (int i = 0; i < kC; ++i)
          if ((i >> 4) > rb) Xs[sidx(t2, i)] = 0.f;
      }
      named_bar(1, 128);
      // (2) level-1 merges: X_{2m+1,2m} = -X_{2m+1,2m+1} (A_{2m+1,2m} X_{2m,2m})
      {
        const int m = it >> 6, e2 = it & 63, rr = e2 >> 2, j0 = (e2 & 3) * 4;
        const int ro = (2 * m + 1) * 16, co = 2 * m * 16;
        float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float av = As[sidx(ro + rr, co + i)];
#pragma unroll
          for (int u = 0; u < 4; ++u) t[u] = fmaf(av, Xs[sidx(co + i, co + j0 + u)], t[u]);
        }
        // temp T in A's unused upper block (rows co..co+15, cols ro..ro+15)
#pragma unroll
        for (int u = 0; u < 4; ++u) As[sidx(co + rr, ro + j0 + u)] = t[u];
      }
      named_bar(1, 128);
      {
        const int m = it >> 6, e2 = it & 63, rr = e2 >> 2, j0 = (e2 & 3) * 4;
        const int ro = (2 * m + 1) * 16, co = 2 * m * 16;
        float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float xv = Xs[sidx(ro + rr, ro + i)];
#pragma unroll
          for (int u = 0; u < 4; ++u) t[u] = fmaf(xv, As[sidx(co + i, ro + j0 + u)], t[u]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) Xs[sidx(ro + rr, co + j0 + u)] = -t[u];
      }
      named_bar(1, 128);
      // (3) level-2 merge: X_21 = -X_22 (A_21 X_11), 32x32 blocks
      {
        const int rr = it >> 2, j0 = (it & 3) * 8;
        float t[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) t[u] = 0.f;
#pragma unroll 8
        for (int i = 0; i < 32; ++i) {
          const float av = As[sidx(32 + rr, i)];
#pragma unroll
          for (int u = 0; u < 8; ++u) t[u] = fmaf(av, Xs[sidx(i, j0 + u)], t[u]);
        }
        // temp T2 in A's unused upper-right quadrant (rows 0..31, cols 32..63)
#pragma unroll
        for (int u = 0; u < 8; ++u) As[sidx(rr, 32 + j0 + u)] = t[u];
      }
      named_bar(1, 128);
      {
        const int rr = it >> 2, j0 = (it & 3) * 8;
        float t[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) t[u] = 0.f;
#pragma unroll 8
        for (int i = 0; i < 32; ++i) {
          const float xv = Xs[sidx(32 + rr, 32 + i)];
#pragma unroll
          for (int u = 0; u < 8; ++u) t[u] = fmaf(xv, As[sidx(i, 32 + j0 + u)], t[u]);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) Xs[sidx(32 + rr, j0 + u)] = -t[u];
      }
      named_bar(1, 128);
      // Tm = X Diag(beta) -> bf16 -> TM (row r, half hh)
      {
        const int rr = it >> 1, hh = it & 1;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = hh * 4 + jj;
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i0 = j * 8 + u * 2;
            const float v0 = (i0 <= rr) ? Xs[sidx(rr, i0)] * s->beta[i0] : 0.f;
            const float v1 = (i0 + 1 <= rr) ? Xs[sidx(rr, i0 + 1)] * s->beta[i0 + 1] : 0.f;
            w[u] = pack_bf16x2(v0, v1);
          }
          st_chunk(sm, OFF_TM + sw128_off(rr, j), w[0], w[1], w[2], w[3]);
        }
      }
      fence_async_smem();
      named_bar(1, 128);
      // ------------------------------------------------------------- U~ and W
      if (leader_warp) {
        bool okw = wait_bar(p, s, B_V_FULL, gc & 1);
        if (okw && gc > 0) okw = wait_bar(p, s, B_E1, (gc - 1) & 1);  // U region read
        if (okw && lane == 0) {
          tc_fence_after();
          const uint32_t idu = idesc_bf16(128, 64, 1, 0), idw = idesc_bf16(128, 64, 0, 0);
#pragma unroll
          for (int st = 0; st < 4; ++st) {
            const uint64_t b = sdesc_sw128(sbase + OFF_TM + st * 32, 16, 1024);
            mma_bf16(tbase + TM_U, sdesc_sw128(sbase + OFF_VB + st * 2048, 8192, 1024), b, idu,
                     st > 0 ? 1u : 0u);
            mma_bf16(tbase + TM_AB, sdesc_sw128(sbase + OFF_KG + st * 32, 16, 1024), b, idw,
                     st > 0 ? 1u : 0u);
          }
          mma_commit(&s->bar[B_UW_DONE]);
          mma_commit(&s->bar[B_VB_FREE]);
        }
        __syncwarp();
      }
      wait_bar(p, s, B_UW_DONE, gc & 1);
      tc_fence_after();
      // -W^T rows -> WB (row = channel tl)
      if (gc > 0) wait_bar(p, s, B_M1A, (gc - 1) & 1);
#pragma unroll
      for (int cq = 0; cq < 4; ++cq) {
        float wv[16];
        tmem_ld16(taddr_q + TM_AB + cq * 16, wv);
        tmem_ld_wait();
        uint32_t w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) w[u] = pack_bf16x2(-wv[2 * u], -wv[2 * u + 1]);
        st_chunk(sm, OFF_WB + sw128_off(tl, cq * 2), w[0], w[1], w[2], w[3]);
        st_chunk(sm, OFF_WB + sw128_off(tl, cq * 2 + 1), w[4], w[5], w[6], w[7]);
      }
      tc_fence_before();
      // KR = (k kap) F_s : scaled copy of CB block 0 row `ch` into KR
      if (gc > 0) wait_bar(p, s, B_M3B, (gc - 1) & 1);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 src = *reinterpret_cast<const uint4*>(sm + OFF_CB + sw128_off(ch, j));
        const float f = Fs[j >> 1];
        const uint32_t in[4] = {src.x, src.y, src.z, src.w};
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          w[u] = pack_bf16x2(bf_bits(in[u] & 0xFFFFu) * f, bf_bits(in[u] >> 16) * f);
        st_chunk(sm, OFF_KR + sw128_off(ch, j), w[0], w[1], w[2], w[3]);
      }
      fence_async_smem();
      named_bar(1, 128);
      if (it == 0) mbar_arrive(&s->bar[B_REC_READY]);
    }
    if (stop) break;
  }
  // drain this group's MMAs before the CTA can release TMEM
  named_bar(1, 128);
  if (leader_warp) {
    if (lane == 0) mma_commit(&s->bar[B_DRAIN_IG]);
    __syncwarp();
    wait_bar(p, s, B_DRAIN_IG, 0);
  }
}

// ======================================================================================
// Recurrence group (warps 5-8): state update and output, chunk by chunk.
// ======================================================================================
template <typename ST>
__device__ void run_recurrence(const TcParams& p, uint8_t* sm, Small* s, uint32_t tbase) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int v = quad * 32 + lane;  // TMEM lane = value channel
  const int rt = threadIdx.x - 160;
  const bool leader_warp = (warp == 5);
  const uint32_t taddr_q = tbase + ((uint32_t)(quad * 32) << 16);
  const uint32_t sbase = smem_u32(sm);
  uint32_t gc = 0;
  // deferred output epilogue of the previous chunk
  bool pend = false;
  int64_t pend_t0 = 0;
  int pend_cv = 0, pend_h = 0;
  uint32_t pend_gc = 0;

  auto o_epilogue = [&]() {
    if (!pend) return;
    pend = false;
    if (!wait_bar(p, s, B_M3A, pend_gc & 1)) return;
    tc_fence_after();
    __nv_bfloat16* op = p.o + ((size_t)pend_t0 * p.Hv + pend_h) * kV + v;
#pragma unroll
    for (int cq = 0; cq < 4; ++cq) {
      float ov[16];
      tmem_ld16(taddr_q + TM_O + 64 * (pend_gc & 1) + cq * 16, ov);
      tmem_ld_wait();
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int r = cq * 16 + u;
        if (r < pend_cv) op[(size_t)r * p.Hv * kV] = __float2bfloat16_rn(ov[u]);
      }
    }
    tc_fence_before();
  };

  for (int k = 0;; ++k) {
    bool ok;
    const ItemInfo info = next_item(p, s, k, rt == 0, 2, ok);
    if (info.done) break;
    const int h = info.h;
    const ST* src = nullptr;
    ST* dst = nullptr;
    const size_t hoff = (size_t)h * kK * kV;
    if (info.slot >= 0) {
      src = static_cast<const ST*>(p.state_in) + info.slot * p.slot_stride + hoff;
      dst = static_cast<ST*>(p.state_out) + info.slot * p.slot_stride + hoff;
    } else {
      if (p.state_in) src = static_cast<const ST*>(p.state_in) + ((size_t)info.n * p.Hv) * kK * kV + hoff;
      if (p.state_out) dst = static_cast<ST*>(p.state_out) + ((size_t)info.n * p.Hv) * kK * kV + hoff;
    }
    if (info.nchunks == 0) {  // empty sequence: the final state is the initial one
      if (dst && dst != src)
        for (int c = 0; c < kK; ++c) dst[(size_t)c * kV + v] = src ? src[(size_t)c * kV + v] : ST(0.f);
      continue;
    }
    // ---- initial state: S^T row v -> ST (bf16) and TMEM S (pre-decayed by gamma of chunk 0)
    wait_bar(p, s, B_GAMMA0 + (gc & 1), (gc >> 1) & 1);
#pragma unroll
    for (int kq = 0; kq < 8; ++kq) {
      float sv[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int c = kq * 16 + u;
        sv[u] = src ? to_f32(src[(size_t)c * kV + v]) : 0.f;
      }
      uint32_t w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) w[u] = pack_bf16x2(sv[2 * u], sv[2 * u + 1]);
      const uint32_t cj = kq * 2;
      st_chunk(sm, OFF_ST + (cj >> 3) * 16384 + sw128_off(v, cj & 7), w[0], w[1], w[2], w[3]);
      st_chunk(sm, OFF_ST + ((cj + 1) >> 3) * 16384 + sw128_off(v, (cj + 1) & 7), w[4], w[5], w[6], w[7]);
#pragma unroll
      for (int u = 0; u < 16; ++u) sv[u] *= s->gamma[gc & 1][kq * 16 + u];
      tmem_st16(taddr_q + TM_S + kq * 16, sv);
    }
    tmem_st_wait();
    tc_fence_before();
    fence_async_smem();
    named_bar(2, 128);

    bool stop = false;
    for (int lc = 0; lc < info.nchunks; ++lc, ++gc) {
      if (named_bar_any(2, 128, aborted(s))) { stop = true; break; }
      const int64_t t0 = info.bos + (int64_t)lc * kC;
      const int cv = (int)min((int64_t)kC, info.eos - t0);
      const bool last = (lc + 1 == info.nchunks);
      // ---- R1: U~ -= S W^T ; O = S QG^T   (leader warp)
      if (leader_warp) {
        const bool okr = wait_bar(p, s, B_REC_READY, gc & 1);
        if (okr && lane == 0) {
          tc_fence_after();
          const uint32_t id1 = idesc_bf16(128, 64, 0, 1);
#pragma unroll
          for (int st = 0; st < 8; ++st) {
            const uint64_t a = sdesc_sw128(sbase + OFF_ST + (st >> 2) * 16384 + (st & 3) * 32, 16, 1024);
            mma_bf16(tbase + TM_U, a, sdesc_sw128(sbase + OFF_WB + st * 2048, 16384, 1024), id1, 1u);
          }
          mma_commit(&s->bar[B_M1A]);
#pragma unroll
          for (int st = 0; st < 8; ++st) {
            const uint64_t a = sdesc_sw128(sbase + OFF_ST + (st >> 2) * 16384 + (st & 3) * 32, 16, 1024);
            mma_bf16(tbase + TM_O + 64 * (gc & 1), a,
                     sdesc_sw128(sbase + OFF_QG + st * 2048, 16384, 1024), id1, st > 0 ? 1u : 0u);
          }
          mma_commit(&s->bar[B_M1B]);
        }
        __syncwarp();
      }
      o_epilogue();
      // ---- E1: U^T row v -> UT (bf16)
      wait_bar(p, s, B_M1A, gc & 1);
      tc_fence_after();
#pragma unroll
      for (int cq = 0; cq < 4; ++cq) {
        float uv[16];
        tmem_ld16(taddr_q + TM_U + cq * 16, uv);
        tmem_ld_wait();
        uint32_t w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) w[u] = pack_bf16x2(uv[2 * u], uv[2 * u + 1]);
        st_chunk(sm, OFF_UT + sw128_off(v, cq * 2), w[0], w[1], w[2], w[3]);
        st_chunk(sm, OFF_UT + sw128_off(v, cq * 2 + 1), w[4], w[5], w[6], w[7]);
      }
      tc_fence_before();
      fence_async_smem();
      named_bar(2, 128);
      if (rt == 0) {
        mbar_arrive(&s->bar[B_E1]);
        tc_fence_after();
        const uint32_t id3 = idesc_bf16(128, 128, 0, 0), id3o = idesc_bf16(128, 64, 0, 0);
#pragma unroll
        for (int st = 0; st < 4; ++st)
          mma_bf16(tbase + TM_S, sdesc_sw128(sbase + OFF_UT + st * 32, 16, 1024),
                   sdesc_sw128(sbase + OFF_KR + st * 32, 16, 1024), id3, 1u);
        mma_commit(&s->bar[B_M3B]);
#pragma unroll
        for (int st = 0; st < 4; ++st)
          mma_bf16(tbase + TM_O + 64 * (gc & 1), sdesc_sw128(sbase + OFF_UT + st * 32, 16, 1024),
                   sdesc_sw128(sbase + OFF_BB + st * 32, 16, 1024), id3o, 1u);
        mma_commit(&s->bar[B_M3A]);
      }
      // ---- E2: S -> ST (bf16) and pre-decay for the next chunk, or the final store
      wait_bar(p, s, B_M3B, gc & 1);
      tc_fence_after();
      if (!last) wait_bar(p, s, B_GAMMA0 + ((gc + 1) & 1), ((gc + 1) >> 1) & 1);
#pragma unroll
      for (int kq = 0; kq < 8; ++kq) {
        float sv[16];
        tmem_ld16(taddr_q + TM_S + kq * 16, sv);
        tmem_ld_wait();
        if (!last) {
          uint32_t w[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) w[u] = pack_bf16x2(sv[2 * u], sv[2 * u + 1]);
          const uint32_t cj = kq * 2;
          st_chunk(sm, OFF_ST + (cj >> 3) * 16384 + sw128_off(v, cj & 7), w[0], w[1], w[2], w[3]);
          st_chunk(sm, OFF_ST + ((cj + 1) >> 3) * 16384 + sw128_off(v, (cj + 1) & 7), w[4], w[5], w[6], w[7]);
          const float* gm = s->gamma[(gc + 1) & 1];
#pragma unroll
          for (int u = 0; u < 16; ++u) sv[u] *= gm[kq * 16 + u];
          tmem_st16(taddr_q + TM_S + kq * 16, sv);
        } else if (dst) {
#pragma unroll
          for (int u = 0; u < 16; ++u) dst[(size_t)(kq * 16 + u) * kV + v] = from_f32<ST>(sv[u]);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      fence_async_smem();
      named_bar(2, 128);
      pend = true;
      pend_t0 = t0;
      pend_cv = cv;
      pend_h = h;
      pend_gc = gc;
    }
    if (stop) break;
  }
  o_epilogue();
  named_bar(2, 128);
  if (leader_warp) {
    if (lane == 0) mma_commit(&s->bar[B_DRAIN_RG]);
    __syncwarp();
    wait_bar(p, s, B_DRAIN_RG, 0);
  }
}

template <typename ST>
__global__ void __launch_bounds__(kThreads, 1) kda_prefill_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  Small* s = reinterpret_cast<Small*>(sm + OFF_SMALL);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int b = 0; b < B_COUNT; ++b) mbar_init(&s->bar[b], 1);
    for (int r = 0; r < kRing; ++r) mbar_init(&s->bar[B_ITEM_EMPTY + r], 2);
    s->abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&p.tm_q);
    prefetch_tensormap(&p.tm_k);
    prefetch_tensormap(&p.tm_v);
    prefetch_tensormap(&p.tm_g);
  }
  if (warp == 0) tmem_alloc(&s->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s->tmem_base;
  if (warp == 0) {
    if ((threadIdx.x & 31) == 0) run_producer(p, sm, s);
  } else if (warp <= 4) {
    run_intra(p, sm, s, tbase);
  } else {
    run_recurrence<ST>(p, sm, s, tbase);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

// Sequences ordered longest first (ties by index) so the longest (sequence, head)
// chains start first on the persistent grid.
__global__ void kda_order_kernel(const int32_t* __restrict__ cu, int N, int64_t T,
                                 int32_t* __restrict__ order) {
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    const int64_t a = cu[n], b = cu[n + 1];
    const int64_t ln = (a >= 0 && b >= a && b <= T) ? b - a : 0;
    int rank = 0;
    for (int m = 0; m < N; ++m) {
      const int64_t am = cu[m], bm = cu[m + 1];
      const int64_t lm = (am >= 0 && bm >= am && bm <= T) ? bm - am : 0;
      rank += (lm > ln) || (lm == ln && m < n);
    }
    order[rank] = n;
  }
}
__global__ void kda_identity_order_kernel(int N, int32_t* __restrict__ order) {
  for (int n = blockIdx.x * blockDim.x + threadIdx.x; n < N; n += gridDim.x * blockDim.x)
    order[n] = n;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 3-D map over a [T, H, D] row-major tensor: box {64 (or D), 1, 64 tokens}.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem, int64_t T,
              int H, int D, int box_inner, CUtensorMapSwizzle sw) {
  auto enc = get_encoder();
  if (!enc) return false;
  const int64_t rows = T > 0 ? T : 1;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * elem, (cuuint64_t)H * D * elem};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, 1u, (cuuint32_t)kC};
  cuuint32_t es[3] = {1u, 1u, 1u};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

}  // namespace

bool prefill_tc_supported(const kda_desc_t& d) {
  return d.qkv_dtype == KDA_BF16 && d.head_k_dim == kK && d.head_v_dim == kV &&
         (d.flags & KDA_FLAG_CUDA_CORE_PATH) == 0u;
}

size_t prefill_tc_workspace(const kda_desc_t& d) { return (size_t)d.num_seqs * sizeof(int32_t); }

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t st) {
  const kda_desc_t& d = a.d;
  if (d.total_tokens == 0 && d.num_seqs == 0) return cudaSuccess;
  TcParams p;
  memset(&p, 0, sizeof(p));
  const int64_t T = d.total_tokens;
  if (T > 0) {
    if (!make_map(&p.tm_q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, d.num_k_heads, kK, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&p.tm_k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, d.num_k_heads, kK, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&p.tm_v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, d.num_v_heads, kV, 64,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&p.tm_g, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, T, d.num_v_heads, kK, kK,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  int32_t* order = reinterpret_cast<int32_t*>(a.ws + kWsPayload);
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k = static_cast<const __nv_bfloat16*>(a.k);
  p.g = a.g;
  p.beta = a.beta;
  p.cu = a.cu;
  p.idx = a.idx;
  p.order = order;
  p.state_in = a.state_in;
  p.state_out = a.state_out;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.status = a.status;
  p.next_item = &reinterpret_cast<WsHeader*>(a.ws)->next_item;
  p.N = d.num_seqs;
  p.Hk = d.num_k_heads;
  p.Hv = d.num_v_heads;
  p.num_items = d.num_seqs * d.num_v_heads;
  p.T = T;
  p.num_slots = d.num_slots;
  p.slot_stride = a.slot_stride;
  p.scale = a.scale;

  if (d.num_seqs <= 8192)
    kda_order_kernel<<<1, 1024, 0, st>>>(a.cu, d.num_seqs, T, order);
  else
    kda_identity_order_kernel<<<64, 256, 0, st>>>(d.num_seqs, order);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int grid = std::min(sm_count(), std::max(1, p.num_items));
  if (d.state_dtype == KDA_BF16) {
    auto kern = kda_prefill_tc_kernel<__nv_bfloat16>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    kern<<<grid, kThreads, kSmemBytes, st>>>(p);
  } else {
    auto kern = kda_prefill_tc_kernel<float>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    kern<<<grid, kThreads, kSmemBytes, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace kda
