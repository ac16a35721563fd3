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
//   computed by ONE MMA  [k rho; q rho] (128 x 128) x CB^T (128 x 176) where
//   CB holds the column tokens pre-scaled for each sub-chunk reference:
//     block 0: k kap                  (adjacent sub-chunk pairs)
//     block 1: k kap / pi_s = k / rho (diagonal sub-chunks) on channels whose
//              sub-chunk product pi_s >= 2^-100; the remaining ("unsafe")
//              channels get their diagonal terms from an exact pairwise loop.
//     block 2: k kap pi_1, k kap pi_1 pi_2, k kap pi_2   (distance 2 and 3)
//   Tm = (I + A)^-1 Diag(beta): 16x16 diagonal blocks by fp32 forward
//   substitution, off-diagonal blocks by block forward substitution with tf32
//   warp MMAs (tiny, latency-bound 16x16 products)
//   per chunk, sequentially (state S^T fp32 in TMEM, lanes = value channel;
//   KG = k rho E, QG = scale q rho E, KR = k kap F, gamma = prod e):
//     [-Y^T | O^T] = [-V^T | 0] + S^T [KG | QG]^T   (one N = 128 MMA; Tm-independent)
//     U^T = Y^T Tm^T                   (U = Tm (V - KG S), the delta-rule correction)
//     O^T += U^T B^T
//     S^T = S^T Diag(gamma) + U^T KR
//
// CTA = 12 warps, one CTA per SM, persistent over (sequence, head) items sorted
// longest first and claimed from a global counter near the end of the item before:
//   warps 0-7   intra group (S-independent work of chunk c+1 up to the inverted 16x16
//               diagonal blocks of (I + A))
//   warps 8-11  recurrence group (the rest of the inverse, Tm, state update and output
//               of chunk c)
// Pool I/O (sglang PR 30169 digest, 实现拆解 items 1-3) is fused: the
// recurrence group reads h0 from pool[state_indices[n]] (-1 -> last slot) and
// writes the final state back to the same row.
#include <cudaTypedefs.h>

#include <cstddef>

#include "kda_internal.cuh"
#include "tc_ptx.cuh"

namespace kda {
namespace {

KDA_DEBUG_FLAG_DEFINE();
using namespace tc;

constexpr int kC = 64;
constexpr int kK = 128;
constexpr int kV = 128;
constexpr int kThreads = 384;
constexpr int kRing = 4;
// Sub-chunk gate products down to 2^-100 keep k rho >= |k| 2^-100 and k / rho <= 2^100
// normal in bf16 and fp32 (8 exponent bits): the factorised diagonal blocks stay exact to
// bf16 rounding.  Below it a channel takes the pairwise path.
constexpr float kSafeMin = 7.888609052210118e-31f;  // 2^-100

// ---- shared memory map (offsets from a 1024-aligned base) -------------------------
constexpr uint32_t OFF_QK = 0;        // [2 K-atoms][128 rows: k 0-63 | q 64-127][128 B]
constexpr uint32_t OFF_VB = 32768;    // [2 v-blocks][64 tokens][128 B]        (MN-major A)
constexpr uint32_t OFF_CB = 49152;    // [3 blocks][128 ch][128 B]             (MN-major B)
constexpr uint32_t OFF_KG = 98304;    // [128 ch][64 tokens]                   (K-major A)
constexpr uint32_t OFF_TM = 114688;   // [64 r][64 i]                          (K-major B)
constexpr uint32_t OFF_WB = 122880;   // [64 tokens][128 v]   output tile (TMA store)
constexpr uint32_t OFF_QG = 139264;   // [128 ch][64 tokens]  QG              (MN-major B)
constexpr uint32_t OFF_BB = 155648;   // [64 r][64 i]         B               (K-major B)
constexpr uint32_t OFF_KR = 163840;   // [128 ch][64 tokens]  KR              (K-major B)
constexpr uint32_t OFF_AM = 180224;   // [k | q][128 ch][128 B]  k rho, q rho (MN-major A)
constexpr uint32_t OFF_PI = 212992;   // [4 sub-chunks][128 ch] fp32 gate products
constexpr uint32_t OFF_NI = 215040;   // [64 n][64 k] -I (K-major B; builds other than the plain gate)
constexpr uint32_t OFF_SMALL = 229376;
// After MMA-AB completes, the AM buffer holds the fp32 scratch of the inverse (A and B
// rows, then X = (I + A)^-1) until Tm is written, the q/k buffer q and k of the next
// chunk, and CB blocks 1-2 the TMA-staged gate of the next chunk, which the B group turns
// into e = exp(g) ([64][128] fp32) in the same buffer when that chunk is in the same item
// (otherwise each prologue thread forms its e in registers).
constexpr uint32_t OFF_AS = OFF_AM;
constexpr uint32_t OFF_XS = OFF_AM + 16384;
constexpr uint32_t OFF_G = OFF_CB + 16384;

// ---- TMEM columns ------------------------------------------------------------------
// U | O is the N = 128 result of MMA-X, O | S the N = 192 result of MMA-3
constexpr uint32_t TM_U = 0;     // -V^T -> -Y^T -> U^T (64)
constexpr uint32_t TM_O = 64;    // O^T (64)
constexpr uint32_t TM_S = 128;   // S^T fp32 (128)
constexpr uint32_t TM_SB = 256;  // S^T as bf16 pairs: A operand of MMA-X (64); after MMA-X, Y^T
                                 // (32) and U^T (32) as bf16 pairs: A of MMA-U and MMA-3
constexpr uint32_t TM_AB = 320;  // A/B result: 176 of 192 columns, or 64 in the whole-chunk form

constexpr int kIG = 256;  // intra-group threads (warps 0-7)
constexpr int kRG = 128;  // recurrence-group threads (warps 8-11)
constexpr uint32_t BAR_IG = 1, BAR_RG = 2, BAR_A = 3, BAR_B = 4;

enum Bar {
  B_QK_FULL, B_V_FULL, B_G_FULL, B_AB_DONE, B_UW_DONE, B_GAMMA0, B_GAMMA1, B_REC_READY,
  B_M1B, B_M3, B_DRAIN_IG, B_DRAIN_RG,
  B_ITEM_FULL, B_ITEM_EMPTY = B_ITEM_FULL + kRing, B_COUNT = B_ITEM_EMPTY + kRing
};

// Kinds of work-list entries.  A long sequence may be cut in two at a chunk boundary
// (see kda_plan_kernel): its head runs as usual but leaves its final state S_p in the
// split scratch; its tail runs twice from the cut, once from a zero state (outputs o_loc,
// final state S_loc) and once with the values set to zero from the identity matrix
// (outputs y_t = scale M_t^T q_t into the split scratch, final state M, the product of the
// tail's transition matrices).  The state is affine in its start value, so the combine
// kernel completes the tail as o_t = o_loc_t + S_p^T y_t and S_end = M S_p + S_loc.
enum ItemKind : int32_t { KIND_WHOLE = 0, KIND_HEAD = 1, KIND_TAIL = 2, KIND_TAIL_ID = 3 };

struct SplitInfo {  // one cut sequence
  int32_t n, cut;     // sequence, chunks in its head
  int32_t ytok0;      // first row of its tail in the y scratch
  int32_t ntok;       // tokens in its tail
};

struct ItemInfo {
  int32_t n, h, kh, nchunks;
  int64_t bos, eos, slot;  // slot: pool row, or -1 in dense mode
  int32_t done, kind, split, ybase;  // ybase: y-scratch row of token bos (KIND_TAIL_ID)
};

// Scheduling and load state of the threads that claim items and issue loads, kept in
// shared memory so that it holds no registers across the chunk loop.
struct NextChunk {  // the chunk after chunk gc of this CTA, if known when gc's MMA-AB ran
  int32_t have, kh, h, t0, cv;
};
struct LoaderState {
  int32_t pushed, fetched_done;
  uint32_t n_qk, n_g, n_v;  // chunks whose loads were issued (by whichever thread issued them)
  NextChunk nx[2];          // by chunk parity
};

struct Small {
  uint64_t bar[B_COUNT];
  ItemInfo ring[kRing];
  // beta of the chunk, by chunk parity: written after pass B, read by the chunk's extraction
  // and by the recurrence group's Tm, which may still be running when the next chunk writes its
  // own (nothing orders that chunk's pass B after this chunk's Tm)
  alignas(16) float beta[2][kC];   // read as float4
  float inv_nrm[128];              // q/k row norms of the staged chunk (KDA_FLAG_QK_L2NORM)
  alignas(16) float gamma[2][kK];  // read as float4
  // [chunk parity][sub-chunk][half][parity]: bit l = channel 64*half + 2l + parity
  uint32_t unsafe[2][4][2][2];
  LoaderState ld;
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t num_items;  // work-list entries x Hv
  uint32_t whole[2];   // [chunk parity]: the chunk runs as one 64-token sub-chunk
};
// The operand tiles need a 1024-byte aligned base.  The dynamic shared window of a CTA
// starts 1024-byte aligned (after the 1 KB the system reserves per block), so the slack is
// normally unused; a base that would need more than the slack is refused at run time.
constexpr uint32_t kAlignSlack = 232448u - OFF_SMALL - (uint32_t)sizeof(Small) < 1024u
                                     ? (232448u - OFF_SMALL - (uint32_t)sizeof(Small)) & ~15u
                                     : 1024u;
constexpr uint32_t kSmemBytes = OFF_SMALL + sizeof(Small) + kAlignSlack;
static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
static_assert(offsetof(Small, beta) % 16 == 0 && offsetof(Small, gamma) % 16 == 0,
              "vector-read arrays must be 16-byte aligned");

struct TcParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_g;
  CUtensorMap tm_o;   // o [T, Hv, V] bf16, boxes of 64 tokens x one head x 128 values (stores)
  const __nv_bfloat16 *q, *k;
  const float *g, *beta;
  GateAct act;        // act.a set: tm_g maps the gate input a (bf16) instead of g
  uint32_t g_bytes;   // bytes of one staged gate tile (g: 32768, a: 16384; scalar gate: 1024)
  int gate_k;         // 128, or 1 for a scalar gate ([T, Hv]: tiles of 64 tokens x gw heads)
  int gw;             // scalar gate: heads per staged row (4 fp32 g or 8 bf16 a = 16 bytes)
  int l2norm;         // normalise the staged q/k rows (x / max(||x||, 1e-12), back to bf16)
  int state_vk;       // state buffers hold each head's state as [V][K] (KDA_FLAG_STATE_VK)
  const int32_t *cu, *idx;
  const uint32_t* work;      // work list: sequence | kind << 28, longest first
  const SplitInfo* splits;   // cut sequences
  const WsHeader* hdr;       // entries and cuts of the work list
  float *sp, *sl, *mm;       // split scratch: [cuts][Hv][K][V] fp32 each
  __nv_bfloat16* y;          // split scratch: [tail tokens][Hv][K]
  const void* state_in;
  void* state_out;
  __nv_bfloat16* o;
  uint32_t* status;
  uint32_t* next_item;
  uint64_t wait_limit_ns;    // bound of the pipeline waits (kWaitLimitNs unless set shorter)
  int32_t max_cuts, ytok_cap;  // capacities of the split scratch (bounds checks)
  int32_t N, Hk, Hv;
  int64_t T, num_slots, slot_stride;
  float scale;
};

// ---- small helpers -----------------------------------------------------------------
__device__ __forceinline__ float bf_bits(uint32_t b16) { return __uint_as_float(b16 << 16); }
// (a, b) *= (x, y) as one packed fp32 multiply (round to nearest each)
__device__ __forceinline__ void mul2(float& a, float& b, float x, float y) {
  unsigned long long ab, xy;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ab) : "f"(a), "f"(b));
  asm("mov.b64 %0, {%1, %2};" : "=l"(xy) : "f"(x), "f"(y));
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(ab) : "l"(xy));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(ab));
}
// Element (row, ch) of a K-major operand with 128 channels in two 64-wide atoms.
__device__ __forceinline__ uint32_t kmaj_elem(uint32_t row, uint32_t ch, uint32_t rows_per_atom) {
  const uint32_t off = (ch >> 6) * rows_per_atom * 128u + sw128_off(row, (ch & 63u) >> 3) + (ch & 7u) * 2u;
  return KDA_CHECK(off + 4u <= 2u * rows_per_atom * 128u) ? off : 0u;  // inside its tile
}
__device__ __forceinline__ void st_chunk(uint8_t* sm, uint32_t off, uint32_t a, uint32_t b,
                                         uint32_t c, uint32_t d) {
  if (KDA_CHECK(off % 16u == 0u && off + 16u <= OFF_SMALL))  // inside the operand tiles
    *reinterpret_cast<uint4*>(sm + off) = make_uint4(a, b, c, d);
}
// fp32 64x64 scratch index with an XOR swizzle (conflict-free row and fragment reads); the
// debug build maps an index outside the 64x64 tile to element 0 after recording it
__device__ __forceinline__ int sidx(int r, int i) {
  if (!KDA_CHECK(r >= 0 && r < 64 && i >= 0 && i < 64)) return 0;
  return r * 64 + (i ^ ((r & 7) << 2));
}

__device__ __forceinline__ bool aborted(Small* s) {
  return *reinterpret_cast<volatile uint32_t*>(&s->abort) != 0u;
}
// Bounded wait of the pipeline, given up after p.wait_limit_ns.  A timeout marks the CTA
// aborted and every later wait fails at once; callers never branch on the result inside a
// chunk (control flow stays uniform so every named barrier is reached), they leave at chunk
// boundaries, no load is issued once the CTA is aborted, and the drains before the CTA
// exits keep the full limit (mbar_wait), so that no MMA or TMA is in flight when it frees
// its tensor memory.
// A bound shorter than the suspend hint polls with test_wait (try_wait may itself suspend
// the thread until the phase completes, which would let a short bound never run out).  The
// waiting loop is out of line: every wait of the pipeline runs the same few instructions
// rather than a copy per call site, which keeps the chunk loop's code in the SM's
// instruction cache.
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                           uint32_t* abort_flag, uint32_t* status) {
  const bool poll = limit_ns < kSleepHintNs;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (*reinterpret_cast<volatile uint32_t*>(abort_flag) != 0u) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      if (atomicExch(abort_flag, 1u) == 0u) raise_status(status, KDA_DEVICE_PIPE_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_bar(const TcParams& p, Small* s, int b, uint32_t parity) {
  if (mbar_test_wait(&s->bar[b], parity)) return true;
  return wait_bar_slow(&s->bar[b], parity, p.wait_limit_ns, &s->abort, p.status);
}

// Fetches the next valid item (work-list entry, head) from the global counter.
__device__ ItemInfo fetch_item(const TcParams& p, Small* s) {
  ItemInfo info{};
  for (;;) {
    const uint32_t it = aborted(s) ? s->num_items : atomicAdd(p.next_item, 1u);
    if (it >= s->num_items) { info.done = 1; return info; }
    if (!KDA_CHECK(it / (uint32_t)p.Hv < (uint32_t)p.N + 2u * (uint32_t)p.max_cuts)) continue;
    const uint32_t code = p.work[it / p.Hv];
    const int n = (int)(code & 0x0FFFFFFFu), kind = (int)(code >> 28), h = it % p.Hv;
    int64_t bos, eos;
    if (!seq_bounds(p.cu, n, p.T, &bos, &eos)) { raise_status(p.status, KDA_DEVICE_BAD_SEQLENS); continue; }
    int64_t sl = -1;
    if (p.idx) {
      sl = resolve_slot(p.idx, n, p.num_slots);
      if (sl < 0) { raise_status(p.status, KDA_DEVICE_BAD_SLOT); continue; }
    }
    info.split = -1;
    info.ybase = 0;
    if (kind != KIND_WHOLE) {
      const int ns = (int)p.hdr->num_splits;
      for (int i = 0; i < ns; ++i)
        if (p.splits[i].n == n) info.split = i;
      if (info.split < 0 || !KDA_CHECK(info.split < p.max_cuts)) continue;
      const SplitInfo sp = p.splits[info.split];
      const int64_t cut = bos + (int64_t)sp.cut * kC;
      if (kind == KIND_HEAD) {
        eos = cut;
      } else {
        bos = cut;
        info.ybase = sp.ytok0;
      }
    }
    info.n = n; info.h = h; info.kh = h / (p.Hv / p.Hk);
    info.bos = bos; info.eos = eos; info.slot = sl;
    info.nchunks = (int)((eos - bos + kC - 1) / kC);
    info.kind = kind;
    info.done = 0;
    return info;
  }
}

// Reads ring entry k (whole group) and releases it; `done` is uniform.
__device__ __forceinline__ ItemInfo next_item(const TcParams& p, Small* s, int k, bool leader,
                                              uint32_t bar_id, uint32_t nthreads) {
  const int slot = k % kRing;
  const bool ok = wait_bar(p, s, B_ITEM_FULL + slot, (k / kRing) & 1);
  ItemInfo info = s->ring[slot];
  const bool stop = named_bar_any(bar_id, nthreads, !ok || info.done != 0 || aborted(s));
  if (leader && ok) mbar_arrive(&s->bar[B_ITEM_EMPTY + slot]);
  info.done = stop ? 1 : 0;
  return info;
}

// ---- warp-level 16x16x16 products on the legacy tensor path (tf32) ------------------
// acc[nt] (16 x 8 tile nt of a 16x16 result) += M1[r1.., c1..] * M2[r2.., c2..]
__device__ __forceinline__ void blk_mma(float acc[2][4], const float* M1, int r1, int c1,
                                        const float* M2, int r2, int c2, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    uint32_t a[4];
    a[0] = to_tf32(M1[sidx(r1 + g, c1 + 8 * ks + t)]);
    a[1] = to_tf32(M1[sidx(r1 + g + 8, c1 + 8 * ks + t)]);
    a[2] = to_tf32(M1[sidx(r1 + g, c1 + 8 * ks + t + 4)]);
    a[3] = to_tf32(M1[sidx(r1 + g + 8, c1 + 8 * ks + t + 4)]);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      uint32_t b[2];
      b[0] = to_tf32(M2[sidx(r2 + 8 * ks + t, c2 + 8 * nt + g)]);
      b[1] = to_tf32(M2[sidx(r2 + 8 * ks + t + 4, c2 + 8 * nt + g)]);
      mma_tf32_16x8x8(acc[nt], a, b);
    }
  }
}
__device__ __forceinline__ void blk_store(float* M, int r, int c, const float acc[2][4], float sgn,
                                          int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {  // column pairs stay adjacent under the swizzle
    *reinterpret_cast<float2*>(M + sidx(r + g, c + 8 * nt + 2 * t)) =
        make_float2(sgn * acc[nt][0], sgn * acc[nt][1]);
    *reinterpret_cast<float2*>(M + sidx(r + g + 8, c + 8 * nt + 2 * t)) =
        make_float2(sgn * acc[nt][2], sgn * acc[nt][3]);
  }
}

// ======================================================================================
// Intra group (warps 0-7, 256 threads): S-independent work of each chunk.  Its
// thread 0 claims the first item (the recurrence group each later one).  A TMA issue
// blocks its thread for hundreds of cycles, so each load is issued by a thread with
// slack at a point where that thread already knows the target buffer is free: for a
// chunk found by the lookahead, q/k by warp 4 while MMA-AB of the chunk before runs and
// the gate by warp 4 while warps 0-1 invert its diagonal blocks; for a chunk not known
// one chunk ahead, by thread 0; v of every chunk by warp 5 during its own MMA-AB.
// ======================================================================================
struct Loader {  // item claims and loads, by the threads named at each call
  LoaderState* st;

  __device__ void push_one(const TcParams& p, Small* s) {
    if (st->fetched_done) return;
    const int pushed = st->pushed;
    const int slot = pushed % kRing;
    if (pushed >= kRing) wait_bar(p, s, B_ITEM_EMPTY + slot, ((pushed / kRing) - 1) & 1);
    const ItemInfo info = fetch_item(p, s);
    s->ring[slot] = info;
    mbar_arrive(&s->bar[B_ITEM_FULL + slot]);
    st->pushed = pushed + 1;
    if (info.done) st->fetched_done = 1;
  }
  // Each load is issued only while the CTA is not aborted: the issuing thread has then
  // seen the buffer's previous phase complete (its own wait succeeded), so no two loads
  // of one buffer are ever in flight.
  __device__ void load_qk(const TcParams& p, uint8_t* sm, Small* s, int kh, int t0) {
    if (aborted(s)) return;
    mbar_expect_tx(&s->bar[B_QK_FULL], 32768);
    tma_load_3d(sm + OFF_QK + 0, &p.tm_k, &s->bar[B_QK_FULL], 0, kh, t0);
    tma_load_3d(sm + OFF_QK + 16384, &p.tm_k, &s->bar[B_QK_FULL], 64, kh, t0);
    tma_load_3d(sm + OFF_QK + 8192, &p.tm_q, &s->bar[B_QK_FULL], 0, kh, t0);
    tma_load_3d(sm + OFF_QK + 24576, &p.tm_q, &s->bar[B_QK_FULL], 64, kh, t0);
    atomicAdd(&st->n_qk, 1u);
  }
  __device__ void load_g(const TcParams& p, uint8_t* sm, Small* s, int h, int t0) {
    if (aborted(s)) return;
    mbar_expect_tx(&s->bar[B_G_FULL], p.g_bytes);
    if (p.gate_k == 1)  // x = first head of the 16-byte group holding h
      tma_load_2d(sm + OFF_G, &p.tm_g, &s->bar[B_G_FULL], h & ~(p.gw - 1), t0);
    else
      tma_load_3d(sm + OFF_G, &p.tm_g, &s->bar[B_G_FULL], 0, h, t0);
    atomicAdd(&st->n_g, 1u);
  }
  __device__ void load_v(const TcParams& p, uint8_t* sm, Small* s, int h, int t0) {
    if (aborted(s)) return;
    mbar_expect_tx(&s->bar[B_V_FULL], 16384);
    tma_load_3d(sm + OFF_VB + 0, &p.tm_v, &s->bar[B_V_FULL], 0, h, t0);
    tma_load_3d(sm + OFF_VB + 8192, &p.tm_v, &s->bar[B_V_FULL], 64, h, t0);
    atomicAdd(&st->n_v, 1u);
  }
  // Chunk after (item k, local chunk lc), if already known without blocking: item k+1
  // counts once its ring entry is complete (its ITEM_FULL phase, which also orders the
  // entry's contents).  Ring slots k and k+1 cannot be refilled during item k.
  __device__ bool next_chunk(Small* s, int k, int lc, int& kh, int& h, int& t0, int& cv) const {
    const ItemInfo& cur = s->ring[k % kRing];
    if (lc + 1 < cur.nchunks) {
      kh = cur.kh; h = cur.h; t0 = (int)(cur.bos + (int64_t)(lc + 1) * kC);
      cv = (int)min((int64_t)kC, cur.eos - t0);
      return true;
    }
    if (mbar_try_wait(&s->bar[B_ITEM_FULL + (k + 1) % kRing], ((k + 1) / kRing) & 1)) {
      const ItemInfo& nx = s->ring[(k + 1) % kRing];
      if (!nx.done && nx.nchunks > 0) {
        kh = nx.kh; h = nx.h; t0 = (int)nx.bos;
        cv = (int)min((int64_t)kC, nx.eos - nx.bos);
        return true;
      }
    }
    return false;
  }
  __device__ void prefetch_l2(const TcParams& p, int h, int t0) {  // the gate
    if (p.gate_k > 1) tma_prefetch_3d(&p.tm_g, 0, h, t0);
  }
};

// Exact pairwise terms of the diagonal sub-chunk blocks on "unsafe" channels (sub-chunk
// gate product below 2^-100), added to the raw A (As) and B (Xs) rows: thread = TMEM
// lane L (row L & 63 of A for L < 64, of B otherwise).  Kept out of line: it never
// runs at ordinary gates and would otherwise raise the register pressure of the
// chunk loop.
__device__ __noinline__ void unsafe_diag_terms(const TcParams& p, const uint32_t (*uns)[2][2], float* As,
                                               float* Xs, const float* inv_nrm, int L, int64_t t0,
                                               int cv, int kh, int h) {
  const int r = L & 63, a = r >> 4;
  const bool isB = L >= 64;
  const uint32_t anya = uns[a][0][0] | uns[a][0][1] | uns[a][1][0] | uns[a][1][1];
  if (anya != 0u && r < cv) {
    float* row = isB ? Xs : As;
    const __nv_bfloat16* xsrc = isB ? p.q : p.k;
    for (int wd = 0; wd < 4; ++wd) {
      uint32_t m = uns[a][wd >> 1][wd & 1];
      while (m) {
        const int c = 64 * (wd >> 1) + 2 * (__ffs(m) - 1) + (wd & 1);
        m &= m - 1;
        const float xr = __bfloat162float(xsrc[((size_t)(t0 + r) * p.Hk + kh) * kK + c]) *
                         (p.l2norm ? inv_nrm[isB ? 64 + r : r] : 1.f);
        float pr = 1.f;
        for (int i = r; i >= a * 16; --i) {
          const float ki = __bfloat162float(p.k[((size_t)(t0 + i) * p.Hk + kh) * kK + c]) *
                           (p.l2norm ? inv_nrm[i] : 1.f);
          row[sidx(r, i)] += xr * ki * pr;
          const int gk = p.gate_k, gcol = gk > 1 ? c : 0;
          const size_t gi = ((size_t)(t0 + i) * p.Hv + h) * gk + gcol;
          float gv;
          if (p.act.a) {
            const float x = __bfloat162float(static_cast<const __nv_bfloat16*>(p.act.a)[gi]) +
                            (p.act.dt_bias ? p.act.dt_bias[(size_t)h * gk + gcol] : 0.f);
            gv = fmaxf(-__expf(p.act.A_log[h]) * softplus_f32(x), p.act.lb);
          } else {
            gv = p.g[gi];
          }
          pr *= __expf(gv);
          if (pr == 0.f) break;
        }
      }
    }
  }
}

// exp(x) as one ex2 on the multi-function unit, results below 2^-126 flushed to zero:
// an e that low puts its channel's sub-chunk product below 2^-100, so the channel takes
// the pairwise path, and products formed from it differ from exact by under 2^-126.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float exp_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));  // log2(e)
  return y;
}

// e = exp(g) of sub-chunks sc0 .. sc1-1 of one chunk in place over its staged fp32 gate g
// ([64 tokens][128 channels]; each element read and written by the same thread; rows >= cv:
// 1), their products pi into the PI buffer ([4][128] fp32) and the masks of "unsafe"
// channels (pi below 2^-100, or not finite) into `uns`.  Run by nw warps (wg = index among
// them): warp wg covers channels 64 (wg & 1) .. 64 (wg & 1) + 63 of sub-chunks
// sc0 + wg / 2 + i nw / 2, so its reads and writes are full rows.  The products are taken
// token by token in order, as the prologue forms them.
__device__ __forceinline__ void gate_exp_inplace(uint8_t* sm, uint32_t (*uns)[2][2], int cv, int wg, int nw,
                                                 int lane, int sc0, int sc1) {
  const int half = wg & 1, c0 = 2 * (half * 32 + lane);
  float* Es = reinterpret_cast<float*>(sm + OFF_G);
  float* pis = reinterpret_cast<float*>(sm + OFF_PI);
  for (int sc = sc0 + (wg >> 1); sc < sc1; sc += nw >> 1) {
    float pm0 = 1.f, pm1 = 1.f;
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
      const int r = sc * 16 + j;
      float2* ep = reinterpret_cast<float2*>(Es + r * kK + c0);
      const float2 gv = *ep;
      float e0 = gv.x, e1 = gv.y;
      mul2(e0, e1, 1.4426950408889634f, 1.4426950408889634f);  // log2(e)
      e0 = (r < cv) ? ex2_ftz(e0) : 1.f;  // padded rows: decay 1
      e1 = (r < cv) ? ex2_ftz(e1) : 1.f;
      *ep = make_float2(e0, e1);
      mul2(pm0, pm1, e0, e1);
    }
    *reinterpret_cast<float2*>(pis + sc * kK + c0) = make_float2(pm0, pm1);
    const uint32_t m0 = __ballot_sync(0xffffffffu, !(pm0 >= kSafeMin));
    const uint32_t m1 = __ballot_sync(0xffffffffu, !(pm1 >= kSafeMin));
    if (lane == 0) {
      uns[sc][half][0] = m0;
      uns[sc][half][1] = m1;
    }
  }
}

// The rest of X = (I + A)^-1 from its inverted 16x16 diagonal blocks, by the four warps of
// a group (aw = 0..3 within it, named barrier `bar` of 128 threads), with tf32 warp MMAs:
// the two 32x32 diagonal halves X_{a+1,a} = -X_{a+1,a+1} (A_{a+1,a} X_aa) for a = 0, 2 (the
// product staged in the unused upper block (a, a+1) of A), then the lower-left 32x32 block
// -X2 (A21 X1): P_kj = sum_l A_kl X_lj into the upper blocks (k-2, j+2), one 16x16 block per
// warp, and X_ij = -sum_{2<=k<=i} X_ik P_kj.  Ends with X complete (barrier).
__device__ __forceinline__ void inverse_merges(float* As, float* Xs, int aw, int lane, uint32_t bar) {
  if (aw < 2) {
    const int a = aw * 2;
    float acc[2][4] = {};
    blk_mma(acc, As, (a + 1) * 16, a * 16, Xs, a * 16, a * 16, lane);
    blk_store(As, a * 16, (a + 1) * 16, acc, 1.f, lane);
    __syncwarp();
    float acc2[2][4] = {};
    blk_mma(acc2, Xs, (a + 1) * 16, (a + 1) * 16, As, a * 16, (a + 1) * 16, lane);
    blk_store(Xs, (a + 1) * 16, a * 16, acc2, -1.f, lane);
  }
  named_bar(bar, 128);
  {
    const int kb = 2 + (aw >> 1), jb = aw & 1;
    float acc[2][4] = {};
#pragma unroll 1
    for (int l = jb; l < 2; ++l) blk_mma(acc, As, kb * 16, l * 16, Xs, l * 16, jb * 16, lane);
    blk_store(As, (kb - 2) * 16, (jb + 2) * 16, acc, 1.f, lane);
  }
  named_bar(bar, 128);
  {
    const int ib = 2 + (aw >> 1), jb = aw & 1;
    float acc[2][4] = {};
#pragma unroll 1
    for (int kb = 2; kb <= ib; ++kb) blk_mma(acc, Xs, ib * 16, kb * 16, As, (kb - 2) * 16, (jb + 2) * 16, lane);
    blk_store(Xs, ib * 16, jb * 16, acc, -1.f, lane);
  }
  named_bar(bar, 128);
}

// Tm = X Diag(beta) -> bf16, K-major rows in the TM buffer, by 128 threads (row r = i & 63,
// columns 32 (i >> 6) ..).
__device__ __forceinline__ void form_tm(uint8_t* sm, const float* Xs, const float* beta, int i) {
  const int r = i & 63, qq = i >> 6;
#pragma unroll 1
  for (int u2 = 0; u2 < 4; ++u2) {
    const int j = qq * 4 + u2;
    const float4 xa = *reinterpret_cast<const float4*>(Xs + sidx(r, j * 8));
    const float4 xb = *reinterpret_cast<const float4*>(Xs + sidx(r, j * 8 + 4));
    const float4 ba = *reinterpret_cast<const float4*>(beta + j * 8);
    const float4 bb4 = *reinterpret_cast<const float4*>(beta + j * 8 + 4);
    const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
    const float bv[8] = {ba.x, ba.y, ba.z, ba.w, bb4.x, bb4.y, bb4.z, bb4.w};
    uint32_t w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i0 = j * 8 + u * 2;
      w[u] = pack_bf16x2((i0 <= r) ? xv[2 * u] * bv[2 * u] : 0.f,
                         (i0 + 1 <= r) ? xv[2 * u + 1] * bv[2 * u + 1] : 0.f);
    }
    st_chunk(sm, OFF_TM + sw128_off(r, j), w[0], w[1], w[2], w[3]);
  }
}

// MODE: the gate forms the kernel is compiled for, so that a common case's chunk loop carries
// none of the other forms' code:
//   0  the plain fp32 per-channel gate, no q/k normalisation;
//   1  the activated per-channel gate (bf16 or fp32 pre-activation), no q/k normalisation;
//   2  any gate form, with or without KDA_FLAG_QK_L2NORM.
template <int MODE>
__device__ void run_intra(const TcParams& p, uint8_t* sm, Small* s, uint32_t tbase) {
  const int t = threadIdx.x;  // 0..255
  const int warp = t >> 5, lane = t & 31;
  const int quad = warp & 3, hx = warp >> 2;
  const int L = quad * 32 + lane;  // TMEM lane of this thread
  const uint32_t taddr_q = tbase + ((uint32_t)(quad * 32) << 16);
  const uint32_t sbase = smem_u32(sm);
  Loader ld{&s->ld};
  uint32_t gc = 0;
  float bt_next = 0.f;  // beta of the next chunk, read one chunk ahead (threads 0-63)
  bool bt_ok = false;

  // item 0; each later item is claimed by the recurrence group near the end of the one
  // before it
  if (t == 0) ld.push_one(p, s);
  __syncwarp();
  for (int k = 0;; ++k) {
    const ItemInfo info = next_item(p, s, k, t == 0, BAR_IG, kIG);
    if (info.done) break;
    const int h = info.h, kh = info.kh;
    bool stop = false;
    for (int lc = 0; lc < info.nchunks; ++lc, ++gc) {
      if (named_bar_any(BAR_IG, kIG, aborted(s))) { stop = true; break; }
      const int64_t t0 = info.bos + (int64_t)lc * kC;
      const int cv = (int)min((int64_t)kC, info.eos - t0);
      // q/k and the gate of this chunk were issued during the previous chunk iff its
      // lookahead found this one; otherwise thread 0 issues them here.  A plain fp32
      // per-channel gate was turned into e (in its staging buffer) by the B group while the
      // A group inverted the diagonal blocks of the chunk before in the same item; an
      // activated gate (three multi-function operations per element) or a scalar gate, and
      // the first chunk of an item, are turned into e here by all intra threads.
      // (v: during MMA-AB.)
      const bool ahead = gc > 0 && ld.st->nx[(gc - 1) & 1].have;
      const bool plain_gate = MODE == 0 || (MODE == 2 && p.gate_k > 1 && !p.act.a);
      const bool e_ahead = plain_gate && lc > 0;
      if (t == 0) {
        if (!ahead) ld.load_qk(p, sm, s, kh, (int)t0);
        if (ld.st->n_g == gc) ld.load_g(p, sm, s, h, (int)t0);
      }
      __syncwarp();
      // ------------------------------------------------------------- prologue
      // thread = (channel pair c0 = 2*cp, c0+1; sub-chunk sc).  A warp covers 64
      // consecutive channels of one 16-token sub-chunk, so its gate, k and q reads are
      // full rows; row writes alternate the two channels across lane groups so eight
      // consecutive lanes always hit eight different 16-byte positions of the swizzle.
      const int sc = warp >> 1, cp = (warp & 1) * 32 + lane, c0 = 2 * cp;
      const int wsel = (lane >> 2) & 1;  // channel this lane writes first
      float bt = 0.f;  // beta of token t, needed only after the prologue
      if (t < kC && t < cv && KDA_CHECK(t0 + t < p.T))
        bt = bt_ok ? bt_next : p.beta[(size_t)(t0 + t) * p.Hv + h];
      bt_ok = false;
      float e0[16], e1[16];
      if (!e_ahead) {  // e of this chunk from the staged gate, into registers
        wait_bar(p, s, B_G_FULL, gc & 1);
        const float* Gs = reinterpret_cast<const float*>(sm + OFF_G);
        float gA = 0.f, gdb0 = 0.f, gdb1 = 0.f;  // activation constants of head h, channels c0, c0+1
        if (MODE == 1 || (MODE == 2 && p.act.a)) {
          gA = __expf(p.act.A_log[h]);
          if (p.act.dt_bias) {
            const int gk = p.gate_k;
            gdb0 = p.act.dt_bias[(size_t)h * gk + (gk > 1 ? c0 : 0)];
            gdb1 = p.act.dt_bias[(size_t)h * gk + (gk > 1 ? c0 + 1 : 0)];
          }
        }
        // one loop per gate form, so that only the form in use sits in the executed code
        if (MODE == 2 && p.gate_k == 1) {  // scalar gate: staged [64 tokens][gw heads], one value per token
          const int col = h & (p.gw - 1);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = sc * 16 + j;
            float g0;
            if (p.act.a) {
              const float x = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(sm + OFF_G)[r * 8 + col]) + gdb0;
              g0 = fmaxf(-gA * (fmaxf(x, 0.f) + __logf(1.f + __expf(-fabsf(x)))), p.act.lb);
            } else {
              g0 = Gs[r * 4 + col];
            }
            e0[j] = e1[j] = (r < cv) ? exp_ftz(g0) : 1.f;  // padded rows: decay 1
          }
        } else if (MODE == 0 || (MODE == 2 && !p.act.a)) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = sc * 16 + j;
            const float2 gv = *reinterpret_cast<const float2*>(Gs + r * kK + c0);
            e0[j] = (r < cv) ? exp_ftz(gv.x) : 1.f;
            e1[j] = (r < cv) ? exp_ftz(gv.y) : 1.f;
          }
        } else {  // staged tile is a ([64][128] bf16): g = max(-A softplus(a + dt_bias), lb)
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = sc * 16 + j;
            const uint32_t w = *reinterpret_cast<const uint32_t*>(sm + OFF_G + r * 256 + c0 * 2);
            const float x0 = bf_bits(w & 0xFFFFu) + gdb0, x1 = bf_bits(w >> 16) + gdb1;
            const float g0 = fmaxf(-gA * (fmaxf(x0, 0.f) + __logf(1.f + __expf(-fabsf(x0)))), p.act.lb);
            const float g1 = fmaxf(-gA * (fmaxf(x1, 0.f) + __logf(1.f + __expf(-fabsf(x1)))), p.act.lb);
            e0[j] = (r < cv) ? exp_ftz(g0) : 1.f;
            e1[j] = (r < cv) ? exp_ftz(g1) : 1.f;
          }
        }
        float pm0 = 1.f, pm1 = 1.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          pm0 *= e0[j];
          pm1 *= e1[j];
        }
        *reinterpret_cast<float2*>(reinterpret_cast<float*>(sm + OFF_PI) + sc * kK + c0) = make_float2(pm0, pm1);
        const uint32_t m0 = __ballot_sync(0xffffffffu, !(pm0 >= kSafeMin));
        const uint32_t m1 = __ballot_sync(0xffffffffu, !(pm1 >= kSafeMin));
        if (lane == 0) {
          s->unsafe[gc & 1][sc][warp & 1][0] = m0;
          s->unsafe[gc & 1][sc][warp & 1][1] = m1;
        }
      } else {  // turned into e in place by the B group during the previous chunk
        const float* Es = reinterpret_cast<const float*>(sm + OFF_G);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 ev = *reinterpret_cast<const float2*>(Es + (sc * 16 + j) * kK + c0);
          e0[j] = ev.x;
          e1[j] = ev.y;
        }
      }
      wait_bar(p, s, B_QK_FULL, gc & 1);
      if (MODE == 2 && p.l2norm) {
        // staged rows (k 0-63, q 64-127) -> x / max(||x||, 1e-12), re-rounded to bf16 as a
        // caller's normalise-then-cast would; thread = (row, 64-channel half).  The inverse
        // norms are kept for the pairwise path, which reads q and k from global memory.
        const int row = t >> 1, hf = t & 1;
        uint8_t* base = sm + OFF_QK + hf * 16384;
        float ss = 0.f;
#pragma unroll 2
        for (int j = 0; j < 8; ++j) {
          const uint4 w = *reinterpret_cast<const uint4*>(base + sw128_off(row, j));
          const uint32_t u4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float x0 = bf_bits(u4[u] & 0xFFFFu), x1 = bf_bits(u4[u] >> 16);
            ss = fmaf(x0, x0, fmaf(x1, x1, ss));
          }
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        const float inv = 1.f / fmaxf(sqrtf(ss), 1e-12f);
#pragma unroll 2
        for (int j = 0; j < 8; ++j) {
          const uint4 w = *reinterpret_cast<const uint4*>(base + sw128_off(row, j));
          const uint32_t u4[4] = {w.x, w.y, w.z, w.w};
          uint32_t o4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            o4[u] = pack_bf16x2(bf_bits(u4[u] & 0xFFFFu) * inv, bf_bits(u4[u] >> 16) * inv);
          st_chunk(sm, OFF_QK + hf * 16384 + sw128_off(row, j), o4[0], o4[1], o4[2], o4[3]);
        }
        if (hf == 0) s->inv_nrm[row] = inv;
      }
      named_bar(BAR_IG, kIG);  // the products visible
      const float* pis = reinterpret_cast<const float*>(sm + OFF_PI);
      float pi0[4], pi1[4];
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2) {
        const float2 pv = *reinterpret_cast<const float2*>(pis + q2 * kK + c0);
        pi0[q2] = pv.x;
        pi1[q2] = pv.y;
      }
      // pi of this thread's own sub-chunk
      const float pm0 = sc == 0 ? pi0[0] : sc == 1 ? pi0[1] : sc == 2 ? pi0[2] : pi0[3];
      const float pm1 = sc == 0 ? pi1[0] : sc == 1 ? pi1[1] : sc == 2 ? pi1[2] : pi1[3];
      // Every warp holds e and the products before pass A/B overwrite CB and AM.  The same
      // barrier takes the vote on the chunk's form: when the whole-chunk product gamma of
      // every channel is >= 2^-100 (which puts every sub-chunk product above it too), the
      // chunk runs as ONE 64-token sub-chunk -- the diagonal-block factorisation of the
      // four-sub-chunk form applied to the whole chunk: A/B from [k rho; q rho] x (k/rho)^T
      // with rho, the inclusive product from the chunk start, >= 2^-100, so that k rho and
      // k/rho stay normal in bf16.  One CB block instead of three, no block-2 references,
      // an N = 64 MMA-AB, and KG / QG are the MMA-AB operand itself.  Otherwise the chunk
      // takes the four-sub-chunk form with its exact pairwise fallback.
      const float gm0 = pi0[0] * pi0[1] * pi0[2] * pi0[3], gm1 = pi1[0] * pi1[1] * pi1[2] * pi1[3];
      // gamma of this chunk (by warps 6-7, which hold all 128 channels), published by the
      // vote's barrier: the recurrence group reads it at the end of the chunk before, to
      // pre-decay the state it hands on, or at the start of the item.  The value it replaces
      // (two chunks back) was last read before MMA-X of the chunk before that, which the chunk
      // before waited for.
      if (sc == 3) *reinterpret_cast<float2*>(&s->gamma[gc & 1][c0]) = make_float2(gm0, gm1);
      const bool whole = !named_bar_any(BAR_IG, kIG, !(gm0 >= kSafeMin) || !(gm1 >= kSafeMin));
      if (t == 0) {
        s->whole[gc & 1] = whole ? 1u : 0u;
        mbar_arrive(&s->bar[B_GAMMA0 + (gc & 1)]);
      }
      // the gate staging (CB blocks 1-2) is free from here on when this chunk is whole (every
      // thread holds its e, and the one-sub-chunk form neither writes nor reads blocks 1-2):
      // the next chunk of this item gets its gate now, a whole chunk ahead of its use
      if (t == 128 && whole && lc + 1 < info.nchunks && ld.st->n_g == gc + 1)
        ld.load_g(p, sm, s, h, (int)(t0 + kC));
      // inverse scratch: in AM (free after MMA-AB) for the four-sub-chunk form; in the KG and
      // QG buffers when AM is itself KG / QG
      float* As = reinterpret_cast<float*>(sm + (whole ? OFF_KG : OFF_AS));
      float* Xs = reinterpret_cast<float*>(sm + (whole ? OFF_QG : OFF_XS));
      // the chunk before ran as one sub-chunk (its inverse scratch in the KG / QG buffers)
      const bool prev_whole = gc > 0 && s->whole[(gc - 1) & 1] != 0u;
      const float E0 = (sc > 0 ? pi0[0] : 1.f) * (sc > 1 ? pi0[1] : 1.f) * (sc > 2 ? pi0[2] : 1.f);
      const float E1 = (sc > 0 ? pi1[0] : 1.f) * (sc > 1 ? pi1[1] : 1.f) * (sc > 2 ? pi1[2] : 1.f);
      {
        const float ip0 = (pm0 >= kSafeMin) ? __fdividef(1.f, pm0) : 0.f;  // pm = pi of this sub-chunk
        const float ip1 = (pm1 >= kSafeMin) ? __fdividef(1.f, pm1) : 0.f;
        // pass A, tokens in descending order: kap (exclusive product to the sub-chunk
        // end) needs no array.  Writes CB block 0 (k kap), block 1 (k/rho on safe channels:
        // the diagonal sub-chunk blocks) and, by sub-chunk, the block-2 references of the
        // blocks two and three sub-chunks below the diagonal: sub-chunk 0 -> k kap pi_1
        // (chunk jh) and k kap pi_1 pi_2 (chunk 2+jh), sub-chunk 1 -> k kap pi_2 (chunk 4+jh).
        float ka0 = 1.f, ka1 = 1.f;
        if (whole) {
          // one sub-chunk: k / rho_r = (k kap_r) F_sc / gamma = (k kap_r) / (E_sc pi_sc),
          // rounded once, into CB block 0
          // (plain-gate build: the running product starts at fw and takes kap_r on the way)
          const float fw0 = __fdividef(1.f, E0 * pm0), fw1 = __fdividef(1.f, E1 * pm1);
          if (MODE == 0) {
            ka0 = fw0;
            ka1 = fw1;
          }
#pragma unroll
          for (int jh = 1; jh >= 0; --jh) {
            uint32_t xw[2][4];
#pragma unroll
            for (int u = 7; u >= 0; --u) {
              const int j = jh * 8 + u, r = sc * 16 + j;
              const uint32_t kv = (r < cv) ? *reinterpret_cast<const uint32_t*>(sm + OFF_QK + kmaj_elem(r, c0, 128)) : 0u;
              float k0, k1;
              if (MODE == 0) {
                k0 = bf_bits(kv & 0xFFFFu);
                k1 = bf_bits(kv >> 16);
                mul2(k0, k1, ka0, ka1);
                mul2(ka0, ka1, e0[j], e1[j]);
              } else {
                k0 = bf_bits(kv & 0xFFFFu) * (ka0 * fw0);
                k1 = bf_bits(kv >> 16) * (ka1 * fw1);
                ka0 *= e0[j];
                ka1 *= e1[j];
              }
              if (u & 1) {
                xw[0][u >> 1] = __float_as_uint(k0);  // odd token: the high half, packed below
                xw[1][u >> 1] = __float_as_uint(k1);
              } else {
                xw[0][u >> 1] = pack_bf16x2(k0, __uint_as_float(xw[0][u >> 1]));
                xw[1][u >> 1] = pack_bf16x2(k1, __uint_as_float(xw[1][u >> 1]));
              }
            }
            const uint32_t cj = sc * 2 + jh;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
              const int c = c2 ^ wsel;
              st_chunk(sm, OFF_CB + sw128_off(c0 + c, cj), c ? xw[1][0] : xw[0][0], c ? xw[1][1] : xw[0][1],
                       c ? xw[1][2] : xw[0][2], c ? xw[1][3] : xw[0][3]);
            }
          }
        } else {
#pragma unroll
        for (int jh = 1; jh >= 0; --jh) {
          float kk[2][8];
#pragma unroll
          for (int u = 7; u >= 0; --u) {
            const int j = jh * 8 + u, r = sc * 16 + j;
            const uint32_t kv = (r < cv) ? *reinterpret_cast<const uint32_t*>(sm + OFF_QK + kmaj_elem(r, c0, 128)) : 0u;
            kk[0][u] = bf_bits(kv & 0xFFFFu) * ka0;
            kk[1][u] = bf_bits(kv >> 16) * ka1;
            ka0 *= e0[j];
            ka1 *= e1[j];
          }
          const uint32_t cj = sc * 2 + jh;
          // both channels' 8 tokens as bf16 pairs: k kap, and k kap / pi rounded once from
          // fp32 (a second rounding on the diagonal blocks shows in the output); the
          // references scale the k kap pairs with one packed bf16 product each
          uint32_t xa[2][4], xd[2][4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            xa[0][u] = pack_bf16x2(kk[0][2 * u], kk[0][2 * u + 1]);
            xa[1][u] = pack_bf16x2(kk[1][2 * u], kk[1][2 * u + 1]);
            xd[0][u] = pack_bf16x2(kk[0][2 * u] * ip0, kk[0][2 * u + 1] * ip0);
            xd[1][u] = pack_bf16x2(kk[1][2 * u] * ip1, kk[1][2 * u + 1] * ip1);
          }
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            const int c = c2 ^ wsel;
            const int row = c0 + c;
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) w[u] = c ? xa[1][u] : xa[0][u];
            st_chunk(sm, OFF_CB + sw128_off(row, cj), w[0], w[1], w[2], w[3]);
            st_chunk(sm, OFF_CB + 16384 + sw128_off(row, cj), c ? xd[1][0] : xd[0][0], c ? xd[1][1] : xd[0][1],
                     c ? xd[1][2] : xd[0][2], c ? xd[1][3] : xd[0][3]);
            if (sc < 2) {
              const float p1 = c ? pi1[1] : pi0[1], p2 = c ? pi1[2] : pi0[2];
              const uint32_t ff = (sc == 0) ? pack_bf16x2(p1, p1) : pack_bf16x2(p2, p2);
              st_chunk(sm, OFF_CB + 32768 + sw128_off(row, (sc == 0 ? 0 : 4) + jh), bmul2(w[0], ff),
                       bmul2(w[1], ff), bmul2(w[2], ff), bmul2(w[3], ff));
              if (sc == 0) {
                const uint32_t f2 = pack_bf16x2(p1 * p2, p1 * p2);
                st_chunk(sm, OFF_CB + 32768 + sw128_off(row, 2 + jh), bmul2(w[0], f2), bmul2(w[1], f2),
                         bmul2(w[2], f2), bmul2(w[3], f2));
              }
            }
          }
        }
        }
        // pass B, ascending: rho (inclusive product from the sub-chunk start); q and k
        // rows of the MMA-AB operand in place, and KG, QG.  The recurrence group reads the
        // chunk before's KG and QG with its MMA-X (waited for in the prologue), and its inverse
        // scratch -- the AM buffer when that chunk took the four-sub-chunk form, the KG / QG
        // buffers otherwise -- up to its Tm (UW_DONE of that chunk).
        const float qs0 = p.scale * E0, qs1 = p.scale * E1;
        // the KG and QG tiles (the operand buffer AM of a whole chunk) and the v buffer are free
        // once MMA-X of the previous chunk ran
        if (gc > 0) wait_bar(p, s, B_M1B, (gc - 1) & 1);
        // tokens 8 jh .. 8 jh + 7 of channels c0, c0+1 of the staged k (row0 = 0) or q (row0 =
        // 64) rows, times m rho, packed as token pairs; rho is carried in r0, r1 (in the
        // plain-gate build they start at m and carry m rho, and m is not applied again)
        auto rows = [&](int row0, int jh, float& r0, float& r1, float m0, float m1, uint32_t (&aw)[2][4]) {
          uint32_t xw[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int r = sc * 16 + jh * 8 + u;
            xw[u] = (r < cv) ? *reinterpret_cast<const uint32_t*>(sm + OFF_QK + kmaj_elem(row0 + r, c0, 128)) : 0u;
          }
          float pa0 = 0.f, pa1 = 0.f;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int j = jh * 8 + u;
            float x0, x1;
            if (MODE == 0) {
              mul2(r0, r1, e0[j], e1[j]);
              x0 = bf_bits(xw[u] & 0xFFFFu);
              x1 = bf_bits(xw[u] >> 16);
              mul2(x0, x1, r0, r1);
            } else {
              r0 *= e0[j];
              r1 *= e1[j];
              x0 = bf_bits(xw[u] & 0xFFFFu) * (r0 * m0);
              x1 = bf_bits(xw[u] >> 16) * (r1 * m1);
            }
            if (u & 1) {
              aw[0][u >> 1] = pack_bf16x2(pa0, x0);
              aw[1][u >> 1] = pack_bf16x2(pa1, x1);
            } else {
              pa0 = x0;
              pa1 = x1;
            }
          }
        };
        // rows as the MN-major A operand of MMA-AB: k into AM, q into AM + 16 KB
        auto store_rows = [&](uint32_t base, uint32_t cj, int c, const uint32_t (&aw)[2][4]) {
          st_chunk(sm, base + sw128_off(c0 + c, cj), c ? aw[1][0] : aw[0][0], c ? aw[1][1] : aw[0][1],
                   c ? aw[1][2] : aw[0][2], c ? aw[1][3] : aw[0][3]);
        };
        if (whole) {
          // one sub-chunk: the operand rows are k rho E and scale q rho E themselves (one
          // rounding), which are KG and QG too
          if (gc > 0 && !prev_whole) wait_bar(p, s, B_UW_DONE, (gc - 1) & 1);
          float r0 = MODE == 0 ? qs0 : 1.f, r1 = MODE == 0 ? qs1 : 1.f;
#pragma unroll
          for (int jh = 0; jh < 2; ++jh) {
            uint32_t aw[2][4];
            rows(64, jh, r0, r1, qs0, qs1, aw);
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) store_rows(OFF_AM + 16384, sc * 2 + jh, c2 ^ wsel, aw);
          }
          r0 = MODE == 0 ? E0 : 1.f;
          r1 = MODE == 0 ? E1 : 1.f;
#pragma unroll
          for (int jh = 0; jh < 2; ++jh) {
            uint32_t aw[2][4];
            rows(0, jh, r0, r1, E0, E1, aw);
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) store_rows(OFF_AM, sc * 2 + jh, c2 ^ wsel, aw);
          }
        } else {
          if (gc > 0) wait_bar(p, s, B_UW_DONE, (gc - 1) & 1);
          float rk0 = 1.f, rk1 = 1.f, rq0 = 1.f, rq1 = 1.f;
#pragma unroll
          for (int jh = 0; jh < 2; ++jh) {
            uint32_t kaw[2][4], qaw[2][4];
            rows(0, jh, rk0, rk1, 1.f, 1.f, kaw);
            rows(64, jh, rq0, rq1, 1.f, 1.f, qaw);
            const uint32_t cj = sc * 2 + jh;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
              const int c = c2 ^ wsel;
              const int row = c0 + c;
              store_rows(OFF_AM, cj, c, kaw);
              store_rows(OFF_AM + 16384, cj, c, qaw);
              // KG = (k rho) E and QG = (q rho) scale E as packed products of the pairs above
              const uint32_t eg = c ? pack_bf16x2(E1, E1) : pack_bf16x2(E0, E0);
              st_chunk(sm, OFF_KG + sw128_off(row, cj), bmul2(c ? kaw[1][0] : kaw[0][0], eg),
                       bmul2(c ? kaw[1][1] : kaw[0][1], eg), bmul2(c ? kaw[1][2] : kaw[0][2], eg),
                       bmul2(c ? kaw[1][3] : kaw[0][3], eg));
              const uint32_t eq = c ? pack_bf16x2(qs1, qs1) : pack_bf16x2(qs0, qs0);
              st_chunk(sm, OFF_QG + sw128_off(row, cj), bmul2(c ? qaw[1][0] : qaw[0][0], eq),
                       bmul2(c ? qaw[1][1] : qaw[0][1], eq), bmul2(c ? qaw[1][2] : qaw[0][2], eq),
                       bmul2(c ? qaw[1][3] : qaw[0][3], eq));
            }
          }
        }
      }
      if (t < kC) s->beta[gc & 1][t] = bt;
      fence_async_smem();
      named_bar(BAR_IG, kIG);
      if (t == 0) {
        tc_fence_after();
        // four sub-chunks: CB blocks 0-2 (the last 16 columns unused); one: block 0
        const uint32_t idesc = whole ? idesc_bf16(128, 64, 1, 1) : idesc_bf16(128, 176, 1, 1);
#pragma unroll 1
        for (int st = 0; st < 8; ++st) {
          const uint64_t a = sdesc_sw128(sbase + OFF_AM + st * 2048, 16384, 1024);
          const uint64_t b = sdesc_sw128(sbase + OFF_CB + st * 2048, 16384, 1024);
          mma_bf16(tbase + TM_AB, a, b, idesc, st > 0 ? 1u : 0u);
        }
        mma_commit(&s->bar[B_AB_DONE]);
      } else if (t == 128) {
        // meanwhile, on warp 4: the chunk after this one (read by the A group after a
        // later barrier, by the whole group after the one before Tm, by the recurrence
        // group after REC_READY); its q/k, and its gate into L2
        NextChunk nx{};
        nx.have = ld.next_chunk(s, k, lc, nx.kh, nx.h, nx.t0, nx.cv);
        ld.st->nx[gc & 1] = nx;
        if (nx.have) {
          ld.load_qk(p, sm, s, nx.kh, nx.t0);  // q/k buffer free since pass B
          ld.prefetch_l2(p, nx.h, nx.t0);
        }
      } else if (t == 160) {
        // and on warp 5: v of this chunk, which the recurrence group turns into -V^T in TMEM
        // before its MMA-X (the v buffer is free once MMA-X of the previous chunk ran); the
        // identity pass of a cut tail has zero values, so its phase completes bare
        if (info.kind == KIND_TAIL_ID) {
          if (!aborted(s)) {
            mbar_arrive(&s->bar[B_V_FULL]);
            atomicAdd(&ld.st->n_v, 1u);
          }
        } else {
          ld.load_v(p, sm, s, h, (int)t0);
        }
      }
      __syncwarp();
      // a whole chunk followed by one in the same item has that chunk's gate in flight since the
      // vote: the A group, idle during MMA-AB, turns its sub-chunks 0-1 into e (warps 0, 1, 4, 5
      // -> units 0-3), warps 2-5 the rest while warps 0-1 invert
      const bool e_split = plain_gate && whole && lc + 1 < info.nchunks;
      if (quad < 2 && e_split) {
        const int ncv = (int)min((int64_t)kC, info.eos - (t0 + kC));
        wait_bar(p, s, B_G_FULL, (gc + 1) & 1);
        gate_exp_inplace(sm, s->unsafe[(gc + 1) & 1], ncv, (warp & 1) | (hx << 1), 4, lane, 0, 2);
      }
      if (quad >= 2) {
        // KR = (k kap) F_s for sub-chunks sc-1 and sc of this thread's channel pair
        // (F_s = product of pi after s), by the B group while the tensor core runs MMA-AB;
        // one sub-chunk: KR = (k / rho) gamma
        if (gc > 0) wait_bar(p, s, B_M3, (gc - 1) & 1);
#pragma unroll 1
        for (int s2 = 0; s2 < 2; ++s2) {
          const int sk = sc - 1 + s2;
          const float fs0 = whole ? gm0 : (sk < 1 ? pi0[1] : 1.f) * (sk < 2 ? pi0[2] : 1.f) * (sk < 3 ? pi0[3] : 1.f);
          const float fs1 = whole ? gm1 : (sk < 1 ? pi1[1] : 1.f) * (sk < 2 ? pi1[2] : 1.f) * (sk < 3 ? pi1[3] : 1.f);
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            const int c = c2 ^ wsel;
            const float f = c ? fs1 : fs0;
#pragma unroll 1
            for (int jj = 0; jj < 2; ++jj) {
              const int j = sk * 2 + jj;
              const uint4 src = *reinterpret_cast<const uint4*>(sm + OFF_CB + sw128_off(c0 + c, j));
              const uint32_t in[4] = {src.x, src.y, src.z, src.w};
              uint32_t w[4];
#pragma unroll
              for (int u = 0; u < 4; ++u)
                w[u] = pack_bf16x2(bf_bits(in[u] & 0xFFFFu) * f, bf_bits(in[u] >> 16) * f);
              st_chunk(sm, OFF_KR + sw128_off(c0 + c, j), w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
      // ------------------------------------------------------------- A / B rows
      wait_bar(p, s, B_AB_DONE, gc & 1);
      // a whole chunk's inverse scratch is the KG / QG buffers, which hold the chunk before's
      // scratch when that chunk was whole too: read by its recurrence up to Tm
      if (whole && prev_whole) wait_bar(p, s, B_UW_DONE, (gc - 1) & 1);
      tc_fence_after();

      __syncwarp();
      uint32_t any_unsafe = 0;
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2)
        any_unsafe |= s->unsafe[gc & 1][q2][0][0] | s->unsafe[gc & 1][q2][0][1] | s->unsafe[gc & 1][q2][1][0] |
                      s->unsafe[gc & 1][q2][1][1];
      {
        const int r = L & 63, a = r >> 4;
        const bool isB = L >= 64;
        const int a0 = (L & 32) ? 2 : 0;  // sub-chunks a0, a0+1 live in this warp
        float x[32];
        if (whole) {  // one sub-chunk: token column i of every row is TMEM column i
#pragma unroll
          for (int bb = 0; bb < 2; ++bb) {
            float v0[16];
            tmem_ld16(taddr_q + TM_AB + 16 * (hx * 2 + bb), v0);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) x[bb * 16 + j] = v0[j];
          }
        } else {
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const int b = hx * 2 + bb;
          auto colof = [](int aa, int b_) -> int {
            if (b_ == aa) return 64 + 16 * aa;
            if (b_ == aa - 1) return 16 * b_;
            if (b_ == aa - 2) return aa == 2 ? 128 : 160;
            if (b_ == aa - 3) return 144;
            return -1;
          };
          const int cc0 = (b <= a0) ? colof(a0, b) : -1;
          const int cc1 = (b <= a0 + 1) ? colof(a0 + 1, b) : -1;
          float v0[16], v1[16];
          if (cc0 >= 0) tmem_ld16(taddr_q + TM_AB + cc0, v0);
          if (cc1 >= 0) tmem_ld16(taddr_q + TM_AB + cc1, v1);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float val = 0.f;
            if (a == a0 && cc0 >= 0) val = v0[j];
            if (a == a0 + 1 && cc1 >= 0) val = v1[j];
            x[bb * 16 + j] = val;
          }
        }
        }
        tc_fence_before();
        if (any_unsafe == 0u) {
          // fast path: mask and scale straight from TMEM
          if (!isB) {
            const float br = s->beta[gc & 1][r];
#pragma unroll
            for (int jc = 0; jc < 8; ++jc) {
              float4 w4;
              const int i = hx * 32 + jc * 4;
              if ((i >> 4) > a) continue;  // blocks above the diagonal are never read
              w4.x = (i + 0 < r) ? br * x[jc * 4 + 0] : 0.f;
              w4.y = (i + 1 < r) ? br * x[jc * 4 + 1] : 0.f;
              w4.z = (i + 2 < r) ? br * x[jc * 4 + 2] : 0.f;
              w4.w = (i + 3 < r) ? br * x[jc * 4 + 3] : 0.f;
              *reinterpret_cast<float4*>(As + sidx(r, i)) = w4;
            }
          } else {
            if (gc > 0) wait_bar(p, s, B_M3, (gc - 1) & 1);  // BB free
            const float bsc = whole ? 1.f : p.scale;  // one sub-chunk: the q rows carry it
#pragma unroll
            for (int jc = 0; jc < 4; ++jc) {
              uint32_t w[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int i0 = hx * 32 + jc * 8 + u * 2;
                w[u] = pack_bf16x2((i0 <= r) ? bsc * x[jc * 8 + u * 2] : 0.f,
                                   (i0 + 1 <= r) ? bsc * x[jc * 8 + u * 2 + 1] : 0.f);
              }
              st_chunk(sm, OFF_BB + sw128_off(r, hx * 4 + jc), w[0], w[1], w[2], w[3]);
            }
          }
        } else {
          float* row = isB ? Xs : As;
#pragma unroll
          for (int jc = 0; jc < 8; ++jc)
            *reinterpret_cast<float4*>(row + sidx(r, hx * 32 + jc * 4)) =
                make_float4(x[jc * 4], x[jc * 4 + 1], x[jc * 4 + 2], x[jc * 4 + 3]);
        }
      }
      // TMEM lanes 0-63 (A rows) belong to warps 0, 1, 4, 5 (the "A group"), lanes
      // 64-127 (B rows) to warps 2, 3, 6, 7; on the fast path the A group goes on to the
      // inverse while the B group writes KR.
      const bool agrp = quad < 2;
      if (any_unsafe == 0u) {
        if (agrp) named_bar(BAR_A, 128);
      } else {
        named_bar(BAR_IG, kIG);
        // exact pairwise terms of the diagonal sub-chunk blocks on "unsafe" channels
        if (hx == 0)
          unsafe_diag_terms(p, s->unsafe[gc & 1], As, Xs, s->inv_nrm,
                            L, t0, cv, kh, h);
        named_bar(BAR_IG, kIG);
        // A: mask + beta_r (in place, fp32); B: mask + scale -> bf16 -> BB
        {
          const int r = L & 63;
          if (L < 64) {
            const float br = s->beta[gc & 1][r];
#pragma unroll
            for (int jc = 0; jc < 8; ++jc) {
              const int i = hx * 32 + jc * 4;
              float4 w4 = *reinterpret_cast<const float4*>(As + sidx(r, i));
              w4.x = (i + 0 < r) ? br * w4.x : 0.f;
              w4.y = (i + 1 < r) ? br * w4.y : 0.f;
              w4.z = (i + 2 < r) ? br * w4.z : 0.f;
              w4.w = (i + 3 < r) ? br * w4.w : 0.f;
              *reinterpret_cast<float4*>(As + sidx(r, i)) = w4;
            }
          } else {
            if (gc > 0) wait_bar(p, s, B_M3, (gc - 1) & 1);  // BB free
#pragma unroll
            for (int jc = 0; jc < 4; ++jc) {
              const int i = hx * 32 + jc * 8;
              const float4 lo = *reinterpret_cast<const float4*>(Xs + sidx(r, i));
              const float4 hi = *reinterpret_cast<const float4*>(Xs + sidx(r, i + 4));
              const float vv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
              uint32_t w[4];
#pragma unroll
              for (int u = 0; u < 4; ++u)
                w[u] = pack_bf16x2((i + 2 * u <= r) ? p.scale * vv[2 * u] : 0.f,
                                   (i + 2 * u + 1 <= r) ? p.scale * vv[2 * u + 1] : 0.f);
              st_chunk(sm, OFF_BB + sw128_off(r, hx * 4 + jc), w[0], w[1], w[2], w[3]);
            }
          }
        }
        named_bar(BAR_IG, kIG);
      }
      // ------------------------------------------------------------- inverse
      // X = (I + A)^-1: the 16x16 diagonal blocks here, by forward substitution on warps 0-1
      // (one column per lane, two blocks per warp); the recurrence group, idle by then, forms
      // the rest from them (inverse_merges) and Tm.
      // While warps 0-1 invert the diagonal blocks, warps 2-5 (one per SM sub-partition, so
      // that the exponentials spread over all four multi-function units) turn the staged gate
      // of the next chunk of this item into e, its products and masks (sub-chunks 2-3 when the
      // A group did 0-1 during MMA-AB), after the B group's rows (barrier of warps 2-7).
      // Warp 4 first issues that gate load if the vote did not (CB 1-2 are free since MMA-AB).
      if (t == 128 && ld.st->nx[gc & 1].have && ld.st->n_g == gc + 1) {
        const NextChunk& nx = ld.st->nx[gc & 1];
        ld.load_g(p, sm, s, nx.h, nx.t0);
      }
      if (warp < 2) {
        // lane = column j of diagonal block o (two blocks per warp).  Its 8x8 diagonal
        // sub-blocks are inverted by forward substitution side by side (columns 0-7
        // take rows 0-7, columns 8-15 rows 8-15; rows of A read as broadcast float4),
        // then columns 0-7 get rows 8-15 as -X22 (A21 x), A21 the lower-left 8x8.
        const int o = (warp * 2 + (lane >> 4)) * 16, j = lane & 15;
        const int hb = j & 8;
        float xv[8];
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) xv[rr] = (hb + rr == j) ? 1.f : 0.f;
#pragma unroll
        for (int rr = 1; rr < 8; ++rr) {
          const float4 a0 = *reinterpret_cast<const float4*>(As + sidx(o + hb + rr, o + hb));
          const float4 a1 = *reinterpret_cast<const float4*>(As + sidx(o + hb + rr, o + hb + 4));
          const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          float acc[2] = {0.f, 0.f};
#pragma unroll
          for (int i = 0; i < rr; ++i) acc[i & 1] = fmaf(av[i], xv[i], acc[i & 1]);
          if (hb + rr > j) xv[rr] = -(acc[0] + acc[1]);
        }
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) Xs[sidx(o + hb + rr, o + j)] = xv[rr];
        // upper-right 8x8 is zero: one float4 per lane (row j/2, columns 8 + 4 (j&1) ..)
        *reinterpret_cast<float4*>(Xs + sidx(o + (j >> 1), o + 8 + 4 * (j & 1))) =
            make_float4(0.f, 0.f, 0.f, 0.f);
        __syncwarp();
        if (!hb) {
          float y[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 a0 = *reinterpret_cast<const float4*>(As + sidx(o + 8 + i, o));
            const float4 a1 = *reinterpret_cast<const float4*>(As + sidx(o + 8 + i, o + 4));
            y[i] = fmaf(a0.x, xv[0], fmaf(a0.y, xv[1], fmaf(a0.z, xv[2], a0.w * xv[3]))) +
                   fmaf(a1.x, xv[4], fmaf(a1.y, xv[5], fmaf(a1.z, xv[6], a1.w * xv[7])));
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 x0 = *reinterpret_cast<const float4*>(Xs + sidx(o + 8 + i, o + 8));
            const float4 x1 = *reinterpret_cast<const float4*>(Xs + sidx(o + 8 + i, o + 12));
            const float xr[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            float acc[2] = {0.f, 0.f};
#pragma unroll
            for (int m = 0; m <= i; ++m) acc[m & 1] = fmaf(xr[m], y[m], acc[m & 1]);
            Xs[sidx(o + 8 + i, o + j)] = -(acc[0] + acc[1]);
          }
        }
      } else if (plain_gate && lc + 1 < info.nchunks) {
        // (the lookahead within an item always succeeds, so the gate load was issued)
        named_bar(BAR_B, 192);
        if (warp < 6) {
          const int ncv = (int)min((int64_t)kC, info.eos - (t0 + kC));
          const int wgb = (warp ^ 4) & 3;  // warps 4, 5, 2, 3 -> 0-3
          wait_bar(p, s, B_G_FULL, (gc + 1) & 1);
          gate_exp_inplace(sm, s->unsafe[(gc + 1) & 1], ncv, wgb, 4, lane, e_split ? 2 : 0, 4);
        }
      }
      // B rows (BB) visible to the tensor core; the diagonal blocks of X complete
      fence_async_smem();
      named_bar(BAR_IG, kIG);
      if (t < kC && ld.st->nx[gc & 1].have) {
        const NextChunk& nx = ld.st->nx[gc & 1];
        if (t < nx.cv && KDA_CHECK((int64_t)nx.t0 + t < p.T))
          bt_next = p.beta[(size_t)(nx.t0 + t) * p.Hv + nx.h];
        bt_ok = true;
      }
      // hand the chunk to the recurrence group: it issues MMA-X, completes X and Tm, and runs
      // MMA-U and MMA-3
      if (t == 0) mbar_arrive(&s->bar[B_REC_READY]);
      __syncwarp();
    }
    if (stop) break;
  }
  // drain: this group's MMAs, before the CTA releases TMEM (loads drain at the end)
  named_bar(BAR_IG, kIG);
  if (warp == 0) {
    if (lane == 0) mma_commit(&s->bar[B_DRAIN_IG]);
    __syncwarp();
    mbar_wait(&s->bar[B_DRAIN_IG], 0);  // the full limit, aborted or not
  }
}

// 32 consecutive key channels of row v of a transposed ([V][K]) state, as fp32, with
// 16-byte loads and stores (each thread owns its row).
__device__ __forceinline__ void row32_load(const float* p, float* r) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 x = reinterpret_cast<const float4*>(p)[i];
    r[4 * i] = x.x; r[4 * i + 1] = x.y; r[4 * i + 2] = x.z; r[4 * i + 3] = x.w;
  }
}
__device__ __forceinline__ void row32_load(const __nv_bfloat16* p, float* r) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 x = reinterpret_cast<const uint4*>(p)[i];
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      r[8 * i + 2 * j] = bf_bits(w[j] & 0xFFFFu);
      r[8 * i + 2 * j + 1] = bf_bits(w[j] >> 16);
    }
  }
}
__device__ __forceinline__ void row32_store(float* p, const float* r) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
    reinterpret_cast<float4*>(p)[i] = make_float4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
}
__device__ __forceinline__ void row32_store(__nv_bfloat16* p, const float* r) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
    reinterpret_cast<uint4*>(p)[i] =
        make_uint4(pack_bf16x2(r[8 * i], r[8 * i + 1]), pack_bf16x2(r[8 * i + 2], r[8 * i + 3]),
                   pack_bf16x2(r[8 * i + 4], r[8 * i + 5]), pack_bf16x2(r[8 * i + 6], r[8 * i + 7]));
}

// ======================================================================================
// Recurrence group (warps 8-11): state update and output, chunk by chunk.
// ======================================================================================
template <typename ST, int MODE>
__device__ void run_recurrence(const TcParams& p, uint8_t* sm, Small* s, uint32_t tbase) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int v = quad * 32 + lane;  // TMEM lane = value channel
  const int rt = threadIdx.x - kIG;
  const bool leader_warp = (warp == kIG / 32);
  const uint32_t taddr_q = tbase + ((uint32_t)(quad * 32) << 16);
  const uint32_t sbase = smem_u32(sm);
  Loader ld{&s->ld};
  uint32_t gc = 0;
  if (MODE != 0) {
    // the -I tile of V-in (B operand, K-major, 128-byte swizzle): row n holds -1 at column n;
    // visible to the tensor core after the first barrier of the item loop
    for (int c = rt; c < 64 * 8; c += kRG) {
      const int n = c >> 3, j = c & 7;
      const uint32_t m1 = (n >> 3) == j ? (0xBF80u << (16 * (n & 1))) : 0u;  // bf16 -1 at column n
      const int w = (n & 7) >> 1;
      st_chunk(sm, OFF_NI + sw128_off(n, j), w == 0 ? m1 : 0u, w == 1 ? m1 : 0u, w == 2 ? m1 : 0u,
               w == 3 ? m1 : 0u);
    }
    fence_async_smem();
  }

  for (int k = 0;; ++k) {
    const ItemInfo info = next_item(p, s, k, rt == 0, BAR_RG, kRG);
    if (info.done) break;
    const int h = info.h;
    const ST* src = nullptr;
    ST* dst = nullptr;
    float* dst32 = nullptr;  // final state of a cut sequence's part, into the split scratch
    const bool ident = info.kind == KIND_TAIL_ID;  // starts from I, zero values, o -> y
    const size_t hoff = (size_t)h * kK * kV;
    if (info.kind == KIND_WHOLE || info.kind == KIND_HEAD) {
      if (info.slot >= 0) {
        src = static_cast<const ST*>(p.state_in) + info.slot * p.slot_stride + hoff;
        dst = static_cast<ST*>(p.state_out) + info.slot * p.slot_stride + hoff;
      } else {
        if (p.state_in) src = static_cast<const ST*>(p.state_in) + ((size_t)info.n * p.Hv) * kK * kV + hoff;
        if (p.state_out) dst = static_cast<ST*>(p.state_out) + ((size_t)info.n * p.Hv) * kK * kV + hoff;
      }
    }
    if (info.kind != KIND_WHOLE) {
      const size_t so = ((size_t)info.split * p.Hv) * kK * kV + hoff;
      dst32 = (info.kind == KIND_HEAD ? p.sp : info.kind == KIND_TAIL ? p.sl : p.mm) + so;
      dst = nullptr;
    }
    if (info.nchunks == 0) {  // empty sequence: the final state is the initial one
      if (rt == 32) ld.push_one(p, s);  // claim of the next item (see the chunk loop)
      if (dst && dst != src)
        for (int c = 0; c < kK; ++c) dst[(size_t)c * kV + v] = src ? src[(size_t)c * kV + v] : ST(0.f);
      continue;
    }
    // ---- initial state: S^T row v -> TMEM as bf16 pairs (MMA-X operand) and as fp32
    // pre-decayed by gamma of chunk 0
    wait_bar(p, s, B_GAMMA0 + (gc & 1), (gc >> 1) & 1);
#pragma unroll 1
    for (int kq = 0; kq < 4; ++kq) {
      float sv[32], pw[16];
      if (src && p.state_vk) {
        row32_load(src + (size_t)v * kK + kq * 32, sv);  // row v: S[k][v] for 32 k
      } else {
#pragma unroll
        for (int u = 0; u < 32; ++u)
          sv[u] = src ? to_f32(src[(size_t)(kq * 32 + u) * kV + v]) : (ident && kq * 32 + u == v ? 1.f : 0.f);
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) pw[u] = __uint_as_float(pack_bf16x2(sv[2 * u], sv[2 * u + 1]));
      tmem_st16(taddr_q + TM_SB + kq * 16, pw);
#pragma unroll
      for (int u = 0; u < 32; ++u) sv[u] *= s->gamma[gc & 1][kq * 32 + u];
      tmem_st16(taddr_q + TM_S + kq * 32, sv);
      tmem_st16(taddr_q + TM_S + kq * 32 + 16, sv + 16);
    }
    tmem_st_wait();
    tc_fence_before();
    named_bar(BAR_RG, kRG);

    bool stop = false;
    for (int lc = 0; lc < info.nchunks; ++lc, ++gc) {
      // the output staging tile (the WB buffer) is read by the TMA store of the chunk
      // before, if any, before this chunk writes its own there
      if (rt == 0) bulk_wait_read();
      if (named_bar_any(BAR_RG, kRG, aborted(s))) { stop = true; break; }
      const int64_t t0 = info.bos + (int64_t)lc * kC;
      const int cv = (int)min((int64_t)kC, info.eos - t0);
      const bool last = (lc + 1 == info.nchunks);
      // claim the next item late, about two chunks before this one ends, so that a CTA
      // takes new work only when it is about to run out (dynamic longest-first
      // scheduling); the claim's global round trips overlap this group's slack
      if (rt == 32 && lc == (info.nchunks > 3 ? info.nchunks - 3 : 0)) ld.push_one(p, s);
      // ---- V-in, in the group's slack before the hand-over: -V^T into the U columns (lane =
      // value channel v, column = token; zero values in the identity pass) and zeros into O,
      // which MMA-X accumulates onto.  The plain-gate build reads v with per-thread loads; the
      // other builds form -V^T as V^T (-I), four MMAs with the staged v tile as the A operand
      // (MN-major: value channels contiguous, the two 64-value halves 8 KB apart), issued by the
      // thread that issues MMA-X after them (on their workloads the group has more slack).
      if (MODE == 0) {
        wait_bar(p, s, B_V_FULL, gc & 1);
        const uint8_t* vb = sm + OFF_VB + (v >> 6) * 8192 + (v & 7) * 2;
        const uint32_t vc = (uint32_t)(v & 63) >> 3;
        float z[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) z[u] = 0.f;
#pragma unroll 1
        for (int cq = 0; cq < 4; ++cq) {
          float nv[16];
#pragma unroll
          for (int u = 0; u < 16; ++u)
            nv[u] = ident ? 0.f : -bf_bits(*reinterpret_cast<const uint16_t*>(vb + sw128_off(cq * 16 + u, vc)));
          tmem_st16(taddr_q + TM_U + cq * 16, nv);
          tmem_st16(taddr_q + TM_O + cq * 16, z);
        }
        tmem_st_wait();
      } else {
        float z[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) z[u] = 0.f;
#pragma unroll 1
        for (int cq = 0; cq < 4; ++cq) {
          tmem_st16(taddr_q + TM_O + cq * 16, z);
          if (ident) tmem_st16(taddr_q + TM_U + cq * 16, z);
        }
        tmem_st_wait();
        if (rt == 64) {
          wait_bar(p, s, B_V_FULL, gc & 1);
          if (!ident) {
            tc_fence_after();
            const uint32_t idv = idesc_bf16(128, 64, 1, 0);
#pragma unroll 1
            for (int st = 0; st < 4; ++st)
              mma_bf16(tbase + TM_U, sdesc_sw128(sbase + OFF_VB + st * 2048, 8192, 1024),
                       sdesc_sw128(sbase + OFF_NI + st * 32, 16, 1024), idv, st > 0 ? 1u : 0u);
          }
        }
      }
      tc_fence_before();
      // ---- R0: the hand-over.  MMA-X first (it frees KG, QG, v and gamma for the next
      // chunk's prologue), then X = (I + A)^-1 and Tm from the diagonal blocks the intra group
      // inverted, then Y^T -> TMEM (bf16 pairs) and U^T = Y^T Tm^T
      wait_bar(p, s, B_REC_READY, gc & 1);
      // a chunk run as one sub-chunk keeps KG and QG in the MMA-AB operand buffer, and the
      // inverse scratch in the KG / QG buffers
      const bool whole = s->whole[gc & 1] != 0u;
      named_bar(BAR_RG, kRG);  // every lane's V-in is in TMEM
      // MMA-X: [U | O] (N = 128) += S^T [KG | QG]^T, B = the KG and QG tiles as two 64-token
      // blocks LBO apart.  Issued by warp 10, idle during the first step of the merges (an MMA
      // issue holds its thread for about as long as the tensor core takes to run it).
      if (rt == 64) {
        tc_fence_after();
        const uint32_t off_b = whole ? OFF_AM : OFF_KG;
        const uint32_t lbo = whole ? 16384u : OFF_QG - OFF_KG;
        const uint32_t idx = idesc_bf16(128, 128, 0, 1);
#pragma unroll 1
        for (int st = 0; st < 8; ++st)
          mma_bf16_ta(tbase + TM_U, tbase + TM_SB + st * 8, sdesc_sw128(sbase + off_b + st * 2048, lbo, 1024),
                      idx, 1u);
        mma_commit(&s->bar[B_M1B]);
      }
      {
        float* As = reinterpret_cast<float*>(sm + (whole ? OFF_KG : OFF_AS));
        float* Xs = reinterpret_cast<float*>(sm + (whole ? OFF_QG : OFF_XS));
        inverse_merges(As, Xs, warp - kIG / 32, lane, BAR_RG);
        form_tm(sm, Xs, s->beta[gc & 1], rt);
      }
      // ---- Y^T = -(the U columns) -> TMEM as bf16 pairs (columns 0-31 of the S^T pairs, free
      // once MMA-X ran): the A operand of MMA-U
      wait_bar(p, s, B_M1B, gc & 1);
      tc_fence_after();
#pragma unroll 1
      for (int cq = 0; cq < 2; ++cq) {  // tokens 32 cq ..
        float yv[32], pw[16];
        tmem_ld16(taddr_q + TM_U + cq * 32, yv);
        tmem_ld16(taddr_q + TM_U + cq * 32 + 16, yv + 16);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 16; ++u) pw[u] = __uint_as_float(pack_bf16x2(-yv[2 * u], -yv[2 * u + 1]));
        tmem_st16(taddr_q + TM_SB + cq * 16, pw);
      }
      tmem_st_wait();
      tc_fence_before();
      fence_async_smem();
      named_bar(BAR_RG, kRG);  // Tm in shared memory, Y^T in TMEM, the U columns read out
      // ---- MMA-U: U^T = Y^T Tm^T (onto the U columns)
      if (rt == 0) {
        tc_fence_after();
        const uint32_t idu = idesc_bf16(128, 64, 0, 0);
#pragma unroll 1
        for (int st = 0; st < 4; ++st)
          mma_bf16_ta(tbase + TM_U, tbase + TM_SB + st * 8, sdesc_sw128(sbase + OFF_TM + st * 32, 16, 1024), idu,
                      st > 0 ? 1u : 0u);
        mma_commit(&s->bar[B_UW_DONE]);
      }
      __syncwarp();
      // ---- E1: U^T row v -> TMEM as bf16 pairs (columns 32-63 of the S^T pairs): the A operand
      // of MMA-3
      wait_bar(p, s, B_UW_DONE, gc & 1);
      tc_fence_after();
#pragma unroll 1
      for (int cq = 0; cq < 2; ++cq) {
        float uv[32], pw[16];
        tmem_ld16(taddr_q + TM_U + cq * 32, uv);
        tmem_ld16(taddr_q + TM_U + cq * 32 + 16, uv + 16);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 16; ++u) pw[u] = __uint_as_float(pack_bf16x2(uv[2 * u], uv[2 * u + 1]));
        tmem_st16(taddr_q + TM_SB + 32 + cq * 16, pw);
      }
      tmem_st_wait();
      tc_fence_before();
      named_bar(BAR_RG, kRG);
      // ---- MMA-3: [O | S] (N = 192) += U^T [B | KR]^T, B = the BB rows (64 tokens) and the
      // KR rows (128 channels) right after them, K-major.  (MMA-X, which wrote O, completed
      // before Y^T was read out.)
      if (rt == 0) {
        tc_fence_after();
        const uint32_t id3 = idesc_bf16(128, 192, 0, 0);
#pragma unroll 1
        for (int st = 0; st < 4; ++st)
          mma_bf16_ta(tbase + TM_O, tbase + TM_SB + 32 + st * 8, sdesc_sw128(sbase + OFF_BB + st * 32, 16, 1024),
                      id3, 1u);
        mma_commit(&s->bar[B_M3]);
      }
      __syncwarp();
      // ---- E2: S -> TMEM bf16 pairs for the next chunk's MMA-X, and back as fp32 pre-decayed
      // by that chunk's gamma (its MMA-3 accumulates onto Diag(gamma) S); or the final state
      // store
      wait_bar(p, s, B_M3, gc & 1);
      if (!last) wait_bar(p, s, B_GAMMA0 + ((gc + 1) & 1), ((gc + 1) >> 1) & 1);
      tc_fence_after();
      if (!last) {
        const float* gn = s->gamma[(gc + 1) & 1];
#pragma unroll 1
        for (int kq = 0; kq < 4; ++kq) {
          float sv[32], pw[16];
          tmem_ld16(taddr_q + TM_S + kq * 32, sv);
          tmem_ld16(taddr_q + TM_S + kq * 32 + 16, sv + 16);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 16; ++u) pw[u] = __uint_as_float(pack_bf16x2(sv[2 * u], sv[2 * u + 1]));
          tmem_st16(taddr_q + TM_SB + kq * 16, pw);
#pragma unroll
          for (int u4 = 0; u4 < 8; ++u4) {
            const float4 g4 = *reinterpret_cast<const float4*>(gn + kq * 32 + u4 * 4);
            mul2(sv[u4 * 4 + 0], sv[u4 * 4 + 1], g4.x, g4.y);
            mul2(sv[u4 * 4 + 2], sv[u4 * 4 + 3], g4.z, g4.w);
          }
          tmem_st16(taddr_q + TM_S + kq * 32, sv);
          tmem_st16(taddr_q + TM_S + kq * 32 + 16, sv + 16);
        }
      } else if (dst32 || dst) {  // the final state (a cut part's into the split scratch)
#pragma unroll 1
        for (int kq = 0; kq < 4; ++kq) {
          float sv[32];
          tmem_ld16(taddr_q + TM_S + kq * 32, sv);
          tmem_ld16(taddr_q + TM_S + kq * 32 + 16, sv + 16);
          tmem_ld_wait();
          if (dst32) {
#pragma unroll
            for (int u = 0; u < 32; ++u) dst32[(size_t)(kq * 32 + u) * kV + v] = sv[u];
          } else if (p.state_vk) {
            row32_store(dst + (size_t)v * kK + kq * 32, sv);
          } else {
#pragma unroll
            for (int u = 0; u < 32; ++u) dst[(size_t)(kq * 32 + u) * kV + v] = from_f32<ST>(sv[u]);
          }
        }
      }
      tmem_st_wait();
      // ---- output of this chunk, complete once MMA-3 ran: a full chunk through a shared-memory
      // tile and one TMA store; a partial chunk or the identity pass by per-thread stores
      if (!ident && cv == kC) {
        // a full chunk of o: rows of the [64 tokens][128 values] tile in the WB buffer (free: the
        // chunk before's store has read it), each thread writing its value channel, then one TMA
        // store
        __nv_bfloat16* os = reinterpret_cast<__nv_bfloat16*>(sm + OFF_WB);
#pragma unroll 1
        for (int cq = 0; cq < 4; ++cq) {
          float ov[16];
          tmem_ld16(taddr_q + TM_O + cq * 16, ov);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 16; ++u) os[(cq * 16 + u) * kV + v] = __float2bfloat16_rn(ov[u]);
        }
        fence_async_smem();
        named_bar(BAR_RG, kRG);
        if (rt == 0 && KDA_CHECK(t0 + kC <= p.T)) {
          tma_store_3d(&p.tm_o, os, 0, h, (int)t0);
          bulk_commit();
        }
      } else {
        // a partial chunk (its tile would cover the next sequence's rows) or the identity
        // pass (y into the split scratch instead of o): each thread stores its column
        __nv_bfloat16* od = ident ? p.y + ((size_t)(t0 - info.bos + info.ybase) * p.Hv + h) * kV + v
                                  : p.o + ((size_t)t0 * p.Hv + h) * kV + v;
        const size_t rs = (size_t)p.Hv * kV;
#pragma unroll 1
        for (int cq = 0; cq < 4; ++cq) {
          float ov[16];
          tmem_ld16(taddr_q + TM_O + cq * 16, ov);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 16; ++u)
            if (cq * 16 + u < cv &&
                KDA_CHECK(ident ? t0 - info.bos + info.ybase + cq * 16 + u < p.ytok_cap
                                : t0 + cq * 16 + u < p.T))
              od[(size_t)(cq * 16 + u) * rs] = __float2bfloat16_rn(ov[u]);
        }
      }
      tc_fence_before();
    }
    if (stop) break;
  }
  if (rt == 0) bulk_wait_all();  // the output stores this thread issued have completed
  named_bar(BAR_RG, kRG);
  // the two threads that issue this group's MMAs (rt 0, 64) each commit once
  if (rt == 0 || rt == 64) mma_commit(&s->bar[B_DRAIN_RG]);
  if (leader_warp) mbar_wait(&s->bar[B_DRAIN_RG], 0);  // the full limit, aborted or not
}

template <typename ST, int MODE>
__global__ void __launch_bounds__(kThreads, 1) kda_prefill_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, formed as an offset into the shared array (not through an
  // integer round trip) so that the compiler keeps every derived pointer in the shared
  // window and emits shared loads and stores rather than generic ones
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad > kAlignSlack) {  // uniform: no barrier, load or TMEM has been touched yet
    if (threadIdx.x == 0) raise_status(p.status, KDA_DEVICE_PIPE_TIMEOUT);
    return;
  }
  uint8_t* sm = smem_raw + pad;
  Small* s = reinterpret_cast<Small*>(sm + OFF_SMALL);
  const int warp = threadIdx.x >> 5;
  // the combine kernel after this one may be scheduled as SMs free up (it waits for this
  // grid before reading anything)
  grid_dep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int b = 0; b < B_COUNT; ++b) mbar_init(&s->bar[b], b == B_DRAIN_RG ? 2 : 1);
    for (int r = 0; r < kRing; ++r) mbar_init(&s->bar[B_ITEM_EMPTY + r], 2);
    s->abort = 0;
    s->ld = LoaderState{};
    fence_mbar_init();
    prefetch_tensormap(&p.tm_q);
    prefetch_tensormap(&p.tm_k);
    prefetch_tensormap(&p.tm_v);
    prefetch_tensormap(&p.tm_g);
    prefetch_tensormap(&p.tm_o);
  }
  if (warp == 0) tmem_alloc(&s->tmem_base, 512);
  // everything above overlaps the planning kernel; the work list is read only after it
  grid_dep_wait();
  if (threadIdx.x == 0) s->num_items = p.hdr->num_entries * (uint32_t)p.Hv;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s->tmem_base;
  if (threadIdx.x < kIG) run_intra<MODE>(p, sm, s, tbase);
  else run_recurrence<ST, MODE>(p, sm, s, tbase);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {  // loads still in flight (issued ahead of a chunk never run)
    const LoaderState* L = &s->ld;
    if (L->n_qk > 0) mbar_wait(&s->bar[B_QK_FULL], (L->n_qk - 1) & 1);
    if (L->n_g > 0) mbar_wait(&s->bar[B_G_FULL], (L->n_g - 1) & 1);
    if (L->n_v > 0) mbar_wait(&s->bar[B_V_FULL], (L->n_v - 1) & 1);
  }
  if (warp == 0) tmem_dealloc(tbase, 512);
  if (threadIdx.x == 0) KDA_DEBUG_FOLD(p.status);
}

// ---- planning: the work list, longest first, with the longest sequences cut in two --------
// One block of kOrderKeys threads, before the prefill kernel on the same stream (no host
// sync).  Entries are ordered by chunk count, most chunks first, so that the longest
// (entry, head) chains start first on the persistent grid; a counting sort over the chunk
// counts (a histogram, an exclusive scan over the keys in descending order, a scatter), O(N)
// for any N.  Counts of kOrderKeys - 1 or more share the top key; ties land in any order,
// which only decides which CTA claims an item first -- every item computes the same result
// on any CTA.
//
// Cuts.  The grid runs about L = Hv * (all chunks) / grid chunks per CTA; a sequence longer
// than 1.05 L (and of at least kCutMinChunks chunks) would hold its CTAs well past the others,
// so up to `max_cuts` of the longest such sequences are cut after a = max(ceil(c / 2), ceil(L))
// of their c chunks.  Each cut adds the tail's identity pass (the tail's chunks once more) and
// shortens the longest chain from c to a; the combine kernel finishes the tail.  A cut needs
// room for its tail's y rows (ytok_max rows in all).  The cuts depend only on the sequence
// lengths, Hv, the grid and the workspace size, so pool and dense calls cut alike.
constexpr int kOrderKeys = 1024;
constexpr int kMaxCuts = 4;
constexpr int kCutMinChunks = 8;
constexpr uint32_t kCodeN = 0x0FFFFFFFu;

__device__ __forceinline__ int64_t seq_len_checked(const int32_t* cu, int n, int64_t T) {
  const int64_t a = cu[n], b = cu[n + 1];
  return (a >= 0 && b >= a && b <= T) ? b - a : 0;  // bad bounds: reported by the prefill
}
__device__ __forceinline__ int order_key(int64_t chunks) {
  return (int)min(chunks, (int64_t)(kOrderKeys - 1));
}
// Exclusive scan over the keys in descending order: cnt[k] becomes the first position of
// key k in the list.  Thread t holds key kOrderKeys-1-t.
__device__ void scan_keys_desc(int* cnt, int* wsum) {
  const int t = threadIdx.x, lane = t & 31, wp = t >> 5;
  const int kb = kOrderKeys - 1 - t;
  const int c = cnt[kb];
  int x = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[wp] = x;
  __syncthreads();
  if (wp == 0) {
    int w = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  cnt[kb] = x - c + (wp > 0 ? wsum[wp - 1] : 0);
  __syncthreads();
}

constexpr int kPlanCache = 4096;  // sequences whose lengths and order the block keeps on chip

__global__ void __launch_bounds__(kOrderKeys) kda_plan_kernel(const int32_t* __restrict__ cu, int N,
                                                              int64_t T, int Hv, int grid, int max_cuts,
                                                              int ytok_max, uint32_t* __restrict__ work,
                                                              SplitInfo* __restrict__ splits,
                                                              WsHeader* __restrict__ hdr) {
  __shared__ int cnt[kOrderKeys];
  __shared__ int wsum[kOrderKeys / 32];
  grid_dep_launch_dependents();  // the prefill kernel may start its prologue meanwhile
  __shared__ int len_s[kPlanCache];       // lengths of the first kPlanCache sequences
  __shared__ uint32_t order_s[kPlanCache];  // the first kPlanCache entries of the order
  __shared__ unsigned long long total;
  __shared__ int cut_n[kMaxCuts], cut_a[kMaxCuts], ncut;
  const int t = threadIdx.x;
  // lengths from cu_seqlens once; later reads come from shared memory
  auto len_of = [&](int n) -> int64_t { return n < kPlanCache ? (int64_t)len_s[n] : seq_len_checked(cu, n, T); };
  auto chunks = [&](int n) -> int64_t { return (len_of(n) + kC - 1) / kC; };
  cnt[t] = 0;
  if (t == 0) total = 0ull;
  for (int n = t; n < N && n < kPlanCache; n += kOrderKeys) len_s[n] = (int)seq_len_checked(cu, n, T);
  __syncthreads();
  unsigned long long mine = 0;
  for (int n = t; n < N; n += kOrderKeys) {
    const int64_t c = chunks(n);
    mine += (unsigned long long)c;
    atomicAdd(&cnt[order_key(c)], 1);
  }
  // one shared atomic per warp (1024 on one address would serialise)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if ((t & 31) == 0) atomicAdd(&total, mine);
  __syncthreads();
  scan_keys_desc(cnt, wsum);
  for (int n = t; n < N; n += kOrderKeys) {
    const int pos = atomicAdd(&cnt[order_key(chunks(n))], 1);
    if (KDA_CHECK(pos >= 0 && pos < N)) work[pos] = (uint32_t)n;
    if (pos < kPlanCache) order_s[pos] = (uint32_t)n;
  }
  __syncthreads();
  if (t == 0) {  // the cuts, longest sequence first
    int nc = 0, ytok = 0;
    // L = Hv total / grid; c > 1.05 L and ceil(L) in exact 64-bit integer arithmetic (the
    // double-precision unit is slow on this part)
    const int64_t hvt = (int64_t)Hv * (int64_t)total;
    const int64_t ceil_l = (hvt + grid - 1) / grid;
    for (int i = 0; i < N && nc < max_cuts; ++i) {
      const int n = (int)(i < kPlanCache ? order_s[i] : work[i]);
      const int64_t c = chunks(n);
      if (c < kCutMinChunks) break;
      if (100 * c * (int64_t)grid <= 105 * hvt) {
        if (order_key(c) < kOrderKeys - 1) break;  // sorted exactly below the top key
        continue;
      }
      const int64_t a = max((c + 1) / 2, ceil_l);
      if (a >= c) continue;
      const int64_t tail = len_of(n) - a * kC;
      if ((int64_t)ytok + tail > (int64_t)ytok_max) continue;
      splits[nc] = SplitInfo{n, (int32_t)a, ytok, (int32_t)tail};
      cut_n[nc] = n;
      cut_a[nc] = (int)a;
      ytok += (int)tail;
      ++nc;
    }
    ncut = nc;
    hdr->num_splits = (uint32_t)nc;
    hdr->num_entries = (uint32_t)(N + 2 * nc);
  }
  __syncthreads();
  if (ncut == 0) {  // the sequence order stands
    if (t == 0) KDA_DEBUG_FOLD(&hdr->status);
    return;
  }
  // the list again with the cut sequences' three entries (head; tail; tail identity pass)
  cnt[t] = 0;
  __syncthreads();
  const int nc = ncut;
  auto cut_of = [&](int n) -> int {
    for (int i = 0; i < nc; ++i)
      if (cut_n[i] == n) return i;
    return -1;
  };
  for (int n = t; n < N; n += kOrderKeys) {
    const int64_t c = chunks(n);
    const int i = cut_of(n);
    if (i < 0) {
      atomicAdd(&cnt[order_key(c)], 1);
    } else {
      atomicAdd(&cnt[order_key(cut_a[i])], 1);
      atomicAdd(&cnt[order_key(c - cut_a[i])], 2);
    }
  }
  __syncthreads();
  scan_keys_desc(cnt, wsum);
  for (int n = t; n < N; n += kOrderKeys) {
    const int64_t c = chunks(n);
    const int i = cut_of(n);
    const int cap = N + 2 * nc;
    if (i < 0) {
      const int pos = atomicAdd(&cnt[order_key(c)], 1);
      if (KDA_CHECK(pos >= 0 && pos < cap)) work[pos] = (uint32_t)n;
    } else {
      const int ph = atomicAdd(&cnt[order_key(cut_a[i])], 1);
      if (KDA_CHECK(ph >= 0 && ph < cap)) work[ph] = (uint32_t)n | ((uint32_t)KIND_HEAD << 28);
      const int k = order_key(c - cut_a[i]);
      const int pos = atomicAdd(&cnt[k], 2);
      if (KDA_CHECK(pos >= 0 && pos + 1 < cap)) {
        work[pos] = (uint32_t)n | ((uint32_t)KIND_TAIL << 28);
        work[pos + 1] = (uint32_t)n | ((uint32_t)KIND_TAIL_ID << 28);
      }
    }
  }
  __syncthreads();
  if (t == 0) KDA_DEBUG_FOLD(&hdr->status);
}

// ---- combine: completes the tails of the cut sequences --------------------------------------
// For cut s and v-head h, with S_p the head's final state, M and S_loc the final states of the
// tail's identity and zero-start passes, and y the identity pass's outputs:
//   o_t += S_p^T y_t          for every tail token t (bf16 warp MMAs, fp32 sums, o re-rounded)
//   S_end = M S_p + S_loc     into the pool row or the dense final state (fp32 FMAs)
// Units: (cut, head, group of kCombTok tail tokens) for o and (cut, head, 16 state rows) for
// the state, over a grid that leaves at once when the planning kernel made no cut.  Global
// accesses are 16-byte and coalesced; o is read, corrected and written a row piece at a time.
constexpr int kCombThreads = 256;
constexpr int kCombTok = 256;
constexpr int kCombPitch = 136;  // bf16 row pitch of the staged S_p and y tiles
constexpr int kCombAccPitch = 132;  // fp32 row pitch of the staged correction
constexpr uint32_t kCombSmem = (128 + 64) * kCombPitch * 2 + 64 * kCombAccPitch * 4;
static_assert((16 + 128) * 128 * 4 <= kCombSmem, "state units stage M rows and S_p");

struct CombineParams {
  const WsHeader* hdr;
  const SplitInfo* splits;
  const float *sp, *sl, *mm;
  const __nv_bfloat16* y;
  __nv_bfloat16* o;
  const int32_t *cu, *idx;
  void* state_out;
  uint32_t* status;
  int32_t Hv, state_vk, ytok_cap;
  int64_t num_slots, slot_stride, T;
};

__device__ __forceinline__ void mma_bf16_16816(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9},"
      " {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Four 8x8 bf16 matrices, transposed on the way: lanes 8m..8m+7 give the row addresses of
// matrix m; each lane receives the (2 tq, 2 tq + 1) x g elements of each matrix.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t r[4], const void* addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(addr)));
}

__device__ __forceinline__ int comb_o_units(const SplitInfo& sp, int Hv) {
  return (sp.ntok + kCombTok - 1) / kCombTok * Hv;
}

template <typename ST>
__global__ void __launch_bounds__(kCombThreads) kda_combine_kernel(const __grid_constant__ CombineParams p) {
  grid_dep_wait();  // the prefill grid has finished and its writes are visible
  const int ns = (int)p.hdr->num_splits;
  if (ns == 0) return;
  extern __shared__ __align__(16) uint8_t csm[];
  __nv_bfloat16* spk = reinterpret_cast<__nv_bfloat16*>(csm);            // S_p [k][v] bf16
  __nv_bfloat16* yt = spk + 128 * kCombPitch;                            // y [64 tokens][k]
  float* acc_s = reinterpret_cast<float*>(yt + 64 * kCombPitch);         // [64 tokens][v]
  float* ms = reinterpret_cast<float*>(csm);                             // state units: M rows
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hv = p.Hv;
  int total = 0;
  for (int i = 0; i < ns; ++i) total += comb_o_units(p.splits[i], Hv) + 8 * Hv;
  for (int u = blockIdx.x; u < total; u += gridDim.x) {
    int si = 0, r = u;
    for (; si < ns; ++si) {
      const int per = comb_o_units(p.splits[si], Hv) + 8 * Hv;
      if (r < per) break;
      r -= per;
    }
    const SplitInfo sp = p.splits[si];
    const int no = comb_o_units(sp, Hv);
    const size_t so = ((size_t)si * Hv) * 16384;
    __syncthreads();  // the previous unit's shared memory is no longer read
    if (r < no) {
      // ---- o of tail tokens [g * kCombTok, ...) of head h; the y rows and o pieces of a
      // 64-token tile are loaded into registers one tile ahead of the MMAs that use them
      const int h = r % Hv, g = r / Hv;
      const float4* S4 = reinterpret_cast<const float4*>(p.sp + so + (size_t)h * 16384);
      float4 sreg[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) sreg[i] = S4[tid + i * kCombThreads];  // all in flight
      const int64_t tail0 = (int64_t)p.cu[sp.n] + (int64_t)sp.cut * kC;  // first tail token
      const int t_beg = g * kCombTok, t_end = min(sp.ntok, (g + 1) * kCombTok);
      auto load_y = [&](int tb, uint4 (&yr)[4]) {
        const int nt = min(64, t_end - tb);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int e = tid + i * kCombThreads, row = e >> 4, c8 = (e & 15) * 8;
          yr[i] = row < nt && KDA_CHECK(sp.ytok0 + tb + row < p.ytok_cap)
                      ? *reinterpret_cast<const uint4*>(p.y + ((size_t)(sp.ytok0 + tb + row) * Hv + h) * 128 + c8)
                      : make_uint4(0u, 0u, 0u, 0u);
        }
      };
      uint4 yr[4];
      load_y(t_beg, yr);
#pragma unroll
      for (int i = 0; i < 16; ++i) {  // S_p [k][v] as bf16
        const int e = tid + i * kCombThreads, k = e >> 5, v4 = (e & 31) * 4;
        uint2 w;
        w.x = pack_bf16x2(sreg[i].x, sreg[i].y);
        w.y = pack_bf16x2(sreg[i].z, sreg[i].w);
        *reinterpret_cast<uint2*>(spk + k * kCombPitch + v4) = w;
      }
      for (int tb = t_beg; tb < t_end; tb += 64) {
        const int nt = min(64, t_end - tb);
        __syncthreads();  // acc_s / yt of the previous tile consumed
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int e = tid + i * kCombThreads, row = e >> 4, c8 = (e & 15) * 8;
          *reinterpret_cast<uint4*>(yt + row * kCombPitch + c8) = yr[i];
        }
        // this tile's o pieces and the next tile's y rows, in flight during the MMAs
        uint4 orr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int e = tid + i * kCombThreads, row = e >> 4, c8 = (e & 15) * 8;
          orr[i] = row < nt && KDA_CHECK(tail0 + tb + row < p.T)
                       ? *reinterpret_cast<const uint4*>(p.o + ((size_t)(tail0 + tb + row) * Hv + h) * 128 + c8)
                       : make_uint4(0u, 0u, 0u, 0u);
        }
        if (tb + 64 < t_end) load_y(tb + 64, yr);
        __syncthreads();
        // warp: tokens r0..r0+15, values n0..n0+63
        const int r0 = (warp & 3) * 16, n0 = (warp >> 2) * 64;
        const int gq = lane >> 2, tq = lane & 3;
        float acc[8][4] = {};
#pragma unroll
        for (int kb = 0; kb < 128; kb += 16) {
          uint32_t a[4];
          a[0] = *reinterpret_cast<const uint32_t*>(yt + (r0 + gq) * kCombPitch + kb + 2 * tq);
          a[1] = *reinterpret_cast<const uint32_t*>(yt + (r0 + gq + 8) * kCombPitch + kb + 2 * tq);
          a[2] = *reinterpret_cast<const uint32_t*>(yt + (r0 + gq) * kCombPitch + kb + 2 * tq + 8);
          a[3] = *reinterpret_cast<const uint32_t*>(yt + (r0 + gq + 8) * kCombPitch + kb + 2 * tq + 8);
#pragma unroll
          for (int np = 0; np < 4; ++np) {  // two 8-wide value tiles per ldmatrix
            uint32_t b[4];
            const int mrow = kb + (lane & 15);
            const int mcol = n0 + np * 16 + (lane >> 4) * 8;
            ldsm_x4_trans(b, spk + mrow * kCombPitch + mcol);
            mma_bf16_16816(acc[np * 2], a, b[0], b[1]);
            mma_bf16_16816(acc[np * 2 + 1], a, b[2], b[3]);
          }
        }
#pragma unroll
        for (int nt8 = 0; nt8 < 8; ++nt8) {
          const int col = n0 + nt8 * 8 + 2 * tq;
          *reinterpret_cast<float2*>(acc_s + (r0 + gq) * kCombAccPitch + col) =
              make_float2(acc[nt8][0], acc[nt8][1]);
          *reinterpret_cast<float2*>(acc_s + (r0 + gq + 8) * kCombAccPitch + col) =
              make_float2(acc[nt8][2], acc[nt8][3]);
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // o rows, 16 bytes at a time
          const int e = tid + i * kCombThreads, row = e >> 4, c8 = (e & 15) * 8;
          if (row < nt && KDA_CHECK(tail0 + tb + row < p.T)) {
            const float* cs = acc_s + row * kCombAccPitch + c8;
            const uint32_t in[4] = {orr[i].x, orr[i].y, orr[i].z, orr[i].w};
            uint32_t outw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
              outw[j] = pack_bf16x2(__uint_as_float(in[j] << 16) + cs[2 * j],
                                    __uint_as_float(in[j] & 0xFFFF0000u) + cs[2 * j + 1]);
            *reinterpret_cast<uint4*>(p.o + ((size_t)(tail0 + tb + row) * Hv + h) * 128 + c8) =
                make_uint4(outw[0], outw[1], outw[2], outw[3]);
          }
        }
      }
    } else {
      // ---- rows 16 rb .. 16 rb + 15 of head h's final state: S_end = M S_p + S_loc, with
      // S_p and the 16 rows of M staged in shared memory (every load in flight at once)
      const int rr = r - no, h = rr >> 3, rb = rr & 7;
      ST* dst = nullptr;
      if (p.state_out) {
        if (p.idx) {
          const int64_t sl = resolve_slot(p.idx, sp.n, p.num_slots);
          if (sl >= 0) dst = static_cast<ST*>(p.state_out) + sl * p.slot_stride + (size_t)h * 16384;
        } else {
          dst = static_cast<ST*>(p.state_out) + ((size_t)sp.n * Hv + h) * 16384;
        }
      }
      if (!dst) continue;
      const float4* M4 = reinterpret_cast<const float4*>(p.mm + so + (size_t)h * 16384 + rb * 16 * 128);
      const float4* S4 = reinterpret_cast<const float4*>(p.sp + so + (size_t)h * 16384);
      const float* SL = p.sl + so + (size_t)h * 16384;
      float* ss = ms + 16 * 128;  // S_p [j][v]
      const int v = tid & 127, k0 = (tid >> 7) * 8;  // rows 16 rb + k0 .. + 7
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = SL[(size_t)(rb * 16 + k0 + i) * 128 + v];
#pragma unroll
      for (int i = 0; i < 2; ++i) reinterpret_cast<float4*>(ms)[tid + i * kCombThreads] = M4[tid + i * kCombThreads];
#pragma unroll 4
      for (int i = 0; i < 16; ++i) reinterpret_cast<float4*>(ss)[tid + i * kCombThreads] = S4[tid + i * kCombThreads];
      __syncthreads();
#pragma unroll 8
      for (int j = 0; j < 128; ++j) {
        const float sv = ss[j * 128 + v];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(ms[(k0 + i) * 128 + j], sv, acc[i]);
      }
      if (p.state_vk) {  // row v, key channels 16 rb + k0 .. + 7: two 16-byte pieces (fp32)
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[(size_t)v * 128 + rb * 16 + k0 + i] = from_f32<ST>(acc[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[(size_t)(rb * 16 + k0 + i) * 128 + v] = from_f32<ST>(acc[i]);
      }
    }
  }
  if (threadIdx.x == 0) KDA_DEBUG_FOLD(p.status);
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

// [T, Hv] gate (scalar per token and head): 2-D map, boxes of 64 tokens x (16 bytes of heads).
bool make_map_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem, int64_t T,
                 int H, int box_inner) {
  auto enc = get_encoder();
  if (!enc) return false;
  const int64_t rows = T > 0 ? T : 1;
  cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)H * elem};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)kC};
  cuuint32_t es[2] = {1u, 1u};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The prefill kernel, and the combine kernel when cuts are possible, each launched with
// programmatic stream serialisation: a kernel may be scheduled while the one before it on
// the stream still runs, and waits for it in grid_dep_wait before reading its results.
template <typename KP, typename KC>
cudaError_t launch_pair(KP kern, KC comb, const TcParams& p, const CombineParams& cp, int grid,
                        int cgrid, bool with_combine, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  err = cudaLaunchKernelEx(&cfg, kern, p);
  if (err != cudaSuccess || !with_combine) return err;
  err = cudaFuncSetAttribute(comb, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCombSmem);
  if (err != cudaSuccess) return err;
  cfg.gridDim = dim3((unsigned)cgrid);
  cfg.blockDim = dim3(kCombThreads);
  cfg.dynamicSmemBytes = kCombSmem;
  return cudaLaunchKernelEx(&cfg, comb, cp);
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
  // a scalar gate is staged by 16-byte groups of heads (8 bf16 a): Hv % 8 == 0
  return d.qkv_dtype == KDA_BF16 && d.head_k_dim == kK && d.head_v_dim == kV &&
         (d.flags & KDA_FLAG_CUDA_CORE_PATH) == 0u &&
         ((d.flags & KDA_FLAG_SCALAR_GATE) == 0u || d.num_v_heads % 8 == 0);
}

namespace {
// Workspace after the 256-byte header: the work list (one 32-bit entry per sequence plus two
// per cut), then, when cuts are allowed, the cut records, the head / tail / identity-pass
// final states (fp32 [cuts][Hv][K][V] each) and the y rows of the tails ([rows][Hv][K] bf16).
struct WsLayout {
  size_t work, splits, sp, sl, mm, y, end;
};
WsLayout ws_layout(const kda_desc_t& d, int cuts, int64_t ytok) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  WsLayout L;
  size_t off = kWsPayload;
  L.work = off;
  off += up(sizeof(uint32_t) * ((size_t)d.num_seqs + 2 * (size_t)cuts));
  L.splits = off;
  off += up(sizeof(SplitInfo) * (size_t)cuts);
  const size_t st = (size_t)cuts * d.num_v_heads * kK * kV * sizeof(float);
  L.sp = off;
  off += st;
  L.sl = off;
  off += st;
  L.mm = off;
  off += st;
  L.y = off;
  off += up((size_t)ytok * d.num_v_heads * kK * sizeof(__nv_bfloat16));
  L.end = off;
  return L;
}
// Cut capacity of a workspace of the full size: up to kMaxCuts sequences, tails of up to
// 8192 tokens in all.
int full_cuts(const kda_desc_t& d) { return (int)std::min<int64_t>(d.num_seqs, kMaxCuts); }
int64_t full_ytok(const kda_desc_t& d) { return std::min<int64_t>(d.total_tokens, 8192); }
}  // namespace

size_t prefill_tc_workspace(const kda_desc_t& d) {
  return ws_layout(d, full_cuts(d), full_ytok(d)).end - kWsPayload;
}
size_t prefill_tc_min_workspace(const kda_desc_t& d) { return ws_layout(d, 0, 0).end - kWsPayload; }

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
        !make_map(&p.tm_o, a.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T, d.num_v_heads, kV, kV,
                  CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !(a.gate_k == 1
              ? (a.act.a ? make_map_2d(&p.tm_g, a.act.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T,
                                       d.num_v_heads, 8)
                         : make_map_2d(&p.tm_g, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, T,
                                       d.num_v_heads, 4))
              : a.act.a ? make_map(&p.tm_g, a.act.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T,
                                   d.num_v_heads, kK, kK, CU_TENSOR_MAP_SWIZZLE_NONE)
                        : make_map(&p.tm_g, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, T,
                                   d.num_v_heads, kK, kK, CU_TENSOR_MAP_SWIZZLE_NONE)))
      return cudaErrorInvalidValue;
  }
  // cuts only with a workspace of the full size (a smaller one, down to the minimum, runs
  // every sequence whole)
  const WsLayout full = ws_layout(d, full_cuts(d), full_ytok(d));
  const bool can_cut = a.ws_bytes >= full.end && d.num_seqs < (int)kCodeN;
  const WsLayout L = can_cut ? full : ws_layout(d, 0, 0);
  p.work = reinterpret_cast<const uint32_t*>(a.ws + L.work);
  p.splits = reinterpret_cast<const SplitInfo*>(a.ws + L.splits);
  p.hdr = reinterpret_cast<const WsHeader*>(a.ws);
  p.sp = reinterpret_cast<float*>(a.ws + L.sp);
  p.sl = reinterpret_cast<float*>(a.ws + L.sl);
  p.mm = reinterpret_cast<float*>(a.ws + L.mm);
  p.y = reinterpret_cast<__nv_bfloat16*>(a.ws + L.y);
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k = static_cast<const __nv_bfloat16*>(a.k);
  p.g = a.g;
  p.act = a.act;
  p.gate_k = a.gate_k;
  p.l2norm = a.l2norm ? 1 : 0;
  p.state_vk = a.state_vk ? 1 : 0;
  p.gw = a.act.a ? 8 : 4;
  p.g_bytes = a.gate_k == 1 ? 1024u : (a.act.a ? 16384u : 32768u);
  p.beta = a.beta;
  p.cu = a.cu;
  p.idx = a.idx;
  p.state_in = a.state_in;
  p.state_out = a.state_out;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.status = a.status;
  p.next_item = &reinterpret_cast<WsHeader*>(a.ws)->next_item;
  p.N = d.num_seqs;
  p.Hk = d.num_k_heads;
  p.Hv = d.num_v_heads;
  p.T = T;
  p.num_slots = d.num_slots;
  p.slot_stride = a.slot_stride;
  p.scale = a.scale;
  p.wait_limit_ns = pipeline_wait_limit_ns();
  p.max_cuts = can_cut ? full_cuts(d) : 0;
  p.ytok_cap = can_cut ? (int32_t)full_ytok(d) : 0;

  const int max_cuts = can_cut ? full_cuts(d) : 0;
  const int64_t max_items = ((int64_t)d.num_seqs + 2 * max_cuts) * d.num_v_heads;
  const int grid = (int)std::min<int64_t>(sm_count(), std::max<int64_t>(1, max_items));
  kda_plan_kernel<<<1, kOrderKeys, 0, st>>>(a.cu, d.num_seqs, T, d.num_v_heads, grid, max_cuts,
                                            can_cut ? (int)full_ytok(d) : 0,
                                            reinterpret_cast<uint32_t*>(a.ws + L.work),
                                            reinterpret_cast<SplitInfo*>(a.ws + L.splits),
                                            reinterpret_cast<WsHeader*>(a.ws));
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  CombineParams cp;
  cp.hdr = p.hdr;
  cp.splits = p.splits;
  cp.sp = p.sp;
  cp.sl = p.sl;
  cp.mm = p.mm;
  cp.y = p.y;
  cp.o = p.o;
  cp.cu = p.cu;
  cp.idx = p.idx;
  cp.state_out = p.state_out;
  cp.Hv = d.num_v_heads;
  cp.status = p.status;
  cp.ytok_cap = p.ytok_cap;
  cp.T = T;
  cp.state_vk = a.state_vk ? 1 : 0;
  cp.num_slots = d.num_slots;
  cp.slot_stride = a.slot_stride;
  const int cgrid = 2 * sm_count();
  // the plain fp32 per-channel gate and the activated per-channel gate, without normalisation,
  // each run the kernel compiled for that form alone
  const int mode = (p.gate_k == 1 || p.l2norm) ? 2 : (p.act.a != nullptr ? 1 : 0);
  const bool cut = max_cuts > 0;
  if (d.state_dtype == KDA_BF16) {
    using C = __nv_bfloat16;
    return mode == 0 ? launch_pair(kda_prefill_tc_kernel<C, 0>, kda_combine_kernel<C>, p, cp, grid, cgrid, cut, st)
         : mode == 1 ? launch_pair(kda_prefill_tc_kernel<C, 1>, kda_combine_kernel<C>, p, cp, grid, cgrid, cut, st)
                     : launch_pair(kda_prefill_tc_kernel<C, 2>, kda_combine_kernel<C>, p, cp, grid, cgrid, cut, st);
  }
  return mode == 0 ? launch_pair(kda_prefill_tc_kernel<float, 0>, kda_combine_kernel<float>, p, cp, grid, cgrid, cut, st)
       : mode == 1 ? launch_pair(kda_prefill_tc_kernel<float, 1>, kda_combine_kernel<float>, p, cp, grid, cgrid, cut, st)
                   : launch_pair(kda_prefill_tc_kernel<float, 2>, kda_combine_kernel<float>, p, cp, grid, cgrid, cut, st);
}

}  // namespace kda
