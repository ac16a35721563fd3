/*
 * kda.h -- C ABI of the GB300 (sm_103a) chunked KDA prefill and decode library.
 *
 * KDA is the gated delta rule with a per-channel (per key channel) decay gate.
 * Per v-head, token by token:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * The prefill evaluates this in chunks of 64 tokens (intra-chunk work in
 * parallel, one sequential state pass across chunks), which is the pipeline of
 * the sglang PR 27488 digest "KDA SM100 CuteDSL prefill" (sections 实现拆解 /
 * implementation breakdown and 关键文件 / key files: gate prologue, KKT inverse
 * and U/W, h (state) kernel, output kernel).  The state pool I/O follows the
 * sglang PR 30169 digest "pool state I/O fused into the h kernel" (实现拆解
 * items 1-3).  The decode grid rule follows the sglang PR 37317 digest "FLA/MoE
 * grid split" (实现拆解 item 1: sequences and heads on separate grid axes).
 *
 * General rules for every entry point
 * -----------------------------------
 *  - All tensor pointers are DEVICE pointers, owned by the caller; tensors are
 *    packed, contiguous and row-major with the shapes given below.  The library
 *    sees no sizes: every buffer must hold at least the shape stated for it
 *    (the Python binding checks shapes before calling).
 *  - q, k, v, g (or a), o and the state buffers must be 16-byte aligned (they
 *    are moved by TMA); an unaligned one is KDA_ERR_INVALID_ARGUMENT.
 *  - Calls are asynchronous on `stream`.  They never allocate device memory and
 *    never synchronise the host (the pages measured both as the dominant host
 *    cost: a ~200 MB re-allocation per call and a device->host `.item()` in the
 *    metadata step -- PR 27488 digest, 功能与动机 and 关键源码片段).
 *  - Host-checkable errors return synchronously and nothing is enqueued.
 *  - Errors found in device data (a slot index out of range, a non-monotone or
 *    out-of-range cu_seqlens) set bits in a status word kept in the workspace;
 *    the offending sequence is skipped (its outputs and state rows are left
 *    untouched) and every other sequence is computed normally.  Read the word
 *    with kda_read_device_status().  Kernels never trap.
 *  - Thread safety: calls that share a workspace must be ordered on one stream.
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARGUMENT = 1,   /* bad pointer, shape or mode combination      */
    KDA_ERR_UNSUPPORTED = 2,        /* valid but not implemented (dtype, head dims) */
    KDA_ERR_WORKSPACE_TOO_SMALL = 3,
    KDA_ERR_CUDA = 4,               /* a CUDA launch or copy failed                */
    KDA_ERR_DEVICE_DATA = 5         /* kda_read_device_status: device data invalid */
} kda_status_t;

typedef enum { KDA_BF16 = 0, KDA_F32 = 1 } kda_dtype_t;

/* Device status bits (kda_read_device_status). */
#define KDA_DEVICE_BAD_SLOT      0x1u  /* state index < -1 or >= num_slots          */
#define KDA_DEVICE_BAD_SEQLENS   0x2u  /* cu_seqlens not monotone / outside [0, T]  */
#define KDA_DEVICE_PIPE_TIMEOUT  0x4u  /* an internal pipeline wait gave up         */
#define KDA_DEVICE_DEBUG_BOUNDS  0x8u  /* debug build only: a computed index fell outside
                                          its buffer (the access was skipped)         */

/* Descriptor flags. */
#define KDA_FLAG_CUDA_CORE_PATH  0x1u  /* prefill: run the fp32 CUDA-core kernel even where
                                          the tensor-core kernel applies (cross-checks) */
#define KDA_FLAG_SCALAR_GATE     0x2u  /* prefill and decode: the gate carries one value per
                                          (token, v-head), shared by all key channels -- the
                                          gated-delta-net (GDN) form that the pages' pool test
                                          runs (PR 30169 digest, 关键源码片段).  g is then
                                          [>=T, Hv] fp32 and, for kda_chunk_prefill_act, a is
                                          [>=T, Hv] and dt_bias [Hv]. */
#define KDA_FLAG_QK_L2NORM       0x4u  /* prefill and decode: q and k are L2-normalised per
                                          (token, head) inside the kernel, x / max(||x||, 1e-12),
                                          as the pages' callers do before the call (PR 27488
                                          digest, 关键源码片段 CuteDSLKDAKernel.extend; the
                                          tensor-core kernel re-rounds them to bf16 as the
                                          caller's normalise-then-cast does). */

#define KDA_FLAG_STATE_VK        0x8u  /* prefill and decode: every state buffer (pool, dense
                                          initial / final states, draft-step cache) holds each
                                          head's state transposed, [V][K] (row v is the state's
                                          column v), the [num_slots, Hv, head_v_dim, head_k_dim]
                                          pool of the pages' GDN test (PR 30169 digest, 关键源码
                                          片段).  Default: [K][V].  The prefill runs the same
                                          arithmetic either way (results bit-identical to the
                                          default layout's, transposed); the decode reduces over
                                          the key channels in another order. */

/* Problem descriptor shared by prefill and decode. */
typedef struct {
    int32_t num_seqs;          /* N (prefill: packed sequences; decode: rows)          */
    int64_t total_tokens;      /* T: rows of q/k/v/o.  Authoritative: g and beta may be
                                  longer (CUDA-graph padding); only T rows are read
                                  (PR 27488 digest, 实现拆解 item 3).  Decode: T == N. */
    int32_t num_k_heads;       /* Hk (q and k heads)                                    */
    int32_t num_v_heads;       /* Hv; Hv % Hk == 0; v-head h reads k/q head h/(Hv/Hk)   */
    int32_t head_k_dim;        /* K in {64, 128}                                        */
    int32_t head_v_dim;        /* V in {64, 128}                                        */
    kda_dtype_t qkv_dtype;     /* dtype of q, k, v and o                                */
    kda_dtype_t state_dtype;   /* dtype of the state / pool (math is fp32 inside)       */
    float scale;               /* output scale; <= 0 selects K^-0.5                     */
    int32_t chunk_size;        /* must be 64                                            */
    int64_t num_slots;         /* pool mode: rows of the pool; slot num_slots-1 is the
                                  sentinel that index -1 maps to                        */
    int64_t slot_stride_elems; /* pool: elements between consecutive slots; 0 means
                                  Hv*K*V.  Must be >= Hv*K*V.  (The pitch is passed, not
                                  inferred from a shape: PR 37317 digest, 实现拆解 item 2.) */
    uint32_t flags;            /* KDA_FLAG_* bits; every other bit must be 0           */
} kda_desc_t;

/* Bytes of workspace kda_chunk_prefill() wants for this descriptor (0 on an
 * invalid descriptor).  The workspace is caller-owned device memory, aligned to
 * 256 bytes, reusable across calls on the same stream; its contents need no
 * initialisation.  It holds the device status word, the work list and, for the
 * tensor-core path, room to cut up to 4 of the longest sequences in two (the
 * final states of the parts and up to 8192 rows of tail outputs, [rows][Hv][K]
 * bf16): a sequence much longer than the batch's share per SM would keep its
 * SMs busy long after the others, so its tail runs in parallel with its head
 * and is completed by an exact affine combine (the state after the cut is
 * M S_p + S_loc; outputs gain S_p^T y).  With Hv = 32 that is up to ~88 MB. */
size_t kda_chunk_prefill_workspace_size(const kda_desc_t *desc);

/* The least workspace kda_chunk_prefill() accepts (status word and work list):
 * with less than kda_chunk_prefill_workspace_size() bytes no sequence is cut,
 * which gives the same results up to rounding, more slowly when one sequence
 * dominates the batch. */
size_t kda_chunk_prefill_min_workspace_size(const kda_desc_t *desc);

/* Bytes of workspace kda_decode() needs (status word only). */
size_t kda_decode_workspace_size(const kda_desc_t *desc);

/*
 * Chunked KDA prefill over packed variable-length sequences.
 *
 *   q, k         [T, Hk, K]  qkv_dtype.  Expected L2-normalised per head (the
 *                            caller normalises, as on the pages: PR 27488 digest,
 *                            CuteDSLKDAKernel.extend); not re-normalised here.
 *   v            [T, Hv, V]  qkv_dtype
 *   g            [>=T, Hv, K] fp32 natural-log decay per key channel (g <= 0)
 *   beta         [>=T, Hv]    fp32
 *   cu_seqlens   [N+1] int32, cu_seqlens[0] = 0, non-decreasing, cu_seqlens[N] <= T.
 *                Chunks start at each sequence's first token; the last chunk of a
 *                sequence may be partial.
 *   state        pool mode (state_indices != NULL): the pool, num_slots rows of
 *                [Hv, K, V] (row pitch slot_stride_elems), read and written IN
 *                PLACE: sequence n starts from slot s_n and its final state is
 *                written back to slot s_n, where s_n = state_indices[n] if >= 0,
 *                else num_slots-1 (PR 30169 digest, 实现拆解 items 1-3).  Rows not
 *                named are not touched.  Indices should be distinct (a repeated
 *                slot, e.g. the sentinel, gets an unspecified one of the results).
 *                dense mode (state_indices == NULL): initial states [N, Hv, K, V],
 *                or NULL for zero initial states.
 *   state_indices  [N] int32 or NULL (selects the mode)
 *   final_state  pool mode: must be NULL or equal to `state`.
 *                dense mode: [N, Hv, K, V] state_dtype, or NULL to skip; may
 *                equal `state` (in-place update).
 *   o            [T, Hv, V] qkv_dtype, fully overwritten for every valid token.
 *   workspace    kda_chunk_prefill_workspace_size(desc) bytes (at least
 *                kda_chunk_prefill_min_workspace_size(desc)), 256-byte aligned.
 *
 * State layout: S[k][v] row-major per (slot or sequence, v-head).
 * Pool mode and dense mode run the same kernels and the same arithmetic; only
 * the addresses differ, so o and the written state rows are bit-identical
 * between the two modes (PR 30169 digest, 实现拆解 item 4).
 * Run to run, results are bit-identical (no atomics in any reduction), for the
 * same inputs and workspace size; which sequences are cut depends only on the
 * sequence lengths, Hv, the GPU's SM count and the workspace size.
 */
kda_status_t kda_chunk_prefill(const kda_desc_t *desc, const void *q, const void *k,
                               const void *v, const float *g, const float *beta,
                               const int32_t *cu_seqlens, void *state,
                               const int32_t *state_indices, void *final_state, void *o,
                               void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Chunked KDA prefill with the gate activation computed in the kernel: instead of
 * reading the fp32 log-decay g, it reads the pre-activation a and computes, per
 * (token t, v-head h, key channel c),
 *
 *   g[t,h,c] = max( -exp(A_log[h]) * softplus(a[t,h,c] + dt_bias[h,c]), lower_bound )
 *
 * with softplus(x) = log(1 + exp(x)).  The -exp(A_log) * softplus(a + dt_bias) form
 * is the gate of the pages' tests (PR 30169 digest, 关键源码片段, the GDN pool test;
 * PR 27488 digest, 关键源码片段: CuteDSLKDAKernel.extend takes A_log, dt_bias and
 * lower_bound); here it is per key channel, as KDA's gate is.  The pages name
 * lower_bound without a formula; it is read as a floor on g.
 *
 *   a            [>=T, Hv, K] qkv_dtype (16-byte aligned)
 *   A_log        [Hv] fp32
 *   dt_bias      [Hv, K] fp32, or NULL for zero
 *   lower_bound  <= 0; -INFINITY for none (NaN or > 0 is KDA_ERR_INVALID_ARGUMENT)
 *
 * Every other argument, the workspace, the modes and the error behaviour are those
 * of kda_chunk_prefill().  The bf16 a is half the bytes of the fp32 g it replaces.
 */
kda_status_t kda_chunk_prefill_act(const kda_desc_t *desc, const void *q, const void *k,
                                   const void *v, const void *a, const float *A_log,
                                   const float *dt_bias, float lower_bound, const float *beta,
                                   const int32_t *cu_seqlens, void *state,
                                   const int32_t *state_indices, void *final_state, void *o,
                                   void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * One-token-per-row KDA decode, updating a state pool in place.
 *
 *   q, k   [N, Hk, K]   v [N, Hv, V]   g [>=N, Hv, K] fp32   beta [>=N, Hv] fp32
 *   state_pool     num_slots rows of [Hv, K, V] (pitch slot_stride_elems)
 *   state_indices  [N] int32; -1 (padding) maps to the sentinel slot num_slots-1;
 *                  NULL means row n uses slot n.  Rows that share a slot (padding
 *                  rows on the sentinel) race: their outputs and that slot's final
 *                  contents are unspecified.
 *   o      [N, Hv, V] qkv_dtype
 * The grid keeps rows and heads on separate axes with rows on grid.x, so any
 * N < 2^31 launches (PR 37317 digest, 实现拆解 item 1 and 风险与影响 item 5:
 * folding N*Hv into one 65535-limited axis made large decode batches fail).
 */
kda_status_t kda_decode(const kda_desc_t *desc, const void *q, const void *k, const void *v,
                        const float *g, const float *beta, void *state_pool,
                        const int32_t *state_indices, void *o, void *workspace,
                        size_t workspace_bytes, cudaStream_t stream);

/*
 * Decode of speculative draft steps with a per-step state cache.  Row n of the batch is a
 * request whose draft tokens cu_seqlens[n] .. cu_seqlens[n+1]-1 (at most max_steps of
 * them) run one after another from pool[s_n] (s_n as in kda_decode; state_indices NULL
 * means s_n = n).  The state after draft step j is written to
 *
 *     step_cache + n * cache_pitch_elems + j * (Hv*K*V)      ([Hv, K, V], state_dtype)
 *
 * so that a caller can keep the state of the accepted prefix.  The per-request pitch is
 * passed explicitly: the pages fixed a cache-stride bug that inferred it from the buffer's
 * shape, which changes when the number of drafts does (PR 37317 digest, 实现拆解 item 2).
 * The pool row is written with the last step's state only if update_pool != 0.
 *
 *   desc          num_seqs = N requests, total_tokens = T draft tokens in all
 *   q, k [T,Hk,K]; v, o [T,Hv,V]; g [T,Hv,K] (or [T,Hv] with KDA_FLAG_SCALAR_GATE);
 *   beta [T,Hv]; cu_seqlens [N+1] int32
 *   step_cache    NULL (no per-step states) or 16-byte aligned, with
 *                 cache_pitch_elems >= max_steps*Hv*K*V and a multiple of 8
 * A request longer than max_steps, or a bad cu_seqlens, sets KDA_DEVICE_BAD_SEQLENS and
 * is skipped.  Same grid rule as kda_decode (rows on grid.x).  Errors as kda_decode.
 */
kda_status_t kda_decode_draft(const kda_desc_t *desc, const void *q, const void *k,
                              const void *v, const float *g, const float *beta,
                              const int32_t *cu_seqlens, void *state_pool,
                              const int32_t *state_indices, void *step_cache,
                              int64_t cache_pitch_elems, int32_t max_steps, int update_pool,
                              void *o, void *workspace, size_t workspace_bytes,
                              cudaStream_t stream);

/*
 * Allocation-free prefill.  The pages have no counterpart of this entry point.
 *
 * For callers that cannot allocate device memory when they run the prefill:
 * plug-in hosts whose device allocator belongs to someone else, and real-time paths
 * that forbid allocation after start-up.  It
 * takes the same arguments as kda_chunk_prefill() minus the workspace: the scratch
 * the prefill needs (status word, work counter, sequence order) comes from a fixed
 * array of KDA_NOALLOC_SCRATCH_BYTES bytes in the library's device memory, which
 * every GPU that loads the library holds until the process exits.  The call never
 * calls cudaMalloc, cudaFree or any allocating library routine.  The array has no
 * room to cut long sequences, so every sequence runs whole (the results of
 * kda_chunk_prefill() with kda_chunk_prefill_min_workspace_size() bytes).
 *
 *  - Limit: num_seqs <= KDA_NOALLOC_MAX_SEQS; a larger batch returns
 *    KDA_ERR_WORKSPACE_TOO_SMALL and enqueues nothing.
 *  - The first call on a device looks up that device's copy of the array
 *    (cudaGetSymbolAddress) and caches it; make that first call before any
 *    stream capture.
 *  - Every call on a device shares the one array and it keeps the last call's
 *    contents (each call clears what must start at zero).  Calls that overlap on
 *    the GPU (different streams, no ordering between them) race on it: order them.
 *  - Device-data errors are recorded in the shared array's status word, which this
 *    entry point offers no way to read back; use kda_chunk_prefill() with a
 *    workspace to diagnose inputs.
 */
#define KDA_NOALLOC_MAX_SEQS 16384
#define KDA_NOALLOC_SCRATCH_BYTES (256 + 4 * KDA_NOALLOC_MAX_SEQS)
kda_status_t kda_chunk_prefill_noalloc(const kda_desc_t *desc, const void *q, const void *k,
                                       const void *v, const float *g, const float *beta,
                                       const int32_t *cu_seqlens, void *state,
                                       const int32_t *state_indices, void *final_state,
                                       void *o, cudaStream_t stream);

/*
 * Bound of the internal pipeline waits of the tensor-core prefill, for launches made
 * after the call (process-wide; 0 restores the default of 2 seconds; more than 2 s is
 * KDA_ERR_INVALID_ARGUMENT).  The pages have no counterpart: it is the watchdog of this
 * library's own kernels.  Every wait between the kernel's producer and consumer warps
 * gives up after this long; the kernel then sets KDA_DEVICE_PIPE_TIMEOUT, stops taking
 * work, lets the loads and matrix operations it issued finish (those last waits keep the
 * full 2 s bound) and returns -- it never traps.  Outputs of such a call are unspecified;
 * the next call starts clean.  A bound far below a chunk's latency (a microsecond or
 * less) makes the waits give up on purpose, which is how the failure path is tested.
 */
kda_status_t kda_set_pipeline_wait_limit(uint64_t nanoseconds);

/* Synchronises `stream`, then reads the device status word left in `workspace`
 * by the last prefill or decode call that used it.  Returns KDA_OK or
 * KDA_ERR_DEVICE_DATA (raw bits in *bits_out if bits_out != NULL), or
 * KDA_ERR_CUDA if the synchronisation or copy failed. */
kda_status_t kda_read_device_status(const void *workspace, uint32_t *bits_out,
                                    cudaStream_t stream);

/* Which prefill kernel path a descriptor selects: 1 = fused tensor-core
 * (tcgen05) path, 0 = CUDA-core (fp32 FFMA) path, -1 = invalid descriptor. */
int kda_chunk_prefill_path(const kda_desc_t *desc);

/* Human-readable name of a status code (static storage). */
const char *kda_status_string(kda_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* KDA_GB300_H */
