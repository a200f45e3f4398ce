/*
 * kda.h -- C ABI of libkda.so: Kimi Delta Attention (KDA) prefill and decode
 * on one NVIDIA GB300 (sm_103a).
 *
 * KDA is the gated delta rule with a per-channel decay.  For every (sequence,
 * head) it carries a matrix state S in R^{dk x dv}, held in fp32, and for each
 * token t with query q_t, key k_t (dk), value v_t (dv), log-decay g_t (dk) and
 * write strength beta_t (scalar) it computes
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *
 * ("Kimi K3 on vLLM: Up to 370 Tokens/sec", section "Kimi Delta Attention: a
 * hybrid recurrent + full-attention stack": a linear-attention mechanism with a
 * fixed-size recurrent state; "Kimi K3 + vLLM: Inside the Day-0 Production
 * Integration", section "Kimi Delta Attention: When Prefix Caching Meets
 * Recurrent State": a fixed-size matrix-like recurrent state per layer).
 * g is used as given (exp g is the decay; no activation is applied) and there
 * is no in-kernel normalisation or 1/sqrt(dk) scaling of q or k.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument of the compute calls is caller-owned DEVICE memory
 *   (cu_seqlens, init_slots and slot_ids included).  The library allocates no
 *   device memory in these calls; scratch lives in the caller's workspace.
 * - All arrays are dense, row-major, contiguous, with 16-byte aligned base
 *   pointers.  q, k, v, g, beta and out share the element type a->dtype.
 *   Token-major layouts: q, k, g: [T][H][dk]; v, out: [T][H][dv]; beta: [T][H].
 *   States: state_pool [n_slots][H][dk][dv] fp32, row i of a state is the
 *   key channel i.
 * - The calls are asynchronous and stream-ordered on a->stream (a
 *   cudaStream_t; NULL is the legacy default stream).
 * - Errors that the host can see (null pointers, bad sizes, unsupported
 *   shapes, a too-small workspace) return immediately without launching
 *   anything.  Errors that only the device can see (a slot id out of range, a
 *   duplicate destination slot, non-monotone cu_seqlens, too small a snapshot
 *   buffer) are recorded in a sticky error word in the workspace, the
 *   offending sequence's writes are skipped (nothing outside the caller's
 *   buffers is touched), and kda_device_status() reports and clears them.
 * - Results are deterministic: no floating-point atomics, no order-dependent
 *   reductions.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,   /* a host-visible argument is wrong; nothing launched */
  KDA_ERR_UNSUPPORTED = 2,   /* valid but not supported (shape, dtype, algo) */
  KDA_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch, sync) */
  KDA_ERR_DEVICE_CHECK = 4,  /* a device-side argument check failed (see kda_device_status) */
  KDA_ERR_TIMEOUT = 5        /* a bounded device-side wait gave up */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Which prefill algorithm to run.  AUTO picks the tensor-core chunked
 * prefill for bf16 with dk = 128, dv in {64, 128} and snap_interval % 64 == 0,
 * else the token-recurrent CUDA-core kernel (exact fp32 recurrence, any
 * supported shape).  The chunked prefill has two variants: one CTA per
 * (sequence, head, dv block), and, when a batch has at most 64 (sequence,
 * head) pairs with dv = 128 and the workspace was sized for it, a cooperative
 * grid in which the other SMs prepare chunks for the per-pair CTAs.  The
 * cooperative grid carries each pair's state in one CTA, or in two that hold
 * one half of the value columns each (faster per chunk, at the cost of a
 * producer SM per pair: the library takes the halves when that raises the
 * grid's sustained chunk rate, i.e. for the few pairs of long single
 * sequences).  CHUNKED lets the library choose; CHUNKED_PER_STATE,
 * CHUNKED_COOP (one CTA per pair) and CHUNKED_COOP_HALVES (two) force one.
 * A forced choice that does not apply returns KDA_ERR_UNSUPPORTED.
 *
 * The chunked algorithm scales its operands by exp(+-(G_r - a)), G_r the
 * in-chunk cumulative log-decay and a its value at mid-chunk, which stays
 * within fp32 range while one channel's decay within half a chunk is at most
 * 80 nats.  A (sequence, head) that goes beyond is recomputed in the same
 * call, outputs, snapshots and final state, by the exact token-recurrent
 * kernel (launched after every chunked prefill; its CTAs return at once when
 * no unit needs it), so every finite gate gives the recurrence's result. */
typedef enum {
  KDA_ALGO_AUTO = 0,
  KDA_ALGO_RECURRENT = 1,
  KDA_ALGO_CHUNKED = 2,
  KDA_ALGO_CHUNKED_PER_STATE = 3,
  KDA_ALGO_CHUNKED_COOP = 4,
  KDA_ALGO_CHUNKED_COOP_HALVES = 5
} kda_algo;

typedef struct {
  int32_t B;              /* prefill: sequences in the packed batch; decode: N sequences */
  int32_t T_total;        /* prefill: cu_seqlens[B]; decode: N * n_tok */
  int32_t H;              /* heads */
  int32_t dk, dv;         /* key / value head dims: each one of 16, 32, 64, 128 */
  int32_t n_slots;        /* state_pool slots */
  int32_t dtype;          /* kda_dtype of q, k, v, g, beta, out */
  int32_t algo;           /* kda_algo (prefill only) */
  int64_t snaps_capacity; /* prefill: snapshots the snaps buffer holds */
  void *stream;           /* cudaStream_t */
  void *workspace;        /* device scratch: >= kda_workspace_bytes(this), 256-byte aligned,
                             ZERO-FILLED ONCE after allocation; reusable across calls that
                             are ordered on one stream; never shared by concurrent calls */
  size_t workspace_bytes;
  void *ev_begin;         /* optional cudaEvent_t recorded on stream just before the main
                             compute kernel of the call (NULL: none); for timing */
  void *ev_end;           /* optional cudaEvent_t recorded just after it */
} kda_args;

/*
 * Varlen chunked prefill with copy-on-write resume and state snapshots.
 *
 * Serving semantics follow the hybrid prefix cache of the Day-0 integration
 * page: "Separating Physical Blocks, Scheduler Alignment, and Prefix Matching"
 * (a cached state is copied into a private destination before extension;
 * valid states are registered at fine prefix boundaries) and "Interval-Based
 * and Marconi-Style Retention" (checkpoints at a fixed token interval, the
 * prompt boundary always kept).
 *
 * q, k, g    [T_total][H][dk]   dtype        packed tokens of B sequences
 * v          [T_total][H][dv]   dtype
 * beta       [T_total][H]       dtype
 * cu_seqlens [B+1]              int32        cu[0] = 0, non-decreasing, cu[B] = T_total;
 *                                            sequence b owns tokens [cu[b], cu[b+1])
 * init_slots [B][2]             int32        {src, dst}: sequence b starts from
 *                                            state_pool[src] (src = -1: zero state) and its
 *                                            final state is written to state_pool[dst].
 *                                            src is only read (unless src == dst, which
 *                                            extends in place).  dst slots must be distinct
 *                                            and no src may be another sequence's dst.
 * state_pool [n_slots][H][dk][dv] fp32       read at src, written at dst; all other slots
 *                                            are left bit-identical
 * out        [T_total][H][dv]   dtype        o_t (round-to-nearest-even for bf16)
 * snap_interval                              0, or a positive interval: snapshot j of
 *                                            sequence b is its state after (j+1)*interval
 *                                            tokens of this segment (segment-relative)
 * snaps      [n_snaps][H][dk][dv] fp32       snapshots, sequence-major then position:
 *                                            sequence b's start at the exclusive scan of
 *                                            floor(L_b / interval); NULL when interval == 0
 *                                            (or when a->snaps_capacity == 0);
 *                                            n_snaps = kda_snapshot_count(...)
 *                                            <= a->snaps_capacity
 * Callers align segment starts to the interval (a scheduler invariant) so that
 * segment-relative snapshots fall on absolute prefix boundaries.
 */
kda_status kda_prefill_varlen(const void *q, const void *k, const void *v, const void *g,
                              const void *beta, const int32_t *cu_seqlens,
                              const int32_t *init_slots, float *state_pool, void *out,
                              int32_t snap_interval, float *snaps, const kda_args *a);

/*
 * kda_prefill_varlen with a snapshot retention map: the same computation, but
 * each snapshot either goes straight into a pool slot or is not written.
 *
 * Retention follows "Kimi K3 + vLLM: Inside the Day-0 Production
 * Integration", section "Interval-Based and Marconi-Style Retention": a
 * serving scheduler keeps states at a fixed token interval (the prompt
 * boundary always) or only for prefixes seen a second time, so most interval
 * positions of a long prompt need no state.  The scheduler's decision, made
 * before the call, is the map; the final state still always goes to dst.
 *
 * snap_slots [n_snaps] int32 (device)  for snapshot s, numbered as for the
 *                                      snaps buffer of kda_prefill_varlen
 *                                      (sequence-major, then position):
 *                                      -1 = not retained, else the pool slot
 *                                      that receives the state, written like a
 *                                      final state ([H][dk][dv] fp32)
 * a->snaps_capacity                    entries of snap_slots (>= n_snaps)
 * All other arguments are those of kda_prefill_varlen.  A retained slot must
 * be in [0, n_slots) and may not be any sequence's src or dst nor another
 * retained snapshot's slot; a violation is a device-side error (bit 1 or 2)
 * and the sequence that owns the offending snapshot is skipped.
 */
kda_status kda_prefill_varlen_retain(const void *q, const void *k, const void *v, const void *g,
                                     const void *beta, const int32_t *cu_seqlens,
                                     const int32_t *init_slots, float *state_pool, void *out,
                                     int32_t snap_interval, const int32_t *snap_slots,
                                     const kda_args *a);

/*
 * Single- and multi-token decode in place on the state pool (the fused decode
 * step of "Kimi K3 on vLLM: Up to 370 Tokens/sec", section "Kimi Delta
 * Attention: a hybrid recurrent + full-attention stack", and the multi-token
 * verify pass used under speculative decoding).
 *
 * q, k, g    [N*n_tok][H][dk]   dtype        sequence n owns rows [n*n_tok, (n+1)*n_tok)
 * v, out     [N*n_tok][H][dv]   dtype
 * beta       [N*n_tok][H]       dtype
 * slot_ids   [N]                int32        distinct slots in [0, n_slots)
 * state_pool [n_slots][H][dk][dv] fp32       slot_ids[n] advanced in place by n_tok tokens
 * n_tok      >= 1
 * per_tok_states [N][n_tok][H][dk][dv] fp32 or NULL: the state after each token, for
 *                                            rollback of rejected draft tokens (copy
 *                                            per_tok_states[n][a-1] into the slot)
 * a->B = N, a->T_total = N * n_tok.
 */
kda_status kda_decode(const void *q, const void *k, const void *v, const void *g,
                      const void *beta, const int32_t *slot_ids, float *state_pool, void *out,
                      int32_t n_tok, float *per_tok_states, const kda_args *a);

/*
 * Speculative verify with an in-kernel commit of the previous verify step.
 *
 * Under speculative decoding every step verifies 1 + d tokens per sequence
 * (the last accepted token and d draft tokens; the DSpark speculator of
 * "Kimi K3 on vLLM: Up to 370 Tokens/sec" proposes 7, the vLLM recipe page
 * for Kimi-K3 configures 8).  How many of them
 * are accepted is known only after the verify pass, so kda_decode must either
 * dump the state after every verified token (per_tok_states) or advance the
 * slot past tokens that may be rejected.  This call instead carries the
 * commit into the next step: sequence n
 *   1. reads state_pool[slot_ids[n]] -- the state before the previous verify
 *      step's tokens;
 *   2. replays the first accepted_prev[n] of those tokens (rows
 *      n*n_prev + j, j < accepted_prev[n], of k_prev, v_prev, g_prev,
 *      beta_prev -- the previous step's own k, v, g, beta, which the caller
 *      keeps) and, if accepted_prev[n] > 0, writes the result into the slot:
 *      the committed state;
 *   3. runs this step's n_tok tokens (rows n*n_tok + j of q, k, v, g, beta)
 *      from the committed state and writes their outputs o_t = S_t^T q_t to
 *      out.  The slot is NOT advanced past the committed state: these tokens
 *      are next call's "previous step".
 * One state is read and at most one written per (sequence, head) and step,
 * instead of n_tok + 1 writes with per-token states.
 *
 * q, k, g          [N*n_tok][H][dk]  dtype   this step's tokens (may be NULL when n_tok == 0)
 * v, out           [N*n_tok][H][dv]  dtype
 * beta             [N*n_tok][H]      dtype
 * slot_ids         [N]               int32   distinct slots in [0, n_slots)
 * state_pool       [n_slots][H][dk][dv] fp32 slot_ids[n] receives the committed state
 * n_tok            >= 0 (0: commit only, nothing is verified)
 * k_prev, g_prev   [N*n_prev][H][dk] dtype   the previous step's tokens (NULL when n_prev == 0)
 * v_prev           [N*n_prev][H][dv] dtype
 * beta_prev        [N*n_prev][H]     dtype
 * accepted_prev    [N]               int32   in [0, n_prev]: tokens of the previous step
 *                                            kept for sequence n (NULL when n_prev == 0);
 *                                            a value outside the range is a device-side
 *                                            error (bit 64) and that sequence's slot and
 *                                            outputs are left unwritten
 * n_prev           >= 0 (0: nothing to commit; the slot is only read)
 * a->B = N, a->T_total = N * n_tok.  per-token states are not produced here.
 */
kda_status kda_decode_spec(const void *q, const void *k, const void *v, const void *g,
                           const void *beta, const int32_t *slot_ids, float *state_pool,
                           void *out, int32_t n_tok, const void *k_prev, const void *v_prev,
                           const void *g_prev, const void *beta_prev,
                           const int32_t *accepted_prev, int32_t n_prev, const kda_args *a);

/*
 * kda_decode without a workspace, for callers that may not allocate device
 * memory: code inside a framework that owns every device buffer through its
 * own pool and hands a plugin only the step's tensors, or code on a latency
 * path where cudaMalloc is not allowed because it can synchronise the whole
 * device.  (The pages describe no such entry point; it exists for those
 * callers only.)
 *
 * Same arguments and results as kda_decode, restricted to dk = dv = 128;
 * a->workspace and a->workspace_bytes are ignored.  The scratch the decode
 * kernel needs (its duplicate-slot claim table) is a fixed array inside
 * libkda.so: every GPU that loads the library holds it (2 MiB + 256 bytes)
 * until the process exits, and it covers n_slots * H <= 131072 states; larger
 * pools are refused with KDA_ERR_INVALID_ARG before anything is launched.
 * This call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine).
 *
 * err_bits: NULL, or a caller-owned device uint32 that the kernel ORs the
 * device-side check bits into (same bits as kda_device_status reports); the
 * caller clears it.  With NULL the bits go to a word nobody reads: a slot id
 * out of range or a duplicate slot then skips that sequence with no way for
 * the caller to notice, so pass err_bits unless the slots are known valid.
 *
 * The first call on each device looks up the array's device address on the
 * current device (cudaGetSymbolAddress); make that first call before any
 * stream capture.  Every call shares the one array and leaves its contents
 * behind (claims are stamped with a per-device call count, so nothing needs
 * clearing; when that 32-bit count wraps, after 2^32 - 1 calls on a device,
 * the call clears the array once with a memset on its stream); calls that
 * overlap on the GPU race on it and may miss a duplicate slot, so order them
 * on one stream.
 */
kda_status kda_decode_noalloc(const void *q, const void *k, const void *v, const void *g,
                              const void *beta, const int32_t *slot_ids, float *state_pool,
                              void *out, int32_t n_tok, float *per_tok_states, uint32_t *err_bits,
                              const kda_args *a);

/*
 * The layer around the recurrence: short causal convolution in, gated RMSNorm
 * out ("Kimi K3 + vLLM: Inside the Day-0 Production Integration": a KDA layer
 * keeps "a short causal convolution state" beside its matrix state, section
 * "Kimi Delta Attention: When Prefix Caching Meets Recurrent State", and its
 * fused decode kernel folds the causal convolution, the recurrent state
 * update, the gating and the RMSNorm into one launch, section "Separate
 * Prefill/Decode Code Paths"; the vLLM recipe page for Kimi-K3 fuses the KDA
 * output RMSNorm and its sigmoid gate).  Per (sequence, head), token t:
 *
 *     y~_t[c] = act(sum_i conv_w[h][c][i] * x[t - (W-1) + i][c])   c over [q | k | v]
 *     q_t = y~_q / |y~_q| / sqrt(dk),  k_t = y~_k / |y~_k|,  v_t = y~_v
 *     (the recurrence of kda_prefill_varlen / kda_decode on q, k, v, g, beta)
 *     out_t = o_t / sqrt(mean(o_t^2) + norm_eps) * norm_w * sigmoid(gate_t)
 *
 * where x are the raw (pre-convolution) inputs, W = conv_width taps, and the
 * W-1 inputs before a segment come from the slot's convolution state (zeros
 * for a sequence without a source slot).
 */
typedef struct {
  const void *gate;     /* [T][H][dv] a->dtype: output gate logits */
  const float *conv_w;  /* [H][2 dk + dv][conv_width] fp32: taps per channel, channels in
                           the order q (dk), k (dk), v (dv); tap conv_width-1 multiplies
                           the current token, tap i the token conv_width-1-i steps back */
  const float *norm_w;  /* [dv] fp32: RMSNorm weight, shared by the heads */
  void *conv_pool;      /* [n_slots][H][2 dk + dv][conv_width - 1] a->dtype: per channel
                           its last conv_width-1 raw inputs, oldest first (channel-major,
                           the "DS" layout); indexed by the same slots as state_pool */
  int32_t conv_width;   /* 4 (the only width supported) */
  int32_t conv_act;     /* 0: no activation after the convolution, 1: SiLU */
  float norm_eps;       /* RMSNorm epsilon, >= 0 */
  int32_t reserved;     /* 0 */
} kda_fused_args;

/* Scratch bytes kda_prefill_varlen_fused needs for these sizes (uses T_total,
 * H, dk, dv, dtype): the convolved q, k, v and the recurrence's outputs. */
size_t kda_fused_scratch_bytes(const kda_args *a);

/*
 * kda_prefill_varlen with the layer around it.  xq, xk [T][H][dk] and xv
 * [T][H][dv] are the raw inputs; the convolution of sequence b starts from
 * conv_pool[src_b] (zeros when src_b = -1) and its new state (the last
 * conv_width-1 raw inputs of [old state; segment]) goes to conv_pool[dst_b],
 * copy-on-write exactly like state_pool.  out [T][H][dv] receives the gated
 * RMSNorm of the recurrence's outputs; snapshots and final states are those
 * of the recurrence on the convolved q, k, v (the convolution state at a
 * snapshot is the W-1 raw inputs before that position, which the caller
 * holds).  scratch: device memory of at least kda_fused_scratch_bytes(a)
 * bytes, 16-byte aligned, caller-owned, not shared by concurrent calls.
 * Six kernels in stream order: plan, convolution, convolution states,
 * prefill, exact recomputation (as in kda_prefill_varlen), gated RMSNorm.
 * Same shapes and errors as kda_prefill_varlen.
 */
kda_status kda_prefill_varlen_fused(const void *xq, const void *xk, const void *xv,
                                    const void *g, const void *beta, const int32_t *cu_seqlens,
                                    const int32_t *init_slots, float *state_pool, void *out,
                                    int32_t snap_interval, float *snaps, const kda_fused_args *f,
                                    void *scratch, size_t scratch_bytes, const kda_args *a);

/*
 * kda_decode with the layer around it, in ONE kernel launch (dk = dv = 128):
 * per token the convolution from the slot's convolution state, the
 * normalisation of q and k, the recurrence step in place on the slot and the
 * gated RMSNorm of the output; the slot's convolution state advances with
 * its matrix state.  per_tok_states as in kda_decode (the convolution state
 * after token j is the last conv_width-1 raw inputs up to j, which the caller
 * holds).  Arguments otherwise as kda_decode, raw inputs in place of q, k, v.
 */
kda_status kda_decode_fused(const void *xq, const void *xk, const void *xv, const void *g,
                            const void *beta, const int32_t *slot_ids, float *state_pool,
                            void *out, int32_t n_tok, float *per_tok_states,
                            const kda_fused_args *f, const kda_args *a);

/* Workspace bytes the calls need for these sizes (uses B, H, n_slots).
 * The snapshot interval does not change the size: snapshot offsets live in
 * the per-sequence plan, whose size depends on B only.
 *
 * Stamps that calls leave in a workspace carry a per-workspace call count;
 * when that 32-bit count wraps (after 2^32 - 1 calls on one workspace) the
 * call clears the workspace once (a memset on its stream, keeping the error
 * word) before reusing the count. */
size_t kda_workspace_bytes(const kda_args *a);

/* Number of snapshots a prefill writes: sum over b of floor(L_b / snap_interval),
 * from a HOST copy of cu_seqlens.  Returns -1 on a bad argument. */
int64_t kda_snapshot_count(const int32_t *cu_seqlens_host, int32_t B, int32_t snap_interval);

/* Synchronises a->stream, then returns KDA_OK, KDA_ERR_DEVICE_CHECK or
 * KDA_ERR_TIMEOUT for any device-side error recorded in a->workspace since the
 * last call to this function, and clears the record.  If detail is not NULL
 * it receives the raw error bits (1 slot out of range, 2 duplicate slot or a
 * source that is another sequence's destination, 4 bad cu_seqlens, 8 snapshot
 * buffer too small, 16 wait timeout, 64 an accepted length of kda_decode_spec
 * outside [0, n_prev]; bit 32 is not used).
 *
 * Only a->stream and a->workspace are read.  (The status word lives in the
 * workspace, so the call takes the kda_args that name it rather than only a
 * stream; several workspaces on one stream are queried separately.) */
kda_status kda_device_status(const kda_args *a, uint32_t *detail);

/* Human-readable name of a status code (static string). */
const char *kda_status_string(kda_status s);

/* Kernel launches issued by the last successful compute call on this host
 * thread (for launch accounting). */
int32_t kda_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
