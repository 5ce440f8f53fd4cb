/*
 * gdn.h -- C ABI of libgdn: the Gated DeltaNet layer over a slot-indexed pool
 * of independent per-request recurrent states, for NVIDIA GB300 (sm_103a).
 *
 * Why a pool: one recurrent state per layer forces concurrent requests to run
 * one after another (baseRT issue #31, "Summary" and "Measurement": four
 * requests take four times as long as one).  The fix that page proposes is an
 * outer slot dimension on the state cache and a slot index in the GDN kernels
 * ("Why this looks tractable").  This library is that: a pool of
 * [n_layers][n_slots] states, and kernels that take a list of slot ids.
 *
 * Per value head h of a slot, with key head h' = h / (h_v / h_k), each token
 * applies the gated delta rule
 *     S <- alpha * S (I - beta k k^T) + beta v k^T,      o = scale * S q
 * where S is [dv][dk] (float32 arithmetic), q and k are L2-normalised inside the kernels
 * (x / sqrt(sum x^2 + 1e-6)), alpha = exp(g) with g <= 0 given per token and
 * value head, and o is read from the updated state.
 *
 * Conventions for every call:
 *  - All array arguments are DEVICE pointers (cudaMalloc / torch memory),
 *    owned by the caller; the library never frees them.  Index arrays
 *    (slot_ids, cu_seqlens, advance, accept_len) are int32 device arrays too,
 *    so a call needs no host round trip and can be recorded into a stream.
 *  - Every compute call is asynchronous on `stream` (NULL = legacy default
 *    stream).  The returned status covers argument validation and the launch.
 *  - With desc.host_checks != 0 the library additionally copies the index
 *    arrays to the host (synchronising `stream`) and validates them: slot ids
 *    in range and not repeated, cu_seqlens[0] == 0 and non-decreasing and
 *    ending at total_tokens, 0 <= advance/accept_len <= the sequence length;
 *    it also checks that every pointer is device-accessible.  A failed check
 *    launches nothing.
 *  - With host checks off, kernels still guard their indexes: an entry with a
 *    slot id out of range or a malformed length is skipped and a bit is set in
 *    the pool's device error word (see gdn_pool_get_error).  Kernels never
 *    trap.  Repeated slot ids in one call are not detected on the device and
 *    give unspecified results for those slots.
 *  - n == 0 / empty sequences are valid no-ops.
 *  - The state layout is [n_layers][n_slots][h_v][dv][dk] in the pool's
 *    state_dtype (float32 unless chosen otherwise) and the conv cache
 *    [n_layers][n_slots][conv_ch][conv_k-1] in conv_dtype, oldest input
 *    first; both are plain caller memory, so a state can be written, read,
 *    copied or saved with ordinary memcpy.
 *  - Not thread-safe per pool: calls on one pool from several host threads
 *    must be serialised by the caller.  Calls on different streams that touch
 *    the same slot race.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *gdn_stream; /* identical to cudaStream_t */

typedef enum {
  GDN_OK = 0,
  GDN_ERR_ARG = 1,         /* null pointer, negative count, bad layer, misaligned pointer */
  GDN_ERR_SLOT = 2,        /* slot id outside [0, n_slots) (host check) */
  GDN_ERR_DUP_SLOT = 3,    /* a slot id repeated within one call (host check) */
  GDN_ERR_DTYPE = 4,       /* dtype not supported for this argument */
  GDN_ERR_SIZE = 5,        /* buffer too small, malformed cu_seqlens, length/T out of range */
  GDN_ERR_UNSUPPORTED = 6, /* a shape the library has no kernel for (see gdn_pool_create) */
  GDN_ERR_CUDA = 7         /* a CUDA runtime call failed (gdn_last_error_message has it) */
} gdn_status;

/* Element types.  Activations (q, k, v, g, beta, x, y, o) and the conv cache
 * are GDN_F32 or GDN_BF16; the recurrent state may also be GDN_F16. */
typedef enum { GDN_F32 = 0, GDN_BF16 = 1, GDN_F16 = 2 } gdn_dtype;

/* Bits of the pool's device error word. */
#define GDN_DEVERR_SLOT 1u   /* an entry with an out-of-range slot id was skipped */
#define GDN_DEVERR_SEQ 2u    /* an entry with a malformed cu_seqlens range was skipped */
#define GDN_DEVERR_COUNT 4u  /* an advance/accept_len outside [0, length] was clamped */
#define GDN_DEVERR_TIMEOUT 8u /* a bounded wait on an asynchronous copy gave up; outputs of
                                 that CTA are missing (never expected; reported, not hung) */

/* Shape of every GDN layer in the pool.  Supported: dk in {16, 32, 64, 128},
 * dv a multiple of 4 (<= 4096), h_v a multiple of h_k, 2 <= conv_k <= 8,
 * conv_ch >= 1, conv_dtype GDN_F32 or GDN_BF16. */
typedef struct {
  int32_t n_layers;
  int32_t n_slots;
  int32_t h_v;        /* value heads (one state per value head) */
  int32_t h_k;        /* key/query heads; value head h uses key head h / (h_v / h_k) */
  int32_t dk;         /* key head dim = state columns */
  int32_t dv;         /* value head dim = state rows */
  int32_t conv_ch;    /* channels of the short conv */
  int32_t conv_k;     /* conv width; the cache keeps conv_k - 1 inputs */
  gdn_dtype conv_dtype; /* dtype of conv inputs/outputs and of the cache */
  int32_t host_checks;  /* nonzero: validate index arrays on the host (syncs) */
  /* Upper bound (bytes) on the workspace one gdn_prefill_chunked call may take
   * for its two-launch tensor-core path (about 32 KiB per 64-token chunk per
   * value head); 0 means 8 GiB.  Calls that would need more, or whose
   * workspace cannot be allocated, run the single-launch kernel instead. */
  uint64_t prefill_workspace_max;
  /* Storage type of the recurrent state: GDN_F32, or a half-precision state
   * (GDN_BF16 / GDN_F16) that halves the state's memory and its HBM traffic
   * (baseRT issue #31, "Why this looks tractable": the gdn_mp_factor_f16 /
   * gdn_mp_scan_f16 kernels; the pages do not say what they compute, and the
   * reading used here is half-precision storage with float32 arithmetic).  A
   * kernel widens the stored state to float32, keeps it in float32 for the
   * whole call, and rounds it to nearest-even once when it writes it back (a
   * decode step: every token; a prefill call: at the end of each sequence
   * and at each checkpoint; a verify: at commit).  Every entry point accepts
   * such a pool; chunked prefill runs its two-launch tensor-core path where
   * that applies (dk = dv = 128 with a workspace) and the token-by-token
   * kernel otherwise, and verify runs its CUDA-core kernel. */
  gdn_dtype state_dtype;
} gdn_pool_desc;

/* Per-token inputs of the recurrence for `tokens` tokens.
 *   q, k  [tokens][h_k][dk]  token stride ld_qk elements (0: h_k*dk)
 *   v     [tokens][h_v][dv]  token stride ld_v elements  (0: h_v*dv)
 *   g     [tokens][h_v]      log of the decay, alpha = exp(g) (g <= 0 expected)
 *   beta  [tokens][h_v]      delta-rule write strength
 * All five have type `dtype`.  Each head row must start 16-byte aligned for
 * GDN_F32 and 8-byte aligned for GDN_BF16 (base pointers and strides). */
typedef struct {
  const void *q, *k, *v, *g, *beta;
  int64_t ld_qk, ld_v;
  gdn_dtype dtype;
} gdn_qkv;

typedef struct gdn_pool gdn_pool;

/* Bytes of state / conv-cache memory a pool with this shape needs. */
size_t gdn_pool_state_bytes(const gdn_pool_desc *desc);
size_t gdn_pool_conv_bytes(const gdn_pool_desc *desc);

/* State cache create (baseRT issue #31, "Why this looks tractable":
 * GDNStateCache::create sized by layers, heads, head dim and conv_k, plus the
 * slot dimension that page asks for).  Wraps caller memory: state_mem and
 * conv_mem (256-byte aligned device memory of at least the sizes above) are
 * NOT cleared -- call gdn_pool_reset for new requests, or write states
 * directly.  The pool allocates a small zeroed device array (the error word
 * and 4 bytes per layer, slot and key head for gdn_decode_step_conv) and owns
 * a stream-ordered memory pool from which chunked prefill takes its
 * workspace (kept for reuse until gdn_pool_destroy).  On success *out
 * receives the handle. */
gdn_status gdn_pool_create(const gdn_pool_desc *desc, void *state_mem, size_t state_bytes,
                           void *conv_mem, size_t conv_bytes, gdn_pool **out);

/* Zero the state and conv cache of slots slot_ids[0..n) in every layer
 * (ai-infra-handbooks, "Project: adding the hybrid model Qwen3.5", "What to
 * do", State row: a new request starts from zero; a reused slot is cleared).
 * Other slots are not touched. */
gdn_status gdn_pool_reset(gdn_pool *pool, const int32_t *slot_ids, int32_t n, gdn_stream stream);

/* Copy the state and conv cache of slot src_slots[i] into slot dst_slots[i],
 * in every layer (state checkpoints for prefix caching: a recurrent state can
 * only be saved and copied whole -- ai-infra-handbooks, "Project: adding the
 * hybrid model Qwen3.5", "What to do", Prefix cache row, and "Why it is worth
 * doing").  Destinations must be distinct and must not also be sources (host
 * checks reject it; without them the result is unspecified). */
gdn_status gdn_pool_copy(gdn_pool *pool, const int32_t *src_slots, const int32_t *dst_slots,
                         int32_t n, gdn_stream stream);

/* State cache destroy (baseRT issue #31, "Why this looks tractable":
 * GDNStateCache::destroy).  Releases the handle, its error word and tickets
 * and its workspace memory pool (caller memory is left alone).
 * Synchronises the device before freeing. NULL is a no-op. */
gdn_status gdn_pool_destroy(gdn_pool *pool);

/* Wait for the device, return the device error word (GDN_DEVERR_* bits
 * accumulated since the last call) in *dev_err and clear it.  The pages have
 * no counterpart: baseRT issue #31 ("Why this looks tractable") names only
 * GDNStateCache::{create,destroy}; the word is how kernels that never trap
 * report a skipped entry or an expired wait. */
gdn_status gdn_pool_get_error(gdn_pool *pool, uint32_t *dev_err);

/* Test hook (no counterpart on the pages; 0 in normal use).  With
 * GDN_TEST_DECODE_WAIT_TIMEOUT set, the decode kernels of this pool
 * (gdn_decode_step, gdn_decode_step_conv) make each CTA's copy barrier expect
 * 16 bytes more than its state-tile copy delivers: the copy lands, the
 * bounded wait runs out (a second or two), the CTA sets GDN_DEVERR_TIMEOUT,
 * leaves its state rows and its rows of o unwritten and exits with no copy
 * in flight.  It exercises the error path of the waits without a fault; flags
 * other than that bit are GDN_ERR_ARG. */
#define GDN_TEST_DECODE_WAIT_TIMEOUT 1u
gdn_status gdn_pool_set_test_flags(gdn_pool *pool, uint32_t flags);

/* Causal depthwise conv of width conv_k followed by SiLU (baseRT issue #31,
 * "Why this looks tractable": gdn_conv_silu), on each sequence's slot cache.
 * Sequence i is tokens cu_seqlens[i] .. cu_seqlens[i+1]-1 of x and uses the
 * cache of slot slot_ids[i]; cu_seqlens == NULL means one token per sequence
 * (decode).  For each token t and channel c:
 *     y[t][c] = silu(sum_j w[c][j] * win[j] + bias[c]),
 *     win = (cache[c][0..conv_k-2], x[t-conv_k+1..t][c]) restricted to the
 *     conv_k most recent inputs, w[c][conv_k-1] on the current token.
 * x, y: [total_tokens][conv_ch] in the pool's conv_dtype with row strides
 * ld_x / ld_y elements (0: conv_ch); w: [conv_ch][conv_k] float32;
 * bias: [conv_ch] float32 or NULL.  y may be NULL (cache update only).
 * The cache then holds the conv_k-1 raw inputs preceding token advance[i] of
 * the sequence (advance == NULL: the whole sequence), so speculative tokens
 * can be run without moving the cache and committed later.
 * max_seqlen: an upper bound of the sequence lengths, used only to size the
 * grid (any value >= 1 is correct; a tight one is fastest). */
gdn_status gdn_conv_silu(gdn_pool *pool, int32_t layer, const int32_t *slot_ids,
                         const int32_t *cu_seqlens, int32_t n_seqs, int32_t total_tokens,
                         int32_t max_seqlen, const void *x, int64_t ld_x, gdn_dtype x_dtype,
                         const float *w, const float *bias, void *y, int64_t ld_y,
                         const int32_t *advance, gdn_stream stream);

/* One decode token for each of n active slots (baseRT issue #31, "Why this
 * looks tractable": gdn_recurrence, with the slot index that page asks for).
 * Token i of `in` belongs to slot slot_ids[i]; every head of that slot's
 * state in `layer` is read once and written once.  o: [n][h_v][dv] in
 * o_dtype (GDN_F32 or GDN_BF16), read from the updated state. */
gdn_status gdn_decode_step(gdn_pool *pool, int32_t layer, const int32_t *slot_ids, int32_t n,
                           const gdn_qkv *in, void *o, gdn_dtype o_dtype, float scale,
                           gdn_stream stream);

/* The whole decode step of one layer in one call: gdn_conv_silu in decode
 * mode (one token per slot) on x, writing y, then gdn_decode_step reading q,
 * k and v out of y (b70-optimization-lab research plan, "What the research
 * found": batch-1 decode is latency- and launch-bound, so conv, SiLU and the
 * q/k norm are folded into the decode call).  y: [n][conv_ch] in `dtype` with
 * row stride ld_y (0: conv_ch), split as q = y[:, 0 : h_k*dk],
 * k = y[:, h_k*dk : 2*h_k*dk], v = y[:, 2*h_k*dk :]; the pool's conv_ch must
 * be 2*h_k*dk + h_v*dv (else GDN_ERR_SIZE).  x: [n][conv_ch] with row stride
 * ld_x (0: conv_ch); x, y, g and beta are all in `dtype`, which must be the
 * pool's conv_dtype (else GDN_ERR_DTYPE); w, bias as in gdn_conv_silu; o, g,
 * beta, scale as in gdn_decode_step.  Results, y, cache and state are those
 * of the two calls made one after the other, bit for bit.
 * Three forms, chosen by size and shape: while the decode grid (h_v *
 * ceil(dv / rows per CTA) CTAs per slot) fits on the device at once, ONE
 * kernel does it all -- each CTA convolves the q/k channels of its key head
 * and the v channels of its state rows itself while its state tile is in
 * flight, and the last of the CTAs sharing a key head (a per-slot ticket in
 * pool memory, no waiting) shifts that head's q/k cache.  Larger calls with
 * dk = 128, a float32 state, h_v / h_k <= 2 and dv a multiple of 32 run ONE
 * kernel with a CTA per (slot, key head) that convolves each channel once
 * while the key head's value-head states stream in.  Other larger calls
 * launch the conv and then the decode as its programmatic dependent launch,
 * which fetches its state tiles (untouched by the conv) before it waits for
 * the conv grid to complete and reads y.  Caller owns every buffer.  An argument or host-check error
 * launches nothing; GDN_ERR_CUDA from the second launch of the two-launch
 * form leaves the conv (cache advanced, y written) launched without its
 * decode. */
gdn_status gdn_decode_step_conv(gdn_pool *pool, int32_t layer, const int32_t *slot_ids,
                                int32_t n, const void *x, int64_t ld_x, const float *w,
                                const float *bias, void *y, int64_t ld_y, const void *g,
                                const void *beta, gdn_dtype dtype, void *o, gdn_dtype o_dtype,
                                float scale, gdn_stream stream);

/* The number of kernel launches gdn_decode_step_conv makes for n active slots
 * on this pool with these dtypes (1: one of the fused forms; 2: the conv and
 * the decode; 0 for n = 0), chosen by the same rule, without launching
 * anything (a not-in-the-pages companion of gdn_decode_step_conv, for callers
 * that count or budget launches, e.g. when sizing a CUDA graph).  *launches:
 * host int32.  Errors: GDN_ERR_ARG (NULL launches, n outside [0, 65535], the
 * pool's device not current), GDN_ERR_DTYPE as in gdn_decode_step_conv,
 * GDN_ERR_CUDA (the occupancy query failed). */
gdn_status gdn_decode_step_conv_launches(gdn_pool *pool, int32_t n, gdn_dtype dtype,
                                         gdn_dtype o_dtype, int32_t *launches);

/* Input projection of the layer (baseRT issue #31, "Why this looks
 * tractable": the gdn_in_proj kernel, named there without its formula; the
 * plain reading is the layer's linear projection of the hidden states):
 *     y[t][n] = sum_h x[t][h] * w[n][h]     for t < tokens, n < n_out,
 * with x [tokens][hidden] and w [n_out][hidden] in bf16 (row strides ld_x,
 * ld_w elements; 0: hidden), float32 accumulation, and y [tokens][n_out] in
 * y_dtype (GDN_F32 or GDN_BF16, rounded to nearest-even; row stride ld_y,
 * 0: n_out).  The rows of w stack whatever the layer projects to (q | k | v
 * for gdn_conv_silu, the output gate, the beta and decay logits); the
 * library applies no activation.  Pointers and row strides must be 16-byte
 * aligned (GDN_ERR_ARG otherwise).  Runs on the tensor cores (tcgen05, TMA
 * tensor maps); the pool supplies the device and the error word
 * (GDN_DEVERR_TIMEOUT if a bounded wait gives up) and is otherwise unused.
 * tokens == 0 is a no-op. */
gdn_status gdn_in_proj(gdn_pool *pool, int64_t tokens, int32_t hidden, int32_t n_out,
                       const void *x, int64_t ld_x, const void *w, int64_t ld_w, void *y,
                       int64_t ld_y, gdn_dtype y_dtype, gdn_stream stream);

/* Output gated RMSNorm of the layer (ai-infra-handbooks Qwen3.5 project, "Why
 * it is worth doing": the model's two kinds of RMSNorm; the formula is not
 * written out there, and the one used is the plain reading): for each of
 * `rows` rows (one token and value head each) of d elements,
 *     y[r][j] = o[r][j] / sqrt(mean_j o[r][j]^2 + eps) * w[j] * silu(z[r][j]).
 * o (the recurrence output), z (the gate), y: [rows][d] contiguous, each in
 * its own dtype (GDN_F32 or GDN_BF16); w: [d] float32; eps >= 0 and finite
 * (a row of zeros needs eps > 0).  y may not overlap o or z.  No pool is
 * involved.  rows == 0 is a no-op; d < 1, a NULL pointer or a bad dtype is
 * GDN_ERR_ARG / GDN_ERR_DTYPE and nothing is launched. */
gdn_status gdn_gated_rmsnorm(int64_t rows, int32_t d, const void *o, gdn_dtype o_dtype,
                             const void *z, gdn_dtype z_dtype, const float *w, float eps,
                             void *y, gdn_dtype y_dtype, gdn_stream stream);

/* Chunked prefill of packed variable-length sequences (b70-optimization-lab
 * research plan, "What the research found": the chunked delta rule with the
 * (I+A)^{-1} UT transform; ai-infra-handbooks Qwen3.5 project, "What to do",
 * State row: the state is carried from chunk to chunk).  Sequence i is tokens
 * cu_seqlens[i] .. cu_seqlens[i+1]-1 and starts from slot slot_ids[i]'s
 * current state, which holds the final state afterwards, so a long prompt
 * can be fed in several calls.  Chunks are 64 tokens; the last one of each
 * sequence may be partial.  o: [total_tokens][h_v][dv] in o_dtype.
 * max_seqlen as for gdn_conv_silu. */
gdn_status gdn_prefill_chunked(gdn_pool *pool, int32_t layer, const int32_t *slot_ids,
                               const int32_t *cu_seqlens, int32_t n_seqs, int32_t total_tokens,
                               int32_t max_seqlen, const gdn_qkv *in, void *o, gdn_dtype o_dtype,
                               float scale, gdn_stream stream);

/* gdn_prefill_chunked that also stores state checkpoints for prefix caching
 * (ai-infra-handbooks, "Project: adding the hybrid model Qwen3.5", "What to
 * do", Prefix cache row: a cached prefix can resume only where a state
 * checkpoint was stored; "Why it is worth doing": a recurrent state is saved
 * and copied whole).  After (j + 1) * ckpt_every tokens of sequence i in this
 * call, the recurrent state of every value head is written into slot
 * ckpt_slots[i * ckpt_per_seq + j] of the same layer (entries < 0: none;
 * ckpt_every a positive multiple of 64, so checkpoints fall on chunk
 * boundaries).  Only the recurrent state is written: the conv window at a
 * boundary is the last conv_k - 1 conv inputs before it, which the caller
 * holds.  Checkpoint slots must differ from the active slots and from each
 * other (host checks reject it; without them an out-of-range slot sets
 * GDN_DEVERR_SLOT and is skipped).  Needs the two-launch path (dk = dv = 128,
 * 16-byte aligned v rows, workspace within prefill_workspace_max):
 * GDN_ERR_UNSUPPORTED otherwise. */
gdn_status gdn_prefill_chunked_ckpt(gdn_pool *pool, int32_t layer, const int32_t *slot_ids,
                                    const int32_t *cu_seqlens, int32_t n_seqs,
                                    int32_t total_tokens, int32_t max_seqlen, const gdn_qkv *in,
                                    void *o, gdn_dtype o_dtype, float scale,
                                    const int32_t *ckpt_slots, int32_t ckpt_per_seq,
                                    int32_t ckpt_every, gdn_stream stream);

/* Token-by-token prefill: the same contract, arguments and results as
 * gdn_prefill_chunked, computed by applying the recurrence to each token in
 * order (baseRT issue #31, "Why this looks tractable": the per-token
 * gdn_recurrence kernel).  It is the reference point the chunked form is
 * measured against and accepts every supported head dim. */
gdn_status gdn_prefill_recurrent(gdn_pool *pool, int32_t layer, const int32_t *slot_ids,
                                 const int32_t *cu_seqlens, int32_t n_seqs, int32_t total_tokens,
                                 int32_t max_seqlen, const gdn_qkv *in, void *o,
                                 gdn_dtype o_dtype, float scale, gdn_stream stream);

/* Speculative verify of T draft tokens per slot without per-position state
 * snapshots (b70-optimization-lab research plan, "What the research found").
 * Draft t of slot slot_ids[i] is token i*T + t of `in`.  o_t ([n][T][h_v][dv],
 * may be NULL) is what t+1 decode steps from the slot's state would output.
 * accept_len (may be NULL; [n] int32 in [0, T]) commits each slot's state to
 * the state after accept_len[i] tokens, written once; 0 leaves it untouched.
 * With accept_len == NULL the pool is only read (verify-then-commit in two
 * calls, the second recomputing from the same inputs).  o and accept_len
 * must not both be NULL.  1 <= T <= 32.  Calls of more than four tokens per
 * slot on the tensor-core path (dk = dv = 128, float32 state) may take a
 * stream-ordered workspace for the staged drafts from the pool's memory pool
 * (within prefill_workspace_max; released on `stream` when the call's work
 * is done); if it cannot be had, the call runs without it. */
gdn_status gdn_spec_verify(gdn_pool *pool, int32_t layer, const int32_t *slot_ids, int32_t n,
                           int32_t T, const gdn_qkv *in, void *o, gdn_dtype o_dtype,
                           const int32_t *accept_len, float scale, gdn_stream stream);

/* Speculative verify with the commit deferred to the next round
 * (b70-optimization-lab research plan, "What the research found": the
 * drafts' inputs are kept and the full state is written back only later).
 * Each slot first replays the first prev_accept[i] of last round's T_prev
 * drafts (`prev`, draft t of slot i at token i*T_prev + t) and commits the
 * state after them; on that committed state it computes the outputs of this
 * round's T drafts (`in`, draft t at token i*T + t) without committing them.
 * o: [n][T][h_v][dv] in o_dtype, required.  One call reads each state once
 * and writes it at most once; a two-phase round (gdn_spec_verify without,
 * then with, accept_len) reads it twice and writes it once.  The caller
 * keeps this round's inputs until the next call, which passes them as
 * `prev` with the accepted counts; gdn_spec_verify with accept_len flushes
 * them without new drafts.  prev and prev_accept are both NULL (no pending
 * drafts: outputs only) or both set; prev_accept: [n] int32 in [0, T_prev];
 * prev and in share one dtype.  T >= 1, T_prev >= 0, T + T_prev <= 32: the
 * pending drafts plus this round's fit one 32-token window.  Workspace as in
 * gdn_spec_verify (staged drafts when T + T_prev > 4). */
gdn_status gdn_spec_verify_deferred(gdn_pool *pool, int32_t layer, const int32_t *slot_ids,
                                    int32_t n, int32_t T, const gdn_qkv *in, void *o,
                                    gdn_dtype o_dtype, int32_t T_prev, const gdn_qkv *prev,
                                    const int32_t *prev_accept, float scale, gdn_stream stream);

/* gdn_prefill_chunked for callers that must not allocate device memory:
 * code running under an allocator that owns the whole GPU (a serving engine
 * that reserves its memory up front), or with a fixed memory budget where an
 * allocation in the middle of a step is not allowed to fail or wait.  The
 * source pages have no counterpart to this entry point.
 * Arguments, results and errors are those of gdn_prefill_chunked.  Where that
 * function would take its workspace from the pool's memory pool (dk = dv =
 * 128), this one uses a 64 MiB array compiled into the library, which every
 * GPU that loads the library holds until the process exits; it calls no
 * allocator.  A call needing more than 64 MiB -- about 32 KiB per 64-token
 * chunk per value head, counting (tokens / 64 + sequences) chunks -- returns
 * GDN_ERR_SIZE and launches nothing.  Each call looks up the array's device
 * address (cudaGetSymbolAddress, which allocates nothing; the first lookup may
 * load the library's device code, so make the first call before any stream
 * capture).  Every call shares the one array: calls whose work
 * overlaps on the GPU (other streams, other threads, other pools of the same
 * device) race on it and must be serialised by the caller. */
gdn_status gdn_prefill_chunked_noalloc(gdn_pool *pool, int32_t layer, const int32_t *slot_ids,
                                       const int32_t *cu_seqlens, int32_t n_seqs,
                                       int32_t total_tokens, int32_t max_seqlen,
                                       const gdn_qkv *in, void *o, gdn_dtype o_dtype, float scale,
                                       gdn_stream stream);

/* Human-readable name of a status, and the detail of the last failure on
 * this host thread (empty string if none). */
const char *gdn_status_string(gdn_status s);
const char *gdn_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
