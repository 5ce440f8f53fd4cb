// Internal kernel-argument structs and launcher declarations of libgdn.
// Host code in gdn_api.cu validates arguments and calls these launchers; each
// launcher lives next to its kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"

#if defined(__CUDACC__)
#define GDN_HD __host__ __device__ __forceinline__
#else
#define GDN_HD inline
#endif

namespace gdn {

constexpr float kL2Eps = 1e-6f;
constexpr int kChunk = 64;          // prefill chunk length
constexpr int kMaxVerifyT = 32;     // drafts per slot in one verify call

struct PoolView {
  float *state;            // [n_layers][n_slots][h_v][dv][dk] of state_dtype (base address)
  void *conv;              // [n_layers][n_slots][conv_ch][conv_k-1]
  unsigned int *err;       // device error word
  int n_layers, n_slots, h_v, h_k, dk, dv, conv_ch, conv_k;
  gdn_dtype conv_dtype;
  unsigned int *ticks;     // [n_layers][n_slots][h_k] tickets of the one-call decode step
  gdn_dtype state_dtype;   // GDN_F32, or GDN_BF16 / GDN_F16 storage (fp32 arithmetic)
  uint32_t test_flags;     // GDN_TEST_* bits (gdn_pool_set_test_flags); 0 in normal use
  GDN_HD int64_t state_slot_elems() const { return (int64_t)h_v * dv * dk; }
  GDN_HD int64_t conv_slot_elems() const { return (int64_t)conv_ch * (conv_k - 1); }
  GDN_HD int state_esz() const { return state_dtype == GDN_F32 ? 4 : 2; }
  // element index of row 0 of head h of (layer, slot)
  GDN_HD int64_t state_head_elem(int layer, int slot, int h) const {
    return ((int64_t)layer * n_slots + slot) * state_slot_elems() + (int64_t)h * dv * dk;
  }
  // address of state element e
  GDN_HD char *state_at(int64_t e) const {
    return reinterpret_cast<char *>(state) + e * state_esz();
  }
};

struct QKV {
  const void *q, *k, *v, *g, *beta;
  int64_t ld_qk, ld_v;     // resolved (never 0)
  gdn_dtype dtype;
};

// Per-slot token range of a call: sequence i covers tokens [tok0, tok0 + len).
struct SeqIndex {
  const int32_t *slot_ids;
  const int32_t *cu_seqlens;   // NULL: one token per sequence
  int n_seqs;
  int total_tokens;            // rows of the packed token arrays
};

// State checkpoints during a chunked prefill: after (j + 1) * every tokens of
// sequence i in the call, the state goes to slot slots[i * per_seq + j] (if
// that entry is >= 0).  every == 0: none.
struct Checkpoints {
  const int32_t *slots;
  int per_seq;
  int every;                   // a multiple of the chunk (64)
};

cudaError_t launch_pool_reset(const PoolView &p, const int32_t *slot_ids, int n,
                              cudaStream_t s);

// y[r][j] = o[r][j] * rsqrt(mean_j o[r][j]^2 + eps) * w[j] * silu(z[r][j]) over
// rows x d contiguous elements.
cudaError_t launch_gated_rmsnorm(const void *o, gdn_dtype ot, const void *z, gdn_dtype zt,
                                 const float *w, float eps, void *y, gdn_dtype yt, int64_t rows,
                                 int d, cudaStream_t s);

// y[t][n] = sum_h x[t][h] * w[n][h]: bf16 x [M][K] (row stride ld_x) and w
// [N][K] (ld_w), float32 accumulation, y [M][N] (ld_y) in y_dtype; timeouts
// set GDN_DEVERR_TIMEOUT in *err.  Rows and strides 16-byte aligned.
cudaError_t launch_in_proj(int64_t M, int N, int K, const void *x, int64_t ld_x, const void *w,
                           int64_t ld_w, void *y, int64_t ld_y, gdn_dtype y_dtype,
                           unsigned int *err, int sm_count, cudaStream_t s);

cudaError_t launch_pool_copy(const PoolView &p, const int32_t *src, const int32_t *dst, int n,
                             cudaStream_t s);

cudaError_t launch_conv_silu(const PoolView &p, int layer, const SeqIndex &seq,
                             int max_seqlen, const void *x, int64_t ld_x,
                             const float *w, const float *bias, void *y, int64_t ld_y,
                             const int32_t *advance, cudaStream_t s);

// The conv kernels let a programmatic dependent launch that follows them start
// as soon as every conv CTA is running.  after_conv: launch the decode kernel
// as such a dependent of the kernel before it on `s`; it fetches its state
// tiles first and reads q, k, v, g and beta only once that kernel has completed
// and its writes are visible.  Only for a decode whose preceding launch on `s`
// is the conv of the same step (it writes neither the state nor slot_ids).
cudaError_t launch_decode(const PoolView &p, const void *tmap, int layer,
                          const int32_t *slot_ids, int n, const QKV &in, void *o,
                          gdn_dtype o_dtype, float scale, cudaStream_t s,
                          bool after_conv = false);

// conv + SiLU, the q/k norm and the decode step of one layer in one kernel
// (one token per slot): y = conv(x) split as q | k | v.  Results, y, cache and
// state equal launch_conv_silu followed by launch_decode, bit for bit.  Needs
// conv_ch == 2*h_k*dk + h_v*dv and p.ticks (all zero between launches).
// CTAs of the decode kernels' grid for n slots, and how many CTAs of the fused
// conv + decode kernel the device (sm_count SMs) holds resident at once.
int64_t decode_grid_ctas(const PoolView &p, int n);
cudaError_t decode_conv_resident_ctas(const PoolView &p, gdn_dtype dtype, gdn_dtype o_dtype,
                                      int sm_count, int64_t *ctas);

cudaError_t launch_decode_conv(const PoolView &p, int layer, const int32_t *slot_ids, int n,
                               const void *x, int64_t ld_x, const float *w, const float *bias,
                               void *y, int64_t ld_y, const void *g, const void *beta,
                               gdn_dtype dtype, void *o, gdn_dtype o_dtype, float scale,
                               cudaStream_t s);

// The same step with one CTA per (slot, key head): each conv channel once,
// the key head's value-head states streamed through a ring of bulk tiles; no
// tickets.  For dk = 128, a float32 state, h_v / h_k <= 2 and dv a multiple
// of 32 (decode_conv_group_ok); the same results, bit for bit.
bool decode_conv_group_ok(const PoolView &p);
cudaError_t launch_decode_conv_group(const PoolView &p, int layer, const int32_t *slot_ids,
                                     int n, const void *x, int64_t ld_x, const float *w,
                                     const float *bias, void *y, int64_t ld_y, const void *g,
                                     const void *beta, gdn_dtype dtype, void *o,
                                     gdn_dtype o_dtype, float scale, cudaStream_t s);

// Speculative verify of T new drafts per slot.  Normal mode: commit at
// accept_len[i] (or after all T with commit_all).  Deferred mode (prev.q set):
// slot i first replays the first prev_accept[i] drafts of the previous round
// (token i*T_prev + t of prev), commits the state right after them, and then
// runs the new drafts for their outputs only.
struct VerifyArgs {
  const int32_t *slot_ids;
  int n;
  int T;
  QKV in;
  const int32_t *accept_len;
  int commit_all;
  QKV prev;                    // prev.q == NULL: no pending drafts
  int T_prev;
  const int32_t *prev_accept;
  float scale;
  float *stage;                // workspace for the staged drafts (tensor-core path), or NULL
};

// tmap: the pool's state tensor map (CUtensorMap), or NULL
cudaError_t launch_verify(const PoolView &p, const void *tmap, int layer, const VerifyArgs &va,
                          void *o, gdn_dtype o_dtype, cudaStream_t s);

cudaError_t launch_verify_tma(const PoolView &p, const void *tmap, int layer,
                              const VerifyArgs &va, void *o, gdn_dtype o_dtype, cudaStream_t s);
// Bytes of the draft-staging workspace the tensor-core verify can use (0: that
// path does not apply).
size_t verify_stage_workspace_bytes(const PoolView &p, const VerifyArgs &va);

cudaError_t launch_prefill_recurrent(const PoolView &p, int layer, const SeqIndex &seq,
                                     const QKV &in, void *o, gdn_dtype o_dtype, float scale,
                                     cudaStream_t s);

cudaError_t launch_prefill_tc(const PoolView &p, int layer, const SeqIndex &seq, const QKV &in,
                              void *o, gdn_dtype o_dtype, float scale, cudaStream_t s);

// Two-launch chunked prefill (dk = dv = 128): key-side tiles of every chunk
// in parallel into `work`, then the state side sequence by sequence.
size_t prefill_split_workspace_bytes(int n_seqs, int total_tokens, int h_v);
cudaError_t launch_prefill_split(const PoolView &p, int layer, const SeqIndex &seq,
                                 const QKV &in, void *o, gdn_dtype o_dtype, float scale,
                                 void *work, cudaStream_t s, const Checkpoints &ck = {});

// Workspace bytes the chunked prefill of this call would use, or 0 when it
// runs without one (not the tensor-core shape, or more than `limit` bytes).
size_t prefill_workspace_bytes(const PoolView &p, const SeqIndex &seq, const QKV &in,
                               size_t limit);

// Chunked prefill; `work` is a device workspace of prefill_workspace_bytes()
// bytes, or NULL (the single-launch kernels, which need none).
cudaError_t launch_prefill(const PoolView &p, int layer, const SeqIndex &seq, const QKV &in,
                           void *o, gdn_dtype o_dtype, float scale, void *work,
                           cudaStream_t s);

}  // namespace gdn
