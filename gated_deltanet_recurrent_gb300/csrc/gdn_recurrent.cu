// Token-by-token prefill: the gated delta rule applied to every token of a
// packed variable-length sequence in order (baseRT issue #31, "Why this looks
// tractable": the per-token gdn_recurrence kernel), with the state carried in
// the slot like the chunked prefill.  It is the reference point the chunked
// form is measured against, and it has no chunk-size or head-dim constraint.
//
// CTA = 32 state rows of one (sequence, value head); each row lives in the
// registers of 4 lanes (dk/4 columns each) for the whole call, in float32
// whatever the pool's storage type (rounded back once, at the end).  Tokens are
// staged 32 at a time (normalised q, k; this CTA's slice of v; alpha, beta);
// per token each row does p = s.k, s = alpha s + beta (v - alpha p) k,
// o = s.q, with 2-shuffle reductions over its 4 lanes.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kRT = 128;  // threads
constexpr int kRR = 32;   // rows per CTA
constexpr int kTB = 32;   // tokens staged per block

template <int DK, typename TI, typename TO>
__global__ void __launch_bounds__(kRT)
    recurrent_prefill_kernel(PoolView p, int layer, SeqIndex seq, QKV in, TO *__restrict__ o,
                             float scale) {
  constexpr int LPR = 4;         // lanes per row
  constexpr int C4 = DK / 16;    // float4 chunks per lane
  __shared__ float4 sk[kTB][DK / 4];
  __shared__ float4 sq[kTB][DK / 4];
  __shared__ float sv[kTB][kRR];
  __shared__ float sal[kTB], sbe[kTB];

  const int si = blockIdx.z, h = blockIdx.y;
  const int r0 = blockIdx.x * kRR;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = seq.slot_ids[si];
  const bool first = blockIdx.x == 0 && h == 0 && tid == 0;
  if (slot < 0 || slot >= p.n_slots) {
    if (first) raise_error(p.err, GDN_DEVERR_SLOT);
    return;
  }
  const int64_t lo = seq.cu_seqlens[si];
  const int64_t hi = seq.cu_seqlens[si + 1];
  if (hi < lo || lo < 0 || hi > seq.total_tokens) {
    if (first) raise_error(p.err, GDN_DEVERR_SEQ);
    return;
  }
  const int len = (int)(hi - lo);
  if (len == 0) return;
  const int hk = h / (p.h_v / p.h_k);
  const int sub = lane % LPR, rho = lane / LPR;
  const int rl = warp * (32 / LPR) + rho;   // row within the CTA
  const int r = r0 + rl;
  const bool live = r < p.dv;
  const int rot = rho % C4;                  // chunk rotation per row (bank spread)
  const gdn_dtype sd = p.state_dtype;
  char *Srow = p.state_at(p.state_head_elem(layer, slot, h) + (int64_t)(live ? r : 0) * DK);

  float4 s[C4];
#pragma unroll
  for (int j = 0; j < C4; ++j) {
    const int cj = ((j + rot) % C4) * LPR + sub;
    s[j] = live ? state_ld4(Srow, 4 * cj, sd) : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  const TI *qg = static_cast<const TI *>(in.q);
  const TI *kg = static_cast<const TI *>(in.k);
  const TI *vg = static_cast<const TI *>(in.v);
  const TI *gg = static_cast<const TI *>(in.g);
  const TI *bg = static_cast<const TI *>(in.beta);
  TO *ob = o + (int64_t)h * p.dv + r;
  const int64_t o_tok = (int64_t)p.h_v * p.dv;

  for (int b0 = 0; b0 < len; b0 += kTB) {
    const int nb = min(kTB, len - b0);
    __syncthreads();  // previous block consumed
    for (int t = warp; t < nb; t += kRT / 32) {
      const int64_t tok = lo + b0 + t;
      float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f), k4 = q4;
      if (lane < DK / 4) {
        q4 = Elem<TI>::load4(qg + tok * in.ld_qk + (int64_t)hk * DK + 4 * lane);
        k4 = Elem<TI>::load4(kg + tok * in.ld_qk + (int64_t)hk * DK + 4 * lane);
      }
      const float qq = group_sum<32>(dot4(q4, q4));
      const float kk = group_sum<32>(dot4(k4, k4));
      if (lane < DK / 4) {
        sq[t][lane] = scale4(rsqrtf(qq + kL2Eps), q4);
        sk[t][lane] = scale4(rsqrtf(kk + kL2Eps), k4);
      }
    }
    for (int e = tid; e < nb * kRR; e += kRT) {
      const int t = e / kRR, rr = e % kRR;
      sv[t][rr] = r0 + rr < p.dv
                      ? Elem<TI>::load1(vg + (lo + b0 + t) * in.ld_v + (int64_t)h * p.dv + r0 + rr)
                      : 0.f;
    }
    if (tid < nb) {
      const int64_t tok = lo + b0 + tid;
      sal[tid] = expf(Elem<TI>::load1(gg + tok * p.h_v + h));
      sbe[tid] = Elem<TI>::load1(bg + tok * p.h_v + h);
    }
    __syncthreads();
#pragma unroll 1
    for (int t = 0; t < nb; ++t) {
      float ak = 0.f;
#pragma unroll
      for (int j = 0; j < C4; ++j) ak += dot4(s[j], sk[t][((j + rot) % C4) * LPR + sub]);
      ak = group_sum<LPR>(ak);
      const float al = sal[t];
      const float d = sbe[t] * (sv[t][rl] - al * ak);
      float aq = 0.f;
#pragma unroll
      for (int j = 0; j < C4; ++j) {
        const int cj = ((j + rot) % C4) * LPR + sub;
        s[j] = axpby4(al, s[j], d, sk[t][cj]);
        aq += dot4(s[j], sq[t][cj]);
      }
      aq = group_sum<LPR>(aq);
      if (live && sub == (t & (LPR - 1))) Elem<TO>::store1(ob + (lo + b0 + t) * o_tok, scale * aq);
    }
  }
  if (live) {
#pragma unroll
    for (int j = 0; j < C4; ++j) {
      const int cj = ((j + rot) % C4) * LPR + sub;
      state_st4<false>(Srow, 4 * cj, s[j], sd);
    }
  }
}

template <int DK, typename TI, typename TO>
struct RecurrentF {
  static cudaError_t run(const PoolView &p, int layer, const SeqIndex &seq, const QKV &in,
                         void *o, float scale, cudaStream_t s) {
    dim3 grid((p.dv + kRR - 1) / kRR, p.h_v, seq.n_seqs);
    recurrent_prefill_kernel<DK, TI, TO><<<grid, kRT, 0, s>>>(p, layer, seq, in,
                                                                static_cast<TO *>(o), scale);
    return cudaGetLastError();
  }
};

}  // namespace

cudaError_t launch_prefill_recurrent(const PoolView &p, int layer, const SeqIndex &seq,
                                     const QKV &in, void *o, gdn_dtype o_dtype, float scale,
                                     cudaStream_t s) {
#define GDN_RT(DK, TI, TO) return RecurrentF<DK, TI, TO>::run(p, layer, seq, in, o, scale, s)
#define GDN_RK(DK)                                                        \
  if (p.dk == DK) {                                                       \
    if (in.dtype == GDN_F32 && o_dtype == GDN_F32) GDN_RT(DK, float, float); \
    if (in.dtype == GDN_F32 && o_dtype == GDN_BF16) GDN_RT(DK, float, bf16); \
    if (in.dtype == GDN_BF16 && o_dtype == GDN_F32) GDN_RT(DK, bf16, float); \
    if (in.dtype == GDN_BF16 && o_dtype == GDN_BF16) GDN_RT(DK, bf16, bf16); \
  }
  GDN_RK(16)
  GDN_RK(32)
  GDN_RK(64)
  GDN_RK(128)
#undef GDN_RK
#undef GDN_RT
  return cudaErrorNotSupported;
}

}  // namespace gdn
