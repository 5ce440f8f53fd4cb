// Chunked prefill of packed variable-length sequences on the slot pool.
//
// One CTA per (sequence, value head) walks its sequence in chunks of 64
// tokens with the [dv][dk] state resident in shared memory (read from the
// slot once at the start, written back once at the end).  Within a chunk of
// n tokens, with local cumulative log-decay G_t and gamma_t = exp(G_t), the
// chunked delta rule (b70-optimization-lab research plan, "What the research
// found": the (I+A)^{-1} UT transform) gives, exactly up to rounding,
//     A[t][i] = beta_t exp(G_t - G_i) k_t.k_i              (i < t)
//     [W | U] = (I + A)^{-1} [diag(beta gamma) K | diag(beta) V]
//     Delta   = U - W S^T                                   (n x dv)
//     O       = diag(gamma) Q S^T + (exp(G_t - G_i) q_t.k_i)_{i<=t} Delta
//     S      <- gamma_n S + Delta^T diag(exp(G_n - G)) K
// The triangular system is solved by forward substitution, one column per
// thread.  A partial last chunk is padded with zero tokens (g = beta = 0,
// q = k = v = 0), which leaves every real output and the state unchanged.
// All arithmetic is float32 on CUDA cores.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kC = kChunk;       // 64
constexpr int kPT = 256;         // threads per CTA

template <int DK, int DV>
struct PrefillSmem {
  static constexpr int KS = DK + 4;            // padded row strides (floats)
  static constexpr int XS = DK + DV + 4;
  static constexpr int AS = kC + 4;
  static constexpr int SS = DK + 4;
  static constexpr int kK = 0;                           // Kc [kC][KS]
  static constexpr int kQ = kK + kC * KS;                // Qc [kC][KS] (later O staging)
  static constexpr int kX = kQ + kC * KS;                // [W | U -> Delta] [kC][XS]
  static constexpr int kA = kX + kC * XS;                // A, then P [kC][AS]
  static constexpr int kS = kA + kC * AS;                // S [DV][SS]
  static constexpr int kG = kS + DV * SS;                // G [kC]
  static constexpr int kGam = kG + kC;                   // gamma [kC]
  static constexpr int kB = kGam + kC;                   // beta [kC]
  static constexpr int kTotal = kB + kC;
  static constexpr size_t bytes = sizeof(float) * kTotal;
};

template <int DK, int DV, typename TI, typename TO>
__global__ void __launch_bounds__(kPT, 1)
    prefill_simt_kernel(PoolView p, int layer, SeqIndex seq, QKV in, TO *__restrict__ o,
                        float scale) {
  using L = PrefillSmem<DK, DV>;
  extern __shared__ float4 smem4[];
  float *sm = reinterpret_cast<float *>(smem4);
  float *Kc = sm + L::kK, *Qc = sm + L::kQ, *X = sm + L::kX, *A = sm + L::kA, *S = sm + L::kS;
  float *G = sm + L::kG, *Gam = sm + L::kGam, *Bt = sm + L::kB;

  const int h = blockIdx.x;
  const int si = blockIdx.y;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int slot = seq.slot_ids[si];
  const bool first = h == 0 && tid == 0;
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
  float *Sg = p.state + ((int64_t)layer * p.n_slots + slot) * p.state_slot_elems() +
              (int64_t)h * DV * DK;

  // state -> shared
  for (int e = tid; e < DV * DK / 4; e += kPT) {
    const int r = e / (DK / 4), c4 = e % (DK / 4);
    reinterpret_cast<float4 *>(S + r * L::SS)[c4] = reinterpret_cast<const float4 *>(Sg)[e];
  }

  const TI *qg = static_cast<const TI *>(in.q);
  const TI *kg = static_cast<const TI *>(in.k);
  const TI *vg = static_cast<const TI *>(in.v);
  const TI *gg = static_cast<const TI *>(in.g);
  const TI *bg = static_cast<const TI *>(in.beta);

  for (int c0 = 0; c0 < len; c0 += kC) {
    const int n = min(kC, len - c0);
    __syncthreads();  // previous chunk fully consumed

    // 1. stage normalised q, k, raw v; g, beta.  Warp per token.
    for (int t = warp; t < kC; t += kPT / 32) {
      const bool real = t < n;
      const int64_t tok = lo + c0 + t;
      float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f), k4 = q4;
      if (real && lane < DK / 4) {
        q4 = Elem<TI>::load4(qg + tok * in.ld_qk + (int64_t)hk * DK + 4 * lane);
        k4 = Elem<TI>::load4(kg + tok * in.ld_qk + (int64_t)hk * DK + 4 * lane);
      }
      const float qq = group_sum<32>(dot4(q4, q4));
      const float kk = group_sum<32>(dot4(k4, k4));
      if (lane < DK / 4) {
        reinterpret_cast<float4 *>(Qc + t * L::KS)[lane] = scale4(rsqrtf(qq + kL2Eps), q4);
        reinterpret_cast<float4 *>(Kc + t * L::KS)[lane] = scale4(rsqrtf(kk + kL2Eps), k4);
      }
      for (int c = lane; c < DV; c += 32)
        X[t * L::XS + DK + c] =
            real ? Elem<TI>::load1(vg + tok * in.ld_v + (int64_t)h * DV + c) : 0.f;
      if (lane == 0) {
        G[t] = real ? Elem<TI>::load1(gg + tok * p.h_v + h) : 0.f;
        Bt[t] = real ? Elem<TI>::load1(bg + tok * p.h_v + h) : 0.f;
      }
    }
    __syncthreads();

    // 2. cumulative log-decay (warp 0, two values per lane)
    if (warp == 0) {
      float a = G[2 * lane], b = G[2 * lane + 1];
      float pair = a + b;
      float incl = pair;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float up = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += up;
      }
      const float excl = incl - pair;
      G[2 * lane] = excl + a;
      G[2 * lane + 1] = incl;
      Gam[2 * lane] = expf(excl + a);
      Gam[2 * lane + 1] = expf(incl);
    }
    __syncthreads();

    // 3. right-hand sides: W part = beta gamma k, U part = beta v
    for (int e = tid; e < kC * (DK + DV); e += kPT) {
      const int t = e / (DK + DV), c = e % (DK + DV);
      X[t * L::XS + c] = c < DK ? Bt[t] * Gam[t] * Kc[t * L::KS + c] : Bt[t] * X[t * L::XS + c];
    }
    // 4. A[t][i] = beta_t exp(G_t - G_i) k_t . k_i for i < t (zero elsewhere)
    {
      const int tr = tid % 16, tc = tid / 16;
      float acc[4][4] = {};
      for (int k4 = 0; k4 < DK / 4; ++k4) {
        float4 kt[4], ki[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) kt[a] = reinterpret_cast<const float4 *>(Kc + (tr + 16 * a) * L::KS)[k4];
#pragma unroll
        for (int b = 0; b < 4; ++b) ki[b] = reinterpret_cast<const float4 *>(Kc + (tc + 16 * b) * L::KS)[k4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) acc[a][b] += dot4(kt[a], ki[b]);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int t = tr + 16 * a, i = tc + 16 * b;
          A[t * L::AS + i] = i < t ? Bt[t] * expf(G[t] - G[i]) * acc[a][b] : 0.f;
        }
    }
    __syncthreads();

    // 5. forward substitution: (I + A) X = RHS, one column per thread
    if (tid < DK + DV) {
      float *col = X + tid;
      for (int t = 1; t < n; ++t) {
        const float *arow = A + t * L::AS;
        float acc0 = col[t * L::XS], acc1 = 0.f;
        int i = 0;
        for (; i + 1 < t; i += 2) {
          acc0 -= arow[i] * col[i * L::XS];
          acc1 -= arow[i + 1] * col[(i + 1) * L::XS];
        }
        if (i < t) acc0 -= arow[i] * col[i * L::XS];
        col[t * L::XS] = acc0 + acc1;
      }
    }
    __syncthreads();

    // 5b. P[t][i] = exp(G_t - G_i) q_t . k_i for i <= t, into A's buffer
    {
      const int tr = tid % 16, tc = tid / 16;
      float acc[4][4] = {};
      for (int k4 = 0; k4 < DK / 4; ++k4) {
        float4 qt[4], ki[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) qt[a] = reinterpret_cast<const float4 *>(Qc + (tr + 16 * a) * L::KS)[k4];
#pragma unroll
        for (int b = 0; b < 4; ++b) ki[b] = reinterpret_cast<const float4 *>(Kc + (tc + 16 * b) * L::KS)[k4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) acc[a][b] += dot4(qt[a], ki[b]);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int t = tr + 16 * a, i = tc + 16 * b;
          A[t * L::AS + i] = i <= t ? expf(G[t] - G[i]) * acc[a][b] : 0.f;
        }
    }

    // 6. Delta = U - W S^T and O = diag(gamma) Q S^T (registers)
    constexpr int NB = DV / 16;
    const int tr = tid % 16, tc = tid / 16;
    float ox[4][NB];
    {
      float dx[4][NB];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < NB; ++b) dx[a][b] = ox[a][b] = 0.f;
      for (int k4 = 0; k4 < DK / 4; ++k4) {
        float4 wt[4], qt[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          wt[a] = reinterpret_cast<const float4 *>(X + (tr + 16 * a) * L::XS)[k4];
          qt[a] = reinterpret_cast<const float4 *>(Qc + (tr + 16 * a) * L::KS)[k4];
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const float4 sv = reinterpret_cast<const float4 *>(S + (tc + 16 * b) * L::SS)[k4];
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            dx[a][b] += dot4(wt[a], sv);
            ox[a][b] += dot4(qt[a], sv);
          }
        }
      }
      __syncthreads();  // all reads of W (and U below) and Q done before overwriting
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int t = tr + 16 * a;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          float *u = X + t * L::XS + DK + tc + 16 * b;
          *u = *u - dx[a][b];
          ox[a][b] *= Gam[t];
        }
      }
    }
    __syncthreads();

    // 7. O += P Delta; stage scale * O in Qc's buffer, then write out coalesced
    {
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int t = tr + 16 * a;
        const float *prow = A + t * L::AS;
        for (int i = 0; i <= t; ++i) {
          const float pv = prow[i];
          const float *drow = X + i * L::XS + DK + tc;
#pragma unroll
          for (int b = 0; b < NB; ++b) ox[a][b] += pv * drow[16 * b];
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) Qc[t * L::KS + tc + 16 * b] = scale * ox[a][b];
      }
    }
    __syncthreads();
    for (int e = tid; e < n * DV; e += kPT) {
      const int t = e / DV, c = e % DV;
      Elem<TO>::store1(o + ((lo + c0 + t) * p.h_v + h) * DV + c, Qc[t * L::KS + c]);
    }

    // 8. S <- gamma_n S + Delta^T diag(exp(G_n - G)) K
    {
      const float gl = G[kC - 1];        // padded tokens carry g = 0
      const float gam_n = Gam[kC - 1];
      constexpr int NA = DV / 16;        // rows v = tr + 16 a
      constexpr int NK = (DK / 4 + 15) / 16;
      for (int kb = 0; kb < NK; ++kb) {
        const int kq = tc + 16 * kb;
        if (kq >= DK / 4) break;
        float4 acc[NA];
#pragma unroll
        for (int a = 0; a < NA; ++a) {
          const float4 s0 = reinterpret_cast<const float4 *>(S + (tr + 16 * a) * L::SS)[kq];
          acc[a] = scale4(gam_n, s0);
        }
        for (int i = 0; i < n; ++i) {
          const float dec = expf(gl - G[i]);
          const float4 ki = scale4(dec, reinterpret_cast<const float4 *>(Kc + i * L::KS)[kq]);
          const float *drow = X + i * L::XS + DK + tr;
#pragma unroll
          for (int a = 0; a < NA; ++a) {
            const float d = drow[16 * a];
            acc[a] = axpby4(1.f, acc[a], d, ki);
          }
        }
#pragma unroll
        for (int a = 0; a < NA; ++a)
          reinterpret_cast<float4 *>(S + (tr + 16 * a) * L::SS)[kq] = acc[a];
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < DV * DK / 4; e += kPT) {
    const int r = e / (DK / 4), c4 = e % (DK / 4);
    reinterpret_cast<float4 *>(Sg)[e] = reinterpret_cast<const float4 *>(S + r * L::SS)[c4];
  }
}

template <int DK, int DV, typename TI, typename TO>
cudaError_t launch_prefill_t(const PoolView &p, int layer, const SeqIndex &seq, const QKV &in,
                             void *o, float scale, cudaStream_t s) {
  using L = PrefillSmem<DK, DV>;
  auto kern = prefill_simt_kernel<DK, DV, TI, TO>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)L::bytes);
  if (e != cudaSuccess) return e;
  dim3 grid(p.h_v, seq.n_seqs);
  kern<<<grid, kPT, L::bytes, s>>>(p, layer, seq, in, static_cast<TO *>(o), scale);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_prefill_d(const PoolView &p, int layer, const SeqIndex &seq, const QKV &in,
                             void *o, gdn_dtype o_dtype, float scale, cudaStream_t s) {
  if (in.dtype == GDN_F32 && o_dtype == GDN_F32)
    return launch_prefill_t<D, D, float, float>(p, layer, seq, in, o, scale, s);
  if (in.dtype == GDN_F32 && o_dtype == GDN_BF16)
    return launch_prefill_t<D, D, float, bf16>(p, layer, seq, in, o, scale, s);
  if (in.dtype == GDN_BF16 && o_dtype == GDN_F32)
    return launch_prefill_t<D, D, bf16, float>(p, layer, seq, in, o, scale, s);
  return launch_prefill_t<D, D, bf16, bf16>(p, layer, seq, in, o, scale, s);
}

}  // namespace

namespace {

// tensor-core paths: dk = dv = 128 and 128-bit aligned rows of v
bool tc_shape(const PoolView &p, const QKV &in) {
  const size_t es = in.dtype == GDN_F32 ? 4 : 2;
  const size_t al = in.dtype == GDN_F32 ? 16 : 8;
  return p.dk == 128 && p.dv == 128 && (uintptr_t)in.v % al == 0 &&
         ((size_t)in.ld_v * es) % al == 0;
}

}  // namespace

size_t prefill_workspace_bytes(const PoolView &p, const SeqIndex &seq, const QKV &in,
                               size_t limit) {
  if (!tc_shape(p, in)) return 0;
  const size_t b = prefill_split_workspace_bytes(seq.n_seqs, seq.total_tokens, p.h_v);
  return b <= limit ? b : 0;
}

cudaError_t launch_prefill(const PoolView &p, int layer, const SeqIndex &seq, const QKV &in,
                           void *o, gdn_dtype o_dtype, float scale, void *work,
                           cudaStream_t s) {
  if (tc_shape(p, in) && work != nullptr)
    return launch_prefill_split(p, layer, seq, in, o, o_dtype, scale, work, s);
  // a bf16 / f16 state is read and written by the two-launch path above and by
  // the token-by-token kernel; the single-launch chunked kernels keep float32
  if (p.state_dtype != GDN_F32)
    return launch_prefill_recurrent(p, layer, seq, in, o, o_dtype, scale, s);
  if (p.dk != p.dv) return cudaErrorNotSupported;
  if (tc_shape(p, in)) return launch_prefill_tc(p, layer, seq, in, o, o_dtype, scale, s);
  switch (p.dk) {
    case 16: return launch_prefill_d<16>(p, layer, seq, in, o, o_dtype, scale, s);
    case 32: return launch_prefill_d<32>(p, layer, seq, in, o, o_dtype, scale, s);
    case 64: return launch_prefill_d<64>(p, layer, seq, in, o, o_dtype, scale, s);
    case 128: return launch_prefill_d<128>(p, layer, seq, in, o, o_dtype, scale, s);
  }
  return cudaErrorNotSupported;
}

}  // namespace gdn
