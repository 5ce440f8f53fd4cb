// Speculative verify over a slot-indexed pool of Gated DeltaNet states
// (b70-optimization-lab research plan, "What the research found": outputs for
// every draft position without per-position state snapshots), with the state
// committed once at each slot's accepted length.
#include "gdn_rows.cuh"

namespace gdn {
namespace {

using rows::kThreads;
using rows::dispatch;

constexpr int kTileBytes = 32768;  // state tile per CTA (one bulk copy)

// Row-level WY form for T tokens (speculative verify; decode is T = 1).
//
// With G_t the cumulative log-decay after t tokens (G_0 = 0) and
// D[a][b] = exp(G_a - G_b), the state after t tokens is
//     S_t = D[t][0] S_0 + sum_{i<=t} D[t][i] delta_i k_i^T,
// so for one row r of S_0 (s = S_0[r]) every quantity follows from the 2T
// dot products s.k_t, s.q_t and the CTA-wide Gram scalars k_i.k_t, k_i.q_t:
//     p_t     = D[t-1][0] s.k_t + sum_{i<t} D[t-1][i] delta_i k_i.k_t
//     delta_t = beta_t (v_t[r] - alpha_t p_t)
//     o_t[r]  = scale (D[t][0] s.q_t + sum_{i<=t} D[t][i] delta_i k_i.q_t)
//     S_a[r]  = D[a][0] s + sum_{i<=a} D[a][i] delta_i k_i          (commit)
// (tokens 1-based here; the code is 0-based).  The 2T dot products are
// independent, so each row is split over only 4 lanes (2-shuffle reductions)
// and the state row is rebuilt once, at the accepted length, instead of
// being updated T times.  The CTA's state tile (32 KiB of float32, 16 KiB of
// a bf16 / f16 state, widened to float32 as rows are read and rounded back
// when they are written) arrives by one bulk copy while the tokens are
// staged.  grid (ceil(dv / R), h_v, n).
template <int DK, int TMAX, typename TI, typename TO>
__global__ void __launch_bounds__(kThreads)
    rows_kernel(PoolView p, int layer, VerifyArgs va, TO *__restrict__ o) {
  constexpr int R = kTileBytes / (DK * 4);   // rows per CTA
  constexpr int LPR = 4;                     // lanes per row
  constexpr int C4 = DK / 16;                // float4 chunks per lane per row
  constexpr int RPP = 32 / LPR;              // rows per warp pass
  constexpr int RPW = R / (kThreads / 32);   // rows per warp
  constexpr int PASSES = RPW / RPP;
  static_assert(PASSES >= 1 && RPW % RPP == 0, "row mapping");
  __shared__ __align__(128) float4 tile[kTileBytes / 16];
  __shared__ __align__(8) uint64_t bar;
  // dynamic: k, q [T][DK]; v [T][R]; Gram KK, KQ [T][T]; D [(T+1)][(T+1)]; alpha, beta [T];
  // G [T+1]
  // (sized for Tb = T_prev + T tokens; this CTA runs T = ap + T_new <= Tb)
  extern __shared__ float4 dsm[];
  const int Tb = va.T + va.T_prev;
  float4 *sk4 = dsm;
  float4 *sq4 = sk4 + Tb * (DK / 4);
  float *sv = reinterpret_cast<float *>(sq4 + Tb * (DK / 4));
  float *KK = sv + Tb * R;
  float *KQ = KK + Tb * Tb;
  float *Dm = KQ + Tb * Tb;
  float *sal = Dm + (Tb + 1) * (Tb + 1);
  float *sbe = sal + Tb;
  float *sG = sbe + Tb;  // cumulative log-decay after t tokens, t = 0..T
  // looped variant only (TMAX > 8): per-row dot products and deltas, [32 rows][T] each
  float *rdk = sG + Tb + 1;
  float *rdq = rdk + 32 * Tb;
  float *rdl = rdq + 32 * Tb;

  const int i = blockIdx.z;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  const int slot = va.slot_ids[i];
  if (slot < 0 || slot >= p.n_slots) {
    if (blockIdx.x == 0 && h == 0 && tid == 0) raise_error(p.err, GDN_DEVERR_SLOT);
    return;
  }
  const bool deferred = va.prev.q != nullptr && va.prev_accept != nullptr;
  int ap = deferred ? va.prev_accept[i] : 0;  // pending drafts replayed first
  if (ap < 0 || ap > va.T_prev) {
    if (blockIdx.x == 0 && h == 0 && tid == 0) raise_error(p.err, GDN_DEVERR_COUNT);
    ap = ap < 0 ? 0 : va.T_prev;
  }
  const int T = ap + va.T;
  int a = deferred ? ap : (va.commit_all ? T : (va.accept_len ? va.accept_len[i] : 0));
  if (a < 0 || a > T) {
    if (blockIdx.x == 0 && h == 0 && tid == 0) raise_error(p.err, GDN_DEVERR_COUNT);
    a = a < 0 ? 0 : T;
  }
  // token t of this slot's sequence: pending draft t, or new draft t - ap
  // (register copies: no address of the parameter block is taken)
  const QKV cur = va.in, prv = va.prev;
  const int T_new = va.T, T_old = va.T_prev;
  auto src_of = [&](int t, int64_t &row) -> QKV {
    const bool pend = t < ap;
    row = pend ? (int64_t)i * T_old + t : (int64_t)i * T_new + (t - ap);
    return pend ? prv : cur;
  };
  const int r0 = blockIdx.x * R;
  const int nrows = min(R, p.dv - r0);
  char *S = p.state_at(p.state_head_elem(layer, slot, h) + (int64_t)r0 * DK);
  const gdn_dtype sd = p.state_dtype;
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t bytes = (uint32_t)nrows * DK * p.state_esz();
    mbar_arrive_expect_tx(&bar, bytes);
    bulk_g2s(tile, S, bytes, &bar);
  }

  // ---- stage the T tokens (overlaps the bulk copy)
  const int lane = tid & 31, warp = tid >> 5;
  const int hk = h / (p.h_v / p.h_k);
  for (int t = warp; t < T; t += kThreads / 32) {
    int64_t tok;
    const QKV src = src_of(t, tok);
    float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f), k4 = q4;
    if (lane < DK / 4) {
      q4 = Elem<TI>::load4(static_cast<const TI *>(src.q) + tok * src.ld_qk + (int64_t)hk * DK + 4 * lane);
      k4 = Elem<TI>::load4(static_cast<const TI *>(src.k) + tok * src.ld_qk + (int64_t)hk * DK + 4 * lane);
    }
    const float qq = group_sum<32>(dot4(q4, q4));
    const float kk = group_sum<32>(dot4(k4, k4));
    if (lane < DK / 4) {
      sq4[t * (DK / 4) + lane] = scale4(rsqrtf(qq + kL2Eps), q4);
      sk4[t * (DK / 4) + lane] = scale4(rsqrtf(kk + kL2Eps), k4);
    }
  }
  for (int e = tid; e < T * R; e += kThreads) {
    const int t = e / R, rl = e % R;
    int64_t tok;
    const QKV src = src_of(t, tok);
    sv[e] = rl < nrows ? Elem<TI>::load1(static_cast<const TI *>(src.v) + tok * src.ld_v +
                                        (int64_t)h * p.dv + r0 + rl)
                       : 0.f;
  }
  if (tid < T) {  // g_t into sG[t + 1] (summed below), alpha_t, beta_t
    int64_t tok;
    const QKV src = src_of(tid, tok);
    const float gt = Elem<TI>::load1(static_cast<const TI *>(src.g) + tok * p.h_v + h);
    sG[tid + 1] = gt;
    sal[tid] = expf(gt);
    sbe[tid] = Elem<TI>::load1(static_cast<const TI *>(src.beta) + tok * p.h_v + h);
  }
  __syncthreads();
  if (tid == 0) {  // G_t = g_0 + ... + g_{t-1}
    float acc = 0.f;
    sG[0] = 0.f;
    for (int t = 1; t <= T; ++t) sG[t] = (acc += sG[t]);
  }
  __syncthreads();
  // Gram scalars k_i.k_t and k_i.q_t (four lanes per pair) and the decay table
  for (int e0 = 0; e0 < 2 * T * T; e0 += kThreads / 4) {
    const int e = e0 + tid / 4, sub4 = tid % 4;
    float acc = 0.f;
    if (e < 2 * T * T) {
      const int which = e / (T * T), ii = (e / T) % T, tt = e % T;
      const float4 *x = sk4 + ii * (DK / 4);
      const float4 *y = (which ? sq4 : sk4) + tt * (DK / 4);
#pragma unroll
      for (int j = 0; j < DK / 16; ++j) {
        const int c = ((j + e) % (DK / 16)) * 4 + sub4;
        acc += dot4(x[c], y[c]);
      }
    }
    acc = group_sum<4>(acc);
    if (e < 2 * T * T && sub4 == 0) {
      const int which = e / (T * T), ii = (e / T) % T, tt = e % T;
      (which ? KQ : KK)[ii * T + tt] = acc;
    }
  }
  for (int e = tid; e < (T + 1) * (T + 1); e += kThreads) {
    const int aa = e / (T + 1), bb = e % (T + 1);
    Dm[e] = bb <= aa ? expf(sG[aa] - sG[bb]) : 0.f;
  }
  __syncthreads();

  if (!mbar_wait_bounded(&bar, 0)) {
    if (tid == 0) raise_error(p.err, GDN_DEVERR_TIMEOUT);
    mbar_wait_bounded(&bar, 0);
    return;
  }

  const int sub = lane % LPR;
  const int rho = lane / LPR;
  const int rot = rho % C4;  // per-row rotation of the chunk order (bank spread)
  const int64_t o_tok = (int64_t)p.h_v * p.dv;
  // output of token t >= ap: new draft t - ap of slot i
  TO *obase = o == nullptr ? nullptr : o + ((int64_t)i * va.T * p.h_v + h) * p.dv + r0;
  const float scale = va.scale;
#pragma unroll
  for (int ps = 0; ps < PASSES; ++ps) {
    const int rl = warp * RPW + ps * RPP + rho;
    const bool live = rl < nrows;
    float4 s[C4];
#pragma unroll
    for (int j = 0; j < C4; ++j) {
      const int cj = ((j + rot) % C4) * LPR + sub;   // float4 index within the row
      s[j] = live ? state_ld4(tile, (int64_t)rl * DK + 4 * cj, sd) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if constexpr (TMAX <= 8) {
      // fully unrolled: per-row scalars in registers
      float dk[TMAX], dq[TMAX], dl[TMAX];
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        float ak = 0.f, aq = 0.f;
        if (t < T) {
#pragma unroll
          for (int j = 0; j < C4; ++j) {
            const int cj = ((j + rot) % C4) * LPR + sub;
            ak += dot4(s[j], sk4[t * (DK / 4) + cj]);
            if (o != nullptr) aq += dot4(s[j], sq4[t * (DK / 4) + cj]);
          }
        }
        dk[t] = group_sum<LPR>(ak);
        dq[t] = group_sum<LPR>(aq);
      }
      // scalar recurrences (every lane of the row computes them)
#pragma unroll
      for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
          float pt = Dm[t * (T + 1)] * dk[t];
#pragma unroll
          for (int ii = 0; ii < TMAX; ++ii)
            if (ii < t) pt += Dm[t * (T + 1) + ii + 1] * dl[ii] * KK[ii * T + t];
          dl[t] = sbe[t] * (sv[t * R + (live ? rl : 0)] - sal[t] * pt);
          if (o != nullptr) {
            float ot = Dm[(t + 1) * (T + 1)] * dq[t];
#pragma unroll
            for (int ii = 0; ii < TMAX; ++ii)
              if (ii <= t) ot += Dm[(t + 1) * (T + 1) + ii + 1] * dl[ii] * KQ[ii * T + t];
            if (live && t >= ap && (t % LPR) == sub)
              Elem<TO>::store1(obase + (t - ap) * o_tok + rl, scale * ot);
          }
        } else {
          dl[t] = 0.f;
        }
      }
      if (a > 0 && live) {
        const float c0 = Dm[a * (T + 1)];
#pragma unroll
        for (int j = 0; j < C4; ++j) {
          const int cj = ((j + rot) % C4) * LPR + sub;
          float4 acc = scale4(c0, s[j]);
#pragma unroll
          for (int ii = 0; ii < TMAX; ++ii)
            if (ii < a) acc = axpby4(1.f, acc, Dm[a * (T + 1) + ii + 1] * dl[ii],
                                     sk4[ii * (DK / 4) + cj]);
          state_st4<true>(S, (int64_t)rl * DK + 4 * cj, acc, sd);
        }
      }
    } else {
      // long drafts: loops, per-row scalars in shared memory (one row per 4 lanes)
      const int rs = (warp * RPP + rho) * T;
#pragma unroll 1
      for (int t = 0; t < T; ++t) {
        float ak = 0.f, aq = 0.f;
#pragma unroll
        for (int j = 0; j < C4; ++j) {
          const int cj = ((j + rot) % C4) * LPR + sub;
          ak += dot4(s[j], sk4[t * (DK / 4) + cj]);
          if (o != nullptr) aq += dot4(s[j], sq4[t * (DK / 4) + cj]);
        }
        ak = group_sum<LPR>(ak);
        aq = group_sum<LPR>(aq);
        if (sub == 0) {
          rdk[rs + t] = ak;
          rdq[rs + t] = aq;
        }
      }
      __syncwarp();
      if (sub == 0) {
#pragma unroll 1
        for (int t = 0; t < T; ++t) {
          float pt = Dm[t * (T + 1)] * rdk[rs + t];
          for (int ii = 0; ii < t; ++ii) pt += Dm[t * (T + 1) + ii + 1] * rdl[rs + ii] * KK[ii * T + t];
          const float d = sbe[t] * (sv[t * R + (live ? rl : 0)] - sal[t] * pt);
          rdl[rs + t] = d;
          if (o != nullptr) {
            float ot = Dm[(t + 1) * (T + 1)] * rdq[rs + t];
            for (int ii = 0; ii <= t; ++ii)
              ot += Dm[(t + 1) * (T + 1) + ii + 1] * rdl[rs + ii] * KQ[ii * T + t];
            if (live && t >= ap) Elem<TO>::store1(obase + (t - ap) * o_tok + rl, scale * ot);
          }
        }
      }
      __syncwarp();
      if (a > 0 && live) {
        const float c0 = Dm[a * (T + 1)];
#pragma unroll
        for (int j = 0; j < C4; ++j) {
          const int cj = ((j + rot) % C4) * LPR + sub;
          float4 acc = scale4(c0, s[j]);
#pragma unroll 1
          for (int ii = 0; ii < a; ++ii)
            acc = axpby4(1.f, acc, Dm[a * (T + 1) + ii + 1] * rdl[rs + ii],
                         sk4[ii * (DK / 4) + cj]);
          state_st4<true>(S, (int64_t)rl * DK + 4 * cj, acc, sd);
        }
      }
      __syncwarp();
    }
  }
}

inline size_t rows_smem_bytes(int DK, int R, int T, bool looped) {
  return (size_t)T * (DK / 4) * sizeof(float4) * 2 +
         ((size_t)T * R + 2 * (size_t)T * T + (size_t)(T + 1) * (T + 1) + 3 * (size_t)T + 1 +
          (looped ? 3 * 32 * (size_t)T : 0)) *
             sizeof(float);
}

template <int DK, int TMAX, typename TI, typename TO>
cudaError_t launch_rows_t(const PoolView &p, int layer, const VerifyArgs &va, void *o,
                          cudaStream_t s) {
  constexpr int R = kTileBytes / (DK * 4);
  const size_t smem = rows_smem_bytes(DK, R, va.T + va.T_prev, TMAX > 8);
  auto kern = rows_kernel<DK, TMAX, TI, TO>;
  // the static tile counts against the default 48 KiB per-block limit
  if (smem + kTileBytes + 64 > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((p.dv + R - 1) / R, p.h_v, va.n);
  kern<<<grid, kThreads, smem, s>>>(p, layer, va, static_cast<TO *>(o));
  return cudaGetLastError();
}

template <int DK, typename TI, typename TO>
struct VerifyF {
  static cudaError_t run(const PoolView &p, int layer, const VerifyArgs &va, void *o,
                         cudaStream_t s) {
    if (va.T + va.T_prev <= 4) return launch_rows_t<DK, 4, TI, TO>(p, layer, va, o, s);
    return launch_rows_t<DK, 32, TI, TO>(p, layer, va, o, s);
  }
};

}  // namespace

cudaError_t launch_verify(const PoolView &p, const void *tmap, int layer, const VerifyArgs &va,
                          void *o, gdn_dtype o_dtype, cudaStream_t s) {
  const cudaError_t e = launch_verify_tma(p, tmap, layer, va, o, o_dtype, s);
  if (e != cudaErrorNotSupported) return e;
  return dispatch<VerifyF>(p.dk, va.in.dtype, o_dtype, p, layer, va, o, s);
}

}  // namespace gdn
