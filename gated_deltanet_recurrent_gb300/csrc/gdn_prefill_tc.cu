// Chunked prefill on the 5th-generation tensor cores (tcgen05, kind::tf32),
// for dk = dv = 128.
//
// One CTA (256 threads) per (sequence, value head) walks the sequence in
// 64-token chunks.  The float32 state S [dv][dk] lives in tensor memory for
// the whole call (TMEM columns 0..127, row v in lane v) and is the A operand
// of the state-dependent products, so it never leaves the SM between chunks.
// Per chunk (notation of the chunked delta rule, b70-optimization-lab research
// plan, "What the research found": the (I+A)^{-1} UT transform):
//   MMA1  D1 = [Q;K] K^T                     -> A = beta e^{dG} KK^T (strict),
//                                              P = e^{dG} QK^T (lower, incl. diag)
//   solve (I + A) [W | U] = [diag(beta gamma) K | diag(beta) V]   (CUDA cores)
//   MMA2  D2 = S W^T,  MMA3  D3 = S Q^T      -> Delta^T = U^T - D2;  S <- gamma_n S
//   MMA4  D4 = Delta^T P^T                    -> O^T = diag(gamma) D3 + D4
//   MMA5  S += Delta^T Ktil,  Ktil = diag(e^{G_n - G}) K
// TMEM lanes are split over warps w and w+4 (same lane quadrant, column
// halves).  Operands are K-major, no-swizzle core-matrix tiles in shared
// memory (see gdn_tc.cuh).
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int C = kChunk;   // 64
constexpr int D = 128;      // dk = dv
constexpr int NT = 256;     // threads
constexpr int XS = D + 4;   // plain row stride (floats) of the solve buffers
constexpr int AS = C + 4;   // plain row stride of the A matrix

// shared-memory map (bytes)
constexpr int OFF_QK = 0;                          // [Q;K] then [Q;W], 128 x 128 core tile
constexpr int OFF_XW = OFF_QK + 128 * D * 4;       // W solve (plain 64 x XS), then Delta^T tile
constexpr int OFF_XU = OFF_XW + C * XS * 4;        // U solve (plain 64 x XS)
constexpr int OFF_AP = OFF_XU + C * XS * 4;        // A (plain 64 x AS), then P tile 64 x 64
constexpr int OFF_KT = OFF_AP + C * AS * 4;        // Ktil^T tile 128 x 64
constexpr int OFF_SC = OFF_KT + D * C * 4;         // scalars
constexpr int SMEM_BYTES = OFF_SC + 4 * C * 4 + 64;
static_assert(OFF_XW % 1024 == 0 && OFF_KT % 16 == 0 && OFF_AP % 16 == 0, "alignment");
static_assert(128 * C * 4 <= C * XS * 4, "Delta^T tile fits the W solve buffer");
static_assert(C * C * 4 <= C * AS * 4, "P tile fits the A buffer");

// TMEM columns
constexpr uint32_t T_S = 0, T_D1 = 128, T_D2 = 192, T_D3 = 256, T_D4 = 320;
constexpr uint32_t TMEM_COLS = 512;

template <typename TI, typename TO>
__global__ void __launch_bounds__(NT, 1)
    prefill_tc_kernel(PoolView p, int layer, SeqIndex seq, QKV in, TO *__restrict__ o,
                      float scale) {
  extern __shared__ __align__(1024) unsigned char smem[];
  float *QK = reinterpret_cast<float *>(smem + OFF_QK);
  float *XW = reinterpret_cast<float *>(smem + OFF_XW);
  float *XU = reinterpret_cast<float *>(smem + OFF_XU);
  float *AP = reinterpret_cast<float *>(smem + OFF_AP);
  float *KT = reinterpret_cast<float *>(smem + OFF_KT);
  float *sG = reinterpret_cast<float *>(smem + OFF_SC);
  float *sGam = sG + C;
  float *sBeta = sGam + C;
  float *sDte = sBeta + C;
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;

  const int h = blockIdx.x;
  const int si = blockIdx.y;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int quad = warp & 3;                    // TMEM lane quadrant of this warp
  const int half = warp >> 2;                   // which half of the columns it takes
  const int row = 32 * quad + lane;             // TMEM lane = accumulator row
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
              (int64_t)h * D * D;

  if (warp == 0) tc::tmem_alloc(&tmem_slot, TMEM_COLS);
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = tmem_slot;
  const uint32_t lrow = tm + ((uint32_t)(32 * quad) << 16);  // this warp's TMEM lanes

  // state row `row`, column half `half` -> TMEM
  {
    const float4 *src = reinterpret_cast<const float4 *>(Sg + (int64_t)row * D + 64 * half);
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 x = src[c * 4 + j];
        v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
      }
      tc::tmem_st16(lrow + T_S + 64 * half + c * 16, v);
    }
    tc::tmem_st_wait();
  }

  const TI *qg = static_cast<const TI *>(in.q);
  const TI *kg = static_cast<const TI *>(in.k);
  const TI *vg = static_cast<const TI *>(in.v);
  const TI *gg = static_cast<const TI *>(in.g);
  const TI *bg = static_cast<const TI *>(in.beta);
  const uint32_t qk_s = smem_addr(QK);
  const uint32_t k_s = qk_s + 64 * D * 4;  // rows 64..127 of the [Q;K] tile
  const uint32_t dt_s = smem_addr(XW);
  const uint32_t p_s = smem_addr(AP);
  const uint32_t kt_s = smem_addr(KT);
  constexpr uint32_t SBO_D = tc::sbo_bytes(D);  // 4096
  constexpr uint32_t SBO_C = tc::sbo_bytes(C);  // 2048
  constexpr uint32_t KSTEP = 2 * tc::kLBO;      // one K = 8 step spans two core matrices
  uint32_t phase = 0;
  bool alive = true;

  for (int c0 = 0; c0 < len && alive; c0 += C) {
    const int n = min(C, len - c0);

    // ---- S0: stage normalised q, k (core tiles), beta v (plain), g, beta.
    // Warp w takes tokens 8w .. 8w+7; lane = token (3 bits) + 8 * chunk group, so a
    // quarter-warp writes the 8 rows of one core matrix (contiguous 128 bytes).
    {
      const int tl = lane & 7, cg = lane >> 3;      // token in group, chunk group 0..3
      const int t = 8 * warp + tl;
      const int64_t tok = lo + c0 + t;
      const bool real = t < n;
      float4 q4[D / 16], k4[D / 16], v4[D / 16];   // chunks c = cg + 4 j
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        const int c = cg + 4 * j;
        q4[j] = k4[j] = v4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (real) {
          q4[j] = Elem<TI>::load4(qg + tok * in.ld_qk + (int64_t)hk * D + 4 * c);
          k4[j] = Elem<TI>::load4(kg + tok * in.ld_qk + (int64_t)hk * D + 4 * c);
          v4[j] = Elem<TI>::load4(vg + tok * in.ld_v + (int64_t)h * D + 4 * c);
        }
      }
      const float gt = real ? Elem<TI>::load1(gg + tok * p.h_v + h) : 0.f;
      const float bt = real ? Elem<TI>::load1(bg + tok * p.h_v + h) : 0.f;
      float qq = 0.f, kk = 0.f;
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        qq += dot4(q4[j], q4[j]);
        kk += dot4(k4[j], k4[j]);
      }
      // reduce over the four chunk groups of this token (lane bits 3 and 4)
      qq += __shfl_xor_sync(0xffffffffu, qq, 8);
      qq += __shfl_xor_sync(0xffffffffu, qq, 16);
      kk += __shfl_xor_sync(0xffffffffu, kk, 8);
      kk += __shfl_xor_sync(0xffffffffu, kk, 16);
      const float qs = rsqrtf(qq + kL2Eps), ks = rsqrtf(kk + kL2Eps);
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        const int c = cg + 4 * j;
        *reinterpret_cast<float4 *>(QK + tc::core_off(t, 4 * c, D)) = scale4(qs, q4[j]);
        *reinterpret_cast<float4 *>(QK + tc::core_off(64 + t, 4 * c, D)) = scale4(ks, k4[j]);
        *reinterpret_cast<float4 *>(XU + t * XS + 4 * c) = scale4(bt, v4[j]);
      }
      if (cg == 0) {
        sG[t] = gt;
        sBeta[t] = bt;
      }
    }
    __syncthreads();
    if (warp == 0) {  // cumulative log-decay over the chunk (padded tokens carry g = 0)
      const float a = sG[2 * lane], b = sG[2 * lane + 1];
      float incl = a + b;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float up = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += up;
      }
      const float g0 = incl - b;
      const float gl = __shfl_sync(0xffffffffu, incl, 31);
      sG[2 * lane] = g0;
      sG[2 * lane + 1] = incl;
      sGam[2 * lane] = expf(g0);
      sGam[2 * lane + 1] = expf(incl);
      sDte[2 * lane] = expf(gl - g0);
      sDte[2 * lane + 1] = expf(gl - incl);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---- S1: MMA1  D1 = [Q;K] K^T  (M 128, N 64, K 128)
    if (tid == 0) {
      constexpr uint32_t id = tc::idesc_tf32(128, 64);
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
        tc::mma_ss(tm + T_D1, tc::smem_desc(qk_s + j * KSTEP, tc::kLBO, SBO_D),
                   tc::smem_desc(k_s + j * KSTEP, tc::kLBO, SBO_D), id, j > 0);
      tc::mma_commit(&bar);
    }
    // meanwhile: W right-hand side (beta gamma k, plain) and the Ktil^T tile
    for (int e = tid; e < C * (D / 4); e += NT) {
      const int t = e % C, c4 = e / C;
      const float4 k4 = *reinterpret_cast<const float4 *>(QK + tc::core_off(64 + t, 4 * c4, D));
      *reinterpret_cast<float4 *>(XW + t * XS + 4 * c4) = scale4(sBeta[t] * sGam[t], k4);
    }
    {
      const int kc = tid & 127;            // row k of Ktil^T
      const int ib = (tid >> 7) * (C / 8); // which half of the i chunks
#pragma unroll 2
      for (int q = 0; q < C / 8; ++q) {
        const int i4 = ib + ((q + (kc >> 2)) & (C / 8 - 1));   // rotated: spreads banks
        float4 x;
        x.x = sDte[4 * i4 + 0] * QK[tc::core_off(64 + 4 * i4 + 0, kc, D)];
        x.y = sDte[4 * i4 + 1] * QK[tc::core_off(64 + 4 * i4 + 1, kc, D)];
        x.z = sDte[4 * i4 + 2] * QK[tc::core_off(64 + 4 * i4 + 2, kc, D)];
        x.w = sDte[4 * i4 + 3] * QK[tc::core_off(64 + 4 * i4 + 3, kc, D)];
        *reinterpret_cast<float4 *>(KT + tc::core_off(kc, 4 * i4, C)) = x;
      }
    }
    alive = __syncthreads_and(mbar_wait_bounded(&bar, phase));
    if (!alive) break;
    phase ^= 1;
    tc::fence_after_sync();

    // ---- S2: A[t][i] = beta_t e^{G_t - G_i} (k_t . k_i), i < t   (rows 64..127 of D1)
    if (quad >= 2) {
      const int t = row - 64;
      const float bt = sBeta[t], gt = sG[t];
#pragma unroll 1
      for (int cb = 0; cb < 2; ++cb) {
        float v[16];
        const int i0 = 32 * half + 16 * cb;
        tc::tmem_ld16(lrow + T_D1 + i0, v);
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          float4 a;
          const int i = i0 + j;
          a.x = i + 0 < t ? bt * expf(gt - sG[i + 0]) * v[j + 0] : 0.f;
          a.y = i + 1 < t ? bt * expf(gt - sG[i + 1]) * v[j + 1] : 0.f;
          a.z = i + 2 < t ? bt * expf(gt - sG[i + 2]) * v[j + 2] : 0.f;
          a.w = i + 3 < t ? bt * expf(gt - sG[i + 3]) * v[j + 3] : 0.f;
          *reinterpret_cast<float4 *>(AP + t * AS + i) = a;
        }
      }
    }
    __syncthreads();

    // ---- S3: forward substitution (I + A) X = RHS; thread = one column of [W | U]
    {
      float *Xc = (tid < D ? XW + tid : XU + (tid - D));
      float x[C];
#pragma unroll
      for (int t = 0; t < C; ++t) x[t] = Xc[t * XS];
#pragma unroll
      for (int t = 1; t < C; ++t) {
        const float *ar = AP + t * AS;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int i = 0; i + 3 < t; i += 4) {
          const float4 av = *reinterpret_cast<const float4 *>(ar + i);
          a0 += av.x * x[i];
          a1 += av.y * x[i + 1];
          a2 += av.z * x[i + 2];
          a3 += av.w * x[i + 3];
        }
#pragma unroll
        for (int i = (t / 4) * 4; i < t; ++i) a0 += ar[i] * x[i];
        x[t] -= (a0 + a1) + (a2 + a3);
      }
#pragma unroll
      for (int t = 0; t < C; ++t) Xc[t * XS] = x[t];
    }
    __syncthreads();

    // ---- S4: W -> rows 64..127 of the [Q;K] tile; P tile (rows 0..63 of D1)
    for (int e = tid; e < C * (D / 4); e += NT) {
      const int t = e % C, c4 = e / C;
      *reinterpret_cast<float4 *>(QK + tc::core_off(64 + t, 4 * c4, D)) =
          *reinterpret_cast<const float4 *>(XW + t * XS + 4 * c4);
    }
    if (quad < 2) {
      const int t = row;
      const float gt = sG[t];
#pragma unroll 1
      for (int cb = 0; cb < 2; ++cb) {
        float v[16];
        const int i0 = 32 * half + 16 * cb;
        tc::tmem_ld16(lrow + T_D1 + i0, v);
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          float4 pv;
          const int i = i0 + j;
          pv.x = i + 0 <= t ? expf(gt - sG[i + 0]) * v[j + 0] : 0.f;
          pv.y = i + 1 <= t ? expf(gt - sG[i + 1]) * v[j + 1] : 0.f;
          pv.z = i + 2 <= t ? expf(gt - sG[i + 2]) * v[j + 2] : 0.f;
          pv.w = i + 3 <= t ? expf(gt - sG[i + 3]) * v[j + 3] : 0.f;
          *reinterpret_cast<float4 *>(AP + tc::core_off(t, i, C)) = pv;
        }
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---- S5: MMA2  D2 = S W^T,  MMA3  D3 = S Q^T   (M 128, N 64, K 128; A from TMEM)
    if (tid == 0) {
      constexpr uint32_t id = tc::idesc_tf32(128, 64);
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
        tc::mma_ts(tm + T_D2, tm + T_S + j * 8,
                   tc::smem_desc(k_s + j * KSTEP, tc::kLBO, SBO_D), id, j > 0);
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
        tc::mma_ts(tm + T_D3, tm + T_S + j * 8,
                   tc::smem_desc(qk_s + j * KSTEP, tc::kLBO, SBO_D), id, j > 0);
      tc::mma_commit(&bar);
    }
    alive = __syncthreads_and(mbar_wait_bounded(&bar, phase));
    if (!alive) break;
    phase ^= 1;
    tc::fence_after_sync();

    // ---- S6: Delta^T[v][t] = U[t][v] - D2[v][t] (tile, K = t); o part = gamma_t D3[v][t];
    //          S <- gamma_n S (MMA5 then accumulates Delta^T Ktil into it)
    float op[C / 2];
    {
      const int v = row;
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        const int t0 = 32 * half + 16 * cb;
        float d2[16], d3[16];
        tc::tmem_ld16(lrow + T_D2 + t0, d2);
        tc::tmem_ld16(lrow + T_D3 + t0, d3);
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          const int t = t0 + j;
          float4 dd;
          dd.x = XU[(t + 0) * XS + v] - d2[j + 0];
          dd.y = XU[(t + 1) * XS + v] - d2[j + 1];
          dd.z = XU[(t + 2) * XS + v] - d2[j + 2];
          dd.w = XU[(t + 3) * XS + v] - d2[j + 3];
          *reinterpret_cast<float4 *>(XW + tc::core_off(v, t, C)) = dd;
#pragma unroll
          for (int q = 0; q < 4; ++q) op[16 * cb + j + q] = sGam[t + q] * d3[j + q];
        }
      }
      const float gn = sGam[C - 1];
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        float s[16];
        tc::tmem_ld16(lrow + T_S + 64 * half + 16 * cb, s);
#pragma unroll
        for (int j = 0; j < 16; ++j) s[j] *= gn;
        tc::tmem_st16(lrow + T_S + 64 * half + 16 * cb, s);
      }
      tc::tmem_st_wait();
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---- S7: MMA4  D4 = Delta^T P^T (N 64),  MMA5  S += Delta^T Ktil (N 128); K = 64
    if (tid == 0) {
#pragma unroll
      for (int j = 0; j < C / 8; ++j)
        tc::mma_ss(tm + T_D4, tc::smem_desc(dt_s + j * KSTEP, tc::kLBO, SBO_C),
                   tc::smem_desc(p_s + j * KSTEP, tc::kLBO, SBO_C), tc::idesc_tf32(128, 64),
                   j > 0);
#pragma unroll
      for (int j = 0; j < C / 8; ++j)
        tc::mma_ss(tm + T_S, tc::smem_desc(dt_s + j * KSTEP, tc::kLBO, SBO_C),
                   tc::smem_desc(kt_s + j * KSTEP, tc::kLBO, SBO_C), tc::idesc_tf32(128, 128),
                   1);
      tc::mma_commit(&bar);
    }
    alive = __syncthreads_and(mbar_wait_bounded(&bar, phase));
    if (!alive) break;
    phase ^= 1;
    tc::fence_after_sync();

    // ---- S8: outputs o[t][v] = scale (gamma_t D3 + D4), this warp's half of t
    {
      const int v = row;
      TO *ob = o + (lo + c0) * p.h_v * D + (int64_t)h * D + v;
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        const int t0 = 32 * half + 16 * cb;
        float d4[16];
        tc::tmem_ld16(lrow + T_D4 + t0, d4);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = t0 + j;
          if (t < n)
            Elem<TO>::store1(ob + (int64_t)t * p.h_v * D, scale * (op[16 * cb + j] + d4[j]));
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
  }

  if (alive) {
    float4 *dst = reinterpret_cast<float4 *>(Sg + (int64_t)row * D + 64 * half);
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float v[16];
      tc::tmem_ld16(lrow + T_S + 64 * half + c * 16, v);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        dst[c * 4 + j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
  } else {
    if (tid == 0) raise_error(p.err, GDN_DEVERR_TIMEOUT);
    mbar_wait_bounded(&bar, phase);  // give the outstanding MMA group a second bounded chance
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tm, TMEM_COLS);
}

template <typename TI, typename TO>
cudaError_t launch_tc(const PoolView &p, int layer, const SeqIndex &seq, const QKV &in, void *o,
                      float scale, cudaStream_t s) {
  auto kern = prefill_tc_kernel<TI, TO>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(p.h_v, seq.n_seqs);
  kern<<<grid, NT, SMEM_BYTES, s>>>(p, layer, seq, in, static_cast<TO *>(o), scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const PoolView &p, int layer, const SeqIndex &seq, const QKV &in,
                              void *o, gdn_dtype o_dtype, float scale, cudaStream_t s) {
  if (in.dtype == GDN_F32 && o_dtype == GDN_F32)
    return launch_tc<float, float>(p, layer, seq, in, o, scale, s);
  if (in.dtype == GDN_F32 && o_dtype == GDN_BF16)
    return launch_tc<float, bf16>(p, layer, seq, in, o, scale, s);
  if (in.dtype == GDN_BF16 && o_dtype == GDN_F32)
    return launch_tc<bf16, float>(p, layer, seq, in, o, scale, s);
  return launch_tc<bf16, bf16>(p, layer, seq, in, o, scale, s);
}

}  // namespace gdn
