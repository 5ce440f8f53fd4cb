// Chunked prefill on the 5th-generation tensor cores (tcgen05, kind::tf32),
// for dk = dv = 128.
//
// One CTA (128 threads) per (sequence, value head) walks the sequence in
// 64-token chunks.  The float32 state S [dv][dk] lives in tensor memory for
// the whole call (TMEM columns 0..127, row v in lane v) and is the A operand
// of the state-dependent products, so it never leaves the SM between chunks.
// Per chunk (notation of the chunked delta rule, b70-optimization-lab research
// plan, "What the research found": the (I+A)^{-1} UT transform):
//   MMA1  D1 = [Q;K] K^T                     -> A = beta e^{dG} KK^T (strict),
//                                              P = e^{dG} QK^T (lower, incl. diag)
//   solve (I + A) [W | U] = [diag(beta gamma) K | diag(beta) V]   (CUDA cores)
//   MMA2  D2 = S W^T,  MMA3  D3 = S Q^T      -> Delta^T = U^T - D2
//   MMA4  D4 = Delta^T P^T                    -> O^T = diag(gamma) D3 + D4
//   MMA5  D5 = Delta^T Ktil, Ktil = diag(e^{G_n - G}) K  -> S <- gamma_n S + D5
// Everything that is not S-dependent (the stage, MMA1, the solve) is on the
// chunk's critical path too in this version.  Operands are K-major,
// no-swizzle core-matrix tiles in shared memory (see gdn_tc.cuh).
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int C = kChunk;   // 64
constexpr int D = 128;      // dk = dv
constexpr int NT = 128;     // threads
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
constexpr uint32_t T_S = 0, T_D1 = 128, T_D2 = 192, T_D3 = 256, T_D4 = 320, T_D5 = 384;
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
  const uint32_t lrow = tm + ((uint32_t)(32 * warp) << 16);  // this warp's TMEM lanes

  // state row tid -> TMEM (lane tid, columns 0..127)
  {
    const float4 *src = reinterpret_cast<const float4 *>(Sg + (int64_t)tid * D);
#pragma unroll 1
    for (int c = 0; c < D / 16; ++c) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 x = src[c * 4 + j];
        v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
      }
      tc::tmem_st16(lrow + T_S + c * 16, v);
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

    // ---- S0: stage normalised q, k (core tiles), beta v (plain), g, beta
    for (int t = warp; t < C; t += NT / 32) {
      const bool real = t < n;
      const int64_t tok = lo + c0 + t;
      float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f), k4 = q4, v4 = q4;
      float gt = 0.f, bt = 0.f;
      if (real) {
        q4 = Elem<TI>::load4(qg + tok * in.ld_qk + (int64_t)hk * D + 4 * lane);
        k4 = Elem<TI>::load4(kg + tok * in.ld_qk + (int64_t)hk * D + 4 * lane);
        v4 = Elem<TI>::load4(vg + tok * in.ld_v + (int64_t)h * D + 4 * lane);
        gt = Elem<TI>::load1(gg + tok * p.h_v + h);
        bt = Elem<TI>::load1(bg + tok * p.h_v + h);
      }
      const float qq = group_sum<32>(dot4(q4, q4));
      const float kk = group_sum<32>(dot4(k4, k4));
      *reinterpret_cast<float4 *>(QK + tc::core_off(t, 4 * lane, D)) =
          scale4(rsqrtf(qq + kL2Eps), q4);
      *reinterpret_cast<float4 *>(QK + tc::core_off(64 + t, 4 * lane, D)) =
          scale4(rsqrtf(kk + kL2Eps), k4);
      *reinterpret_cast<float4 *>(XU + t * XS + 4 * lane) = scale4(bt, v4);
      if (lane == 0) {
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
    // meanwhile: W right-hand side (beta gamma k, plain) and Ktil^T tile
    for (int e = tid; e < C * (D / 4); e += NT) {
      const int t = e % C, c4 = e / C;
      const float4 k4 = *reinterpret_cast<const float4 *>(QK + tc::core_off(64 + t, 4 * c4, D));
      *reinterpret_cast<float4 *>(XW + t * XS + 4 * c4) = scale4(sBeta[t] * sGam[t], k4);
    }
    {
      const int kc = tid;  // row k of Ktil^T
#pragma unroll 4
      for (int i4 = 0; i4 < C / 4; ++i4) {
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
    if (warp >= 2) {
      const int t = tid - 64;
      const float bt = sBeta[t], gt = sG[t];
#pragma unroll 1
      for (int cb = 0; cb < C / 16; ++cb) {
        float v[16];
        tc::tmem_ld16(lrow + T_D1 + cb * 16, v);
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          float4 a;
          const int i = cb * 16 + j;
          a.x = i + 0 < t ? bt * expf(gt - sG[i + 0]) * v[j + 0] : 0.f;
          a.y = i + 1 < t ? bt * expf(gt - sG[i + 1]) * v[j + 1] : 0.f;
          a.z = i + 2 < t ? bt * expf(gt - sG[i + 2]) * v[j + 2] : 0.f;
          a.w = i + 3 < t ? bt * expf(gt - sG[i + 3]) * v[j + 3] : 0.f;
          *reinterpret_cast<float4 *>(AP + t * AS + i) = a;
        }
      }
    }
    __syncthreads();

    // ---- S3: forward substitution (I + A) X = RHS; thread = one W and one U column
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      float *Xc = (pass == 0 ? XW : XU) + tid;
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
    if (warp < 2) {
      const int t = tid;
      const float gt = sG[t];
#pragma unroll 1
      for (int cb = 0; cb < C / 16; ++cb) {
        float v[16];
        tc::tmem_ld16(lrow + T_D1 + cb * 16, v);
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          float4 pv;
          const int i = cb * 16 + j;
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
        tc::mma_ts(tm + T_D2, tm + T_S + j * 8, tc::smem_desc(k_s + j * KSTEP, tc::kLBO, SBO_D), id,
                   j > 0);
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
        tc::mma_ts(tm + T_D3, tm + T_S + j * 8, tc::smem_desc(qk_s + j * KSTEP, tc::kLBO, SBO_D),
                   id, j > 0);
      tc::mma_commit(&bar);
    }
    alive = __syncthreads_and(mbar_wait_bounded(&bar, phase));
    if (!alive) break;
    phase ^= 1;
    tc::fence_after_sync();

    // ---- S6: Delta^T[v][t] = U[t][v] - D2[v][t]  (tile, K = t);  o part = gamma_t D3[v][t]
    float op[C];
    {
      const int v = tid;
#pragma unroll
      for (int cb = 0; cb < C / 16; ++cb) {
        float d2[16], d3[16];
        tc::tmem_ld16(lrow + T_D2 + cb * 16, d2);
        tc::tmem_ld16(lrow + T_D3 + cb * 16, d3);
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          const int t = cb * 16 + j;
          float4 dd;
          dd.x = XU[(t + 0) * XS + v] - d2[j + 0];
          dd.y = XU[(t + 1) * XS + v] - d2[j + 1];
          dd.z = XU[(t + 2) * XS + v] - d2[j + 2];
          dd.w = XU[(t + 3) * XS + v] - d2[j + 3];
          *reinterpret_cast<float4 *>(XW + tc::core_off(v, t, C)) = dd;
#pragma unroll
          for (int q = 0; q < 4; ++q) op[t + q] = sGam[t + q] * d3[j + q];
        }
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---- S7: MMA4  D4 = Delta^T P^T (N 64),  MMA5  D5 = Delta^T Ktil (N 128); K = 64
    if (tid == 0) {
#pragma unroll
      for (int j = 0; j < C / 8; ++j)
        tc::mma_ss(tm + T_D4, tc::smem_desc(dt_s + j * KSTEP, tc::kLBO, SBO_C),
                   tc::smem_desc(p_s + j * KSTEP, tc::kLBO, SBO_C), tc::idesc_tf32(128, 64), j > 0);
#pragma unroll
      for (int j = 0; j < C / 8; ++j)
        tc::mma_ss(tm + T_D5, tc::smem_desc(dt_s + j * KSTEP, tc::kLBO, SBO_C),
                   tc::smem_desc(kt_s + j * KSTEP, tc::kLBO, SBO_C), tc::idesc_tf32(128, 128),
                   j > 0);
      tc::mma_commit(&bar);
    }
    alive = __syncthreads_and(mbar_wait_bounded(&bar, phase));
    if (!alive) break;
    phase ^= 1;
    tc::fence_after_sync();

    // ---- S8: outputs and the state update
    {
      const int v = tid;
      TO *ob = o + (lo + c0) * p.h_v * D + (int64_t)h * D + v;
#pragma unroll
      for (int cb = 0; cb < C / 16; ++cb) {
        float d4[16];
        tc::tmem_ld16(lrow + T_D4 + cb * 16, d4);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = cb * 16 + j;
          if (t < n) Elem<TO>::store1(ob + (int64_t)t * p.h_v * D, scale * (op[t] + d4[j]));
        }
      }
      const float gn = sGam[C - 1];
#pragma unroll 1
      for (int cb = 0; cb < D / 16; ++cb) {
        float s[16], d5[16];
        tc::tmem_ld16(lrow + T_S + cb * 16, s);
        tc::tmem_ld16(lrow + T_D5 + cb * 16, d5);
#pragma unroll
        for (int j = 0; j < 16; ++j) s[j] = gn * s[j] + d5[j];
        tc::tmem_st16(lrow + T_S + cb * 16, s);
      }
      tc::tmem_st_wait();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
  }

  if (alive) {
    float4 *dst = reinterpret_cast<float4 *>(Sg + (int64_t)tid * D);
#pragma unroll 1
    for (int c = 0; c < D / 16; ++c) {
      float v[16];
      tc::tmem_ld16(lrow + T_S + c * 16, v);
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
