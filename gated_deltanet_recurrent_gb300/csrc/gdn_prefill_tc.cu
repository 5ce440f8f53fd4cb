// Chunked prefill on the 5th-generation tensor cores (tcgen05, kind::tf32),
// for dk = dv = 128.
//
// One CTA (256 threads) per (sequence, value head) walks the sequence in
// 64-token chunks.  The float32 state S [dv][dk] lives in tensor memory for
// the whole call (TMEM columns 0..127, row v in lane v) and is the A operand
// of the state products, so it never leaves the SM between chunks.
// The chunked delta rule (b70-optimization-lab research plan, "What the
// research found": the (I+A)^{-1} UT transform) gives, with T = (I + A)^{-1},
//   W = T diag(beta gamma) K,  U = T diag(beta) V,  Delta = U - W S^T.
// Re-associating, Delta^T = F T^T with F = diag(beta) (V^T - E diag(gamma))
// and E = S K^T, so W and U are never formed and the only triangular work is
// the 64 x 64 inverse T.  Per chunk:
//   MMA1  D1 = [Q;K] K^T,  MMAE  E = S K^T,  MMA3  D3 = S Q^T     (one batch)
//         -> A = beta e^{dG} KK^T (strict), P = e^{dG} QK^T (lower, incl. diag),
//            F into TMEM, S <- gamma_n S;  T = (I + A)^{-1} by 16 x 16 blocks
//   MMAD  Dd = F T^T                 (= Delta^T, stays in TMEM)
//   MMA4  D4 = Delta^T P^T  -> O^T = diag(gamma) D3 + D4
//   MMA5  S += Delta^T Ktil,  Ktil = diag(e^{G_n - G}) K
// TMEM lanes are split over warps w and w+4 (same lane quadrant, column
// halves).  Operands are K-major, no-swizzle core-matrix tiles in shared
// memory (see gdn_tc.cuh); F and Delta^T are A operands read from TMEM.
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int C = kChunk;   // 64
constexpr int D = 128;      // dk = dv
constexpr int NT = 256;     // threads
constexpr int XS = D + 4;   // plain row stride (floats) of the staged values
constexpr int AS = C + 4;   // plain row stride of A and of T

// shared-memory map (bytes)
constexpr int OFF_QK = 0;                          // [Q;K] core tile, 128 x 128
constexpr int OFF_XU = OFF_QK + 128 * D * 4;       // beta v (plain 64 x XS)
constexpr int OFF_AP = OFF_XU + C * XS * 4;        // A (plain 64 x AS)
constexpr int OFF_TP = OFF_AP + C * AS * 4;        // T (plain 64 x AS)
constexpr int OFF_PT = OFF_TP + C * AS * 4;        // P tile [t][i], 64 x 64
constexpr int OFF_TT = OFF_PT + C * C * 4;         // T tile [t][i], 64 x 64
constexpr int OFF_KT = OFF_TT + C * C * 4;         // Ktil^T tile [k][i], 128 x 64
constexpr int OFF_MS = OFF_KT + D * C * 4;         // block-inverse scratch, 3 x 16 x 16
constexpr int OFF_SC = OFF_MS + 3 * 256 * 4;       // scalars
constexpr int SMEM_BYTES = OFF_SC + 4 * C * 4 + 64;
static_assert(OFF_PT % 16 == 0 && OFF_TT % 16 == 0 && OFF_KT % 16 == 0, "tile alignment");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

// TMEM columns
constexpr uint32_t T_S = 0, T_D1 = 128, T_E = 192, T_D3 = 256, T_F = 320, T_DD = 384,
                   T_D4 = 448;
constexpr uint32_t TMEM_COLS = 512;

template <typename TI, typename TO>
__global__ void __launch_bounds__(NT, 1)
    prefill_tc_kernel(PoolView p, int layer, SeqIndex seq, QKV in, TO *__restrict__ o,
                      float scale) {
  extern __shared__ __align__(1024) unsigned char smem[];
  float *QK = reinterpret_cast<float *>(smem + OFF_QK);
  float *XU = reinterpret_cast<float *>(smem + OFF_XU);
  float *AP = reinterpret_cast<float *>(smem + OFF_AP);
  float *TP = reinterpret_cast<float *>(smem + OFF_TP);
  float *PT = reinterpret_cast<float *>(smem + OFF_PT);
  float *TT = reinterpret_cast<float *>(smem + OFF_TT);
  float *KT = reinterpret_cast<float *>(smem + OFF_KT);
  float *MS = reinterpret_cast<float *>(smem + OFF_MS);
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
  // T is lower triangular: its strictly-upper 16 x 16 blocks stay zero
  for (int e = tid; e < C * C; e += NT) {
    const int r = e / C, c = e % C;
    if ((c >> 4) > (r >> 4)) TP[r * AS + c] = 0.f;
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
  const uint32_t pt_s = smem_addr(PT);
  const uint32_t tt_s = smem_addr(TT);
  const uint32_t kt_s = smem_addr(KT);
  constexpr uint32_t SBO_D = tc::sbo_bytes(D);  // 4096
  constexpr uint32_t SBO_C = tc::sbo_bytes(C);  // 2048
  constexpr uint32_t KSTEP = 2 * tc::kLBO;      // one K = 8 step spans two core matrices
  uint32_t phase = 0;
  bool alive = true;

  for (int c0 = 0; c0 < len && alive; c0 += C) {
    const int n = min(C, len - c0);

    // ---- P0: stage normalised q, k (core tiles), beta v (plain), g, beta.
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

    // ---- P1: MMA1 D1 = [Q;K] K^T  (M 128, N 64, K 128)
    if (tid == 0) {
      constexpr uint32_t id = tc::idesc_tf32(128, 64);
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
        tc::mma_ss(tm + T_D1, tc::smem_desc(qk_s + j * KSTEP, tc::kLBO, SBO_D),
                   tc::smem_desc(k_s + j * KSTEP, tc::kLBO, SBO_D), id, j > 0);
      tc::mma_commit(&bar);
    }
    // meanwhile: the Ktil^T tile, Ktil = diag(e^{G_n - G}) K
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

    // ---- P2: A (plain) and P (tile) from D1; o part and F from D3 and E; S <- gamma_n S
    const int i0 = 32 * half;  // this warp's half of the 64 chunk columns
    if (quad >= 2) {           // rows 64..127 of D1: A[t][i] = beta_t e^{G_t - G_i} k_t.k_i, i < t
      const int t = row - 64;
      const float bt = sBeta[t], gt = sG[t];
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        float v[16];
        tc::tmem_ld16(lrow + T_D1 + i0 + 16 * cb, v);
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          const int i = i0 + 16 * cb + j;
          float4 a;
          a.x = i + 0 < t ? bt * __expf(gt - sG[i + 0]) * v[j + 0] : 0.f;
          a.y = i + 1 < t ? bt * __expf(gt - sG[i + 1]) * v[j + 1] : 0.f;
          a.z = i + 2 < t ? bt * __expf(gt - sG[i + 2]) * v[j + 2] : 0.f;
          a.w = i + 3 < t ? bt * __expf(gt - sG[i + 3]) * v[j + 3] : 0.f;
          *reinterpret_cast<float4 *>(AP + t * AS + i) = a;
        }
      }
    } else {                   // rows 0..63 of D1: P[t][i] = e^{G_t - G_i} q_t.k_i, i <= t
      const int t = row;
      const float gt = sG[t];
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        float v[16];
        tc::tmem_ld16(lrow + T_D1 + i0 + 16 * cb, v);
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          const int i = i0 + 16 * cb + j;
          float4 pv;
          pv.x = i + 0 <= t ? __expf(gt - sG[i + 0]) * v[j + 0] : 0.f;
          pv.y = i + 1 <= t ? __expf(gt - sG[i + 1]) * v[j + 1] : 0.f;
          pv.z = i + 2 <= t ? __expf(gt - sG[i + 2]) * v[j + 2] : 0.f;
          pv.w = i + 3 <= t ? __expf(gt - sG[i + 3]) * v[j + 3] : 0.f;
          *reinterpret_cast<float4 *>(PT + tc::core_off(t, i, C)) = pv;
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // MMAE  E = S K^T, MMA3  D3 = S Q^T (A = S from TMEM): run while the CUDA cores invert
    if (tid == 0) {
      constexpr uint32_t id = tc::idesc_tf32(128, 64);
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
        tc::mma_ts(tm + T_E, tm + T_S + j * 8, tc::smem_desc(k_s + j * KSTEP, tc::kLBO, SBO_D),
                   id, j > 0);
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
        tc::mma_ts(tm + T_D3, tm + T_S + j * 8,
                   tc::smem_desc(qk_s + j * KSTEP, tc::kLBO, SBO_D), id, j > 0);
      tc::mma_commit(&bar);
    }

    // ---- P3: T = (I + A)^{-1} by 16 x 16 blocks.  First pull the next chunk's
    // q, k, v rows towards L2 so its staging loads do not wait on HBM.
    {
      const int t = tid & (C - 1);
      const int64_t tok = lo + c0 + C + t;
      if (tok < hi) {
        constexpr int LINES = (D * (int)sizeof(TI) + 127) / 128;  // 128-byte lines per row
        const char *qr = reinterpret_cast<const char *>(qg + tok * in.ld_qk + (int64_t)hk * D);
        const char *kr = reinterpret_cast<const char *>(kg + tok * in.ld_qk + (int64_t)hk * D);
        const char *vr = reinterpret_cast<const char *>(vg + tok * in.ld_v + (int64_t)h * D);
        for (int l = tid >> 6; l < 3 * LINES; l += NT / C) {
          const char *base = l < LINES ? qr : (l < 2 * LINES ? kr : vr);
          asm volatile("prefetch.global.L2 [%0];" ::"l"(base + 128 * (l % LINES)));
        }
      }
    }
    if (tid < C) {  // diagonal blocks: column j of (I + A_bb)^{-1} by forward substitution
      const int bb = tid >> 4, j = tid & 15;
      const float *Ab = AP + (16 * bb) * AS + 16 * bb;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float acc = r == j ? 1.f : 0.f;
#pragma unroll
        for (int c = 0; c < r; ++c) acc -= Ab[r * AS + c] * x[c];
        x[r] = acc;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) TP[(16 * bb + r) * AS + 16 * bb + j] = x[r];
    }
    __syncthreads();
#pragma unroll 1
    for (int d = 1; d < 4; ++d) {
      // M_ij = sum_{k=j}^{i-1} A_ik T_kj for the blocks (i, j) = (b + d, b)
      for (int e = tid; e < (4 - d) * 256; e += NT) {
        const int b = e >> 8, r = (e >> 4) & 15, c = e & 15;
        const int bi = b + d;
        float acc = 0.f;
        for (int kb = b; kb < bi; ++kb) {
          const float *ar = AP + (16 * bi + r) * AS + 16 * kb;
          const float *tcol = TP + (16 * kb) * AS + 16 * b + c;
#pragma unroll
          for (int m = 0; m < 16; ++m) acc += ar[m] * tcol[m * AS];
        }
        MS[e] = acc;
      }
      __syncthreads();
      // T_ij = -T_ii M_ij
      for (int e = tid; e < (4 - d) * 256; e += NT) {
        const int b = e >> 8, r = (e >> 4) & 15, c = e & 15;
        const int bi = b + d;
        const float *tr = TP + (16 * bi + r) * AS + 16 * bi;
        const float *mc = MS + (b << 8) + c;
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) acc += tr[m] * mc[m * 16];
        TP[(16 * bi + r) * AS + 16 * b + c] = -acc;
      }
      __syncthreads();
    }
    for (int e = tid; e < C * (C / 4); e += NT) {  // T tile [t][i]
      const int t = e % C, c4 = e / C;
      *reinterpret_cast<float4 *>(TT + tc::core_off(t, 4 * c4, C)) =
          *reinterpret_cast<const float4 *>(TP + t * AS + 4 * c4);
    }
    alive = __syncthreads_and(mbar_wait_bounded(&bar, phase));
    if (!alive) break;
    phase ^= 1;
    tc::fence_after_sync();
    // F[v][t] = beta_t v_t[v] - beta_t gamma_t E[v][t] into TMEM; o part; S <- gamma_n S
    float op[C / 2];  // gamma_t (S Q^T)[v][t] for this warp's half of t
    {
      const int v = row;
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        const int t0 = i0 + 16 * cb;
        float e[16], d3[16], f[16];
        tc::tmem_ld16(lrow + T_E + t0, e);
        tc::tmem_ld16(lrow + T_D3 + t0, d3);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = t0 + j;
          op[16 * cb + j] = sGam[t] * d3[j];
          f[j] = XU[t * XS + v] - sBeta[t] * sGam[t] * e[j];   // F[v][t]
        }
        tc::tmem_st16(lrow + T_F + t0, f);
      }
      const float gn = sGam[C - 1];
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        float sv[16];
        tc::tmem_ld16(lrow + T_S + 64 * half + 16 * cb, sv);
#pragma unroll
        for (int j = 0; j < 16; ++j) sv[j] *= gn;
        tc::tmem_st16(lrow + T_S + 64 * half + 16 * cb, sv);
      }
      tc::tmem_st_wait();
    }

    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---- P4: MMAD  Delta^T = F T^T  (A = F from TMEM, M 128, N 64, K 64)
    if (tid == 0) {
#pragma unroll
      for (int j = 0; j < C / 8; ++j)
        tc::mma_ts(tm + T_DD, tm + T_F + j * 8, tc::smem_desc(tt_s + j * KSTEP, tc::kLBO, SBO_C),
                   tc::idesc_tf32(128, 64), j > 0);
      tc::mma_commit(&bar);
    }
    alive = __syncthreads_and(mbar_wait_bounded(&bar, phase));
    if (!alive) break;
    phase ^= 1;
    tc::fence_after_sync();

    // ---- P5: MMA4  D4 = Delta^T P^T (N 64),  MMA5  S += Delta^T Ktil (N 128); K = 64
    if (tid == 0) {
#pragma unroll
      for (int j = 0; j < C / 8; ++j)
        tc::mma_ts(tm + T_D4, tm + T_DD + j * 8, tc::smem_desc(pt_s + j * KSTEP, tc::kLBO, SBO_C),
                   tc::idesc_tf32(128, 64), j > 0);
#pragma unroll
      for (int j = 0; j < C / 8; ++j)
        tc::mma_ts(tm + T_S, tm + T_DD + j * 8, tc::smem_desc(kt_s + j * KSTEP, tc::kLBO, SBO_C),
                   tc::idesc_tf32(128, 128), 1);
      tc::mma_commit(&bar);
    }
    alive = __syncthreads_and(mbar_wait_bounded(&bar, phase));
    if (!alive) break;
    phase ^= 1;
    tc::fence_after_sync();

    // ---- P6: outputs o[t][v] = scale (gamma_t D3 + D4), this warp's half of t
    {
      const int v = row;
      TO *ob = o + (lo + c0) * p.h_v * D + (int64_t)h * D + v;
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        const int t0 = i0 + 16 * cb;
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
