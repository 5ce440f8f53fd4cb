// Chunked prefill in two launches, for dk = dv = 128 (tcgen05, kind::tf32).
//
// The chunked delta rule (b70-optimization-lab research plan, "What the
// research found": the (I+A)^{-1} UT transform) splits each 64-token chunk
// into work that depends only on the chunk's own keys, queries, gates and
// betas, and work that needs the state carried in from the previous chunk:
//
//   key side (no state):  A = beta e^{dG} K K^T (strict),  T = (I + A)^{-1},
//                         P = e^{dG} Q K^T (lower, incl. diagonal)
//   state side:           E = S K^T,  F = diag(beta) (V^T - E diag(gamma)),
//                         Delta^T = F T^T,  O^T = diag(gamma) S Q^T + Delta^T P^T,
//                         S <- gamma_n S + Delta^T Ktil,  Ktil = diag(e^{G_n - G}) K
//
// Only the state side is sequential along a sequence.  `prep_kernel` runs the
// key side of every (chunk, value head) of the call in parallel (one CTA
// each, two CTAs per SM) and writes P and T as ready-made tensor-core operand
// tiles to a workspace; `seq_kernel` then walks each (sequence, value head)
// chunk by chunk with the state resident in TMEM, fetching each chunk's P and
// T tiles with one bulk copy issued a chunk ahead.  The arithmetic is the
// single-launch kernel's, step for step, so results agree with it.
//
// Workspace: (n_seqs + 1) int32 chunk offsets (256-byte aligned), then per
// (chunk, value head) 32 KiB: the P tile, then the T tile, each 64 x 64 float32
// in the K-major core-matrix layout of gdn_tc.cuh.  Chunks are numbered
// sequence by sequence; offsets[i] is the first chunk of sequence i.
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int C = kChunk;   // 64
constexpr int D = 128;      // dk = dv
constexpr int NT = 256;     // threads of both kernels
constexpr int XS = D + 4;   // plain row stride (floats) of staged values
constexpr int AS = C + 4;   // plain row stride of A and T
constexpr int TILE = C * C; // floats of one 64 x 64 tile
constexpr uint32_t kTileBytes = TILE * 4;

__host__ __device__ inline size_t offsets_bytes(int n_seqs) {
  return (((size_t)n_seqs + 1) * 4 + 255) & ~(size_t)255;
}
__host__ __device__ inline int64_t max_chunks(int n_seqs, int total_tokens) {
  return (int64_t)total_tokens / C + n_seqs;  // >= sum over sequences of ceil(len / 64)
}

__device__ __forceinline__ int seq_chunks(const SeqIndex &seq, int i) {
  const int64_t lo = seq.cu_seqlens[i], hi = seq.cu_seqlens[i + 1];
  if (hi < lo || lo < 0 || hi > seq.total_tokens) return 0;  // the state kernel reports it
  return (int)((hi - lo + C - 1) / C);
}

// offsets[i] = number of chunks before sequence i; offsets[n_seqs] = total.
// Offsets saturate at cap + 1 (only overlapping sequences can exceed the
// workspace's cap chunks; the state kernel rejects them).
__global__ void __launch_bounds__(1024)
    chunk_offsets_kernel(SeqIndex seq, int32_t *off, int64_t cap) {
  __shared__ int64_t part[1024];
  const int n = seq.n_seqs, tid = threadIdx.x;
  const int per = (n + 1023) / 1024;
  const int b = min(n, tid * per), e = min(n, b + per);
  int64_t sum = 0;
  for (int i = b; i < e; ++i) sum += seq_chunks(seq, i);
  part[tid] = sum;
  __syncthreads();
  for (int d = 1; d < 1024; d <<= 1) {  // inclusive scan
    const int64_t add = tid >= d ? part[tid - d] : 0;
    __syncthreads();
    part[tid] += add;
    __syncthreads();
  }
  int64_t run = tid ? part[tid - 1] : 0;
  for (int i = b; i < e; ++i) {
    off[i] = (int32_t)min(run, cap + 1);
    run += seq_chunks(seq, i);
  }
  if (tid == 1023) off[n] = (int32_t)min(part[1023], cap + 1);
}

// Stage normalised q and k of one chunk as the [Q;K] core tile (rows 0..63 Q,
// 64..127 K; padded tokens zero) and g, beta into shared memory.  Warp w takes
// tokens 8w .. 8w+7; lane = token (3 bits) + 8 * chunk group, so a quarter-warp
// writes the 8 rows of one core matrix (contiguous 128 bytes).
template <typename TI, bool WITH_V>
__device__ __forceinline__ void stage_chunk(const QKV &in, const PoolView &p, int h, int hk,
                                            int64_t tok0, int n, float *QK, float *XU,
                                            float *sG, float *sBeta) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tl = lane & 7, cg = lane >> 3;
  const int t = 8 * warp + tl;
  const int64_t tok = tok0 + t;
  const bool real = t < n;
  const TI *qg = static_cast<const TI *>(in.q);
  const TI *kg = static_cast<const TI *>(in.k);
  const TI *vg = static_cast<const TI *>(in.v);
  float4 q4[D / 16], k4[D / 16], v4[D / 16];
#pragma unroll
  for (int j = 0; j < D / 16; ++j) {
    const int c = cg + 4 * j;
    q4[j] = k4[j] = v4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (real) {
      q4[j] = Elem<TI>::load4(qg + tok * in.ld_qk + (int64_t)hk * D + 4 * c);
      k4[j] = Elem<TI>::load4(kg + tok * in.ld_qk + (int64_t)hk * D + 4 * c);
      if (WITH_V) v4[j] = Elem<TI>::load4(vg + tok * in.ld_v + (int64_t)h * D + 4 * c);
    }
  }
  const float gt = real ? Elem<TI>::load1(static_cast<const TI *>(in.g) + tok * p.h_v + h) : 0.f;
  const float bt = real ? Elem<TI>::load1(static_cast<const TI *>(in.beta) + tok * p.h_v + h) : 0.f;
  float qq = 0.f, kk = 0.f;
#pragma unroll
  for (int j = 0; j < D / 16; ++j) {
    qq += dot4(q4[j], q4[j]);
    kk += dot4(k4[j], k4[j]);
  }
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
    if (WITH_V) *reinterpret_cast<float4 *>(XU + t * XS + 4 * c) = scale4(bt, v4[j]);
  }
  if (cg == 0) {
    sG[t] = gt;
    sBeta[t] = bt;
  }
}

// ----------------------------------------------------------------- key side
// shared-memory map of prep_kernel (bytes)
constexpr int P_QK = 0;                        // [Q;K] core tile 128 x 128
constexpr int P_AP = P_QK + 128 * D * 4;       // A (plain 64 x AS)
constexpr int P_TP = P_AP + C * AS * 4;        // T (plain 64 x AS)
constexpr int P_MS = P_TP + C * AS * 4;        // block-inverse scratch 3 x 16 x 16
constexpr int P_SC = P_MS + 3 * 256 * 4;       // G, beta
constexpr int PREP_SMEM = P_SC + 2 * C * 4;
static_assert(2 * (PREP_SMEM + 1024) <= 228 * 1024, "two prep CTAs per SM");

template <typename TI>
__global__ void __launch_bounds__(NT, 2)
    prep_kernel(PoolView p, SeqIndex seq, QKV in, const int32_t *__restrict__ off,
                float *__restrict__ work) {
  extern __shared__ __align__(1024) unsigned char smem[];
  float *QK = reinterpret_cast<float *>(smem + P_QK);
  float *AP = reinterpret_cast<float *>(smem + P_AP);
  float *TP = reinterpret_cast<float *>(smem + P_TP);
  float *MS = reinterpret_cast<float *>(smem + P_MS);
  float *sG = reinterpret_cast<float *>(smem + P_SC);
  float *sBeta = sG + C;
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;

  const int cidx = blockIdx.x, h = blockIdx.y;
  if (cidx >= off[seq.n_seqs]) return;
  int si = 0;  // the sequence holding chunk cidx: the last i with off[i] <= cidx
  for (int b = seq.n_seqs - 1; si < b;) {
    const int m = (si + b + 1) >> 1;
    if (off[m] <= cidx) si = m; else b = m - 1;
  }
  const int64_t lo = seq.cu_seqlens[si], hi = seq.cu_seqlens[si + 1];
  const int c0 = (cidx - off[si]) * C;
  const int64_t rest = hi - lo - c0;
  const int n = rest < C ? (int)rest : C;
  const int hk = h / (p.h_v / p.h_k);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int quad = warp & 3, half = warp >> 2;
  const int row = 32 * quad + lane;

  if (warp == 0) tc::tmem_alloc(&tmem_slot, 64);
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  for (int e = tid; e < C * C; e += NT) {  // T's strictly-upper 16 x 16 blocks stay zero
    const int r = e / C, c = e % C;
    if ((c >> 4) > (r >> 4)) TP[r * AS + c] = 0.f;
  }
  stage_chunk<TI, false>(in, p, h, hk, lo + c0, n, QK, nullptr, sG, sBeta);
  __syncthreads();
  if (warp == 0) {  // cumulative log-decay over the chunk (padded tokens carry g = 0)
    const float a = sG[2 * lane], b = sG[2 * lane + 1];
    float incl = a + b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float up = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += up;
    }
    sG[2 * lane] = incl - b;
    sG[2 * lane + 1] = incl;
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = tmem_slot;
  const uint32_t lrow = tm + ((uint32_t)(32 * quad) << 16);

  // D1 = [Q;K] K^T  (M 128, N 64, K 128)
  if (tid == 0) {
    const uint32_t qk_s = smem_addr(QK), k_s = qk_s + 64 * D * 4;
    constexpr uint32_t SBO_D = tc::sbo_bytes(D), KSTEP = 2 * tc::kLBO;
#pragma unroll
    for (int j = 0; j < D / 8; ++j)
      tc::mma_ss(tm, tc::smem_desc(qk_s + j * KSTEP, tc::kLBO, SBO_D),
                 tc::smem_desc(k_s + j * KSTEP, tc::kLBO, SBO_D), tc::idesc_tf32(128, 64), j > 0);
    tc::mma_commit(&bar);
  }
  const bool alive = __syncthreads_and(mbar_wait_bounded(&bar, 0));
  tc::fence_after_sync();
  float *Pg = work + ((int64_t)cidx * p.h_v + h) * (2 * TILE);
  float *Tg = Pg + TILE;
  if (alive) {
    const int i0 = 32 * half;
    if (quad >= 2) {  // rows 64..127: A[t][i] = beta_t e^{G_t - G_i} k_t.k_i, i < t
      const int t = row - 64;
      const float bt = sBeta[t], gt = sG[t];
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        float v[16];
        tc::tmem_ld16(lrow + i0 + 16 * cb, v);
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
    } else {  // rows 0..63: P[t][i] = e^{G_t - G_i} q_t.k_i, i <= t, straight to the workspace
      const int t = row;
      const float gt = sG[t];
#pragma unroll
      for (int cb = 0; cb < 2; ++cb) {
        float v[16];
        tc::tmem_ld16(lrow + i0 + 16 * cb, v);
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          const int i = i0 + 16 * cb + j;
          float4 pv;
          pv.x = i + 0 <= t ? __expf(gt - sG[i + 0]) * v[j + 0] : 0.f;
          pv.y = i + 1 <= t ? __expf(gt - sG[i + 1]) * v[j + 1] : 0.f;
          pv.z = i + 2 <= t ? __expf(gt - sG[i + 2]) * v[j + 2] : 0.f;
          pv.w = i + 3 <= t ? __expf(gt - sG[i + 3]) * v[j + 3] : 0.f;
          *reinterpret_cast<float4 *>(Pg + tc::core_off(t, i, C)) = pv;
        }
      }
    }
  } else {
    if (tid == 0) raise_error(p.err, GDN_DEVERR_TIMEOUT);
    mbar_wait_bounded(&bar, 0);  // a second bounded chance before TMEM is released
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tm, 64);
  if (!alive) return;

  // T = (I + A)^{-1} by 16 x 16 blocks: diagonal blocks by forward substitution
  // (one column per thread), then block row d below the diagonal from the rows above.
  if (tid < C) {
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
  for (int e = tid; e < C * (C / 4); e += NT) {  // T tile [t][i] -> workspace
    const int t = e % C, c4 = e / C;
    *reinterpret_cast<float4 *>(Tg + tc::core_off(t, 4 * c4, C)) =
        *reinterpret_cast<const float4 *>(TP + t * AS + 4 * c4);
  }
}

// --------------------------------------------------------------- state side
// shared-memory map of seq_kernel (bytes)
constexpr int S_QK = 0;                        // [Q;K] core tile 128 x 128
constexpr int S_XU = S_QK + 128 * D * 4;       // beta v (plain 64 x XS)
constexpr int S_PT = S_XU + C * XS * 4;        // P tile (from the workspace)
constexpr int S_TT = S_PT + TILE * 4;          // T tile (same bulk copy)
constexpr int S_KT = S_TT + TILE * 4;          // Ktil^T tile [k][i], 128 x 64
constexpr int S_SC = S_KT + D * C * 4;         // G, gamma, beta, e^{G_n - G}
constexpr int SEQ_SMEM = S_SC + 4 * C * 4;
static_assert(S_PT % 16 == 0 && S_KT % 16 == 0, "tile alignment");
static_assert(SEQ_SMEM <= 227 * 1024, "shared memory");

// TMEM columns
constexpr uint32_t T_S = 0, T_E = 128, T_D3 = 192, T_F = 256, T_DD = 320, T_D4 = 384;
constexpr uint32_t SEQ_TMEM = 512;

template <typename TI, typename TO>
__global__ void __launch_bounds__(NT, 1)
    seq_kernel(PoolView p, int layer, SeqIndex seq, QKV in, TO *__restrict__ o, float scale,
               const int32_t *__restrict__ off, int64_t cap, const float *__restrict__ work) {
  extern __shared__ __align__(1024) unsigned char smem[];
  float *QK = reinterpret_cast<float *>(smem + S_QK);
  float *XU = reinterpret_cast<float *>(smem + S_XU);
  float *PT = reinterpret_cast<float *>(smem + S_PT);
  float *KT = reinterpret_cast<float *>(smem + S_KT);
  float *sG = reinterpret_cast<float *>(smem + S_SC);
  float *sGam = sG + C;
  float *sBeta = sGam + C;
  float *sDte = sBeta + C;
  __shared__ __align__(8) uint64_t bar;    // MMA completion
  __shared__ __align__(8) uint64_t tbar;   // P / T tiles landed
  __shared__ uint32_t tmem_slot;

  const int h = blockIdx.x, si = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int quad = warp & 3, half = warp >> 2;
  const int row = 32 * quad + lane;
  const int slot = seq.slot_ids[si];
  const bool first = h == 0 && tid == 0;
  if (slot < 0 || slot >= p.n_slots) {
    if (first) raise_error(p.err, GDN_DEVERR_SLOT);
    return;
  }
  const int64_t lo = seq.cu_seqlens[si], hi = seq.cu_seqlens[si + 1];
  if (hi < lo || lo < 0 || hi > seq.total_tokens) {
    if (first) raise_error(p.err, GDN_DEVERR_SEQ);
    return;
  }
  const int len = (int)(hi - lo);
  if (len == 0) return;
  if (off[si] < 0 || off[si + 1] > cap || off[si + 1] - off[si] != (len + C - 1) / C) {
    if (first) raise_error(p.err, GDN_DEVERR_SEQ);  // overlapping sequences
    return;
  }
  const int hk = h / (p.h_v / p.h_k);
  float *Sg = p.state + ((int64_t)layer * p.n_slots + slot) * p.state_slot_elems() +
              (int64_t)h * D * D;
  const float *wsq = work + ((int64_t)off[si] * p.h_v + h) * (2 * TILE);  // chunk 0's tiles
  const int64_t wstep = (int64_t)p.h_v * (2 * TILE);                      // next chunk

  if (warp == 0) tc::tmem_alloc(&tmem_slot, SEQ_TMEM);
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&tbar, 1);
    mbar_fence_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0) {  // chunk 0's P and T tiles
    mbar_arrive_expect_tx(&tbar, 2 * kTileBytes);
    bulk_g2s(PT, wsq, 2 * kTileBytes, &tbar);
  }
  const uint32_t tm = tmem_slot;
  const uint32_t lrow = tm + ((uint32_t)(32 * quad) << 16);
  {  // state row `row`, column half `half` -> TMEM
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
  const uint32_t qk_s = smem_addr(QK);
  const uint32_t k_s = qk_s + 64 * D * 4;
  const uint32_t pt_s = smem_addr(PT);
  const uint32_t tt_s = pt_s + kTileBytes;
  const uint32_t kt_s = smem_addr(KT);
  constexpr uint32_t SBO_D = tc::sbo_bytes(D);
  constexpr uint32_t SBO_C = tc::sbo_bytes(C);
  constexpr uint32_t KSTEP = 2 * tc::kLBO;
  uint32_t phase = 0, tphase = 0;
  bool alive = true;

  for (int c0 = 0; c0 < len && alive; c0 += C) {
    const int n = min(C, len - c0);
    stage_chunk<TI, true>(in, p, h, hk, lo + c0, n, QK, XU, sG, sBeta);
    __syncthreads();
    if (warp == 0) {  // cumulative log-decay (padded tokens carry g = 0)
      const float a = sG[2 * lane], b = sG[2 * lane + 1];
      float incl = a + b;
#pragma unroll
      for (int s = 1; s < 32; s <<= 1) {
        const float up = __shfl_up_sync(0xffffffffu, incl, s);
        if (lane >= s) incl += up;
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

    // E = S K^T, D3 = S Q^T (A = S from TMEM; M 128, N 64, K 128)
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
    // meanwhile: the Ktil^T tile, and the next chunk's rows pulled towards L2
    {
      const int kc = tid & 127;
      const int ib = (tid >> 7) * (C / 8);
#pragma unroll 2
      for (int q = 0; q < C / 8; ++q) {
        const int i4 = ib + ((q + (kc >> 2)) & (C / 8 - 1));
        float4 x;
        x.x = sDte[4 * i4 + 0] * QK[tc::core_off(64 + 4 * i4 + 0, kc, D)];
        x.y = sDte[4 * i4 + 1] * QK[tc::core_off(64 + 4 * i4 + 1, kc, D)];
        x.z = sDte[4 * i4 + 2] * QK[tc::core_off(64 + 4 * i4 + 2, kc, D)];
        x.w = sDte[4 * i4 + 3] * QK[tc::core_off(64 + 4 * i4 + 3, kc, D)];
        *reinterpret_cast<float4 *>(KT + tc::core_off(kc, 4 * i4, C)) = x;
      }
      const int t = tid & (C - 1);
      const int64_t tok = lo + c0 + C + t;
      if (tok < hi) {
        constexpr int LINES = (D * (int)sizeof(TI) + 127) / 128;
        const char *qr = reinterpret_cast<const char *>(qg + tok * in.ld_qk + (int64_t)hk * D);
        const char *kr = reinterpret_cast<const char *>(kg + tok * in.ld_qk + (int64_t)hk * D);
        const char *vr = reinterpret_cast<const char *>(vg + tok * in.ld_v + (int64_t)h * D);
        for (int l = tid >> 6; l < 3 * LINES; l += NT / C) {
          const char *base = l < LINES ? qr : (l < 2 * LINES ? kr : vr);
          asm volatile("prefetch.global.L2 [%0];" ::"l"(base + 128 * (l % LINES)));
        }
      }
    }
    alive = __syncthreads_and(mbar_wait_bounded(&bar, phase));
    if (!alive) break;
    phase ^= 1;
    tc::fence_after_sync();

    // F[v][t] = beta_t v_t[v] - beta_t gamma_t E[v][t] into TMEM; o part; S <- gamma_n S
    const int i0 = 32 * half;
    float op[C / 2];
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
          f[j] = XU[t * XS + v] - sBeta[t] * sGam[t] * e[j];
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
    // this chunk's P and T tiles must have landed
    alive = __syncthreads_and(mbar_wait_bounded(&tbar, tphase));
    if (!alive) break;
    tphase ^= 1;
    tc::fence_after_sync();

    // Delta^T = F T^T  (A = F from TMEM, M 128, N 64, K 64)
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

    // D4 = Delta^T P^T (N 64),  S += Delta^T Ktil (N 128); K = 64
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
    if (tid == 0 && c0 + C < len) {  // the tiles are free again: fetch the next chunk's
      mbar_arrive_expect_tx(&tbar, 2 * kTileBytes);
      bulk_g2s(PT, wsq + (int64_t)(c0 / C + 1) * wstep, 2 * kTileBytes, &tbar);
    }

    // outputs o[t][v] = scale (gamma_t D3 + D4), this warp's half of t
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
    // give outstanding MMA groups and tile copies a second bounded chance to finish
    mbar_wait_bounded(&bar, phase);
    mbar_wait_bounded(&tbar, tphase);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tm, SEQ_TMEM);
}

template <typename TI, typename TO>
cudaError_t launch_t(const PoolView &p, int layer, const SeqIndex &seq, const QKV &in, void *o,
                     float scale, void *work, cudaStream_t s) {
  int32_t *off = static_cast<int32_t *>(work);
  float *tiles = reinterpret_cast<float *>(static_cast<char *>(work) + offsets_bytes(seq.n_seqs));
  const int64_t nc = max_chunks(seq.n_seqs, seq.total_tokens);
  chunk_offsets_kernel<<<1, 1024, 0, s>>>(seq, off, nc);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto prep = prep_kernel<TI>;
  e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, PREP_SMEM);
  if (e != cudaSuccess) return e;
  prep<<<dim3((unsigned)nc, p.h_v), NT, PREP_SMEM, s>>>(p, seq, in, off, tiles);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  auto kern = seq_kernel<TI, TO>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SEQ_SMEM);
  if (e != cudaSuccess) return e;
  kern<<<dim3(p.h_v, seq.n_seqs), NT, SEQ_SMEM, s>>>(p, layer, seq, in, static_cast<TO *>(o),
                                                     scale, off, nc, tiles);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_split_workspace_bytes(int n_seqs, int total_tokens, int h_v) {
  return offsets_bytes(n_seqs) +
         (size_t)max_chunks(n_seqs, total_tokens) * h_v * 2 * kTileBytes;
}

cudaError_t launch_prefill_split(const PoolView &p, int layer, const SeqIndex &seq,
                                 const QKV &in, void *o, gdn_dtype o_dtype, float scale,
                                 void *work, cudaStream_t s) {
  if (p.dk != D || p.dv != D) return cudaErrorNotSupported;
  if (in.dtype == GDN_F32 && o_dtype == GDN_F32)
    return launch_t<float, float>(p, layer, seq, in, o, scale, work, s);
  if (in.dtype == GDN_F32 && o_dtype == GDN_BF16)
    return launch_t<float, bf16>(p, layer, seq, in, o, scale, work, s);
  if (in.dtype == GDN_BF16 && o_dtype == GDN_F32)
    return launch_t<bf16, float>(p, layer, seq, in, o, scale, work, s);
  return launch_t<bf16, bf16>(p, layer, seq, in, o, scale, work, s);
}

}  // namespace gdn
