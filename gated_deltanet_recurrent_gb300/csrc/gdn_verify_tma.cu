// Speculative verify for dk = dv = 128 and T <= 8, with the state head moved
// by the TMA engine and the row dot products on the tensor cores.
//
// One CTA (128 threads) per (slot, value head).  Four tensor-map loads bring
// the head's 128 x 128 float32 state into shared memory in the 128-byte
// swizzled layout, which tcgen05 reads directly as a K-major A operand.  One
// MMA batch computes every row's 2T dot products with the staged, normalised
// keys and queries (D = S [K;Q]^T, M 128, N 16, into TMEM).  Thread v then
// owns state row v: the row-level WY recurrences of the verify (see
// gdn_verify.cu) give its o_t and delta_t, and when the slot commits it
// rebuilds its row in place (the swizzle makes these row-per-thread accesses
// conflict-free) before four tensor-map stores write the head back.
#include <cuda.h>

#include "gdn_rows.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int D = 128;
constexpr int NT = 128;
constexpr int TMX = 8;            // drafts handled here (2T <= 16 MMA columns)
constexpr int NX = 16;            // rows of the [K; Q] operand
constexpr int TILE = D * D * 4;   // 64 KiB
constexpr int SLAB = 128 * 32 * 4;  // 16 KiB: 128 rows x 32 floats (one swizzle column)

// shared-memory map after the 1024-byte alignment pad (bytes)
constexpr int O_X = TILE;                    // [K;Q] core tile 16 x 128
constexpr int O_KK = O_X + NX * D * 4;       // Gram k.k [8][8]
constexpr int O_KQ = O_KK + TMX * TMX * 4;   // Gram k.q [8][8]
constexpr int O_DM = O_KQ + TMX * TMX * 4;   // decay table [9][9]
constexpr int O_SC = O_DM + 96 * 4;          // alpha, beta, G
constexpr int SMEM = 1024 + O_SC + 32 * 4;

// ---- draft staging, once per (slot, key head)
// Workspace of a staged call: per (slot i, key head) a block of kXBlock floats
// -- the [K;Q] core tile X (normalised k rows 0..T-1, q rows T..2T-1, zero
// rows up to NX), then KK and KQ -- and after all of those, per (slot i,
// value head) kGBlock floats: the decay table Dm, then alpha, beta and the
// cumulative G.  The same arithmetic as the verify kernel's own staging, so
// both forms give the same bits; the verify kernel bulk-copies its two blocks
// next to the head instead of loading and reducing the drafts itself.
constexpr int kXBlock = NX * D + 2 * TMX * TMX;  // 2176 floats (8704 bytes)
constexpr int kGBlock = 128;                     // 96 (Dm) + 8 + 8 + 16 floats
static_assert(O_KK == O_X + NX * D * 4 && O_KQ == O_KK + TMX * TMX * 4 &&
                  O_SC == O_DM + 96 * 4 && (kGBlock - 96) * 4 == 32 * 4,
              "staged blocks mirror the shared-memory map");

__host__ __device__ inline size_t verify_stage_bytes(int n, int h_k, int h_v) {
  return (size_t)n * ((size_t)h_k * kXBlock + (size_t)h_v * kGBlock) * 4;
}

// Token t of slot i: pending draft t (deferred round), or new draft t - ap.
__device__ __forceinline__ QKV verify_src(const VerifyArgs &va, bool deferred, int ap, int i,
                                          int t, int64_t &row) {
  const bool pend = deferred && t < ap;
  row = pend ? (int64_t)i * va.T_prev + t : (int64_t)i * va.T + (t - ap);
  return pend ? va.prev : va.in;
}

// Pending drafts replayed first (deferred round only), clamped as the verify
// kernel clamps them (which also raises the error).
__device__ __forceinline__ int verify_pending(const VerifyArgs &va, bool deferred, int i) {
  if (!deferred) return 0;
  const int ap = va.prev_accept[i];
  return ap < 0 ? 0 : (ap > va.T_prev ? va.T_prev : ap);
}

// grid (h_k, n), 128 threads
template <typename TI, bool DEFERRED>
__global__ void __launch_bounds__(NT)
    verify_stage_kernel(int h_v, int h_k, VerifyArgs va, float *__restrict__ st) {
  __shared__ __align__(16) float Xs[NX * D];
  __shared__ float sg[TMX + 1];
  // the verify grid may start now: it issues its head loads before waiting for
  // this grid (a programmatic dependent launch)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int kh = blockIdx.x, i = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ap = verify_pending(va, DEFERRED, i);
  const int T = ap + va.T;
  for (int e = tid; e < (NX - 2 * T) * (D / 4); e += NT) {  // zero the unused rows
    const int r = 2 * T + e / (D / 4), c4 = e % (D / 4);
    *reinterpret_cast<float4 *>(Xs + tc::core_off(r, 4 * c4, D)) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int t = warp; t < T; t += NT / 32) {
    int64_t tok;
    const QKV src = verify_src(va, DEFERRED, ap, i, t, tok);
    float4 q4 = Elem<TI>::load4(static_cast<const TI *>(src.q) + tok * src.ld_qk + (int64_t)kh * D + 4 * lane);
    float4 k4 = Elem<TI>::load4(static_cast<const TI *>(src.k) + tok * src.ld_qk + (int64_t)kh * D + 4 * lane);
    const float qq = group_sum<32>(dot4(q4, q4));
    const float kk = group_sum<32>(dot4(k4, k4));
    *reinterpret_cast<float4 *>(Xs + tc::core_off(t, 4 * lane, D)) = scale4(rsqrtf(kk + kL2Eps), k4);
    *reinterpret_cast<float4 *>(Xs + tc::core_off(T + t, 4 * lane, D)) =
        scale4(rsqrtf(qq + kL2Eps), q4);
  }
  __syncthreads();
  float *xb = st + ((int64_t)i * h_k + kh) * kXBlock;
  for (int e = tid; e < NX * D / 4; e += NT)
    reinterpret_cast<float4 *>(xb)[e] = reinterpret_cast<const float4 *>(Xs)[e];
  // Gram scalars, four lanes per pair (the verify kernel's reduction order)
  for (int e0 = 0; e0 < 2 * T * T; e0 += NT / 4) {
    const int e = e0 + tid / 4, sub4 = tid % 4;
    float acc = 0.f;
    const int which = e / (T * T), ii = (e / T) % T, tt = e % T;
    if (e < 2 * T * T) {
      const int ry = which ? T + tt : tt;
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        const int c = 4 * (4 * j + sub4);
        acc += dot4(*reinterpret_cast<const float4 *>(Xs + tc::core_off(ii, c, D)),
                    *reinterpret_cast<const float4 *>(Xs + tc::core_off(ry, c, D)));
      }
    }
    acc = group_sum<4>(acc);
    if (e < 2 * T * T && sub4 == 0) xb[NX * D + which * TMX * TMX + ii * TMX + tt] = acc;
  }
  // per value head of the group: the decay table, alpha, beta, G
  const int G = h_v / h_k;
  for (int g = 0; g < G; ++g) {
    const int h = kh * G + g;
    float *gbk = st + (int64_t)va.n * h_k * kXBlock + ((int64_t)i * h_v + h) * kGBlock;
    float gt = 0.f;
    if (tid < T) {
      int64_t tok;
      const QKV src = verify_src(va, DEFERRED, ap, i, tid, tok);
      gt = Elem<TI>::load1(static_cast<const TI *>(src.g) + tok * h_v + h);
      gbk[96 + tid] = expf(gt);
      gbk[104 + tid] = Elem<TI>::load1(static_cast<const TI *>(src.beta) + tok * h_v + h);
      sg[tid + 1] = gt;
    }
    __syncthreads();
    if (tid == 0) {  // G_t = g_0 + ... + g_{t-1}, T <= 8 terms
      float acc = 0.f;
      sg[0] = 0.f;
#pragma unroll
      for (int t = 1; t <= TMX; ++t)
        if (t <= T) sg[t] = (acc += sg[t]);
    }
    __syncthreads();
    if (tid <= T) gbk[112 + tid] = sg[tid];
    for (int e = tid; e < (T + 1) * (T + 1); e += NT) {
      const int aa = e / (T + 1), bb = e % (T + 1);
      gbk[aa * (TMX + 1) + bb] = bb <= aa ? expf(sg[aa] - sg[bb]) : 0.f;
    }
    __syncthreads();
  }
}

template <typename TI, typename TO, bool DEFERRED>
__global__ void __launch_bounds__(NT)
    verify_tma_kernel(PoolView p, const __grid_constant__ CUtensorMap tmap, int layer,
                      VerifyArgs va, TO *__restrict__ o, const float *__restrict__ staged) {
  const bool pre = staged != nullptr;  // the drafts were staged by verify_stage_kernel
  extern __shared__ __align__(1024) unsigned char dsm[];
  unsigned char *base = dsm + ((1024u - (smem_addr(dsm) & 1023u)) & 1023u);
  unsigned char *tile = base;
  float *X = reinterpret_cast<float *>(base + O_X);
  float *KK = reinterpret_cast<float *>(base + O_KK);
  float *KQ = reinterpret_cast<float *>(base + O_KQ);
  float *Dm = reinterpret_cast<float *>(base + O_DM);
  float *sal = reinterpret_cast<float *>(base + O_SC);
  float *sbe = sal + TMX;
  float *sG = sbe + TMX;
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;

  const int h = blockIdx.x, i = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = va.slot_ids[i];
  if (slot < 0 || slot >= p.n_slots) {
    if (h == 0 && tid == 0) raise_error(p.err, GDN_DEVERR_SLOT);
    return;
  }
  const int row0 = ((layer * p.n_slots + slot) * p.h_v + h) * D;  // tensor-map row
  const int hk = h / (p.h_v / p.h_k);
  if (warp == 0) tc::tmem_alloc(&tmem_slot, 32);
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }

  int ap = 0;  // pending drafts replayed first (deferred commit only)
  if constexpr (DEFERRED) {
    ap = va.prev_accept[i];
    if (ap < 0 || ap > va.T_prev) {
      if (h == 0 && tid == 0) raise_error(p.err, GDN_DEVERR_COUNT);
      ap = ap < 0 ? 0 : va.T_prev;
    }
  }
  const int T = ap + va.T;  // <= TMX (checked by the launcher)
  int a = DEFERRED ? ap : (va.commit_all ? T : (va.accept_len ? va.accept_len[i] : 0));
  if (a < 0 || a > T) {
    if (h == 0 && tid == 0) raise_error(p.err, GDN_DEVERR_COUNT);
    a = a < 0 ? 0 : T;
  }
  // token t of this slot's sequence: pending draft t, or new draft t - ap
  // (register copies: no address of the parameter block is taken)
  const QKV cur = va.in, prv = va.prev;
  const int T_new = va.T, T_old = va.T_prev;
  auto src_of = [&](int t, int64_t &row) -> QKV {
    const bool pend = DEFERRED && t < ap;
    row = pend ? (int64_t)i * T_old + t : (int64_t)i * T_new + (t - ap);
    return pend ? prv : cur;
  };
  // ---- the drafts' loads go out before the head's: they are small and every
  // step after them waits on them, while the head is needed only by the MMA.
  // Warp w takes tokens w and w + 4 (q and k rows), thread v its row's v of
  // each token, threads t < T the gates.
  float4 q4[2], k4[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int t = warp + 4 * r;
    q4[r] = k4[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!pre && t < T) {
      int64_t tok;
      const QKV src = src_of(t, tok);
      q4[r] = Elem<TI>::load4(static_cast<const TI *>(src.q) + tok * src.ld_qk + (int64_t)hk * D + 4 * lane);
      k4[r] = Elem<TI>::load4(static_cast<const TI *>(src.k) + tok * src.ld_qk + (int64_t)hk * D + 4 * lane);
    }
  }
  const int v = tid;  // this thread's state row
  float vr[TMX];
#pragma unroll
  for (int t = 0; t < TMX; ++t) {
    vr[t] = 0.f;
    if (t < T) {
      int64_t tok;
      const QKV src = src_of(t, tok);
      vr[t] = Elem<TI>::load1(static_cast<const TI *>(src.v) + tok * src.ld_v + (int64_t)h * D + v);
    }
  }
  float gt = 0.f, bt = 0.f;
  if (!pre && tid < T) {
    int64_t tok;
    const QKV src = src_of(tid, tok);
    gt = Elem<TI>::load1(static_cast<const TI *>(src.g) + tok * p.h_v + h);
    bt = Elem<TI>::load1(static_cast<const TI *>(src.beta) + tok * p.h_v + h);
  }
  tc::fence_before_sync();
  __syncthreads();  // the barrier is initialised
  tc::fence_after_sync();
  const uint32_t tm = tmem_slot;
  if (tid == 0) {  // the head: four tensor-map loads in the 128-byte swizzle
    mbar_arrive_expect_tx(&bar, TILE + (pre ? (kXBlock + kGBlock) * 4 : 0));
#pragma unroll
    for (int s = 0; s < 4; ++s)
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
          "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(tile + s * SLAB)),
          "l"(reinterpret_cast<uint64_t>(&tmap)), "r"(32 * s), "r"(row0), "r"(smem_addr(&bar))
          : "memory");
    if (pre) {  // the staged [K;Q] tile with KK, KQ, and this head's decays and gates,
                // once the staging grid has completed
      asm volatile("griddepcontrol.wait;" ::: "memory");
      bulk_g2s(X, staged + ((int64_t)i * p.h_k + hk) * kXBlock, kXBlock * 4, &bar);
      bulk_g2s(Dm, staged + (int64_t)va.n * p.h_k * kXBlock + ((int64_t)i * p.h_v + h) * kGBlock,
               kGBlock * 4, &bar);
    }
  }
  if (!pre) {
  for (int e = tid; e < (NX - 2 * T) * (D / 4); e += NT) {  // zero the unused X rows
    const int r = 2 * T + e / (D / 4), c4 = e % (D / 4);
    *reinterpret_cast<float4 *>(X + tc::core_off(r, 4 * c4, D)) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {  // normalised k and q rows of the [K;Q] tile
    const int t = warp + 4 * r;
    if (t < T) {
      const float qq = group_sum<32>(dot4(q4[r], q4[r]));
      const float kk = group_sum<32>(dot4(k4[r], k4[r]));
      *reinterpret_cast<float4 *>(X + tc::core_off(t, 4 * lane, D)) =
          scale4(rsqrtf(kk + kL2Eps), k4[r]);
      *reinterpret_cast<float4 *>(X + tc::core_off(T + t, 4 * lane, D)) =
          scale4(rsqrtf(qq + kL2Eps), q4[r]);
    }
  }
  if (tid < T) {  // g_t into sG[t + 1] (summed below), alpha_t, beta_t
    sG[tid + 1] = gt;
    sal[tid] = expf(gt);
    sbe[tid] = bt;
  }
  __syncthreads();
  if (tid == 0) {  // G_t = g_0 + ... + g_{t-1}, T <= 8 terms
    float acc = 0.f;
    sG[0] = 0.f;
#pragma unroll
    for (int t = 1; t <= TMX; ++t)
      if (t <= T) sG[t] = (acc += sG[t]);
  }
  __syncthreads();
  // Gram scalars (four lanes per pair) and the decay table
  for (int e0 = 0; e0 < 2 * T * T; e0 += NT / 4) {
    const int e = e0 + tid / 4, sub4 = tid % 4;
    float acc = 0.f;
    const int which = e / (T * T), ii = (e / T) % T, tt = e % T;
    if (e < 2 * T * T) {
      const int ry = which ? T + tt : tt;
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        const int c = 4 * (4 * j + sub4);
        acc += dot4(*reinterpret_cast<const float4 *>(X + tc::core_off(ii, c, D)),
                    *reinterpret_cast<const float4 *>(X + tc::core_off(ry, c, D)));
      }
    }
    acc = group_sum<4>(acc);
    if (e < 2 * T * T && sub4 == 0) (which ? KQ : KK)[ii * TMX + tt] = acc;
  }
  for (int e = tid; e < (T + 1) * (T + 1); e += NT) {
    const int aa = e / (T + 1), bb = e % (T + 1);
    Dm[aa * (TMX + 1) + bb] = bb <= aa ? expf(sG[aa] - sG[bb]) : 0.f;
  }
  }  // !pre
  tc::fence_async_smem();
  tc::fence_before_sync();
  bool alive = __syncthreads_and(mbar_wait_bounded(&bar, 0));
  tc::fence_after_sync();

  // ---- D[v][t'] = S[v][:] . X[t'][:]  (M 128, N 16, K 128)
  if (alive && tid == 0) {
    const uint32_t t_s = smem_addr(tile), x_s = smem_addr(X);
#pragma unroll
    for (int s = 0; s < 4; ++s)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        tc::mma_ss(tm, tc::smem_desc_sw128(t_s + s * SLAB + j * 32),
                   tc::smem_desc(x_s + (4 * s + j) * 2 * tc::kLBO, tc::kLBO, tc::sbo_bytes(D)),
                   tc::idesc_tf32(128, NX), (s | j) != 0);
    tc::mma_commit(&bar);
  }
  if (alive) alive = __syncthreads_and(mbar_wait_bounded(&bar, 1));
  tc::fence_after_sync();

  if (alive) {
    float dots[16];
    tc::tmem_ld16(tm + ((uint32_t)(32 * warp) << 16), dots);
    float dl[TMX];
    // output of token t >= ap: new draft t - ap of slot i
    TO *ob = o == nullptr ? nullptr : o + ((int64_t)i * va.T * p.h_v + h) * D + v;
#pragma unroll
    for (int t = 0; t < TMX; ++t) {
      dl[t] = 0.f;
      if (t < T) {
        float pt = Dm[t * (TMX + 1)] * dots[t];
#pragma unroll
        for (int ii = 0; ii < TMX; ++ii)
          if (ii < t) pt += Dm[t * (TMX + 1) + ii + 1] * dl[ii] * KK[ii * TMX + t];
        dl[t] = sbe[t] * (vr[t] - sal[t] * pt);
        if (ob != nullptr && (!DEFERRED || t >= ap)) {
          float dq = 0.f;  // dots[T + t] without a runtime register index
#pragma unroll
          for (int u = 0; u < 16; ++u)
            if (u == T + t) dq = dots[u];
          float ot = Dm[(t + 1) * (TMX + 1)] * dq;
#pragma unroll
          for (int ii = 0; ii < TMX; ++ii)
            if (ii <= t) ot += Dm[(t + 1) * (TMX + 1) + ii + 1] * dl[ii] * KQ[ii * TMX + t];
          Elem<TO>::store1(ob + (int64_t)(t - ap) * p.h_v * D, va.scale * ot);
        }
      }
    }
    if (a > 0) {  // rebuild row v at the accepted length, in place (swizzled)
      const float c0 = Dm[a * (TMX + 1)];
      float cf[TMX];
#pragma unroll
      for (int ii = 0; ii < TMX; ++ii) cf[ii] = ii < a ? Dm[a * (TMX + 1) + ii + 1] * dl[ii] : 0.f;
      unsigned char *rowp = tile + (v >> 3) * 1024 + (v & 7) * 128;
      // One 128-byte segment (8 float4, one slab) at a time: all of its loads
      // are issued before any of its stores, since the row and X share memory.
#pragma unroll 1
      for (int s = 0; s < D / 32; ++s) {
        float4 *sp = reinterpret_cast<float4 *>(rowp + s * SLAB);
        float4 acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = scale4(c0, sp[j ^ (v & 7)]);
#pragma unroll
        for (int ii = 0; ii < TMX; ++ii)
          if (ii < a) {
            const float *xr = X + tc::core_off(ii, 32 * s, D);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              acc[j] = axpby4(1.f, acc[j], cf[ii], *reinterpret_cast<const float4 *>(xr + 32 * j));
          }
#pragma unroll
        for (int j = 0; j < 8; ++j) sp[j ^ (v & 7)] = acc[j];
      }
      tc::fence_async_smem();
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (alive && a > 0 && tid == 0) {
#pragma unroll
    for (int s = 0; s < 4; ++s)
      asm volatile(
          "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
              reinterpret_cast<uint64_t>(&tmap)),
          "r"(32 * s), "r"(row0), "r"(smem_addr(tile + s * SLAB))
          : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  }
  if (!alive) {
    if (tid == 0) raise_error(p.err, GDN_DEVERR_TIMEOUT);
    mbar_wait_bounded(&bar, 0);
    mbar_wait_bounded(&bar, 1);
  }
  tc::fence_after_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tm, 32);
}

template <typename TI, typename TO>
cudaError_t launch_t(const PoolView &p, const CUtensorMap &tmap, int layer, const VerifyArgs &va,
                     void *o, cudaStream_t s) {
  const bool deferred = va.prev.q != nullptr && va.prev_accept != nullptr;
  if (va.stage != nullptr) {  // the drafts staged once per (slot, key head)
    auto stage = deferred ? verify_stage_kernel<TI, true> : verify_stage_kernel<TI, false>;
    stage<<<dim3(p.h_k, va.n), NT, 0, s>>>(p.h_v, p.h_k, va, va.stage);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  auto kern = deferred ? verify_tma_kernel<TI, TO, true> : verify_tma_kernel<TI, TO, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.h_v, va.n);
  if (va.stage == nullptr) {
    kern<<<grid, NT, SMEM, s>>>(p, tmap, layer, va, static_cast<TO *>(o), va.stage);
    return cudaGetLastError();
  }
  // a programmatic dependent of the staging grid: heads load while it runs
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, tmap, layer, va, static_cast<TO *>(o),
                            static_cast<const float *>(va.stage));
}

}  // namespace

size_t verify_stage_workspace_bytes(const PoolView &p, const VerifyArgs &va) {
  // Staged drafts pay off from five tokens per slot (measured on the 128-slot
  // case: 4 tokens 108.7 -> 113.8 us, a deferred round of up to 8 tokens
  // 151.9 -> 139.1 us); with fewer, each block stages its own.
  if (p.state_dtype != GDN_F32 || p.dk != D || p.dv != D || va.T + va.T_prev > TMX ||
      va.T + va.T_prev <= 4)
    return 0;
  return verify_stage_bytes(va.n, p.h_k, p.h_v);
}

cudaError_t launch_verify_tma(const PoolView &p, const void *tmap, int layer,
                              const VerifyArgs &va, void *o, gdn_dtype o_dtype, cudaStream_t s) {
  if (tmap == nullptr || p.state_dtype != GDN_F32 || p.dk != D || p.dv != D ||
      va.T + va.T_prev > TMX)
    return cudaErrorNotSupported;
  const CUtensorMap &m = *static_cast<const CUtensorMap *>(tmap);
  if (va.in.dtype == GDN_F32 && o_dtype == GDN_F32) return launch_t<float, float>(p, m, layer, va, o, s);
  if (va.in.dtype == GDN_F32 && o_dtype == GDN_BF16) return launch_t<float, bf16>(p, m, layer, va, o, s);
  if (va.in.dtype == GDN_BF16 && o_dtype == GDN_F32) return launch_t<bf16, float>(p, m, layer, va, o, s);
  return launch_t<bf16, bf16>(p, m, layer, va, o, s);
}

}  // namespace gdn
