// Decode step over a slot-indexed pool of Gated DeltaNet states.
//
// HBM-bound: per active slot and value head the [dv][dk] float32 state is
// streamed from HBM once and written back once.  The rule
// S <- alpha S (I - beta k k^T) + beta v k^T, o = S q acts on each state row
// independently:
//     p_r   = S_r . k                      (row r of S times the key)
//     S_r  <- alpha S_r + beta (v_r - alpha p_r) k
//     o_r   = scale * S_r . q
// so each row goes to a group of dk/4 lanes holding four columns each, and the
// two dot products are reduced with warp shuffles.  q and k are L2-normalised
// in registers at the start of the CTA.
#include "gdn_rows.cuh"

namespace gdn {
namespace {

using rows::kThreads;
using rows::kBulkBytes;
using rows::dispatch;

// Bulk-staged decode: the CTA's 16 KiB state tile (R rows of one head: 32 of
// float32 or 64 of a bf16 / f16 state at dk = 128) is fetched by one cp.async.bulk onto
// an mbarrier, so every CTA has its whole tile in flight from its first cycle
// while its threads normalise q and k; rows are then read from shared memory,
// widened to float32, updated, and stored back (rounded to the state's
// storage type) with streaming stores.  grid (ceil(dv / R), h_v, n).
// AFTER_CONV: launched as a programmatic dependent of the conv that writes q,
// k and v; the tile fetch is issued before the grid-dependency wait, every
// read of the token inputs after it.
// HALF: the pool stores its state in bf16 or f16 (else float32, no branch).
template <int DK, typename TI, typename TO, bool AFTER_CONV, bool HALF>
__global__ void __launch_bounds__(kThreads, HALF ? 9 : 10)
    decode_bulk_kernel(PoolView p, int layer, const int32_t *__restrict__ slot_ids, QKV in,
                       TO *__restrict__ o, float scale) {
  constexpr int R = kBulkBytes / (DK * (HALF ? 2 : 4));  // rows per CTA: a 16 KiB tile
  constexpr int LPR = DK / 4, RPP = 32 / LPR;
  constexpr int RPW = R / (kThreads / 32);        // rows per warp
  constexpr int U = 4;
  constexpr int PASSES = RPW / (RPP * U);
  static_assert(PASSES >= 1 && RPW % (RPP * U) == 0, "row mapping");
  __shared__ __align__(128) float4 tile[kBulkBytes / 16];
  __shared__ __align__(8) uint64_t bar;

  const int i = blockIdx.z;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  const int slot = slot_ids[i];
  if (slot < 0 || slot >= p.n_slots) {
    if (blockIdx.x == 0 && h == 0 && tid == 0) raise_error(p.err, GDN_DEVERR_SLOT);
    return;
  }
  const int r0 = blockIdx.x * R;
  const int nrows = min(R, p.dv - r0);
  char *S = p.state_at(p.state_head_elem(layer, slot, h) + (int64_t)r0 * DK);
  const gdn_dtype sd = HALF ? p.state_dtype : GDN_F32;
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t bytes = (uint32_t)nrows * DK * p.state_esz();
    // test hook: expect 16 bytes the copy never delivers, so the bounded wait
    // below runs out after the copy itself has landed
    const uint32_t extra = (p.test_flags & GDN_TEST_DECODE_WAIT_TIMEOUT) ? 16u : 0u;
    mbar_arrive_expect_tx(&bar, bytes + extra);
    bulk_g2s(tile, S, bytes, &bar);
  }
  // Returns once the prerequisite grid has completed and its memory is
  // visible (immediately when there is none).
  if (AFTER_CONV) asm volatile("griddepcontrol.wait;" ::: "memory");

  const int lane = tid & 31, warp = tid >> 5;
  const int sub = lane % LPR, grp = lane / LPR;
  const int hk = h / (p.h_v / p.h_k);
  const int64_t qk_off = (int64_t)i * in.ld_qk + (int64_t)hk * DK + 4 * sub;
  float4 q4 = Elem<TI>::load4(static_cast<const TI *>(in.q) + qk_off);
  float4 k4 = Elem<TI>::load4(static_cast<const TI *>(in.k) + qk_off);
  const float kk = group_sum<LPR>(dot4(k4, k4));
  const float qq = group_sum<LPR>(dot4(q4, q4));
  k4 = scale4(rsqrtf(kk + kL2Eps), k4);
  q4 = scale4(rsqrtf(qq + kL2Eps), q4);
  const int64_t gb = (int64_t)i * p.h_v + h;
  const float alpha = expf(Elem<TI>::load1(static_cast<const TI *>(in.g) + gb));
  const float beta = Elem<TI>::load1(static_cast<const TI *>(in.beta) + gb);
  const TI *vp = static_cast<const TI *>(in.v) + (int64_t)i * in.ld_v + (int64_t)h * p.dv + r0;
  TO *op = o + gb * p.dv + r0;
  float vr[PASSES][U];
#pragma unroll
  for (int ps = 0; ps < PASSES; ++ps)
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int rl = warp * RPW + (ps * U + u) * RPP + grp;
      vr[ps][u] = rl < nrows ? Elem<TI>::load1(vp + rl) : 0.f;
    }

  if (!mbar_wait_bounded(&bar, 0)) {
    if (tid == 0) raise_error(p.err, GDN_DEVERR_TIMEOUT);
    mbar_wait_bounded(&bar, 0);  // give the copy a second bounded chance before exiting
    return;
  }

#pragma unroll
  for (int ps = 0; ps < PASSES; ++ps) {
    float4 s[U];
    float acc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int rl = warp * RPW + (ps * U + u) * RPP + grp;
      s[u] = rl < nrows ? state_ld4(tile, (int64_t)rl * DK + 4 * sub, sd)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
      acc[u] = dot4(s[u], k4);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) acc[u] = group_sum<LPR>(acc[u]);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float d = beta * (vr[ps][u] - alpha * acc[u]);
      s[u] = axpby4(alpha, s[u], d, k4);
      acc[u] = dot4(s[u], q4);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) acc[u] = group_sum<LPR>(acc[u]);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int rl = warp * RPW + (ps * U + u) * RPP + grp;
      if (rl < nrows) {
        state_st4<true>(S, (int64_t)rl * DK + 4 * sub, s[u], sd);
        if (sub == 0) Elem<TO>::store1(op + rl, scale * acc[u]);
      }
    }
  }
}

// ---- conv + SiLU, q/k norm and the decode step in one kernel ----
//
// Same grid and state streaming as decode_bulk_kernel.  While its state tile
// is in flight, each CTA computes the conv + SiLU outputs it needs itself:
// the 2*DK q and k channels of its key head and the R v channels of its rows,
// from x, the slot's conv cache and the taps, rounded to the activation dtype
// exactly as the conv kernel stores y.  Outputs, y, cache and state are
// bit-identical to the conv kernel followed by the decode kernel.  Loads that
// do not depend on the slot id (x, taps, g, beta) are issued before it.
//
// Cache update without a grid-wide wait.  A v channel is read by one CTA,
// which shifts its cache in place.  A q/k channel is read by the `readers`
// CTAs that share the key head (value heads of the group x row blocks), so
// its old cache must stay readable until all of them have read it: after its
// reads each CTA takes a ticket for the key head (p.ticks[layer][slot][hk]),
// and the CTA that draws the last one writes the shifted q/k cache (its old
// values are still in its registers) and puts the ticket back to 0.  No CTA
// waits on another; every launch leaves every ticket at 0 (an entry skipped
// for a bad slot id draws none).  The ticket is taken by one thread after a
// CTA barrier (the barrier orders the other threads' cache reads before it,
// as in a grid-wide barrier) and its result is read only after the state
// update, so the round trip stays off the decode's critical path.  The first
// value head of the group, row block 0, writes the q/k part of y.
constexpr int kMaxConvK = 8;

template <typename T>
__device__ __forceinline__ float round_to(float x) {
  return x;
}
template <>
__device__ __forceinline__ float round_to<bf16>(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// One conv channel of one token: taps, raw input and the cached inputs, for
// a conv width W <= WM.
template <int WM>
struct ConvTap {
  float w[WM];
  float b, x;
  float hist[WM - 1];  // the W - 1 cached inputs, oldest first
};

template <int WM, typename T>
__device__ __forceinline__ void tap_load(ConvTap<WM> &t, const T *xrow, const float *w,
                                         const float *bias, int c, int W) {
  const float *wc = w + (int64_t)c * W;
  if (WM == 4 && W == 4 && ((uintptr_t)wc & 15) == 0) {
    const float4 w4 = *reinterpret_cast<const float4 *>(wc);
    t.w[0] = w4.x; t.w[1] = w4.y; t.w[2] = w4.z; t.w[WM - 1] = w4.w;
  } else {
#pragma unroll
    for (int m = 0; m < WM; ++m)
      if (m < W) t.w[m] = wc[m];
  }
  t.b = bias ? bias[c] : 0.f;
  t.x = Elem<T>::load1(xrow + c);
}

template <int WM, typename T>
__device__ __forceinline__ void tap_load_cache(ConvTap<WM> &t, const T *cache, int c, int W) {
  const T *cc = cache + (int64_t)c * (W - 1);
#pragma unroll
  for (int m = 0; m < WM - 1; ++m)
    if (m < W - 1) t.hist[m] = Elem<T>::load1(cc + m);
}

// The conv kernel's arithmetic, in its order, rounded to T as y is stored.
template <int WM, typename T>
__device__ __forceinline__ float tap_conv(const ConvTap<WM> &t, int W) {
  float wl = 0.f;  // t.w[W - 1], selected without a dynamic register index
#pragma unroll
  for (int m = 0; m < WM; ++m)
    if (m == W - 1) wl = t.w[m];
  float u = t.b + wl * t.x;
#pragma unroll
  for (int m = 0; m < WM - 1; ++m)
    if (m < W - 1) u += t.w[m] * t.hist[m];
  return round_to<T>(silu(u));
}

struct ConvStep {
  const void *x;
  int64_t ld_x;
  const float *w;
  const float *bias;
  void *y;
  int64_t ld_y;
  const void *g, *beta;
};

// WM: the largest conv width this instantiation handles (4: exactly 4).
template <int DK, typename TI, typename TO, int WM>
__global__ void __launch_bounds__(kThreads)
    decode_conv_kernel(PoolView p, int layer, const int32_t *__restrict__ slot_ids, ConvStep cs,
                       TO *__restrict__ o, float scale) {
  constexpr int R = kBulkBytes / (DK * 4);
  constexpr int LPR = DK / 4, RPP = 32 / LPR;
  constexpr int RPW = R / (kThreads / 32);
  constexpr int U = 4;
  constexpr int PASSES = RPW / (RPP * U);
  constexpr int NQK = (2 * DK + kThreads - 1) / kThreads;  // q/k channels per thread
  constexpr int NV = (R + kThreads - 1) / kThreads;         // v channels per thread
  constexpr int kTicketThread = kThreads - 1;
  static_assert(PASSES >= 1 && RPW % (RPP * U) == 0, "row mapping");
  __shared__ __align__(128) float4 tile[kBulkBytes / 16];
  __shared__ __align__(16) float sqk[2 * DK];   // conv outputs of q | k (this key head)
  __shared__ float sv[R];                       // conv outputs of this CTA's v rows
  __shared__ TI snew[2 * DK][WM - 1];           // q/k cache after this token (if last)
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_last;

  const int i = blockIdx.z;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  const int slot = slot_ids[i];
  const int group = p.h_v / p.h_k;
  const int hk = h / group;
  const int W = WM == 4 ? 4 : p.conv_k;
  const int nq = p.h_k * DK;
  const int r0 = blockIdx.x * R;
  const int nrows = min(R, p.dv - r0);
  // slot-independent inputs first
  const int64_t gb = (int64_t)i * p.h_v + h;
  const float graw = Elem<TI>::load1(static_cast<const TI *>(cs.g) + gb);
  const float beta = Elem<TI>::load1(static_cast<const TI *>(cs.beta) + gb);
  const TI *xrow = static_cast<const TI *>(cs.x) + (int64_t)i * cs.ld_x;
  auto qk_channel = [&](int j) { return (j < DK ? 0 : nq) + hk * DK + j % DK; };
  ConvTap<WM> tq[NQK], tv[NV];
#pragma unroll
  for (int e = 0; e < NQK; ++e) {
    const int j = tid + e * kThreads;
    if (j < 2 * DK) tap_load<WM, TI>(tq[e], xrow, cs.w, cs.bias, qk_channel(j), W);
  }
#pragma unroll
  for (int e = 0; e < NV; ++e) {
    const int r = tid + e * kThreads;
    if (r < nrows) tap_load<WM, TI>(tv[e], xrow, cs.w, cs.bias, 2 * nq + h * p.dv + r0 + r, W);
  }
  if (slot < 0 || slot >= p.n_slots) {
    if (blockIdx.x == 0 && h == 0 && tid == 0) raise_error(p.err, GDN_DEVERR_SLOT);
    return;
  }
  char *S = p.state_at(p.state_head_elem(layer, slot, h) + (int64_t)r0 * DK);
  const gdn_dtype sd = p.state_dtype;
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t bytes = (uint32_t)nrows * DK * p.state_esz();
    // test hook: expect 16 bytes the copy never delivers, so the bounded wait
    // below runs out after the copy itself has landed
    const uint32_t extra = (p.test_flags & GDN_TEST_DECODE_WAIT_TIMEOUT) ? 16u : 0u;
    mbar_arrive_expect_tx(&bar, bytes + extra);
    bulk_g2s(tile, S, bytes, &bar);
  }

  TI *cache = static_cast<TI *>(p.conv) +
              ((int64_t)layer * p.n_slots + slot) * p.conv_ch * (W - 1);
  TI *yrow = static_cast<TI *>(cs.y) + (int64_t)i * cs.ld_y;
  const bool y_qk_writer = blockIdx.x == 0 && h % group == 0;
#pragma unroll
  for (int e = 0; e < NQK; ++e) {
    const int j = tid + e * kThreads;
    if (j < 2 * DK) tap_load_cache<WM, TI>(tq[e], cache, qk_channel(j), W);
  }
#pragma unroll
  for (int e = 0; e < NV; ++e) {
    const int r = tid + e * kThreads;
    if (r < nrows) tap_load_cache<WM, TI>(tv[e], cache, 2 * nq + h * p.dv + r0 + r, W);
  }
#pragma unroll
  for (int e = 0; e < NQK; ++e) {
    const int j = tid + e * kThreads;
    if (j < 2 * DK) {
      const float yv = tap_conv<WM, TI>(tq[e], W);
      sqk[j] = yv;
      if (y_qk_writer) Elem<TI>::store1(yrow + qk_channel(j), yv);
      // the shifted cache (hist[1 .. W-2], x), kept for the ticket's winner
#pragma unroll
      for (int m = 0; m < WM - 2; ++m)
        if (m < W - 2) Elem<TI>::store1(&snew[j][m], tq[e].hist[m + 1]);
      Elem<TI>::store1(&snew[j][W - 2], tq[e].x);
    }
  }
#pragma unroll
  for (int e = 0; e < NV; ++e) {
    const int r = tid + e * kThreads;
    if (r < nrows) {
      const int c = 2 * nq + h * p.dv + r0 + r;
      const float yv = tap_conv<WM, TI>(tv[e], W);
      sv[r] = yv;
      Elem<TI>::store1(yrow + c, yv);
      // this CTA is the only reader of its v channels: shift in place
      TI *cc = cache + (int64_t)c * (W - 1);
#pragma unroll
      for (int m = 0; m < WM - 2; ++m)
        if (m < W - 2) Elem<TI>::store1(cc + m, tv[e].hist[m + 1]);
      Elem<TI>::store1(cc + (W - 2), tv[e].x);
    }
  }
  __syncthreads();  // every thread's q/k cache reads are done; sqk, sv, snew complete
  unsigned int *ticket = p.ticks + ((int64_t)layer * p.n_slots + slot) * p.h_k + hk;
  unsigned int prev = 0;
  if (tid == kTicketThread) {
    __threadfence();
    prev = atomicAdd(ticket, 1u);  // read only after the state update
  }

  const int lane = tid & 31, warp = tid >> 5;
  const int sub = lane % LPR, grp = lane / LPR;
  float4 q4 = reinterpret_cast<const float4 *>(sqk)[sub];
  float4 k4 = reinterpret_cast<const float4 *>(sqk + DK)[sub];
  const float kk = group_sum<LPR>(dot4(k4, k4));
  const float qq = group_sum<LPR>(dot4(q4, q4));
  k4 = scale4(rsqrtf(kk + kL2Eps), k4);
  q4 = scale4(rsqrtf(qq + kL2Eps), q4);
  const float alpha = expf(graw);
  TO *op = o + gb * p.dv + r0;

  if (mbar_wait_bounded(&bar, 0)) {
#pragma unroll
    for (int ps = 0; ps < PASSES; ++ps) {
      float4 s[U];
      float acc[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int rl = warp * RPW + (ps * U + u) * RPP + grp;
        s[u] = rl < nrows ? state_ld4(tile, (int64_t)rl * DK + 4 * sub, sd)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        acc[u] = dot4(s[u], k4);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = group_sum<LPR>(acc[u]);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int rl = warp * RPW + (ps * U + u) * RPP + grp;
        const float vr = rl < nrows ? sv[rl] : 0.f;
        const float d = beta * (vr - alpha * acc[u]);
        s[u] = axpby4(alpha, s[u], d, k4);
        acc[u] = dot4(s[u], q4);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = group_sum<LPR>(acc[u]);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int rl = warp * RPW + (ps * U + u) * RPP + grp;
        if (rl < nrows) {
          state_st4<true>(S, (int64_t)rl * DK + 4 * sub, s[u], sd);
          if (sub == 0) Elem<TO>::store1(op + rl, scale * acc[u]);
        }
      }
    }
  } else {
    if (tid == 0) raise_error(p.err, GDN_DEVERR_TIMEOUT);
    mbar_wait_bounded(&bar, 0);  // give the copy a second bounded chance before going on
  }

  // the last of the key head's readers writes the shifted q/k cache
  if (tid == kTicketThread) {
    const int readers = group * (int)gridDim.x;
    const int last = prev == (unsigned int)(readers - 1);
    if (last) {
      atomicExch(ticket, 0u);
      __threadfence();
    }
    s_last = last;
  }
  __syncthreads();
  if (s_last) {
    for (int e = tid; e < 2 * DK * (W - 1); e += kThreads) {
      const int j = e / (W - 1), m = e % (W - 1);
      cache[(int64_t)qk_channel(j) * (W - 1) + m] = snew[j][m];
    }
  }
}

// ---- one-call decode step, larger grids: one CTA per (slot, key head) ----
//
// The CTA convolves every channel its key head's decode reads exactly once:
// the 2 * 128 q/k channels and the G * dv v channels of the G value heads
// that share the key head (G = h_v / h_k <= 2), one thread per channel, which
// also shifts that channel's cache in place (no other CTA reads it, so no
// ticket is needed).  Meanwhile the G heads' float32 states stream through a
// ring of kRing 16 KiB tiles (32 rows each; bulk copies issued ahead, one
// mbarrier per buffer), and each tile is updated row by row in the decode
// kernel's arithmetic: outputs, y, cache and state are bit-identical to the
// conv kernel followed by the decode kernel.  dk = 128 (a row is one warp,
// four columns per lane), dv a multiple of 32, float32 state.
constexpr int kGroupThreads = 256;
constexpr int kGroupTile = 16384;                 // bytes of one ring tile
constexpr int kGroupRows = kGroupTile / (128 * 4);  // 32 rows per tile
constexpr int kGroupMaxG = 2;
constexpr int kRing = 3;
constexpr int kGroupNch = (2 * 128 + kGroupMaxG * 128 + kGroupThreads - 1) / kGroupThreads;
constexpr int group_smem_bytes(int dv) {
  return kRing * kGroupTile + (2 * 128 + kGroupMaxG * dv) * 4 + 128;
}

template <typename TI, typename TO, int WM>
__global__ void __launch_bounds__(kGroupThreads, 4)
    decode_conv_group_kernel(PoolView p, int layer, const int32_t *__restrict__ slot_ids,
                             ConvStep cs, TO *__restrict__ o, float scale) {
  constexpr int DK = 128, R = kGroupRows, RPW = R / (kGroupThreads / 32);  // 4 rows per warp
  extern __shared__ __align__(128) unsigned char gsm[];
  float4 *ring = reinterpret_cast<float4 *>(gsm);                  // kRing tiles
  float *sqk = reinterpret_cast<float *>(gsm + kRing * kGroupTile);  // q | k conv outputs
  float *sv = sqk + 2 * DK;                                         // v conv outputs, G heads
  __shared__ __align__(8) uint64_t full[kRing];
  __shared__ float s_alpha[kGroupMaxG], s_beta[kGroupMaxG];

  const int hk = blockIdx.x, i = blockIdx.y, tid = threadIdx.x;
  const int G = p.h_v / p.h_k, dv = p.dv;
  const int W = WM == 4 ? 4 : p.conv_k;
  const int nq = p.h_k * DK;
  const int nch = 2 * DK + G * dv;          // channels this CTA convolves
  const int tph = dv / R, ntiles = G * tph;  // tiles per head, per CTA
  const int slot = slot_ids[i];
  auto channel = [&](int j) {  // the CTA's j-th channel: q, k, then the G heads' v
    return j < 2 * DK ? (j < DK ? 0 : nq) + hk * DK + j % DK
                      : 2 * nq + hk * G * dv + (j - 2 * DK);
  };
  // slot-independent inputs first
  const TI *xrow = static_cast<const TI *>(cs.x) + (int64_t)i * cs.ld_x;
  ConvTap<WM> tap[kGroupNch];
#pragma unroll
  for (int e = 0; e < kGroupNch; ++e) {
    const int j = tid + e * kGroupThreads;
    if (j < nch) tap_load<WM, TI>(tap[e], xrow, cs.w, cs.bias, channel(j), W);
  }
  float graw = 0.f, braw = 0.f;
  if (tid < G) {
    const int64_t gb = (int64_t)i * p.h_v + hk * G + tid;
    graw = Elem<TI>::load1(static_cast<const TI *>(cs.g) + gb);
    braw = Elem<TI>::load1(static_cast<const TI *>(cs.beta) + gb);
  }
  if (slot < 0 || slot >= p.n_slots) {
    if (hk == 0 && tid == 0) raise_error(p.err, GDN_DEVERR_SLOT);
    return;
  }
  auto tile_src = [&](int t) {  // tile t: rows (t % tph) * R .. of head hk * G + t / tph
    return p.state_at(p.state_head_elem(layer, slot, hk * G + t / tph) +
                      (int64_t)(t % tph) * R * DK);
  };
  auto issue = [&](int t) {  // one thread
    uint64_t *b = &full[t % kRing];
    // test hook: expect 16 bytes the copy never delivers, so the bounded wait
    // runs out after the copy itself has landed
    const uint32_t extra =
        (t == 0 && (p.test_flags & GDN_TEST_DECODE_WAIT_TIMEOUT)) ? 16u : 0u;
    mbar_arrive_expect_tx(b, kGroupTile + extra);
    bulk_g2s(ring + (t % kRing) * (kGroupTile / 16), tile_src(t), kGroupTile, b);
  };
  if (tid == 0) {
    for (int b = 0; b < kRing; ++b) mbar_init(&full[b], 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int t = 0; t < kRing && t < ntiles; ++t) issue(t);

  TI *cache = static_cast<TI *>(p.conv) +
              ((int64_t)layer * p.n_slots + slot) * p.conv_ch * (W - 1);
  TI *yrow = static_cast<TI *>(cs.y) + (int64_t)i * cs.ld_y;
#pragma unroll
  for (int e = 0; e < kGroupNch; ++e) {
    const int j = tid + e * kGroupThreads;
    if (j < nch) tap_load_cache<WM, TI>(tap[e], cache, channel(j), W);
  }
#pragma unroll
  for (int e = 0; e < kGroupNch; ++e) {
    const int j = tid + e * kGroupThreads;
    if (j < nch) {
      const int c = channel(j);
      const float yv = tap_conv<WM, TI>(tap[e], W);
      if (j < 2 * DK) sqk[j] = yv; else sv[j - 2 * DK] = yv;
      Elem<TI>::store1(yrow + c, yv);
      // this CTA is the only reader of the channel: shift its cache in place
      TI *cc = cache + (int64_t)c * (W - 1);
#pragma unroll
      for (int m = 0; m < WM - 2; ++m)
        if (m < W - 2) Elem<TI>::store1(cc + m, tap[e].hist[m + 1]);
      Elem<TI>::store1(cc + (W - 2), tap[e].x);
    }
  }
  if (tid < G) {
    s_alpha[tid] = expf(graw);
    s_beta[tid] = braw;
  }
  __syncthreads();  // sqk, sv, s_alpha, s_beta complete

  const int lane = tid & 31, warp = tid >> 5;
  float4 q4 = reinterpret_cast<const float4 *>(sqk)[lane];
  float4 k4 = reinterpret_cast<const float4 *>(sqk + DK)[lane];
  const float kk = group_sum<32>(dot4(k4, k4));
  const float qq = group_sum<32>(dot4(q4, q4));
  k4 = scale4(rsqrtf(kk + kL2Eps), k4);
  q4 = scale4(rsqrtf(qq + kL2Eps), q4);

  for (int t = 0; t < ntiles; ++t) {
    const int b = t % kRing;
    if (!__syncthreads_and(mbar_wait_bounded(&full[b], (uint32_t)(t / kRing) & 1u))) {
      if (tid == 0) {
        raise_error(p.err, GDN_DEVERR_TIMEOUT);
        // a second bounded chance for every copy still in flight
        const int issued = min(t + kRing, ntiles);
        for (int u = t; u < issued; ++u)
          mbar_wait_bounded(&full[u % kRing], (uint32_t)(u / kRing) & 1u);
      }
      __syncthreads();
      return;
    }
    const int vh = t / tph, r0 = (t % tph) * R;
    const int h = hk * G + vh;
    const float alpha = s_alpha[vh], beta = s_beta[vh];
    const float4 *tile = ring + b * (kGroupTile / 16);
    char *S = tile_src(t);
    TO *op = o + ((int64_t)i * p.h_v + h) * dv + r0;
    float4 sr[RPW];
    float acc[RPW];
#pragma unroll
    for (int u = 0; u < RPW; ++u) {
      const int rl = warp * RPW + u;
      sr[u] = tile[rl * (DK / 4) + lane];
      acc[u] = dot4(sr[u], k4);
    }
#pragma unroll
    for (int u = 0; u < RPW; ++u) acc[u] = group_sum<32>(acc[u]);
#pragma unroll
    for (int u = 0; u < RPW; ++u) {
      const int rl = warp * RPW + u;
      const float d = beta * (sv[vh * dv + r0 + rl] - alpha * acc[u]);
      sr[u] = axpby4(alpha, sr[u], d, k4);
      acc[u] = dot4(sr[u], q4);
    }
#pragma unroll
    for (int u = 0; u < RPW; ++u) acc[u] = group_sum<32>(acc[u]);
#pragma unroll
    for (int u = 0; u < RPW; ++u) {
      const int rl = warp * RPW + u;
      state_st4<true>(S, (int64_t)rl * DK + 4 * lane, sr[u], GDN_F32);
      if (lane == 0) Elem<TO>::store1(op + rl, scale * acc[u]);
    }
    __syncthreads();  // every thread is done with buffer b
    if (tid == 0 && t + kRing < ntiles) issue(t + kRing);
  }
}

template <typename TI, typename TO>
cudaError_t launch_group_t(const PoolView &p, int layer, const int32_t *slot_ids, int n,
                           const ConvStep &cs, void *o, float scale, cudaStream_t s) {
  const int bytes = group_smem_bytes(p.dv);
  const dim3 grid(p.h_k, n);
  auto kern = p.conv_k == 4 ? decode_conv_group_kernel<TI, TO, 4>
                            : decode_conv_group_kernel<TI, TO, kMaxConvK>;
  const cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kGroupThreads, bytes, s>>>(p, layer, slot_ids, cs, static_cast<TO *>(o), scale);
  return cudaGetLastError();
}

template <int DK, typename TI, typename TO>
struct DecodeConvF {
  static cudaError_t run(const PoolView &p, int layer, const int32_t *slot_ids, int n,
                         const ConvStep &cs, void *o, float scale, cudaStream_t s) {
    constexpr int R = kBulkBytes / (DK * 4);
    dim3 grid((p.dv + R - 1) / R, p.h_v, n);
    if (p.conv_k == 4)
      decode_conv_kernel<DK, TI, TO, 4><<<grid, kThreads, 0, s>>>(p, layer, slot_ids, cs,
                                                                   static_cast<TO *>(o), scale);
    else
      decode_conv_kernel<DK, TI, TO, kMaxConvK><<<grid, kThreads, 0, s>>>(
          p, layer, slot_ids, cs, static_cast<TO *>(o), scale);
    return cudaGetLastError();
  }
};

// CTAs of the fused kernel one SM holds at once (looked up once per
// instantiation; every device this library runs on is the same part).
template <int DK, typename TI, typename TO>
struct DecodeConvOcc {
  static cudaError_t run(const PoolView &p, int *per_sm) {
    static int occ4 = -1, occ8 = -1;
    int &occ = p.conv_k == 4 ? occ4 : occ8;
    if (occ < 0) {
      int v = 0;
      const cudaError_t e =
          p.conv_k == 4
              ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    &v, decode_conv_kernel<DK, TI, TO, 4>, kThreads, 0)
              : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    &v, decode_conv_kernel<DK, TI, TO, kMaxConvK>, kThreads, 0);
      if (e != cudaSuccess) return e;
      occ = v;
    }
    *per_sm = occ;
    return cudaSuccess;
  }
};

template <int DK, typename TI, typename TO>
cudaError_t launch_decode_t(const PoolView &p, int layer, const int32_t *slot_ids, int n,
                            const QKV &in, void *o, float scale, cudaStream_t s,
                            bool after_conv) {
  const bool half = p.state_dtype != GDN_F32;
  const int R = kBulkBytes / (DK * (half ? 2 : 4));
  dim3 grid((p.dv + R - 1) / R, p.h_v, n);
  if (!after_conv) {
    if (half)
      decode_bulk_kernel<DK, TI, TO, false, true><<<grid, kThreads, 0, s>>>(
          p, layer, slot_ids, in, static_cast<TO *>(o), scale);
    else
      decode_bulk_kernel<DK, TI, TO, false, false><<<grid, kThreads, 0, s>>>(
          p, layer, slot_ids, in, static_cast<TO *>(o), scale);
    return cudaGetLastError();
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (half)
    return cudaLaunchKernelEx(&cfg, decode_bulk_kernel<DK, TI, TO, true, true>, p, layer,
                              slot_ids, in, static_cast<TO *>(o), scale);
  return cudaLaunchKernelEx(&cfg, decode_bulk_kernel<DK, TI, TO, true, false>, p, layer,
                            slot_ids, in, static_cast<TO *>(o), scale);
}

template <int DK, typename TI, typename TO>
struct DecodeF {
  static cudaError_t run(const PoolView &p, int layer, const int32_t *slot_ids, int n,
                         const QKV &in, void *o, float scale, cudaStream_t s, bool after_conv) {
    return launch_decode_t<DK, TI, TO>(p, layer, slot_ids, n, in, o, scale, s, after_conv);
  }
};

}  // namespace

cudaError_t launch_decode(const PoolView &p, const void *tmap, int layer,
                          const int32_t *slot_ids, int n, const QKV &in, void *o,
                          gdn_dtype o_dtype, float scale, cudaStream_t s, bool after_conv) {
  // The tensor-map path of the verify kernel (T = 1, always committing) computes
  // the same step but keeps 64 KiB per CTA in flight, three CTAs per SM; the
  // 16 KiB bulk tiles above sustain more bytes in flight per SM, so decode
  // does not use the map.
  (void)tmap;
  return dispatch<DecodeF>(p.dk, in.dtype, o_dtype, p, layer, slot_ids, n, in, o, scale, s,
                           after_conv);
}

cudaError_t decode_conv_resident_ctas(const PoolView &p, gdn_dtype dtype, gdn_dtype o_dtype,
                                      int sm_count, int64_t *ctas) {
  int per_sm = 0;
  const cudaError_t e = dispatch<DecodeConvOcc>(p.dk, dtype, o_dtype, p, &per_sm);
  *ctas = (int64_t)per_sm * sm_count;
  return e;
}

int64_t decode_grid_ctas(const PoolView &p, int n) {
  const int R = kBulkBytes / (p.dk * 4);
  return (int64_t)((p.dv + R - 1) / R) * p.h_v * n;
}

bool decode_conv_group_ok(const PoolView &p) {
  return p.dk == 128 && p.state_dtype == GDN_F32 && p.h_k > 0 && p.h_v % p.h_k == 0 &&
         p.h_v / p.h_k <= kGroupMaxG && p.dv % kGroupRows == 0 && p.dv > 0 &&
         group_smem_bytes(p.dv) <= 227 * 1024 && p.conv_k >= 2 && p.conv_k <= kMaxConvK;
}

cudaError_t launch_decode_conv_group(const PoolView &p, int layer, const int32_t *slot_ids,
                                     int n, const void *x, int64_t ld_x, const float *w,
                                     const float *bias, void *y, int64_t ld_y, const void *g,
                                     const void *beta, gdn_dtype dtype, void *o,
                                     gdn_dtype o_dtype, float scale, cudaStream_t s) {
  if (!decode_conv_group_ok(p)) return cudaErrorInvalidValue;
  const ConvStep cs{x, ld_x, w, bias, y, ld_y, g, beta};
  if (dtype == GDN_BF16)
    return o_dtype == GDN_BF16 ? launch_group_t<bf16, bf16>(p, layer, slot_ids, n, cs, o, scale, s)
                               : launch_group_t<bf16, float>(p, layer, slot_ids, n, cs, o, scale, s);
  return o_dtype == GDN_BF16 ? launch_group_t<float, bf16>(p, layer, slot_ids, n, cs, o, scale, s)
                             : launch_group_t<float, float>(p, layer, slot_ids, n, cs, o, scale, s);
}

cudaError_t launch_decode_conv(const PoolView &p, int layer, const int32_t *slot_ids, int n,
                              const void *x, int64_t ld_x, const float *w, const float *bias,
                              void *y, int64_t ld_y, const void *g, const void *beta,
                              gdn_dtype dtype, void *o, gdn_dtype o_dtype, float scale,
                              cudaStream_t s) {
  if (p.ticks == nullptr || p.conv_k > kMaxConvK) return cudaErrorInvalidValue;
  const ConvStep cs{x, ld_x, w, bias, y, ld_y, g, beta};
  return dispatch<DecodeConvF>(p.dk, dtype, o_dtype, p, layer, slot_ids, n, cs, o, scale, s);
}

}  // namespace gdn
