// Chunked prefill in two launches, for dk = dv = 128 (tcgen05).
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
// tiles to a workspace; a state kernel then walks each (sequence, value head)
// chunk by chunk with the state resident in TMEM, fetching each chunk's P and
// T tiles with bulk copies issued ahead: `seq_bf16_kernel` when the bf16 rows
// can come by tensor map (S [Q;K]^T on kind::f16 over the raw tiles),
// `seq_kernel` otherwise (rows staged from global memory as float32 operand
// tiles, kind::tf32).
//
// Workspace: (n_seqs + 1) int32 chunk offsets and the sequence order (256-byte
// aligned), then per (chunk, value head) 32 KiB: the P tile, then the T tile,
// each 64 x 64 float32 in the K-major core-matrix layout of gdn_tc.cuh; then,
// when q and k came by tensor map, per (chunk, value head) the state walk's
// per-token scalars (5 x 64 float32, below).  Chunks are numbered sequence by
// sequence; offsets[i] is the first chunk of sequence i.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <type_traits>

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
// The state walk's per-token scalars of one (chunk, value head), written by the
// key-side kernel when q and k come by tensor map: gamma_t = e^{G_t}, beta_t,
// gamma_t / |q_t| (scales column t of S Q^T), beta_t gamma_t / |k_t| (column t
// of S K^T), e^{G_n - G_t} / |k_t| (token t of Ktil); 64 floats each.
constexpr int kSGam = 0, kSBeta = C, kSQ = 2 * C, kSK = 3 * C, kSKt = 4 * C, kScal = 5 * C;

// Calls of up to this many sequences walk them longest first.
constexpr int kOrderMax = 256;
__host__ __device__ inline int64_t max_chunks(int n_seqs, int total_tokens) {
  return (int64_t)total_tokens / C + n_seqs;  // >= sum over sequences of ceil(len / 64)
}
// offsets and the state kernels' sequence order (both int32), then per chunk
// (up to cap chunks) its first token and token count (int2)
__host__ __device__ inline size_t chunk_table_offset(int n_seqs) {
  return ((2 * (size_t)n_seqs + 1) * 4 + 7) & ~(size_t)7;
}
__host__ __device__ inline size_t offsets_bytes(int n_seqs, int64_t cap) {
  return (chunk_table_offset(n_seqs) + (size_t)cap * 8 + 255) & ~(size_t)255;
}

__device__ __forceinline__ int seq_chunks(const SeqIndex &seq, int i) {
  const int64_t lo = seq.cu_seqlens[i], hi = seq.cu_seqlens[i + 1];
  if (hi < lo || lo < 0 || hi > seq.total_tokens) return 0;  // the state kernel reports it
  return (int)((hi - lo + C - 1) / C);
}

// offsets[i] = number of chunks before sequence i; offsets[n_seqs] = total.
// Offsets saturate at cap + 1 (only overlapping sequences can exceed the
// workspace's cap chunks; the state kernel rejects them).  Then order[r]
// (after offsets[n_seqs]) = the sequence with the r-th most chunks, ties by
// index, so that the state kernels start the longest sequences first
// (identity order past kOrderMax sequences).  Then table[c] = (first token,
// tokens) of chunk c < cap, for the key-side kernel.
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
  int2 *table = reinterpret_cast<int2 *>(reinterpret_cast<char *>(off) + chunk_table_offset(n));
  for (int i = b; i < e; ++i) {
    off[i] = (int32_t)min(run, cap + 1);
    const int nc = seq_chunks(seq, i);
    const int lo = nc > 0 ? (int)seq.cu_seqlens[i] : 0;
    const int len = nc > 0 ? (int)seq.cu_seqlens[i + 1] - lo : 0;
    for (int j = 0; j < nc && run + j < cap; ++j)
      table[run + j] = make_int2(lo + j * C, min(C, len - j * C));
    run += nc;
  }
  if (tid == 1023) off[n] = (int32_t)min(part[1023], cap + 1);
  int32_t *order = off + n + 1;
  __shared__ int cnt[kOrderMax];
  if (n <= kOrderMax) {
    if (tid < n) cnt[tid] = seq_chunks(seq, tid);
    __syncthreads();
    if (tid < n) {
      const int ci = cnt[tid];
      int rank = 0;
      for (int j = 0; j < n; ++j) rank += (cnt[j] > ci || (cnt[j] == ci && j < tid)) ? 1 : 0;
      order[rank] = tid;
    }
  } else {
    for (int i = tid; i < n; i += 1024) order[i] = i;
  }
}

// This thread's token in the staging map below (warp w: tokens 8w .. 8w+7).
__device__ __forceinline__ int stage_token() { return 8 * (threadIdx.x >> 5) + (threadIdx.x & 7); }

// g and beta of this thread's token of the chunk starting at tok0 (0 if padded).
template <typename TI>
__device__ __forceinline__ void load_gb(const QKV &in, const PoolView &p, int h, int64_t tok0,
                                        int n, float &gt, float &bt) {
  const int t = stage_token();
  gt = bt = 0.f;
  if (t < n) {
    gt = Elem<TI>::load1(static_cast<const TI *>(in.g) + (tok0 + t) * p.h_v + h);
    bt = Elem<TI>::load1(static_cast<const TI *>(in.beta) + (tok0 + t) * p.h_v + h);
  }
}

// Stage normalised q and k of one chunk as the [Q;K] core tile (rows 0..63 Q,
// 64..127 K; padded tokens zero), beta v (plain rows) and g, beta.  Row t of
// q, k, v starts at q0 + t ldq (k0 + t ldq, v0 + t ldv): global memory, or the
// raw copy of the chunk in shared memory.  Warp w takes tokens 8w .. 8w+7;
// lane = token (3 bits) + 8 * chunk group, so a quarter-warp writes the 8 rows
// of one core matrix (contiguous 128 bytes).
template <typename TI, bool WITH_V>
__device__ __forceinline__ void stage_rows(const TI *q0, const TI *k0, const TI *v0, int64_t ldq,
                                           int64_t ldv, int n, float gt, float bt, float *QK,
                                           float *XU, float *sG, float *sBeta) {
  const int lane = threadIdx.x & 31;
  const int cg = lane >> 3;
  const int t = stage_token();
  const bool real = t < n;
  // q, then k (normalised rows of the core tile), then beta v: one row in registers at a time
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const TI *src = (which == 0 ? q0 : k0) + t * ldq;
    float4 x4[D / 16];
    float xx = 0.f;
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      x4[j] = real ? Elem<TI>::load4(src + 4 * (cg + 4 * j)) : make_float4(0.f, 0.f, 0.f, 0.f);
      xx += dot4(x4[j], x4[j]);
    }
    xx += __shfl_xor_sync(0xffffffffu, xx, 8);
    xx += __shfl_xor_sync(0xffffffffu, xx, 16);
    const float xs = rsqrtf(xx + kL2Eps);
#pragma unroll
    for (int j = 0; j < D / 16; ++j)
      *reinterpret_cast<float4 *>(QK + tc::core_off(64 * which + t, 4 * (cg + 4 * j), D)) =
          scale4(xs, x4[j]);
  }
  if (WITH_V) {
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      const int c = cg + 4 * j;
      const float4 v4 = real ? Elem<TI>::load4(v0 + t * ldv + 4 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4 *>(XU + t * XS + 4 * c) = scale4(bt, v4);
    }
  }
  if (cg == 0) {
    sG[t] = gt;
    sBeta[t] = bt;
  }
}

// The same from global memory, for the chunk starting at token tok0.
template <typename TI, bool WITH_V>
__device__ __forceinline__ void stage_chunk(const QKV &in, const PoolView &p, int h, int hk,
                                            int64_t tok0, int n, float *QK, float *XU,
                                            float *sG, float *sBeta) {
  float gt, bt;
  load_gb<TI>(in, p, h, tok0, n, gt, bt);
  stage_rows<TI, WITH_V>(static_cast<const TI *>(in.q) + tok0 * in.ld_qk + (int64_t)hk * D,
                         static_cast<const TI *>(in.k) + tok0 * in.ld_qk + (int64_t)hk * D,
                         static_cast<const TI *>(in.v) + tok0 * in.ld_v + (int64_t)h * D,
                         in.ld_qk, in.ld_v, n, gt, bt, QK, XU, sG, sBeta);
}

// Tensor maps of a call's bf16 rows (16-byte aligned): q, k and v are fetched
// as 64-column halves of [64 tokens][64] bf16 in the 128-byte swizzled layout
// (8 KiB each, 1024-byte aligned).
struct InMaps {
  CUtensorMap q, k, v;  // {128, heads, tokens}
  CUtensorMap o;        // bf16 outputs {128, h_v, tokens}, stores of whole chunks
};
constexpr int kRawHalf = C * 64 * 2;  // 8 KiB

__device__ __forceinline__ void tma3(void *dst, const CUtensorMap *m, int x, int y, int z,
                                     uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// Tensor-map store of a shared-memory box (one thread), and the bulk-group
// commit / waits that order it: .read once the source may be overwritten, the
// full wait before the block exits.
__device__ __forceinline__ void tma3_store(const CUtensorMap *m, int x, int y, int z,
                                           const void *src) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(x), "r"(y), "r"(z), "r"(smem_addr(src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// One thread: the chunk's v halves to vdst, vdst + kRawHalf onto vbar.
__device__ __forceinline__ void prefetch_v(const InMaps &m, int h, int64_t tok0,
                                           unsigned char *vdst, uint64_t *vbar) {
  mbar_arrive_expect_tx(vbar, 2 * kRawHalf);
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) tma3(vdst + hf * kRawHalf, &m.v, 64 * hf, h, (int)tok0, vbar);
}
// One thread: the chunk's q and k halves into a [q h0 | k h0 | q h1 | k h1]
// buffer (each half-pair a 128-row [Q;K] operand block) onto bar, which also
// expects extra_tx bytes of copies the caller issues next.
__device__ __forceinline__ void prefetch_qk_pairs(const InMaps &m, int hk, int64_t tok0,
                                                  unsigned char *qk, uint64_t *bar,
                                                  uint32_t extra_tx) {
  mbar_arrive_expect_tx(bar, 4 * kRawHalf + extra_tx);
  const int z = (int)tok0;
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    tma3(qk + (2 * hf) * kRawHalf, &m.q, 64 * hf, hk, z, bar);
    tma3(qk + (2 * hf + 1) * kRawHalf, &m.k, 64 * hf, hk, z, bar);
  }
}

// ----------------------------------------------------------------- key side
// Raw bf16 q and k rows of one chunk as the [Q;K] 16-bit core tile (rows 0..63
// Q, 64..127 K; padded tokens zero), with rq[t], rk[t] = 1 / |q_t|, 1 / |k_t|
// (epsilon as everywhere).  The tile feeds a kind::f16 MMA on the exact input
// values; the norms are applied to its products.  Warp w takes tokens
// 8w .. 8w+7; lane = token (3 bits) + 8 * part, part p holding the 4-element
// pieces p, p+4, ..., so one store instruction fills two whole core matrices.
__device__ __forceinline__ void stage_qk_bf16(const bf16 *q0, const bf16 *k0, int64_t ld, int n,
                                              unsigned char *tile, float *rq, float *rk) {
  const int lane = threadIdx.x & 31;
  const int part = lane >> 3;
  const int t = stage_token();
  const bool real = t < n;
  uint2 qv[8], kv[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int c = part + 4 * m;
    qv[m] = kv[m] = make_uint2(0u, 0u);
    if (real) {
      qv[m] = *reinterpret_cast<const uint2 *>(q0 + t * ld + 4 * c);
      kv[m] = *reinterpret_cast<const uint2 *>(k0 + t * ld + 4 * c);
    }
  }
  float qq = 0.f, kk = 0.f;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float a0 = __uint_as_float(qv[m].x << 16), a1 = __uint_as_float(qv[m].x & 0xffff0000u);
    const float a2 = __uint_as_float(qv[m].y << 16), a3 = __uint_as_float(qv[m].y & 0xffff0000u);
    const float b0 = __uint_as_float(kv[m].x << 16), b1 = __uint_as_float(kv[m].x & 0xffff0000u);
    const float b2 = __uint_as_float(kv[m].y << 16), b3 = __uint_as_float(kv[m].y & 0xffff0000u);
    qq += a0 * a0 + a1 * a1 + a2 * a2 + a3 * a3;
    kk += b0 * b0 + b1 * b1 + b2 * b2 + b3 * b3;
  }
  qq += __shfl_xor_sync(0xffffffffu, qq, 8);
  qq += __shfl_xor_sync(0xffffffffu, qq, 16);
  kk += __shfl_xor_sync(0xffffffffu, kk, 8);
  kk += __shfl_xor_sync(0xffffffffu, kk, 16);
  constexpr uint32_t SBO = tc::sbo_bytes16(D);
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int c = part + 4 * m;  // elements 4c .. 4c+3
    const uint32_t off = (uint32_t)(c >> 1) * tc::kLBO + (uint32_t)(t & 7) * 16 + (c & 1) * 8;
    *reinterpret_cast<uint2 *>(tile + (t >> 3) * SBO + off) = qv[m];
    *reinterpret_cast<uint2 *>(tile + (8 + (t >> 3)) * SBO + off) = kv[m];
  }
  if (part == 0) {
    rq[t] = rsqrtf(qq + kL2Eps);
    rk[t] = rsqrtf(kk + kL2Eps);
  }
}

__device__ __forceinline__ void group_sync(int id) {  // one 128-thread warpgroup
  asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}

// T = (I + A)^{-1} for a strictly lower 64 x 64 A (plain rows, stride AS), by
// one warpgroup (thread tt of 128, named barrier `bar`).  T's strictly-upper
// 16 x 16 blocks must be zero on entry; X is 1024 floats of scratch.  With
// T_b the inverse of diagonal block b and lower-triangular blocks throughout,
//   T_{b+1,b} = -T_{b+1,b+1} A_{b+1,b} T_{b,b}            (16 x 16, b = 0, 2)
//   T_L       = -T_hi A_L T_lo                             (32 x 32 lower left)
// where T_lo, T_hi are the finished upper-left and lower-right 32 x 32 halves.
__device__ __forceinline__ void invert_unit_lower(const float *A, float *T, float *X, int tt,
                                                  int bar) {
  if (tt < C) {  // diagonal blocks: column j of (I + A_bb)^{-1} by forward substitution
    const int bb = tt >> 4, j = tt & 15;
    const float *Ab = A + (16 * bb) * AS + 16 * bb;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = r == j ? 1.f : 0.f;
#pragma unroll
      for (int c = 0; c < r; ++c) acc -= Ab[r * AS + c] * x[c];
      x[r] = acc;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) T[(16 * bb + r) * AS + 16 * bb + j] = x[r];
  }
  group_sync(bar);
  // The products below run over the whole K range, fully unrolled, with two
  // partial sums each: the triangular factors' zero upper parts add exact
  // zeros, and every thread gets the same work.
  const int which = tt >> 6, r = (tt >> 2) & 15, q0 = 4 * (tt & 3);
  const int b = 2 * which;
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  {  // X_b = A_{b+1,b} T_{b,b}
    const float *ar = A + (16 * (b + 1) + r) * AS + 16 * b;
    const float *tb = T + (16 * b) * AS + 16 * b + q0;
    float4 x0 = z4, x1 = z4;
#pragma unroll
    for (int k = 0; k < 16; k += 4) {
      const float4 a4 = *reinterpret_cast<const float4 *>(ar + k);
      x0 = axpby4(1.f, x0, a4.x, *reinterpret_cast<const float4 *>(tb + (k + 0) * AS));
      x1 = axpby4(1.f, x1, a4.y, *reinterpret_cast<const float4 *>(tb + (k + 1) * AS));
      x0 = axpby4(1.f, x0, a4.z, *reinterpret_cast<const float4 *>(tb + (k + 2) * AS));
      x1 = axpby4(1.f, x1, a4.w, *reinterpret_cast<const float4 *>(tb + (k + 3) * AS));
    }
    *reinterpret_cast<float4 *>(X + which * 256 + r * 16 + q0) = axpby4(1.f, x0, 1.f, x1);
  }
  group_sync(bar);
  {  // T_{b+1,b} = -T_{b+1,b+1} X_b
    const float *tr = T + (16 * (b + 1) + r) * AS + 16 * (b + 1);
    const float *xb = X + which * 256 + q0;
    float4 y0 = z4, y1 = z4;
#pragma unroll
    for (int k = 0; k < 16; k += 4) {
      const float4 t4 = *reinterpret_cast<const float4 *>(tr + k);
      y0 = axpby4(1.f, y0, t4.x, *reinterpret_cast<const float4 *>(xb + (k + 0) * 16));
      y1 = axpby4(1.f, y1, t4.y, *reinterpret_cast<const float4 *>(xb + (k + 1) * 16));
      y0 = axpby4(1.f, y0, t4.z, *reinterpret_cast<const float4 *>(xb + (k + 2) * 16));
      y1 = axpby4(1.f, y1, t4.w, *reinterpret_cast<const float4 *>(xb + (k + 3) * 16));
    }
    *reinterpret_cast<float4 *>(T + (16 * (b + 1) + r) * AS + 16 * b + q0) =
        axpby4(-1.f, y0, -1.f, y1);
  }
  group_sync(bar);
  const int r0 = 2 * (tt >> 3), c0 = 4 * (tt & 7);
  {  // Y = A_L T_lo  (rows 32 + r0, 33 + r0)
    const float *a0 = A + (32 + r0) * AS, *a1 = a0 + AS;
    float4 y00 = z4, y01 = z4, y10 = z4, y11 = z4;
#pragma unroll
    for (int k = 0; k < 32; k += 4) {
      const float4 u = *reinterpret_cast<const float4 *>(a0 + k);
      const float4 w = *reinterpret_cast<const float4 *>(a1 + k);
      const float4 t0 = *reinterpret_cast<const float4 *>(T + (k + 0) * AS + c0);
      const float4 t1 = *reinterpret_cast<const float4 *>(T + (k + 1) * AS + c0);
      const float4 t2 = *reinterpret_cast<const float4 *>(T + (k + 2) * AS + c0);
      const float4 t3 = *reinterpret_cast<const float4 *>(T + (k + 3) * AS + c0);
      y00 = axpby4(1.f, y00, u.x, t0);
      y01 = axpby4(1.f, y01, u.y, t1);
      y10 = axpby4(1.f, y10, w.x, t0);
      y11 = axpby4(1.f, y11, w.y, t1);
      y00 = axpby4(1.f, y00, u.z, t2);
      y01 = axpby4(1.f, y01, u.w, t3);
      y10 = axpby4(1.f, y10, w.z, t2);
      y11 = axpby4(1.f, y11, w.w, t3);
    }
    *reinterpret_cast<float4 *>(X + r0 * 32 + c0) = axpby4(1.f, y00, 1.f, y01);
    *reinterpret_cast<float4 *>(X + (r0 + 1) * 32 + c0) = axpby4(1.f, y10, 1.f, y11);
  }
  group_sync(bar);
  {  // T_L = -T_hi Y  (rows 32 + r0, 33 + r0)
    const float *t0 = T + (32 + r0) * AS + 32, *t1 = t0 + AS;
    float4 y00 = z4, y01 = z4, y10 = z4, y11 = z4;
#pragma unroll
    for (int k = 0; k < 32; k += 4) {
      const float4 u = *reinterpret_cast<const float4 *>(t0 + k);
      const float4 w = *reinterpret_cast<const float4 *>(t1 + k);
      const float4 x0 = *reinterpret_cast<const float4 *>(X + (k + 0) * 32 + c0);
      const float4 x1 = *reinterpret_cast<const float4 *>(X + (k + 1) * 32 + c0);
      const float4 x2 = *reinterpret_cast<const float4 *>(X + (k + 2) * 32 + c0);
      const float4 x3 = *reinterpret_cast<const float4 *>(X + (k + 3) * 32 + c0);
      y00 = axpby4(1.f, y00, u.x, x0);
      y01 = axpby4(1.f, y01, u.y, x1);
      y10 = axpby4(1.f, y10, w.x, x0);
      y11 = axpby4(1.f, y11, w.y, x1);
      y00 = axpby4(1.f, y00, u.z, x2);
      y01 = axpby4(1.f, y01, u.w, x3);
      y10 = axpby4(1.f, y10, w.z, x2);
      y11 = axpby4(1.f, y11, w.w, x3);
    }
    *reinterpret_cast<float4 *>(T + (32 + r0) * AS + c0) = axpby4(-1.f, y00, -1.f, y01);
    *reinterpret_cast<float4 *>(T + (33 + r0) * AS + c0) = axpby4(-1.f, y10, -1.f, y11);
  }
  group_sync(bar);
}

// shared-memory map of prep_kernel: the [Q;K] tile, then per value head of
// the CTA's pair: A and T (plain 64 x AS), 1024 floats of inverse scratch,
// G and beta; then rq, rk.
constexpr int kHeadFloats = 2 * C * AS + 1024 + 2 * C;
template <typename TI>
constexpr int prep_tile_bytes() { return std::is_same<TI, bf16>::value ? 128 * D * 2 : 128 * D * 4; }
template <typename TI>
constexpr int prep_smem() {  // + 1024: the tile is aligned to 1024 bytes inside the allocation
  return prep_tile_bytes<TI>() + (2 * kHeadFloats + 2 * C) * 4 + 1024;
}
static_assert(2 * (prep_smem<bf16>() + 1024 + 64) <= 228 * 1024, "two bf16 prep CTAs per SM");
static_assert(prep_smem<float>() <= 227 * 1024, "shared memory");

// Persistent: each CTA takes the work items blockIdx.x, blockIdx.x + gridDim.x,
// ... of the call, item = (chunk, key head, pair of the value heads that read
// that key head), chunk-major.  Both warpgroups share the staged [Q;K] tile
// and the Gram product D1 = [Q;K] K^T; warpgroup wg then forms P and A for
// value head 2 pair + wg of the group and inverts I + A.  Once the Gram MMA
// has read the tile, the next item's q/k copies (tensor-map rows) and its g,
// beta loads are issued, so they land while this item's P, A and T are formed.
// nc: the chunk capacity of the workspace; table: each chunk's first token
// and token count.
template <typename TI>
__global__ void __launch_bounds__(NT, 2)
    prep_kernel(PoolView p, SeqIndex seq, QKV in, const int32_t *__restrict__ off,
                const int2 *__restrict__ table, float *__restrict__ work, int64_t nc,
                const __grid_constant__ InMaps maps, int raw_rows) {
  constexpr bool B16 = std::is_same<TI, bf16>::value;  // raw bf16 tile, kind::f16
  // 16-byte aligned bf16 rows: the tile arrives by tensor-map copies in the 128-byte
  // swizzle, two K halves [Q;K] x 64 columns (16 KiB each), read by swizzled descriptors
  const bool TMAQK = B16 && raw_rows != 0;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *tile = smem + ((1024u - (smem_addr(smem) & 1023u)) & 1023u);
  float *heads = reinterpret_cast<float *>(tile + prep_tile_bytes<TI>());
  float *rq = heads + 2 * kHeadFloats;
  float *rk = rq + C;
  __shared__ __align__(8) uint64_t bar;
  __shared__ __align__(8) uint64_t lbar;   // tensor-map copies of q, k
  __shared__ uint32_t tmem_slot;

  // the state kernel may start its prologue now (it waits for this grid
  // before it reads the workspace)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int G = p.h_v / p.h_k, npair = (G + 1) / 2;
  const int ny = p.h_k * npair;
  // (offsets past the capacity come only from overlapping sequences, which the
  // state kernel rejects; no chunk beyond it is formed)
  const int64_t items = min((int64_t)off[seq.n_seqs], nc) * ny;
  if ((int64_t)blockIdx.x >= items) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wg = warp >> 2, quad = warp & 3, tt = tid & 127;
  float *AP = heads + wg * kHeadFloats;
  float *TP = AP + C * AS;
  float *XS_ = TP + C * AS;
  float *sG = XS_ + 1024;
  float *sBeta = sG + C;

  // work item -> chunk, its sequence's token range, key head, pair
  struct Item {
    int cidx, n, kh, pair;
    int64_t tok0;
  };
  auto locate = [&](int64_t it, int2 tc) {  // tc = table[it / ny]
    Item w;
    w.cidx = (int)(it / ny);
    const int y = (int)(it % ny);
    w.kh = y / npair;
    w.pair = y % npair;
    w.tok0 = tc.x;
    w.n = tc.y;
    return w;
  };
  auto head_of = [&](const Item &w) {
    const bool lv = 2 * w.pair + wg < G;  // this warpgroup has a value head
    return w.kh * G + (lv ? 2 * w.pair + wg : 0);
  };
  // thread tt < C of each warpgroup: its head's g and beta of token tt (padded 0)
  auto load_gb1 = [&](const Item &w, float &gt, float &bt) {
    gt = bt = 0.f;
    if (tt < w.n && 2 * w.pair + wg < G) {
      const int h = head_of(w);
      gt = Elem<TI>::load1(static_cast<const TI *>(in.g) + (w.tok0 + tt) * p.h_v + h);
      bt = Elem<TI>::load1(static_cast<const TI *>(in.beta) + (w.tok0 + tt) * p.h_v + h);
    }
  };
  auto issue_rows = [&](const Item &w) {  // one thread
    mbar_arrive_expect_tx(&lbar, 4 * kRawHalf);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      tma3(tile + hf * 2 * kRawHalf, &maps.q, 64 * hf, w.kh, (int)w.tok0, &lbar);
      tma3(tile + hf * 2 * kRawHalf + kRawHalf, &maps.k, 64 * hf, w.kh, (int)w.tok0, &lbar);
    }
  };

  if (warp == 0) tc::tmem_alloc(&tmem_slot, 64);
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&lbar, 1);
    mbar_fence_init();
  }
  for (int e = tt; e < C * C; e += 128) {  // T's strictly-upper 16 x 16 blocks stay zero
    const int r = e / C, c = e % C;
    if ((c >> 4) > (r >> 4)) TP[r * AS + c] = 0.f;
  }
  Item w = locate(blockIdx.x, table[blockIdx.x / ny]);
  float g_nx = 0.f, b_nx = 0.f;  // the next item's g, beta (threads tt < C)
  load_gb1(w, g_nx, b_nx);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = tmem_slot;
  const uint32_t lrow = tm + ((uint32_t)(32 * quad) << 16);
  if (TMAQK && tid == 0) issue_rows(w);

  bool ok = true;        // every wait so far completed
  bool pending = TMAQK;  // a row copy onto lbar is in flight
  bool mma_out = false;  // a Gram MMA onto bar is in flight
  uint32_t ph = 0;       // phase of bar and lbar for this item
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x, ph ^= 1u) {
    const int cidx = w.cidx, n = w.n;
    const int64_t nx = it + gridDim.x;
    const int2 tc_nx = nx < items ? table[nx / ny] : make_int2(0, 0);  // used at the prefetch
    const int64_t tok0 = w.tok0;
    const int kh = w.kh, pair = w.pair;
    const bool live = 2 * pair + wg < G;
    const int h = head_of(w);
    if (tt < C) {
      sG[tt] = g_nx;
      sBeta[tt] = b_nx;
    }
    const TI *q0 = static_cast<const TI *>(in.q) + tok0 * in.ld_qk + (int64_t)kh * D;
    const TI *k0 = static_cast<const TI *>(in.k) + tok0 * in.ld_qk + (int64_t)kh * D;
    bool loaded = true;
    if (TMAQK) {  // norms of the tensor-map rows, summed in stage_qk_bf16's order
      loaded = mbar_wait_bounded(&lbar, ph);
      const int t = stage_token(), part = lane >> 3;
      float qq = 0.f, kk = 0.f;
      if (loaded) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int c = part + 4 * m;                  // elements 4c .. 4c+3
          const int col = (4 * c) & 63, hf = (4 * c) >> 6;
          const int off8 = t * 128 + ((((col >> 3) ^ (t & 7))) << 4) + (col & 7) * 2;
          const uint2 qv = *reinterpret_cast<const uint2 *>(tile + hf * 2 * kRawHalf + off8);
          const uint2 kv =
              *reinterpret_cast<const uint2 *>(tile + hf * 2 * kRawHalf + kRawHalf + off8);
          const float a0 = __uint_as_float(qv.x << 16), a1 = __uint_as_float(qv.x & 0xffff0000u);
          const float a2 = __uint_as_float(qv.y << 16), a3 = __uint_as_float(qv.y & 0xffff0000u);
          const float b0 = __uint_as_float(kv.x << 16), b1 = __uint_as_float(kv.x & 0xffff0000u);
          const float b2 = __uint_as_float(kv.y << 16), b3 = __uint_as_float(kv.y & 0xffff0000u);
          qq += a0 * a0 + a1 * a1 + a2 * a2 + a3 * a3;
          kk += b0 * b0 + b1 * b1 + b2 * b2 + b3 * b3;
        }
      }
      qq += __shfl_xor_sync(0xffffffffu, qq, 8);
      qq += __shfl_xor_sync(0xffffffffu, qq, 16);
      kk += __shfl_xor_sync(0xffffffffu, kk, 8);
      kk += __shfl_xor_sync(0xffffffffu, kk, 16);
      if (part == 0) {
        rq[t] = rsqrtf(qq + kL2Eps);
        rk[t] = rsqrtf(kk + kL2Eps);
      }
    } else if constexpr (B16) {
      stage_qk_bf16(q0, k0, in.ld_qk, n, tile, rq, rk);
    } else {
      // normalised float32 rows; rq = rk = 1 (written through the g / beta slots)
      stage_rows<TI, false>(q0, k0, nullptr, in.ld_qk, 0, n, 1.f, 1.f,
                            reinterpret_cast<float *>(tile), nullptr, rq, rk);
    }
    if (!__syncthreads_and(loaded)) {  // the q, k copies never landed
      ok = false;
      break;
    }
    pending = false;
    if (quad == 0 && tt < 32) {  // warp 4 wg: cumulative log-decay of this head
      const float a = sG[2 * lane], b = sG[2 * lane + 1];
      float incl = a + b;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float up = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += up;
      }
      sG[2 * lane] = incl - b;
      sG[2 * lane + 1] = incl;
      // cf[i] = e^{G_e - G_i} / |k_i|, e the last token of i's 16-token block (so at
      // most 1 / |k_i|): the column factor of P and A left of the diagonal blocks
      const float Ge = __shfl_sync(0xffffffffu, incl, (lane & ~7) | 7);
      XS_[2 * lane] = rk[2 * lane] * __expf(Ge - (incl - b));
      XS_[2 * lane + 1] = rk[2 * lane + 1] * __expf(Ge - incl);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // D1 = [Q;K] K^T  (M 128, N 64, K 128)
    if (tid == 0) {
      const uint32_t a_s = smem_addr(tile);
      constexpr uint32_t KSTEP = 2 * tc::kLBO;
      if (TMAQK) {  // K halves of 64: 4 steps of 16 (32 bytes) inside each 128-byte row
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc::mma_ss_f16(tm, tc::smem_desc_sw128(a_s + hf * 2 * kRawHalf + 32 * j),
                           tc::smem_desc_sw128(a_s + hf * 2 * kRawHalf + kRawHalf + 32 * j),
                           tc::idesc_bf16(128, 64), (hf | j) != 0);
      } else if constexpr (B16) {
        constexpr uint32_t SBO = tc::sbo_bytes16(D);
        const uint32_t b_s = a_s + 8 * SBO;
#pragma unroll
        for (int j = 0; j < D / 16; ++j)
          tc::mma_ss_f16(tm, tc::smem_desc(a_s + j * KSTEP, tc::kLBO, SBO),
                         tc::smem_desc(b_s + j * KSTEP, tc::kLBO, SBO), tc::idesc_bf16(128, 64),
                         j > 0);
      } else {
        constexpr uint32_t SBO = tc::sbo_bytes(D);
        const uint32_t b_s = a_s + 8 * SBO;
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
          tc::mma_ss(tm, tc::smem_desc(a_s + j * KSTEP, tc::kLBO, SBO),
                     tc::smem_desc(b_s + j * KSTEP, tc::kLBO, SBO), tc::idesc_tf32(128, 64),
                     j > 0);
      }
      tc::mma_commit(&bar);
    }
    mma_out = true;
    const bool alive = __syncthreads_and(mbar_wait_bounded(&bar, ph));
    tc::fence_after_sync();
    if (!alive) {
      ok = false;
      break;
    }
    mma_out = false;
    // the tile is free again: the next item's rows and scalars travel under this one
    if (nx < items) {
      w = locate(nx, tc_nx);
      if (TMAQK) pending = true;
      if (TMAQK && tid == 0) issue_rows(w);
      load_gb1(w, g_nx, b_nx);
    }
    float *Pg = work + ((int64_t)cidx * p.h_v + h) * (2 * TILE);
    float *Tg = Pg + TILE;
    if (live) {
      // rows 0..63: P[t][i] = e^{G_t - G_i} q~_t.k~_i (i <= t), to the workspace;
      // rows 64..127: A[t][i] = beta_t e^{G_t - G_i} k~_t.k~_i (i < t), to smem.
      // Warp w (w % 2 = q2) holds rows t = 32 q2 .. 32 q2 + 31 of one of them.
      // Columns of the 16-token blocks left of its rows (q2 = 1: i < 32) take
      // e^{G_t - G_i} = e^{G_t - G_e} e^{G_e - G_i} with e the block's last token
      // (both factors at most 1, so no overflow at any decay); the warp's own 32
      // columns take the exact exponential; columns right of them are zero.
      const int row = 32 * quad + lane;
      const bool isA = quad >= 2;
      const int t = isA ? row - 64 : row;
      const int q2 = quad & 1;
      const float sc = isA ? sBeta[t] * rk[t] : rq[t];
      const float gt = sG[t];
      const float *cf = XS_;
      auto put = [&](int i, float4 x) {
        if (isA) *reinterpret_cast<float4 *>(AP + t * AS + i) = x;
        else *reinterpret_cast<float4 *>(Pg + tc::core_off(t, i, C)) = x;
      };
      if (q2 == 1) {
        const float rf0 = sc * __expf(gt - sG[15]), rf1 = sc * __expf(gt - sG[31]);
        float v2[32];
        tc::tmem_ld32(lrow, lrow + 16, v2);
#pragma unroll
        for (int j2 = 0; j2 < 32; j2 += 4) {
          const float rf = j2 < 16 ? rf0 : rf1;
          const float4 c4 = *reinterpret_cast<const float4 *>(cf + j2);
          put(j2, make_float4(rf * c4.x * v2[j2], rf * c4.y * v2[j2 + 1], rf * c4.z * v2[j2 + 2],
                              rf * c4.w * v2[j2 + 3]));
        }
      }
      {
        const int cb = 32 * q2;
        const int lim = isA ? t : t + 1;  // columns i < lim are kept
        float v2[32];
        tc::tmem_ld32(lrow + cb, lrow + cb + 16, v2);
#pragma unroll
        for (int j2 = 0; j2 < 32; j2 += 4) {
          const int i = cb + j2;
          const float4 r4 = *reinterpret_cast<const float4 *>(rk + i);
          const float4 g4 = *reinterpret_cast<const float4 *>(sG + i);
          float4 x;
          x.x = i + 0 < lim ? sc * r4.x * __expf(gt - g4.x) * v2[j2 + 0] : 0.f;
          x.y = i + 1 < lim ? sc * r4.y * __expf(gt - g4.y) * v2[j2 + 1] : 0.f;
          x.z = i + 2 < lim ? sc * r4.z * __expf(gt - g4.z) * v2[j2 + 2] : 0.f;
          x.w = i + 3 < lim ? sc * r4.w * __expf(gt - g4.w) * v2[j2 + 3] : 0.f;
          put(i, x);
        }
      }
      if (q2 == 0 && !isA) {  // P's zero columns 32..63 (A's upper part is never read)
#pragma unroll
        for (int j2 = 0; j2 < 32; j2 += 4) put(32 + j2, make_float4(0.f, 0.f, 0.f, 0.f));
      }
    }
    // D1 is read out (the next Gram product overwrites it), and every thread is
    // past its reads of rq, rk and the tile before the next item rewrites them
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (live) {
      if (TMAQK && tt >= C) {  // (idle in the inversion's first phase) the state
        // walk's per-token scalars of this (chunk, head), token i
        const int i = tt - C;
        float *sb = work + nc * p.h_v * (2 * TILE) + ((int64_t)cidx * p.h_v + h) * kScal;
        const float G = sG[i], gam = expf(G), be = sBeta[i], ik = rk[i];
        sb[kSGam + i] = gam;
        sb[kSBeta + i] = be;
        sb[kSQ + i] = gam * rq[i];
        sb[kSK + i] = be * gam * ik;
        sb[kSKt + i] = expf(sG[C - 1] - G) * ik;
      }
      invert_unit_lower(AP, TP, XS_, tt, 1 + wg);
#pragma unroll
      for (int i4 = 0; i4 < C * (C / 4) / 128; ++i4) {  // T tile [t][i] -> workspace
        const int e = tt + 128 * i4;
        const int t = e % C, c4 = e / C;
        *reinterpret_cast<float4 *>(Tg + tc::core_off(t, 4 * c4, C)) =
            *reinterpret_cast<const float4 *>(TP + t * AS + 4 * c4);
      }
    }
  }
  if (!ok) {
    if (tid == 0) raise_error(p.err, GDN_DEVERR_TIMEOUT);
    // a second bounded chance for copies and MMAs in flight before TMEM and
    // shared memory are released
    if (pending) mbar_wait_bounded(&lbar, ph);
    if (mma_out) mbar_wait_bounded(&bar, ph);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tm, 64);
}

// --------------------------------------------------------------- state side
// shared-memory map of seq_kernel (bytes)
constexpr int S_QK = 0;                        // [Q;K] core tile 128 x 128
constexpr int S_OS = S_QK + 128 * D * 4;       // outputs of a chunk, [64 tokens][128], for
                                               // whole-row stores (up to 32 KiB)
constexpr int S_PT = S_OS + C * XS * 4;        // P tile (from the workspace)
constexpr int S_KT = S_PT + TILE * 4;          // Ktil^T tile [k][i], 128 x 64, right after P:
                                               // [P; Ktil^T] is one 192-row B operand
constexpr int S_TT = S_KT + D * C * 4;         // T tile (from the workspace)
constexpr int S_SC = S_TT + TILE * 4;          // G, gamma, beta, e^{G_n - G}
constexpr int S_XU = S_SC + 4 * C * 4;         // beta v (plain 64 x XS float32)
constexpr int kSeqSmem = S_XU + C * XS * 4;
static_assert(C * D * 4 <= S_PT - S_OS, "shared-memory regions");
static_assert(S_PT % 16 == 0 && S_KT == S_PT + TILE * 4 && S_TT % 16 == 0 && S_XU % 16 == 0,
              "tile alignment");
static_assert(kSeqSmem <= 227 * 1024, "shared memory");

// Roles in seq_kernel: warps 0..7 compute (warp w reads TMEM lanes
// 32 (w % 4) .. +31, column half w / 4) and meet on named barrier 1; warp 8
// issues the MMA groups and the P / T tile copies.  The compute warps hand
// work to warp 8 through mbarriers with one arrival per warp, so a thread that
// stalls issuing a long MMA group holds up no CUDA-core work.
constexpr int kMmaWarp = 8;
constexpr int NTS = NT + 32;
// Compute thread that issues the tensor-map stores of whole output chunks (warp 6).
constexpr int kCopier = 192;

// TMEM columns
// [S Q^T | S K^T] is one N = 128 product over the [Q;K] tile: D3 then E
// [D4 | S] is one N = 192 accumulator over [P; Ktil^T]: output part then state
constexpr uint32_t T_D4 = 0, T_S = 64, T_D3 = 192, T_E = 256, T_F = 320, T_DD = 384;
constexpr uint32_t SEQ_TMEM = 512;

__device__ __forceinline__ void cw_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// The 256 compute threads meet; true when p holds for every one of them.
__device__ __forceinline__ bool cw_and(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\t"
      "bar.red.and.pred b, 1, 256, a;\n\tselp.u32 %0, 1, 0, b;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p)
      : "memory");
  return r != 0;
}
// Bounded wait that also gives up as soon as the other role has failed.
__device__ __forceinline__ bool wait_live(uint64_t *bar, uint32_t parity,
                                          const volatile int *dead) {
  for (uint32_t it = 0; it < (1u << 20); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*dead) return false;
  }
  return false;
}
// This warp's TMEM stores have completed (each lane waited) and its operand
// writes to shared memory are fenced for the tensor core: one arrival.
__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
  tc::fence_before_sync();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

template <typename TI, typename TO>
__global__ void __launch_bounds__(NTS, 1)
    seq_kernel(PoolView p, int layer, SeqIndex seq, QKV in, TO *__restrict__ o, float scale,
               const int32_t *__restrict__ off, int64_t cap, const float *__restrict__ work,
               Checkpoints ck) {
  extern __shared__ __align__(1024) unsigned char smem[];
  float *QK = reinterpret_cast<float *>(smem + S_QK);
  TO *OS = reinterpret_cast<TO *>(smem + S_OS);
  float *XU = reinterpret_cast<float *>(smem + S_XU);
  float *PT = reinterpret_cast<float *>(smem + S_PT);
  float *KT = reinterpret_cast<float *>(smem + S_KT);
  float *TT = reinterpret_cast<float *>(smem + S_TT);
  float *sG = reinterpret_cast<float *>(smem + S_SC);
  float *sGam = sG + C;
  float *sBeta = sGam + C;
  float *sDte = sBeta + C;
  __shared__ __align__(8) uint64_t b_ed3, b_dd, b_upd;  // MMA groups done
  __shared__ __align__(8) uint64_t tbar;                 // P / T tiles landed
  __shared__ __align__(8) uint64_t f_rdy, g_rdy, s_rdy;  // compute warps -> MMA warp
  __shared__ uint32_t tmem_slot;
  __shared__ int dead;  // set by the role that gave up waiting

  const int h = blockIdx.x, si = off[seq.n_seqs + 1 + blockIdx.y];  // longest first
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int quad = warp & 3, half = (warp >> 2) & 1;
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
  const int nch = (len + C - 1) / C;
  const int hk = h / (p.h_v / p.h_k);
  const gdn_dtype sd = p.state_dtype;
  char *Sg = p.state_at(p.state_head_elem(layer, slot, h));  // float32, bf16 or f16 elements
  const float *wsq = work + ((int64_t)off[si] * p.h_v + h) * (2 * TILE);  // chunk 0's tiles
  const int64_t wstep = (int64_t)p.h_v * (2 * TILE);                      // next chunk

  if (warp == 0) tc::tmem_alloc(&tmem_slot, SEQ_TMEM);
  if (tid == 0) {
    mbar_init(&b_ed3, 1);
    mbar_init(&b_dd, 1);
    mbar_init(&b_upd, 1);
    mbar_init(&tbar, 1);
    mbar_init(&f_rdy, 8);
    mbar_init(&g_rdy, 8);
    mbar_init(&s_rdy, 8);
    dead = 0;
    mbar_fence_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = tmem_slot;
  volatile int *vdead = &dead;

  if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA warp
    // Per chunk c: [F_c staged, P/T tiles] -> Delta^T = F T^T -> [S scaled,
    // Ktil^T] -> [D4 | S] += Delta^T [P; Ktil^T]^T -> next tiles; [chunk c+1
    // staged] -> [D3 | E] of chunk c+1.  Lane 0 issues; the warp waits together.
    const uint32_t qk_s = smem_addr(QK), pt_s = smem_addr(PT), tt_s = smem_addr(TT);
    constexpr uint32_t SBO_D = tc::sbo_bytes(D);
    constexpr uint32_t SBO_C = tc::sbo_bytes(C);
    constexpr uint32_t KSTEP = 2 * tc::kLBO;
    const bool leader = lane == 0;
    auto all_lanes = [](bool x) { return __all_sync(0xffffffffu, x) != 0; };
    auto load_tiles = [&](int c) {  // P and T tiles of chunk c onto tbar
      if (leader) {
        const float *src = wsq + (int64_t)c * wstep;
        mbar_arrive_expect_tx(&tbar, 2 * kTileBytes);
        bulk_g2s(PT, src, kTileBytes, &tbar);
        bulk_g2s(TT, src + TILE, kTileBytes, &tbar);
      }
    };
    // [D3 | E] = S [Q;K]^T  (A = S from TMEM; M 128, N 128, K 128)
    auto issue_ed3 = [&]() {
      if (leader) {
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
          tc::mma_ts(tm + T_D3, tm + T_S + j * 8,
                     tc::smem_desc(qk_s + j * KSTEP, tc::kLBO, SBO_D), tc::idesc_tf32(128, 128),
                     j > 0);
        tc::mma_commit(&b_ed3);
      }
      __syncwarp();
    };
    int n_ed3 = 0, n_dd = 0, n_upd = 0, n_t = 1;  // groups issued, tile loads armed
    load_tiles(0);
    bool ok = all_lanes(wait_live(&s_rdy, 0, vdead));  // chunk 0 staged, state in TMEM
    if (ok) {
      tc::fence_after_sync();
      issue_ed3();
      n_ed3 = 1;
    }
    for (int c = 0; ok && c < nch; ++c) {
      const uint32_t par = c & 1;
      ok = all_lanes(wait_live(&f_rdy, par, vdead) && wait_live(&tbar, par, vdead));
      if (!ok) break;
      tc::fence_after_sync();
      if (leader) {  // Delta^T = F T^T  (A = F from TMEM; M 128, N 64, K 64)
#pragma unroll
        for (int j = 0; j < C / 8; ++j)
          tc::mma_ts(tm + T_DD, tm + T_F + j * 8,
                     tc::smem_desc(tt_s + j * KSTEP, tc::kLBO, SBO_C), tc::idesc_tf32(128, 64),
                     j > 0);
        tc::mma_commit(&b_dd);
      }
      __syncwarp();
      ++n_dd;
      ok = all_lanes(wait_live(&b_dd, par, vdead) && wait_live(&g_rdy, par, vdead));
      if (!ok) break;
      tc::fence_after_sync();
      // [D4 | S] += Delta^T [P; Ktil^T]^T: D4 (onto gamma S Q^T) and the state update in
      // one N = 192 chain; K = 64
      if (leader) {
#pragma unroll
        for (int j = 0; j < C / 8; ++j)
          tc::mma_ts(tm + T_D4, tm + T_DD + j * 8,
                     tc::smem_desc(pt_s + j * KSTEP, tc::kLBO, SBO_C), tc::idesc_tf32(128, 192),
                     1);
        tc::mma_commit(&b_upd);
      }
      __syncwarp();
      ++n_upd;
      ok = all_lanes(wait_live(&b_upd, par, vdead));
      if (!ok || c + 1 == nch) break;
      load_tiles(c + 1);  // both tiles are free again
      ++n_t;
      ok = all_lanes(wait_live(&s_rdy, (c + 1) & 1, vdead));
      if (!ok) break;
      tc::fence_after_sync();
      issue_ed3();
      ++n_ed3;
    }
    if (!ok) {
      if (leader) {
        *vdead = 1;
        raise_error(p.err, GDN_DEVERR_TIMEOUT);
      }
      // at most one group per barrier and one tile load can be in flight: let
      // them finish before TMEM and shared memory are released
      if (n_ed3) mbar_wait_bounded(&b_ed3, (n_ed3 - 1) & 1);
      if (n_dd) mbar_wait_bounded(&b_dd, (n_dd - 1) & 1);
      if (n_upd) mbar_wait_bounded(&b_upd, (n_upd - 1) & 1);
      mbar_wait_bounded(&tbar, (n_t - 1) & 1);
    }
  } else {
    // ----------------------------------------------------------- compute warps
    const uint32_t lrow = tm + ((uint32_t)(32 * quad) << 16);
    {  // state row `row`, column half `half` -> TMEM (float32)
      const int64_t e0 = (int64_t)row * D + 64 * half;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float v[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 x = state_ld4(Sg, e0 + (c * 4 + j) * 4, sd);
          v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
        }
        tc::tmem_st16(lrow + T_S + 64 * half + c * 16, v);
      }
      tc::tmem_st_wait();
    }

    const bool ovec = ((uintptr_t)o & 15) == 0;  // output rows start 16-byte aligned
    const TI *qg = static_cast<const TI *>(in.q);
    const TI *kg = static_cast<const TI *>(in.k);
    const TI *vg = static_cast<const TI *>(in.v);
    bool alive = true;

    // Stage chunk c0s into QK, XU and the scalars, and form its cumulative
    // decays.  Ends with the tile writes fenced for the tensor core.
    auto stage_next = [&](int c0s) {
      const int ns = min(C, len - c0s);
      stage_chunk<TI, true>(in, p, h, hk, lo + c0s, ns, QK, XU, sG, sBeta);
      cw_sync();
      if (warp == 7) {  // cumulative log-decay (padded tokens carry g = 0)
        const float a = sG[2 * lane], b = sG[2 * lane + 1];
        float incl = a + b;
#pragma unroll
        for (int sh = 1; sh < 32; sh <<= 1) {
          const float up = __shfl_up_sync(0xffffffffu, incl, sh);
          if (lane >= sh) incl += up;
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
    };
    // The Ktil^T tile of the staged chunk (needs its sDte), and rows `ahead`
    // chunks further on pulled towards L2.
    // Each thread reads 4 consecutive k of one token (a 16-byte piece of the K
    // core tile), the 4 lanes of a quad transpose their 4 x 4 block with two
    // xor-shuffle rounds, and each stores 4 consecutive tokens of one k.
    auto build_kt = [&](int c0s) {
      const int l4 = lane & 3;
#pragma unroll 4
      for (int it = 0; it < 8; ++it) {
        const int blk = it * 8 + warp;                 // 8 token groups x 8 k-quad groups
        const int i = 8 * (blk & 7) + (lane & 7);
        const int k4 = 4 * (blk >> 3) + (lane >> 3);   // columns 4 k4 .. 4 k4 + 3
        const float4 x = *reinterpret_cast<const float4 *>(QK + tc::core_off(64 + i, 4 * k4, D));
        const float d = sDte[i];
        const float v0 = d * x.x, v1 = d * x.y, v2 = d * x.z, v3 = d * x.w;
        // stage 1 (xor 2): lanes 0,1 keep columns 0,1 and take rows 2,3's; lanes 2,3 the rest
        const bool hi2 = (l4 & 2) != 0;
        const float r0 = __shfl_xor_sync(0xffffffffu, hi2 ? v0 : v2, 2);
        const float r1 = __shfl_xor_sync(0xffffffffu, hi2 ? v1 : v3, 2);
        const float a0 = hi2 ? r0 : v0, a1 = hi2 ? r1 : v1;
        const float a2 = hi2 ? v2 : r0, a3 = hi2 ? v3 : r1;
        // stage 2 (xor 1): 2 x 2 transposes
        const bool hi1 = (l4 & 1) != 0;
        const float s0 = __shfl_xor_sync(0xffffffffu, hi1 ? a0 : a1, 1);
        const float s1 = __shfl_xor_sync(0xffffffffu, hi1 ? a2 : a3, 1);
        const float4 w = hi1 ? make_float4(s0, a1, s1, a3) : make_float4(a0, s0, a2, s1);
        // lane l4 now holds column k = 4 k4 + l4 of tokens ib .. ib + 3
        const int ib = 8 * (blk & 7) + (lane & 4);
        *reinterpret_cast<float4 *>(KT + tc::core_off(4 * k4 + l4, ib, C)) = w;
      }
      const int t = tid & (C - 1);
      const int64_t tok = lo + c0s + 2 * C + t;
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
      tc::fence_async_smem();
    };

    // chunk 0: stage it and hand it (with the state) to the MMA warp, then build
    // its Ktil^T while [D3 | E] runs
    stage_next(0);
    alive = cw_and(alive);
    if (alive) warp_arrive(&s_rdy);
    if (alive) build_kt(0);

    // Per chunk the state chain is [D3 | E] -> F -> Delta -> state update ->
    // next [D3 | E]; the next chunk is staged under the Delta MMAs, and this
    // chunk's outputs and the next Ktil^T under the next [D3 | E].
    for (int c = 0; c < nch && alive; ++c) {
      const int c0 = c * C;
      const uint32_t par = c & 1;
      const int n = min(C, len - c0);
      const bool last = c + 1 == nch;
      alive = cw_and(wait_live(&b_ed3, par, vdead));  // [D3 | E] done
      if (!alive) break;
      tc::fence_after_sync();

      // F[v][t] = beta_t v_t[v] - beta_t gamma_t E[v][t] into TMEM; the output's state
      // part gamma_t (S Q^T)[v][t] into the D4 columns (the Delta^T P^T MMA adds to it)
      const int i0 = 32 * half;
      {
        const int v = row;
        // this thread's 32 columns of E and D3, all four loads under one wait
        float e[32], d3[32];
        tc::tmem_ld16x4(lrow + T_E + i0, lrow + T_E + i0 + 16, lrow + T_D3 + i0,
                        lrow + T_D3 + i0 + 16, e, d3);
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
          const int t0 = i0 + 16 * cb;
          float f[16], dd[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = t0 + j;
            dd[j] = d3[16 * cb + j] * sGam[t];
            const float bv = XU[t * XS + v];  // beta_t v_t[v] (0 for padded tokens)
            f[j] = bv - sBeta[t] * sGam[t] * e[16 * cb + j];
          }
          tc::tmem_st16(lrow + T_F + t0, f);
          tc::tmem_st16(lrow + T_D4 + t0, dd);
        }
        tc::tmem_st_wait();
      }
      warp_arrive(&f_rdy);
      {  // S <- gamma_n S, under Delta^T = F T^T (which reads neither)
        const float gn = sGam[C - 1];
#pragma unroll 1
        for (int cb = 0; cb < 2; ++cb) {
          float sv[32];
          const uint32_t sc = lrow + T_S + 64 * half + 32 * cb;
          tc::tmem_ld32(sc, sc + 16, sv);
#pragma unroll
          for (int j = 0; j < 32; ++j) sv[j] *= gn;
          tc::tmem_st16(sc, sv);
          tc::tmem_st16(sc + 16, sv + 16);
        }
        tc::tmem_st_wait();
      }
      warp_arrive(&g_rdy);  // (this chunk's Ktil^T was fenced when it was built)

      if (!last) {
        cw_sync();  // every warp is past its reads of XU, gamma and beta
        stage_next(c0 + C);
        if (alive) warp_arrive(&s_rdy);
      }
      alive = cw_and(alive && wait_live(&b_upd, par, vdead));  // D4, new state ready
      if (!alive) break;
      tc::fence_after_sync();
      if (ck.every > 0 && c0 + C <= len && (c0 + C) % ck.every == 0) {  // checkpoint: copy S out
        const int j = (c0 + C) / ck.every - 1;
        const int ds = j < ck.per_seq ? ck.slots[(int64_t)si * ck.per_seq + j] : -1;
        if (ds >= p.n_slots) {
          if (tid == 0) raise_error(p.err, GDN_DEVERR_SLOT);
        } else if (ds >= 0) {
          char *dst = p.state_at(p.state_head_elem(layer, ds, h));
          const int64_t e0 = (int64_t)row * D + 64 * half;
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {
            float v[16];
            tc::tmem_ld16(lrow + T_S + 64 * half + 16 * cb, v);
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4)
              state_st4<false>(dst, e0 + (cb * 4 + j4) * 4,
                               make_float4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]),
                               sd);
          }
        }
      }

      // outputs o[t][v] = scale D4[v][t] (gamma_t S Q^T + Delta^T P^T): this warp's half
      // of t into the [t][v] staging tile, then whole 16-byte pieces of token rows out
      {
        const int v = row;
        const int64_t ostep = (int64_t)p.h_v * D;
        float d4[32];
        tc::tmem_ld32(lrow + T_D4 + i0, lrow + T_D4 + i0 + 16, d4);
        if (ovec) {
#pragma unroll
          for (int j = 0; j < 32; ++j) Elem<TO>::store1(OS + (i0 + j) * D + v, scale * d4[j]);
          cw_sync();
          constexpr int VEC = 16 / (int)sizeof(TO), PIECES = D / VEC;  // per token row
          TO *ob = o + (lo + c0) * ostep + (int64_t)h * D;
          for (int e = tid; e < n * PIECES; e += NT) {
            const int t = e / PIECES, pc = e % PIECES;
            *reinterpret_cast<uint4 *>(ob + t * ostep + pc * VEC) =
                *reinterpret_cast<const uint4 *>(OS + t * D + pc * VEC);
          }
        } else {
          TO *ob = o + (lo + c0 + i0) * ostep + (int64_t)h * D + v;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (i0 + j < n) Elem<TO>::store1(ob + (int64_t)j * ostep, scale * d4[j]);
        }
      }
      if (!last) build_kt(c0 + C);
    }

    if (alive) {
      const int64_t e0 = (int64_t)row * D + 64 * half;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float v[16];
        tc::tmem_ld16(lrow + T_S + 64 * half + c * 16, v);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          state_st4<false>(Sg, e0 + (c * 4 + j) * 4,
                           make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]), sd);
      }
    } else {
      *vdead = 1;
      if (tid == 0) raise_error(p.err, GDN_DEVERR_TIMEOUT);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tm, SEQ_TMEM);
}

// ------------------------------------------------- state side, bf16 rows
// The state walk for bf16 q, k, v whose rows arrive by tensor-map copies.
// [D3 | E] = S [Q;K]^T runs on kind::f16 over the raw tiles themselves (the
// exact input values, two chunks of q, k buffered ahead: bf16 operands,
// float32 accumulation), with the state rounded to nearest bf16 and packed
// two per column into the free F columns of TMEM; the L2 norms of q and k
// scale the products' columns.  Delta^T = F T^T and the N = 192 output /
// state update stay on kind::tf32 as in seq_kernel; so do the roles of the
// nine warps.  The state's carried value stays float32 in TMEM: only this
// product sees it rounded, and its rounding is not the dominant error (a
// second bf16 term for the remainder left the errors against the float64
// recurrence unchanged to four digits).

// TMEM columns of seq_bf16_kernel: [D4a | S | D4b | D3 | E | F | Delta].  The
// output part alternates between D4a (even chunks: [D4a | S] += Delta [P; Ktil^T])
// and D4b (odd chunks: [S | D4b] += Delta [Ktil^T; P]), so a chunk's outputs
// can be read while the next chunk's update runs.  S_bf16 shares F's columns.
constexpr uint32_t U_D4A = 0, U_S = 64, U_D4B = 192, U_D3 = 256, U_E = 320, U_F = 384,
                   U_DD = 448;
__device__ __forceinline__ uint32_t u_d4(int c) { return (c & 1) ? U_D4B : U_D4A; }

// shared-memory map of seq_bf16_kernel (bytes from a 1024-byte aligned base)
constexpr int kQKBuf = 4 * kRawHalf;            // raw [q h0 | k h0 | q h1 | k h1], 32 KiB
constexpr int B_QK = 0;                         // two q, k buffers (chunk c in buffer c % 2)
constexpr int B_V = B_QK + 2 * kQKBuf;          // raw v [v h0 | v h1]
constexpr int B_OS = B_V + 2 * kRawHalf;        // outputs of a chunk, [64 tokens][128]
constexpr int B_PT = B_OS + C * D * 4;          // P tile of even chunks
constexpr int B_KT = B_PT + TILE * 4;           // Ktil^T tile: [P0; Ktil^T] and
constexpr int B_PT1 = B_KT + D * C * 4;         // [Ktil^T; P1] are contiguous operands
constexpr int B_TT = B_PT1 + TILE * 4;          // T tile
constexpr int B_SB = B_TT + TILE * 4;           // two per-token scalar blocks (chunk c in c % 2)
constexpr int kSeqBf16Smem = B_SB + 2 * kScal * 4 + 1024;  // + alignment slack
static_assert(B_V % 1024 == 0 && B_PT % 16 == 0 && B_SB % 16 == 0 && B_KT == B_PT + TILE * 4 &&
                  B_PT1 == B_KT + D * C * 4,
              "tile alignment");
static_assert(kSeqBf16Smem <= 227 * 1024, "shared memory");


template <typename TO>
__global__ void __launch_bounds__(NTS, 1)
    seq_bf16_kernel(PoolView p, int layer, SeqIndex seq, QKV in, TO *__restrict__ o, float scale,
                    const int32_t *__restrict__ off, int64_t cap, const float *__restrict__ work,
                    const __grid_constant__ InMaps maps, int o_map, Checkpoints ck) {
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *sm = smem + ((1024u - (smem_addr(smem) & 1023u)) & 1023u);
  unsigned char *RQK = sm + B_QK;
  unsigned char *RV = sm + B_V;
  TO *OS = reinterpret_cast<TO *>(sm + B_OS);
  // staged outputs: bf16 as two 64-column halves of [64 tokens][64] in the
  // 128-byte swizzle (the output map's boxes); float32 as plain [64][128] rows
  constexpr bool OB16 = std::is_same<TO, bf16>::value;
  constexpr int kOSRow = D;
  static_assert(B_OS % 1024 == 0, "output staging alignment");
  float *PT = reinterpret_cast<float *>(sm + B_PT);
  float *PT1 = reinterpret_cast<float *>(sm + B_PT1);
  float *KT = reinterpret_cast<float *>(sm + B_KT);
  float *TT = reinterpret_cast<float *>(sm + B_TT);
  // chunk c's per-token scalars (from the key-side kernel), buffer c % 2
  float *SB = reinterpret_cast<float *>(sm + B_SB);
  auto scal = [&](int c) -> const float * { return SB + (c & 1) * kScal; };
  __shared__ __align__(8) uint64_t b_ed3, b_dd, b_upd;  // MMA groups done
  __shared__ __align__(8) uint64_t tbar, vbar;           // P / T tiles, raw v landed
  __shared__ __align__(8) uint64_t rbar[2];              // raw q, k and scalars landed
  __shared__ __align__(8) uint64_t f_rdy, g_rdy, s_rdy;  // compute warps -> MMA warp
  __shared__ uint32_t tmem_slot;
  __shared__ int dead;  // set by the role that gave up waiting

  const int h = blockIdx.x, si = off[seq.n_seqs + 1 + blockIdx.y];  // longest first
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int quad = warp & 3, half = (warp >> 2) & 1;
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
  const int nch = (len + C - 1) / C;
  const int hk = h / (p.h_v / p.h_k);
  const gdn_dtype sd = p.state_dtype;
  char *Sg = p.state_at(p.state_head_elem(layer, slot, h));  // float32, bf16 or f16 elements
  const float *wsq = work + ((int64_t)off[si] * p.h_v + h) * (2 * TILE);  // chunk 0's tiles
  // chunk 0's per-token scalars (written by the key-side kernel), next chunk h_v blocks on
  const float *wscal = work + cap * p.h_v * (2 * TILE) + ((int64_t)off[si] * p.h_v + h) * kScal;
  const int64_t wstep = (int64_t)p.h_v * (2 * TILE);                      // next chunk

  if (warp == 0) tc::tmem_alloc(&tmem_slot, SEQ_TMEM);
  if (tid == 0) {
    mbar_init(&b_ed3, 1);
    mbar_init(&b_dd, 1);
    mbar_init(&b_upd, 1);
    mbar_init(&tbar, 1);
    mbar_init(&vbar, 1);
    mbar_init(&rbar[0], 1);
    mbar_init(&rbar[1], 1);
    mbar_init(&f_rdy, 8);
    mbar_init(&g_rdy, 8);
    mbar_init(&s_rdy, 8);
    dead = 0;
    mbar_fence_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tm = tmem_slot;
  volatile int *vdead = &dead;

  if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA warp
    const uint32_t pt_s = smem_addr(PT), kt_s = smem_addr(KT), tt_s = smem_addr(TT);
    constexpr uint32_t SBO_C = tc::sbo_bytes(C);
    constexpr uint32_t KSTEP = 2 * tc::kLBO;
    const bool leader = lane == 0;
    auto all_lanes = [](bool x) { return __all_sync(0xffffffffu, x) != 0; };
    // Row copies: v of chunk c onto vbar; q, k of chunk c into buffer c % 2
    // with the chunk's per-token scalars from the key-side kernel onto rbar[c % 2]
    // (scalars = false: issued later, once the key-side grid has finished)
    int n_r0 = 0, n_r1 = 0, n_v = 0;  // copies armed per barrier
    auto fetch_v = [&](int c) {
      if (leader) prefetch_v(maps, h, lo + (int64_t)c * C, RV, &vbar);
      ++n_v;
    };
    auto fetch_scal = [&](int c) {
      if (leader)
        bulk_g2s(SB + (c & 1) * kScal, wscal + (int64_t)c * p.h_v * kScal, kScal * 4,
                 &rbar[c & 1]);
    };
    auto fetch_qk = [&](int c, bool scalars) {
      const int b = c & 1;
      if (leader) {
        prefetch_qk_pairs(maps, hk, lo + (int64_t)c * C, RQK + b * kQKBuf, &rbar[b], kScal * 4);
        if (scalars) fetch_scal(c);
      }
      if (b) ++n_r1; else ++n_r0;
    };
    auto load_tiles = [&](int c) {  // P and T tiles of chunk c onto tbar
      if (leader) {
        const float *src = wsq + (int64_t)c * wstep;
        mbar_arrive_expect_tx(&tbar, 2 * kTileBytes);
        bulk_g2s((c & 1) ? PT1 : PT, src, kTileBytes, &tbar);
        bulk_g2s(TT, src + TILE, kTileBytes, &tbar);
      }
    };
    // [D3 | E] = S_bf16 [Q;K]^T over the raw rows of chunk c: M 128, N 128,
    // K 128 in steps of 16 (four 32-byte steps inside each swizzled 64-column half)
    // Descriptor bases, built once: a K step adds its byte offset / 16 to the
    // 14-bit address field (every operand lies below 256 KiB: no carry out).
    const uint64_t ed3_d0 = tc::smem_desc_sw128(smem_addr(RQK));
    const uint64_t ed3_d1 = tc::smem_desc_sw128(smem_addr(RQK + kQKBuf));
    const uint64_t dd_d = tc::smem_desc(tt_s, tc::kLBO, SBO_C);
    const uint64_t up_d0 = tc::smem_desc(pt_s, tc::kLBO, SBO_C);
    const uint64_t up_d1 = tc::smem_desc(kt_s, tc::kLBO, SBO_C);
    auto issue_ed3 = [&](int c) {
      if (leader) {
        const uint64_t b0 = (c & 1) ? ed3_d1 : ed3_d0;
        constexpr uint32_t id = tc::idesc_bf16(128, 128);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t bd = b0 + (uint64_t)((((ks >> 2) * 2 * kRawHalf) + 32 * (ks & 3)) >> 4);
          tc::mma_ts_f16(tm + U_D3, tm + U_F + 8 * ks, bd, id, ks > 0);
        }
        tc::mma_commit(&b_ed3);
      }
      __syncwarp();
    };
    int n_ed3 = 0, n_dd = 0, n_upd = 0, n_t = 1;  // groups issued, tile loads armed
    fetch_v(0);
    fetch_qk(0, false);
    if (nch > 1) fetch_qk(1, false);
    // the key-side grid has written the tiles and scalars (this launch may
    // start before it ends)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    fetch_scal(0);
    if (nch > 1) fetch_scal(1);
    load_tiles(0);
    bool ok = all_lanes(wait_live(&s_rdy, 0, vdead) && wait_live(&rbar[0], 0, vdead));
    if (ok) {
      tc::fence_after_sync();
      issue_ed3(0);
      n_ed3 = 1;
    }
    for (int c = 0; ok && c < nch; ++c) {
      const uint32_t par = c & 1;
      ok = all_lanes(wait_live(&f_rdy, par, vdead) && wait_live(&tbar, par, vdead));
      if (!ok) break;
      tc::fence_after_sync();
      if (leader) {  // Delta^T = F T^T  (A = F from TMEM; M 128, N 64, K 64)
#pragma unroll
        for (int j = 0; j < C / 8; ++j)
          tc::mma_ts(tm + U_DD, tm + U_F + j * 8, dd_d + (uint64_t)((j * KSTEP) >> 4),
                     tc::idesc_tf32(128, 64), j > 0);
        tc::mma_commit(&b_dd);
      }
      __syncwarp();
      ++n_dd;
      ok = all_lanes(wait_live(&b_dd, par, vdead) && wait_live(&g_rdy, par, vdead));
      if (!ok) break;
      tc::fence_after_sync();
      if (leader) {  // [D4a | S] += Delta^T [P0; Ktil^T]^T (even c) or
                     // [S | D4b] += Delta^T [Ktil^T; P1]^T (odd c): N 192, K 64
        const uint32_t dcol = (c & 1) ? U_S : U_D4A;
        const uint64_t b0 = (c & 1) ? up_d1 : up_d0;
#pragma unroll
        for (int j = 0; j < C / 8; ++j)
          tc::mma_ts(tm + dcol, tm + U_DD + j * 8, b0 + (uint64_t)((j * KSTEP) >> 4),
                     tc::idesc_tf32(128, 192), 1);
        tc::mma_commit(&b_upd);
      }
      __syncwarp();
      ++n_upd;
      // under the update: the v tile is free (every warp's F pass is done), and
      // so is the q, k buffer of chunk c (its [D3 | E], F and Ktil^T are done)
      if (c + 1 < nch) fetch_v(c + 1);
      if (c + 2 < nch) fetch_qk(c + 2, true);
      ok = all_lanes(wait_live(&b_upd, par, vdead));
      if (!ok || c + 1 == nch) break;
      load_tiles(c + 1);  // both tiles are free again
      ++n_t;
      ok = all_lanes(wait_live(&s_rdy, (c + 1) & 1, vdead) &&
                     wait_live(&rbar[(c + 1) & 1], ((c + 1) >> 1) & 1, vdead));
      if (!ok) break;
      tc::fence_after_sync();
      issue_ed3(c + 1);
      ++n_ed3;
    }
    if (!ok) {
      if (leader) {
        *vdead = 1;
        raise_error(p.err, GDN_DEVERR_TIMEOUT);
      }
      if (n_ed3) mbar_wait_bounded(&b_ed3, (n_ed3 - 1) & 1);
      if (n_dd) mbar_wait_bounded(&b_dd, (n_dd - 1) & 1);
      if (n_upd) mbar_wait_bounded(&b_upd, (n_upd - 1) & 1);
      mbar_wait_bounded(&tbar, (n_t - 1) & 1);
      // row copies still in flight land before shared memory is released
      if (n_r0 > 0) mbar_wait_bounded(&rbar[0], (n_r0 - 1) & 1);
      if (n_r1 > 0) mbar_wait_bounded(&rbar[1], (n_r1 - 1) & 1);
      if (n_v > 0) mbar_wait_bounded(&vbar, (n_v - 1) & 1);
    }
  } else {
    // ----------------------------------------------------------- compute warps
    const uint32_t lrow = tm + ((uint32_t)(32 * quad) << 16);
    const bool ovec = ((uintptr_t)o & 15) == 0;  // output rows start 16-byte aligned
    {  // state row `row`, column half `half` -> TMEM (float32)
      const int64_t e0 = (int64_t)row * D + 64 * half;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float v[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 x = state_ld4(Sg, e0 + (c * 4 + j) * 4, sd);
          v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
        }
        tc::tmem_st16(lrow + U_S + 64 * half + c * 16, v);
      }
      tc::tmem_st_wait();
    }
    bool alive = true;

    // chunk c's copies have landed (every compute thread waits itself)
    auto rows_landed = [&](int c) { return wait_live(&rbar[c & 1], (c >> 1) & 1, vdead); };
    // S (float32) -> S_bf16 at the F columns, packed two per column (lower k in
    // the low half), for the next [D3 | E], and S <- gn S in place for the next
    // state update (which S_bf16 does not see).  Arrives on s_rdy once all of
    // it is in TMEM.
    auto split_scale = [&](float gn) {
#pragma unroll 1
      for (int cb = 0; cb < 2; ++cb) {
        float sv[32], hp[16];
        const uint32_t sc = lrow + U_S + 64 * half + 32 * cb;
        tc::tmem_ld32(sc, sc + 16, sv);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float s0 = sv[2 * m], s1 = sv[2 * m + 1];
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(s0, s1);
          hp[m] = __uint_as_float(*reinterpret_cast<const uint32_t *>(&h2));
        }
        tc::tmem_st16(lrow + U_F + 32 * half + 16 * cb, hp);
#pragma unroll
        for (int j = 0; j < 32; ++j) sv[j] *= gn;
        tc::tmem_st16(sc, sv);
        tc::tmem_st16(sc + 16, sv + 16);
      }
      tc::tmem_st_wait();
      warp_arrive(&s_rdy);
    };
    // Ktil^T of chunk c (tokens past the chunk's end zero) from its raw k rows.
    // A warp task is one
    // token quad x 32 consecutive k (one k per lane): four 16-bit reads (one
    // per token, 64 contiguous bytes of a swizzled row per warp), scaled, and
    // one 16-byte store (a quarter-warp fills one core matrix).
    auto build_kt = [&](int c) {
      const int nn = min(C, len - c * C);
      const unsigned char *kb = RQK + (c & 1) * kQKBuf + kRawHalf;
      const float *sKt = scal(c) + kSKt;
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int task = it * 8 + warp;
        const int tq = task & 15, k = 32 * (task >> 4) + lane;
        const unsigned char *kc = kb + (k >> 6) * 2 * kRawHalf + (k & 7) * 2;
        const int piece = (k & 63) >> 3;
        const float4 d4 = *reinterpret_cast<const float4 *>(sKt + 4 * tq);
        const float d[4] = {d4.x, d4.y, d4.z, d4.w};
        float w[4];
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
          const int i = 4 * tq + ii;
          const uint32_t u =
              *reinterpret_cast<const unsigned short *>(kc + i * 128 + ((piece ^ (i & 7)) << 4));
          w[ii] = d[ii] * __uint_as_float(u << 16);
          if (nn < C && i >= nn) w[ii] = 0.f;
        }
        *reinterpret_cast<float4 *>(KT + tc::core_off(k, 4 * tq, C)) =
            make_float4(w[0], w[1], w[2], w[3]);
      }
      tc::fence_async_smem();
    };
    // F[v][t] = beta_t v_t[v] - (beta_t gamma_t / |k_t|) (S K^T)[v][t] and the
    // output's state part (gamma_t / |q_t|) (S Q^T)[v][t] into TMEM, this
    // thread's 32 tokens; padded tokens (FULL false) give 0
    auto f_pass = [&](auto full, int n, int i0, uint32_t d4c, const float *sc) {
      constexpr bool FULL = decltype(full)::value;
      const float *sBeta = sc + kSBeta, *sQ = sc + kSQ, *sK = sc + kSK;
      const int v = row;
      const unsigned char *vr = RV + (v >> 6) * kRawHalf + (v & 7) * 2;
      const int vpiece = (v & 63) >> 3;
#pragma unroll 1
      for (int cb = 0; cb < 2; ++cb) {
        const int t0 = i0 + 16 * cb;
        float ed[32], f[16], dd[16];  // ed: 16 columns of E, then the same of D3
        tc::tmem_ld32(lrow + U_E + t0, lrow + U_D3 + t0, ed);
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {  // four tokens' scalars per vector load
          const float4 b4 = *reinterpret_cast<const float4 *>(sBeta + t0 + 4 * j4);
          const float4 q4 = *reinterpret_cast<const float4 *>(sQ + t0 + 4 * j4);
          const float4 k4 = *reinterpret_cast<const float4 *>(sK + t0 + 4 * j4);
          const float be[4] = {b4.x, b4.y, b4.z, b4.w}, qs[4] = {q4.x, q4.y, q4.z, q4.w};
          const float ks[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int j = 4 * j4 + jj, t = t0 + j;
            const uint32_t u = *reinterpret_cast<const unsigned short *>(
                vr + t * 128 + ((vpiece ^ (t & 7)) << 4));
            const float bv = be[jj] * __uint_as_float(u << 16);
            dd[j] = ed[16 + j] * qs[jj];
            f[j] = bv - ks[jj] * ed[j];
            if (!FULL && t >= n) dd[j] = f[j] = 0.f;
          }
        }
        tc::tmem_st16(lrow + U_F + t0, f);
        tc::tmem_st16(lrow + d4c + t0, dd);
      }
      tc::tmem_st_wait();
    };

    // outputs of chunk cc, o[t][v] = scale D4[v][t]: this warp's half of t into the
    // [t][v] staging tile (free once the last tensor-map store has read it), then
    // whole 16-byte pieces of token rows out
    auto out_chunk = [&](int cc) {
      const int c0 = cc * C, n = min(C, len - c0), i0 = 32 * half;
      if (tid == kCopier) bulk_wait_read();
      cw_sync();
      {
        const int v = row;
        const int64_t ostep = (int64_t)p.h_v * D;
        float d4[32];
        tc::tmem_ld32(lrow + u_d4(cc) + i0, lrow + u_d4(cc) + i0 + 16, d4);
        if (ovec) {
          if constexpr (OB16) {
            // lanes v, v ^ 1 swap one value per token pair (j, j + 4) of each group of
            // 8: the even lane writes (v, v + 1) of token j, the odd lane (v - 1, v) of
            // token j + 4; the two rows differ in the swizzle's bit 2, so the two
            // halves of the warp store to disjoint banks
            const bool odd = (lane & 1) != 0;
            unsigned char *oh = reinterpret_cast<unsigned char *>(OS) + (v >> 6) * kRawHalf +
                                (v & 6) * 2;
            const int vp = (v & 63) >> 3;
#pragma unroll
            for (int j8 = 0; j8 < 32; j8 += 8)
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const int j = j8 + jj;
                const float a = scale * d4[j], b = scale * d4[j + 4];
                const float x = __shfl_xor_sync(0xffffffffu, odd ? a : b, 1);
                const int t = i0 + j + (odd ? 4 : 0);
                *reinterpret_cast<__nv_bfloat162 *>(oh + t * 128 + ((vp ^ (t & 7)) << 4)) =
                    odd ? __floats2bfloat162_rn(x, b) : __floats2bfloat162_rn(a, x);
              }
            tc::fence_async_smem();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) OS[(i0 + j) * kOSRow + v] = scale * d4[j];
          }
          cw_sync();
          if (OB16 && o_map != 0 && n == C) {  // a whole chunk: two tensor-map stores
            if (tid == kCopier) {
              tma3_store(&maps.o, 0, h, (int)(lo + c0), OS);
              tma3_store(&maps.o, 64, h, (int)(lo + c0),
                         reinterpret_cast<unsigned char *>(OS) + kRawHalf);
              bulk_commit();
            }
          } else {
            constexpr int VEC = 16 / (int)sizeof(TO), PIECES = D / VEC;  // per token row
            TO *ob = o + (lo + c0) * ostep + (int64_t)h * D;
            for (int e = tid; e < n * PIECES; e += NT) {
              const int t = e / PIECES, pc = e % PIECES;
              const unsigned char *src =
                  OB16 ? reinterpret_cast<const unsigned char *>(OS) + (pc >> 3) * kRawHalf +
                             t * 128 + (((pc & 7) ^ (t & 7)) << 4)
                       : reinterpret_cast<const unsigned char *>(OS + t * kOSRow + pc * VEC);
              *reinterpret_cast<uint4 *>(ob + t * ostep + pc * VEC) =
                  *reinterpret_cast<const uint4 *>(src);
            }
          }
        } else {
          TO *ob = o + (lo + c0 + i0) * ostep + (int64_t)h * D + v;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (i0 + j < n) Elem<TO>::store1(ob + (int64_t)j * ostep, scale * d4[j]);
        }
      }
    };

    // chunk 0's rows and scalars (fetched by the MMA warp) landed: the split
    // and scaled state to the MMA warp
    alive = cw_and(rows_landed(0));
    if (alive) split_scale(scal(0)[kSGam + C - 1]);

    // Per chunk c: [D3 | E] -> F -> (MMA warp: Delta) while Ktil^T is built ->
    // (MMA warp: state update, then the next row copies) -> split and scale the
    // new state (the next [D3 | E] starts) -> this chunk's outputs under it.
    for (int c = 0; c < nch && alive; ++c) {
      const int c0 = c * C;
      const uint32_t par = c & 1;
      const int n = min(C, len - c0);
      const bool last = c + 1 == nch;
      alive = cw_and(wait_live(&b_ed3, par, vdead) &&    // [D3 | E] done, v landed
                     wait_live(&vbar, par, vdead));
      if (!alive) break;
      tc::fence_after_sync();

      const int i0 = 32 * half;
      if (n == C) f_pass(std::true_type(), n, i0, u_d4(c), scal(c));
      else f_pass(std::false_type(), n, i0, u_d4(c), scal(c));
      warp_arrive(&f_rdy);
      build_kt(c);  // the previous update has read the last Ktil^T
      warp_arrive(&g_rdy);

      // D4 and the new state ready; the next chunk's scalars landed
      alive = cw_and(alive && wait_live(&b_upd, par, vdead) && (last || rows_landed(c + 1)));
      if (!alive) break;
      tc::fence_after_sync();
      if (ck.every > 0 && c0 + C <= len && (c0 + C) % ck.every == 0) {  // checkpoint: copy S out
        const int j = (c0 + C) / ck.every - 1;
        const int ds = j < ck.per_seq ? ck.slots[(int64_t)si * ck.per_seq + j] : -1;
        if (ds >= p.n_slots) {
          if (tid == 0) raise_error(p.err, GDN_DEVERR_SLOT);
        } else if (ds >= 0) {
          char *dst = p.state_at(p.state_head_elem(layer, ds, h));
          const int64_t e0 = (int64_t)row * D + 64 * half;
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {
            float v[16];
            tc::tmem_ld16(lrow + U_S + 64 * half + 16 * cb, v);
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4)
              state_st4<false>(dst, e0 + (cb * 4 + j4) * 4,
                               make_float4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]),
                               sd);
          }
        }
      }
      if (!last) {
        split_scale(scal(c + 1)[kSGam + C - 1]);  // the next [D3 | E] starts here
        out_chunk(c);              // under it (the next update writes the other D4)
      }
    }

    if (alive) out_chunk(nch - 1);
    if (tid == kCopier) bulk_wait_all();  // output stores complete before the block exits
    if (alive) {
      const int64_t e0 = (int64_t)row * D + 64 * half;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float v[16];
        tc::tmem_ld16(lrow + U_S + 64 * half + c * 16, v);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          state_st4<false>(Sg, e0 + (c * 4 + j) * 4,
                           make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]), sd);
      }
    } else {
      *vdead = 1;
      if (tid == 0) raise_error(p.err, GDN_DEVERR_TIMEOUT);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tm, SEQ_TMEM);
}

// Tensor maps for the bf16 inputs of a call: q, k {128, h_k, tokens} and v
// {128, h_v, tokens} with boxes {64, 1, 64} in the 128-byte swizzle (rows and
// strides 16-byte aligned).  False: stage from global memory.
// With o_bf16 (a bf16 output tensor [tokens][h_v][128]) also its map, boxes
// {64, 1, 64} in the 128-byte swizzle, when it starts 16-byte aligned (om).
bool encode_in_maps(const PoolView &p, const SeqIndex &seq, const QKV &in, InMaps &m,
                    const void *o_bf16, bool &om) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      fn = nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  om = false;
  if (encode == nullptr) return false;
  const size_t es = 2;
  auto a16 = [](const void *x) { return (uintptr_t)x % 16 == 0; };
  if (!a16(in.q) || !a16(in.k) || !a16(in.v) || (in.ld_qk * es) % 16 || (in.ld_v * es) % 16)
    return false;
  const cuuint64_t tokens = (cuuint64_t)seq.total_tokens;
  cuuint32_t box[3] = {64, 1, C}, elem[3] = {1, 1, 1};
  auto map3 = [&](CUtensorMap *dst, const void *base, int heads, int64_t ld) {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, tokens};
    cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)ld * es};
    return encode(dst, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                  strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
  };
  if (!map3(&m.q, in.q, p.h_k, in.ld_qk) || !map3(&m.k, in.k, p.h_k, in.ld_qk) ||
      !map3(&m.v, in.v, p.h_v, in.ld_v))
    return false;
  if (o_bf16 != nullptr && a16(o_bf16))
    om = map3(&m.o, o_bf16, p.h_v, (int64_t)p.h_v * D);
  return true;
}

// SMs of the current device (queried once per device)
int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 1;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

template <typename TI, typename TO>
cudaError_t launch_t(const PoolView &p, int layer, const SeqIndex &seq, const QKV &in, void *o,
                     float scale, void *work, cudaStream_t s, const Checkpoints &ck) {
  int32_t *off = static_cast<int32_t *>(work);
  const int64_t nc = max_chunks(seq.n_seqs, seq.total_tokens);
  const int2 *table =
      reinterpret_cast<const int2 *>(static_cast<char *>(work) + chunk_table_offset(seq.n_seqs));
  float *tiles =
      reinterpret_cast<float *>(static_cast<char *>(work) + offsets_bytes(seq.n_seqs, nc));
  chunk_offsets_kernel<<<1, 1024, 0, s>>>(seq, off, nc);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  InMaps maps;
  bool om = false;
  const bool raw = std::is_same<TI, bf16>::value &&
                   encode_in_maps(p, seq, in, maps,
                                  std::is_same<TO, bf16>::value ? o : nullptr, om);
  auto prep = prep_kernel<TI>;
  constexpr int prep_bytes = prep_smem<TI>();
  e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, prep_bytes);
  if (e != cudaSuccess) return e;
  const int npair = (p.h_v / p.h_k + 1) / 2;
  // persistent: two CTAs per SM (or one per item when there are fewer)
  const int64_t items = nc * p.h_k * npair;
  const int64_t grid = items < 2 * (int64_t)sm_count() ? items : 2 * (int64_t)sm_count();
  prep<<<(unsigned)grid, NT, prep_bytes, s>>>(p, seq, in, off, table, tiles, nc, maps,
                                               raw ? 1 : 0);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (raw) {  // bf16 rows by tensor map: [D3 | E] on kind::f16 over the raw rows
    auto kern = seq_bf16_kernel<TO>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSeqBf16Smem);
    if (e != cudaSuccess) return e;
    // a programmatic dependent of the key-side kernel: its prologue (state
    // load, first row copies) overlaps that kernel's tail
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.h_v, seq.n_seqs);
    cfg.blockDim = dim3(NTS);
    cfg.dynamicSmemBytes = kSeqBf16Smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, layer, seq, in, static_cast<TO *>(o), scale,
                              static_cast<const int32_t *>(off), nc,
                              static_cast<const float *>(tiles), maps, om ? 1 : 0, ck);
  }
  auto kern = seq_kernel<TI, TO>;  // rows staged from global memory
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSeqSmem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(p.h_v, seq.n_seqs), NTS, kSeqSmem, s>>>(p, layer, seq, in, static_cast<TO *>(o),
                                                         scale, off, nc, tiles, ck);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_split_workspace_bytes(int n_seqs, int total_tokens, int h_v) {
  const int64_t nc = max_chunks(n_seqs, total_tokens);
  return offsets_bytes(n_seqs, nc) + (size_t)nc * h_v * (2 * kTileBytes + kScal * 4);
}

cudaError_t launch_prefill_split(const PoolView &p, int layer, const SeqIndex &seq,
                                 const QKV &in, void *o, gdn_dtype o_dtype, float scale,
                                 void *work, cudaStream_t s, const Checkpoints &ck) {
  if (p.dk != D || p.dv != D) return cudaErrorNotSupported;
  if (in.dtype == GDN_F32 && o_dtype == GDN_F32)
    return launch_t<float, float>(p, layer, seq, in, o, scale, work, s, ck);
  if (in.dtype == GDN_F32 && o_dtype == GDN_BF16)
    return launch_t<float, bf16>(p, layer, seq, in, o, scale, work, s, ck);
  if (in.dtype == GDN_BF16 && o_dtype == GDN_F32)
    return launch_t<bf16, float>(p, layer, seq, in, o, scale, work, s, ck);
  return launch_t<bf16, bf16>(p, layer, seq, in, o, scale, work, s, ck);
}

}  // namespace gdn
