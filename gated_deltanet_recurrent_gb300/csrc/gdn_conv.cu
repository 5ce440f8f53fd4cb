// Causal depthwise short conv + SiLU on the slot conv caches, and the pool
// reset (zeroing of listed slots).
//
// Conv: thread = one channel of one sequence, walking a block of kTokBlock
// consecutive tokens with the conv_k - 1 previous raw inputs in registers.
// Token blocks of one sequence run in parallel; only block 0 reads the old
// cache (kTokBlock >= conv_k - 1), and the same thread writes the new cache
// after it has read the old one, so one launch updates caches in place.
// Each conv CTA first allows a programmatic dependent launch that follows it
// (the decode of the same step) to start; such a dependent waits for the conv
// grid to complete before it reads anything the conv writes.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kConvThreads = 128;
constexpr int kTokBlock = 16;
constexpr int kMaxGridY = 2048;

template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads)
    conv_silu_kernel(PoolView p, int layer, SeqIndex seq, const T *__restrict__ x, int64_t ld_x,
                     const float *__restrict__ w, const float *__restrict__ bias,
                     T *__restrict__ y, int64_t ld_y, const int32_t *__restrict__ advance) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int c = blockIdx.x * kConvThreads + threadIdx.x;
  const int i = blockIdx.z;
  const int slot = seq.slot_ids[i];
  const bool first = blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0;
  if (slot < 0 || slot >= p.n_slots) {
    if (first) raise_error(p.err, GDN_DEVERR_SLOT);
    return;
  }
  int64_t lo = i;
  int len = 1;
  if (seq.cu_seqlens != nullptr) {
    lo = seq.cu_seqlens[i];
    const int64_t hi = seq.cu_seqlens[i + 1];
    if (hi < lo || lo < 0 || hi > seq.total_tokens) {
      if (first) raise_error(p.err, GDN_DEVERR_SEQ);
      return;
    }
    len = (int)(hi - lo);
  }
  if (c >= p.conv_ch) return;
  int a = advance ? advance[i] : len;
  if (a < 0 || a > len) {
    if (first) raise_error(p.err, GDN_DEVERR_COUNT);
    a = a < 0 ? 0 : len;
  }
  T *cache = static_cast<T *>(p.conv) +
             (((int64_t)layer * p.n_slots + slot) * p.conv_ch + c) * (W - 1);
  float wr[W];
#pragma unroll
  for (int j = 0; j < W; ++j) wr[j] = w[(int64_t)c * W + j];
  const float b = bias ? bias[c] : 0.f;
  const T *xc = x + lo * ld_x + c;

  for (int blk = blockIdx.y; blk * kTokBlock < len; blk += gridDim.y) {
    const int t0 = blk * kTokBlock;
    float old[W - 1];  // the old cache (block 0 only)
    float hst[W - 1];  // raw inputs at times t0-(W-1) .. t0-1
#pragma unroll
    for (int j = 0; j < W - 1; ++j) {
      const int tt = t0 - (W - 1) + j;
      old[j] = blk == 0 ? Elem<T>::load1(cache + j) : 0.f;
      hst[j] = tt < 0 ? Elem<T>::load1(cache + (W - 1) + tt) : Elem<T>::load1(xc + tt * ld_x);
    }
    const int t1 = min(t0 + kTokBlock, len);
    for (int t = t0; t < t1; ++t) {
      const float xt = Elem<T>::load1(xc + (int64_t)t * ld_x);
      float u = b + wr[W - 1] * xt;
#pragma unroll
      for (int j = 0; j < W - 1; ++j) u += wr[j] * hst[j];
      if (y != nullptr) Elem<T>::store1(y + (lo + t) * ld_y + c, silu(u));
#pragma unroll
      for (int j = 0; j < W - 2; ++j) hst[j] = hst[j + 1];
      hst[W - 2] = xt;
    }
    if (blk == 0) {
      // new cache = raw inputs at times a-(W-1) .. a-1 (old cache below 0)
#pragma unroll
      for (int j = 0; j < W - 1; ++j) {
        const int tt = a - (W - 1) + j;
        float val = 0.f;
        if (tt < 0) {
#pragma unroll
          for (int m = 0; m < W - 1; ++m)  // old[(W - 1) + tt] without a dynamic index
            if (m == (W - 1) + tt) val = old[m];
        } else {
          val = Elem<T>::load1(xc + (int64_t)tt * ld_x);
        }
        Elem<T>::store1(cache + j, val);
      }
    }
  }
}

// 16-byte vector access: VEC consecutive channels per thread.
template <typename T>
struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
  static __device__ __forceinline__ void unpack(const uint4 r, float *f);
  static __device__ __forceinline__ uint4 pack(const float *f);
};
template <>
__device__ __forceinline__ void Vec16<float>::unpack(const uint4 r, float *f) {
  f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
  f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
}
template <>
__device__ __forceinline__ uint4 Vec16<float>::pack(const float *f) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}
template <>
__device__ __forceinline__ void Vec16<bf16>::unpack(const uint4 r, float *f) {
  const unsigned w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
}
template <>
__device__ __forceinline__ uint4 Vec16<bf16>::pack(const float *f) {
  unsigned w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
    w[j] = *reinterpret_cast<const unsigned *>(&b2);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Same contract as conv_silu_kernel; each thread owns VEC = 16/sizeof(T)
// consecutive channels, so x, y, the cache ((W-1) x 16 bytes per thread) and
// the taps move in 16-byte accesses.  Needs conv_ch % VEC == 0 and 16-byte
// aligned rows of x and y (checked by the launcher).
template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads)
    conv_silu_vec_kernel(PoolView p, int layer, SeqIndex seq, const T *__restrict__ x,
                         int64_t ld_x, const float *__restrict__ w,
                         const float *__restrict__ bias, T *__restrict__ y, int64_t ld_y,
                         const int32_t *__restrict__ advance) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int V = Vec16<T>::N;
  const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * V;
  const int i = blockIdx.z;
  const int slot = seq.slot_ids[i];
  const bool first = blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0;
  if (slot < 0 || slot >= p.n_slots) {
    if (first) raise_error(p.err, GDN_DEVERR_SLOT);
    return;
  }
  int64_t lo = i;
  int len = 1;
  if (seq.cu_seqlens != nullptr) {
    lo = seq.cu_seqlens[i];
    const int64_t hi = seq.cu_seqlens[i + 1];
    if (hi < lo || lo < 0 || hi > seq.total_tokens) {
      if (first) raise_error(p.err, GDN_DEVERR_SEQ);
      return;
    }
    len = (int)(hi - lo);
  }
  if (c0 >= p.conv_ch) return;
  int a = advance ? advance[i] : len;
  if (a < 0 || a > len) {
    if (first) raise_error(p.err, GDN_DEVERR_COUNT);
    a = a < 0 ? 0 : len;
  }
  // this thread's cache: V channels x (W-1) taps, channel-major, (W-1) x 16 bytes
  uint4 *cache = reinterpret_cast<uint4 *>(
      static_cast<T *>(p.conv) + (((int64_t)layer * p.n_slots + slot) * p.conv_ch + c0) * (W - 1));
  float wr[V][W];
#pragma unroll
  for (int j = 0; j < V; ++j)
#pragma unroll
    for (int m = 0; m < W; m += 4) {
      if (W % 4 == 0) {
        const float4 w4 = *reinterpret_cast<const float4 *>(w + (int64_t)(c0 + j) * W + m);
        wr[j][m] = w4.x; wr[j][m + 1] = w4.y; wr[j][m + 2] = w4.z; wr[j][m + 3] = w4.w;
      } else {
#pragma unroll
        for (int mm = m; mm < m + 4 && mm < W; ++mm) wr[j][mm] = w[(int64_t)(c0 + j) * W + mm];
      }
    }
  float b[V];
#pragma unroll
  for (int j = 0; j < V; ++j) b[j] = bias ? bias[c0 + j] : 0.f;
  const T *xc = x + lo * ld_x + c0;

  for (int blk = blockIdx.y; blk * kTokBlock < len; blk += gridDim.y) {
    const int t0 = blk * kTokBlock;
    float old[V][W - 1];
    float hst[V][W - 1];
    if (blk == 0) {
      float flat[V * (W - 1)];
#pragma unroll
      for (int q = 0; q < W - 1; ++q) Vec16<T>::unpack(cache[q], flat + q * V);
#pragma unroll
      for (int j = 0; j < V; ++j)
#pragma unroll
        for (int m = 0; m < W - 1; ++m) old[j][m] = flat[j * (W - 1) + m];
    }
    // block 0 starts at t0 = 0, so its history is exactly the old cache;
    // later blocks start at t0 >= kTokBlock >= W - 1 and read x only
#pragma unroll
    for (int m = 0; m < W - 1; ++m) {
      if (blk == 0) {
#pragma unroll
        for (int j = 0; j < V; ++j) hst[j][m] = old[j][m];
      } else {
        float f[V];
        Vec16<T>::unpack(
            *reinterpret_cast<const uint4 *>(xc + (int64_t)(t0 - (W - 1) + m) * ld_x), f);
#pragma unroll
        for (int j = 0; j < V; ++j) hst[j][m] = f[j];
      }
    }
    const int t1 = min(t0 + kTokBlock, len);
    for (int t = t0; t < t1; ++t) {
      float xt[V], out[V];
      Vec16<T>::unpack(*reinterpret_cast<const uint4 *>(xc + (int64_t)t * ld_x), xt);
#pragma unroll
      for (int j = 0; j < V; ++j) {
        float u = b[j] + wr[j][W - 1] * xt[j];
#pragma unroll
        for (int m = 0; m < W - 1; ++m) u += wr[j][m] * hst[j][m];
        out[j] = silu(u);
#pragma unroll
        for (int m = 0; m < W - 2; ++m) hst[j][m] = hst[j][m + 1];
        hst[j][W - 2] = xt[j];
      }
      if (y != nullptr)
        *reinterpret_cast<uint4 *>(y + (lo + t) * ld_y + c0) = Vec16<T>::pack(out);
    }
    if (blk == 0) {
      // new cache = raw inputs at times a-(W-1) .. a-1 (old cache below 0)
      float flat[V * (W - 1)];
#pragma unroll
      for (int m = 0; m < W - 1; ++m) {
        const int tt = a - (W - 1) + m;
        float f[V];
        if (tt < 0) {
#pragma unroll
          for (int j = 0; j < V; ++j) {
            f[j] = 0.f;
#pragma unroll
            for (int mm = 0; mm < W - 1; ++mm)
              if (mm == (W - 1) + tt) f[j] = old[j][mm];
          }
        } else {
          Vec16<T>::unpack(*reinterpret_cast<const uint4 *>(xc + (int64_t)tt * ld_x), f);
        }
#pragma unroll
        for (int j = 0; j < V; ++j) flat[j * (W - 1) + m] = f[j];
      }
#pragma unroll
      for (int q = 0; q < W - 1; ++q) cache[q] = Vec16<T>::pack(flat + q * V);
    }
  }
}

template <typename T>
__device__ __forceinline__ void zero_elems(T *base, int64_t n, int64_t start, int64_t stride) {
  for (int64_t e = start; e < n; e += stride) base[e] = T(0.f);
}

// grid (blocks, n_layers, n); zero state and conv cache of each listed slot.
__global__ void reset_kernel(PoolView p, const int32_t *__restrict__ slot_ids) {
  const int i = blockIdx.z;
  const int layer = blockIdx.y;
  const int slot = slot_ids[i];
  if (slot < 0 || slot >= p.n_slots) {
    if (blockIdx.x == 0 && layer == 0 && threadIdx.x == 0) raise_error(p.err, GDN_DEVERR_SLOT);
    return;
  }
  const int64_t start = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  // the slot's state as 16-byte words (dk * element size is a multiple of 16)
  uint4 *st = reinterpret_cast<uint4 *>(p.state_at(p.state_head_elem(layer, slot, 0)));
  const int64_t n16 = p.state_slot_elems() * p.state_esz() / 16;
  for (int64_t e = start; e < n16; e += stride) st[e] = make_uint4(0u, 0u, 0u, 0u);
  const int64_t nc = p.conv_slot_elems();
  const int64_t coff = ((int64_t)layer * p.n_slots + slot) * nc;
  if (p.conv_dtype == GDN_F32)
    zero_elems(static_cast<float *>(p.conv) + coff, nc, start, stride);
  else
    zero_elems(static_cast<bf16 *>(p.conv) + coff, nc, start, stride);
}

// grid (blocks, n_layers, n); copy state and conv cache of src[i] to dst[i].
__global__ void copy_kernel(PoolView p, const int32_t *__restrict__ src,
                            const int32_t *__restrict__ dst) {
  const int i = blockIdx.z;
  const int layer = blockIdx.y;
  const int a = src[i], b = dst[i];
  if (a < 0 || a >= p.n_slots || b < 0 || b >= p.n_slots) {
    if (blockIdx.x == 0 && layer == 0 && threadIdx.x == 0) raise_error(p.err, GDN_DEVERR_SLOT);
    return;
  }
  const int64_t start = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t n16 = p.state_slot_elems() * p.state_esz() / 16;
  const uint4 *sa = reinterpret_cast<const uint4 *>(p.state_at(p.state_head_elem(layer, a, 0)));
  uint4 *sb = reinterpret_cast<uint4 *>(p.state_at(p.state_head_elem(layer, b, 0)));
  for (int64_t e = start; e < n16; e += stride) sb[e] = sa[e];
  const int64_t nc = p.conv_slot_elems();
  if (p.conv_dtype == GDN_F32) {
    const float *ca = static_cast<const float *>(p.conv) + ((int64_t)layer * p.n_slots + a) * nc;
    float *cb = static_cast<float *>(p.conv) + ((int64_t)layer * p.n_slots + b) * nc;
    for (int64_t e = start; e < nc; e += stride) cb[e] = ca[e];
  } else {
    const bf16 *ca = static_cast<const bf16 *>(p.conv) + ((int64_t)layer * p.n_slots + a) * nc;
    bf16 *cb = static_cast<bf16 *>(p.conv) + ((int64_t)layer * p.n_slots + b) * nc;
    for (int64_t e = start; e < nc; e += stride) cb[e] = ca[e];
  }
}

template <typename T, int W>
cudaError_t launch_conv_t(const PoolView &p, int layer, const SeqIndex &seq, int max_seqlen,
                          const void *x, int64_t ld_x, const float *w, const float *bias,
                          void *y, int64_t ld_y, const int32_t *advance, cudaStream_t s) {
  const int blocks_y = seq.cu_seqlens == nullptr
                           ? 1
                           : min(kMaxGridY, max(1, (max_seqlen + kTokBlock - 1) / kTokBlock));
  constexpr int V = Vec16<T>::N;
  const bool vec_ok = p.conv_ch % V == 0 && (uintptr_t)x % 16 == 0 &&
                      (ld_x * sizeof(T)) % 16 == 0 && (uintptr_t)w % 16 == 0 &&
                      (y == nullptr || ((uintptr_t)y % 16 == 0 && (ld_y * sizeof(T)) % 16 == 0));
  if (vec_ok) {
    const int threads = p.conv_ch / V;
    dim3 grid((threads + kConvThreads - 1) / kConvThreads, blocks_y, seq.n_seqs);
    conv_silu_vec_kernel<T, W><<<grid, kConvThreads, 0, s>>>(
        p, layer, seq, static_cast<const T *>(x), ld_x, w, bias, static_cast<T *>(y), ld_y,
        advance);
  } else {
    dim3 grid((p.conv_ch + kConvThreads - 1) / kConvThreads, blocks_y, seq.n_seqs);
    conv_silu_kernel<T, W><<<grid, kConvThreads, 0, s>>>(
        p, layer, seq, static_cast<const T *>(x), ld_x, w, bias, static_cast<T *>(y), ld_y,
        advance);
  }
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_conv_w(const PoolView &p, int layer, const SeqIndex &seq, int max_seqlen,
                          const void *x, int64_t ld_x, const float *w, const float *bias,
                          void *y, int64_t ld_y, const int32_t *advance, cudaStream_t s) {
  switch (p.conv_k) {
#define GDN_W(W) \
  case W: return launch_conv_t<T, W>(p, layer, seq, max_seqlen, x, ld_x, w, bias, y, ld_y, advance, s);
    GDN_W(2) GDN_W(3) GDN_W(4) GDN_W(5) GDN_W(6) GDN_W(7) GDN_W(8)
#undef GDN_W
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_pool_copy(const PoolView &p, const int32_t *src, const int32_t *dst, int n,
                             cudaStream_t s) {
  const int64_t per_slot = p.state_slot_elems() / 4;
  const int threads = 256;
  int64_t blocks = (per_slot + threads * 8 - 1) / (threads * 8);
  blocks = blocks < 1 ? 1 : (blocks > 64 ? 64 : blocks);
  dim3 grid((unsigned)blocks, p.n_layers, n);
  copy_kernel<<<grid, threads, 0, s>>>(p, src, dst);
  return cudaGetLastError();
}

cudaError_t launch_conv_silu(const PoolView &p, int layer, const SeqIndex &seq, int max_seqlen,
                             const void *x, int64_t ld_x, const float *w, const float *bias,
                             void *y, int64_t ld_y, const int32_t *advance, cudaStream_t s) {
  if (p.conv_dtype == GDN_F32)
    return launch_conv_w<float>(p, layer, seq, max_seqlen, x, ld_x, w, bias, y, ld_y, advance, s);
  return launch_conv_w<bf16>(p, layer, seq, max_seqlen, x, ld_x, w, bias, y, ld_y, advance, s);
}

cudaError_t launch_pool_reset(const PoolView &p, const int32_t *slot_ids, int n,
                              cudaStream_t s) {
  const int64_t per_slot = p.state_slot_elems() / 4;
  const int threads = 256;
  int64_t blocks = (per_slot + threads * 8 - 1) / (threads * 8);
  blocks = blocks < 1 ? 1 : (blocks > 64 ? 64 : blocks);
  dim3 grid((unsigned)blocks, p.n_layers, n);
  reset_kernel<<<grid, threads, 0, s>>>(p, slot_ids);
  return cudaGetLastError();
}

}  // namespace gdn
