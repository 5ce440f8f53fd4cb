// Output gated RMSNorm of a GDN layer: for each row r (one token, one value
// head) of the recurrence output o [rows][d],
//     y[r][j] = o[r][j] * rsqrt(mean_j o[r][j]^2 + eps) * w[j] * silu(z[r][j]).
//
// HBM-bound: o and z are read once and y written once.  One warp per row,
// grid-stride over rows, the sum of squares reduced with warp shuffles.
// Rows of d = 128 * C elements (C = 1, 2, 4, 8) with aligned rows take the
// vector kernel: lane l holds elements 128 c + 4 l .. + 3 of o and z in
// registers, fetched as 16- or 8-byte vectors before the reduction (two rows
// per warp at C <= 2, to keep more bytes in flight), and writes y as one
// vector per piece.  Other shapes take the scalar kernel, whose lanes walk
// the row element by element and re-read o from L1 in a second pass.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int kNormThreads = 256;

template <typename TO, typename TZ, typename TY>
__global__ void __launch_bounds__(kNormThreads)
    gated_rmsnorm_kernel(const TO *__restrict__ o, const TZ *__restrict__ z,
                         const float *__restrict__ w, float eps, TY *__restrict__ y,
                         int64_t rows, int d) {
  const int lane = threadIdx.x & 31;
  const int64_t first = ((int64_t)blockIdx.x * kNormThreads + threadIdx.x) >> 5;
  const int64_t stride = ((int64_t)gridDim.x * kNormThreads) >> 5;
  const float inv_d = 1.0f / (float)d;
  for (int64_t r = first; r < rows; r += stride) {
    const TO *orow = o + r * d;
    float ss = 0.f;
    for (int j = lane; j < d; j += 32) {
      const float v = Elem<TO>::load1(orow + j);
      ss += v * v;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = rsqrtf(ss * inv_d + eps);
    const TZ *zrow = z + r * d;
    TY *yrow = y + r * d;
    for (int j = lane; j < d; j += 32)
      Elem<TY>::store1(yrow + j,
                       Elem<TO>::load1(orow + j) * inv * w[j] * silu(Elem<TZ>::load1(zrow + j)));
  }
}

__device__ __forceinline__ void store4(float *p, float4 v) {
  *reinterpret_cast<float4 *>(p) = v;
}

__device__ __forceinline__ void store4(bf16 *p, float4 v) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<const unsigned *>(&lo);
  u.y = *reinterpret_cast<const unsigned *>(&hi);
  *reinterpret_cast<uint2 *>(p) = u;
}

template <typename TO, typename TZ, typename TY, int C, int RPW>
__global__ void __launch_bounds__(kNormThreads)
    gated_rmsnorm_vec_kernel(const TO *__restrict__ o, const TZ *__restrict__ z,
                             const float *__restrict__ w, float eps, TY *__restrict__ y,
                             int64_t rows) {
  constexpr int D = 128 * C;
  const int lane = threadIdx.x & 31;
  const int64_t first = ((int64_t)blockIdx.x * kNormThreads + threadIdx.x) >> 5;
  const int64_t stride = ((int64_t)gridDim.x * kNormThreads) >> 5;
  for (int64_t r0 = first * RPW; r0 < rows; r0 += stride * RPW) {
    float4 ov[RPW][C], zv[RPW][C];
#pragma unroll
    for (int q = 0; q < RPW; ++q) {
      const int64_t r = r0 + q;  // the same for every lane of the warp
#pragma unroll
      for (int c = 0; c < C; ++c) {
        if (r < rows) {
          ov[q][c] = Elem<TO>::load4(o + r * D + 128 * c + 4 * lane);
          zv[q][c] = Elem<TZ>::load4(z + r * D + 128 * c + 4 * lane);
        } else {
          ov[q][c] = zv[q][c] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < RPW; ++q) {
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < C; ++c) ss += dot4(ov[q][c], ov[q][c]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float inv = rsqrtf(ss * (1.0f / (float)D) + eps);
      const int64_t r = r0 + q;
      if (r < rows) {
#pragma unroll
        for (int c = 0; c < C; ++c) {
          const float4 wv = *reinterpret_cast<const float4 *>(w + 128 * c + 4 * lane);
          const float4 a = ov[q][c], g = zv[q][c];
          store4(y + r * D + 128 * c + 4 * lane,
                 make_float4(a.x * inv * wv.x * silu(g.x), a.y * inv * wv.y * silu(g.y),
                             a.z * inv * wv.z * silu(g.z), a.w * inv * wv.w * silu(g.w)));
        }
      }
    }
  }
}

template <typename TO, typename TZ, typename TY, int C, int RPW>
cudaError_t launch_vec(const void *o, const void *z, const float *w, float eps, void *y,
                       int64_t rows, cudaStream_t s) {
  const int64_t warps = (rows + RPW - 1) / RPW;
  int64_t blocks = (warps + kNormThreads / 32 - 1) / (kNormThreads / 32);
  const int64_t cap = 152 * 8;  // one wave of 8 resident blocks per SM, then grid-stride
  if (blocks > cap) blocks = cap;
  gated_rmsnorm_vec_kernel<TO, TZ, TY, C, RPW><<<(unsigned)blocks, kNormThreads, 0, s>>>(
      static_cast<const TO *>(o), static_cast<const TZ *>(z), w, eps, static_cast<TY *>(y),
      rows);
  return cudaGetLastError();
}

bool aligned(const void *p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

template <typename TO, typename TZ, typename TY>
cudaError_t launch_t(const void *o, const void *z, const float *w, float eps, void *y,
                     int64_t rows, int d, cudaStream_t s) {
  // vector path: whole 16-byte (float32) / 8-byte (bf16) pieces of aligned rows
  if (d % 128 == 0 && aligned(o, 4 * sizeof(TO)) && aligned(z, 4 * sizeof(TZ)) &&
      aligned(y, 4 * sizeof(TY)) && aligned(w, 16)) {
    switch (d / 128) {
      case 1: return launch_vec<TO, TZ, TY, 1, 2>(o, z, w, eps, y, rows, s);
      case 2: return launch_vec<TO, TZ, TY, 2, 2>(o, z, w, eps, y, rows, s);
      case 4: return launch_vec<TO, TZ, TY, 4, 1>(o, z, w, eps, y, rows, s);
      case 8: return launch_vec<TO, TZ, TY, 8, 1>(o, z, w, eps, y, rows, s);
      default: break;
    }
  }
  const int64_t warps_per_block = kNormThreads / 32;
  int64_t blocks = (rows + warps_per_block - 1) / warps_per_block;
  const int64_t cap = 152 * 16;  // grid-stride beyond 16 resident blocks per SM
  if (blocks > cap) blocks = cap;
  gated_rmsnorm_kernel<TO, TZ, TY><<<(unsigned)blocks, kNormThreads, 0, s>>>(
      static_cast<const TO *>(o), static_cast<const TZ *>(z), w, eps, static_cast<TY *>(y),
      rows, d);
  return cudaGetLastError();
}

template <typename TO, typename TZ>
cudaError_t by_out(gdn_dtype yt, const void *o, const void *z, const float *w, float eps,
                   void *y, int64_t rows, int d, cudaStream_t s) {
  return yt == GDN_F32 ? launch_t<TO, TZ, float>(o, z, w, eps, y, rows, d, s)
                       : launch_t<TO, TZ, bf16>(o, z, w, eps, y, rows, d, s);
}

template <typename TO>
cudaError_t by_gate(gdn_dtype zt, gdn_dtype yt, const void *o, const void *z, const float *w,
                    float eps, void *y, int64_t rows, int d, cudaStream_t s) {
  return zt == GDN_F32 ? by_out<TO, float>(yt, o, z, w, eps, y, rows, d, s)
                       : by_out<TO, bf16>(yt, o, z, w, eps, y, rows, d, s);
}

}  // namespace

cudaError_t launch_gated_rmsnorm(const void *o, gdn_dtype ot, const void *z, gdn_dtype zt,
                                 const float *w, float eps, void *y, gdn_dtype yt, int64_t rows,
                                 int d, cudaStream_t s) {
  return ot == GDN_F32 ? by_gate<float>(zt, yt, o, z, w, eps, y, rows, d, s)
                       : by_gate<bf16>(zt, yt, o, z, w, eps, y, rows, d, s);
}

}  // namespace gdn
