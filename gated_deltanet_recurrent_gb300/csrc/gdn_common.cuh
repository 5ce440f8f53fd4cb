// Device helpers shared by the libgdn kernels: typed loads/stores of float32
// and bf16 inputs, group reductions over warp lanes, the error word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_internal.h"

namespace gdn {

typedef __nv_bfloat16 bf16;

template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static __device__ __forceinline__ float4 load4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
  }
  static __device__ __forceinline__ float load1(const float *p) { return *p; }
  static __device__ __forceinline__ void store1(float *p, float x) { *p = x; }
  static __device__ __forceinline__ float from_bits(float x) { return x; }
};

template <>
struct Elem<bf16> {
  // four consecutive bf16 values (8-byte aligned) widened to float32
  static __device__ __forceinline__ float4 load4(const bf16 *p) {
    const uint2 raw = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                       __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u));
  }
  static __device__ __forceinline__ float load1(const bf16 *p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ void store1(bf16 *p, float x) { *p = __float2bfloat16_rn(x); }
};

// ---- state storage: float32, or bf16 / f16 elements converted to and from
// float32 registers (round to nearest even on every store) ----

// four consecutive state elements starting at element e (a multiple of 4) of
// `base` (global or shared memory)
__device__ __forceinline__ float4 state_ld4(const void *base, int64_t e, gdn_dtype sd) {
  if (sd == GDN_F32) return reinterpret_cast<const float4 *>(base)[e / 4];
  const uint2 r = reinterpret_cast<const uint2 *>(base)[e / 4];
  if (sd == GDN_BF16)
    return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u),
                       __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xffff0000u));
  const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// store four state elements at element e; STREAM: evict-first global store
template <bool STREAM>
__device__ __forceinline__ void state_st4(void *base, int64_t e, float4 v, gdn_dtype sd) {
  if (sd == GDN_F32) {
    float4 *p = reinterpret_cast<float4 *>(base) + e / 4;
    if (STREAM) __stcs(p, v); else *p = v;
    return;
  }
  uint2 r;
  if (sd == GDN_BF16) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    r.x = *reinterpret_cast<const unsigned *>(&a);
    r.y = *reinterpret_cast<const unsigned *>(&b);
  } else {
    const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    r.x = *reinterpret_cast<const unsigned *>(&a);
    r.y = *reinterpret_cast<const unsigned *>(&b);
  }
  uint2 *p = reinterpret_cast<uint2 *>(base) + e / 4;
  if (STREAM) __stcs(p, r); else *p = r;
}

__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
  return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

__device__ __forceinline__ float4 axpby4(float a, const float4 x, float b, const float4 y) {
  return make_float4(a * x.x + b * y.x, a * x.y + b * y.y, a * x.z + b * y.z, a * x.w + b * y.w);
}

__device__ __forceinline__ float4 scale4(float a, const float4 x) {
  return make_float4(a * x.x, a * x.y, a * x.z, a * x.w);
}

// Sum over aligned groups of LANES consecutive lanes; every lane of the group
// receives the total.  All 32 lanes must call it.
template <int LANES>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int off = LANES / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

__device__ __forceinline__ void raise_error(unsigned int *err, unsigned int bit) {
  atomicOr(err, bit);
}

__device__ __forceinline__ float silu(float u) { return u / (1.0f + expf(-u)); }


// ---- bulk-copy (TMA engine) and mbarrier helpers, sm_90+ PTX ----

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// make the initialised barrier visible to the async (bulk-copy) proxy
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

// global -> shared bulk copy of `bytes` (multiple of 16, both ends 16-byte
// aligned), completing on `bar` as transaction bytes
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase: gives up after `limit` polls (each poll
// may itself suspend the thread for a while) and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint32_t limit = (1u << 20)) {
  for (uint32_t it = 0; it < limit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

}  // namespace gdn
