// Shared pieces of the row-streaming kernels (decode and verify): CTA size,
// state addressing, the bulk tile size and the (dk, dtype) dispatch.
#pragma once

#include "gdn_common.cuh"

namespace gdn {
namespace rows {

constexpr int kThreads = 128;    // 4 warps per CTA
constexpr int kBulkBytes = 16384;  // state tile per CTA (one bulk copy)

__device__ __forceinline__ float *state_head(const PoolView &p, int layer, int slot, int h) {
  return p.state + ((int64_t)layer * p.n_slots + slot) * p.state_slot_elems() +
         (int64_t)h * p.dv * p.dk;
}

// Dispatch over (dk, input dtype, output dtype) to F<DK, TI, TO>::run.
template <template <int, typename, typename> class F, typename... Args>
cudaError_t dispatch(int dk, gdn_dtype ti, gdn_dtype to, Args... args) {
#define GDN_DT(DK, TI, TO) return F<DK, TI, TO>::run(args...)
#define GDN_DK(DK)                                                     \
  if (dk == DK) {                                                      \
    if (ti == GDN_F32 && to == GDN_F32) GDN_DT(DK, float, float);      \
    if (ti == GDN_F32 && to == GDN_BF16) GDN_DT(DK, float, bf16);      \
    if (ti == GDN_BF16 && to == GDN_F32) GDN_DT(DK, bf16, float);      \
    if (ti == GDN_BF16 && to == GDN_BF16) GDN_DT(DK, bf16, bf16);      \
  }
  GDN_DK(16)
  GDN_DK(32)
  GDN_DK(64)
  GDN_DK(128)
#undef GDN_DK
#undef GDN_DT
  return cudaErrorInvalidValue;
}

}  // namespace rows
}  // namespace gdn
