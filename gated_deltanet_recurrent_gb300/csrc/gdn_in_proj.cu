// Input projection of a GDN layer (baseRT issue #31, "Why this looks
// tractable": the gdn_in_proj kernel): y = x W^T for bf16 activations
// x [tokens][hidden] and bf16 weights W [n_out][hidden] (the layer's q | k | v
// conv inputs, the output gate and the per-head beta / decay logits, stacked
// along n_out), float32 accumulation, y in float32 or bf16.
//
// One CTA computes a 128 x BN tile of y on the 5th-generation tensor cores:
//   warp 0, one thread: TMA producer -- 128 x 64 tiles of x and BN x 64 tiles
//     of W (tensor maps, 128-byte swizzle) into a ring of STAGES stages, each
//     completing on its `full` mbarrier;
//   warp 1, one thread: MMA issuer -- per stage four tcgen05.mma kind::f16
//     (M 128, N BN, K 16) from the swizzled shared-memory tiles into a float32
//     accumulator in TMEM; tcgen05.commit frees the stage (`empty`) and, after
//     the last one, signals the epilogue (`done`); warp 1 also owns the TMEM
//     allocation;
//   warps 2..5: epilogue -- each reads its 32 TMEM lanes (rows) with
//     tcgen05.ld and stores them (16-byte stores, masked at the edges).
// Two CTAs fit one SM (shared memory and TMEM), so one CTA's epilogue overlaps
// the other's main loop (BN 128); for few tokens 96-column tiles with a
// 6-stage ring put one wave of CTAs on the GPU.  K tails are zero-filled by the tensor map; M and N
// tails are masked in the epilogue.  Every mbarrier wait is bounded: a wait
// that gives up sets GDN_DEVERR_TIMEOUT, the CTA skips its stores and waits
// (bounded) for its copies and MMAs in flight before it frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int kBM = 128, kBK = 64;
constexpr int kGemmThreads = 192;
constexpr int kTileA = kBM * kBK * 2;  // 16 KiB of x per stage

template <int BN>
struct GemmCfg {
  static constexpr int kTileB = BN * kBK * 2;
  static constexpr int kStage = kTileA + kTileB;
  // BN 128: two CTAs per SM; BN 96 (few tokens): one CTA per SM, a deep ring
  static constexpr int kStages = BN == 128 ? 3 : 6;
  static constexpr int kSmem = kStages * kStage + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = BN <= 64 ? 64 : (BN <= 128 ? 128 : 256);  // power of 2
};

__device__ __forceinline__ void tma_load2(void *dst, const CUtensorMap *m, int x, int y,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

template <typename TO>
__device__ __forceinline__ void store_row16(TO *dst, const float *v, int n_valid);

template <>
__device__ __forceinline__ void store_row16<float>(float *dst, const float *v, int n_valid) {
  if (n_valid >= 16) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      reinterpret_cast<float4 *>(dst)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2],
                                                       v[4 * j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < n_valid) dst[j] = v[j];
  }
}

template <>
__device__ __forceinline__ void store_row16<bf16>(bf16 *dst, const float *v, int n_valid) {
  if (n_valid >= 16) {
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
      w[j] = *reinterpret_cast<const uint32_t *>(&b2);
    }
    reinterpret_cast<uint4 *>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4 *>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < n_valid) dst[j] = __float2bfloat16_rn(v[j]);
  }
}

template <int BN, typename TO>
__global__ void __launch_bounds__(kGemmThreads, 2)
    in_proj_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mw,
                   int M, int N, int K, TO *__restrict__ y, int64_t ld_y,
                   unsigned int *__restrict__ err) {
  using Cfg = GemmCfg<BN>;
  constexpr int S = Cfg::kStages;
  extern __shared__ unsigned char dsm_raw[];
  __shared__ __align__(8) uint64_t full[S], empty[S], done, drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int s_abort;
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  auto tileA = [&](int s) { return smem + s * Cfg::kStage; };
  auto tileB = [&](int s) { return smem + s * Cfg::kStage + kTileA; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * BN;
  const int KB = (K + kBK - 1) / kBK;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    mbar_init(&drain, 1);
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_slot, Cfg::kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  volatile int *abort_flag = &s_abort;

  if (warp == 0 && lane == 0) {
    // producer
    int issued = 0;
    for (int kb = 0; kb < KB; ++kb) {
      const int s = kb % S;
      if (kb >= S && !mbar_wait_bounded(&empty[s], ((kb / S) - 1) & 1)) {
        *abort_flag = 1;
        raise_error(err, GDN_DEVERR_TIMEOUT);
        break;
      }
      if (*abort_flag) break;
      mbar_arrive_expect_tx(&full[s], Cfg::kStage);
      tma_load2(tileA(s), &mx, kb * kBK, m0, &full[s]);
      tma_load2(tileB(s), &mw, kb * kBK, n0, &full[s]);
      issued = kb + 1;
    }
    if (*abort_flag) {  // let the copies still in flight land before the CTA exits
      for (int kb = issued - S < 0 ? 0 : issued - S; kb < issued; ++kb)
        mbar_wait_bounded(&full[kb % S], (kb / S) & 1);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    constexpr uint32_t idesc = tc::idesc_bf16(kBM, BN);
    bool ok = true;
    for (int kb = 0; kb < KB && ok; ++kb) {
      const int s = kb % S;
      if (!mbar_wait_bounded(&full[s], (kb / S) & 1) || *abort_flag) {
        *abort_flag = 1;
        raise_error(err, GDN_DEVERR_TIMEOUT);
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t a = smem_addr(tileA(s)), b = smem_addr(tileB(s));
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        tc::mma_ss_f16(tmem, tc::smem_desc_sw128(a + 32 * kk), tc::smem_desc_sw128(b + 32 * kk),
                       idesc, (kb | kk) ? 1u : 0u);
      tc::mma_commit(&empty[s]);
    }
    tc::mma_commit(ok ? &done : &drain);
    if (!ok) mbar_wait_bounded(&drain, 0);  // MMAs in flight finish before TMEM is freed
  } else if (warp >= 2) {
    // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31
    const int quad = warp & 3;
    const int row = m0 + 32 * quad + lane;
    // warp-uniform decision: tcgen05.ld is a whole-warp instruction
    const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(&done, 0));
    if (!got) {
      *abort_flag = 1;
      if (lane == 0) raise_error(err, GDN_DEVERR_TIMEOUT);
    } else if (!__any_sync(0xffffffffu, *abort_flag != 0)) {
      tc::fence_after_sync();
      TO *yrow = y + (int64_t)row * ld_y + n0;
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        float v[16];
        tc::tmem_ld16(tmem + ((uint32_t)(32 * quad) << 16) + 16 * c, v);
        const int nv = N - (n0 + 16 * c);
        if (row < M && nv > 0) store_row16<TO>(yrow + 16 * c, v, nv);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

// ---- persistent form for many tiles (prefill-sized token counts) ----
//
// One CTA per SM walks the output tiles t = blockIdx.x, blockIdx.x + grid, ...
// (128 x 256 each, column block fastest: the CTAs in flight cover a few row
// blocks of x and all of W, which stays resident in L2).  The producer and MMA threads run across tile
// boundaries through one 4-stage ring (48 KiB per stage); the accumulator is
// double-buffered in TMEM (2 x 256 columns), so the four epilogue warps drain
// tile i while the MMAs of tile i + 1 run.  Barriers: full / empty per stage
// (as above), acc_full[b] (MMA commit) and acc_empty[b] (one arrival per
// epilogue warp once it has read buffer b).
constexpr int kPBN = 256;
constexpr int kPStages = 4;
constexpr int kPStage = kTileA + kPBN * kBK * 2;         // 48 KiB
constexpr int kPSmem = kPStages * kPStage + 1024;

template <typename TO>
__global__ void __launch_bounds__(kGemmThreads, 1)
    in_proj_persistent_kernel(const __grid_constant__ CUtensorMap mx,
                              const __grid_constant__ CUtensorMap mw, int M, int N, int K,
                              TO *__restrict__ y, int64_t ld_y, unsigned int *__restrict__ err) {
  constexpr int S = kPStages;
  extern __shared__ unsigned char dsm_raw[];
  __shared__ __align__(8) uint64_t full[S], empty[S], acc_full[2], acc_empty[2], drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int s_abort;
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  auto tileA = [&](int s) { return smem + s * kPStage; };
  auto tileB = [&](int s) { return smem + s * kPStage + kTileA; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int KB = (K + kBK - 1) / kBK;
  const int m_tiles = (M + kBM - 1) / kBM;
  const int n_tiles = (N + kPBN - 1) / kPBN;
  const int tiles = m_tiles * n_tiles;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(&drain, 1);
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_slot, 2 * kPBN);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  volatile int *abort_flag = &s_abort;
  auto fail = [&]() {
    *abort_flag = 1;
    raise_error(err, GDN_DEVERR_TIMEOUT);
  };

  if (warp == 0 && lane == 0) {
    // producer: one k-block per stage, across tiles
    int64_t g = 0, issued = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
      const int m0 = (t / n_tiles) * kBM, n0 = (t % n_tiles) * kPBN;
      for (int kb = 0; kb < KB; ++kb, ++g) {
        const int s = (int)(g % S);
        const int64_t u = g / S;
        if ((u > 0 && !mbar_wait_bounded(&empty[s], (uint32_t)((u - 1) & 1))) || *abort_flag) {
          fail();
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kPStage);
        tma_load2(tileA(s), &mx, kb * kBK, m0, &full[s]);
        tma_load2(tileB(s), &mw, kb * kBK, n0, &full[s]);
        issued = g + 1;
      }
    }
    if (!ok) {  // the copies still in flight land before the CTA exits
      for (int64_t q = issued - S < 0 ? 0 : issued - S; q < issued; ++q)
        mbar_wait_bounded(&full[q % S], (uint32_t)((q / S) & 1));
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    constexpr uint32_t idesc = tc::idesc_bf16(kBM, kPBN);
    int64_t g = 0;
    int i = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++i) {
      const int b = i & 1, v = i >> 1;
      if ((v > 0 && !mbar_wait_bounded(&acc_empty[b], (uint32_t)((v - 1) & 1))) || *abort_flag) {
        fail();
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t acc = tmem + (uint32_t)(b * kPBN);
      for (int kb = 0; kb < KB; ++kb, ++g) {
        const int s = (int)(g % S);
        if (!mbar_wait_bounded(&full[s], (uint32_t)((g / S) & 1)) || *abort_flag) {
          fail();
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t a = smem_addr(tileA(s)), bb = smem_addr(tileB(s));
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          tc::mma_ss_f16(acc, tc::smem_desc_sw128(a + 32 * kk), tc::smem_desc_sw128(bb + 32 * kk),
                         idesc, (kb | kk) ? 1u : 0u);
        tc::mma_commit(&empty[s]);
      }
      if (ok) tc::mma_commit(&acc_full[b]);
    }
    if (!ok) {
      tc::mma_commit(&drain);
      mbar_wait_bounded(&drain, 0);  // MMAs in flight finish before TMEM is freed
    }
  } else if (warp >= 2) {
    // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 of buffer i % 2
    const int quad = warp & 3;
    int i = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
      const int b = i & 1, v = i >> 1;
      const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_full[b], (uint32_t)(v & 1)));
      if (!got || __any_sync(0xffffffffu, *abort_flag != 0)) {
        if (!got && lane == 0) fail();
        break;
      }
      tc::fence_after_sync();
      const int m0 = (t / n_tiles) * kBM, n0 = (t % n_tiles) * kPBN;
      const int row = m0 + 32 * quad + lane;
      TO *yrow = y + (int64_t)row * ld_y + n0;
      const uint32_t acc = tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(b * kPBN);
#pragma unroll 1
      for (int c = 0; c < kPBN / 32; ++c) {
        float v32[32];
        tc::tmem_ld32(acc + 32 * c, acc + 32 * c + 16, v32);
        const int nv = N - (n0 + 32 * c);
        if (row < M && nv > 0) {
          store_row16<TO>(yrow + 32 * c, v32, nv);
          if (nv > 16) store_row16<TO>(yrow + 32 * c + 16, v32 + 16, nv - 16);
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 2 * kPBN);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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
  return encode;
}

// [rows][cols] bf16 with row stride ld elements, box {64, box_rows}, 128-byte swizzle
bool encode_rows(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld,
                 int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  cuuint32_t elem[2] = {1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int BN, typename TO>
cudaError_t launch_in_proj_t(int64_t M, int N, int K, const void *x, int64_t ld_x, const void *w,
                             int64_t ld_w, void *y, int64_t ld_y, unsigned int *err,
                             cudaStream_t s) {
  CUtensorMap mx, mw;
  if (!encode_rows(&mx, x, M, K, ld_x, kBM) || !encode_rows(&mw, w, N, K, ld_w, BN))
    return cudaErrorInvalidValue;
  auto kern = in_proj_kernel<BN, TO>;
  const cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GemmCfg<BN>::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + kBM - 1) / kBM));
  kern<<<grid, kGemmThreads, GemmCfg<BN>::kSmem, s>>>(mx, mw, (int)M, N, K,
                                                       static_cast<TO *>(y), ld_y, err);
  return cudaGetLastError();
}

template <typename TO>
cudaError_t launch_in_proj_persistent(int64_t M, int N, int K, const void *x, int64_t ld_x,
                                      const void *w, int64_t ld_w, void *y, int64_t ld_y,
                                      unsigned int *err, int sm_count, cudaStream_t s) {
  CUtensorMap mx, mw;
  if (!encode_rows(&mx, x, M, K, ld_x, kBM) || !encode_rows(&mw, w, N, K, ld_w, kPBN))
    return cudaErrorInvalidValue;
  auto kern = in_proj_persistent_kernel<TO>;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kPSmem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kPBN - 1) / kPBN);
  const int grid = (int)(tiles < sm_count ? tiles : sm_count);
  kern<<<grid, kGemmThreads, kPSmem, s>>>(mx, mw, (int)M, N, K, static_cast<TO *>(y), ld_y,
                                          err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_in_proj(int64_t M, int N, int K, const void *x, int64_t ld_x, const void *w,
                           int64_t ld_w, void *y, int64_t ld_y, gdn_dtype y_dtype,
                           unsigned int *err, int sm_count, cudaStream_t s) {
  // many 128 x 256 tiles (prefill-sized token counts): the persistent kernel;
  // else 128-column tiles unless that leaves SMs idle (a decode step: 64-column)
  const int64_t m_tiles = (M + kBM - 1) / kBM;
  if (m_tiles * ((N + kPBN - 1) / kPBN) >= 4 * (int64_t)sm_count)
    return y_dtype == GDN_F32
               ? launch_in_proj_persistent<float>(M, N, K, x, ld_x, w, ld_w, y, ld_y, err,
                                                  sm_count, s)
               : launch_in_proj_persistent<bf16>(M, N, K, x, ld_x, w, ld_w, y, ld_y, err,
                                                 sm_count, s);
  const bool narrow = m_tiles * ((N + 127) / 128) < 2 * (int64_t)sm_count;
  if (y_dtype == GDN_F32)
    return narrow ? launch_in_proj_t<96, float>(M, N, K, x, ld_x, w, ld_w, y, ld_y, err, s)
                  : launch_in_proj_t<128, float>(M, N, K, x, ld_x, w, ld_w, y, ld_y, err, s);
  return narrow ? launch_in_proj_t<96, bf16>(M, N, K, x, ld_x, w, ld_w, y, ld_y, err, s)
                : launch_in_proj_t<128, bf16>(M, N, K, x, ld_x, w, ld_w, y, ld_y, err, s);
}

}  // namespace gdn
