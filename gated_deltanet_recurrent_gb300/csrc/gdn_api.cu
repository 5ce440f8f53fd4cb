// extern "C" entry points of libgdn: argument validation (always), optional
// host-side validation of the index arrays, and the kernel launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>

#include <cmath>
#include <string>
#include <vector>

#include "gdn_internal.h"

struct gdn_pool {
  gdn::PoolView view;
  gdn_pool_desc desc;
  int device;
  int sm_count;
  bool has_tmap;
  alignas(64) CUtensorMap tmap;  // the state as a [rows][dk] float32 tensor (TMA)
  cudaMemPool_t work_pool;       // stream-ordered prefill workspaces (kept until destroy)
};

namespace {

thread_local std::string g_last_msg;

gdn_status fail(gdn_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_msg = buf;
  return s;
}

gdn_status ok() {
  g_last_msg.clear();
  return GDN_OK;
}

gdn_status cuda_fail(cudaError_t e, const char *what) {
  return fail(GDN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool dtype_ok(gdn_dtype d) { return d == GDN_F32 || d == GDN_BF16; }
size_t dtype_size(gdn_dtype d) { return d == GDN_F32 ? 4 : 2; }
bool dk_supported(int dk) { return dk == 16 || dk == 32 || dk == 64 || dk == 128; }

gdn_status check_desc(const gdn_pool_desc *d) {
  if (!d) return fail(GDN_ERR_ARG, "desc is NULL");
  if (d->n_layers < 1 || d->n_slots < 1 || d->h_v < 1 || d->h_k < 1 || d->dk < 1 || d->dv < 1 ||
      d->conv_ch < 1 || d->conv_k < 1)
    return fail(GDN_ERR_ARG, "pool dimensions must be positive");
  if (d->h_v % d->h_k != 0) return fail(GDN_ERR_ARG, "h_v (%d) is not a multiple of h_k (%d)",
                                        d->h_v, d->h_k);
  if (!dtype_ok(d->conv_dtype)) return fail(GDN_ERR_DTYPE, "conv_dtype must be F32 or BF16");
  if (d->state_dtype != GDN_F32 && d->state_dtype != GDN_BF16 && d->state_dtype != GDN_F16)
    return fail(GDN_ERR_DTYPE, "state_dtype must be F32, BF16 or F16");
  if (!dk_supported(d->dk)) return fail(GDN_ERR_UNSUPPORTED, "dk=%d (supported: 16,32,64,128)",
                                        d->dk);
  if (d->dv % 4 != 0 || d->dv > 4096) return fail(GDN_ERR_UNSUPPORTED,
                                                  "dv=%d must be a multiple of 4, <= 4096", d->dv);
  if (d->conv_k < 2 || d->conv_k > 8) return fail(GDN_ERR_UNSUPPORTED, "conv_k=%d (2..8)",
                                                  d->conv_k);
  if (d->n_slots > 65535) return fail(GDN_ERR_UNSUPPORTED, "n_slots=%d (max 65535)", d->n_slots);
  return GDN_OK;
}

gdn_status check_pool(const gdn_pool *p, int layer) {
  if (!p) return fail(GDN_ERR_ARG, "pool is NULL");
  if (layer < 0 || layer >= p->desc.n_layers)
    return fail(GDN_ERR_ARG, "layer %d outside [0, %d)", layer, p->desc.n_layers);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != p->device)
    return fail(GDN_ERR_ARG, "current device %d is not the pool's device %d", dev, p->device);
  return GDN_OK;
}

// Under host checks: is this pointer something the device can dereference?
gdn_status check_device_ptr(const void *ptr, const char *name) {
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, ptr);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(GDN_ERR_ARG, "%s: cudaPointerGetAttributes failed", name);
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return fail(GDN_ERR_ARG, "%s is not device memory", name);
  return GDN_OK;
}

gdn_status fetch(std::vector<int32_t> &dst, const int32_t *src, size_t n, cudaStream_t s,
                 const char *name) {
  dst.resize(n);
  if (n == 0) return GDN_OK;
  gdn_status st = check_device_ptr(src, name);
  if (st != GDN_OK) return st;
  cudaError_t e = cudaMemcpyAsync(dst.data(), src, n * sizeof(int32_t), cudaMemcpyDefault, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "copying index array to host");
  return GDN_OK;
}

gdn_status check_slots(const gdn_pool *p, const int32_t *slot_ids, int n, cudaStream_t s) {
  std::vector<int32_t> h;
  gdn_status st = fetch(h, slot_ids, (size_t)n, s, "slot_ids");
  if (st != GDN_OK) return st;
  std::vector<unsigned char> seen((size_t)p->desc.n_slots, 0);
  for (int i = 0; i < n; ++i) {
    if (h[i] < 0 || h[i] >= p->desc.n_slots)
      return fail(GDN_ERR_SLOT, "slot_ids[%d] = %d outside [0, %d)", i, h[i], p->desc.n_slots);
    if (seen[h[i]]) return fail(GDN_ERR_DUP_SLOT, "slot id %d repeated (entry %d)", h[i], i);
    seen[h[i]] = 1;
  }
  return GDN_OK;
}

gdn_status check_cu(const int32_t *cu, int n_seqs, int total, cudaStream_t s,
                    std::vector<int32_t> &h) {
  gdn_status st = fetch(h, cu, (size_t)n_seqs + 1, s, "cu_seqlens");
  if (st != GDN_OK) return st;
  if (h[0] != 0) return fail(GDN_ERR_SIZE, "cu_seqlens[0] = %d, expected 0", h[0]);
  for (int i = 0; i < n_seqs; ++i)
    if (h[i + 1] < h[i]) return fail(GDN_ERR_SIZE, "cu_seqlens decreases at %d", i);
  if (h[n_seqs] != total)
    return fail(GDN_ERR_SIZE, "cu_seqlens[%d] = %d, expected total_tokens %d", n_seqs, h[n_seqs],
                total);
  return GDN_OK;
}

gdn_status check_counts(const int32_t *cnt, int n, const std::vector<int32_t> *cu, int fixed,
                        cudaStream_t s, const char *name) {
  std::vector<int32_t> h;
  gdn_status st = fetch(h, cnt, (size_t)n, s, name);
  if (st != GDN_OK) return st;
  for (int i = 0; i < n; ++i) {
    const int lim = cu ? (*cu)[i + 1] - (*cu)[i] : fixed;
    if (h[i] < 0 || h[i] > lim)
      return fail(GDN_ERR_SIZE, "%s[%d] = %d outside [0, %d]", name, i, h[i], lim);
  }
  return GDN_OK;
}

// Validate and resolve a gdn_qkv for `tokens` tokens.
gdn_status resolve_qkv(const gdn_pool *p, const gdn_qkv *in, int64_t tokens, gdn::QKV &out) {
  if (!in) return fail(GDN_ERR_ARG, "inputs struct is NULL");
  if (!dtype_ok(in->dtype)) return fail(GDN_ERR_DTYPE, "input dtype must be F32 or BF16");
  if (!in->q || !in->k || !in->v || !in->g || !in->beta)
    return fail(GDN_ERR_ARG, "q, k, v, g and beta must all be non-NULL");
  const gdn_pool_desc &d = p->desc;
  const int64_t ld_qk = in->ld_qk ? in->ld_qk : (int64_t)d.h_k * d.dk;
  const int64_t ld_v = in->ld_v ? in->ld_v : (int64_t)d.h_v * d.dv;
  if (ld_qk < (int64_t)d.h_k * d.dk || ld_v < (int64_t)d.h_v * d.dv)
    return fail(GDN_ERR_ARG, "token strides smaller than a token (ld_qk %lld, ld_v %lld)",
                (long long)ld_qk, (long long)ld_v);
  const size_t es = dtype_size(in->dtype);
  const size_t al = in->dtype == GDN_F32 ? 16 : 8;
  if ((uintptr_t)in->q % al || (uintptr_t)in->k % al || ((size_t)ld_qk * es) % al)
    return fail(GDN_ERR_ARG, "q/k rows must start %zu-byte aligned", al);
  if (p->desc.host_checks && tokens > 0) {
    gdn_status st;
    if ((st = check_device_ptr(in->q, "q")) || (st = check_device_ptr(in->k, "k")) ||
        (st = check_device_ptr(in->v, "v")) || (st = check_device_ptr(in->g, "g")) ||
        (st = check_device_ptr(in->beta, "beta")))
      return st;
  }
  out = gdn::QKV{in->q, in->k, in->v, in->g, in->beta, ld_qk, ld_v, in->dtype};
  return GDN_OK;
}

// Tensor map over the whole state viewed as [n_layers*n_slots*h_v*dv][dk]
// float32, box 128 rows x 32 columns, 128-byte swizzle (one value head of
// 128 x 128 is four boxes).  Encoded through the runtime's driver entry
// point, so the library does not link libcuda.  Returns false if unavailable.
bool encode_state_map(gdn_pool *p) {
  const gdn_pool_desc &d = p->desc;
  if (d.dk != 128 || d.dv != 128 || d.state_dtype != GDN_F32) return false;
  const uint64_t rows = (uint64_t)d.n_layers * d.n_slots * d.h_v * d.dv;
  if (rows > 0x7fffffffull) return false;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      fn == nullptr || q != cudaDriverEntryPointSuccess) {
    cudaGetLastError();
    return false;
  }
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  cuuint64_t dims[2] = {(cuuint64_t)d.dk, rows};
  cuuint64_t strides[1] = {(cuuint64_t)d.dk * sizeof(float)};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t elem[2] = {1, 1};
  return encode(&p->tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p->view.state, dims, strides, box,
                elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

extern "C" {

const char *gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_ARG: return "GDN_ERR_ARG";
    case GDN_ERR_SLOT: return "GDN_ERR_SLOT";
    case GDN_ERR_DUP_SLOT: return "GDN_ERR_DUP_SLOT";
    case GDN_ERR_DTYPE: return "GDN_ERR_DTYPE";
    case GDN_ERR_SIZE: return "GDN_ERR_SIZE";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
  }
  return "GDN_ERR_<unknown>";
}

const char *gdn_last_error_message(void) { return g_last_msg.c_str(); }

size_t gdn_pool_state_bytes(const gdn_pool_desc *d) {
  if (!d || d->n_layers < 0 || d->n_slots < 0) return 0;
  return (size_t)d->n_layers * d->n_slots * d->h_v * d->dv * d->dk *
         (d->state_dtype == GDN_F32 ? sizeof(float) : 2);
}

size_t gdn_pool_conv_bytes(const gdn_pool_desc *d) {
  if (!d || d->n_layers < 0 || d->n_slots < 0 || d->conv_k < 1) return 0;
  return (size_t)d->n_layers * d->n_slots * d->conv_ch * (d->conv_k - 1) *
         dtype_size(d->conv_dtype);
}

gdn_status gdn_pool_create(const gdn_pool_desc *desc, void *state_mem, size_t state_bytes,
                           void *conv_mem, size_t conv_bytes, gdn_pool **out) {
  if (!out) return fail(GDN_ERR_ARG, "out is NULL");
  *out = nullptr;
  gdn_status st = check_desc(desc);
  if (st != GDN_OK) return st;
  if (!state_mem || !conv_mem) return fail(GDN_ERR_ARG, "state_mem and conv_mem must be non-NULL");
  if ((uintptr_t)state_mem % 16 || (uintptr_t)conv_mem % 16)
    return fail(GDN_ERR_ARG, "state_mem and conv_mem must be 16-byte aligned");
  if (state_bytes < gdn_pool_state_bytes(desc))
    return fail(GDN_ERR_SIZE, "state_bytes %zu < %zu needed", state_bytes,
                gdn_pool_state_bytes(desc));
  if (conv_bytes < gdn_pool_conv_bytes(desc))
    return fail(GDN_ERR_SIZE, "conv_bytes %zu < %zu needed", conv_bytes, gdn_pool_conv_bytes(desc));
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (desc->host_checks) {
    if ((st = check_device_ptr(state_mem, "state_mem")) ||
        (st = check_device_ptr(conv_mem, "conv_mem")))
      return st;
  }
  // one allocation: the error word, then the one-call decode step's tickets
  // (one per layer, slot and key head), all zero
  const size_t n_ticks = (size_t)desc->n_layers * desc->n_slots * desc->h_k;
  const size_t aux_bytes = (1 + n_ticks) * sizeof(unsigned int);
  unsigned int *err = nullptr;
  e = cudaMalloc(&err, aux_bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(error word and tickets)");
  e = cudaMemset(err, 0, aux_bytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(err);
    return cuda_fail(e, "cudaMemset(error word and tickets)");
  }
  int sm_count = 0;
  e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    cudaFree(err);
    return cuda_fail(e, "cudaDeviceGetAttribute(multiprocessor count)");
  }
  gdn_pool *p = new gdn_pool;
  p->desc = *desc;
  p->device = dev;
  p->sm_count = sm_count;
  p->view = gdn::PoolView{static_cast<float *>(state_mem), conv_mem, err,
                          desc->n_layers, desc->n_slots, desc->h_v, desc->h_k, desc->dk,
                          desc->dv, desc->conv_ch, desc->conv_k, desc->conv_dtype, err + 1,
                          desc->state_dtype, 0u};
  p->has_tmap = encode_state_map(p);
  cudaMemPoolProps props = {};
  props.allocType = cudaMemAllocationTypePinned;
  props.location.type = cudaMemLocationTypeDevice;
  props.location.id = dev;
  e = cudaMemPoolCreate(&p->work_pool, &props);
  if (e == cudaSuccess) {
    uint64_t keep = UINT64_MAX;  // keep freed workspace for the next call
    e = cudaMemPoolSetAttribute(p->work_pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) cudaMemPoolDestroy(p->work_pool);
  }
  if (e != cudaSuccess) {
    cudaFree(err);
    delete p;
    return cuda_fail(e, "creating the workspace memory pool");
  }
  *out = p;
  return ok();
}

gdn_status gdn_pool_destroy(gdn_pool *p) {
  if (!p) return ok();
  cudaError_t e = cudaDeviceSynchronize();
  cudaError_t e2 = cudaFree(p->view.err);  // the error word and the tickets
  cudaError_t e3 = cudaMemPoolDestroy(p->work_pool);
  if (e2 == cudaSuccess) e2 = e3;
  delete p;
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaFree(error word)");
  return ok();
}

gdn_status gdn_pool_set_test_flags(gdn_pool *p, uint32_t flags) {
  if (!p) return fail(GDN_ERR_ARG, "pool is NULL");
  if (flags & ~(uint32_t)GDN_TEST_DECODE_WAIT_TIMEOUT)
    return fail(GDN_ERR_ARG, "unknown test flags 0x%x", flags);
  p->view.test_flags = flags;
  return ok();
}

gdn_status gdn_pool_get_error(gdn_pool *p, uint32_t *dev_err) {
  if (!p || !dev_err) return fail(GDN_ERR_ARG, "pool and dev_err must be non-NULL");
  unsigned int h = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&h, p->view.err, sizeof(h), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(p->view.err, 0, sizeof(h));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  *dev_err = h;
  return ok();
}

gdn_status gdn_pool_reset(gdn_pool *p, const int32_t *slot_ids, int32_t n, gdn_stream stream) {
  gdn_status st = check_pool(p, 0);
  if (st != GDN_OK) return st;
  if (n < 0) return fail(GDN_ERR_ARG, "n = %d < 0", n);
  if (n == 0) return ok();
  if (!slot_ids) return fail(GDN_ERR_ARG, "slot_ids is NULL");
  if (n > 65535) return fail(GDN_ERR_SIZE, "n = %d > 65535", n);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->desc.host_checks && (st = check_slots(p, slot_ids, n, s))) return st;
  cudaError_t e = gdn::launch_pool_reset(p->view, slot_ids, n, s);
  if (e != cudaSuccess) return cuda_fail(e, "pool reset launch");
  return ok();
}

gdn_status gdn_pool_copy(gdn_pool *p, const int32_t *src_slots, const int32_t *dst_slots,
                         int32_t n, gdn_stream stream) {
  gdn_status st = check_pool(p, 0);
  if (st != GDN_OK) return st;
  if (n < 0) return fail(GDN_ERR_ARG, "n = %d < 0", n);
  if (n == 0) return ok();
  if (!src_slots || !dst_slots) return fail(GDN_ERR_ARG, "src_slots and dst_slots must be non-NULL");
  if (n > 65535) return fail(GDN_ERR_SIZE, "n = %d > 65535", n);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->desc.host_checks) {
    if ((st = check_slots(p, dst_slots, n, s))) return st;
    std::vector<int32_t> hs, hd;
    if ((st = fetch(hs, src_slots, (size_t)n, s, "src_slots")) ||
        (st = fetch(hd, dst_slots, (size_t)n, s, "dst_slots")))
      return st;
    std::vector<unsigned char> is_dst((size_t)p->desc.n_slots, 0);
    for (int i = 0; i < n; ++i) is_dst[hd[i]] = 1;
    for (int i = 0; i < n; ++i) {
      if (hs[i] < 0 || hs[i] >= p->desc.n_slots)
        return fail(GDN_ERR_SLOT, "src_slots[%d] = %d outside [0, %d)", i, hs[i], p->desc.n_slots);
      if (is_dst[hs[i]])
        return fail(GDN_ERR_DUP_SLOT, "slot %d is both a source and a destination", hs[i]);
    }
  }
  cudaError_t e = gdn::launch_pool_copy(p->view, src_slots, dst_slots, n, s);
  if (e != cudaSuccess) return cuda_fail(e, "pool copy launch");
  return ok();
}

gdn_status gdn_conv_silu(gdn_pool *p, int32_t layer, const int32_t *slot_ids,
                         const int32_t *cu_seqlens, int32_t n_seqs, int32_t total_tokens,
                         int32_t max_seqlen, const void *x, int64_t ld_x, gdn_dtype x_dtype,
                         const float *w, const float *bias, void *y, int64_t ld_y,
                         const int32_t *advance, gdn_stream stream) {
  gdn_status st = check_pool(p, layer);
  if (st != GDN_OK) return st;
  if (n_seqs < 0 || total_tokens < 0) return fail(GDN_ERR_ARG, "negative n_seqs/total_tokens");
  if (n_seqs > 65535) return fail(GDN_ERR_SIZE, "n_seqs = %d > 65535", n_seqs);
  if (!cu_seqlens && total_tokens != n_seqs)
    return fail(GDN_ERR_SIZE, "without cu_seqlens total_tokens must equal n_seqs");
  if (n_seqs == 0 || total_tokens == 0) return ok();
  if (x_dtype != p->desc.conv_dtype)
    return fail(GDN_ERR_DTYPE, "x dtype differs from the pool's conv_dtype");
  if (!slot_ids || !x || !w) return fail(GDN_ERR_ARG, "slot_ids, x and w must be non-NULL");
  const int64_t C = p->desc.conv_ch;
  if (ld_x == 0) ld_x = C;
  if (ld_y == 0) ld_y = C;
  if (ld_x < C || ld_y < C) return fail(GDN_ERR_ARG, "row strides smaller than conv_ch");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->desc.host_checks) {
    if ((st = check_slots(p, slot_ids, n_seqs, s))) return st;
    std::vector<int32_t> cu;
    if (cu_seqlens && (st = check_cu(cu_seqlens, n_seqs, total_tokens, s, cu))) return st;
    if (advance && (st = check_counts(advance, n_seqs, cu_seqlens ? &cu : nullptr, 1, s,
                                      "advance")))
      return st;
    if ((st = check_device_ptr(x, "x")) || (st = check_device_ptr(w, "w")) ||
        (bias && (st = check_device_ptr(bias, "bias"))) ||
        (y && (st = check_device_ptr(y, "y"))))
      return st;
  }
  gdn::SeqIndex seq{slot_ids, cu_seqlens, n_seqs, total_tokens};
  cudaError_t e = gdn::launch_conv_silu(p->view, layer, seq, max_seqlen < 1 ? 1 : max_seqlen, x,
                                        ld_x, w, bias, y, ld_y, advance, s);
  if (e != cudaSuccess) return cuda_fail(e, "conv launch");
  return ok();
}

gdn_status gdn_decode_step(gdn_pool *p, int32_t layer, const int32_t *slot_ids, int32_t n,
                           const gdn_qkv *in, void *o, gdn_dtype o_dtype, float scale,
                           gdn_stream stream) {
  gdn_status st = check_pool(p, layer);
  if (st != GDN_OK) return st;
  if (n < 0) return fail(GDN_ERR_ARG, "n = %d < 0", n);
  if (n == 0) return ok();
  if (n > 65535) return fail(GDN_ERR_SIZE, "n = %d > 65535", n);
  if (!slot_ids || !o) return fail(GDN_ERR_ARG, "slot_ids and o must be non-NULL");
  if (!dtype_ok(o_dtype)) return fail(GDN_ERR_DTYPE, "o dtype must be F32 or BF16");
  gdn::QKV q;
  if ((st = resolve_qkv(p, in, n, q))) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->desc.host_checks) {
    if ((st = check_slots(p, slot_ids, n, s)) || (st = check_device_ptr(o, "o"))) return st;
  }
  cudaError_t e = gdn::launch_decode(p->view, p->has_tmap ? &p->tmap : nullptr, layer, slot_ids,
                                     n, q, o, o_dtype, scale, s);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return ok();
}

}  // extern "C"

namespace {

// The form gdn_decode_step_conv takes for n slots: one fused kernel per (row
// block, value head, slot) while that grid is resident at once (small n: one
// launch and one wave; beyond that its CTAs each recompute their key head's q
// and k conv), else one fused kernel per (slot, key head) where the shape
// allows it, else the conv launch followed by the decode as a programmatic
// dependent launch (the decode fetches its state tiles while the conv runs).
enum class StepConvForm { kFusedRows, kFusedGroup, kPair };

cudaError_t step_conv_form(const gdn_pool *p, int32_t n, gdn_dtype dtype, gdn_dtype o_dtype,
                           StepConvForm *form) {
  int64_t resident = 0;
  const cudaError_t e =
      gdn::decode_conv_resident_ctas(p->view, dtype, o_dtype, p->sm_count, &resident);
  if (e != cudaSuccess) return e;
  if (gdn::decode_grid_ctas(p->view, n) <= resident) *form = StepConvForm::kFusedRows;
  else if (gdn::decode_conv_group_ok(p->view)) *form = StepConvForm::kFusedGroup;
  else *form = StepConvForm::kPair;
  return cudaSuccess;
}

}  // namespace

extern "C" {

gdn_status gdn_decode_step_conv_launches(gdn_pool *p, int32_t n, gdn_dtype dtype,
                                         gdn_dtype o_dtype, int32_t *launches) {
  gdn_status st = check_pool(p, 0);
  if (st != GDN_OK) return st;
  if (!launches) return fail(GDN_ERR_ARG, "launches must be non-NULL");
  if (n < 0 || n > 65535) return fail(GDN_ERR_ARG, "n = %d outside [0, 65535]", n);
  if (dtype != p->desc.conv_dtype) return fail(GDN_ERR_DTYPE, "dtype differs from the pool's conv_dtype");
  if (!dtype_ok(o_dtype)) return fail(GDN_ERR_DTYPE, "o dtype must be F32 or BF16");
  if (n == 0) {
    *launches = 0;
    return ok();
  }
  StepConvForm form;
  const cudaError_t e = step_conv_form(p, n, dtype, o_dtype, &form);
  if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
  *launches = form == StepConvForm::kPair ? 2 : 1;
  return ok();
}

gdn_status gdn_decode_step_conv(gdn_pool *p, int32_t layer, const int32_t *slot_ids,
                                int32_t n, const void *x, int64_t ld_x, const float *w,
                                const float *bias, void *y, int64_t ld_y, const void *g,
                                const void *beta, gdn_dtype dtype, void *o, gdn_dtype o_dtype,
                                float scale, gdn_stream stream) {
  gdn_status st = check_pool(p, layer);
  if (st != GDN_OK) return st;
  if (n < 0) return fail(GDN_ERR_ARG, "n = %d < 0", n);
  if (n == 0) return ok();
  if (n > 65535) return fail(GDN_ERR_SIZE, "n = %d > 65535", n);
  const gdn_pool_desc &d = p->desc;
  const int64_t C = d.conv_ch, nqk = (int64_t)d.h_k * d.dk;
  if (C != 2 * nqk + (int64_t)d.h_v * d.dv)
    return fail(GDN_ERR_SIZE, "conv_ch = %lld is not 2*h_k*dk + h_v*dv = %lld", (long long)C,
                (long long)(2 * nqk + (int64_t)d.h_v * d.dv));
  if (dtype != d.conv_dtype) return fail(GDN_ERR_DTYPE, "dtype differs from the pool's conv_dtype");
  if (!dtype_ok(o_dtype)) return fail(GDN_ERR_DTYPE, "o dtype must be F32 or BF16");
  if (!slot_ids || !x || !w || !y || !o)
    return fail(GDN_ERR_ARG, "slot_ids, x, w, y and o must be non-NULL");
  if (ld_x == 0) ld_x = C;
  if (ld_y == 0) ld_y = C;
  if (ld_x < C || ld_y < C) return fail(GDN_ERR_ARG, "row strides smaller than conv_ch");
  const size_t es = dtype_size(dtype);
  unsigned char *yb = static_cast<unsigned char *>(y);
  const gdn_qkv in{yb, yb + nqk * es, yb + 2 * nqk * es, g, beta, ld_y, ld_y, dtype};
  gdn::QKV q;
  if ((st = resolve_qkv(p, &in, n, q))) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (d.host_checks) {
    if ((st = check_slots(p, slot_ids, n, s)) || (st = check_device_ptr(x, "x")) ||
        (st = check_device_ptr(w, "w")) || (bias && (st = check_device_ptr(bias, "bias"))) ||
        (st = check_device_ptr(o, "o")))
      return st;
  }
  StepConvForm form;
  cudaError_t e = step_conv_form(p, n, dtype, o_dtype, &form);
  if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
  if (form == StepConvForm::kFusedRows) {
    e = gdn::launch_decode_conv(p->view, layer, slot_ids, n, x, ld_x, w, bias, y, ld_y, g, beta,
                                dtype, o, o_dtype, scale, s);
    if (e != cudaSuccess) return cuda_fail(e, "conv + decode launch");
    return ok();
  }
  if (form == StepConvForm::kFusedGroup) {
    e = gdn::launch_decode_conv_group(p->view, layer, slot_ids, n, x, ld_x, w, bias, y, ld_y, g,
                                      beta, dtype, o, o_dtype, scale, s);
    if (e != cudaSuccess) return cuda_fail(e, "conv + decode launch");
    return ok();
  }
  gdn::SeqIndex seq{slot_ids, nullptr, n, n};
  e = gdn::launch_conv_silu(p->view, layer, seq, 1, x, ld_x, w, bias, y, ld_y, nullptr, s);
  if (e != cudaSuccess) return cuda_fail(e, "conv launch");
  e = gdn::launch_decode(p->view, p->has_tmap ? &p->tmap : nullptr, layer, slot_ids, n, q, o,
                         o_dtype, scale, s, /*after_conv=*/true);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return ok();
}

gdn_status gdn_in_proj(gdn_pool *p, int64_t tokens, int32_t hidden, int32_t n_out,
                       const void *x, int64_t ld_x, const void *w, int64_t ld_w, void *y,
                       int64_t ld_y, gdn_dtype y_dtype, gdn_stream stream) {
  gdn_status st = check_pool(p, 0);
  if (st != GDN_OK) return st;
  if (tokens < 0 || hidden < 1 || n_out < 1)
    return fail(GDN_ERR_ARG, "tokens = %lld, hidden = %d, n_out = %d", (long long)tokens, hidden,
                n_out);
  if (!dtype_ok(y_dtype)) return fail(GDN_ERR_DTYPE, "y dtype must be F32 or BF16");
  if (tokens == 0) return ok();
  if (tokens > INT32_MAX) return fail(GDN_ERR_SIZE, "tokens = %lld > 2^31 - 1", (long long)tokens);
  if (!x || !w || !y) return fail(GDN_ERR_ARG, "x, w and y must be non-NULL");
  if (ld_x == 0) ld_x = hidden;
  if (ld_w == 0) ld_w = hidden;
  if (ld_y == 0) ld_y = n_out;
  if (ld_x < hidden || ld_w < hidden || ld_y < n_out)
    return fail(GDN_ERR_ARG, "row strides smaller than a row");
  const size_t ye = dtype_size(y_dtype);
  if ((uintptr_t)x % 16 || (uintptr_t)w % 16 || (uintptr_t)y % 16 || (ld_x * 2) % 16 ||
      (ld_w * 2) % 16 || (ld_y * (int64_t)ye) % 16)
    return fail(GDN_ERR_ARG, "x, w and y rows must start 16-byte aligned (pointers and strides)");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->desc.host_checks) {
    if ((st = check_device_ptr(x, "x")) || (st = check_device_ptr(w, "w")) ||
        (st = check_device_ptr(y, "y")))
      return st;
  }
  const cudaError_t e = gdn::launch_in_proj(tokens, n_out, hidden, x, ld_x, w, ld_w, y, ld_y,
                                            y_dtype, p->view.err, p->sm_count, s);
  if (e == cudaErrorInvalidValue)
    return fail(GDN_ERR_UNSUPPORTED, "no tensor map for these operands (driver entry point)");
  if (e != cudaSuccess) return cuda_fail(e, "input projection launch");
  return ok();
}

gdn_status gdn_gated_rmsnorm(int64_t rows, int32_t d, const void *o, gdn_dtype o_dtype,
                             const void *z, gdn_dtype z_dtype, const float *w, float eps,
                             void *y, gdn_dtype y_dtype, gdn_stream stream) {
  if (rows < 0) return fail(GDN_ERR_ARG, "rows = %lld < 0", (long long)rows);
  if (d < 1) return fail(GDN_ERR_ARG, "d = %d < 1", d);
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(GDN_ERR_ARG, "eps must be finite and >= 0");
  if (!dtype_ok(o_dtype) || !dtype_ok(z_dtype) || !dtype_ok(y_dtype))
    return fail(GDN_ERR_DTYPE, "o, z and y dtypes must be F32 or BF16");
  if (rows == 0) return ok();
  if (!o || !z || !w || !y) return fail(GDN_ERR_ARG, "o, z, w and y must be non-NULL");
  if (rows > INT64_MAX / d) return fail(GDN_ERR_SIZE, "rows * d overflows");
  cudaError_t e = gdn::launch_gated_rmsnorm(o, o_dtype, z, z_dtype, w, eps, y, y_dtype, rows, d,
                                            reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gated RMSNorm launch");
  return ok();
}

namespace {

// A verify launch with its drafts staged in a stream-ordered workspace (the
// tensor-core path, when the pool's memory pool grants it within
// prefill_workspace_max; otherwise each block stages its own drafts).
cudaError_t verify_with_stage(gdn_pool *p, int32_t layer, gdn::VerifyArgs &va, void *o,
                              gdn_dtype o_dtype, cudaStream_t s) {
  void *stage = nullptr;
  const uint64_t lim = p->desc.prefill_workspace_max ? p->desc.prefill_workspace_max
                                                     : (uint64_t)8 << 30;
  const size_t sb = p->has_tmap ? gdn::verify_stage_workspace_bytes(p->view, va) : 0;
  if (sb > 0 && sb <= lim && cudaMallocFromPoolAsync(&stage, sb, p->work_pool, s) != cudaSuccess) {
    cudaGetLastError();
    stage = nullptr;
  }
  va.stage = static_cast<float *>(stage);
  cudaError_t e =
      gdn::launch_verify(p->view, p->has_tmap ? &p->tmap : nullptr, layer, va, o, o_dtype, s);
  if (stage != nullptr) {
    const cudaError_t ef = cudaFreeAsync(stage, s);
    if (e == cudaSuccess) e = ef;
  }
  return e;
}

}  // namespace

gdn_status gdn_spec_verify(gdn_pool *p, int32_t layer, const int32_t *slot_ids, int32_t n,
                           int32_t T, const gdn_qkv *in, void *o, gdn_dtype o_dtype,
                           const int32_t *accept_len, float scale, gdn_stream stream) {
  gdn_status st = check_pool(p, layer);
  if (st != GDN_OK) return st;
  if (n < 0) return fail(GDN_ERR_ARG, "n = %d < 0", n);
  if (T < 1 || T > gdn::kMaxVerifyT)
    return fail(GDN_ERR_SIZE, "T = %d outside [1, %d]", T, gdn::kMaxVerifyT);
  if (!o && !accept_len) return fail(GDN_ERR_ARG, "o and accept_len are both NULL");
  if (n == 0) return ok();
  if (n > 65535) return fail(GDN_ERR_SIZE, "n = %d > 65535", n);
  if (!slot_ids) return fail(GDN_ERR_ARG, "slot_ids is NULL");
  if (!dtype_ok(o_dtype)) return fail(GDN_ERR_DTYPE, "o dtype must be F32 or BF16");
  gdn::QKV q;
  if ((st = resolve_qkv(p, in, (int64_t)n * T, q))) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->desc.host_checks) {
    if ((st = check_slots(p, slot_ids, n, s))) return st;
    if (accept_len && (st = check_counts(accept_len, n, nullptr, T, s, "accept_len"))) return st;
    if (o && (st = check_device_ptr(o, "o"))) return st;
  }
  gdn::VerifyArgs va{slot_ids, n, T, q, accept_len, 0, gdn::QKV{}, 0, nullptr, scale, nullptr};
  const cudaError_t e = verify_with_stage(p, layer, va, o, o_dtype, s);
  if (e != cudaSuccess) return cuda_fail(e, "verify launch");
  return ok();
}

gdn_status gdn_spec_verify_deferred(gdn_pool *p, int32_t layer, const int32_t *slot_ids,
                                    int32_t n, int32_t T, const gdn_qkv *in, void *o,
                                    gdn_dtype o_dtype, int32_t T_prev, const gdn_qkv *prev,
                                    const int32_t *prev_accept, float scale, gdn_stream stream) {
  gdn_status st = check_pool(p, layer);
  if (st != GDN_OK) return st;
  if (n < 0) return fail(GDN_ERR_ARG, "n = %d < 0", n);
  if (T < 1 || T_prev < 0 || T + T_prev > gdn::kMaxVerifyT)
    return fail(GDN_ERR_SIZE, "T = %d, T_prev = %d: need T >= 1, T_prev >= 0, T + T_prev <= %d",
                T, T_prev, gdn::kMaxVerifyT);
  if (!o) return fail(GDN_ERR_ARG, "o is NULL");
  if (n == 0) return ok();
  if (n > 65535) return fail(GDN_ERR_SIZE, "n = %d > 65535", n);
  if (!slot_ids) return fail(GDN_ERR_ARG, "slot_ids is NULL");
  if (!dtype_ok(o_dtype)) return fail(GDN_ERR_DTYPE, "o dtype must be F32 or BF16");
  const bool pending = prev != nullptr && prev_accept != nullptr && T_prev > 0;
  if ((prev != nullptr) != (prev_accept != nullptr))
    return fail(GDN_ERR_ARG, "prev and prev_accept must both be set or both be NULL");
  gdn::QKV q, qp{};
  if ((st = resolve_qkv(p, in, (int64_t)n * T, q))) return st;
  if (pending) {
    if ((st = resolve_qkv(p, prev, (int64_t)n * T_prev, qp))) return st;
    if (qp.dtype != q.dtype) return fail(GDN_ERR_DTYPE, "prev and in must share one dtype");
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->desc.host_checks) {
    if ((st = check_slots(p, slot_ids, n, s)) || (st = check_device_ptr(o, "o"))) return st;
    if (pending && (st = check_counts(prev_accept, n, nullptr, T_prev, s, "prev_accept")))
      return st;
  }
  gdn::VerifyArgs va{slot_ids, n, T, q, nullptr, 0, pending ? qp : gdn::QKV{},
                     pending ? T_prev : 0, pending ? prev_accept : nullptr, scale, nullptr};
  const cudaError_t e = verify_with_stage(p, layer, va, o, o_dtype, s);
  if (e != cudaSuccess) return cuda_fail(e, "deferred verify launch");
  return ok();
}

namespace {

gdn_status prefill_common(gdn_pool *p, int32_t layer, const int32_t *slot_ids,
                          const int32_t *cu_seqlens, int32_t n_seqs, int32_t total_tokens,
                          int32_t max_seqlen, const gdn_qkv *in, void *o, gdn_dtype o_dtype,
                          float scale, gdn_stream stream, bool chunked) {
  gdn_status st = check_pool(p, layer);
  if (st != GDN_OK) return st;
  if (n_seqs < 0 || total_tokens < 0) return fail(GDN_ERR_ARG, "negative n_seqs/total_tokens");
  if (n_seqs == 0 || total_tokens == 0) return ok();
  if (n_seqs > 65535) return fail(GDN_ERR_SIZE, "n_seqs = %d > 65535", n_seqs);
  if (!slot_ids || !cu_seqlens || !o)
    return fail(GDN_ERR_ARG, "slot_ids, cu_seqlens and o must be non-NULL");
  if (!dtype_ok(o_dtype)) return fail(GDN_ERR_DTYPE, "o dtype must be F32 or BF16");
  gdn::QKV q;
  if ((st = resolve_qkv(p, in, total_tokens, q))) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->desc.host_checks) {
    std::vector<int32_t> cu;
    if ((st = check_slots(p, slot_ids, n_seqs, s)) ||
        (st = check_cu(cu_seqlens, n_seqs, total_tokens, s, cu)) ||
        (st = check_device_ptr(o, "o")))
      return st;
  }
  gdn::SeqIndex seq{slot_ids, cu_seqlens, n_seqs, total_tokens};
  cudaError_t e;
  if (chunked) {
    // the two-launch path keeps per-chunk tiles in a stream-ordered workspace;
    // without one (allocation refused) the single-launch kernel runs instead
    void *work = nullptr;
    const uint64_t lim = p->desc.prefill_workspace_max ? p->desc.prefill_workspace_max
                                                       : (uint64_t)8 << 30;
    const size_t wb = gdn::prefill_workspace_bytes(p->view, seq, q, (size_t)lim);
    if (wb > 0 && cudaMallocFromPoolAsync(&work, wb, p->work_pool, s) != cudaSuccess) {
      cudaGetLastError();
      work = nullptr;
    }
    e = gdn::launch_prefill(p->view, layer, seq, q, o, o_dtype, scale, work, s);
    if (work != nullptr) {
      const cudaError_t ef = cudaFreeAsync(work, s);
      if (e == cudaSuccess) e = ef;
    }
  } else {
    e = gdn::launch_prefill_recurrent(p->view, layer, seq, q, o, o_dtype, scale, s);
  }
  if (e == cudaErrorNotSupported)
    return fail(GDN_ERR_UNSUPPORTED, "prefill is not available for this shape");
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return ok();
}

}  // namespace

gdn_status gdn_prefill_chunked(gdn_pool *p, int32_t layer, const int32_t *slot_ids,
                               const int32_t *cu_seqlens, int32_t n_seqs, int32_t total_tokens,
                               int32_t max_seqlen, const gdn_qkv *in, void *o, gdn_dtype o_dtype,
                               float scale, gdn_stream stream) {
  return prefill_common(p, layer, slot_ids, cu_seqlens, n_seqs, total_tokens, max_seqlen, in, o,
                        o_dtype, scale, stream, true);
}

gdn_status gdn_prefill_chunked_ckpt(gdn_pool *p, int32_t layer, const int32_t *slot_ids,
                                    const int32_t *cu_seqlens, int32_t n_seqs,
                                    int32_t total_tokens, int32_t max_seqlen, const gdn_qkv *in,
                                    void *o, gdn_dtype o_dtype, float scale,
                                    const int32_t *ckpt_slots, int32_t ckpt_per_seq,
                                    int32_t ckpt_every, gdn_stream stream) {
  (void)max_seqlen;
  gdn_status st = check_pool(p, layer);
  if (st != GDN_OK) return st;
  if (n_seqs < 0 || total_tokens < 0) return fail(GDN_ERR_ARG, "negative n_seqs/total_tokens");
  if (n_seqs == 0 || total_tokens == 0) return ok();
  if (n_seqs > 65535) return fail(GDN_ERR_SIZE, "n_seqs = %d > 65535", n_seqs);
  if (!slot_ids || !cu_seqlens || !o || !ckpt_slots)
    return fail(GDN_ERR_ARG, "slot_ids, cu_seqlens, o and ckpt_slots must be non-NULL");
  if (ckpt_every < gdn::kChunk || ckpt_every % gdn::kChunk != 0 || ckpt_per_seq < 1)
    return fail(GDN_ERR_ARG, "ckpt_every = %d must be a positive multiple of %d, ckpt_per_seq = %d >= 1",
                ckpt_every, gdn::kChunk, ckpt_per_seq);
  if (!dtype_ok(o_dtype)) return fail(GDN_ERR_DTYPE, "o dtype must be F32 or BF16");
  gdn::QKV q;
  if ((st = resolve_qkv(p, in, total_tokens, q))) return st;
  gdn::SeqIndex seq{slot_ids, cu_seqlens, n_seqs, total_tokens};
  const uint64_t lim = p->desc.prefill_workspace_max ? p->desc.prefill_workspace_max
                                                     : (uint64_t)8 << 30;
  const size_t wb = gdn::prefill_workspace_bytes(p->view, seq, q, (size_t)lim);
  if (wb == 0)
    return fail(GDN_ERR_UNSUPPORTED,
                "checkpoints need the two-launch path: dk = dv = 128, 16-byte aligned v rows "
                "and a workspace within prefill_workspace_max");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->desc.host_checks) {
    std::vector<int32_t> cu, act, ck;
    if ((st = check_slots(p, slot_ids, n_seqs, s)) ||
        (st = check_cu(cu_seqlens, n_seqs, total_tokens, s, cu)) ||
        (st = check_device_ptr(o, "o")) || (st = fetch(act, slot_ids, (size_t)n_seqs, s, "slot_ids")) ||
        (st = fetch(ck, ckpt_slots, (size_t)n_seqs * ckpt_per_seq, s, "ckpt_slots")))
      return st;
    std::vector<char> used((size_t)p->desc.n_slots, 0);
    for (int32_t a : act) used[(size_t)a] = 1;
    for (size_t e = 0; e < ck.size(); ++e) {
      const int32_t d = ck[e];
      if (d < 0) continue;
      if (d >= p->desc.n_slots)
        return fail(GDN_ERR_SLOT, "ckpt_slots[%zu] = %d outside [0, %d)", e, d, p->desc.n_slots);
      if (used[(size_t)d])
        return fail(GDN_ERR_DUP_SLOT, "ckpt_slots[%zu] = %d is an active or repeated slot", e, d);
      used[(size_t)d] = 1;
    }
  }
  void *work = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&work, wb, p->work_pool, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "prefill workspace");
  }
  gdn::Checkpoints ck{ckpt_slots, ckpt_per_seq, ckpt_every};
  e = gdn::launch_prefill_split(p->view, layer, seq, q, o, o_dtype, scale, work, s, ck);
  const cudaError_t ef = cudaFreeAsync(work, s);
  if (e == cudaSuccess) e = ef;
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return ok();
}

gdn_status gdn_prefill_recurrent(gdn_pool *p, int32_t layer, const int32_t *slot_ids,
                                 const int32_t *cu_seqlens, int32_t n_seqs, int32_t total_tokens,
                                 int32_t max_seqlen, const gdn_qkv *in, void *o,
                                 gdn_dtype o_dtype, float scale, gdn_stream stream) {
  return prefill_common(p, layer, slot_ids, cu_seqlens, n_seqs, total_tokens, max_seqlen, in, o,
                        o_dtype, scale, stream, false);
}

}  // extern "C"

// ------------------------------------------------------------------
// Chunked prefill that allocates no device memory: the two-launch path's
// workspace lives in one file-scope device array, shared by every call.

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)64 << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_prefill_scratch[kNoAllocScratchBytes];

// The array's device address on the current device, looked up on every call
// (cheap once the module is loaded, and never stale after a context reset).
// In host code the array's name is only a stand-in, never a pointer a kernel
// may be given.
cudaError_t noalloc_scratch(void **out) {
  return cudaGetSymbolAddress(out, g_prefill_scratch);
}

}  // namespace

extern "C" {

gdn_status gdn_prefill_chunked_noalloc(gdn_pool *p, int32_t layer, const int32_t *slot_ids,
                                       const int32_t *cu_seqlens, int32_t n_seqs,
                                       int32_t total_tokens, int32_t max_seqlen,
                                       const gdn_qkv *in, void *o, gdn_dtype o_dtype, float scale,
                                       gdn_stream stream) {
  (void)max_seqlen;
  gdn_status st = check_pool(p, layer);
  if (st != GDN_OK) return st;
  if (n_seqs < 0 || total_tokens < 0) return fail(GDN_ERR_ARG, "negative n_seqs/total_tokens");
  if (n_seqs == 0 || total_tokens == 0) return ok();
  if (n_seqs > 65535) return fail(GDN_ERR_SIZE, "n_seqs = %d > 65535", n_seqs);
  if (!slot_ids || !cu_seqlens || !o)
    return fail(GDN_ERR_ARG, "slot_ids, cu_seqlens and o must be non-NULL");
  if (!dtype_ok(o_dtype)) return fail(GDN_ERR_DTYPE, "o dtype must be F32 or BF16");
  gdn::QKV q;
  if ((st = resolve_qkv(p, in, total_tokens, q))) return st;
  gdn::SeqIndex seq{slot_ids, cu_seqlens, n_seqs, total_tokens};
  // no workspace limit here: the check below is against the fixed array
  const size_t wb = gdn::prefill_workspace_bytes(p->view, seq, q, (size_t)-1);
  if (wb > kNoAllocScratchBytes)
    return fail(GDN_ERR_SIZE,
                "prefill needs %zu bytes of scratch, more than the %zu-byte array of "
                "gdn_prefill_chunked_noalloc (%d value heads, %d tokens, %d sequences); split "
                "the call into fewer tokens",
                wb, kNoAllocScratchBytes, p->desc.h_v, total_tokens, n_seqs);
  void *work = nullptr;
  if (wb > 0) {
    const cudaError_t e = noalloc_scratch(&work);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(prefill scratch)");
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->desc.host_checks) {
    std::vector<int32_t> cu;
    if ((st = check_slots(p, slot_ids, n_seqs, s)) ||
        (st = check_cu(cu_seqlens, n_seqs, total_tokens, s, cu)) ||
        (st = check_device_ptr(o, "o")))
      return st;
  }
  const cudaError_t e = gdn::launch_prefill(p->view, layer, seq, q, o, o_dtype, scale, work, s);
  if (e == cudaErrorNotSupported)
    return fail(GDN_ERR_UNSUPPORTED, "prefill is not available for this shape");
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return ok();
}

}  // extern "C"
