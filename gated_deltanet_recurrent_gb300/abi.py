"""Thin Python binding of libgdn's C ABI (include/gdn.h).

Argument marshalling only: torch tensors supply device memory and the
current CUDA stream; every step of the computation runs in libgdn's CUDA
kernels.  The functions carry the C names.  If libgdn.so has not been built
the first call raises -- there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn.so")

GDN_F32, GDN_BF16, GDN_F16 = 0, 1, 2
STATUS = {0: "GDN_OK", 1: "GDN_ERR_ARG", 2: "GDN_ERR_SLOT", 3: "GDN_ERR_DUP_SLOT",
          4: "GDN_ERR_DTYPE", 5: "GDN_ERR_SIZE", 6: "GDN_ERR_UNSUPPORTED", 7: "GDN_ERR_CUDA"}
DEVERR_SLOT, DEVERR_SEQ, DEVERR_COUNT, DEVERR_TIMEOUT = 1, 2, 4, 8
TEST_DECODE_WAIT_TIMEOUT = 1

EXPORTED = ("gdn_pool_state_bytes", "gdn_pool_conv_bytes", "gdn_pool_create", "gdn_pool_reset",
            "gdn_pool_copy",
            "gdn_pool_destroy", "gdn_pool_get_error", "gdn_pool_set_test_flags", "gdn_conv_silu",
            "gdn_decode_step",
            "gdn_decode_step_conv", "gdn_decode_step_conv_launches", "gdn_gated_rmsnorm",
            "gdn_in_proj",
            "gdn_prefill_chunked", "gdn_prefill_recurrent", "gdn_spec_verify",
            "gdn_spec_verify_deferred", "gdn_prefill_chunked_noalloc", "gdn_prefill_chunked_ckpt",
            "gdn_status_string",
            "gdn_last_error_message")


class GDNError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.name = STATUS.get(status, str(status))


class gdn_pool_desc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_slots", ctypes.c_int32),
                ("h_v", ctypes.c_int32), ("h_k", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("conv_ch", ctypes.c_int32), ("conv_k", ctypes.c_int32),
                ("conv_dtype", ctypes.c_int), ("host_checks", ctypes.c_int32),
                ("prefill_workspace_max", ctypes.c_uint64), ("state_dtype", ctypes.c_int)]


class gdn_qkv(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p),
                ("ld_qk", ctypes.c_int64), ("ld_v", ctypes.c_int64), ("dtype", ctypes.c_int)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgdn.so (once).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libgdn.so not found at {path}; build it with "
                           "`python -m gated_deltanet_recurrent_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, i64, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int
    P = ctypes.POINTER
    sig = {
        "gdn_pool_state_bytes": (ctypes.c_size_t, [P(gdn_pool_desc)]),
        "gdn_pool_conv_bytes": (ctypes.c_size_t, [P(gdn_pool_desc)]),
        "gdn_pool_create": (st, [P(gdn_pool_desc), vp, ctypes.c_size_t, vp, ctypes.c_size_t,
                                 P(vp)]),
        "gdn_pool_reset": (st, [vp, vp, i32, vp]),
        "gdn_pool_copy": (st, [vp, vp, vp, i32, vp]),
        "gdn_pool_destroy": (st, [vp]),
        "gdn_pool_get_error": (st, [vp, P(ctypes.c_uint32)]),
        "gdn_pool_set_test_flags": (st, [vp, ctypes.c_uint32]),
        "gdn_conv_silu": (st, [vp, i32, vp, vp, i32, i32, i32, vp, i64, st, vp, vp, vp, i64,
                               vp, vp]),
        "gdn_decode_step": (st, [vp, i32, vp, i32, P(gdn_qkv), vp, st, ctypes.c_float, vp]),
        "gdn_decode_step_conv": (st, [vp, i32, vp, i32, vp, i64, vp, vp, vp, i64, vp, vp, st,
                                      vp, st, ctypes.c_float, vp]),
        "gdn_decode_step_conv_launches": (st, [vp, i32, st, st, P(i32)]),
        "gdn_gated_rmsnorm": (st, [i64, i32, vp, st, vp, st, vp, ctypes.c_float, vp, st, vp]),
        "gdn_in_proj": (st, [vp, i64, i32, i32, vp, i64, vp, i64, vp, i64, st, vp]),
        "gdn_prefill_chunked": (st, [vp, i32, vp, vp, i32, i32, i32, P(gdn_qkv), vp, st,
                                     ctypes.c_float, vp]),
        "gdn_prefill_recurrent": (st, [vp, i32, vp, vp, i32, i32, i32, P(gdn_qkv), vp, st,
                                       ctypes.c_float, vp]),
        "gdn_spec_verify": (st, [vp, i32, vp, i32, i32, P(gdn_qkv), vp, st, vp,
                                 ctypes.c_float, vp]),
        "gdn_spec_verify_deferred": (st, [vp, i32, vp, i32, i32, P(gdn_qkv), vp, st, i32,
                                          P(gdn_qkv), vp, ctypes.c_float, vp]),
        "gdn_prefill_chunked_noalloc": (st, [vp, i32, vp, vp, i32, i32, i32, P(gdn_qkv), vp, st,
                                             ctypes.c_float, vp]),
        "gdn_prefill_chunked_ckpt": (st, [vp, i32, vp, vp, i32, i32, i32, P(gdn_qkv), vp, st,
                                          ctypes.c_float, vp, i32, i32, vp]),
        "gdn_status_string": (ctypes.c_char_p, [st]),
        "gdn_last_error_message": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        msg = load_library().gdn_last_error_message().decode()
        raise GDNError(status, msg)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GDN_F32
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    raise GDNError(4, f"unsupported dtype {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _idx(t: Optional[torch.Tensor], name: str):
    if t is None:
        return None
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise GDNError(1, f"{name} must be a contiguous int32 tensor")
    return _ptr(t)


def _token_rows(t: torch.Tensor, heads: int, dim: int, name: str) -> int:
    """Token stride (elements) of a [tokens, heads, dim] view whose heads are packed."""
    if t.dim() != 3 or t.shape[1] != heads or t.shape[2] != dim:
        raise GDNError(5, f"{name} must be [tokens, {heads}, {dim}], got {tuple(t.shape)}")
    if t.stride(2) != 1 or t.stride(1) != dim:
        raise GDNError(1, f"{name}: heads must be packed (strides {t.stride()})")
    return t.stride(0)


def _qkv(pool: "Pool", q, k, v, g, beta) -> gdn_qkv:
    d = pool.desc
    ld_q = _token_rows(q, d.h_k, d.dk, "q")
    ld_k = _token_rows(k, d.h_k, d.dk, "k")
    ld_v = _token_rows(v, d.h_v, d.dv, "v")
    if ld_q != ld_k:
        raise GDNError(1, "q and k must share one token stride")
    for name, t in (("g", g), ("beta", beta)):
        if t.shape != (q.shape[0], d.h_v) or not t.is_contiguous():
            raise GDNError(5, f"{name} must be contiguous [tokens, {d.h_v}]")
    dts = {_dt(t) for t in (q, k, v, g, beta)}
    if len(dts) != 1:
        raise GDNError(4, "q, k, v, g and beta must share one dtype")
    return gdn_qkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(),
                   ld_q, ld_v, dts.pop())


_STATE_DTYPES = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16, torch.float16: GDN_F16}


class Pool:
    """A pool handle plus the torch tensors holding its state and conv cache:
    state [n_layers, n_slots, h_v, dv, dk] in state_dtype (float32, or
    bfloat16 / float16 storage), conv [n_layers, n_slots, conv_ch, conv_k-1]
    in conv_dtype.  Both start at zero."""

    def __init__(self, n_layers, n_slots, h_v, h_k, dk, dv, conv_ch, conv_k,
                 conv_dtype=torch.bfloat16, host_checks=True, device="cuda",
                 prefill_workspace_max=0, state_dtype=torch.float32):
        if state_dtype not in _STATE_DTYPES:
            raise GDNError(4, f"unsupported state dtype {state_dtype}")
        self.desc = gdn_pool_desc(n_layers, n_slots, h_v, h_k, dk, dv, conv_ch, conv_k,
                                  GDN_F32 if conv_dtype == torch.float32 else GDN_BF16,
                                  1 if host_checks else 0, prefill_workspace_max,
                                  _STATE_DTYPES[state_dtype])
        self.state = torch.zeros((n_layers, n_slots, h_v, dv, dk), dtype=state_dtype,
                                 device=device)
        self.conv = torch.zeros((n_layers, n_slots, conv_ch, conv_k - 1), dtype=conv_dtype,
                                device=device)
        self.handle = gdn_pool_create(self.desc, self.state, self.conv)

    @classmethod
    def for_shape(cls, shape, n_layers, n_slots, conv_dtype=torch.bfloat16, host_checks=True,
                  device="cuda", prefill_workspace_max=0, state_dtype=torch.float32):
        return cls(n_layers, n_slots, shape.h_v, shape.h_k, shape.dk, shape.dv,
                   shape.conv_ch, shape.conv_k, conv_dtype, host_checks, device,
                   prefill_workspace_max, state_dtype)

    def set_host_checks(self, on: bool):
        """Recreate the handle with host checks switched on or off (same memory)."""
        self.close()
        self.desc.host_checks = 1 if on else 0
        self.handle = gdn_pool_create(self.desc, self.state, self.conv)

    def close(self):
        if getattr(self, "handle", None):
            gdn_pool_destroy(self)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# --------------------------------------------------------------- entry points

def gdn_pool_state_bytes(desc: gdn_pool_desc) -> int:
    return load_library().gdn_pool_state_bytes(ctypes.byref(desc))


def gdn_pool_conv_bytes(desc: gdn_pool_desc) -> int:
    return load_library().gdn_pool_conv_bytes(ctypes.byref(desc))


def gdn_pool_create(desc: gdn_pool_desc, state: torch.Tensor, conv: torch.Tensor):
    lib = load_library()
    out = ctypes.c_void_p()
    _check(lib.gdn_pool_create(ctypes.byref(desc), _ptr(state),
                               state.numel() * state.element_size(), _ptr(conv),
                               conv.numel() * conv.element_size(), ctypes.byref(out)))
    return out


def gdn_pool_destroy(pool: Pool):
    _check(load_library().gdn_pool_destroy(pool.handle))


def gdn_pool_reset(pool: Pool, slot_ids: torch.Tensor, stream=None):
    _check(load_library().gdn_pool_reset(pool.handle, _idx(slot_ids, "slot_ids"),
                                         slot_ids.numel(), _stream(stream)))


def gdn_pool_copy(pool: Pool, src_slots: torch.Tensor, dst_slots: torch.Tensor, stream=None):
    if src_slots.numel() != dst_slots.numel():
        raise GDNError(5, "src_slots and dst_slots differ in length")
    _check(load_library().gdn_pool_copy(pool.handle, _idx(src_slots, "src_slots"),
                                        _idx(dst_slots, "dst_slots"), src_slots.numel(),
                                        _stream(stream)))


def gdn_pool_get_error(pool: Pool) -> int:
    err = ctypes.c_uint32(0)
    _check(load_library().gdn_pool_get_error(pool.handle, ctypes.byref(err)))
    return err.value


def gdn_pool_set_test_flags(pool: Pool, flags: int):
    """Test hook of the C ABI (see gdn.h); 0 restores normal operation."""
    _check(load_library().gdn_pool_set_test_flags(pool.handle, flags))


def gdn_conv_silu(pool: Pool, layer: int, slot_ids: torch.Tensor, x: torch.Tensor,
                  w: torch.Tensor, y: Optional[torch.Tensor] = None,
                  cu_seqlens: Optional[torch.Tensor] = None, bias=None, advance=None,
                  max_seqlen: int = 0, stream=None):
    """x, y [tokens, conv_ch] (row stride may exceed conv_ch); w [conv_ch, conv_k] float32."""
    n = slot_ids.numel()
    if w.dtype != torch.float32 or not w.is_contiguous():
        raise GDNError(1, "w must be contiguous float32 [conv_ch, conv_k]")
    if x.dim() != 2 or x.stride(1) != 1 or (y is not None and y.stride(1) != 1):
        raise GDNError(1, "x and y must be [tokens, channels] with unit channel stride")
    if max_seqlen <= 0:
        max_seqlen = x.shape[0]
    _check(load_library().gdn_conv_silu(
        pool.handle, layer, _idx(slot_ids, "slot_ids"), _idx(cu_seqlens, "cu_seqlens"), n,
        x.shape[0], max_seqlen, _ptr(x), x.stride(0), _dt(x), _ptr(w), _ptr(bias), _ptr(y),
        0 if y is None else y.stride(0), _idx(advance, "advance"), _stream(stream)))
    return y


def gdn_decode_step(pool: Pool, layer: int, slot_ids: torch.Tensor, q, k, v, g, beta,
                    o: torch.Tensor, scale: float = 1.0, stream=None):
    """q, k [n, h_k, dk]; v [n, h_v, dv]; g, beta [n, h_v]; o [n, h_v, dv]."""
    inp = _qkv(pool, q, k, v, g, beta)
    _check(load_library().gdn_decode_step(pool.handle, layer, _idx(slot_ids, "slot_ids"),
                                          slot_ids.numel(), ctypes.byref(inp), _ptr(o),
                                          _dt(o), scale, _stream(stream)))
    return o


def gdn_decode_step_conv(pool: Pool, layer: int, slot_ids: torch.Tensor, x: torch.Tensor,
                         w: torch.Tensor, y: torch.Tensor, g, beta, o: torch.Tensor, bias=None,
                         scale: float = 1.0, stream=None):
    """conv + SiLU then the decode step in one call.  x, y [n, conv_ch] (row
    stride may exceed conv_ch; y is split into q | k | v); w [conv_ch, conv_k]
    float32; g, beta [n, h_v] in x's dtype; o [n, h_v, dv]."""
    n = slot_ids.numel()
    if w.dtype != torch.float32 or not w.is_contiguous():
        raise GDNError(1, "w must be contiguous float32 [conv_ch, conv_k]")
    for name, t in (("x", x), ("y", y)):
        if t.dim() != 2 or t.stride(1) != 1 or t.shape[0] != n:
            raise GDNError(1, f"{name} must be [n, channels] with unit channel stride")
    for name, t in (("g", g), ("beta", beta)):
        if t.shape != (n, pool.desc.h_v) or not t.is_contiguous():
            raise GDNError(5, f"{name} must be contiguous [n, {pool.desc.h_v}]")
    dts = {_dt(t) for t in (x, y, g, beta)}
    if len(dts) != 1:
        raise GDNError(4, "x, y, g and beta must share one dtype")
    _check(load_library().gdn_decode_step_conv(
        pool.handle, layer, _idx(slot_ids, "slot_ids"), n, _ptr(x), x.stride(0), _ptr(w),
        _ptr(bias), _ptr(y), y.stride(0), _ptr(g), _ptr(beta), dts.pop(), _ptr(o), _dt(o), scale,
        _stream(stream)))
    return o


def gdn_decode_step_conv_launches(pool: Pool, n: int, dtype: torch.dtype,
                                  o_dtype: torch.dtype = torch.float32) -> int:
    """Kernel launches gdn_decode_step_conv makes for n slots (1 or 2; 0 if n = 0)."""
    codes = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16, torch.float16: GDN_F16}
    out = ctypes.c_int32(-1)
    _check(load_library().gdn_decode_step_conv_launches(pool.handle, n, codes[dtype],
                                                         codes[o_dtype], ctypes.byref(out)))
    return out.value


def gdn_in_proj(pool: Pool, x: torch.Tensor, w: torch.Tensor,
                y: Optional[torch.Tensor] = None, stream=None):
    """y = x w^T: x [tokens, hidden] bf16, w [n_out, hidden] bf16 (unit
    column strides), y [tokens, n_out] float32 or bf16 (default float32)."""
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
        raise GDNError(4, "x and w must be bf16")
    if x.dim() != 2 or w.dim() != 2 or x.stride(1) != 1 or w.stride(1) != 1 or \
            x.shape[1] != w.shape[1]:
        raise GDNError(1, "x [tokens, hidden] and w [n_out, hidden] with unit column strides")
    if y is None:
        y = torch.empty(x.shape[0], w.shape[0], dtype=torch.float32, device=x.device)
    if y.dim() != 2 or y.stride(1) != 1 or tuple(y.shape) != (x.shape[0], w.shape[0]):
        raise GDNError(1, "y must be [tokens, n_out] with a unit column stride")
    _check(load_library().gdn_in_proj(pool.handle, x.shape[0], x.shape[1], w.shape[0], _ptr(x),
                                      x.stride(0), _ptr(w), w.stride(0), _ptr(y), y.stride(0),
                                      _dt(y), _stream(stream)))
    return y


def gdn_gated_rmsnorm(o: torch.Tensor, z: torch.Tensor, w: torch.Tensor,
                      y: Optional[torch.Tensor] = None, eps: float = 1e-6, stream=None):
    """Output gated RMSNorm over the last axis: o, z, y [..., d] contiguous
    (each float32 or bf16; y defaults to float32), w [d] float32."""
    d = o.shape[-1]
    if y is None:
        y = torch.empty(o.shape, dtype=torch.float32, device=o.device)
    for name, t in (("o", o), ("z", z), ("y", y)):
        if t.shape != o.shape or not t.is_contiguous():
            raise GDNError(1, f"{name} must be contiguous with o's shape {tuple(o.shape)}")
    if w.dtype != torch.float32 or not w.is_contiguous() or w.numel() != d:
        raise GDNError(1, f"w must be contiguous float32 [{d}]")
    _check(load_library().gdn_gated_rmsnorm(o.numel() // max(d, 1), d, _ptr(o), _dt(o), _ptr(z),
                                            _dt(z), _ptr(w), eps, _ptr(y), _dt(y),
                                            _stream(stream)))
    return y


def gdn_prefill_chunked(pool: Pool, layer: int, slot_ids: torch.Tensor,
                        cu_seqlens: torch.Tensor, q, k, v, g, beta, o: torch.Tensor,
                        scale: float = 1.0, max_seqlen: int = 0, stream=None):
    """Packed varlen tokens: q, k [T, h_k, dk]; v [T, h_v, dv]; o [T, h_v, dv]."""
    inp = _qkv(pool, q, k, v, g, beta)
    if max_seqlen <= 0:
        max_seqlen = q.shape[0]
    _check(load_library().gdn_prefill_chunked(
        pool.handle, layer, _idx(slot_ids, "slot_ids"), _idx(cu_seqlens, "cu_seqlens"),
        slot_ids.numel(), q.shape[0], max_seqlen, ctypes.byref(inp), _ptr(o), _dt(o), scale,
        _stream(stream)))
    return o


def gdn_prefill_recurrent(pool: Pool, layer: int, slot_ids: torch.Tensor,
                          cu_seqlens: torch.Tensor, q, k, v, g, beta, o: torch.Tensor,
                          scale: float = 1.0, max_seqlen: int = 0, stream=None):
    """Token-by-token prefill; same arguments and results as gdn_prefill_chunked."""
    inp = _qkv(pool, q, k, v, g, beta)
    if max_seqlen <= 0:
        max_seqlen = q.shape[0]
    _check(load_library().gdn_prefill_recurrent(
        pool.handle, layer, _idx(slot_ids, "slot_ids"), _idx(cu_seqlens, "cu_seqlens"),
        slot_ids.numel(), q.shape[0], max_seqlen, ctypes.byref(inp), _ptr(o), _dt(o), scale,
        _stream(stream)))
    return o


def gdn_spec_verify(pool: Pool, layer: int, slot_ids: torch.Tensor, T: int, q, k, v, g, beta,
                    o: Optional[torch.Tensor] = None,
                    accept_len: Optional[torch.Tensor] = None, scale: float = 1.0,
                    stream=None):
    """Draft t of slot i is token i*T + t; o [n, T, h_v, dv] (or None)."""
    inp = _qkv(pool, q, k, v, g, beta)
    o_dt = GDN_F32 if o is None else _dt(o)
    _check(load_library().gdn_spec_verify(
        pool.handle, layer, _idx(slot_ids, "slot_ids"), slot_ids.numel(), T,
        ctypes.byref(inp), _ptr(o), o_dt, _idx(accept_len, "accept_len"), scale,
        _stream(stream)))
    return o


def gdn_spec_verify_deferred(pool: Pool, layer: int, slot_ids: torch.Tensor, T: int, q, k, v, g,
                             beta, o: torch.Tensor, prev=None,
                             prev_accept: Optional[torch.Tensor] = None, scale: float = 1.0,
                             stream=None):
    """Commit the first prev_accept[i] of last round's drafts, then output this
    round's T drafts without committing them.  prev = (q, k, v, g, beta) of
    last round ([n*T_prev, ...] each) or None; o [n, T, h_v, dv]."""
    inp = _qkv(pool, q, k, v, g, beta)
    n = slot_ids.numel()
    T_prev, pin = 0, None
    if prev is not None:
        pin = _qkv(pool, *prev)
        if n == 0 or prev[0].shape[0] % n:
            raise GDNError(5, "prev holds no whole number of drafts per slot")
        T_prev = prev[0].shape[0] // n
    _check(load_library().gdn_spec_verify_deferred(
        pool.handle, layer, _idx(slot_ids, "slot_ids"), n, T, ctypes.byref(inp), _ptr(o),
        _dt(o), T_prev, None if pin is None else ctypes.byref(pin),
        _idx(prev_accept, "prev_accept"), scale, _stream(stream)))
    return o


def gdn_prefill_chunked_noalloc(pool: Pool, layer: int, slot_ids: torch.Tensor,
                                cu_seqlens: torch.Tensor, q, k, v, g, beta, o: torch.Tensor,
                                scale: float = 1.0, max_seqlen: int = 0, stream=None):
    """gdn_prefill_chunked without any device allocation: its workspace is a
    fixed 64 MiB array inside the library, shared by all calls."""
    inp = _qkv(pool, q, k, v, g, beta)
    if max_seqlen <= 0:
        max_seqlen = q.shape[0]
    _check(load_library().gdn_prefill_chunked_noalloc(
        pool.handle, layer, _idx(slot_ids, "slot_ids"), _idx(cu_seqlens, "cu_seqlens"),
        slot_ids.numel(), q.shape[0], max_seqlen, ctypes.byref(inp), _ptr(o), _dt(o), scale,
        _stream(stream)))
    return o


def gdn_prefill_chunked_ckpt(pool: Pool, layer: int, slot_ids: torch.Tensor,
                             cu_seqlens: torch.Tensor, q, k, v, g, beta, o: torch.Tensor,
                             ckpt_slots: torch.Tensor, ckpt_every: int, scale: float = 1.0,
                             max_seqlen: int = 0, stream=None):
    """gdn_prefill_chunked that also writes the state after every ckpt_every
    tokens of sequence i into slot ckpt_slots[i, j] (int32 [n_seqs, m], -1: none)."""
    inp = _qkv(pool, q, k, v, g, beta)
    if max_seqlen <= 0:
        max_seqlen = q.shape[0]
    if ckpt_slots.dim() != 2 or ckpt_slots.shape[0] != slot_ids.numel():
        raise GDNError(5, "ckpt_slots must be [n_seqs, m]")
    _check(load_library().gdn_prefill_chunked_ckpt(
        pool.handle, layer, _idx(slot_ids, "slot_ids"), _idx(cu_seqlens, "cu_seqlens"),
        slot_ids.numel(), q.shape[0], max_seqlen, ctypes.byref(inp), _ptr(o), _dt(o), scale,
        _idx(ckpt_slots.contiguous(), "ckpt_slots"), ckpt_slots.shape[1], ckpt_every,
        _stream(stream)))
    return o
