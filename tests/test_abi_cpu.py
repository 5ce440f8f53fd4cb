"""CPU-side checks of the C ABI: the library builds, loads and exports every
function include/gdn.h declares; size helpers and argument validation that
fail before any CUDA call behave as documented.  No kernel runs here."""
import ctypes
import os
import re

import pytest

from gated_deltanet_recurrent_gb300 import abi
from gated_deltanet_recurrent_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return abi.load_library()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for required in ("gdn_pool_create", "gdn_pool_reset", "gdn_pool_destroy", "gdn_conv_silu",
                     "gdn_decode_step", "gdn_prefill_chunked", "gdn_spec_verify"):
        assert required in names


def test_library_exports_every_declared_function(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(abi.EXPORTED) == set(_declared_functions())


def _desc(**kw):
    d = dict(n_layers=2, n_slots=5, h_v=4, h_k=2, dk=16, dv=8, conv_ch=64, conv_k=4,
             conv_dtype=abi.GDN_BF16, host_checks=1)
    d.update(kw)
    return abi.gdn_pool_desc(**d)


def test_pool_byte_sizes(lib):
    d = _desc()
    assert abi.gdn_pool_state_bytes(d) == 2 * 5 * 4 * 8 * 16 * 4
    assert abi.gdn_pool_conv_bytes(d) == 2 * 5 * 64 * 3 * 2
    d.conv_dtype = abi.GDN_F32
    assert abi.gdn_pool_conv_bytes(d) == 2 * 5 * 64 * 3 * 4


def _create(lib, d, state=0x1000, conv=0x2000, sb=1 << 40, cb=1 << 40):
    out = ctypes.c_void_p()
    st = lib.gdn_pool_create(ctypes.byref(d) if d is not None else None, state, sb, conv, cb,
                             ctypes.byref(out))
    return st, out


@pytest.mark.parametrize("kw,status", [
    (dict(n_layers=0), "GDN_ERR_ARG"),
    (dict(h_v=3, h_k=2), "GDN_ERR_ARG"),
    (dict(dk=24), "GDN_ERR_UNSUPPORTED"),
    (dict(dv=6), "GDN_ERR_UNSUPPORTED"),
    (dict(conv_k=1), "GDN_ERR_UNSUPPORTED"),
    (dict(conv_k=9), "GDN_ERR_UNSUPPORTED"),
    (dict(conv_dtype=7), "GDN_ERR_DTYPE"),
])
def test_pool_create_rejects_bad_shapes(lib, kw, status):
    st, out = _create(lib, _desc(**kw))
    assert abi.STATUS[st] == status
    assert out.value is None
    assert lib.gdn_last_error_message().decode()


def test_pool_create_rejects_null_small_and_misaligned(lib):
    assert abi.STATUS[_create(lib, None)[0]] == "GDN_ERR_ARG"
    assert abi.STATUS[_create(lib, _desc(), state=0)[0]] == "GDN_ERR_ARG"
    assert abi.STATUS[_create(lib, _desc(), state=0x1004)[0]] == "GDN_ERR_ARG"
    assert abi.STATUS[_create(lib, _desc(), sb=100)[0]] == "GDN_ERR_SIZE"
    assert abi.STATUS[_create(lib, _desc(), cb=100)[0]] == "GDN_ERR_SIZE"


def test_calls_on_a_null_pool_fail_cleanly(lib):
    assert abi.STATUS[lib.gdn_decode_step(None, 0, None, 1, None, None, 0, 1.0, None)] == \
        "GDN_ERR_ARG"
    assert abi.STATUS[lib.gdn_pool_reset(None, None, 1, None)] == "GDN_ERR_ARG"
    assert lib.gdn_pool_destroy(None) == 0
    assert lib.gdn_status_string(5).decode() == "GDN_ERR_SIZE"


def test_no_compute_path_through_the_oracle():
    """The product package never imports the oracle."""
    pkg = os.path.join(ROOT, "gated_deltanet_recurrent_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b|gdn_oracle|oracle/",
                                     text, flags=re.M), f


def test_one_call_decode_step_on_a_null_pool_fails_cleanly(lib):
    st = lib.gdn_decode_step_conv(None, 0, None, 1, None, 0, None, None, None, 0, None, None,
                                  abi.GDN_BF16, None, abi.GDN_F32, 1.0, None)
    assert abi.STATUS[st] == "GDN_ERR_ARG"
    assert "pool" in lib.gdn_last_error_message().decode()


@pytest.mark.parametrize("args,status", [
    (dict(rows=-1), "GDN_ERR_ARG"),
    (dict(d=0), "GDN_ERR_ARG"),
    (dict(eps=-1e-6), "GDN_ERR_ARG"),
    (dict(eps=float("inf")), "GDN_ERR_ARG"),
    (dict(eps=float("nan")), "GDN_ERR_ARG"),
    (dict(o_dtype=7), "GDN_ERR_DTYPE"),
    (dict(y_dtype=2), "GDN_ERR_DTYPE"),
    (dict(o=None), "GDN_ERR_ARG"),             # rows > 0 needs every pointer
    (dict(rows=0, o=None, z=None, w=None, y=None), "GDN_OK"),   # empty: no-op
])
def test_gated_rmsnorm_argument_checks(lib, args, status):
    """Validation runs before any CUDA call (fake non-NULL pointers are never
    dereferenced on these paths)."""
    a = dict(rows=4, d=16, o=0x1000, o_dtype=abi.GDN_F32, z=0x2000, z_dtype=abi.GDN_BF16,
             w=0x3000, eps=1e-6, y=0x4000, y_dtype=abi.GDN_F32)
    a.update(args)
    st = lib.gdn_gated_rmsnorm(a["rows"], a["d"], a["o"], a["o_dtype"], a["z"], a["z_dtype"],
                               a["w"], a["eps"], a["y"], a["y_dtype"], None)
    assert abi.STATUS[st] == status
