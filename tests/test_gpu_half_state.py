"""Pools that store the recurrent state in half precision (bf16 or binary16)
with float32 arithmetic, against the float64 oracle with the same storage
rule (oracle.OraclePool(state_round=...)): the state is carried unrounded
within a call and rounded to nearest-even when the call stores it.

Tolerance.  The GPU rounds a float32 value and the oracle a float64 one, so a
stored element may differ by one unit in the last place of the format where
the two straddle a rounding boundary (2^-8 relative for bf16, 2^-11 for
binary16), and such differences are carried (contracted: alpha <= 1 and
I - beta k k^T has norm <= 1) by later steps.  States and outputs are held to
the bf16-input criterion |gpu - ref| <= 1e-2 + 1e-2 |ref| elementwise and to
max|gpu - ref| <= 4 ulp * max|ref| per tensor (4 * 2^-8 for bf16, 4 * 2^-11
for binary16).  Paths that run the same kernels (one call against two
calls) are compared bit for bit; reset and copy are bit-exact."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrent_gb300 import abi, synth
from oracle import gdn_oracle as O
from tests.gpu_util import assert_close_bf16, assert_maxrel, dev, dev_i32, host, tok_dev, tok_np

pytestmark = pytest.mark.gpu

FMT = {"bf16": (torch.bfloat16, O.round_bf16, 2.0 ** -8),
       "f16": (torch.float16, O.round_f16, 2.0 ** -11)}


def _check(got, ref, fmt, what, extra=0.0):
    """extra: a kernel's own arithmetic bound added to the storage bound."""
    assert_close_bf16(got, ref, what=what)
    assert_maxrel(got, ref, 4 * FMT[fmt][2] + extra, what)


def _pools(shape, n_layers, n_slots, fmt, conv_dtype=torch.bfloat16, **kw):
    tdt, rnd, _ = FMT[fmt]
    gpu = abi.Pool.for_shape(shape, n_layers, n_slots, conv_dtype=conv_dtype, state_dtype=tdt,
                             **kw)
    ref = O.OraclePool(n_layers, n_slots, shape.h_v, shape.h_k, shape.dk, shape.dv,
                       shape.conv_ch, shape.conv_k, state_round=rnd)
    return gpu, ref


def _set_states(gpu, ref, layer, ids, S0, fmt):
    S0 = FMT[fmt][1](S0)                      # representable in the storage format
    gpu.state[layer, torch.from_numpy(np.asarray(ids)).long().cuda()] = \
        torch.from_numpy(S0.astype(np.float32)).cuda().to(gpu.state.dtype)
    ref.S[layer, ids] = S0


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_decode_steps_half_state_pool256_active64(fmt):
    wl = synth.decode_workload(seed=1)
    shape, ids = wl["shape"], wl["slot_ids"]
    gpu, ref = _pools(shape, 1, wl["n_slots"], fmt)
    _set_states(gpu, ref, 0, ids, wl["states"], fmt)
    lid = torch.from_numpy(ids).long().cuda()
    rng = np.random.default_rng(80)
    n = len(ids)
    for step in range(6):
        tok = synth.token_inputs(rng, n, shape, "bf16")
        o = torch.empty(n, shape.h_v, shape.dv, device="cuda")
        abi.gdn_decode_step(gpu, 0, dev_i32(ids), *tok_dev(tok, "bf16"), o)
        o_ref = ref.decode_step(0, ids, *tok_np(tok))
        _check(host(o), o_ref, fmt, f"o step {step}")
    S = gpu.state[0, lid]
    _check(host(S), ref.S[0, ids], fmt, "S")
    assert gpu.state.dtype == FMT[fmt][0]
    assert abi.gdn_pool_get_error(gpu) == 0


@pytest.mark.parametrize("n", [4, 64])
@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_one_call_step_half_state_equals_two_calls(fmt, n):
    """n = 4: the fused kernel; n = 64: the conv + dependent decode pair."""
    shape = synth.GDN_LAYER
    rng = np.random.default_rng(81)
    ids = dev_i32(rng.choice(128, n, replace=False).astype(np.int32))
    tdt = FMT[fmt][0]
    one, two = (abi.Pool.for_shape(shape, 1, 128, state_dtype=tdt) for _ in range(2))
    gen = torch.Generator(device="cuda").manual_seed(8)
    one.state.copy_((0.1 * torch.randn(one.state.shape, device="cuda", generator=gen)).to(tdt))
    one.conv.copy_(torch.randn(one.conv.shape, device="cuda", generator=gen))
    two.state.copy_(one.state)
    two.conv.copy_(one.conv)
    w = dev(synth.conv_weights(rng, shape.conv_ch, shape.conv_k))
    nq = shape.h_k * shape.dk
    for step in range(3):
        x = dev(synth.conv_input(rng, n, shape.conv_ch, "bf16"), "bf16")
        tok = synth.token_inputs(rng, n, shape, "bf16")
        g, b = dev(tok["g"], "bf16"), dev(tok["beta"], "bf16")
        y1 = torch.empty(n, shape.conv_ch, device="cuda", dtype=torch.bfloat16)
        y2 = torch.empty_like(y1)
        o1 = torch.empty(n, shape.h_v, shape.dv, device="cuda")
        o2 = torch.empty_like(o1)
        abi.gdn_decode_step_conv(one, 0, ids, x, w, y1, g, b, o1)
        abi.gdn_conv_silu(two, 0, ids, x, w, y2)
        abi.gdn_decode_step(two, 0, ids, y2[:, :nq].view(n, shape.h_k, shape.dk),
                            y2[:, nq:2 * nq].view(n, shape.h_k, shape.dk),
                            y2[:, 2 * nq:].view(n, shape.h_v, shape.dv), g, b, o2)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(y1, y2), f"step {step}"
        assert torch.equal(one.state, two.state) and torch.equal(one.conv, two.conv)


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_spec_verify_half_state_commit_then_decode(fmt):
    wl = synth.verify_workload(seed=4, n_decode=4)
    shape, ids, T = wl["shape"], wl["slot_ids"], wl["T"]
    n = len(ids)
    gpu, ref = _pools(shape, 1, wl["n_slots"], fmt)
    _set_states(gpu, ref, 0, ids, wl["states"], fmt)
    lid = torch.from_numpy(ids).long().cuda()
    before = gpu.state.clone()
    o = torch.empty(n, T, shape.h_v, shape.dv, device="cuda")
    abi.gdn_spec_verify(gpu, 0, dev_i32(ids), T, *tok_dev(wl["draft"], "bf16"), o=o,
                        accept_len=dev_i32(wl["accept_len"]))
    o_ref = ref.spec_verify(0, ids, T, *tok_np(wl["draft"]), accept_len=wl["accept_len"])
    _check(host(o), o_ref, fmt, "o_t")
    _check(host(gpu.state[0, lid]), ref.S[0, ids], fmt, "committed S")
    zero = torch.from_numpy(ids[wl["accept_len"] == 0]).long().cuda()
    assert torch.equal(gpu.state[0, zero], before[0, zero]), "accept 0 leaves the bits"
    for step in wl["decode"]:
        od = torch.empty(n, shape.h_v, shape.dv, device="cuda")
        abi.gdn_decode_step(gpu, 0, dev_i32(ids), *tok_dev(step, "bf16"), od)
        _check(host(od), ref.decode_step(0, ids, *tok_np(step)), fmt, "decode after commit")
    _check(host(gpu.state[0, lid]), ref.S[0, ids], fmt, "S after decode")


@pytest.mark.parametrize("entry", ["chunked", "recurrent"])
@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_prefill_half_state_varlen_pieces(fmt, entry):
    """Varlen sequences fed in two calls (the state stored, so rounded, between
    them); dk = dv = 128 runs the two-launch tensor-core path (tf32 products:
    its 5e-3 bound applies on top of the storage rounding)."""
    rng = np.random.default_rng(82)
    shape = synth.LayerShape(4, 2, 128, 128, 16, 4)
    lens = [200, 1, 64, 130]
    ids = np.array([3, 0, 5, 1], dtype=np.int32)
    gpu, ref = _pools(shape, 1, 6, fmt, conv_dtype=torch.float32)
    _set_states(gpu, ref, 0, ids, synth.random_states(rng, len(ids), shape), fmt)
    fn = abi.gdn_prefill_chunked if entry == "chunked" else abi.gdn_prefill_recurrent
    tf32 = 5e-3 if entry == "chunked" else 0.0
    for call in range(2):
        cu = synth.cu_seqlens_of(lens)
        tok = synth.token_inputs(rng, int(cu[-1]), shape, "bf16")
        o = torch.empty(int(cu[-1]), shape.h_v, shape.dv, device="cuda")
        fn(gpu, 0, dev_i32(ids), dev_i32(cu), *tok_dev(tok, "bf16"), o, max_seqlen=max(lens))
        o_ref = ref.prefill(0, ids, cu, *tok_np(tok))
        _check(host(o), o_ref, fmt, f"o call {call}", tf32)
    lid = torch.from_numpy(ids).long().cuda()
    _check(host(gpu.state[0, lid]), ref.S[0, ids], fmt, "S", tf32)
    assert abi.gdn_pool_get_error(gpu) == 0


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_prefill_checkpoints_half_state(fmt):
    rng = np.random.default_rng(83)
    shape = synth.LayerShape(4, 2, 128, 128, 16, 4)
    lens = [200, 130]
    ids = np.array([0, 1], dtype=np.int32)
    cu = synth.cu_seqlens_of(lens)
    gpu, ref = _pools(shape, 1, 8, fmt, conv_dtype=torch.float32)
    _set_states(gpu, ref, 0, ids, synth.random_states(rng, 2, shape), fmt)
    tok = synth.token_inputs(rng, int(cu[-1]), shape, "bf16")
    ck = np.array([[2, 3, 4], [5, 6, -1]], dtype=np.int32)
    o = torch.empty(int(cu[-1]), shape.h_v, shape.dv, device="cuda")
    abi.gdn_prefill_chunked_ckpt(gpu, 0, dev_i32(ids), dev_i32(cu), *tok_dev(tok, "bf16"), o,
                                 dev_i32(ck), 64)
    o_ref = ref.prefill_checkpointed(0, ids, cu, *tok_np(tok), ckpt_slots=ck, ckpt_every=64)
    _check(host(o), o_ref, fmt, "o", 5e-3)
    for d in (2, 3, 4, 5, 6, 0, 1):
        _check(host(gpu.state[0, d]), ref.S[0, d], fmt, f"slot {d}", 5e-3)


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_reset_and_copy_half_state_bit_exact(fmt):
    shape = synth.LayerShape(4, 2, 32, 32, 24, 4)
    tdt = FMT[fmt][0]
    pool = abi.Pool.for_shape(shape, 2, 6, state_dtype=tdt)
    assert abi.gdn_pool_state_bytes(pool.desc) == pool.state.numel() * 2
    gen = torch.Generator(device="cuda").manual_seed(9)
    pool.state.copy_(torch.randn(pool.state.shape, device="cuda", generator=gen).to(tdt))
    before = pool.state.clone()
    abi.gdn_pool_copy(pool, dev_i32([1, 4]), dev_i32([2, 0]))
    abi.gdn_pool_reset(pool, dev_i32([5]))
    torch.cuda.synchronize()
    assert torch.equal(pool.state[:, 2], before[:, 1]) and torch.equal(pool.state[:, 0], before[:, 4])
    assert bool((pool.state[:, 5] == 0).all())
    assert torch.equal(pool.state[:, [1, 3, 4]], before[:, [1, 3, 4]])
