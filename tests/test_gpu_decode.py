"""GPU parity of the pool, conv + SiLU, decode step and speculative verify
against the float64 oracle, through the C ABI.

Tolerances: float32 decode compares o and S by max|gpu - ref| <= 1e-4 * max|ref|
per tensor; bf16-input verify uses |gpu - ref| <= 1e-2 + 1e-2 |ref| elementwise
(and, for head dim 128, whose row dot products run on the tensor cores in
tf32, also max|gpu - ref| <= 5e-3 * max|ref|); the CUDA-core verify of other
head dims keeps 1e-4; slot gather/scatter is checked bit for bit (untouched
slots hold a sentinel and must not change)."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrent_gb300 import abi, synth
from oracle import gdn_oracle as O
from tests.gpu_util import (assert_close_bf16, assert_maxrel, dev, dev_i32, host, tok_dev,
                            tok_np)

pytestmark = pytest.mark.gpu

SENTINEL = 3.25


def _pool(shape, n_layers, n_slots, conv_dtype=torch.bfloat16, host_checks=True):
    p = abi.Pool.for_shape(shape, n_layers, n_slots, conv_dtype=conv_dtype,
                           host_checks=host_checks)
    p.state.fill_(SENTINEL)
    p.conv.fill_(-SENTINEL)
    return p


def _untouched(pool, active, layer=None):
    mask = np.ones(pool.state.shape[1], dtype=bool)
    mask[np.asarray(active, dtype=np.int64)] = False
    idx = torch.from_numpy(np.nonzero(mask)[0]).cuda()
    st = pool.state if layer is None else pool.state[layer:layer + 1]
    cv = pool.conv if layer is None else pool.conv[layer:layer + 1]
    assert bool((st[:, idx] == SENTINEL).all()), "untouched state slots changed"
    assert bool((cv[:, idx] == -SENTINEL).all()), "untouched conv slots changed"


def test_decode_step_matches_oracle_bf16_inputs_pool256_active64():
    wl = synth.decode_workload(seed=1)           # 32/16 heads, K=V=128, bf16
    shape, ids = wl["shape"], wl["slot_ids"]
    pool = _pool(shape, 1, wl["n_slots"])
    pool.state[0, torch.from_numpy(ids).long().cuda()] = dev(wl["states"])
    n = len(ids)
    o = torch.empty(n, shape.h_v, shape.dv, device="cuda")
    abi.gdn_decode_step(pool, 0, dev_i32(ids), *tok_dev(wl["tok"], "bf16"), o)
    S_got = host(pool.state[0, torch.from_numpy(ids).long().cuda()])
    q, k, v, g, beta = tok_np(wl["tok"])
    S_ref = np.empty_like(S_got)
    o_ref = np.empty((n, shape.h_v, shape.dv))
    for i in range(n):
        S_ref[i], o_ref[i] = O.gdn_step(wl["states"][i], q[i], k[i], v[i], g[i], beta[i])
    assert_maxrel(host(o), o_ref, 1e-4, "o")
    assert_maxrel(S_got, S_ref, 1e-4, "S")
    pool.conv.fill_(-SENTINEL)
    _untouched(pool, ids)
    assert abi.gdn_pool_get_error(pool) == 0


@pytest.mark.parametrize("dk,dv,h_v,h_k,out", [(16, 16, 2, 2, "f32"), (32, 24, 4, 2, "f32"),
                                                (64, 40, 4, 1, "bf16"), (128, 12, 2, 1, "f32")])
def test_decode_step_head_dims(dk, dv, h_v, h_k, out):
    rng = np.random.default_rng(dk + dv)
    shape = synth.LayerShape(h_v, h_k, dk, dv, 32, 4)
    ids = np.array([5, 0, 3], dtype=np.int32)
    pool = _pool(shape, 2, 7, conv_dtype=torch.float32)
    S0 = synth.random_states(rng, len(ids), shape)
    pool.state[1, torch.from_numpy(ids).long().cuda()] = dev(S0)
    tok = synth.token_inputs(rng, len(ids), shape, "f32")
    o = torch.empty(len(ids), h_v, dv, device="cuda",
                    dtype=torch.float32 if out == "f32" else torch.bfloat16)
    abi.gdn_decode_step(pool, 1, dev_i32(ids), *tok_dev(tok, "f32"), o, scale=dk ** -0.5)
    q, k, v, g, beta = tok_np(tok)
    for i in range(len(ids)):
        S_ref, o_ref = O.gdn_step(S0[i], q[i], k[i], v[i], g[i], beta[i], scale=dk ** -0.5)
        assert_maxrel(host(pool.state[1, ids[i]]), S_ref, 1e-4, "S")
        if out == "f32":
            assert_maxrel(host(o[i]), o_ref, 1e-4, "o")
        else:
            assert_close_bf16(host(o[i]), o_ref, what="o bf16")
    _untouched(pool, ids, layer=1)
    _untouched(pool, [], layer=0)


def _conv_ref_pool(shape, n_slots, cache_init, slot_list):
    ref = O.OraclePool(1, n_slots, 1, 1, 4, 4, shape.conv_ch, shape.conv_k)
    for j, s in enumerate(slot_list):
        ref.X[0, s] = cache_init[j]
    return ref


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_conv_silu_varlen_and_advance(dtype):
    rng = np.random.default_rng(7)
    shape = synth.LayerShape(2, 1, 16, 16, 8192 if dtype == "bf16" else 200, 4)
    lens = [1, 17, 40, 0, 3, 33]
    ids = np.array([4, 0, 7, 2, 5, 1], dtype=np.int32)
    cu = synth.cu_seqlens_of(lens)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    pool = _pool(shape, 1, 9, conv_dtype=tdt)
    cache0 = synth.random_conv_cache(rng, len(ids), shape, dtype)
    pool.conv[0, torch.from_numpy(ids).long().cuda()] = dev(cache0, dtype)
    x = synth.conv_input(rng, int(cu[-1]), shape.conv_ch, dtype)
    w = synth.conv_weights(rng, shape.conv_ch, shape.conv_k)
    bias = synth.cast(rng.standard_normal(shape.conv_ch), "f32")
    adv = np.array([1, 5, 40, 0, 2, 33], dtype=np.int32)
    y = torch.empty(int(cu[-1]), shape.conv_ch, device="cuda", dtype=tdt)
    abi.gdn_conv_silu(pool, 0, dev_i32(ids), dev(x, dtype), dev(w), y, cu_seqlens=dev_i32(cu),
                      bias=dev(bias), advance=dev_i32(adv), max_seqlen=max(lens))
    ref = _conv_ref_pool(shape, 9, cache0, ids)
    y_ref = ref.conv_silu(0, ids, cu, x, w, bias, advance=adv)
    if dtype == "bf16":
        assert_close_bf16(host(y), y_ref, what="y")
    else:
        assert_maxrel(host(y), y_ref, 1e-5, "y")
    got = host(pool.conv[0, torch.from_numpy(ids).long().cuda()])
    np.testing.assert_array_equal(got, ref.X[0, ids])          # raw inputs: exact
    _untouched(pool, ids)


def test_conv_silu_decode_mode_and_small_max_seqlen():
    rng = np.random.default_rng(8)
    shape = synth.LayerShape(2, 1, 16, 16, 300, 3)
    ids = np.array([2, 6, 1], dtype=np.int32)
    pool = _pool(shape, 1, 8, conv_dtype=torch.float32)
    cache0 = synth.random_conv_cache(rng, 3, shape, "f32")
    pool.conv[0, torch.from_numpy(ids).long().cuda()] = dev(cache0)
    w = synth.conv_weights(rng, shape.conv_ch, shape.conv_k)
    ref = _conv_ref_pool(shape, 8, cache0, ids)
    for step in range(3):                                       # three decode tokens
        x = synth.conv_input(rng, 3, shape.conv_ch, "f32")
        y = torch.empty(3, shape.conv_ch, device="cuda")
        abi.gdn_conv_silu(pool, 0, dev_i32(ids), dev(x), dev(w), y)
        assert_maxrel(host(y), ref.conv_silu(0, ids, None, x, w), 1e-5, "y")
    # a long sequence with a deliberately small max_seqlen hint (grid-stride path)
    x = synth.conv_input(rng, 100, shape.conv_ch, "f32")
    y = torch.empty(100, shape.conv_ch, device="cuda")
    abi.gdn_conv_silu(pool, 0, dev_i32(ids[:1]), dev(x), dev(w), y,
                      cu_seqlens=dev_i32([0, 100]), max_seqlen=1)
    assert_maxrel(host(y), ref.conv_silu(0, ids[:1], [0, 100], x, w), 1e-5, "y")
    np.testing.assert_array_equal(host(pool.conv[0, torch.from_numpy(ids).long().cuda()]),
                                  ref.X[0, ids])


def test_conv_then_decode_chained_on_the_qkv_split():
    """x -> conv + SiLU -> y = [q | k | v] (views, no copies) -> decode."""
    wl = synth.decode_workload(seed=1)
    shape, ids = wl["shape"], wl["slot_ids"]
    n = len(ids)
    pool = _pool(shape, 1, wl["n_slots"])
    lid = torch.from_numpy(ids).long().cuda()
    pool.state[0, lid] = dev(wl["states"])
    pool.conv[0, lid] = dev(wl["conv_cache"], "bf16")
    y = torch.empty(n, shape.conv_ch, device="cuda", dtype=torch.bfloat16)
    abi.gdn_conv_silu(pool, 0, dev_i32(ids), dev(wl["x"], "bf16"), dev(wl["conv_w"]), y)
    nq = shape.h_k * shape.dk
    q = y[:, :nq].view(n, shape.h_k, shape.dk)
    k = y[:, nq:2 * nq].view(n, shape.h_k, shape.dk)
    v = y[:, 2 * nq:].view(n, shape.h_v, shape.dv)
    g = dev(wl["tok"]["g"], "bf16")
    beta = dev(wl["tok"]["beta"], "bf16")
    o = torch.empty(n, shape.h_v, shape.dv, device="cuda")
    abi.gdn_decode_step(pool, 0, dev_i32(ids), q, k, v, g, beta, o)

    o_ref = np.empty((n, shape.h_v, shape.dv))
    for i in range(n):
        yi, _ = O.conv_silu(wl["x"][i:i + 1], wl["conv_cache"][i], wl["conv_w"])
        yi = yi[0]
        _, o_ref[i] = O.gdn_step(wl["states"][i], yi[:nq].reshape(shape.h_k, shape.dk),
                                 yi[nq:2 * nq].reshape(shape.h_k, shape.dk),
                                 yi[2 * nq:].reshape(shape.h_v, shape.dv),
                                 wl["tok"]["g"][i], wl["tok"]["beta"][i])
    assert_close_bf16(host(o), o_ref, what="o (chained)")


def test_spec_verify_commit_then_decode_pool256_active128():
    wl = synth.verify_workload(seed=4)           # 128 active, T = 4, bf16
    shape, ids, T = wl["shape"], wl["slot_ids"], wl["T"]
    n = len(ids)
    lid = torch.from_numpy(ids).long().cuda()
    pool = _pool(shape, 1, wl["n_slots"])
    pool.state[0, lid] = dev(wl["states"])
    draft = tok_dev(wl["draft"], "bf16")
    acc = wl["accept_len"]

    # verify only: outputs, pool untouched
    before = pool.state.clone()
    o1 = torch.empty(n, T, shape.h_v, shape.dv, device="cuda")
    abi.gdn_spec_verify(pool, 0, dev_i32(ids), T, *draft, o=o1)
    assert torch.equal(pool.state, before)
    # commit in one pass with outputs; must equal the verify-only outputs
    o2 = torch.empty_like(o1)
    abi.gdn_spec_verify(pool, 0, dev_i32(ids), T, *draft, o=o2, accept_len=dev_i32(acc))
    assert torch.equal(o1, o2)

    q, k, v, g, beta = tok_np(wl["draft"])
    S_ref = np.empty((n, shape.h_v, shape.dv, shape.dk))
    o_ref = np.empty((n, T, shape.h_v, shape.dv))
    for i in range(n):
        sl = slice(i * T, (i + 1) * T)
        o_ref[i], S_ref[i] = O.spec_verify(wl["states"][i], q[sl], k[sl], v[sl], g[sl],
                                           beta[sl], acc[i])
    # bf16-input verify: the stated elementwise criterion, plus the tf32 bound of
    # the tensor-core path (dot products with tf32 operands, unit roundoff 2^-11)
    assert_close_bf16(host(o2), o_ref, what="o_t")
    assert_maxrel(host(o2), o_ref, 5e-3, "o_t")
    S_got = host(pool.state[0, lid])
    assert_close_bf16(S_got, S_ref, what="committed S")
    assert_maxrel(S_got, S_ref, 5e-3, "committed S")
    zero = acc == 0
    assert np.array_equal(S_got[zero], wl["states"][zero]), "accept 0 must leave bits unchanged"
    _untouched(pool, ids)

    # 16 decode steps on the committed states
    for step in wl["decode"]:
        o = torch.empty(n, shape.h_v, shape.dv, device="cuda")
        abi.gdn_decode_step(pool, 0, dev_i32(ids), *tok_dev(step, "bf16"), o)
        qd, kd, vd, gd, bd = tok_np(step)
        for i in range(n):
            S_ref[i], oi = O.gdn_step(S_ref[i], qd[i], kd[i], vd[i], gd[i], bd[i])
            if i % 16 == 0:
                assert_close_bf16(host(o[i]), oi, what="decode after commit")
    assert_close_bf16(host(pool.state[0, lid]), S_ref, what="S after 16 decode steps")
    assert_maxrel(host(pool.state[0, lid]), S_ref, 5e-3, "S after 16 decode steps")


def test_spec_verify_commit_only_two_phase_and_T_edges():
    rng = np.random.default_rng(9)
    shape = synth.LayerShape(4, 2, 64, 32, 16, 4)
    ids = np.array([1, 4, 2], dtype=np.int32)
    for T in (1, 7, 32):
        pool = _pool(shape, 1, 6, conv_dtype=torch.float32)
        S0 = synth.random_states(rng, 3, shape)
        pool.state[0, torch.from_numpy(ids).long().cuda()] = dev(S0)
        tok = synth.token_inputs(rng, 3 * T, shape, "f32")
        acc = np.array([T, 0, T // 2], dtype=np.int32)
        abi.gdn_spec_verify(pool, 0, dev_i32(ids), T, *tok_dev(tok, "f32"),
                            accept_len=dev_i32(acc))                  # commit only
        q, k, v, g, beta = tok_np(tok)
        for i in range(3):
            sl = slice(i * T, (i + 1) * T)
            _, S_ref = O.spec_verify(S0[i], q[sl], k[sl], v[sl], g[sl], beta[sl], acc[i])
            assert_maxrel(host(pool.state[0, ids[i]]), S_ref, 1e-4, f"T={T} slot {i}")
        _untouched(pool, ids)


def test_pool_reset_zeroes_only_listed_slots():
    shape = synth.LayerShape(4, 2, 32, 32, 24, 4)
    pool = _pool(shape, 3, 10)
    ids = np.array([7, 2, 9], dtype=np.int32)
    abi.gdn_pool_reset(pool, dev_i32(ids))
    lid = torch.from_numpy(ids).long().cuda()
    assert bool((pool.state[:, lid] == 0).all()) and bool((pool.conv[:, lid] == 0).all())
    _untouched(pool, ids)


def test_host_checks_reject_bad_indices_and_launch_nothing():
    shape = synth.LayerShape(2, 1, 16, 16, 16, 4)
    pool = _pool(shape, 1, 4, conv_dtype=torch.float32)
    rng = np.random.default_rng(10)
    tok = tok_dev(synth.token_inputs(rng, 2, shape, "f32"), "f32")
    o = torch.zeros(2, 2, 16, device="cuda")
    before = pool.state.clone()
    for ids, status in (([0, 4], "GDN_ERR_SLOT"), ([1, 1], "GDN_ERR_DUP_SLOT"),
                        ([-1, 2], "GDN_ERR_SLOT")):
        with pytest.raises(abi.GDNError) as e:
            abi.gdn_decode_step(pool, 0, dev_i32(ids), *tok, o)
        assert e.value.name == status
    with pytest.raises(abi.GDNError) as e:     # index array in host memory
        abi.gdn_decode_step(pool, 0, torch.tensor([0, 1], dtype=torch.int32), *tok, o)
    assert e.value.name == "GDN_ERR_ARG"
    with pytest.raises(abi.GDNError) as e:     # accept_len > T
        abi.gdn_spec_verify(pool, 0, dev_i32([0]), 1, *[t[:1] for t in tok],
                            accept_len=dev_i32([2]))
    assert e.value.name == "GDN_ERR_SIZE"
    with pytest.raises(abi.GDNError) as e:     # cu_seqlens not ending at total
        abi.gdn_conv_silu(pool, 0, dev_i32([0]), torch.zeros(3, 16, device="cuda"),
                          torch.zeros(16, 4, device="cuda"), torch.zeros(3, 16, device="cuda"),
                          cu_seqlens=dev_i32([0, 2]))
    assert e.value.name == "GDN_ERR_SIZE"
    with pytest.raises(abi.GDNError) as e:
        abi.gdn_decode_step(pool, 1, dev_i32([0]), *[t[:1] for t in tok], o[:1])
    assert e.value.name == "GDN_ERR_ARG"      # layer out of range
    torch.cuda.synchronize()
    assert torch.equal(pool.state, before)
    assert abi.gdn_pool_get_error(pool) == 0


def test_device_guard_skips_bad_slot_and_sets_error_word():
    shape = synth.LayerShape(2, 1, 16, 16, 16, 4)
    pool = _pool(shape, 1, 4, conv_dtype=torch.float32, host_checks=False)
    rng = np.random.default_rng(11)
    S0 = synth.random_states(rng, 1, shape)
    pool.state[0, 2] = dev(S0[0])
    t = synth.token_inputs(rng, 2, shape, "f32")
    o = torch.zeros(2, 2, 16, device="cuda")
    abi.gdn_decode_step(pool, 0, dev_i32([2, 99]), *tok_dev(t, "f32"), o)
    assert abi.gdn_pool_get_error(pool) == abi.DEVERR_SLOT
    assert abi.gdn_pool_get_error(pool) == 0           # read-and-clear
    q, k, v, g, beta = tok_np(t)
    S_ref, o_ref = O.gdn_step(S0[0], q[0], k[0], v[0], g[0], beta[0])
    assert_maxrel(host(pool.state[0, 2]), S_ref, 1e-4, "valid entry still processed")
    assert bool((o[1] == 0).all())
    _untouched(pool, [2])
    # a malformed cu_seqlens range and an out-of-range advance are flagged too
    x = torch.zeros(4, 16, device="cuda")
    abi.gdn_conv_silu(pool, 0, dev_i32([1]), x, torch.zeros(16, 4, device="cuda"),
                      torch.zeros(4, 16, device="cuda"), cu_seqlens=dev_i32([3, 1]))
    assert abi.gdn_pool_get_error(pool) == abi.DEVERR_SEQ
    abi.gdn_spec_verify(pool, 0, dev_i32([0]), 1, *[tt[:1] for tt in tok_dev(t, "f32")],
                        accept_len=dev_i32([5]))
    assert abi.gdn_pool_get_error(pool) == abi.DEVERR_COUNT


def test_pool_copy_checkpoints_slots_bit_exact():
    shape = synth.LayerShape(4, 2, 32, 32, 24, 4)
    pool = _pool(shape, 3, 8)
    gen = torch.Generator(device="cuda").manual_seed(5)
    pool.state.normal_(generator=gen)
    pool.conv.copy_(torch.randn(pool.conv.shape, device="cuda", generator=gen))
    before = (pool.state.clone(), pool.conv.clone())
    src, dst = [3, 5], [0, 6]
    abi.gdn_pool_copy(pool, dev_i32(src), dev_i32(dst))
    torch.cuda.synchronize()
    for a, b in zip(src, dst):
        assert torch.equal(pool.state[:, b], before[0][:, a])
        assert torch.equal(pool.conv[:, b], before[1][:, a])
    others = [s for s in range(8) if s not in dst]
    assert torch.equal(pool.state[:, others], before[0][:, others])
    assert torch.equal(pool.conv[:, others], before[1][:, others])
    for s_, d_, status in (([1, 2], [4, 4], "GDN_ERR_DUP_SLOT"), ([1, 4], [4, 2], "GDN_ERR_DUP_SLOT"),
                           ([9], [1], "GDN_ERR_SLOT")):
        with pytest.raises(abi.GDNError) as e:
            abi.gdn_pool_copy(pool, dev_i32(s_), dev_i32(d_))
        assert e.value.name == status


def test_pool_copy_then_continue_matches_uninterrupted_request():
    """A checkpoint copied mid-request continues exactly like the original slot."""
    rng = np.random.default_rng(12)
    shape = synth.LayerShape(2, 1, 64, 64, 16, 4)
    pool = _pool(shape, 1, 4, conv_dtype=torch.float32)
    abi.gdn_pool_reset(pool, dev_i32([0, 2]))
    tok = synth.token_inputs(rng, 150, shape, "f32")
    d = tok_dev(tok, "f32")
    o = torch.empty(150, 2, 64, device="cuda")
    abi.gdn_prefill_chunked(pool, 0, dev_i32([0]), dev_i32([0, 100]), *[t[:100] for t in d], o[:100])
    abi.gdn_pool_copy(pool, dev_i32([0]), dev_i32([2]))
    o2 = torch.empty(50, 2, 64, device="cuda")
    abi.gdn_prefill_chunked(pool, 0, dev_i32([0]), dev_i32([0, 50]), *[t[100:] for t in d], o[100:])
    abi.gdn_prefill_chunked(pool, 0, dev_i32([2]), dev_i32([0, 50]), *[t[100:] for t in d], o2)
    assert torch.equal(o[100:], o2)
    assert torch.equal(pool.state[0, 0], pool.state[0, 2])
