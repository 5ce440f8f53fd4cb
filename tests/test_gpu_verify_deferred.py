"""GPU parity of the deferred-commit speculative verify against the float64
oracle, through the C ABI.

Each round commits the accepted part of the previous round's drafts and
outputs the new drafts without committing them; a final gdn_spec_verify with
accept_len flushes the last pending drafts.  Tolerances as for the verify
tests: bf16 inputs |gpu - ref| <= 1e-2 + 1e-2 |ref| elementwise, and for head
dim 128 (tf32 tensor-core dot products) also max|gpu - ref| <= 5e-3 max|ref|;
float32 inputs on the CUDA-core path keep 1e-4 max-relative."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrent_gb300 import abi, synth
from oracle import gdn_oracle as O
from tests.gpu_util import assert_close_bf16, assert_maxrel, dev, dev_i32, host, tok_dev, tok_np

pytestmark = pytest.mark.gpu

SENTINEL = 3.25


def _pool(shape, n_slots):
    p = abi.Pool.for_shape(shape, 1, n_slots, conv_dtype=torch.float32)
    p.state.fill_(SENTINEL)
    return p


def _oracle_pool(shape, n_slots, ids, states):
    op = O.OraclePool(1, n_slots, shape.h_v, shape.h_k, shape.dk, shape.dv, shape.conv_ch,
                      shape.conv_k)
    op.S[0, ids] = states
    return op


def _rounds(pool, op, ids, shape, Ts, accepts, rng, dtype, check):
    """Run deferred rounds on the GPU and in the oracle; flush; compare."""
    n = len(ids)
    prev_d = prev_np = prev_acc = None
    T_prev = 0
    for r, (T, acc) in enumerate(zip(Ts, accepts)):
        tok = synth.token_inputs(rng, n * T, shape, dtype)
        cur_d, cur_np = tok_dev(tok, dtype), tok_np(tok)
        o = torch.empty(n, T, shape.h_v, shape.dv, device="cuda")
        abi.gdn_spec_verify_deferred(pool, 0, dev_i32(ids), T, *cur_d, o, prev=prev_d,
                                     prev_accept=None if prev_acc is None else dev_i32(prev_acc))
        o_ref = op.spec_verify_deferred(0, ids, T, *cur_np, T_prev=T_prev, prev=prev_np,
                                        prev_accept=prev_acc)
        check(host(o), o_ref, f"round {r} outputs")
        prev_d, prev_np, prev_acc, T_prev = cur_d, cur_np, np.asarray(acc, np.int32), T
    abi.gdn_spec_verify(pool, 0, dev_i32(ids), T_prev, *prev_d, accept_len=dev_i32(prev_acc))
    op.spec_verify(0, ids, T_prev, *prev_np, accept_len=prev_acc)
    lid = torch.from_numpy(np.asarray(ids)).long().cuda()
    check(host(pool.state[0, lid]), op.S[0, ids], "state after flush")
    assert abi.gdn_pool_get_error(pool) == 0


def _bf16_check(got, ref, what):
    assert_close_bf16(got, ref, what=what)
    assert_maxrel(got, ref, 5e-3, what)


def test_deferred_rounds_pool256_active128_T4():
    """The verify workload's layer (32/16 heads, K = V = 128, bf16): three
    rounds of 4 drafts, accepted lengths uniform on {0..4}, pending + new
    drafts = 8 (the TMA tensor-core kernel)."""
    wl = synth.verify_workload(seed=4)
    shape, ids = wl["shape"], wl["slot_ids"]
    pool = _pool(shape, wl["n_slots"])
    pool.state[0, torch.from_numpy(ids).long().cuda()] = dev(wl["states"])
    op = _oracle_pool(shape, wl["n_slots"], ids, wl["states"])
    rng = np.random.default_rng(40)
    accepts = [rng.integers(0, 5, len(ids)) for _ in range(3)]
    _rounds(pool, op, ids, shape, [4, 4, 4], accepts, rng, "bf16", _bf16_check)
    mask = np.ones(wl["n_slots"], bool)
    mask[ids] = False
    rest = torch.from_numpy(np.nonzero(mask)[0]).cuda()
    assert bool((pool.state[0, rest] == SENTINEL).all())


def test_deferred_window_edges_head128_rows_kernel():
    """K = V = 128 with pending + new drafts above 8 (the row kernel), up to
    the 32-token window, and pending counts 0 and T_prev."""
    shape = synth.LayerShape(4, 2, 128, 128, 16, 4)
    rng = np.random.default_rng(41)
    ids = np.array([5, 0, 3], dtype=np.int32)
    states = synth.random_states(rng, 3, shape)
    pool = _pool(shape, 6)
    pool.state[0, torch.from_numpy(ids).long().cuda()] = dev(states)
    op = _oracle_pool(shape, 6, ids, states)
    Ts = [6, 9, 23, 1]
    accepts = [[6, 0, 3], [9, 1, 0], [0, 23, 12], [1, 0, 1]]
    _rounds(pool, op, ids, shape, Ts, accepts, rng, "bf16", _bf16_check)


@pytest.mark.parametrize("Ts,accepts", [
    ([2, 2, 1], [[2, 0, 1], [1, 2, 0], [1, 1, 0]]),        # pending + new <= 4
    ([5, 27, 3], [[5, 2, 0], [27, 0, 13], [3, 3, 1]]),     # up to the 32-token window
])
def test_deferred_rounds_small_heads_f32(Ts, accepts):
    shape = synth.LayerShape(4, 2, 64, 32, 16, 4)
    rng = np.random.default_rng(42)
    ids = np.array([1, 4, 2], dtype=np.int32)
    states = synth.random_states(rng, 3, shape)
    pool = _pool(shape, 6)
    pool.state[0, torch.from_numpy(ids).long().cuda()] = dev(states)
    op = _oracle_pool(shape, 6, ids, states)
    check = lambda got, ref, what: assert_maxrel(got, ref, 1e-4, what)
    _rounds(pool, op, ids, shape, Ts, accepts, rng, "f32", check)


def test_deferred_without_pending_is_read_only_and_host_checks():
    shape = synth.LayerShape(2, 1, 16, 16, 16, 4)
    rng = np.random.default_rng(43)
    pool = _pool(shape, 4)
    tok = tok_dev(synth.token_inputs(rng, 2 * 3, shape, "f32"), "f32")
    o = torch.empty(2, 3, 2, 16, device="cuda")
    before = pool.state.clone()
    abi.gdn_spec_verify_deferred(pool, 0, dev_i32([0, 2]), 3, *tok, o)
    torch.cuda.synchronize()
    assert torch.equal(pool.state, before)
    prev = tok_dev(synth.token_inputs(rng, 2 * 4, shape, "f32"), "f32")
    for acc, status in (([5, 0], "GDN_ERR_SIZE"), ([-1, 0], "GDN_ERR_SIZE")):
        with pytest.raises(abi.GDNError) as e:
            abi.gdn_spec_verify_deferred(pool, 0, dev_i32([0, 2]), 3, *tok, o, prev=prev,
                                         prev_accept=dev_i32(acc))
        assert e.value.name == status
    with pytest.raises(abi.GDNError) as e:      # prev given without its counts
        abi.gdn_spec_verify_deferred(pool, 0, dev_i32([0, 2]), 3, *tok, o, prev=prev)
    assert e.value.name == "GDN_ERR_ARG"
    big = tok_dev(synth.token_inputs(rng, 2 * 30, shape, "f32"), "f32")
    with pytest.raises(abi.GDNError) as e:      # 30 pending + 3 new > 32
        abi.gdn_spec_verify_deferred(pool, 0, dev_i32([0, 2]), 3, *tok, o, prev=big,
                                     prev_accept=dev_i32([1, 1]))
    assert e.value.name == "GDN_ERR_SIZE"
    torch.cuda.synchronize()
    assert torch.equal(pool.state, before)
    assert abi.gdn_pool_get_error(pool) == 0
