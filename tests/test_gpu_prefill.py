"""GPU parity of gdn_prefill_chunked (and the tiny end-to-end request flow)
against the float64 oracle, through the C ABI.

float32 inputs: max|gpu - ref| <= 1e-4 * max|ref| per tensor (5e-3 on the tf32
tensor-core path, see _rel_tol).  bf16 inputs:
|gpu - ref| <= 1e-2 + 1e-2 |ref| elementwise.  Full-size cases are checked on
a sample of value heads (the oracle runs only those heads); untouched slots
are checked bit for bit."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrent_gb300 import abi, synth
from oracle import gdn_oracle as O
from tests.gpu_util import (assert_close_bf16, assert_maxrel, dev, dev_i32, host, tdtype, tok_dev,
                            tok_np)
from tests.oracle_par import recurrent_many

pytestmark = pytest.mark.gpu

SENTINEL = 3.25

# Prefill with dk = dv = 128 runs its chunk products on the tensor cores in
# tf32 (10 explicit mantissa bits, unit roundoff u = 2^-11 ~ 4.9e-4), reading
# fp32 operands.  Each output is a sum of products of two rounded operands,
# and the recurrence carries those errors through the state, so a float32
# input case is held to max|gpu - ref| <= 5e-3 * max|ref| (about 10 u) instead
# of the 1e-4 of the pure float32 kernels; smaller head dims run the float32
# CUDA-core kernel and keep 1e-4.
def _rel_tol(D):
    return 5e-3 if D == 128 else 1e-4


def _pool(shape, n_layers, n_slots, conv_dtype=torch.float32, host_checks=True):
    p = abi.Pool.for_shape(shape, n_layers, n_slots, conv_dtype=conv_dtype,
                           host_checks=host_checks)
    p.state.fill_(SENTINEL)
    p.conv.fill_(-SENTINEL)
    return p


def _run_tiny_request_gpu(pool, wl, i, slot):
    seq = wl["seqs"][i]
    L = wl["lengths"][i]
    tok, x = seq["tok"], seq["x"]
    sid = dev_i32([slot])
    ys, os_ = [], []
    w = dev(wl["conv_w"])
    for lo in range(0, L, wl["piece"]):
        hi = min(lo + wl["piece"], L)
        cu = dev_i32([0, hi - lo])
        y = torch.empty(hi - lo, wl["shape"].conv_ch, device="cuda")
        abi.gdn_conv_silu(pool, 0, sid, dev(x[lo:hi]), w, y, cu_seqlens=cu)
        o = torch.empty(hi - lo, wl["shape"].h_v, wl["shape"].dv, device="cuda")
        abi.gdn_prefill_chunked(pool, 0, sid, cu, *[dev(tok[n][lo:hi]) for n in
                                                    ("q", "k", "v", "g", "beta")], o)
        ys.append(y)
        os_.append(o)
    for t in range(L, L + wl["n_decode"]):
        y = torch.empty(1, wl["shape"].conv_ch, device="cuda")
        abi.gdn_conv_silu(pool, 0, sid, dev(x[t:t + 1]), w, y)
        o = torch.empty(1, wl["shape"].h_v, wl["shape"].dv, device="cuda")
        abi.gdn_decode_step(pool, 0, sid, *[dev(tok[n][t:t + 1]) for n in
                                            ("q", "k", "v", "g", "beta")], o)
        ys.append(y)
        os_.append(o)
    return host(torch.cat(ys)), host(torch.cat(os_))


def _run_tiny_request_ref(ref, wl, i, slot):
    seq = wl["seqs"][i]
    L = wl["lengths"][i]
    tok, x = seq["tok"], seq["x"]
    ys, os_ = [], []
    for lo in range(0, L, wl["piece"]):
        hi = min(lo + wl["piece"], L)
        ys.append(ref.conv_silu(0, [slot], [0, hi - lo], x[lo:hi], wl["conv_w"]))
        os_.append(ref.prefill(0, [slot], [0, hi - lo], *(tok[n][lo:hi] for n in
                                                           ("q", "k", "v", "g", "beta"))))
    for t in range(L, L + wl["n_decode"]):
        ys.append(ref.conv_silu(0, [slot], None, x[t:t + 1], wl["conv_w"]))
        os_.append(ref.decode_step(0, [slot], *(tok[n][t:t + 1] for n in
                                                ("q", "k", "v", "g", "beta"))))
    return np.concatenate(ys), np.concatenate(os_)


def test_tiny_request_flow_prefill_decode_reset_rerun():
    """Pool of 4 slots; sequences of 7 and 13 tokens in slots 1 and 3 fed in
    4-token prefill pieces, 5 decode steps; reset slot 1 and rerun it."""
    wl = synth.tiny_workload(0)
    s = wl["shape"]
    pool = _pool(s, 1, wl["n_slots"])
    pool.set_host_checks(True)
    abi.gdn_pool_reset(pool, dev_i32(wl["slots"]))
    ref = O.OraclePool(1, wl["n_slots"], s.h_v, s.h_k, s.dk, s.dv, s.conv_ch, s.conv_k)
    first = []
    for i, slot in enumerate(wl["slots"]):
        y, o = _run_tiny_request_gpu(pool, wl, i, slot)
        y_ref, o_ref = _run_tiny_request_ref(ref, wl, i, slot)
        assert_maxrel(y, y_ref, 1e-5, f"conv y, seq {i}")
        assert_maxrel(o, o_ref, 1e-4, f"o, seq {i}")
        first.append((y, o))
    for slot in wl["slots"]:
        assert_maxrel(host(pool.state[0, slot]), ref.S[0, slot], 1e-4, f"S slot {slot}")
    np.testing.assert_array_equal(host(pool.conv[0, wl["slots"]]), ref.X[0, wl["slots"]])
    S3 = pool.state[0, 3].clone()
    abi.gdn_pool_reset(pool, dev_i32([1]))
    y, o = _run_tiny_request_gpu(pool, wl, 0, 1)
    np.testing.assert_array_equal(y, first[0][0])       # reset slot == fresh slot, bit for bit
    np.testing.assert_array_equal(o, first[0][1])
    assert torch.equal(pool.state[0, 3], S3)
    assert bool((pool.state[:, [0, 2]] == SENTINEL).all())
    assert bool((pool.conv[:, [0, 2]] == -SENTINEL).all())
    assert abi.gdn_pool_get_error(pool) == 0


PREFILL = {"chunked": abi.gdn_prefill_chunked, "recurrent": abi.gdn_prefill_recurrent}


@pytest.mark.parametrize("entry", ["chunked", "recurrent"])
@pytest.mark.parametrize("D", [16, 32, 64, 128])
def test_prefill_varlen_edge_lengths(D, entry):
    rng = np.random.default_rng(40 + D)
    shape = synth.LayerShape(4, 2, D, D, 16, 4)
    lens = [1, 0, 64, 65, 130, 7]
    ids = np.array([6, 2, 0, 5, 1, 3], dtype=np.int32)
    cu = synth.cu_seqlens_of(lens)
    pool = _pool(shape, 2, 8)
    S0 = synth.random_states(rng, len(ids), shape)
    lid = torch.from_numpy(ids).long().cuda()
    pool.state[1, lid] = dev(S0)
    tok = synth.token_inputs(rng, int(cu[-1]), shape, "f32")
    o = torch.empty(int(cu[-1]), shape.h_v, shape.dv, device="cuda")
    PREFILL[entry](pool, 1, dev_i32(ids), dev_i32(cu), *tok_dev(tok, "f32"), o,
                   scale=D ** -0.5, max_seqlen=max(lens))
    ref = O.OraclePool(1, 8, shape.h_v, shape.h_k, shape.dk, shape.dv, 16, 4)
    ref.S[0, ids] = S0
    o_ref = ref.prefill(0, ids, cu, *tok_np(tok), scale=D ** -0.5)
    tol = _rel_tol(D) if entry == "chunked" else 1e-4
    assert_maxrel(host(o), o_ref, tol, "o")
    assert_maxrel(host(pool.state[1, lid]), ref.S[0, ids], tol, "S")
    pool.state[1, lid] = SENTINEL
    assert bool((pool.state == SENTINEL).all())


@pytest.mark.parametrize("entry", ["chunked", "recurrent"])
def test_prefill_split_across_calls_equals_whole_and_token_recurrence(entry):
    rng = np.random.default_rng(41)
    shape = synth.LayerShape(2, 1, 128, 128, 16, 4)
    L = 301
    S0 = synth.random_states(rng, 1, shape)
    tok = synth.token_inputs(rng, L, shape, "f32")
    outs = {}
    for name, cuts in (("whole", [0, L]), ("pieces", [0, 64, 100, 101, 229, L])):
        pool = _pool(shape, 1, 2)
        pool.state[0, 1] = dev(S0[0])
        parts = []
        for lo, hi in zip(cuts[:-1], cuts[1:]):
            o = torch.empty(hi - lo, shape.h_v, shape.dv, device="cuda")
            PREFILL[entry](pool, 0, dev_i32([1]), dev_i32([0, hi - lo]),
                           *[dev(tok[n][lo:hi]) for n in ("q", "k", "v", "g", "beta")], o)
            parts.append(host(o))
        outs[name] = (np.concatenate(parts), host(pool.state[0, 1]))
    S_ref, o_ref = O.gdn_recurrent(S0[0], *tok_np(tok))
    tol = _rel_tol(128) if entry == "chunked" else 1e-4
    for name, (o, S) in outs.items():
        assert_maxrel(o, o_ref, tol, f"o {name}")
        assert_maxrel(S, S_ref, tol, f"S {name}")


@pytest.mark.parametrize("dtype,h_v,h_k", [("f32", 4, 2), ("bf16", 4, 2), ("bf16", 3, 3),
                                           ("bf16", 4, 1), ("f32", 2, 2)])
def test_prefill_two_launch_path_equals_single_launch_kernel(dtype, h_v, h_k):
    """dk = dv = 128: the two-launch path (per-chunk key-side tiles in a
    workspace) against the single-launch kernel (no workspace: forced by a
    1-byte workspace limit), and both against the oracle.  With float32 inputs
    both form the key-side products in tf32 from the same normalised rows, so
    they agree to float32 rounding (1e-5); with bf16 inputs the two-launch path
    multiplies the exact bf16 inputs (kind::f16) and normalises afterwards, so
    the two differ by the single-launch kernel's tf32 rounding (5e-3 bound)."""
    rng = np.random.default_rng(44)
    shape = synth.LayerShape(h_v, h_k, 128, 128, 16, 4)   # value heads per key head: 2, 1, 4
    lens = [200, 0, 1, 64, 129, 77]
    ids = np.array([5, 0, 2, 7, 1, 4], dtype=np.int32)
    cu = synth.cu_seqlens_of(lens)
    S0 = synth.random_states(rng, len(ids), shape)
    tok = synth.token_inputs(rng, int(cu[-1]), shape, dtype)
    lid = torch.from_numpy(ids).long().cuda()
    res = {}
    for name, limit in (("two-launch", 0), ("single", 1)):
        pool = abi.Pool.for_shape(shape, 1, 8, conv_dtype=torch.float32,
                                  prefill_workspace_max=limit)
        pool.state[0, lid] = dev(S0)
        o = torch.empty(int(cu[-1]), shape.h_v, shape.dv, device="cuda")
        abi.gdn_prefill_chunked(pool, 0, dev_i32(ids), dev_i32(cu), *tok_dev(tok, dtype), o,
                                max_seqlen=max(lens))
        res[name] = (host(o), host(pool.state[0, lid]))
        assert abi.gdn_pool_get_error(pool) == 0
    tol = 1e-5 if dtype == "f32" else _rel_tol(128)
    assert_maxrel(res["two-launch"][0], res["single"][0], tol, "o two-launch vs single")
    assert_maxrel(res["two-launch"][1], res["single"][1], tol, "S two-launch vs single")
    ref = O.OraclePool(1, 8, shape.h_v, shape.h_k, shape.dk, shape.dv, 16, 4)
    ref.S[0, ids] = S0
    o_ref = ref.prefill(0, ids, cu, *tok_np(tok))
    assert_maxrel(res["single"][0], o_ref, _rel_tol(128), "o single")
    assert_maxrel(res["two-launch"][0], o_ref, _rel_tol(128), "o")
    assert_maxrel(res["two-launch"][1], ref.S[0, ids], _rel_tol(128), "S")


def test_prefill_two_launch_rows_not_16_byte_aligned():
    """bf16 rows whose token stride is not a multiple of 16 bytes (ld = 260
    elements, allowed: rows need 8-byte alignment) cannot arrive by tensor
    map; the state kernel then stages them from global memory as normalised
    float32 rows (tf32 operands), where aligned rows feed the bf16 products
    directly (kind::f16, the state operand rounded to bf16).  Both paths
    agree with the oracle, and with each other, within the tensor-core bound
    5e-3 * max|ref|."""
    rng = np.random.default_rng(45)
    shape = synth.LayerShape(4, 2, 128, 128, 16, 4)
    lens = [150, 64, 3]
    ids = np.array([2, 0, 3], dtype=np.int32)
    cu = synth.cu_seqlens_of(lens)
    T = int(cu[-1])
    S0 = synth.random_states(rng, len(ids), shape)
    tok = synth.token_inputs(rng, T, shape, "bf16")
    q, k, v, g, beta = tok_dev(tok, "bf16")
    pad = 4
    wide = []
    for x, heads in ((q, shape.h_k), (k, shape.h_k), (v, shape.h_v)):
        buf = torch.zeros(T, heads * 128 + pad, device="cuda", dtype=torch.bfloat16)
        buf[:, :heads * 128] = x.reshape(T, -1)
        wide.append(buf[:, :heads * 128].view(T, heads, 128))   # token stride 8 + 512k bytes
    lid = torch.from_numpy(ids).long().cuda()
    res = []
    for qq, kk, vv in ((q, k, v), tuple(wide)):
        pool = abi.Pool.for_shape(shape, 1, 4, conv_dtype=torch.float32)
        pool.state[0, lid] = dev(S0)
        o = torch.empty(T, shape.h_v, shape.dv, device="cuda")
        abi.gdn_prefill_chunked(pool, 0, dev_i32(ids), dev_i32(cu), qq, kk, vv, g, beta, o)
        res.append((host(o), host(pool.state[0, lid])))
        assert abi.gdn_pool_get_error(pool) == 0
    ref = O.OraclePool(1, 4, shape.h_v, shape.h_k, shape.dk, shape.dv, 16, 4)
    ref.S[0, ids] = S0
    o_ref = ref.prefill(0, ids, cu, *tok_np(tok))
    tol = _rel_tol(128)
    for name, (o, S) in zip(("tensor-map rows", "staged rows"), res):
        assert_maxrel(o, o_ref, tol, f"o {name}")
        assert_maxrel(S, ref.S[0, ids], tol, f"S {name}")
    assert_maxrel(res[0][0], res[1][0], tol, "o aligned vs unaligned")
    assert_maxrel(res[0][1], res[1][1], tol, "S aligned vs unaligned")


def test_prefill_checkpoints_match_oracle_and_resume():
    """gdn_prefill_chunked_ckpt: the state after every 64 tokens goes to the
    requested slots (prefix-cache checkpoints).  Each checkpoint matches the
    oracle's state after that prefix, and a request resumed from a checkpoint
    slot with the rest of its tokens ends where the uninterrupted one does."""
    rng = np.random.default_rng(46)
    shape = synth.LayerShape(4, 2, 128, 128, 16, 4)
    lens = [300, 64, 130]
    ids = np.array([0, 1, 2], dtype=np.int32)
    cu = synth.cu_seqlens_of(lens)
    T = int(cu[-1])
    S0 = synth.random_states(rng, 3, shape)
    tok = synth.token_inputs(rng, T, shape, "bf16")
    ck = np.array([[3, -1, 4, 5], [6, -1, -1, -1], [7, 8, -1, -1]], dtype=np.int32)
    pool = abi.Pool.for_shape(shape, 1, 12, conv_dtype=torch.float32)
    pool.state.fill_(SENTINEL)
    lid = torch.from_numpy(ids).long().cuda()
    pool.state[0, lid] = dev(S0)
    o = torch.empty(T, shape.h_v, shape.dv, device="cuda")
    abi.gdn_prefill_chunked_ckpt(pool, 0, dev_i32(ids), dev_i32(cu), *tok_dev(tok, "bf16"), o,
                                 dev_i32(ck), 64)
    assert abi.gdn_pool_get_error(pool) == 0
    ref = O.OraclePool(1, 12, shape.h_v, shape.h_k, shape.dk, shape.dv, 16, 4)
    ref.S[0, ids] = S0
    o_ref = ref.prefill_checkpointed(0, ids, cu, *tok_np(tok), ckpt_slots=ck, ckpt_every=64)
    assert_close_bf16(host(o), o_ref, what="o")
    assert_maxrel(host(o), o_ref, _rel_tol(128), "o")
    used = sorted(int(d) for d in ck.ravel() if d >= 0)
    for d in used:
        assert_maxrel(host(pool.state[0, d]), ref.S[0, d], _rel_tol(128), f"checkpoint slot {d}")
    assert_maxrel(host(pool.state[0, lid]), ref.S[0, ids], _rel_tol(128), "final S")
    rest = [s for s in range(12) if s not in used and s not in ids]
    assert bool((pool.state[0, rest] == SENTINEL).all())
    # resume sequence 0 from its checkpoint after 192 tokens (slot 4): prefill tokens 192..299
    q, k, v, g, beta = tok_dev(tok, "bf16")
    lo, hi = 192, 300
    o2 = torch.empty(hi - lo, shape.h_v, shape.dv, device="cuda")
    abi.gdn_prefill_chunked(pool, 0, dev_i32([4]), dev_i32([0, hi - lo]),
                            q[lo:hi], k[lo:hi], v[lo:hi], g[lo:hi], beta[lo:hi], o2)
    assert_maxrel(host(pool.state[0, 4]), host(pool.state[0, 0]), _rel_tol(128), "resumed S")
    assert_maxrel(host(o2), host(o[lo:hi]), _rel_tol(128), "resumed o")


def test_prefill_checkpoint_argument_checks():
    shape = synth.LayerShape(2, 1, 128, 128, 16, 4)
    pool = abi.Pool.for_shape(shape, 1, 4, conv_dtype=torch.float32)
    rng = np.random.default_rng(47)
    tok = tok_dev(synth.token_inputs(rng, 70, shape, "bf16"), "bf16")
    o = torch.zeros(70, 2, 128, device="cuda")
    for ck, every, status in (([[0]], 64, "GDN_ERR_DUP_SLOT"), ([[2, 2]], 64, "GDN_ERR_DUP_SLOT"),
                              ([[4]], 64, "GDN_ERR_SLOT"), ([[2]], 32, "GDN_ERR_ARG")):
        with pytest.raises(abi.GDNError) as e:
            abi.gdn_prefill_chunked_ckpt(pool, 0, dev_i32([0]), dev_i32([0, 70]), *tok, o,
                                         dev_i32(ck), every)
        assert e.value.name == status
    small = abi.Pool.for_shape(synth.LayerShape(2, 1, 16, 16, 16, 4), 1, 4,
                               conv_dtype=torch.float32)
    t16 = tok_dev(synth.token_inputs(rng, 70, synth.LayerShape(2, 1, 16, 16, 16, 4), "bf16"),
                  "bf16")
    with pytest.raises(abi.GDNError) as e:
        abi.gdn_prefill_chunked_ckpt(small, 0, dev_i32([0]), dev_i32([0, 70]), *t16,
                                     torch.zeros(70, 2, 16, device="cuda"), dev_i32([[2]]), 64)
    assert e.value.name == "GDN_ERR_UNSUPPORTED"


def _head_sample(tok, heads, group):
    """Slice value heads `heads` (and the key heads they read) out of a token dict."""
    kh = [h // group for h in heads]
    return {"q": tok["q"][:, kh], "k": tok["k"][:, kh], "v": tok["v"][:, heads],
            "g": tok["g"][:, heads], "beta": tok["beta"][:, heads]}


@pytest.mark.parametrize("entry", ["chunked", "recurrent"])
def test_prefill_varlen_pieces_full_size_sampled_heads(entry):
    """8 sequences with lengths uniform in [512, 8192], fed in 2048-token
    pieces with the state carried between calls; bf16 in and out; half the
    slots start from zero, half from N(0, 0.1).  The first piece-call is
    checked on all 32 value heads (outputs and the states it leaves); the
    whole sequences through the last call on value heads 0, 17 and 31."""
    wl = synth.prefill_workload(seed=3)
    s = wl["shape"]
    lens, cu = wl["lengths"], wl["cu_seqlens"]
    pool = _pool(s, 1, len(lens) + 2, conv_dtype=torch.bfloat16)
    ids = wl["slot_ids"] + 1                                   # slots 1..8; 0 and 9 untouched
    lid = torch.from_numpy(ids).long().cuda()
    pool.state[0, lid] = dev(wl["states"])
    tok_all = {n: dev(wl["tok"][n], "bf16") for n in ("q", "k", "v", "g", "beta")}
    o = torch.empty(int(cu[-1]), s.h_v, s.dv, device="cuda", dtype=torch.bfloat16)
    first = None
    for idx, starts, ln in synth.prefill_calls(lens, wl["piece"]):
        rows = np.concatenate([np.arange(cu[i] + st, cu[i] + st + l)
                               for i, st, l in zip(idx, starts, ln)])
        rt = torch.from_numpy(rows).long().cuda()
        packed = [tok_all[n][rt].contiguous() for n in ("q", "k", "v", "g", "beta")]
        ob = torch.empty(len(rows), s.h_v, s.dv, device="cuda", dtype=torch.bfloat16)
        PREFILL[entry](pool, 0, dev_i32(ids[idx]), dev_i32(synth.cu_seqlens_of(ln)),
                       *packed, ob, max_seqlen=max(ln))
        o[rt] = ob
        if first is None:                     # the first piece-call, every head
            first = (host(ob), host(pool.state[0, lid]), ln)
    group = s.h_v // s.h_k
    # all 32 value heads of the first piece-call (the first 2048 tokens of
    # every sequence, 15,204 tokens): one oracle task per sequence and key head
    o1, S1, ln1 = first
    tasks, where = [], []
    for i in range(len(lens)):
        lo = int(cu[i])
        for kh in range(s.h_k):
            hs = list(range(kh * group, (kh + 1) * group))
            sl = slice(lo, lo + ln1[i])
            tasks.append((wl["states"][i][hs], wl["tok"]["q"][sl, kh:kh + 1],
                          wl["tok"]["k"][sl, kh:kh + 1], wl["tok"]["v"][sl][:, hs],
                          wl["tok"]["g"][sl][:, hs], wl["tok"]["beta"][sl][:, hs]))
            where.append((i, hs))
    off = synth.cu_seqlens_of(ln1)
    for (i, hs), (S_ref, o_ref) in zip(where, recurrent_many(tasks)):
        assert_close_bf16(o1[off[i]:off[i + 1]][:, hs], o_ref, what=f"call 0 o seq {i} heads {hs}")
        assert_close_bf16(S1[i][hs], S_ref, what=f"call 0 S seq {i} heads {hs}")
    heads = [0, 17, 31]
    sub = _head_sample(wl["tok"], heads, group)
    for i in range(len(lens)):
        lo, hi = cu[i], cu[i + 1]
        S_ref, o_ref = O.gdn_recurrent(wl["states"][i][heads],
                                       *(sub[n][lo:hi] for n in ("q", "k", "v", "g", "beta")))
        assert_close_bf16(host(o[lo:hi][:, heads]), o_ref, what=f"o seq {i}")
        assert_close_bf16(host(pool.state[0, ids[i]][heads]), S_ref, what=f"S seq {i}")
    assert bool((pool.state[0, [0, 9]] == SENTINEL).all())


def test_prefill_device_guard_and_host_checks():
    shape = synth.LayerShape(2, 1, 16, 16, 16, 4)
    rng = np.random.default_rng(42)
    tok = tok_dev(synth.token_inputs(rng, 10, shape, "f32"), "f32")
    o = torch.zeros(10, 2, 16, device="cuda")
    pool = _pool(shape, 1, 4)
    with pytest.raises(abi.GDNError) as e:
        abi.gdn_prefill_chunked(pool, 0, dev_i32([0, 1]), dev_i32([0, 6, 9]), *tok, o)
    assert e.value.name == "GDN_ERR_SIZE"
    with pytest.raises(abi.GDNError) as e:
        abi.gdn_prefill_chunked(pool, 0, dev_i32([0, 0]), dev_i32([0, 6, 10]), *tok, o)
    assert e.value.name == "GDN_ERR_DUP_SLOT"
    pool.set_host_checks(False)
    abi.gdn_prefill_chunked(pool, 0, dev_i32([7, 1]), dev_i32([0, 6, 10]), *tok, o)
    assert abi.gdn_pool_get_error(pool) == abi.DEVERR_SLOT
    assert bool((pool.state[0, [0, 2, 3]] == SENTINEL).all())
    assert bool((o[:6] == 0).all())


@pytest.mark.parametrize("odt", ["bf16", "f32"])
def test_prefill_many_sequences_unaligned_outputs(odt):
    """dk = dv = 128, bf16 tensor-map rows, 300 sequences: more than the state
    kernel orders longest first (up to 256), so they are walked in index
    order; lengths 1..40 with a few whole and ragged multi-chunk ones; and an
    output tensor that does not start 16-byte aligned, so the state kernel
    stores element by element instead of staging whole rows (and of
    tensor-map stores for bf16).  Every output and every state against the
    oracle."""
    rng = np.random.default_rng(46)
    shape = synth.LayerShape(2, 1, 128, 128, 16, 4)
    n = 300
    lens = rng.integers(1, 41, n)
    lens[[7, 150, 299]] = [64, 130, 65]
    ids = rng.permutation(n + 10)[:n].astype(np.int32)
    cu = synth.cu_seqlens_of(lens)
    T = int(cu[-1])
    S0 = synth.random_states(rng, n, shape)
    tok = synth.token_inputs(rng, T, shape, "bf16")
    pool = _pool(shape, 1, n + 10)
    lid = torch.from_numpy(ids).long().cuda()
    pool.state[0, lid] = dev(S0)
    tdt = tdtype(odt)
    buf = torch.zeros(T * shape.h_v * shape.dv + 1, device="cuda", dtype=tdt)
    o = buf[1:].view(T, shape.h_v, shape.dv)       # one element past a 16-byte boundary
    abi.gdn_prefill_chunked(pool, 0, dev_i32(ids), dev_i32(cu), *tok_dev(tok, "bf16"), o,
                            max_seqlen=int(lens.max()))
    assert abi.gdn_pool_get_error(pool) == 0
    ref = O.OraclePool(1, n + 10, shape.h_v, shape.h_k, shape.dk, shape.dv, 16, 4)
    ref.S[0, ids] = S0
    o_ref = ref.prefill(0, ids, cu, *tok_np(tok))
    assert_close_bf16(host(o), o_ref, what="o")
    assert_maxrel(host(o), o_ref, _rel_tol(128), "o")
    assert_maxrel(host(pool.state[0, lid]), ref.S[0, ids], _rel_tol(128), "S")
    rest = np.setdiff1d(np.arange(n + 10), ids)
    assert bool((pool.state[0, torch.from_numpy(rest).long().cuda()] == SENTINEL).all())


def test_prefill_two_launch_overlapping_sequences_stay_in_bounds():
    """cu_seqlens [0, 200, 0, 200] (host checks off): the middle range is
    reversed and the last overlaps the first, so the sequences claim more
    64-token chunks (8) than the workspace holds (200 / 64 + 3 = 6).  The
    key-side kernel forms only the chunks within that capacity, the state
    kernel rejects the two bad sequences (error word: bad sequence) and leaves
    their slots alone, and the first sequence still matches the oracle."""
    rng = np.random.default_rng(46)
    shape = synth.LayerShape(4, 2, 128, 128, 16, 4)
    T = 200
    S0 = synth.random_states(rng, 1, shape)
    tok = synth.token_inputs(rng, T, shape, "bf16")
    pool = _pool(shape, 1, 4, host_checks=False)
    pool.state[0, 0] = dev(S0[0])
    o = torch.zeros(T, shape.h_v, shape.dv, device="cuda")
    abi.gdn_prefill_chunked(pool, 0, dev_i32([0, 1, 2]), dev_i32([0, T, 0, T]),
                            *tok_dev(tok, "bf16"), o)
    torch.cuda.synchronize()
    assert abi.gdn_pool_get_error(pool) == abi.DEVERR_SEQ
    assert bool((pool.state[0, [1, 2, 3]] == SENTINEL).all())
    ref = O.OraclePool(1, 1, shape.h_v, shape.h_k, shape.dk, shape.dv, 16, 4)
    ref.S[0, [0]] = S0
    o_ref = ref.prefill(0, np.array([0], dtype=np.int32), np.array([0, T]), *tok_np(tok))
    tol = _rel_tol(128)
    assert_maxrel(host(o), o_ref, tol, "o of the valid sequence")
    assert_maxrel(host(pool.state[0, 0]), ref.S[0, 0], tol, "S of the valid sequence")
