"""gdn_decode_step_conv: conv + SiLU and the decode step of one layer in one
call -- one fused kernel per (row block, value head, slot) while its grid fits
the GPU at once (few slots), else one fused kernel per (slot, key head) where
the shape allows it (dk = 128, float32 state, h_v / h_k <= 2), else the conv
launch with the decode as its programmatic dependent launch.  The first two
are exercised here (the decode-step layer with 4 and with 64 slots, and a
two-head layer with 512 slots, conv width 3, float32 activations); the launch
pair runs for the other large shapes.

Checked through the C ABI over three consecutive steps:
  * y against the float64 oracle's conv + SiLU (bf16: |got - ref| <= 1e-2 +
    1e-2 |ref| elementwise; f32: max|got - ref| <= 1e-5 max|ref|), and the
    conv cache bit for bit (it holds raw inputs);
  * o and the state against the oracle's decode step run on the y the GPU
    produced (those are the decode's inputs), max|got - ref| <= 1e-4 max|ref|,
    the tolerance of the plain decode test;
  * every output, cache and state bit-identical to gdn_conv_silu followed by
    gdn_decode_step on a twin pool (same kernels and inputs; only the launch
    overlap differs);
  * slots that are not listed keep a sentinel."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrent_gb300 import abi, synth
from oracle import gdn_oracle as O
from tests.gpu_util import assert_close_bf16, assert_maxrel, dev, dev_i32, host

pytestmark = pytest.mark.gpu

SENTINEL = 3.25

CASES = {
    # decode-step layer shape: 32/16 heads, K = V = 128, 64 of 256 slots, bf16
    "gdn_layer_bf16": dict(shape=synth.GDN_LAYER, n_slots=256, n_active=64, dtype="bf16",
                           pad_x=0, pad_y=0, bias=False, layer=0, n_layers=1),
    # the same layer with 4 slots: one fused kernel
    "gdn_layer_bf16_few": dict(shape=synth.GDN_LAYER, n_slots=256, n_active=4, dtype="bf16",
                               pad_x=0, pad_y=0, bias=False, layer=0, n_layers=1),
    # conv width 3 (the generic-width fused kernel), float32
    "small_f32_w3": dict(shape=synth.LayerShape(4, 2, 32, 32, 256, 3), n_slots=9, n_active=5,
                         dtype="f32", pad_x=0, pad_y=0, bias=True, layer=1, n_layers=2),
    # small heads in float32, second layer of two, with a conv bias
    "small_f32": dict(shape=synth.LayerShape(4, 2, 32, 32, 256, 4), n_slots=9, n_active=5,
                      dtype="f32", pad_x=0, pad_y=0, bias=True, layer=1, n_layers=2),
    # bf16 with padded row strides of x and y
    "small_bf16_strided": dict(shape=synth.LayerShape(4, 2, 64, 64, 512, 4), n_slots=7,
                               n_active=3, dtype="bf16", pad_x=16, pad_y=8, bias=True, layer=0,
                               n_layers=1),
    # the per-(slot, key head) kernel with one value head per key head, conv
    # width 3 (its generic-width instantiation), float32 activations, bias
    "group_f32_w3_g1": dict(shape=synth.LayerShape(2, 2, 128, 128, 768, 3), n_slots=520,
                            n_active=512, dtype="f32", pad_x=0, pad_y=0, bias=True, layer=1,
                            n_layers=2),
    # the decode-step layer at 64 slots with bf16 outputs
    "gdn_layer_bf16_obf16": dict(shape=synth.GDN_LAYER, n_slots=256, n_active=64, dtype="bf16",
                                 pad_x=0, pad_y=0, bias=False, layer=0, n_layers=1,
                                 o_dtype="bf16"),
}


def _pool(shape, n_layers, n_slots, tdt):
    p = abi.Pool.for_shape(shape, n_layers, n_slots, conv_dtype=tdt)
    p.state.fill_(SENTINEL)
    p.conv.fill_(-SENTINEL)
    return p


@pytest.mark.parametrize("case", list(CASES))
def test_decode_step_conv_matches_oracle_and_two_calls(case):
    c = CASES[case]
    shape, dt, L = c["shape"], c["dtype"], c["layer"]
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    rng = np.random.default_rng(60 + len(case))
    ids = rng.choice(c["n_slots"], c["n_active"], replace=False).astype(np.int32)
    lid = torch.from_numpy(ids).long().cuda()
    n = len(ids)
    S0 = synth.random_states(rng, n, shape)
    C0 = synth.random_conv_cache(rng, n, shape, dt)
    w = synth.conv_weights(rng, shape.conv_ch, shape.conv_k)
    bias = synth.cast(rng.standard_normal(shape.conv_ch), "f32") if c["bias"] else None
    fused, split = (_pool(shape, c["n_layers"], c["n_slots"], tdt) for _ in range(2))
    for p in (fused, split):
        p.state[L, lid] = dev(S0)
        p.conv[L, lid] = dev(C0, dt)
    ref = O.OraclePool(1, c["n_slots"], shape.h_v, shape.h_k, shape.dk, shape.dv,
                       shape.conv_ch, shape.conv_k)
    ref.X[0, ids] = C0
    S_ref = S0.astype(np.float64)
    W = dev(w)
    Bias = None if bias is None else dev(bias)
    C, nq = shape.conv_ch, shape.h_k * shape.dk
    scale = shape.dk ** -0.5

    def rows(width):
        return torch.empty(n, width, device="cuda", dtype=tdt)[:, :C]

    for step in range(3):
        x = synth.conv_input(rng, n, C, dt)
        tok = synth.token_inputs(rng, n, shape, dt)
        X = rows(C + c["pad_x"])
        X.copy_(dev(x, dt))
        G, B = dev(tok["g"], dt), dev(tok["beta"], dt)
        Y, Y2 = rows(C + c["pad_y"]), rows(C + c["pad_y"])
        odt = torch.bfloat16 if c.get("o_dtype") == "bf16" else torch.float32
        o = torch.empty(n, shape.h_v, shape.dv, device="cuda", dtype=odt)
        o2 = torch.empty_like(o)
        abi.gdn_decode_step_conv(fused, L, dev_i32(ids), X, W, Y, G, B, o, bias=Bias, scale=scale)
        abi.gdn_conv_silu(split, L, dev_i32(ids), X, W, Y2, bias=Bias)
        abi.gdn_decode_step(split, L, dev_i32(ids), Y2[:, :nq].view(n, shape.h_k, shape.dk),
                            Y2[:, nq:2 * nq].view(n, shape.h_k, shape.dk),
                            Y2[:, 2 * nq:].view(n, shape.h_v, shape.dv), G, B, o2, scale=scale)
        torch.cuda.synchronize()
        what = f"{case} step {step}"
        assert torch.equal(Y, Y2), f"{what}: y differs from the two-call path"
        assert torch.equal(o, o2), f"{what}: o differs from the two-call path"
        assert torch.equal(fused.state, split.state), f"{what}: state differs"
        assert torch.equal(fused.conv, split.conv), f"{what}: conv cache differs"

        y_ref = ref.conv_silu(0, ids, None, x, w, bias)
        if dt == "bf16":
            assert_close_bf16(host(Y), y_ref, what=f"{what}: y")
        else:
            assert_maxrel(host(Y), y_ref, 1e-5, f"{what}: y")
        np.testing.assert_array_equal(host(fused.conv[L, lid]), ref.X[0, ids])
        y = host(Y)
        q = y[:, :nq].reshape(n, shape.h_k, shape.dk)
        k = y[:, nq:2 * nq].reshape(n, shape.h_k, shape.dk)
        v = y[:, 2 * nq:].reshape(n, shape.h_v, shape.dv)
        o_ref = np.empty((n, shape.h_v, shape.dv))
        for i in range(n):
            S_ref[i], o_ref[i] = O.gdn_step(S_ref[i], q[i], k[i], v[i], tok["g"][i],
                                            tok["beta"][i], scale=scale)
        if odt == torch.bfloat16:
            assert_close_bf16(host(o), o_ref, what=f"{what}: o")
        else:
            assert_maxrel(host(o), o_ref, 1e-4, f"{what}: o")
        assert_maxrel(host(fused.state[L, lid]), S_ref, 1e-4, f"{what}: S")

    mask = np.ones(c["n_slots"], dtype=bool)
    mask[ids] = False
    rest = torch.from_numpy(np.nonzero(mask)[0]).cuda()
    assert bool((fused.state[:, rest] == SENTINEL).all()), "unlisted state slots changed"
    assert bool((fused.conv[:, rest] == -SENTINEL).all()), "unlisted conv slots changed"
    if c["n_layers"] > 1:
        assert bool((fused.state[1 - L] == SENTINEL).all()), "other layer's states changed"
    assert abi.gdn_pool_get_error(fused) == 0


def test_decode_step_conv_argument_checks():
    shape = synth.LayerShape(4, 2, 32, 32, 256, 4)
    pool = abi.Pool.for_shape(shape, 1, 4, conv_dtype=torch.bfloat16)
    n = 2
    ids = dev_i32([0, 3])
    w = torch.zeros(shape.conv_ch, shape.conv_k, device="cuda")
    x = torch.zeros(n, shape.conv_ch, device="cuda", dtype=torch.bfloat16)
    y = torch.zeros_like(x)
    g = torch.zeros(n, shape.h_v, device="cuda", dtype=torch.bfloat16)
    b = torch.zeros_like(g)
    o = torch.zeros(n, shape.h_v, shape.dv, device="cuda")
    before = pool.state.clone(), pool.conv.clone()
    # float32 inputs on a bf16 pool
    with pytest.raises(abi.GDNError) as e:
        abi.gdn_decode_step_conv(pool, 0, ids, x.float(), w, y.float(), g.float(), b.float(), o)
    assert e.value.name == "GDN_ERR_DTYPE"
    # conv channels that do not split into q | k | v
    other = synth.LayerShape(4, 2, 32, 32, 264, 4)
    pool2 = abi.Pool.for_shape(other, 1, 4, conv_dtype=torch.bfloat16)
    x2 = torch.zeros(n, other.conv_ch, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(abi.GDNError) as e:
        abi.gdn_decode_step_conv(pool2, 0, ids, x2, torch.zeros(other.conv_ch, other.conv_k,
                                 device="cuda"), torch.zeros_like(x2), g, b, o)
    assert e.value.name == "GDN_ERR_SIZE"
    # a slot outside the pool (host checks on)
    with pytest.raises(abi.GDNError) as e:
        abi.gdn_decode_step_conv(pool, 0, dev_i32([0, 4]), x, w, y, g, b, o)
    assert e.value.name == "GDN_ERR_SLOT"
    torch.cuda.synchronize()
    assert torch.equal(pool.state, before[0]) and torch.equal(pool.conv, before[1])
    assert bool((o == 0).all()) and bool((y == 0).all())


def test_decode_step_conv_alternating_forms_keep_the_cache_consistent():
    """Steps with 4, 64, 4, 64 active slots of one pool (fused kernel, then
    the launch pair, alternately; the fused kernel's tickets must end every
    launch at zero) match a twin pool stepped with the two separate calls,
    bit for bit."""
    shape = synth.GDN_LAYER
    rng = np.random.default_rng(66)
    ids_all = rng.choice(256, 64, replace=False).astype(np.int32)
    one, two = (_pool(shape, 1, 256, torch.bfloat16) for _ in range(2))
    gen = torch.Generator(device="cuda").manual_seed(6)
    one.state.normal_(0.0, 0.1, generator=gen)
    one.conv.copy_(torch.randn(one.conv.shape, device="cuda", generator=gen))
    two.state.copy_(one.state)
    two.conv.copy_(one.conv)
    w = dev(synth.conv_weights(rng, shape.conv_ch, shape.conv_k))
    nq = shape.h_k * shape.dk
    for step, n in enumerate((4, 64, 4, 64, 4)):
        ids = dev_i32(ids_all[:n])
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
        assert torch.equal(y1, y2) and torch.equal(o1, o2), f"step {step} (n = {n})"
        assert torch.equal(one.state, two.state), f"step {step}: state"
        assert torch.equal(one.conv, two.conv), f"step {step}: conv cache"
    assert abi.gdn_pool_get_error(one) == 0


def test_decode_step_conv_launch_count_query():
    """gdn_decode_step_conv_launches reports the form the call takes: one
    launch for the fused forms (few slots; the decode-step layer at 64 slots),
    two for the launch pair (a shape the per-key-head kernel does not take,
    dk = 64, with a grid too large to be resident at once), 0 for no slots;
    bad arguments are refused."""
    big = _pool(synth.GDN_LAYER, 1, 8, torch.bfloat16)
    assert abi.gdn_decode_step_conv_launches(big, 4, torch.bfloat16) == 1
    assert abi.gdn_decode_step_conv_launches(big, 64, torch.bfloat16, torch.bfloat16) == 1
    assert abi.gdn_decode_step_conv_launches(big, 0, torch.bfloat16) == 0
    small = _pool(synth.LayerShape(4, 2, 64, 64, 512, 4), 1, 8, torch.bfloat16)
    assert abi.gdn_decode_step_conv_launches(small, 8000, torch.bfloat16) == 2
    with pytest.raises(abi.GDNError) as e:
        abi.gdn_decode_step_conv_launches(big, -1, torch.bfloat16)
    assert e.value.name == "GDN_ERR_ARG"
    with pytest.raises(abi.GDNError) as e:
        abi.gdn_decode_step_conv_launches(big, 4, torch.float32)
    assert e.value.name == "GDN_ERR_DTYPE"


def test_decode_step_conv_bad_slot_skipped_in_both_fused_forms():
    """Host checks off, one slot id out of range among 4 and among 16 active
    slots of the decode-step layer (the per-row-block and the per-(slot, key
    head) fused kernels): the error word reports the bad slot, its entry
    writes nothing, and every other entry equals the two separate calls on a
    twin pool, bit for bit."""
    shape = synth.GDN_LAYER
    nq = shape.h_k * shape.dk
    rng = np.random.default_rng(67)
    for n in (4, 16):
        pools = []
        for _ in range(2):
            p = abi.Pool.for_shape(shape, 1, 32, conv_dtype=torch.bfloat16, host_checks=False)
            pools.append(p)
        gen = torch.Generator(device="cuda").manual_seed(7)
        pools[0].state.normal_(0.0, 0.1, generator=gen)
        pools[0].conv.copy_(torch.randn(pools[0].conv.shape, device="cuda", generator=gen))
        pools[1].state.copy_(pools[0].state)
        pools[1].conv.copy_(pools[0].conv)
        ids = rng.choice(32, n, replace=False).astype(np.int32)
        ids[1] = 99  # out of range
        good = np.array([i for i in range(n) if i != 1])
        x = dev(synth.conv_input(rng, n, shape.conv_ch, "bf16"), "bf16")
        w = dev(synth.conv_weights(rng, shape.conv_ch, shape.conv_k))
        tok = synth.token_inputs(rng, n, shape, "bf16")
        g, b = dev(tok["g"], "bf16"), dev(tok["beta"], "bf16")
        y1 = torch.zeros(n, shape.conv_ch, device="cuda", dtype=torch.bfloat16)
        y2 = torch.zeros_like(y1)
        o1 = torch.full((n, shape.h_v, shape.dv), 5.0, device="cuda")
        o2 = torch.full_like(o1, 5.0)
        abi.gdn_decode_step_conv(pools[0], 0, dev_i32(ids), x, w, y1, g, b, o1)
        abi.gdn_conv_silu(pools[1], 0, dev_i32(ids), x, w, y2)
        abi.gdn_decode_step(pools[1], 0, dev_i32(ids), y2[:, :nq].view(n, shape.h_k, shape.dk),
                            y2[:, nq:2 * nq].view(n, shape.h_k, shape.dk),
                            y2[:, 2 * nq:].view(n, shape.h_v, shape.dv), g, b, o2)
        torch.cuda.synchronize()
        for p in pools:
            assert abi.gdn_pool_get_error(p) == abi.DEVERR_SLOT, f"n = {n}"
        gi = torch.from_numpy(good).cuda()
        assert torch.equal(y1[gi], y2[gi]) and torch.equal(o1[gi], o2[gi]), f"n = {n}"
        assert bool((o1[1] == 5.0).all()) and bool((y1[1] == 0).all()), f"n = {n}: bad entry"
        assert torch.equal(pools[0].state, pools[1].state), f"n = {n}: state"
        assert torch.equal(pools[0].conv, pools[1].conv), f"n = {n}: conv cache"
