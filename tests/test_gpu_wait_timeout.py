"""The bounded-wait error path of the decode kernels, made to run out without
a fault: the test hook GDN_TEST_DECODE_WAIT_TIMEOUT makes each CTA's copy
barrier expect 16 bytes more than its state-tile copy delivers, so the copy
lands and the bounded wait expires.  The kernel must report
GDN_DEVERR_TIMEOUT in the pool's error word, leave the state and o untouched,
and leave the context usable: with the hook cleared the same pool decodes
correctly (against the oracle) right after."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrent_gb300 import abi, synth
from oracle import gdn_oracle as O
from tests.gpu_util import assert_maxrel, dev, dev_i32, host, tok_dev, tok_np

pytestmark = pytest.mark.gpu


def test_decode_wait_timeout_reports_and_recovers():
    rng = np.random.default_rng(96)
    shape = synth.LayerShape(2, 1, 32, 32, 2 * 32 + 2 * 32, 4)   # one CTA per value head
    pool = abi.Pool.for_shape(shape, 1, 3, conv_dtype=torch.float32)
    S0 = synth.random_states(rng, 3, shape)
    pool.state[0] = dev(S0)
    before = pool.state.clone()
    tok = synth.token_inputs(rng, 1, shape, "f32")
    o = torch.full((1, shape.h_v, shape.dv), 5.0, device="cuda")

    abi.gdn_pool_set_test_flags(pool, abi.TEST_DECODE_WAIT_TIMEOUT)
    abi.gdn_decode_step(pool, 0, dev_i32([1]), *tok_dev(tok, "f32"), o)
    assert abi.gdn_pool_get_error(pool) == abi.DEVERR_TIMEOUT
    assert torch.equal(pool.state, before), "a timed-out CTA must not write its state rows"
    assert bool((o == 5.0).all()), "a timed-out CTA must not write o"
    # the one-call step (one fused kernel at this size) takes the same path
    x = dev(synth.conv_input(rng, 1, shape.conv_ch, "f32"))
    w = dev(synth.conv_weights(rng, shape.conv_ch, shape.conv_k))
    y = torch.empty(1, shape.conv_ch, device="cuda")
    abi.gdn_decode_step_conv(pool, 0, dev_i32([1]), x, w, y, dev(tok["g"]), dev(tok["beta"]), o)
    assert abi.gdn_pool_get_error(pool) == abi.DEVERR_TIMEOUT
    assert torch.equal(pool.state, before)
    assert bool((o == 5.0).all())

    # hook cleared: the same pool and context decode correctly
    abi.gdn_pool_set_test_flags(pool, 0)
    abi.gdn_decode_step(pool, 0, dev_i32([2]), *tok_dev(tok, "f32"), o)
    S_ref, o_ref = O.gdn_step(S0[2], *(a[0] for a in tok_np(tok)))
    assert_maxrel(host(o[0]), o_ref, 1e-4, "o after recovery")
    assert_maxrel(host(pool.state[0, 2]), S_ref, 1e-4, "S after recovery")
    assert abi.gdn_pool_get_error(pool) == 0
    with pytest.raises(abi.GDNError) as e:
        abi.gdn_pool_set_test_flags(pool, 2)
    assert e.value.name == "GDN_ERR_ARG"


def test_fused_step_per_key_head_wait_timeout_reports_and_recovers():
    """The same hook on the one-call step's per-(slot, key head) kernel (the
    decode-step layer at 16 slots: the per-row-block grid does not fit the GPU
    at once, so one launch of 256 CTAs, each streaming its two heads' states
    through a ring of tiles).  Tile 0's wait runs out in every CTA, which then
    waits once more for every tile still in flight and returns: the error word
    says so, no state row and no o changes, and the pool decodes correctly
    afterwards."""
    rng = np.random.default_rng(97)
    shape = synth.GDN_LAYER
    n = 16
    pool = abi.Pool.for_shape(shape, 1, n + 1, conv_dtype=torch.bfloat16)
    gen = torch.Generator(device="cuda").manual_seed(9)
    pool.state.normal_(0.0, 0.1, generator=gen)
    before = pool.state.clone()
    ids = dev_i32(list(range(n)))
    assert abi.gdn_decode_step_conv_launches(pool, n, torch.bfloat16) == 1
    x = dev(synth.conv_input(rng, n, shape.conv_ch, "bf16"), "bf16")
    w = dev(synth.conv_weights(rng, shape.conv_ch, shape.conv_k))
    tok = synth.token_inputs(rng, n, shape, "bf16")
    y = torch.empty(n, shape.conv_ch, device="cuda", dtype=torch.bfloat16)
    o = torch.full((n, shape.h_v, shape.dv), 5.0, device="cuda")

    abi.gdn_pool_set_test_flags(pool, abi.TEST_DECODE_WAIT_TIMEOUT)
    abi.gdn_decode_step_conv(pool, 0, ids, x, w, y, dev(tok["g"], "bf16"),
                             dev(tok["beta"], "bf16"), o)
    assert abi.gdn_pool_get_error(pool) == abi.DEVERR_TIMEOUT
    assert torch.equal(pool.state, before), "a timed-out CTA must not write its state rows"
    assert bool((o == 5.0).all()), "a timed-out CTA must not write o"

    abi.gdn_pool_set_test_flags(pool, 0)
    t1 = synth.token_inputs(rng, 1, shape, "f32")
    o1 = torch.empty(1, shape.h_v, shape.dv, device="cuda")
    S0 = host(pool.state[0, n])
    abi.gdn_decode_step(pool, 0, dev_i32([n]), *tok_dev(t1, "f32"), o1)
    S_ref, o_ref = O.gdn_step(S0, *(a[0] for a in tok_np(t1)))
    assert_maxrel(host(o1[0]), o_ref, 1e-4, "o after recovery")
    assert_maxrel(host(pool.state[0, n]), S_ref, 1e-4, "S after recovery")
    assert abi.gdn_pool_get_error(pool) == 0
