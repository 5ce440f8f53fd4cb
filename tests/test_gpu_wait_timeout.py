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
