"""gdn_prefill_chunked_noalloc: the chunked prefill for callers that cannot
allocate device memory (their allocator owns the GPU, or a step must not
allocate), whose workspace is a fixed 64 MiB array inside the library.

Checked through the C ABI against gdn_prefill_chunked on two calls in a row
(the second continues the first call's sequences from the carried state, and
reuses the array the first call left behind).  Both entry points run the same
kernels, so outputs and states are held to the path-equivalence tolerance of
the prefill tests: max|a - b| <= 1e-5 * max|b|.  A call that needs more
scratch than the array holds is refused with GDN_ERR_SIZE.

This file is collected last on purpose, so that a run stopping at the first
failure has run every other test before it."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrent_gb300 import abi, synth
from tests.gpu_util import assert_maxrel, dev, dev_i32, host, tok_dev

pytestmark = pytest.mark.gpu


def test_noalloc_prefill_matches_chunked_prefill_on_two_calls():
    rng = np.random.default_rng(50)
    shape = synth.LayerShape(32, 16, 128, 128, 16, 4)   # dk = dv = 128: the workspace path
    ids = np.array([3, 0, 5], dtype=np.int32)
    lid = torch.from_numpy(ids).long().cuda()
    S0 = synth.random_states(rng, len(ids), shape)
    pools = {}
    for name in ("noalloc", "chunked"):
        pool = abi.Pool.for_shape(shape, 1, 6, conv_dtype=torch.float32)
        pool.state[0, lid] = dev(S0)
        pools[name] = pool
    fns = {"noalloc": abi.gdn_prefill_chunked_noalloc, "chunked": abi.gdn_prefill_chunked}
    for call, lens in enumerate(([300, 129, 1], [200, 64, 77])):
        cu = synth.cu_seqlens_of(lens)
        tok = tok_dev(synth.token_inputs(rng, int(cu[-1]), shape, "bf16"), "bf16")
        outs = {}
        for name, pool in pools.items():
            o = torch.empty(int(cu[-1]), shape.h_v, shape.dv, device="cuda")
            fns[name](pool, 0, dev_i32(ids), dev_i32(cu), *tok, o, max_seqlen=max(lens))
            outs[name] = host(o)
        assert_maxrel(outs["noalloc"], outs["chunked"], 1e-5, f"o, call {call}")
        assert_maxrel(host(pools["noalloc"].state[0, lid]), host(pools["chunked"].state[0, lid]),
                      1e-5, f"S, call {call}")
    for pool in pools.values():
        assert abi.gdn_pool_get_error(pool) == 0


def test_noalloc_prefill_refuses_calls_beyond_its_array():
    shape = synth.LayerShape(32, 16, 128, 128, 16, 4)
    pool = abi.Pool.for_shape(shape, 1, 2, conv_dtype=torch.float32)
    before = pool.state.clone()
    n = 64 * 64                  # (64 + 1) chunks x 32 heads x 32 KiB > 64 MiB
    rng = np.random.default_rng(51)
    tok = tok_dev(synth.token_inputs(rng, n, shape, "bf16"), "bf16")
    o = torch.zeros(n, shape.h_v, shape.dv, device="cuda")
    with pytest.raises(abi.GDNError) as e:
        abi.gdn_prefill_chunked_noalloc(pool, 0, dev_i32([1]), dev_i32([0, n]), *tok, o)
    assert e.value.name == "GDN_ERR_SIZE"
    torch.cuda.synchronize()
    assert torch.equal(pool.state, before)
    assert bool((o == 0).all())


def test_noalloc_prefill_on_a_side_stream_small_call_then_larger_call():
    """A smaller call followed by a larger one (more sequences, more chunks,
    bf16 outputs), both on a non-default stream: the second call must read
    nothing the first left in the shared array."""
    rng = np.random.default_rng(52)
    shape = synth.LayerShape(8, 4, 128, 128, 16, 4)
    ids = [np.array([2], dtype=np.int32), np.array([4, 1, 0, 6], dtype=np.int32)]
    S0 = synth.random_states(rng, 7, shape)
    pools = {}
    for name in ("noalloc", "chunked"):
        pool = abi.Pool.for_shape(shape, 1, 7, conv_dtype=torch.float32)
        pool.state[0] = dev(S0)
        pools[name] = pool
    fns = {"noalloc": abi.gdn_prefill_chunked_noalloc, "chunked": abi.gdn_prefill_chunked}
    side = torch.cuda.Stream()
    for call, (sid, lens, odt) in enumerate(((ids[0], [70], torch.float32),
                                             (ids[1], [300, 5, 129, 64], torch.bfloat16))):
        cu = synth.cu_seqlens_of(lens)
        tok = tok_dev(synth.token_inputs(rng, int(cu[-1]), shape, "bf16"), "bf16")
        sid_d, cu_d = dev_i32(sid), dev_i32(cu)
        side.wait_stream(torch.cuda.current_stream())      # inputs copied on the default stream
        outs = {}
        with torch.cuda.stream(side):
            for name, pool in pools.items():
                o = torch.empty(int(cu[-1]), shape.h_v, shape.dv, device="cuda", dtype=odt)
                fns[name](pool, 0, sid_d, cu_d, *tok, o, max_seqlen=max(lens), stream=side)
                outs[name] = o
        side.synchronize()
        assert_maxrel(host(outs["noalloc"]), host(outs["chunked"]), 1e-5, f"o, call {call}")
        assert_maxrel(host(pools["noalloc"].state), host(pools["chunked"].state), 1e-5,
                      f"S, call {call}")
    for pool in pools.values():
        assert abi.gdn_pool_get_error(pool) == 0
