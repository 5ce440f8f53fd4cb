"""A decode step of several layers (conv + SiLU, then the decode step, per
layer) captured once into a CUDA graph and replayed with new inputs copied
into its static buffers: the small-batch latency path runs every launch from
one graph.  Replays must match the same calls made eagerly on a twin pool bit
for bit (same kernels, same inputs)."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrent_gb300 import abi, synth
from tests.gpu_util import dev, dev_i32

pytestmark = pytest.mark.gpu


def _step(pool, layers, ids, x, w, g, beta, y, o, shape, stream=None):
    n = ids.numel()
    nq = shape.h_k * shape.dk
    for layer in range(layers):
        abi.gdn_conv_silu(pool, layer, ids, x[layer], w[layer], y[layer], stream=stream)
        q = y[layer][:, :nq].view(n, shape.h_k, shape.dk)
        k = y[layer][:, nq:2 * nq].view(n, shape.h_k, shape.dk)
        v = y[layer][:, 2 * nq:].view(n, shape.h_v, shape.dv)
        abi.gdn_decode_step(pool, layer, ids, q, k, v, g[layer], beta[layer], o[layer],
                            stream=stream)


def test_decode_step_replayed_from_a_cuda_graph_matches_eager_calls():
    rng = np.random.default_rng(70)
    shape = synth.LayerShape(4, 2, 128, 128, 2 * 2 * 128 + 4 * 128, 4)
    layers, n_slots = 3, 6
    ids = dev_i32([4, 1, 5])
    n = ids.numel()
    S0 = synth.random_states(rng, layers * n_slots, shape).reshape(layers, n_slots, shape.h_v,
                                                                     shape.dv, shape.dk)
    pools = []
    for _ in range(2):   # graph pool, eager pool
        pool = abi.Pool.for_shape(shape, layers, n_slots, conv_dtype=torch.bfloat16,
                                  host_checks=False)
        pool.state.copy_(dev(S0))
        pools.append(pool)
    gpool, epool = pools
    w = [dev(synth.conv_weights(rng, shape.conv_ch, shape.conv_k)) for _ in range(layers)]

    def inputs():
        x = [dev(synth.conv_input(rng, n, shape.conv_ch, "bf16"), "bf16") for _ in range(layers)]
        tok = [synth.token_inputs(rng, n, shape, "bf16") for _ in range(layers)]
        return x, [dev(t["g"], "bf16") for t in tok], [dev(t["beta"], "bf16") for t in tok]

    sx, sg, sb = inputs()            # static input buffers of the graph
    sy = [torch.empty(n, shape.conv_ch, device="cuda", dtype=torch.bfloat16) for _ in range(layers)]
    so = [torch.empty(n, shape.h_v, shape.dv, device="cuda") for _ in range(layers)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            _step(gpool, layers, ids, sx, w, sg, sb, sy, so, shape, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    gpool.state.copy_(dev(S0))       # capture runs nothing; start both pools alike
    gpool.conv.zero_()
    epool.conv.zero_()
    ey = [torch.empty_like(t) for t in sy]
    eo = [torch.empty_like(t) for t in so]
    for step in range(3):
        x, g, b = inputs()
        for dst, src in zip(sx + sg + sb, x + g + b):
            dst.copy_(src)
        graph.replay()
        _step(epool, layers, ids, x, w, g, b, ey, eo, shape)
        torch.cuda.synchronize()
        for layer in range(layers):
            assert torch.equal(so[layer], eo[layer]), f"step {step} layer {layer}: outputs"
    assert torch.equal(gpool.state, epool.state)
    assert torch.equal(gpool.conv, epool.conv)
    assert abi.gdn_pool_get_error(gpool) == 0


def test_one_call_decode_step_replayed_from_a_cuda_graph_matches_eager_calls():
    """gdn_decode_step_conv under stream capture: its decode launch depends on
    the conv launch programmatically, an edge the graph must keep."""
    rng = np.random.default_rng(71)
    shape = synth.LayerShape(4, 2, 128, 128, 2 * 2 * 128 + 4 * 128, 4)
    layers, n_slots = 3, 6
    ids = dev_i32([2, 5, 0, 3])
    n = ids.numel()
    S0 = synth.random_states(rng, layers * n_slots, shape).reshape(layers, n_slots, shape.h_v,
                                                                     shape.dv, shape.dk)
    gpool, epool = (abi.Pool.for_shape(shape, layers, n_slots, conv_dtype=torch.bfloat16,
                                       host_checks=False) for _ in range(2))
    w = [dev(synth.conv_weights(rng, shape.conv_ch, shape.conv_k)) for _ in range(layers)]

    def inputs():
        x = [dev(synth.conv_input(rng, n, shape.conv_ch, "bf16"), "bf16") for _ in range(layers)]
        tok = [synth.token_inputs(rng, n, shape, "bf16") for _ in range(layers)]
        return x, [dev(t["g"], "bf16") for t in tok], [dev(t["beta"], "bf16") for t in tok]

    def step(pool, x, g, b, y, o, stream=None):
        for layer in range(layers):
            abi.gdn_decode_step_conv(pool, layer, ids, x[layer], w[layer], y[layer], g[layer],
                                     b[layer], o[layer], scale=shape.dk ** -0.5, stream=stream)

    sx, sg, sb = inputs()
    sy = [torch.empty(n, shape.conv_ch, device="cuda", dtype=torch.bfloat16) for _ in range(layers)]
    so = [torch.empty(n, shape.h_v, shape.dv, device="cuda") for _ in range(layers)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step(gpool, sx, sg, sb, sy, so, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for p in (gpool, epool):
        p.state.copy_(dev(S0))
        p.conv.zero_()
    ey = [torch.empty_like(t) for t in sy]
    eo = [torch.empty_like(t) for t in so]
    for it in range(3):
        x, g, b = inputs()
        for dst, src in zip(sx + sg + sb, x + g + b):
            dst.copy_(src)
        graph.replay()
        step(epool, x, g, b, ey, eo)
        torch.cuda.synchronize()
        for layer in range(layers):
            assert torch.equal(so[layer], eo[layer]), f"step {it} layer {layer}: outputs"
    assert torch.equal(gpool.state, epool.state)
    assert torch.equal(gpool.conv, epool.conv)
    assert abi.gdn_pool_get_error(gpool) == 0
