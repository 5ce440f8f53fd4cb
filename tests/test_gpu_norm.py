"""gdn_gated_rmsnorm (the layer's output gated RMSNorm) against the float64
oracle, through the C ABI.

Tolerances: float32 output max|got - ref| <= 1e-5 * max|ref| (one float32
sum of squares over d <= 1024 terms, rsqrt, expf); bf16 output elementwise
|got - ref| <= 1e-2 + 1e-2 |ref|.  Inputs are the rounded values the kernel
reads, so both sides see the same numbers."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrent_gb300 import abi, synth
from oracle import gdn_oracle as O
from tests.gpu_util import assert_close_bf16, assert_maxrel, dev, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,d,o_dt,z_dt,y_dt", [
    (64 * 32, 128, "f32", "bf16", "bf16"),   # decode-step layer: 64 tokens x 32 heads
    (64 * 32, 128, "f32", "bf16", "f32"),
    (37, 40, "bf16", "f32", "f32"),          # ragged rows, d not a multiple of 32
    (33, 256, "bf16", "bf16", "bf16"),       # vector path, two rows per warp, odd tail
    (7, 512, "f32", "bf16", "f32"),          # vector path, one row per warp
    (5, 1024, "f32", "f32", "f32"),
    (3, 1, "f32", "f32", "bf16"),
])
def test_gated_rmsnorm_matches_oracle(rows, d, o_dt, z_dt, y_dt):
    rng = np.random.default_rng(rows + d)
    o = synth.cast(rng.standard_normal((rows, d)) * 0.3, o_dt)
    z = synth.cast(rng.standard_normal((rows, d)) * 2.0, z_dt)
    w = synth.cast(rng.uniform(0.5, 1.5, d), "f32")
    y = torch.full((rows, d), 7.0, device="cuda",
                   dtype=torch.float32 if y_dt == "f32" else torch.bfloat16)
    abi.gdn_gated_rmsnorm(dev(o, o_dt), dev(z, z_dt), dev(w), y, eps=1e-6)
    ref = O.gated_rmsnorm(o, z, w, eps=1e-6)
    if y_dt == "f32":
        assert_maxrel(host(y), ref, 1e-5, "y")
    else:
        assert_close_bf16(host(y), ref, what="y")


def test_gated_rmsnorm_zero_rows_and_rejects():
    w = torch.ones(16, device="cuda")
    o = torch.zeros(4, 16, device="cuda")
    y = abi.gdn_gated_rmsnorm(o, torch.ones_like(o), w)       # zero rows, eps > 0: zeros
    assert bool((y == 0).all())
    empty = torch.empty(0, 16, device="cuda")
    abi.gdn_gated_rmsnorm(empty, empty, w, torch.empty_like(empty))   # no-op
    with pytest.raises(abi.GDNError) as e:
        abi.gdn_gated_rmsnorm(o, o, w, eps=-1.0)
    assert e.value.name == "GDN_ERR_ARG"
    torch.cuda.synchronize()
