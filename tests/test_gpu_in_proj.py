"""gdn_in_proj (the layer's input projection, y = x w^T on the tensor cores)
against the float64 oracle's in_proj, through the C ABI.

Inputs are bf16 (x ~ N(0, 1), w ~ N(0, 1/hidden)); both sides multiply the
same exact bf16 values.  The GPU accumulates in float32, so a float32 y is
held to max|gpu - ref| <= 1e-5 * max|ref|; a bf16 y is additionally rounded
once, |gpu - ref| <= 2^-8 |ref| + 1e-5 max|ref| elementwise.  Shapes cover a
decode step (64 tokens), ragged token counts (M tails), output widths that
are not a multiple of the tile (N tails) and hidden sizes that are not a
multiple of the 64-wide K block (zero-filled K tails), on each of the three
kernel forms (chosen by the number of output tiles)."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrent_gb300 import abi, synth
from oracle import gdn_oracle as O
from tests.gpu_util import assert_maxrel, host

pytestmark = pytest.mark.gpu

HIDDEN = 2048
N_OUT = 2 * 16 * 128 + 32 * 128 + 32 * 128 + 2 * 32   # q | k | v, gate z, beta and decay logits


def _pool():
    return abi.Pool.for_shape(synth.LayerShape(2, 1, 16, 16, 64, 4), 1, 1,
                              conv_dtype=torch.float32)


def _inputs(rng, tokens, hidden, n_out):
    x = synth.cast(rng.standard_normal((tokens, hidden)), "bf16")
    w = synth.cast(rng.standard_normal((n_out, hidden)) / np.sqrt(hidden), "bf16")
    return x, w


# 64 / 300 tokens: 96-column tiles (one wave); 512, 2000: 128-column tiles, two
# CTAs per SM; 2048 and 4100 (with M, N and K tails): the persistent kernel
# (128 x 256 tiles, double-buffered TMEM)
@pytest.mark.parametrize("tokens,hidden,n_out", [(64, HIDDEN, N_OUT), (300, HIDDEN, N_OUT),
                                                 (512, HIDDEN, N_OUT), (2048, HIDDEN, N_OUT),
                                                 (1, 64, 16), (130, 200, 72), (257, 1000, 344),
                                                 (2000, 520, 3000), (4100, 200, 4904)])
@pytest.mark.parametrize("ydt", ["f32", "bf16"])
def test_in_proj_matches_oracle(tokens, hidden, n_out, ydt):
    rng = np.random.default_rng(tokens + hidden + n_out)
    x, w = _inputs(rng, tokens, hidden, n_out)
    pool = _pool()
    tdt = torch.float32 if ydt == "f32" else torch.bfloat16
    y = torch.full((tokens, n_out), 7.0, device="cuda", dtype=tdt)
    abi.gdn_in_proj(pool, torch.from_numpy(x).cuda().bfloat16(),
                    torch.from_numpy(w).cuda().bfloat16(), y)
    ref = O.in_proj(x, w)
    got = host(y)
    if ydt == "f32":
        assert_maxrel(got, ref, 1e-5, "y")
    else:
        lim = 2.0 ** -8 * np.abs(ref) + 1e-5 * np.abs(ref).max()
        bad = np.abs(got - ref) > lim
        assert not bad.any(), f"{bad.sum()} elements outside the bf16 bound"
    assert abi.gdn_pool_get_error(pool) == 0


def test_in_proj_strided_rows_and_argument_checks():
    """Row strides wider than a row (a view into larger buffers) give the same
    result; misaligned rows, wrong dtypes and zero tokens are handled."""
    rng = np.random.default_rng(95)
    x, w = _inputs(rng, 100, 256, 96)
    pool = _pool()
    xd = torch.from_numpy(x).cuda().bfloat16()
    wd = torch.from_numpy(w).cuda().bfloat16()
    xw = torch.zeros(100, 256 + 64, device="cuda", dtype=torch.bfloat16)
    xw[:, :256] = xd
    yw = torch.zeros(100, 96 + 32, device="cuda")
    abi.gdn_in_proj(pool, xw[:, :256], wd, yw[:, :96])
    y = abi.gdn_in_proj(pool, xd, wd)
    torch.cuda.synchronize()
    assert torch.equal(yw[:, :96], y)
    assert bool((yw[:, 96:] == 0).all())
    assert_maxrel(host(y), O.in_proj(x, w), 1e-5, "y")
    with pytest.raises(abi.GDNError) as e:        # rows not 16-byte aligned
        abi.gdn_in_proj(pool, xw[:, 1:257], wd)
    assert e.value.name == "GDN_ERR_ARG"
    with pytest.raises(abi.GDNError):
        abi.gdn_in_proj(pool, xd.float(), wd)
    empty = abi.gdn_in_proj(pool, xd[:0], wd)
    assert empty.shape == (0, 96)
