"""The method's degenerate cases on the GPU, through every kernel that runs
the recurrence: decode steps, speculative verify with commit, the chunked
prefill (two-launch tensor-core path for head dim 128, CUDA-core kernel for
64) and the token-by-token prefill, each compared with the float64 oracle's
token-by-token recurrence over the same 130 tokens (two full 64-token chunks
and a ragged tail).

Cases (the oracle is pinned to the closed form of each on the CPU):
  beta0           beta = 0: pure decay of the initial state
  overwrite       g = 0, beta = 1: the state maps each new key to its value
  store_retrieve  zero state, g = 0, beta = 1, orthogonal keys (Hadamard
                  rows) stored, then queried with beta = 0: returns the values
  strong_decay    g = -12 on a whole 64-token chunk (its cumulative decay
                  exp(-768) underflows in float32 and float64 alike)
  zero_qk         all-zero q and k rows (whole tokens and single key heads)

Tolerances: the float32 CUDA-core kernels (decode, the CUDA-core verify and
prefill of head dim 64, token-by-token prefill) keep max|gpu - ref| <=
1e-4 * max|ref|; the tensor-core kernels of head dim 128 (verify, chunked
prefill) multiply tf32 operands (unit roundoff 2^-11) and are held to
5e-3 * max|ref|; bf16 inputs are additionally held to the elementwise
criterion |gpu - ref| <= 1e-2 + 1e-2 |ref|."""
import numpy as np
import pytest
import torch

from gated_deltanet_recurrent_gb300 import abi, synth
from oracle import gdn_oracle as O
from tests.gpu_util import assert_close_bf16, assert_maxrel, dev, dev_i32, host, tok_np

pytestmark = pytest.mark.gpu

T = 130
SLOT = 2
SENTINEL = 3.25
CASES = ("beta0", "overwrite", "store_retrieve", "strong_decay", "zero_qk")
PATHS = ("decode", "verify", "chunked", "recurrent")


def _hadamard(n):
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def _case(name, D, dtype, seed):
    shape = synth.LayerShape(4, 2, D, D, 16, 4)
    rng = np.random.default_rng(seed)
    S0 = synth.random_states(rng, 1, shape)[0]
    tok = {n: a.astype(np.float64) for n, a in synth.token_inputs(rng, T, shape, "f32").items()}
    if name == "beta0":
        tok["beta"][:] = 0.0
    elif name == "overwrite":
        tok["g"][:] = 0.0
        tok["beta"][:] = 1.0
    elif name == "store_retrieve":
        S0[:] = 0.0
        m = min(D, 64)
        H = _hadamard(D)
        for kh in range(shape.h_k):
            rows = rng.permutation(D)[:m]
            tok["k"][:m, kh] = H[rows]                  # orthogonal keys, one per token
            picks = rng.integers(0, m, T - m)           # queries read stored keys
            tok["q"][m:, kh] = H[rows[picks]]
        tok["g"][:] = 0.0
        tok["beta"][:m] = 1.0
        tok["beta"][m:] = 0.0
    elif name == "strong_decay":
        tok["g"][64:128] = -12.0                         # the whole second chunk
    elif name == "zero_qk":
        tok["q"][::5] = 0.0
        tok["k"][::5] = 0.0
        tok["q"][3::7, 1] = 0.0
        tok["k"][3::7, 1] = 0.0
    tok = {n: synth.cast(a, dtype) for n, a in tok.items()}
    return shape, S0, tok


def _run(path, shape, S0, tok, dtype):
    pool = abi.Pool.for_shape(shape, 1, 4, conv_dtype=torch.float32)
    pool.state.fill_(SENTINEL)
    pool.state[0, SLOT] = dev(S0)
    d = {n: dev(a, dtype) for n, a in tok.items()}
    args = lambda lo, hi: [d[n][lo:hi] for n in ("q", "k", "v", "g", "beta")]
    o = torch.empty(T, shape.h_v, shape.dv, device="cuda")
    sid = dev_i32([SLOT])
    if path == "decode":
        for t in range(T):
            abi.gdn_decode_step(pool, 0, sid, *args(t, t + 1), o[t:t + 1])
    elif path == "verify":
        for lo in range(0, T, 8):
            hi = min(lo + 8, T)
            ov = o[lo:hi].view(1, hi - lo, shape.h_v, shape.dv)
            abi.gdn_spec_verify(pool, 0, sid, hi - lo, *args(lo, hi), o=ov,
                                accept_len=dev_i32([hi - lo]))
    elif path == "chunked":
        abi.gdn_prefill_chunked(pool, 0, sid, dev_i32([0, T]), *args(0, T), o)
    else:
        abi.gdn_prefill_recurrent(pool, 0, sid, dev_i32([0, T]), *args(0, T), o)
    S = host(pool.state[0, SLOT])
    pool.state[0, SLOT] = SENTINEL
    assert bool((pool.state == SENTINEL).all()), "another slot changed"
    assert abi.gdn_pool_get_error(pool) == 0
    return host(o), S


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("case", CASES)
def test_degenerate_cases_all_paths_match_oracle(case, D, dtype):
    shape, S0, tok = _case(case, D, dtype, seed=CASES.index(case) * 10 + D)
    S_ref, o_ref = O.gdn_recurrent(S0, *tok_np(tok))
    for path in PATHS:
        o, S = _run(path, shape, S0, tok, dtype)
        tensor_core = D == 128 and path in ("verify", "chunked")
        rel = 5e-3 if tensor_core else 1e-4
        what = f"{case} D={D} {dtype} {path}"
        assert_maxrel(o, o_ref, rel, f"o {what}")
        assert_maxrel(S, S_ref, rel, f"S {what}")
        if dtype == "bf16":
            assert_close_bf16(o, o_ref, what=f"o {what}")
            assert_close_bf16(S, S_ref, what=f"S {what}")
        if case == "store_retrieve":
            # queried with beta = 0 and a stored key: o_t is that key's value
            m = min(D, 64)
            keys = tok["k"][:m]
            for t in range(m, T, 17):
                for h in range(shape.h_v):
                    kh = h // (shape.h_v // shape.h_k)
                    j = int(np.nonzero((keys[:, kh] == tok["q"][t, kh]).all(axis=1))[0][0])
                    assert np.max(np.abs(o[t, h] - tok["v"][j, h])) <= \
                        rel * np.max(np.abs(tok["v"])) + 1e-6, f"retrieval {what} t={t}"
