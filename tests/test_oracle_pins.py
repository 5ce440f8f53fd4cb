"""Pins for the CPU oracle: each test checks it against something other than
itself -- a hand-worked example, exact rational brute force, a closed form, a
library routine, or an invariant the pages state -- so that a dropped term, a
wrong sign or index, or a transposed operand fails at least one of them.

Map (oracle function -> pins):
  conv_silu       golden hand example; torch conv1d (float64, groups=C);
                  split invariance; advance == feeding fewer tokens; short seq
  l2_normalize    closed form
  gdn_step /
  gdn_recurrent   golden 2x2 hand example; Fraction brute force of the unrolled
                  product (with a 2-to-1 head grouping); beta = 0 pure decay;
                  beta = 1 overwrite; orthonormal store/retrieve; linearity;
                  q-scale invariance; scale multiplier; contiguous grouping;
                  planted mistakes are caught by the brute force
  gdn_chunked     equals token by token for several chunk sizes; golden example
  spec_verify     equals decode steps; commit at a == a steps; a = 0 unchanged
  spec_verify_deferred  rounds equal the two-phase rounds; the state after
                  the flush equals decoding only the accepted drafts
  prefill_checkpointed  each checkpoint equals the recurrence over the
                  prefix it closes; outputs and final state equal prefill
  OraclePool      N slots == each alone; reset == fresh; prefill split
                  invariance across pieces (chunked-prefill state carry)
  gated_rmsnorm   rows of unit root mean square reduce to o * w * silu(z)
                  with silu from scipy's expit; scale invariance (eps = 0);
                  unit mean square of out / (w silu(z)); z = 0 gives 0; a
                  zero row with eps > 0 gives 0; planted mistakes are caught
  in_proj         brute-force sums over small integers; one-hot rows pick
                  columns of w (catches a transposed weight)
  round_bf16 /
  round_f16       torch's float32 -> bfloat16 and numpy's float64 -> float16
                  conversions (library routines) on values spanning the
                  subnormal, normal and overflow ranges; hand-worked ties
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import gdn_oracle as O
from gated_deltanet_recurrent_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, vals = line.split(":", 1)
            out[key.strip()] = np.array([float(t) for t in vals.split()])
    return out


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# ------------------------------------------------------------------ conv

def test_golden_conv_silu():
    f = _read_fixture("conv_silu_w4.txt")
    w = f["w"].reshape(1, 4)
    cache = f["cache"].reshape(1, 3)
    x = f["x"].reshape(2, 1)
    y, c = O.conv_silu(x, cache, w)
    np.testing.assert_allclose(y[:, 0], f["y"], rtol=1e-14)
    np.testing.assert_array_equal(c[0], f["cache_after"])
    y1, c1 = O.conv_silu(x, cache, w, advance=1)
    np.testing.assert_array_equal(y1, y)
    np.testing.assert_array_equal(c1[0], f["cache_after_advance1"])


@pytest.mark.parametrize("with_bias", [False, True])
def test_conv_matches_torch_conv1d(with_bias):
    rng = np.random.default_rng(11)
    C, W, L = 64, 4, 13
    x = rng.standard_normal((L, C))
    cache = rng.standard_normal((C, W - 1))
    w = 0.25 * rng.standard_normal((C, W))
    b = rng.standard_normal(C) if with_bias else None
    y, c = O.conv_silu(x, cache, w, b)
    inp = torch.from_numpy(np.concatenate([cache, x.T], axis=1))[None]  # [1, C, W-1+L]
    ref = torch.nn.functional.conv1d(
        inp, torch.from_numpy(w)[:, None, :],
        None if b is None else torch.from_numpy(b), groups=C)
    ref = torch.nn.functional.silu(ref)[0].T.numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(c, x[-(W - 1):].T)


def test_conv_split_invariance():
    rng = np.random.default_rng(12)
    C, W, L = 32, 4, 13
    x = rng.standard_normal((L, C))
    cache = rng.standard_normal((C, W - 1))
    w = rng.standard_normal((C, W))
    y, c = O.conv_silu(x, cache, w)
    ys, cc = [], cache
    for lo, hi in [(0, 3), (3, 4), (4, 9), (9, 13)]:
        yy, cc = O.conv_silu(x[lo:hi], cc, w)
        ys.append(yy)
    np.testing.assert_array_equal(np.concatenate(ys), y)
    np.testing.assert_array_equal(cc, c)


def test_conv_advance_equals_fewer_tokens():
    rng = np.random.default_rng(13)
    C, W, L = 16, 4, 5
    x = rng.standard_normal((L, C))
    cache = rng.standard_normal((C, W - 1))
    w = rng.standard_normal((C, W))
    for a in range(L + 1):
        _, c_adv = O.conv_silu(x, cache, w, advance=a)
        _, c_ref = O.conv_silu(x[:a], cache, w) if a else (None, cache)
        np.testing.assert_array_equal(c_adv, c_ref)


def test_conv_short_sequence_shifts_partially():
    cache = np.array([[1.0, 2.0, 3.0]])
    w = np.array([[0.0, 0.0, 0.0, 1.0]])
    _, c = O.conv_silu(np.array([[7.0]]), cache, w)
    np.testing.assert_array_equal(c, [[2.0, 3.0, 7.0]])


# ------------------------------------------------------------- l2 norm

def test_l2_normalize_closed_form():
    np.testing.assert_allclose(O.l2_normalize([3.0, 4.0], eps=0.0), [0.6, 0.8], rtol=1e-15)
    np.testing.assert_allclose(O.l2_normalize([3.0, 4.0]),
                               [0.5999999880000003, 0.7999999840000004], rtol=1e-14)


# --------------------------------------------------------- delta rule

def test_golden_delta_rule_2x2():
    f = _read_fixture("delta_rule_2x2.txt")
    k = f["k"].reshape(2, 1, 2)
    q = f["q"].reshape(2, 1, 2)
    v = f["v"].reshape(2, 1, 2)
    g = np.log(f["alpha"]).reshape(2, 1)
    beta = f["beta"].reshape(2, 1)
    S0 = np.zeros((1, 2, 2))
    S1, o1 = O.gdn_step(S0, q[0], k[0], v[0], g[0], beta[0], eps=0.0)
    np.testing.assert_allclose(S1.ravel(), f["S1"], atol=1e-15)
    np.testing.assert_allclose(o1.ravel(), f["o1"], atol=1e-15)
    S2, o = O.gdn_recurrent(S0, q, k, v, g, beta, eps=0.0)
    np.testing.assert_allclose(S2.ravel(), f["S2"], atol=1e-14)
    np.testing.assert_allclose(o[1].ravel(), f["o2"], atol=1e-14)
    for chunk in (1, 2):
        Sc, oc = O.gdn_chunked(S0, q, k, v, g, beta, chunk=chunk, eps=0.0)
        np.testing.assert_allclose(Sc.ravel(), f["S2"], atol=1e-14)
        np.testing.assert_allclose(oc[1].ravel(), f["o2"], atol=1e-14)


# Rational unit vectors in R^3 (Pythagorean quadruples) so that the key
# normalisation is exact and the whole recurrence stays in the rationals.
_UNIT3 = [(1, 2, 2, 3), (2, 1, -2, 3), (2, 3, 6, 7), (-6, 2, 3, 7), (2, -6, 9, 11),
          (1, 4, 8, 9), (4, -4, 7, 9), (0, 3, 4, 5)]


def _exact_reference(S0, ks, qs, vs, alphas, betas, group):
    """S_T = S0 prod_t A_t + sum_t beta_t v_t k_t^T prod_{s>t} A_s with
    A_t = alpha_t (I - beta_t k_t k_t^T), in exact Fractions, per value head;
    o_t = S_t q_t.  Value head h reads key head h // group."""
    def matmul(X, Y):
        return [[sum(X[i][r] * Y[r][j] for r in range(len(Y))) for j in range(len(Y[0]))]
                for i in range(len(X))]

    h_v = len(S0)
    T = len(ks)
    dim = len(S0[0][0])
    outs = [[None] * h_v for _ in range(T)]
    finals = []
    for h in range(h_v):
        hk = h // group
        for t_end in range(1, T + 1):
            A = []
            for t in range(t_end):
                kv = ks[t][hk]
                A.append([[alphas[t][h] * ((1 if i == j else 0) - betas[t][h] * kv[i] * kv[j])
                           for j in range(dim)] for i in range(dim)])
            St = [row[:] for row in S0[h]]
            for t in range(t_end):
                St = matmul(St, A[t])
            for t in range(t_end):
                term = [[betas[t][h] * vs[t][h][i] * ks[t][hk][j] for j in range(dim)]
                        for i in range(len(vs[t][h]))]
                for s in range(t + 1, t_end):
                    term = matmul(term, A[s])
                St = [[St[i][j] + term[i][j] for j in range(dim)] for i in range(len(St))]
            qv = qs[t_end - 1][hk]
            outs[t_end - 1][h] = [sum(St[i][j] * qv[j] for j in range(dim)) for i in range(len(St))]
            if t_end == T:
                finals.append(St)
    return finals, outs


def _rational_problem(seed, T=4, h_v=2, h_k=1):
    rng = np.random.default_rng(seed)
    dim = 3
    pick = lambda: _UNIT3[int(rng.integers(len(_UNIT3)))]
    unit = lambda u: [Fraction(u[i], u[3]) for i in range(3)]
    ks = [[unit(pick()) for _ in range(h_k)] for _ in range(T)]
    qs = [[unit(pick()) for _ in range(h_k)] for _ in range(T)]
    vs = [[[Fraction(int(rng.integers(-8, 9)), 4) for _ in range(dim)] for _ in range(h_v)]
          for _ in range(T)]
    alphas = [[Fraction(int(rng.integers(1, 8)), 8) for _ in range(h_v)] for _ in range(T)]
    betas = [[Fraction(int(rng.integers(0, 5)), 4) for _ in range(h_v)] for _ in range(T)]
    S0 = [[[Fraction(int(rng.integers(-4, 5)), 8) for _ in range(dim)] for _ in range(dim)]
          for _ in range(h_v)]
    return S0, ks, qs, vs, alphas, betas


def _as_arrays(S0, ks, qs, vs, alphas, betas):
    f = lambda x: np.array(x, dtype=object).astype(np.float64)
    return (f(S0), f(qs), f(ks), f(vs), np.log(f(alphas)), f(betas))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_exact_rational_bruteforce(seed):
    prob = _rational_problem(seed)
    S_ref, o_ref = _exact_reference(*prob, group=2)
    S0, q, k, v, g, beta = _as_arrays(*prob)
    S_T, o = O.gdn_recurrent(S0, q, k, v, g, beta, eps=0.0)
    np.testing.assert_allclose(S_T, np.array(S_ref, dtype=np.float64), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o, np.array(o_ref, dtype=np.float64), rtol=0, atol=1e-12)
    S_c, o_c = O.gdn_chunked(S0, q, k, v, g, beta, chunk=3, eps=0.0)
    np.testing.assert_allclose(S_c, np.array(S_ref, dtype=np.float64), rtol=0, atol=1e-12)
    np.testing.assert_allclose(o_c, np.array(o_ref, dtype=np.float64), rtol=0, atol=1e-12)


def _planted_step(kind):
    """Plausible mistakes, planted in a copy of the oracle's step."""
    def step(S, q, k, v, g, beta, scale=1.0, eps=O.L2_EPS):
        h_v = S.shape[0]
        h_k = q.shape[0]
        if kind == "interleaved_heads":
            kh = np.tile(O.l2_normalize(k, eps), (h_v // h_k, 1))
            qh = np.tile(O.l2_normalize(q, eps), (h_v // h_k, 1))
        else:
            kh = O.expand_key_heads(O.l2_normalize(k, eps), h_v)
            qh = O.expand_key_heads(O.l2_normalize(q, eps), h_v)
        alpha = np.exp(g)[:, None, None]
        b = beta[:, None, None]
        Sk = np.einsum("hvk,hk->hv", S, kh)
        sign = 1.0 if kind == "wrong_sign" else -1.0
        decay_inside = alpha if kind != "alpha_on_input" else 1.0
        S_new = decay_inside * (S + sign * b * Sk[:, :, None] * kh[:, None, :]) \
            + b * v[:, :, None] * kh[:, None, :]
        if kind == "alpha_on_input":
            S_new = alpha * S_new
        if kind == "transposed_state":
            S_new = np.swapaxes(S_new, 1, 2)
        S_read = S if kind == "read_before_update" else S_new
        o = scale * np.einsum("hvk,hk->hv", S_read, qh)
        return S_new, o
    return step


@pytest.mark.parametrize("kind", ["wrong_sign", "alpha_on_input", "transposed_state",
                                  "read_before_update", "interleaved_heads"])
def test_bruteforce_catches_planted_mistakes(kind, monkeypatch):
    # Interleaved vs contiguous head grouping only differs with >1 key head.
    h_v, h_k, group = (4, 2, 2) if kind == "interleaved_heads" else (2, 1, 2)
    prob = _rational_problem(5, h_v=h_v, h_k=h_k)
    S_ref, o_ref = _exact_reference(*prob, group=group)
    S0, q, k, v, g, beta = _as_arrays(*prob)
    monkeypatch.setattr(O, "gdn_step", _planted_step(kind))
    S_T, o = O.gdn_recurrent(S0, q, k, v, g, beta, eps=0.0)
    err = max(np.max(np.abs(S_T - np.array(S_ref, dtype=np.float64))),
              np.max(np.abs(o - np.array(o_ref, dtype=np.float64))))
    assert err > 1e-6, f"planted mistake {kind} went unnoticed"


def _random_problem(seed, T=20, h_v=4, h_k=2, K=8, V=6, beta_val=None, g_val=None):
    rng = np.random.default_rng(seed)
    S0 = 0.3 * rng.standard_normal((h_v, V, K))
    q = rng.standard_normal((T, h_k, K))
    k = rng.standard_normal((T, h_k, K))
    v = rng.standard_normal((T, h_v, V))
    g = -np.logaddexp(0, rng.standard_normal((T, h_v))) if g_val is None else np.full((T, h_v), g_val)
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, h_v)))) if beta_val is None \
        else np.full((T, h_v), beta_val)
    return S0, q, k, v, g, beta


def test_beta_zero_is_pure_decay():
    S0, q, k, v, g, beta = _random_problem(21, beta_val=0.0)
    S_T, o = O.gdn_recurrent(S0, q, k, v, g, beta, scale=0.7)
    G = np.cumsum(g, axis=0)                                # [T, H_v]
    np.testing.assert_allclose(S_T, np.exp(G[-1])[:, None, None] * S0, rtol=1e-12)
    qn = q / np.sqrt(np.sum(q * q, axis=-1, keepdims=True) + O.L2_EPS)
    for t in range(len(q)):
        for h in range(S0.shape[0]):
            ref = 0.7 * np.exp(G[t, h]) * S0[h] @ qn[t, h // 2]
            np.testing.assert_allclose(o[t, h], ref, rtol=1e-12, atol=1e-14)


def test_beta_one_overwrites_key_direction():
    S0, q, k, v, g, beta = _random_problem(22, beta_val=1.0)
    S = S0
    for t in range(len(q)):
        S, _ = O.gdn_step(S, q[t], k[t], v[t], g[t], beta[t], eps=0.0)
        kn = k[t] / np.linalg.norm(k[t], axis=-1, keepdims=True)
        for h in range(S.shape[0]):
            np.testing.assert_allclose(S[h] @ kn[h // 2], v[t, h], rtol=1e-12, atol=1e-12)


def test_orthonormal_keys_store_and_retrieve():
    rng = np.random.default_rng(23)
    K = V = 16
    m = 10
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    keys = Qm[:, :m].T                                      # m orthonormal rows
    vals = rng.standard_normal((m, 1, V))
    S = np.zeros((1, V, K))
    for t in range(m):
        S, _ = O.gdn_step(S, keys[t][None], keys[t][None], vals[t], np.zeros(1),
                          np.ones(1), eps=0.0)
    for j in range(m):
        o = 1.0 * S[0] @ keys[j]
        np.testing.assert_allclose(o, vals[j, 0], atol=1e-12)
        # and through the oracle's own read-out path (g = 0, beta = 0: no change)
        _, oj = O.gdn_step(S, keys[j][None], keys[j][None], np.zeros((1, V)),
                           np.zeros(1), np.zeros(1), eps=0.0)
        np.testing.assert_allclose(oj[0], vals[j, 0], atol=1e-12)


def test_linearity_in_state_and_values():
    S0, q, k, v, g, beta = _random_problem(24)
    S1, o1 = O.gdn_recurrent(S0, q, k, v, g, beta)
    S2, o2 = O.gdn_recurrent(3.5 * S0, q, k, 3.5 * v, g, beta)
    np.testing.assert_allclose(S2, 3.5 * S1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(o2, 3.5 * o1, rtol=1e-12, atol=1e-13)


def test_query_scale_invariance_and_scale_multiplier():
    S0, q, k, v, g, beta = _random_problem(25)
    S1, o1 = O.gdn_recurrent(S0, q, k, v, g, beta, eps=0.0)
    S2, o2 = O.gdn_recurrent(S0, 4.0 * q, k, v, g, beta, eps=0.0)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    S3, o3 = O.gdn_recurrent(S0, q, k, v, g, beta, scale=8 ** -0.5, eps=0.0)
    np.testing.assert_array_equal(S3, S1)
    np.testing.assert_allclose(o3, 8 ** -0.5 * o1, rtol=1e-13)


def test_head_grouping_is_contiguous():
    S0, q, k, v, g, beta = _random_problem(26, h_v=4, h_k=2)
    S_T, o = O.gdn_recurrent(S0, q, k, v, g, beta)
    for h in range(4):
        hk = h // 2
        Sh, oh = O.gdn_recurrent(S0[h:h + 1], q[:, hk:hk + 1], k[:, hk:hk + 1],
                                 v[:, h:h + 1], g[:, h:h + 1], beta[:, h:h + 1])
        np.testing.assert_allclose(S_T[h], Sh[0], rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(o[:, h], oh[:, 0], rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("chunk", [1, 3, 4, 64])
def test_chunked_equals_token_by_token(chunk):
    S0, q, k, v, g, beta = _random_problem(27, T=150, K=16, V=12)
    S_r, o_r = O.gdn_recurrent(S0, q, k, v, g, beta, scale=0.5)
    S_c, o_c = O.gdn_chunked(S0, q, k, v, g, beta, scale=0.5, chunk=chunk)
    assert _rel(S_c, S_r) < 1e-10
    assert _rel(o_c, o_r) < 1e-10


def test_chunked_strong_decay_long_chunk():
    # Large |g| over a 64-token chunk: exp(G_t - G_i) for i > t would overflow
    # if it were not masked before exponentiation.
    S0, q, k, v, g, beta = _random_problem(28, T=64, g_val=-12.0)
    S_r, o_r = O.gdn_recurrent(S0, q, k, v, g, beta)
    S_c, o_c = O.gdn_chunked(S0, q, k, v, g, beta, chunk=64)
    assert np.all(np.isfinite(o_c))
    np.testing.assert_allclose(o_c, o_r, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(S_c, S_r, rtol=1e-9, atol=1e-300)


# ------------------------------------------------------------ verify

def test_spec_verify_identities():
    S0, q, k, v, g, beta = _random_problem(29, T=6)
    T = len(q)
    S = S0.copy()
    steps = [S.copy()]
    outs = []
    for t in range(T):
        S, o = O.gdn_step(S, q[t], k[t], v[t], g[t], beta[t])
        steps.append(S.copy())
        outs.append(o)
    for a in range(T + 1):
        o_v, S_keep = O.spec_verify(S0, q, k, v, g, beta, accept_len=a)
        np.testing.assert_array_equal(o_v, np.stack(outs))
        np.testing.assert_array_equal(S_keep, steps[a])
    o_v, S_keep = O.spec_verify(S0, q, k, v, g, beta)
    np.testing.assert_array_equal(S_keep, S0)


# -------------------------------------------------------------- pool

def _tiny_pool():
    s = synth.TINY_LAYER
    return O.OraclePool(1, 4, s.h_v, s.h_k, s.dk, s.dv, s.conv_ch, s.conv_k)


def _run_tiny_request(pool, wl, i, slot):
    """Prefill sequence i into `slot` in 4-token pieces, then decode 5 tokens."""
    seq = wl["seqs"][i]
    L = wl["lengths"][i]
    tok, x = seq["tok"], seq["x"]
    ys, os_ = [], []
    for lo in range(0, L, wl["piece"]):
        hi = min(lo + wl["piece"], L)
        ys.append(pool.conv_silu(0, [slot], [0, hi - lo], x[lo:hi], wl["conv_w"]))
        os_.append(pool.prefill(0, [slot], [0, hi - lo], *(tok[n][lo:hi] for n in
                   ("q", "k", "v", "g", "beta"))))
    for t in range(L, L + wl["n_decode"]):
        ys.append(pool.conv_silu(0, [slot], None, x[t:t + 1], wl["conv_w"]))
        os_.append(pool.decode_step(0, [slot], *(tok[n][t:t + 1] for n in
                   ("q", "k", "v", "g", "beta"))))
    return np.concatenate(ys), np.concatenate(os_)


def test_pool_slots_independent_and_reset_equals_fresh():
    wl = synth.tiny_workload(0)
    # each request alone in its own fresh pool
    alone = []
    for i, slot in enumerate(wl["slots"]):
        alone.append(_run_tiny_request(_tiny_pool(), wl, i, slot))
    # both requests in one pool, interleaved; sentinel in the untouched slots
    pool = _tiny_pool()
    pool.S[:, [0, 2]] = 123.0
    pool.X[:, [0, 2]] = -7.0
    res = [_run_tiny_request(pool, wl, i, slot) for i, slot in enumerate(wl["slots"])]
    for (ya, oa), (yb, ob) in zip(alone, res):
        np.testing.assert_array_equal(ya, yb)
        np.testing.assert_array_equal(oa, ob)
    assert np.all(pool.S[:, [0, 2]] == 123.0) and np.all(pool.X[:, [0, 2]] == -7.0)
    # reset slot 1 and rerun its request: bit-identical to the first run
    S3 = pool.S[:, 3].copy()
    pool.reset([1])
    again = _run_tiny_request(pool, wl, 0, 1)
    np.testing.assert_array_equal(again[0], res[0][0])
    np.testing.assert_array_equal(again[1], res[0][1])
    np.testing.assert_array_equal(pool.S[:, 3], S3)


def test_pool_batched_varlen_equals_each_alone():
    rng = np.random.default_rng(31)
    shape = synth.LayerShape(4, 2, 8, 8, 16, 4)
    lengths = [5, 0, 9, 3]
    cu = synth.cu_seqlens_of(lengths)
    slots = [2, 0, 5, 3]
    tok = synth.token_inputs(rng, int(cu[-1]), shape)
    args = [tok[n] for n in ("q", "k", "v", "g", "beta")]
    mk = lambda: O.OraclePool(1, 6, shape.h_v, shape.h_k, shape.dk, shape.dv,
                              shape.conv_ch, shape.conv_k)
    pool = mk()
    init = rng.standard_normal(pool.S.shape)
    pool.S[:] = init
    o = pool.prefill(0, slots, cu, *args)
    for i, s in enumerate(slots):
        p1 = mk()
        p1.S[:] = init
        lo, hi = cu[i], cu[i + 1]
        oi = p1.prefill(0, [s], [0, hi - lo], *(a[lo:hi] for a in args))
        np.testing.assert_array_equal(o[lo:hi], oi)
        np.testing.assert_array_equal(pool.S[0, s], p1.S[0, s])


def test_pool_prefill_split_invariance_across_calls():
    rng = np.random.default_rng(32)
    shape = synth.LayerShape(2, 1, 8, 8, 16, 4)
    L = 37
    tok = synth.token_inputs(rng, L, shape)
    args = [tok[n] for n in ("q", "k", "v", "g", "beta")]
    mk = lambda: O.OraclePool(1, 1, shape.h_v, shape.h_k, shape.dk, shape.dv,
                              shape.conv_ch, shape.conv_k)
    whole = mk()
    o_whole = whole.prefill(0, [0], [0, L], *args, chunk=8)
    for cuts in ([0, 8, 16, 37], [0, 5, 6, 30, 37], [0, 1, 37]):
        p = mk()
        outs = []
        for lo, hi in zip(cuts[:-1], cuts[1:]):
            outs.append(p.prefill(0, [0], [0, hi - lo], *(a[lo:hi] for a in args), chunk=8))
        assert _rel(np.concatenate(outs), o_whole) < 1e-11
        assert _rel(p.S, whole.S) < 1e-11


def test_pool_spec_verify_commit_then_decode():
    rng = np.random.default_rng(33)
    shape = synth.LayerShape(2, 1, 8, 8, 16, 4)
    T, n = 3, 3
    draft = synth.token_inputs(rng, n * T, shape)
    args = [draft[nm] for nm in ("q", "k", "v", "g", "beta")]
    mk = lambda: O.OraclePool(1, 4, shape.h_v, shape.h_k, shape.dk, shape.dv,
                              shape.conv_ch, shape.conv_k)
    slots = [3, 0, 2]
    accept = [2, 0, 3]
    p = mk()
    p.S[:] = rng.standard_normal(p.S.shape)
    before = p.S.copy()
    o_read = p.spec_verify(0, slots, T, *args)            # verify only
    np.testing.assert_array_equal(p.S, before)
    o_commit = p.spec_verify(0, slots, T, *args, accept_len=accept)
    np.testing.assert_array_equal(o_read, o_commit)
    for i, s in enumerate(slots):
        ref = mk()
        ref.S[:] = before
        for t in range(accept[i]):
            j = i * T + t
            ref.decode_step(0, [s], *(a[j:j + 1] for a in args))
        np.testing.assert_array_equal(p.S[0, s], ref.S[0, s])
    np.testing.assert_array_equal(p.S[0, 1], before[0, 1])


def test_pool_deferred_rounds_equal_two_phase_rounds():
    """Three speculative rounds with pending commits folded into the next
    round give the outputs of verify-then-commit rounds, and after a final
    flush the states equal decoding only the accepted drafts one by one."""
    rng = np.random.default_rng(34)
    shape = synth.LayerShape(2, 1, 8, 8, 16, 4)
    n, slots = 3, [1, 3, 0]
    Ts = [3, 2, 4]
    accepts = [[2, 0, 3], [1, 2, 0], [4, 1, 2]]
    mk = lambda: O.OraclePool(1, 4, shape.h_v, shape.h_k, shape.dk, shape.dv,
                              shape.conv_ch, shape.conv_k)
    S0 = rng.standard_normal((1, 4, shape.h_v, shape.dv, shape.dk))
    rounds = []
    for T in Ts:
        d = synth.token_inputs(rng, n * T, shape)
        rounds.append([d[nm] for nm in ("q", "k", "v", "g", "beta")])
    two, dfr, dec = mk(), mk(), mk()
    for p in (two, dfr, dec):
        p.S[:] = S0
    prev, T_prev, prev_acc = None, 0, None
    for T, args, acc in zip(Ts, rounds, accepts):
        o_two = two.spec_verify(0, slots, T, *args)
        two.spec_verify(0, slots, T, *args, accept_len=acc)
        o_dfr = dfr.spec_verify_deferred(0, slots, T, *args, T_prev=T_prev, prev=prev,
                                         prev_accept=prev_acc)
        np.testing.assert_allclose(o_dfr, o_two, rtol=1e-12, atol=1e-12)
        for i, s in enumerate(slots):
            for t in range(acc[i]):
                j = i * T + t
                dec.decode_step(0, [s], *(a[j:j + 1] for a in args))
        prev, T_prev, prev_acc = args, T, acc
    # pending drafts are still outstanding: the deferred pool lags until flushed
    assert not np.allclose(dfr.S, two.S)
    dfr.spec_verify(0, slots, T_prev, *prev, accept_len=prev_acc)
    np.testing.assert_allclose(dfr.S, two.S, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dfr.S, dec.S, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(dfr.S[0, 2], S0[0, 2])


def test_pool_prefill_checkpoints_are_prefix_states():
    rng = np.random.default_rng(35)
    shape = synth.LayerShape(2, 1, 8, 8, 16, 4)
    lens = [13, 4, 9]
    cu = synth.cu_seqlens_of(lens)
    tok = synth.token_inputs(rng, int(cu[-1]), shape)
    args = [tok[nm] for nm in ("q", "k", "v", "g", "beta")]
    mk = lambda: O.OraclePool(1, 12, shape.h_v, shape.h_k, shape.dk, shape.dv,
                              shape.conv_ch, shape.conv_k)
    S0 = rng.standard_normal((1, 12, shape.h_v, shape.dv, shape.dk))
    slots = [0, 1, 2]
    ck = [[5, -1, 6], [7, 8, 9], [10, 11, -1]]
    a, b = mk(), mk()
    a.S[:] = S0
    b.S[:] = S0
    o_a = a.prefill_checkpointed(0, slots, cu, *args, ckpt_slots=ck, ckpt_every=4)
    o_b = b.prefill(0, slots, cu, *args)
    np.testing.assert_allclose(o_a, o_b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(a.S[0, slots], b.S[0, slots], rtol=1e-12, atol=1e-12)
    for i, s in enumerate(slots):
        lo = cu[i]
        for j, d in enumerate(ck[i]):
            n = 4 * (j + 1)
            if d < 0:
                continue
            if n > lens[i]:
                np.testing.assert_array_equal(a.S[0, d], S0[0, d])   # never reached
                continue
            S_ref, _ = O.gdn_recurrent(S0[0, s], *(x[lo:lo + n] for x in args))
            np.testing.assert_allclose(a.S[0, d], S_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(a.S[0, [3, 4]], S0[0, [3, 4]])



# ----------------------------------------------------------- gated RMSNorm

def test_gated_rmsnorm_reduces_to_the_gate_on_unit_rms_rows():
    """Rows of +-1 have root mean square 1, so with eps = 0 the norm is the
    identity and the result is o * w * z * expit(z) (scipy's logistic)."""
    from scipy.special import expit
    rng = np.random.default_rng(90)
    o = rng.choice([-1.0, 1.0], size=(5, 3, 24))
    z = rng.standard_normal((5, 3, 24)) * 3
    w = rng.standard_normal(24)
    np.testing.assert_allclose(O.gated_rmsnorm(o, z, w, eps=0.0), o * w * z * expit(z),
                               rtol=1e-13, atol=1e-15)


def test_gated_rmsnorm_invariants():
    rng = np.random.default_rng(91)
    o = rng.standard_normal((7, 40))
    z = rng.standard_normal((7, 40))
    w = rng.uniform(0.5, 2.0, 40)
    out = O.gated_rmsnorm(o, z, w, eps=0.0)
    # scale invariance of the norm
    np.testing.assert_allclose(O.gated_rmsnorm(4.25 * o, z, w, eps=0.0), out, rtol=1e-13)
    # divided by the weight and the gate, every row has mean square exactly 1
    from scipy.special import expit
    normed = out / (w * z * expit(z))
    np.testing.assert_allclose(np.mean(normed ** 2, axis=-1), 1.0, rtol=1e-12)
    # a closed gate (z = 0) gives zero; a zero row with eps > 0 gives zero
    assert np.all(O.gated_rmsnorm(o, np.zeros_like(z), w) == 0.0)
    assert np.all(O.gated_rmsnorm(np.zeros_like(o), z, w, eps=1e-6) == 0.0)


def test_gated_rmsnorm_pins_catch_planted_mistakes():
    """A sum instead of a mean, a sigmoid gate, or a dropped weight each break
    one of the pins above."""
    from scipy.special import expit
    rng = np.random.default_rng(92)
    o = rng.choice([-1.0, 1.0], size=(3, 16))
    z = rng.standard_normal((3, 16))
    w = rng.uniform(0.5, 2.0, 16)
    want = o * w * z * expit(z)

    def sum_not_mean(o, z, w, eps=1e-6):
        o, z = np.asarray(o, float), np.asarray(z, float)
        return o / np.sqrt(np.sum(o * o, -1, keepdims=True) + eps) * w * O.silu(z)

    def sigmoid_gate(o, z, w, eps=1e-6):
        o, z = np.asarray(o, float), np.asarray(z, float)
        return o / np.sqrt(np.mean(o * o, -1, keepdims=True) + eps) * w * expit(z)

    def no_weight(o, z, w, eps=1e-6):
        o, z = np.asarray(o, float), np.asarray(z, float)
        return o / np.sqrt(np.mean(o * o, -1, keepdims=True) + eps) * O.silu(z)

    for wrong in (sum_not_mean, sigmoid_gate, no_weight):
        assert not np.allclose(wrong(o, z, w, eps=0.0), want, rtol=1e-6), wrong.__name__


# ------------------------------------------------------- storage formats

def test_round_bf16_matches_torch_conversion():
    """torch converts float32 to bfloat16 with round-to-nearest-even; on
    float32 inputs (one rounding, no double rounding) it is the definition."""
    rng = np.random.default_rng(90)
    x = rng.standard_normal(100000) * np.exp2(rng.integers(-140, 129, 100000))
    x = x.astype(np.float32)
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(O.round_bf16(x.astype(np.float64)), ref)


def test_round_f16_matches_numpy_conversion():
    rng = np.random.default_rng(91)
    x = rng.standard_normal(100000) * np.exp2(rng.integers(-30, 18, 100000))
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(O.round_f16(x), ref)


def test_round_bf16_hand_worked_ties_and_range():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: the even significand is 1.
    # 1 + 3 2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: even is 1 + 2^-6.
    # 2^-134 is half the smallest subnormal (2^-133): ties to 0.
    # 1.5 2^-133 is halfway between 2^-133 and 2^-132: even is 2^-132.
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2.0 ** -134,
                  1.5 * 2.0 ** -133, 3.4e38])
    want = np.array([1.0, 1 + 2.0 ** -6, -1.0, 0.0, 2.0 ** -132, np.inf])
    np.testing.assert_array_equal(O.round_bf16(x), want)
    # the largest finite bf16 is (2 - 2^-7) 2^127 and stays put
    top = (2 - 2.0 ** -7) * 2.0 ** 127
    assert O.round_bf16(np.array([top]))[0] == top


# -------------------------------------------- half-precision state storage

@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_half_state_pool_stores_representable_states_within_half_an_ulp(fmt):
    """A pool with half-precision state storage keeps every stored state
    exactly representable in the format, and each store is the exact result
    rounded to nearest: within half a unit in the last place (2^-8 relative
    for bf16's 8 significant bits, 2^-11 for binary16's 11; subnormal f16
    values within half of 2^-24)."""
    rnd, p = (O.round_bf16, 8) if fmt == "bf16" else (O.round_f16, 11)
    rng = np.random.default_rng(92)
    shape = synth.LayerShape(2, 1, 8, 8, 4, 4)
    pool = O.OraclePool(1, 3, shape.h_v, shape.h_k, shape.dk, shape.dv, 4, 4, state_round=rnd)
    pool.S[0, 1] = rnd(synth.random_states(rng, 1, shape)[0])
    for step in range(4):
        tok = synth.token_inputs(rng, 1, shape, "f32")
        S_before = pool.S[0, 1].copy()
        pool.decode_step(0, [1], *tok_np_(tok))
        exact, _ = O.gdn_step(S_before, *(tok[n][0] for n in ("q", "k", "v", "g", "beta")))
        np.testing.assert_array_equal(rnd(pool.S[0, 1]), pool.S[0, 1])
        err = np.abs(pool.S[0, 1] - exact)
        tiny = 2.0 ** -25 if fmt == "f16" else 0.0
        assert np.all(err <= 2.0 ** -p * np.abs(exact) + tiny)
        assert np.any(err > 0), "the state was not rounded"


def tok_np_(tok):
    return [tok[n] for n in ("q", "k", "v", "g", "beta")]


def test_half_state_rounds_at_call_boundaries_not_per_token():
    """Within a call the state is carried unrounded: a prefill call of L
    tokens equals the exact recurrence over them followed by ONE rounding,
    whereas L decode calls round after every token.  With beta = 0 and g = 0
    (alpha = 1) a stored state passes through any call bit for bit."""
    rng = np.random.default_rng(93)
    shape = synth.LayerShape(2, 2, 8, 8, 4, 4)
    S0 = O.round_bf16(synth.random_states(rng, 1, shape)[0])
    tok = synth.token_inputs(rng, 12, shape, "f32")
    a = O.OraclePool(1, 2, 2, 2, 8, 8, 4, 4, state_round=O.round_bf16)
    b = O.OraclePool(1, 2, 2, 2, 8, 8, 4, 4, state_round=O.round_bf16)
    a.S[0, 0] = S0
    b.S[0, 0] = S0
    a.prefill(0, [0], [0, 12], *tok_np_(tok))
    for t in range(12):
        b.decode_step(0, [0], *(x[t:t + 1] for x in tok_np_(tok)))
    exact, _ = O.gdn_recurrent(S0, *tok_np_(tok))
    np.testing.assert_array_equal(a.S[0, 0], O.round_bf16(exact))
    assert not np.array_equal(a.S[0, 0], b.S[0, 0]), "per-token rounding must differ"
    assert np.max(np.abs(a.S[0, 0] - b.S[0, 0])) <= 2.0 ** -6 * np.max(np.abs(exact))
    still = {n: x.copy() for n, x in tok.items()}
    still["beta"][:] = 0.0
    still["g"][:] = 0.0
    a.prefill(0, [0], [0, 12], *tok_np_(still))
    np.testing.assert_array_equal(a.S[0, 0], O.round_bf16(exact))


# ------------------------------------------------------- input projection

def test_in_proj_brute_force_and_orientation():
    rng = np.random.default_rng(94)
    x = rng.integers(-3, 4, (5, 7)).astype(float)
    w = rng.integers(-3, 4, (6, 7)).astype(float)
    want = np.array([[sum(x[t, h] * w[n, h] for h in range(7)) for n in range(6)]
                     for t in range(5)])
    np.testing.assert_array_equal(O.in_proj(x, w), want)
    # a one-hot hidden state selects one input column of every weight row
    e = np.zeros((1, 7))
    e[0, 2] = 1.0
    np.testing.assert_array_equal(O.in_proj(e, w)[0], w[:, 2])
