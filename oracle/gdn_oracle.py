"""CPU oracle of the slot-indexed Gated DeltaNet layer -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this module.  It shares no code with the CUDA library (it does not
import the package, and the package never imports it); the two meet only in
the seeded input generators.  Everything is float64 numpy written the plain
way, token by token, so that each line can be checked by eye.

Sources (page title and section):
  [P1] baseRT issue #31, "GDN recurrent state is single-sequence only":
       "Why this looks tractable" lists the per-layer kernels gdn_conv_silu and
       gdn_recurrence and a state cache sized by layers, heads, head_dim and
       conv_k with no slot dimension -- which this pool adds.
  [P2] b70-optimization-lab, "Plan (research-based)": "What the research
       found" -- speculative verify without per-draft-token state snapshots,
       chunked delta rule with the (I+A)^{-1} UT transform.
  [P3] ai-infra-handbooks, "Project: adding the hybrid model Qwen3.5":
       "What to do", State row -- one conv cache and one recurrent state per
       request slot, zero for a new request, carried across chunked-prefill
       chunks.  "Why it is worth doing" names the model's two kinds of
       RMSNorm; the output one (gated_rmsnorm below) is not written out
       there, so its formula is a reading (see that function).

The pages name the recurrence but never write it out.  The rule used is the
gated delta rule of Gated DeltaNet, for each value head:
    S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
    o_t = scale * S_t q_t
with S_t of shape [V, K], q_t and k_t L2-normalised (eps inside the sqrt),
alpha_t = exp(g_t) for the given log-decay g_t <= 0, and value head h reading
key head h // (H_v / H_k).  Readings of points the pages leave open (output
after the update, conv orientation, eps, head grouping) are listed in the
design notes beside this package.

Pins: every function here is checked in tests/test_oracle_pins.py against
closed forms, exact rational brute force, a library convolution and the
invariants the pages state (see that file's docstring for the map).
"""
from __future__ import annotations

import numpy as np

L2_EPS = 1e-6


def _f64(a):
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------- conv + SiLU

def silu(u):
    return u / (1.0 + np.exp(-u))


def conv_silu(x, cache, w, bias=None, advance=None):
    """Causal depthwise short conv followed by SiLU over one sequence [P1].

    x      [L, C]      raw inputs of this call, in time order
    cache  [C, W-1]    the W-1 raw inputs that precede x, oldest first
    w      [C, W]      taps; w[:, W-1] multiplies the current token
    bias   [C] or None
    advance            how many of the L tokens the cache moves past
                       (None: all L).  Outputs are produced for all L.

    Returns (y [L, C], new_cache [C, W-1]).
    """
    x, cache, w = _f64(x), _f64(cache), _f64(w)
    L, C = x.shape
    W = w.shape[1]
    assert cache.shape == (C, W - 1)
    # history row j holds the raw input at time j - (W-1) relative to x[0]
    hist = np.concatenate([cache.T, x], axis=0)
    y = np.empty((L, C))
    for t in range(L):
        window = hist[t:t + W]                      # [W, C], last row is x[t]
        u = np.sum(w.T * window, axis=0)
        if bias is not None:
            u = u + _f64(bias)
        y[t] = silu(u)
    a = L if advance is None else int(advance)
    assert 0 <= a <= L
    new_cache = hist[a:a + W - 1].T.copy()
    return y, new_cache


# ------------------------------------------------- storage formats (rounding)

def round_binary(x, p, emin, emax):
    """Round to the nearest value of a binary floating-point format with p
    significant bits (the leading one included), normal exponents emin..emax
    and subnormals below 2^emin, ties to the even significand; magnitudes
    beyond the format's range become infinities.  This is round-to-nearest-even
    as IEEE 754 defines it, applied once, straight from float64.

    Used where the layer stores an intermediate in a narrower format: the
    conv output in bf16 activations, and the recurrent state of a pool that
    keeps it in half precision."""
    x = _f64(x)
    _, E = np.frexp(np.abs(x))                 # |x| = m 2^E with m in [0.5, 1)
    e = np.maximum(E - 1, emin)                # exponent of the leading bit
    ulp = np.exp2(e - (p - 1))                 # spacing of the format at |x|
    r = np.round(x / ulp) * ulp                # np.round rounds halves to even
    top = (2.0 - 2.0 ** (1 - p)) * 2.0 ** emax
    return np.where(np.abs(r) > top, np.copysign(np.inf, x), r)


def round_bf16(x):
    """bfloat16: 8 significant bits, exponents -126..127."""
    return round_binary(x, 8, -126, 127)


def round_f16(x):
    """IEEE binary16: 11 significant bits, exponents -14..15."""
    return round_binary(x, 11, -14, 15)


# ------------------------------------------------------------ gated delta rule

def l2_normalize(x, eps=L2_EPS):
    """x / sqrt(sum(x^2) + eps) over the last axis."""
    x = _f64(x)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def expand_key_heads(a, h_v):
    """[..., H_k, d] -> [..., H_v, d]: value head h reads key head h // (H_v/H_k)."""
    a = _f64(a)
    h_k = a.shape[-2]
    assert h_v % h_k == 0
    return np.repeat(a, h_v // h_k, axis=-2)


def gdn_step(S, q, k, v, g, beta, scale=1.0, eps=L2_EPS):
    """One token of the gated delta rule for all value heads of one slot.

    S [H_v, V, K]; q, k [H_k, K]; v [H_v, V]; g, beta [H_v].
    Returns (S_new [H_v, V, K], o [H_v, V]); o is read from the updated state.
    """
    S = _f64(S)
    h_v = S.shape[0]
    kh = expand_key_heads(l2_normalize(k, eps), h_v)      # [H_v, K]
    qh = expand_key_heads(l2_normalize(q, eps), h_v)
    v, g, beta = _f64(v), _f64(g), _f64(beta)
    alpha = np.exp(g)
    a3 = alpha[:, None, None]
    b3 = beta[:, None, None]
    # S (I - beta k k^T) = S - beta (S k) k^T
    Sk = np.einsum("hvk,hk->hv", S, kh)
    S_new = a3 * (S - b3 * Sk[:, :, None] * kh[:, None, :]) \
        + b3 * v[:, :, None] * kh[:, None, :]
    o = scale * np.einsum("hvk,hk->hv", S_new, qh)
    return S_new, o


def gdn_recurrent(S0, q, k, v, g, beta, scale=1.0, eps=L2_EPS):
    """Token-by-token recurrence over one sequence of T tokens.

    q, k [T, H_k, K]; v [T, H_v, V]; g, beta [T, H_v].
    Returns (S_T, o [T, H_v, V])."""
    S = _f64(S0).copy()
    T = len(q)
    o = np.empty((T, S.shape[0], S.shape[1]))
    for t in range(T):
        S, o[t] = gdn_step(S, q[t], k[t], v[t], g[t], beta[t], scale, eps)
    return S, o


def gdn_chunked(S0, q, k, v, g, beta, scale=1.0, chunk=64, eps=L2_EPS):
    """The chunked form of the same recurrence [P2, "What the research found":
    chunked delta rule with the (I+A)^{-1} UT transform], kept as a second,
    independent oracle path to pin the identity chunked == token by token.

    Within a chunk of n tokens with local cumulative log-decay G_t = sum_{s<=t} g_s
    and gamma_t = exp(G_t), for each value head:
        A[t,i] = beta_t exp(G_t - G_i) k_t.k_i           (i < t; 0 elsewhere)
        Tm     = (I + A)^{-1}
        W      = Tm diag(beta gamma) K,   U = Tm diag(beta) V
        Delta  = U - W S0^T                  (the effective values, n x V)
        O      = diag(gamma) Q S0^T + (mask(i<=t) * exp(G_t - G_i) * Q K^T) Delta
        S_end  = gamma_n S0 + Delta^T diag(exp(G_n - G)) K
    """
    S = _f64(S0).copy()
    h_v, V, K = S.shape
    T = len(q)
    kh = expand_key_heads(l2_normalize(k, eps), h_v)      # [T, H_v, K]
    qh = expand_key_heads(l2_normalize(q, eps), h_v)
    v, g, beta = _f64(v), _f64(g), _f64(beta)
    o = np.empty((T, h_v, V))
    for h in range(h_v):
        Sh = S[h]
        for c0 in range(0, T, chunk):
            sl = slice(c0, min(c0 + chunk, T))
            Kc, Qc, Vc = kh[sl, h], qh[sl, h], v[sl, h]
            b, gc = beta[sl, h], g[sl, h]
            n = len(gc)
            G = np.cumsum(gc)
            gamma = np.exp(G)
            # exp(G_t - G_i) on and below the diagonal (upper part masked out)
            decay = np.tril(np.exp(np.tril(G[:, None] - G[None, :])))
            A = np.tril(b[:, None] * decay * (Kc @ Kc.T), -1)
            Tm = np.linalg.inv(np.eye(n) + A)
            Wm = Tm @ ((b * gamma)[:, None] * Kc)
            Um = Tm @ (b[:, None] * Vc)
            Delta = Um - Wm @ Sh.T
            P = decay * (Qc @ Kc.T)
            O = gamma[:, None] * (Qc @ Sh.T) + P @ Delta
            Sh = gamma[-1] * Sh + Delta.T @ (np.exp(G[-1] - G)[:, None] * Kc)
            o[sl, h] = scale * O
        S[h] = Sh
    return S, o


def spec_verify(S0, q, k, v, g, beta, accept_len=None, scale=1.0, eps=L2_EPS):
    """Speculative verify over T draft tokens of one slot [P2, "What the
    research found": outputs for every draft position, no per-position
    state snapshots].

    o_t is what t decode steps from the committed S0 give; the returned state
    is the state after `accept_len` steps (S0 itself when None or 0)."""
    S = _f64(S0).copy()
    T = len(q)
    keep = S.copy()
    a = 0 if accept_len is None else int(accept_len)
    assert 0 <= a <= T
    o = np.empty((T, S.shape[0], S.shape[1]))
    for t in range(T):
        S, o[t] = gdn_step(S, q[t], k[t], v[t], g[t], beta[t], scale, eps)
        if t + 1 == a:
            keep = S.copy()
    return o, keep


# ------------------------------------------------------------ input projection

def in_proj(x, w):
    """Input projection of the layer [P1, "Why this looks tractable" names
    gdn_in_proj without its formula; the reading is the layer's linear map of
    the hidden states]: y[t][n] = sum_h x[t][h] w[n][h], x [T, hidden],
    w [n_out, hidden] (one row per output channel), in float64."""
    return _f64(x) @ _f64(w).T


# ------------------------------------------------------ output gated RMSNorm

def gated_rmsnorm(o, z, w, eps=1e-6):
    """Output gated RMSNorm of a GDN layer [P3, "Why it is worth doing": the
    model has two kinds of RMSNorm; the formula is not printed there].
    Reading: each row (one token, one value head) of o is divided by its root
    mean square over the last axis (eps added inside the square root), scaled
    by the per-channel weight w and gated by SiLU of the matching row of z.
    o, z [..., d]; w [d]."""
    o, z, w = _f64(o), _f64(z), _f64(w)
    out = np.empty_like(o)
    rows_o = o.reshape(-1, o.shape[-1])
    rows_z = z.reshape(-1, z.shape[-1])
    rows_out = out.reshape(-1, o.shape[-1])
    for r in range(rows_o.shape[0]):
        mean_square = np.mean(rows_o[r] * rows_o[r])
        rows_out[r] = rows_o[r] / np.sqrt(mean_square + eps) * w * silu(rows_z[r])
    return out


# -------------------------------------------------------------------- the pool

class OraclePool:
    """Slot-indexed pool: per layer and slot a float64 state [H_v, V, K] and a
    conv cache [C, W-1] [P1 "Why this looks tractable"; P3 "What to do",
    State row].  Slots are independent; a new request starts from zero.

    state_round: None (the state is kept exactly), or round_bf16 / round_f16
    for a pool that stores its state in half precision [P1, "Why this looks
    tractable" names gdn_mp_factor_f16 and gdn_mp_scan_f16 without saying what
    they compute; the reading taken is half-precision storage of the state
    with full-precision arithmetic].  Within one call a slot's state is
    carried unrounded; it is rounded when the call stores it: after each
    decode step, at the end of each prefill sequence, at each prefill
    checkpoint, and at a verify's commit."""

    def __init__(self, n_layers, n_slots, h_v, h_k, dk, dv, conv_ch, conv_k,
                 state_round=None):
        self.h_v, self.h_k, self.dk, self.dv = h_v, h_k, dk, dv
        self.conv_ch, self.conv_k = conv_ch, conv_k
        self.S = np.zeros((n_layers, n_slots, h_v, dv, dk))
        self.X = np.zeros((n_layers, n_slots, conv_ch, conv_k - 1))
        self.state_round = state_round

    def _store(self, S):
        """The state as the pool stores it."""
        return S if self.state_round is None else self.state_round(S)

    def reset(self, slot_ids):
        for s in slot_ids:
            self.S[:, s] = 0.0
            self.X[:, s] = 0.0

    def conv_silu(self, layer, slot_ids, cu_seqlens, x, w, bias=None,
                  advance=None):
        """Varlen conv + SiLU: sequence i (tokens cu[i]:cu[i+1] of x) runs on
        slot slot_ids[i]'s cache; cu_seqlens None means one token per slot."""
        x = _f64(x)
        n = len(slot_ids)
        cu = np.arange(n + 1) if cu_seqlens is None else np.asarray(cu_seqlens)
        y = np.empty_like(x)
        for i, s in enumerate(slot_ids):
            lo, hi = int(cu[i]), int(cu[i + 1])
            a = None if advance is None else int(advance[i])
            y[lo:hi], self.X[layer, s] = conv_silu(
                x[lo:hi], self.X[layer, s], w, bias, a)
        return y

    def decode_step(self, layer, slot_ids, q, k, v, g, beta, scale=1.0,
                    eps=L2_EPS):
        """One token per active slot; q, k [N, H_k, K], v [N, H_v, V]."""
        o = np.empty((len(slot_ids), self.h_v, self.dv))
        for i, s in enumerate(slot_ids):
            S, o[i] = gdn_step(self.S[layer, s], q[i], k[i], v[i], g[i], beta[i], scale, eps)
            self.S[layer, s] = self._store(S)
        return o

    def prefill(self, layer, slot_ids, cu_seqlens, q, k, v, g, beta,
                scale=1.0, chunk=None, eps=L2_EPS):
        """Varlen prefill of packed sequences, starting from each slot's
        current state and leaving the final state in the slot [P3, State row].
        chunk None runs token by token, otherwise the chunked form."""
        o = np.empty((len(q), self.h_v, self.dv))
        for i, s in enumerate(slot_ids):
            lo, hi = int(cu_seqlens[i]), int(cu_seqlens[i + 1])
            args = (self.S[layer, s], q[lo:hi], k[lo:hi], v[lo:hi],
                    g[lo:hi], beta[lo:hi])
            if chunk is None:
                S, o[lo:hi] = gdn_recurrent(*args, scale, eps)
            else:
                S, o[lo:hi] = gdn_chunked(*args, scale, chunk, eps)
            self.S[layer, s] = self._store(S)
        return o

    def prefill_checkpointed(self, layer, slot_ids, cu_seqlens, q, k, v, g, beta,
                             ckpt_slots, ckpt_every, scale=1.0, eps=L2_EPS):
        """Prefill token by token that also saves state checkpoints [P3,
        "What to do", Prefix cache row: the prefix cache hits only where a
        state checkpoint was stored; "Why it is worth doing": a state is saved
        and copied whole].  ckpt_slots [n_seqs][m]: after (j + 1) * ckpt_every
        tokens of sequence i in this call, its state is copied into slot
        ckpt_slots[i][j] (skipped when negative)."""
        o = np.empty((len(q), self.h_v, self.dv))
        for i, s in enumerate(slot_ids):
            lo, hi = int(cu_seqlens[i]), int(cu_seqlens[i + 1])
            S = self.S[layer, s].copy()
            for t in range(lo, hi):
                S, o[t] = gdn_step(S, q[t], k[t], v[t], g[t], beta[t], scale, eps)
                n_done = t + 1 - lo
                if n_done % ckpt_every == 0:
                    j = n_done // ckpt_every - 1
                    if j < len(ckpt_slots[i]) and ckpt_slots[i][j] >= 0:
                        self.S[layer, ckpt_slots[i][j]] = self._store(S)
            self.S[layer, s] = self._store(S)
        return o

    def spec_verify(self, layer, slot_ids, T, q, k, v, g, beta,
                    accept_len=None, scale=1.0, eps=L2_EPS):
        """Draft token t of slot i is token i*T + t of q, k, v, g, beta.
        Returns o [N, T, H_v, V]; commits each slot at accept_len[i] when
        accept_len is given, else leaves the pool unchanged."""
        n = len(slot_ids)
        o = np.empty((n, T, self.h_v, self.dv))
        for i, s in enumerate(slot_ids):
            sl = slice(i * T, (i + 1) * T)
            a = None if accept_len is None else accept_len[i]
            o[i], S_keep = spec_verify(self.S[layer, s], q[sl], k[sl], v[sl],
                                       g[sl], beta[sl], a, scale, eps)
            if accept_len is not None and a > 0:
                self.S[layer, s] = self._store(S_keep)
        return o

    def spec_verify_deferred(self, layer, slot_ids, T, q, k, v, g, beta,
                             T_prev=0, prev=None, prev_accept=None, scale=1.0, eps=L2_EPS):
        """Deferred commit [P2, "What the research found": keep the drafts'
        inputs and write the full state back later].  Slot i first advances
        its committed state by the first prev_accept[i] of last round's
        drafts (prev = (q, k, v, g, beta), draft t at token i*T_prev + t) and
        commits it; then its T new drafts (token i*T + t) are verified on that
        state, outputs only.  Returns o [N, T, H_v, V]."""
        n = len(slot_ids)
        o = np.empty((n, T, self.h_v, self.dv))
        for i, s in enumerate(slot_ids):
            S = self.S[layer, s]
            if prev is not None:
                pq, pk, pv, pg, pb = prev
                for t in range(int(prev_accept[i])):
                    r = i * T_prev + t
                    S, _ = gdn_step(S, pq[r], pk[r], pv[r], pg[r], pb[r], scale, eps)
                if int(prev_accept[i]) > 0:
                    self.S[layer, s] = self._store(S)
            sl = slice(i * T, (i + 1) * T)
            o[i], _ = spec_verify(S, q[sl], k[sl], v[sl], g[sl], beta[sl], None, scale, eps)
        return o
