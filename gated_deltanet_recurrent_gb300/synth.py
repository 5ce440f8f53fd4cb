"""Seeded synthetic inputs for the slot-indexed Gated DeltaNet path.

This module holds random draws, dtype rounding and the shapes of the
workloads, nothing of the layer's arithmetic.  It is the one module that both
the CUDA path (tests, benchmark, smoke check) and the CPU oracle are fed from.
It needs only numpy, so a CPU-only process can import it without torch.

Input recipe (the distributions of the tiny correctness workload, reused by
every other workload):
  q, k ~ N(0, 1), then scaled to unit L2 norm per head (the kernels normalise
        again, which is idempotent up to rounding);
  v    ~ N(0, 1);
  beta = sigmoid(N(0, 1));
  g    = -softplus(N(0, 1)) = log(alpha), so alpha = exp(-softplus(z)) in (0, 1);
  conv weights ~ N(0, 0.25^2) (standard deviation 0.25), no bias;
  conv input x ~ N(0, 1);
  non-zero initial states ~ N(0, 0.1^2).
bf16 values are produced by round-to-nearest-even from float32 and kept as
float32 arrays holding exactly representable bf16 numbers, so the oracle
(float64) and the GPU (bf16) consume the very same values.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class LayerShape:
    """Shape of one GDN layer: value heads, key heads, head dims, conv."""
    h_v: int
    h_k: int
    dk: int
    dv: int
    conv_ch: int
    conv_k: int

    @property
    def qkv_channels(self) -> int:
        return 2 * self.h_k * self.dk + self.h_v * self.dv


# 2 value / 2 key heads, K = V = 16, conv_k = 4 over 64 channels.
TINY_LAYER = LayerShape(h_v=2, h_k=2, dk=16, dv=16, conv_ch=64, conv_k=4)
# 32 value heads sharing 16 key heads, K = V = 128, conv_k = 4 over 8192
# channels (8192 = 2*16*128 + 32*128, so the conv output splits into q, k, v).
GDN_LAYER = LayerShape(h_v=32, h_k=16, dk=128, dv=128, conv_ch=8192, conv_k=4)


def round_bf16(x) -> np.ndarray:
    """Round float values to the nearest bf16 (ties to even); float32 result."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).reshape(x.shape)


def cast(x, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    if dtype == "bf16":
        return round_bf16(x)
    raise ValueError(f"unknown dtype {dtype!r}")


def _unit_rows(x: np.ndarray) -> np.ndarray:
    # Input recipe step: draws for q and k are rescaled to unit length per head.
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def token_inputs(rng: np.random.Generator, n_tokens: int, shape: LayerShape,
                 dtype: str = "f32") -> dict:
    """q, k [T, h_k, dk]; v [T, h_v, dv]; g, beta [T, h_v]."""
    q = _unit_rows(rng.standard_normal((n_tokens, shape.h_k, shape.dk)))
    k = _unit_rows(rng.standard_normal((n_tokens, shape.h_k, shape.dk)))
    v = rng.standard_normal((n_tokens, shape.h_v, shape.dv))
    zb = rng.standard_normal((n_tokens, shape.h_v))
    zg = rng.standard_normal((n_tokens, shape.h_v))
    beta = 1.0 / (1.0 + np.exp(-zb))
    g = -np.logaddexp(0.0, zg)
    return {name: cast(a, dtype) for name, a in
            (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta))}


def conv_input(rng: np.random.Generator, n_tokens: int, conv_ch: int,
               dtype: str = "f32") -> np.ndarray:
    return cast(rng.standard_normal((n_tokens, conv_ch)), dtype)


def conv_weights(rng: np.random.Generator, conv_ch: int, conv_k: int) -> np.ndarray:
    """[conv_ch, conv_k] float32; tap conv_k-1 multiplies the current token."""
    return cast(0.25 * rng.standard_normal((conv_ch, conv_k)), "f32")


def random_states(rng: np.random.Generator, n: int, shape: LayerShape,
                  std: float = 0.1) -> np.ndarray:
    """[n, h_v, dv, dk] float32 recurrent states ~ N(0, std^2)."""
    return cast(std * rng.standard_normal((n, shape.h_v, shape.dv, shape.dk)), "f32")


def random_conv_cache(rng: np.random.Generator, n: int, shape: LayerShape,
                      dtype: str) -> np.ndarray:
    """[n, conv_ch, conv_k-1] cached raw conv inputs ~ N(0, 1)."""
    return cast(rng.standard_normal((n, shape.conv_ch, shape.conv_k - 1)), dtype)


def cu_seqlens_of(lengths) -> np.ndarray:
    out = np.zeros(len(lengths) + 1, dtype=np.int32)
    out[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return out


# ----------------------------------------------------------------- workloads

def tiny_workload(seed: int = 0) -> dict:
    """Tiny correctness case: pool of 4 slots, sequences of 7 and 13 tokens in
    slots 1 and 3, fed in 4-token prefill pieces, then 5 decode steps with
    both slots active; afterwards slot 1 is reset and its request rerun.
    float32 throughout."""
    rng = np.random.default_rng(seed)
    shape = TINY_LAYER
    lengths = [7, 13]
    slots = [1, 3]
    n_decode = 5
    seqs = []
    for L in lengths:
        seqs.append({
            "x": conv_input(rng, L + n_decode, shape.conv_ch, "f32"),
            "tok": token_inputs(rng, L + n_decode, shape, "f32"),
        })
    w = conv_weights(rng, shape.conv_ch, shape.conv_k)
    return {"shape": shape, "n_slots": 4, "slots": slots, "lengths": lengths,
            "piece": 4, "n_decode": n_decode, "seqs": seqs, "conv_w": w,
            "dtype": "f32"}


def decode_workload(seed: int = 1, n_slots: int = 256, n_active: int = 64,
                    dtype: str = "bf16", shape: LayerShape = GDN_LAYER,
                    init_states: bool = True) -> dict:
    """One decode step of one layer: a pool of `n_slots`, `n_active` slot ids
    drawn as a random (unsorted) subset, one token per active slot."""
    rng = np.random.default_rng(seed)
    slot_ids = rng.choice(n_slots, n_active, replace=False).astype(np.int32)
    states = random_states(rng, n_active, shape) if init_states else None
    cache = random_conv_cache(rng, n_active, shape, dtype)
    x = conv_input(rng, n_active, shape.conv_ch, dtype)
    tok = token_inputs(rng, n_active, shape, dtype)
    w = conv_weights(rng, shape.conv_ch, shape.conv_k)
    return {"shape": shape, "n_slots": n_slots, "slot_ids": slot_ids,
            "states": states, "conv_cache": cache, "x": x, "tok": tok,
            "conv_w": w, "dtype": dtype}


def prefill_workload(seed: int = 3, n_seqs: int = 8, min_len: int = 512,
                     max_len: int = 8192, piece: int = 2048, dtype: str = "bf16",
                     shape: LayerShape = GDN_LAYER, lengths=None) -> dict:
    """Varlen chunked prefill: `n_seqs` sequences with integer lengths uniform
    on [min_len, max_len], each fed in `piece`-token calls; the first half of
    the sequences start from zeroed slots, the second half from N(0, 0.1)
    states.  Slot i holds sequence i."""
    rng = np.random.default_rng(seed)
    if lengths is None:
        lengths = rng.integers(min_len, max_len + 1, n_seqs)
    lengths = [int(L) for L in lengths]
    n_seqs = len(lengths)
    n_zero = n_seqs // 2
    states = np.zeros((n_seqs, shape.h_v, shape.dv, shape.dk), dtype=np.float32)
    states[n_zero:] = random_states(rng, n_seqs - n_zero, shape)
    total = int(sum(lengths))
    tok = token_inputs(rng, total, shape, dtype)
    return {"shape": shape, "lengths": lengths, "cu_seqlens": cu_seqlens_of(lengths),
            "piece": piece, "states": states, "tok": tok, "dtype": dtype,
            "slot_ids": np.arange(n_seqs, dtype=np.int32)}


def prefill_calls(lengths, piece: int):
    """Split sequences into chunked-prefill calls: call r packs the r-th
    `piece`-token piece of every sequence that still has one.  Returns a list
    of (seq_indices, starts, lens) with starts relative to each sequence."""
    calls = []
    r = 0
    while True:
        idx, starts, lens = [], [], []
        for i, L in enumerate(lengths):
            s = r * piece
            if s < L:
                idx.append(i)
                starts.append(s)
                lens.append(min(piece, L - s))
        if not idx:
            return calls
        calls.append((idx, starts, lens))
        r += 1


def verify_workload(seed: int = 4, n_slots: int = 256, n_active: int = 128,
                    T: int = 4, n_decode: int = 16, dtype: str = "bf16",
                    shape: LayerShape = GDN_LAYER) -> dict:
    """Speculative verify: `n_active` slots each verify T draft tokens; the
    accepted length of each slot is uniform on {0..T}; then `n_decode`
    decode steps run on the committed states."""
    rng = np.random.default_rng(seed)
    slot_ids = rng.choice(n_slots, n_active, replace=False).astype(np.int32)
    states = random_states(rng, n_active, shape)
    draft = token_inputs(rng, n_active * T, shape, dtype)
    accept = rng.integers(0, T + 1, n_active).astype(np.int32)
    decode = [token_inputs(rng, n_active, shape, dtype) for _ in range(n_decode)]
    return {"shape": shape, "n_slots": n_slots, "slot_ids": slot_ids, "T": T,
            "states": states, "draft": draft, "accept_len": accept,
            "decode": decode, "dtype": dtype}


SWEEP_SLOTS = (1, 4, 8, 16, 32, 64, 128, 256, 512)


def sweep_slot_order(seed: int = 2, n_slots: int = 512) -> np.ndarray:
    """Slot-sweep order: the first N entries are the active slots at size N."""
    return np.random.default_rng(seed).permutation(n_slots).astype(np.int32)


def gate_inputs(rng: np.random.Generator, n_tokens: int, h_v: int, dtype: str = "f32"):
    """g, beta [n_tokens, h_v] with the recipe of token_inputs:
    beta = sigmoid(N(0,1)), g = -softplus(N(0,1))."""
    zb = rng.standard_normal((n_tokens, h_v))
    zg = rng.standard_normal((n_tokens, h_v))
    return cast(-np.logaddexp(0.0, zg), dtype), cast(1.0 / (1.0 + np.exp(-zb)), dtype)


def sweep_workload(seed: int = 2, n_layers: int = 18, n_slots: int = 512,
                   n_states: int = 512, table_rows: int = 4096,
                   shape: LayerShape = GDN_LAYER, dtype: str = "bf16") -> dict:
    """Inputs of the stacked-layer slot sweep.

    Fresh draws for every (step, layer, slot) of 128 steps would be 19 GB of
    conv inputs, so each step's rows are picked from seeded tables instead:
    x [table_rows, conv_ch], g and beta [table_rows, h_v], row indices from
    sweep_rows(seed, step, layer, n).  The initial state and conv cache of
    layer l, slot s are entry state_index[l, s] of n_states seeded draws; the
    index is a permutation per layer, so the slots of one layer all start
    from different states.  Active slots at size N: order[:N]."""
    assert n_states >= n_slots
    rng = np.random.default_rng([seed, 0])
    states = random_states(rng, n_states, shape)
    caches = random_conv_cache(rng, n_states, shape, dtype)
    state_index = np.stack([rng.permutation(n_states)[:n_slots] for _ in range(n_layers)])
    x = conv_input(rng, table_rows, shape.conv_ch, dtype)
    g, beta = gate_inputs(rng, table_rows, shape.h_v, dtype)
    w = np.stack([conv_weights(rng, shape.conv_ch, shape.conv_k) for _ in range(n_layers)])
    return {"shape": shape, "n_layers": n_layers, "n_slots": n_slots,
            "order": sweep_slot_order(seed, n_slots), "state_table": states,
            "cache_table": caches, "state_index": state_index.astype(np.int64),
            "x": x, "g": g, "beta": beta, "conv_w": w, "table_rows": table_rows,
            "seed": seed, "dtype": dtype}


def sweep_rows(seed: int, step: int, layer: int, n: int, table_rows: int) -> np.ndarray:
    """Table rows of the inputs of `step` in `layer`: entry i is the row of
    the i-th active slot (order[i])."""
    return np.random.default_rng([seed, 1, step, layer]).integers(0, table_rows, n)
