"""Helpers for the GPU parity tests: move seeded numpy inputs to the device in
the workload's dtype, compare against the oracle with the stated tolerances."""
import numpy as np
import torch

NAMES = ("q", "k", "v", "g", "beta")


def tdtype(dtype: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def dev(a, dtype: str = "f32"):
    """float32 numpy array (bf16-representable when dtype == 'bf16') -> cuda tensor."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device="cuda", dtype=tdtype(dtype))


def dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def tok_dev(tok: dict, dtype: str):
    return [dev(tok[n], dtype) for n in NAMES]


def tok_np(tok: dict):
    return [tok[n] for n in NAMES]


def host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_maxrel(got, ref, rel=1e-4, what=""):
    """max|got - ref| <= rel * max|ref| over the whole tensor."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.max(np.abs(got - ref)) if got.size else 0.0
    lim = rel * max(np.max(np.abs(ref)) if ref.size else 0.0, 1e-30)
    assert err <= lim, f"{what}: max err {err:.3e} > {lim:.3e}"


def assert_close_bf16(got, ref, atol=1e-2, rtol=1e-2, what=""):
    """elementwise |got - ref| <= atol + rtol |ref|."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    bad = np.abs(got - ref) > atol + rtol * np.abs(ref)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance, " \
                          f"max err {np.max(np.abs(got - ref)):.3e}"
