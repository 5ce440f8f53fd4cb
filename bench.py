"""Benchmark of the slot-indexed Gated DeltaNet path on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]

Headline (one JSON line on stdout): decode slot-steps/s for one GDN layer
(32 value heads sharing 16 key heads, K = V = 128, fp32 state, conv_k = 4
over 8192 channels, bf16 activations) on a 256-slot pool with 64 active slot
ids drawn at random.  One step = one gdn_decode_step_conv call: the conv +
SiLU over the 64 new tokens and the decode step on its q, k, v (at this size
one fused kernel, a CTA per (slot, key head)).  L2 is flushed (a 512 MiB
write) between timed steps, outside the timed events.

Also in the line: the same metric end to end through the C ABI with every
step's inputs copied from pinned host memory and its output copied back inside
the timed regions (`e2e`; the copies run on a second stream, double-buffered,
overlapping the neighbouring steps' compute), the same step as two calls
(`two_calls`: gdn_conv_silu, then gdn_decode_step), the decode kernel's HBM
roofline fraction (timed on the decode launch of the two-call step), the
oracle timed on the host cores (`cpu_baseline`: one thread and all cores;
decode, prefill and verify), SM clocks sampled during timing, and
`steady_state` (back-to-back steps over rotating slot sets, no flush), and
`secondary` measurements: the 18-layer slot sweep (N = 1 .. 512), one layer
at N = 1 .. 16 (the small-N latency path),
speculative verify (128 slots, T = 4), varlen chunked prefill with its
roofline, the output gated RMSNorm, the decode step on pools that store the
state in bf16 / binary16, and the layer's input projection (gdn_in_proj).

--impl reference times the float64 CPU oracle on a bounded sample of the same
workload (the pages publish no runnable implementation of this path).
Under torchrun each rank runs its own replica (weak scaling, no data-path
collective); rank 0 prints the line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN decode slot-steps/s"
UNIT = "slot-steps/s"
DECODE_WORKLOAD = ("decode step, one GDN layer: 32 value heads / 16 key heads, K=V=128, "
                   "fp32 state, conv_k=4 over 8192 channels, bf16 activations, pool of 256 "
                   "slots with 64 active slot ids (random subset), one token per active slot")
STATE_BYTES_PER_SLOT_LAYER = 2 * 32 * 128 * 128 * 4          # state read + write
# decode kernel, per slot-step: state r+w, q/k (bf16, 16 heads x 128 each), v (bf16),
# g and beta (bf16, 32 each), o (fp32, 32 x 128)
DECODE_KERNEL_BYTES_PER_SLOT = STATE_BYTES_PER_SLOT_LAYER + 2 * 16 * 128 * 2 + 32 * 128 * 2 \
    + 2 * 32 * 2 + 32 * 128 * 4
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "gdn_decode_pool256_active64.md")
DECODE_SOURCE = os.path.join(ROOT, "gated_deltanet_recurrent_gb300", "csrc", "gdn_decode.cu")
PREFILL_SUMMARY = os.path.join(ROOT, "profiles", "gdn_prefill_split_varlen8_piece2048.md")
PREFILL_SOURCE = os.path.join(ROOT, "gated_deltanet_recurrent_gb300", "csrc",
                              "gdn_prefill_split.cu")
# chunked prefill, algorithmic work per token and value head (chunk 64, K = V = 128,
# triangular blocks exploited): on the tensor cores, in tf32 Delta = F T^T
# (16,640), the state update (32,768) and P Delta (8,320); in bf16 the state
# products with the raw rows, S K^T and S Q^T (2 x 32,768), and the key-side Gram
# products (K K^T 8,064 + Q K^T 8,320); forming T on the CUDA cores (~1,365)
PREFILL_FLOPS_TF32 = 16640 + 32768 + 8320
PREFILL_FLOPS_BF16 = 2 * 32768 + 8064 + 8320
PREFILL_FLOPS_SIMT = 1365
# bytes per token: q, k (16 x 128 each), v (32 x 128), g, beta (32 each) in bf16,
# o (32 x 128) out in bf16; plus the state read and written once per
# (sequence, call): 2 x 32 x 128 x 128 x 4 bytes
PREFILL_BYTES_PER_TOKEN = 2 * (2 * 16 * 128 + 32 * 128 + 2 * 32) + 2 * 32 * 128
PREFILL_STATE_BYTES_PER_SEQ_CALL = STATE_BYTES_PER_SLOT_LAYER


def _parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--sweep-steps", type=int, default=128)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--sections", default="sweep,small_n,verify,prefill,norm,half,in_proj",
                    help="secondary measurements to run (comma list of sweep, small_n, verify, "
                         "prefill, norm, half, in_proj)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-baseline-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    return ap.parse_args()


# ----------------------------------------------------------------- CPU side

def _oracle_decode_sample(n_slots_per_step: int, steps: int, warmup: int):
    """Time the oracle on conv + decode of `n_slots_per_step` slots per step of
    the decode workload; returns (seconds, slot-steps)."""
    import numpy as np
    from gated_deltanet_recurrent_gb300 import synth
    from oracle import gdn_oracle as O
    wl = synth.decode_workload(seed=1)
    s = wl["shape"]
    nq = s.h_k * s.dk
    m = n_slots_per_step
    S = [wl["states"][i].astype(np.float64) for i in range(m)]
    X = [wl["conv_cache"][i].astype(np.float64) for i in range(m)]

    def step():
        for i in range(m):
            y, X[i] = O.conv_silu(wl["x"][i:i + 1], X[i], wl["conv_w"])
            y = y[0]
            S[i], _ = O.gdn_step(S[i], y[:nq].reshape(s.h_k, s.dk),
                                 y[nq:2 * nq].reshape(s.h_k, s.dk),
                                 y[2 * nq:].reshape(s.h_v, s.dv),
                                 wl["tok"]["g"][i], wl["tok"]["beta"][i])

    for _ in range(warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    return time.perf_counter() - t0, steps * m


_WL = {}


def _workloads(n_tok=None):
    """The oracle baseline's inputs, built once per process: the decode and
    spec-verify workloads, and 8 prefill sequences of n_tok tokens drawn with
    the varlen-prefill workload's recipe."""
    from gated_deltanet_recurrent_gb300 import synth
    if "decode" not in _WL:
        _WL["decode"] = synth.decode_workload(seed=1)
        _WL["verify"] = synth.verify_workload(seed=4, n_decode=0)
    if n_tok is not None and _WL.get("prefill_tokens") != n_tok:
        _WL["prefill"] = synth.prefill_workload(seed=3, lengths=[n_tok] * 8)
        _WL["prefill_tokens"] = n_tok
    return _WL


def _decode_slots_task(args):
    """(slot indices, steps) -> (seconds, slot-steps): the oracle's conv +
    decode over those slots of the decode workload, `steps` times."""
    idx, steps = args
    import numpy as np
    from oracle import gdn_oracle as O
    wl = _workloads()["decode"]
    s = wl["shape"]
    nq = s.h_k * s.dk
    S = {i: wl["states"][i].astype(np.float64) for i in idx}
    X = {i: wl["conv_cache"][i].astype(np.float64) for i in idx}
    t0 = time.perf_counter()
    for _ in range(steps):
        for i in idx:
            y, X[i] = O.conv_silu(wl["x"][i:i + 1], X[i], wl["conv_w"])
            y = y[0]
            S[i], _ = O.gdn_step(S[i], y[:nq].reshape(s.h_k, s.dk),
                                 y[nq:2 * nq].reshape(s.h_k, s.dk),
                                 y[2 * nq:].reshape(s.h_v, s.dv),
                                 wl["tok"]["g"][i], wl["tok"]["beta"][i])
    return time.perf_counter() - t0, steps * len(idx)


def _prefill_task(args):
    """(sequence, chunk or None) -> (seconds, tokens): the oracle's prefill of
    one sample sequence (all heads), token by token (chunk None) or in the
    chunked form."""
    seq, chunk = args
    from oracle import gdn_oracle as O
    wl = _WL["prefill"]
    lo, hi = int(wl["cu_seqlens"][seq]), int(wl["cu_seqlens"][seq + 1])
    tok = [wl["tok"][k][lo:hi] for k in ("q", "k", "v", "g", "beta")]
    t0 = time.perf_counter()
    if chunk is None:
        O.gdn_recurrent(wl["states"][seq], *tok)
    else:
        O.gdn_chunked(wl["states"][seq], *tok, chunk=chunk)
    return time.perf_counter() - t0, hi - lo


def _verify_task(args):
    """(slot indices, repeats) -> (seconds, slot-verifies): the oracle's
    speculative verify with commit (T = 4) of those slots of the verify
    workload."""
    idx, reps = args
    from oracle import gdn_oracle as O
    wl = _workloads()["verify"]
    T = wl["T"]
    d = wl["draft"]
    t0 = time.perf_counter()
    for _ in range(reps):
        for i in idx:
            sl = slice(i * T, (i + 1) * T)
            O.spec_verify(wl["states"][i], d["q"][sl], d["k"][sl], d["v"][sl], d["g"][sl],
                          d["beta"][sl], wl["accept_len"][i])
    return time.perf_counter() - t0, reps * len(idx)


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def _timed_parallel(pool, fn, tasks):
    """Wall time of running tasks on the pool; returns (seconds, units)."""
    t0 = time.perf_counter()
    res = pool.map(fn, tasks, chunksize=1)
    return time.perf_counter() - t0, sum(u for _, u in res)


def _cpu_baseline_child(seconds: float):
    """The oracle on the host cores: one thread, then every core (one spawned
    worker process per core, each on its own slots or sequence), for decode,
    prefill (token by token and chunked) and verify.  About `seconds` of
    wall time per one-thread measurement; inputs are built before timing."""
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    out = {"cpu_model": _cpu_model(), "nproc": cores}
    _workloads(32)
    # decode: calibrate one step of 8 slots, then run for about `seconds`
    dt, _ = _decode_slots_task((list(range(8)), 1))
    steps = max(1, int(seconds / max(dt, 1e-6)))
    dt, units = _decode_slots_task((list(range(8)), steps))
    out["decode_1t"] = {"value": units / dt, "seconds": dt, "units": units, "steps": steps}
    # prefill: sequences sized for about seconds / 2 token by token
    t1, _ = _prefill_task((0, None))
    n_tok = max(64, min(2048, int(seconds / 2 / max(t1 / 32, 1e-6))))
    _workloads(n_tok)
    dt, units = _prefill_task((0, None))
    out["prefill_tbt_1t"] = {"value": units / dt, "seconds": dt, "tokens": units}
    dt, units = _prefill_task((0, 64))
    out["prefill_chunked_1t"] = {"value": units / dt, "seconds": dt, "tokens": units}
    # verify
    dv, _ = _verify_task(([0], 1))
    reps = max(1, int(seconds / 2 / max(dv * 8, 1e-6)))
    dt, units = _verify_task((list(range(8)), reps))
    out["verify_1t"] = {"value": units / dt, "seconds": dt, "units": units}
    with mp.get_context("spawn").Pool(cores, initializer=_workloads, initargs=(n_tok,)) as pool:
        pool.map(_verify_task, [([0], 1)] * cores, chunksize=1)   # workers up
        dt, units = _timed_parallel(pool, _decode_slots_task,
                                    [([w % 64], steps * 8) for w in range(cores)])
        out["decode_all"] = {"value": units / dt, "seconds": dt, "units": units}
        dt, units = _timed_parallel(pool, _prefill_task, [(w % 8, None) for w in range(cores)])
        out["prefill_tbt_all"] = {"value": units / dt, "seconds": dt, "tokens": units}
        dt, units = _timed_parallel(pool, _verify_task,
                                    [([w % 128], reps * 8) for w in range(cores)])
        out["verify_all"] = {"value": units / dt, "seconds": dt, "units": units}
    print(json.dumps(out))


def _cpu_env():
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    return env


def cpu_baseline(seconds: float):
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-child",
                        "--cpu-seconds", str(seconds)], capture_output=True, text=True,
                       env=_cpu_env(), cwd=ROOT, timeout=900)
    if r.returncode != 0:
        return {"error": r.stderr[-300:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    one, allc = d["decode_1t"], d["decode_all"]
    return {"value": allc["value"], "unit": UNIT, "cores": d["nproc"], "kind": "oracle",
            "cpu_model": d["cpu_model"],
            "sample": f"float64 numpy oracle, conv+SiLU then gated delta rule on the decode "
                      f"workload: {d['nproc']} worker processes (one per core), each on its "
                      f"own slot for {one['steps'] * 8} steps ({allc['units']} slot-steps, "
                      f"{allc['seconds']:.1f} s wall)",
            "single_thread": {"value": one["value"], "unit": UNIT, "cores": 1,
                              "sample": f"8 slots x {one['steps']} steps, "
                                        f"{one['seconds']:.1f} s"},
            "prefill": {"unit": "tokens/s",
                        "token_by_token_1t": d["prefill_tbt_1t"]["value"],
                        "chunked_1t": d["prefill_chunked_1t"]["value"],
                        "token_by_token_all_cores": d["prefill_tbt_all"]["value"],
                        "sample": f"sequences of {d['prefill_tbt_1t']['tokens']} tokens drawn "
                                  f"with the varlen-prefill recipe (32/16 heads, K = V = 128, "
                                  f"bf16 values); all cores: one sequence per worker"},
            "verify": {"unit": "slot-verifies/s", "one_thread": d["verify_1t"]["value"],
                       "all_cores": d["verify_all"]["value"],
                       "sample": "verify with commit, T = 4, slots of the spec-verify "
                                 "workload"}}


# ------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, on: bool):
        self.windows.append((time.time(), on))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in rows for j in range(4)
                          if r[5 + j].strip().lower() == "active"})
        busy = [x for x in sm if smax and x > 0.3 * max(smax)]
        return {"sm_mhz": statistics.median(busy or sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------------- GPU

def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["hbm_gbs"], d.get("bf16_tflops") or 1900.0, "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def _profile_fields(summary, source):
    """Machine-read fields ('- key: `value`' lines) of a committed ncu summary,
    or None unless it was taken on the current kernel source (its
    source_sha256_16 field matches)."""
    try:
        text = open(summary).read()
        sha = hashlib.sha256(open(source, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    return fields if fields.get("source_sha256_16") == sha else None


def _profiled_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode source."""
    f = _profile_fields(PROFILE_SUMMARY, DECODE_SOURCE)
    try:
        return float(f["dram_bytes_per_launch"]) if f else None
    except (KeyError, ValueError):
        return None


class DecodeBench:
    def __init__(self, torch, abi, synth, device, state_dtype=None):
        self.torch = torch
        self.abi = abi
        wl = synth.decode_workload(seed=1)
        self.shape = s = wl["shape"]
        self.n = n = len(wl["slot_ids"])
        t = lambda a, dt=torch.bfloat16: torch.from_numpy(a).to(device=device, dtype=dt)
        sdt = state_dtype or torch.float32
        self.pool = abi.Pool.for_shape(s, 1, wl["n_slots"], conv_dtype=torch.bfloat16,
                                       host_checks=False, device=device, state_dtype=sdt)
        gen = torch.Generator(device=device).manual_seed(1)
        self.pool.state.copy_(torch.randn(self.pool.state.shape, device=device,
                                          generator=gen).mul_(0.1).to(sdt))
        lid = torch.from_numpy(wl["slot_ids"]).long().to(device)
        self.pool.state[0, lid] = t(wl["states"], torch.float32).to(sdt)
        self.pool.conv[0, lid] = t(wl["conv_cache"])
        self.ids = torch.from_numpy(wl["slot_ids"]).to(device)
        # x, g and beta of a step are packed into one bf16 buffer (x first, each
        # part 16-byte aligned), so the end-to-end leg stages them with one copy;
        # two such buffers (and two o) let step i+1's inputs and step i-1's
        # output move while step i computes
        nx, ng = n * s.conv_ch, n * s.h_v
        self.nx, self.ng = nx, ng
        self.inputs = [torch.empty(nx + 2 * ng, device=device, dtype=torch.bfloat16)
                       for _ in range(2)]
        for buf in self.inputs:
            buf[:nx].copy_(t(wl["x"]).reshape(-1))
            buf[nx:nx + ng].copy_(t(wl["tok"]["g"]).reshape(-1))
            buf[nx + ng:].copy_(t(wl["tok"]["beta"]).reshape(-1))
        self.x, self.g, self.beta = self.parts(0)
        self.w = t(wl["conv_w"], torch.float32)
        self.y = torch.empty(n, s.conv_ch, device=device, dtype=torch.bfloat16)
        nq = s.h_k * s.dk
        self.q = self.y[:, :nq].view(n, s.h_k, s.dk)
        self.k = self.y[:, nq:2 * nq].view(n, s.h_k, s.dk)
        self.v = self.y[:, 2 * nq:].view(n, s.h_v, s.dv)
        self.os = [torch.empty(n, s.h_v, s.dv, device=device) for _ in range(2)]
        self.o = self.os[0]
        self.flush_buf = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=device)
        # pinned host buffers for the end-to-end leg (one per step parity)
        self.inputs_h = [b.cpu().pin_memory() for b in self.inputs]
        self.o_h = [torch.empty(self.o.shape, dtype=torch.float32).pin_memory()
                    for _ in range(2)]
        self.h2d = self.inputs_h[0].numel() * self.inputs_h[0].element_size()
        self.d2h = self.o_h[0].numel() * self.o_h[0].element_size()
        self.copy_stream = torch.cuda.Stream(device=device)

    def parts(self, j):
        s, n, nx, ng = self.shape, self.n, self.nx, self.ng
        b = self.inputs[j]
        return b[:nx].view(n, s.conv_ch), b[nx:nx + ng].view(n, s.h_v), b[nx + ng:].view(n, s.h_v)

    def flush(self):
        self.flush_buf.zero_()

    def step(self, j=0):
        """The decode step of the layer as one call (conv + SiLU, then the
        decode), on input buffer j."""
        x, g, beta = self.parts(j)
        self.abi.gdn_decode_step_conv(self.pool, 0, self.ids, x, self.w, self.y, g, beta,
                                      self.os[j])

    def step_two_calls(self, ev=None):
        """The same step as two calls; ev brackets the decode launch."""
        a = self.abi
        a.gdn_conv_silu(self.pool, 0, self.ids, self.x, self.w, self.y)
        if ev is not None:
            ev[0].record()
        a.gdn_decode_step(self.pool, 0, self.ids, self.q, self.k, self.v, self.g, self.beta,
                          self.o)
        if ev is not None:
            ev[1].record()

    def timed(self, fn, steps, kernel_events=False):
        torch = self.torch
        E = lambda: torch.cuda.Event(enable_timing=True)
        evs = [(E(), E()) for _ in range(steps)]
        kev = [(E(), E()) for _ in range(steps)] if kernel_events else None
        for i in range(steps):
            self.flush()
            evs[i][0].record()
            if kernel_events:
                fn(kev[i])
            else:
                fn()
            evs[i][1].record()
        torch.cuda.synchronize()
        total = sum(a.elapsed_time(b) for a, b in evs) / 1e3
        ktime = sum(a.elapsed_time(b) for a, b in kev) / 1e3 if kernel_events else None
        return total, ktime

    def timed_steady(self, steps):
        """Back-to-back one-call steps with no flush, rotating over four
        disjoint sets of 64 slots (the active set, then the other 192 slots of
        the pool): 512 MiB of state, four times L2, so each step streams its
        state from HBM while the previous step's dirty lines drain, as in a
        long run.  One timed region over all steps; returns seconds."""
        torch = self.torch
        if not hasattr(self, "slot_sets"):
            rest = sorted(set(range(self.pool.state.shape[1])) - set(self.ids.tolist()))
            self.slot_sets = [self.ids] + [
                torch.tensor(rest[64 * j:64 * (j + 1)], dtype=torch.int32, device=self.ids.device)
                for j in range(3)]
        x, g, beta = self.parts(0)

        def one(j):
            self.abi.gdn_decode_step_conv(self.pool, 0, self.slot_sets[j % 4], x, self.w, self.y,
                                          g, beta, self.os[0])

        for j in range(8):
            one(j)
        E = lambda: torch.cuda.Event(enable_timing=True)
        a, b = E(), E()
        torch.cuda.synchronize()
        a.record()
        for j in range(steps):
            one(j)
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3

    def timed_e2e(self, steps):
        """End to end through the C ABI from pinned host memory: every step's
        packed inputs are copied host -> device and its o device -> host, on a
        copy stream, overlapped with the neighbouring steps' compute.  The
        timed region of step i holds its compute and the copies of steps
        i + 1 (in) and i - 1 (out): the compute stream waits for both before
        the region's end event, and a region's copies start only after its
        start event, so no copy runs in the untimed L2 flush between regions.
        A last region holds the final output copy.  Returns seconds."""
        torch = self.torch
        cs, cp = torch.cuda.current_stream(), self.copy_stream
        E = lambda t=True: torch.cuda.Event(enable_timing=t)
        starts = [E() for _ in range(steps + 1)]
        ends = [E() for _ in range(steps + 1)]
        h2d_done = [E(False) for _ in range(steps + 1)]

        def h2d(i):
            self.inputs[i % 2].copy_(self.inputs_h[i % 2], non_blocking=True)
            h2d_done[i].record(cp)

        def d2h(i):
            self.o_h[i % 2].copy_(self.os[i % 2], non_blocking=True)

        torch.cuda.synchronize()
        for i in range(steps + 1):
            self.flush()
            starts[i].record(cs)
            cp.wait_event(starts[i])
            with torch.cuda.stream(cp):
                if i == 0:
                    h2d(0)
                if i > 0:
                    d2h(i - 1)
                if i + 1 < steps:
                    h2d(i + 1)
            if i < steps:
                cs.wait_event(h2d_done[i])
                self.step(i % 2)
            cs.wait_stream(cp)
            ends[i].record(cs)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / 1e3


def half_state_bench(torch, abi, synth, device, steps, peak):
    """The decode-step workload on pools storing the state in bf16 / f16
    (float32 arithmetic): one-call step and the decode kernel alone."""
    out = {}
    for name, dt in (("bf16", torch.bfloat16), ("f16", torch.float16)):
        b = DecodeBench(torch, abi, synth, device, state_dtype=dt)
        for _ in range(3):
            b.step()
            b.step_two_calls()
        torch.cuda.synchronize()
        t_one, _ = b.timed(b.step, steps)
        _, t_kernel = b.timed(b.step_two_calls, steps, kernel_events=True)
        per_slot = DECODE_KERNEL_BYTES_PER_SLOT - STATE_BYTES_PER_SLOT_LAYER // 2
        gbs = per_slot * b.n * steps / t_kernel / 1e9
        out[name] = {"slot_steps_per_s": b.n * steps / t_one,
                     "us_per_step": t_one / steps * 1e6,
                     "decode_kernel_us": t_kernel / steps * 1e6,
                     "decode_algorithmic_bytes_per_launch": per_slot * b.n,
                     "decode_gbs": gbs, "decode_hbm_frac": gbs / peak}
        del b
    out["workload"] = ("decode step workload (64 of 256 slots, one layer, bf16 activations) "
                       "on a pool storing the state in bf16 / binary16, float32 arithmetic; "
                       "L2 flushed between steps")
    return out


def small_n_bench(torch, abi, synth, device, steps):
    """One layer of the decode-step shape on a 256-slot pool with N = 1, 4, 8,
    16 active slots: the one-call step (one fused kernel while its grid fits
    the GPU at once) eager, and replayed from a CUDA graph of that one call.
    L2 flushed between steps."""
    s = synth.GDN_LAYER
    pool = abi.Pool.for_shape(s, 1, 256, conv_dtype=torch.bfloat16, host_checks=False,
                              device=device)
    gen = torch.Generator(device=device).manual_seed(11)
    pool.state.normal_(0.0, 0.1, generator=gen)
    order = torch.from_numpy(synth.sweep_slot_order(2, 256)).to(device)
    w = 0.25 * torch.randn(s.conv_ch, s.conv_k, device=device, generator=gen)
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=device)
    E = lambda: torch.cuda.Event(enable_timing=True)
    out = []
    for N in (1, 4, 8, 16):
        ids = order[:N].contiguous()
        x = torch.randn(N, s.conv_ch, device=device, generator=gen).bfloat16()
        g = (-torch.nn.functional.softplus(torch.randn(N, s.h_v, device=device,
                                                       generator=gen))).bfloat16()
        bt = torch.sigmoid(torch.randn(N, s.h_v, device=device, generator=gen)).bfloat16()
        y = torch.empty(N, s.conv_ch, device=device, dtype=torch.bfloat16)
        o = torch.empty(N, s.h_v, s.dv, device=device)
        step = lambda st=None: abi.gdn_decode_step_conv(pool, 0, ids, x, w, y, g, bt, o,
                                                          stream=st)

        def timed(fn):
            for _ in range(3):
                fn()
            evs = [(E(), E()) for _ in range(steps)]
            torch.cuda.synchronize()
            for a, b in evs:
                flush.zero_()
                a.record()
                fn()
                b.record()
            torch.cuda.synchronize()
            return statistics.median(a.elapsed_time(b) for a, b in evs) / 1e3

        t_eager = timed(step)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                step(side)
        torch.cuda.current_stream().wait_stream(side)
        t_graph = timed(graph.replay)
        del graph
        out.append({"n_active": N, "us_per_step_eager": t_eager * 1e6,
                    "us_per_step_graph": t_graph * 1e6,
                    "state_gbs_graph": N * STATE_BYTES_PER_SLOT_LAYER / t_graph / 1e9})
    del pool
    return {"workload": "one layer of the decode-step shape, 256-slot pool, N active, the "
                        "one-call step (median of the steps), L2 flushed between steps",
            "points": out}


def in_proj_bench(torch, abi, synth, device, steps, hbm_peak, bf16_peak):
    """gdn_in_proj on the layer's projection (hidden 2048 -> q | k | v, gate z,
    beta and decay logits = 12,352 outputs), bf16 in, bf16 out: a decode step
    (64 tokens, weight-read bound) and a prefill piece (16,384 tokens,
    tensor bound).  L2 flushed between timed calls.  torch.matmul (cuBLAS) on
    the same operands is timed beside it as context only."""
    hidden, n_out = 2048, 2 * 16 * 128 + 2 * 32 * 128 + 2 * 32
    gen = torch.Generator(device=device).manual_seed(7)
    w = (torch.randn(n_out, hidden, device=device, generator=gen) / hidden ** 0.5).bfloat16()
    pool = abi.Pool.for_shape(synth.LayerShape(2, 1, 16, 16, 64, 4), 1, 1,
                              conv_dtype=torch.float32, host_checks=False, device=device)
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=device)
    E = lambda: torch.cuda.Event(enable_timing=True)
    out = {}
    for name, tokens in (("decode_64", 64), ("prefill_16384", 16384)):
        x = torch.randn(tokens, hidden, device=device, generator=gen).bfloat16()
        y = torch.empty(tokens, n_out, device=device, dtype=torch.bfloat16)

        def timed(fn):
            for _ in range(3):
                fn()
            evs = [(E(), E()) for _ in range(steps)]
            torch.cuda.synchronize()
            for a, b in evs:
                flush.zero_()
                a.record()
                fn()
                b.record()
            torch.cuda.synchronize()
            return statistics.median(a.elapsed_time(b) for a, b in evs) / 1e3

        t = timed(lambda: abi.gdn_in_proj(pool, x, w, y))
        t_lib = timed(lambda: torch.matmul(x, w.t(), out=y))
        flops = 2.0 * tokens * hidden * n_out
        nbytes = 2.0 * (tokens * hidden + n_out * hidden + tokens * n_out)
        t_roof = max(flops / (bf16_peak * 1e12), nbytes / (hbm_peak * 1e9))
        out[name] = {"tokens": tokens, "us_per_call": t * 1e6, "tflops": flops / t / 1e12,
                     "gbs": nbytes / t / 1e9,
                     "bound": "tensor" if flops / (bf16_peak * 1e12) >= nbytes / (hbm_peak * 1e9)
                     else "hbm",
                     "roofline_frac": t_roof / t, "library_matmul_us": t_lib * 1e6}
    del pool
    out["workload"] = (f"input projection, hidden {hidden} -> {n_out} outputs (q|k|v 8192, gate "
                       f"4096, beta and decay logits 64), bf16 in/out, float32 accumulation; "
                       f"library_matmul_us: torch.matmul on the same operands (context)")
    return out


def sweep_bench(torch, abi, synth, device, steps):
    """18 stacked layers, N active slots of a 512-slot pool, `steps` decode
    steps per N; L2 flushed between steps."""
    s = synth.GDN_LAYER
    L, P = 18, 512
    pool = abi.Pool.for_shape(s, L, P, conv_dtype=torch.bfloat16, host_checks=False,
                              device=device)
    gen = torch.Generator(device=device).manual_seed(2)
    pool.state.normal_(0.0, 0.1, generator=gen)
    order = torch.from_numpy(synth.sweep_slot_order(2, P)).to(device)
    nq = s.h_k * s.dk
    sets = 2
    xs = [torch.randn(P, s.conv_ch, device=device, generator=gen).to(torch.bfloat16)
          for _ in range(sets)]
    w = (0.25 * torch.randn(L, s.conv_ch, s.conv_k, device=device, generator=gen))
    gs = [(-torch.nn.functional.softplus(torch.randn(P, s.h_v, device=device, generator=gen)))
          .to(torch.bfloat16) for _ in range(sets)]
    bs = [torch.sigmoid(torch.randn(P, s.h_v, device=device, generator=gen)).to(torch.bfloat16)
          for _ in range(sets)]
    y = torch.empty(P, s.conv_ch, device=device, dtype=torch.bfloat16)
    o = torch.empty(P, s.h_v, s.dv, device=device)
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=device)
    out = []
    for N in synth.SWEEP_SLOTS:
        ids = order[:N].contiguous()
        q = y[:N, :nq].view(N, s.h_k, s.dk)
        k = y[:N, nq:2 * nq].view(N, s.h_k, s.dk)
        v = y[:N, 2 * nq:].view(N, s.h_v, s.dv)

        def one_step(j):
            for layer in range(L):
                abi.gdn_conv_silu(pool, layer, ids, xs[j % sets][:N], w[layer], y[:N])
                abi.gdn_decode_step(pool, layer, ids, q, k, v, gs[j % sets][:N],
                                    bs[j % sets][:N], o[:N])

        def one_call_step(j):
            for layer in range(L):
                abi.gdn_decode_step_conv(pool, layer, ids, xs[j % sets][:N], w[layer], y[:N],
                                         gs[j % sets][:N], bs[j % sets][:N], o[:N])

        for j in range(3):
            one_step(j)
            one_call_step(j)
        E = lambda: torch.cuda.Event(enable_timing=True)

        def timed(step_fn):
            evs = [(E(), E()) for _ in range(steps)]
            torch.cuda.synchronize()
            for j in range(steps):
                flush.zero_()
                evs[j][0].record()
                step_fn(j)
                evs[j][1].record()
            torch.cuda.synchronize()
            return sum(a.elapsed_time(b) for a, b in evs) / 1e3

        t = timed(one_step)
        t_one = timed(one_call_step)

        def graph_time(step_fn):
            # the step's 36 launches captured once into a CUDA graph and replayed
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                step_fn(0)
            torch.cuda.current_stream().wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                step_fn(0)
            graph.replay()
            tg = timed(lambda j: graph.replay())
            del graph
            return tg

        t_graph = graph_time(one_step)
        t_one_graph = graph_time(one_call_step)
        slot_steps = N * steps
        out.append({"n_active": N, "slot_steps_per_s": slot_steps / t,
                    "slot_layer_steps_per_s": slot_steps * L / t,
                    "state_gbs": slot_steps * L * STATE_BYTES_PER_SLOT_LAYER / t / 1e9,
                    "ms_per_step": t / steps * 1e3,
                    "graph_slot_steps_per_s": slot_steps / t_graph,
                    "graph_state_gbs": slot_steps * L * STATE_BYTES_PER_SLOT_LAYER / t_graph / 1e9,
                    "graph_ms_per_step": t_graph / steps * 1e3,
                    "one_call_slot_steps_per_s": slot_steps / t_one,
                    "one_call_graph_slot_steps_per_s": slot_steps / t_one_graph,
                    "one_call_graph_ms_per_step": t_one_graph / steps * 1e3})
    del pool
    return {"workload": "18 stacked GDN layers (decode-step layer shape), 512-slot pool, "
                        f"N active, {steps} decode steps per N, conv+decode per layer, "
                        "L2 flushed between steps; graph_* = the step's 36 launches replayed "
                        "from one CUDA graph (inputs of step 0 each time); one_call_* = each "
                        "layer as one gdn_decode_step_conv call (decode launch overlapping "
                        "the conv)", "points": out}


def verify_bench(torch, abi, synth, device, steps, peak):
    wl = synth.verify_workload(seed=4)
    s, T = wl["shape"], wl["T"]
    n = len(wl["slot_ids"])
    pool = abi.Pool.for_shape(s, 1, wl["n_slots"], conv_dtype=torch.bfloat16,
                              host_checks=False, device=device)
    lid = torch.from_numpy(wl["slot_ids"]).long().to(device)
    pool.state[0, lid] = torch.from_numpy(wl["states"]).to(device)
    ids = torch.from_numpy(wl["slot_ids"]).to(device)
    draft = [torch.from_numpy(wl["draft"][nm]).to(device=device, dtype=torch.bfloat16)
             for nm in ("q", "k", "v", "g", "beta")]
    acc = torch.from_numpy(wl["accept_len"]).to(device)
    o = torch.empty(n, T, s.h_v, s.dv, device=device, dtype=torch.bfloat16)
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=device)
    E = lambda: torch.cuda.Event(enable_timing=True)

    def timed(round_fn):
        for _ in range(3):
            round_fn()
        evs = [(E(), E()) for _ in range(steps)]
        torch.cuda.synchronize()
        for j in range(steps):
            flush.zero_()
            evs[j][0].record()
            round_fn()
            evs[j][1].record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / 1e3 / steps

    # one pass with the accepted lengths known: outputs + commit
    t = timed(lambda: abi.gdn_spec_verify(pool, 0, ids, T, *draft, o=o, accept_len=acc))
    committing = int((wl["accept_len"] > 0).sum())
    tok_bytes = T * (2 * 16 * 128 * 2 + 32 * 128 * 2 + 2 * 32 * 2 + 32 * 128 * 2)
    per_call = n * STATE_BYTES_PER_SLOT_LAYER / 2 + committing * STATE_BYTES_PER_SLOT_LAYER / 2 \
        + n * tok_bytes
    gbs = per_call / t / 1e9
    # a speculative round when the acceptance is known only after the outputs:
    # two-phase (verify, then commit recomputing the drafts) against deferred
    # (the previous round's accepted drafts committed inside this round's call)
    t_two = timed(lambda: (abi.gdn_spec_verify(pool, 0, ids, T, *draft, o=o),
                           abi.gdn_spec_verify(pool, 0, ids, T, *draft, accept_len=acc)))
    t_def = timed(lambda: abi.gdn_spec_verify_deferred(pool, 0, ids, T, *draft, o, prev=draft,
                                                       prev_accept=acc))
    per_def = per_call + n * tok_bytes
    del pool
    return {"workload": "spec verify, decode-step layer shape, 128 active of 256 slots, T=4, "
                        "bf16 in/out, commit at accepted length U{0..4}, one pass",
            "slot_verifies_per_s": n / t, "us_per_call": t * 1e6,
            "algorithmic_gbs": gbs, "hbm_frac": gbs / peak,
            "round_two_phase_us": t_two * 1e6, "round_deferred_us": t_def * 1e6,
            "round_deferred_speedup": t_two / t_def,
            "deferred_algorithmic_gbs": per_def / t_def / 1e9,
            "deferred_hbm_frac": per_def / t_def / 1e9 / peak}


def norm_bench(torch, abi, device, steps, peak):
    """Output gated RMSNorm over 16,384 tokens x 32 value heads x 128: o fp32,
    z and y bf16 (512 MiB per call, larger than L2, so no flush)."""
    rows, d = 16384 * 32, 128
    gen = torch.Generator(device=device).manual_seed(5)
    o = 0.3 * torch.randn(rows, d, device=device, generator=gen)
    z = (2.0 * torch.randn(rows, d, device=device, generator=gen)).to(torch.bfloat16)
    w = 0.5 + torch.rand(d, device=device, generator=gen)
    y = torch.empty(rows, d, device=device, dtype=torch.bfloat16)
    for _ in range(3):
        abi.gdn_gated_rmsnorm(o, z, w, y)
    E = lambda: torch.cuda.Event(enable_timing=True)
    evs = [(E(), E()) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record()
        abi.gdn_gated_rmsnorm(o, z, w, y)
        b.record()
    torch.cuda.synchronize()
    t = statistics.median(a.elapsed_time(b) for a, b in evs) / 1e3
    nbytes = rows * d * (4 + 2 + 2) + d * 4
    return {"workload": "output gated RMSNorm, 16384 tokens x 32 value heads x 128, o fp32, "
                        "z and y bf16 (512 MiB per call > L2)",
            "us_per_call": t * 1e6, "algorithmic_gbs": nbytes / t / 1e9,
            "hbm_frac": nbytes / t / 1e9 / peak}


def prefill_bench(torch, abi, synth, device, steps, hbm_peak, bf16_peak):
    wl = synth.prefill_workload(seed=3)
    s = wl["shape"]
    lens = wl["lengths"]
    cu = wl["cu_seqlens"]
    pool = abi.Pool.for_shape(s, 1, len(lens), conv_dtype=torch.bfloat16, host_checks=False,
                              device=device)
    init = torch.from_numpy(wl["states"]).to(device)
    tok = [torch.from_numpy(wl["tok"][nm]).to(device=device, dtype=torch.bfloat16)
           for nm in ("q", "k", "v", "g", "beta")]
    o = torch.empty(int(cu[-1]), s.h_v, s.dv, device=device, dtype=torch.bfloat16)
    calls = []
    import numpy as np
    for idx, starts, ln in synth.prefill_calls(lens, wl["piece"]):
        # pack the pieces of this call contiguously
        rows = np.concatenate([np.arange(cu[i] + st, cu[i] + st + l)
                               for i, st, l in zip(idx, starts, ln)])
        rows_t = torch.from_numpy(rows).long().to(device)
        packed = [t[rows_t].contiguous() for t in tok]
        ccu = torch.from_numpy(synth.cu_seqlens_of(ln)).to(device)
        ids = torch.tensor(idx, dtype=torch.int32, device=device)
        ob = torch.empty(len(rows), s.h_v, s.dv, device=device, dtype=torch.bfloat16)
        calls.append((ids, ccu, packed, ob, max(ln)))

    # the same pool memory under a 1-byte workspace limit: the single-launch kernel
    single = abi.Pool.for_shape(s, 1, len(lens), conv_dtype=torch.bfloat16, host_checks=False,
                                device=device, prefill_workspace_max=1)

    def run(fn, pl):
        for ids, ccu, packed, ob, mx in calls:
            fn(pl, 0, ids, ccu, *packed, ob, max_seqlen=mx)

    def timed(fn, pl=pool):
        pl.state[0].copy_(init)
        run(fn, pl)
        E = lambda: torch.cuda.Event(enable_timing=True)
        evs = [(E(), E()) for _ in range(steps)]
        for j in range(steps):
            pl.state[0].copy_(init)
            evs[j][0].record()
            run(fn, pl)
            evs[j][1].record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / 1e3

    try:
        t = timed(abi.gdn_prefill_chunked)
        t_single = timed(abi.gdn_prefill_chunked, single)
        t_rec = timed(abi.gdn_prefill_recurrent)
    except abi.GDNError as e:
        return {"unavailable": str(e)}
    total = int(cu[-1])
    pass_s = t / steps
    seq_calls = sum(int(c[0].numel()) for c in calls)
    nbytes = total * PREFILL_BYTES_PER_TOKEN + seq_calls * PREFILL_STATE_BYTES_PER_SEQ_CALL
    heads = s.h_v
    f_tf32 = total * heads * PREFILL_FLOPS_TF32
    f_bf16 = total * heads * PREFILL_FLOPS_BF16
    flops = f_tf32 + f_bf16 + total * heads * PREFILL_FLOPS_SIMT
    # lower bounds on the pass: HBM traffic at the copy peak, tensor work at the
    # dense bf16 peak (tf32 runs at half of it on this part)
    t_hbm = nbytes / (hbm_peak * 1e9)
    t_tc = f_tf32 / (bf16_peak * 0.5e12) + f_bf16 / (bf16_peak * 1e12)
    prof = _profile_fields(PREFILL_SUMMARY, PREFILL_SOURCE) or {}
    roof = {"bound": "hbm" if t_hbm >= t_tc else "tensor",
            "algorithmic_bytes_per_pass": nbytes, "algorithmic_flops_per_pass": flops,
            "arithmetic_intensity": flops / nbytes,
            "achieved_gbs": nbytes / pass_s / 1e9, "achieved_tflops": flops / pass_s / 1e12,
            "roofline_ms": max(t_hbm, t_tc) * 1e3, "frac": max(t_hbm, t_tc) / pass_s,
            "peaks": f"HBM {hbm_peak:.0f} GB/s, bf16 {bf16_peak:.0f} TFLOP/s, tf32 half of "
                     f"bf16 (MEASURED_PEAKS.json)",
            "tensor_pipe_pct_state_walk": prof.get("tensor_pipe_pct_seq"),
            "tensor_pipe_pct_key_side": prof.get("tensor_pipe_pct_prep"),
            "dram_bytes_first_call": prof.get("dram_bytes_call0")}
    return {"workload": f"varlen chunked prefill, decode-step layer shape, 8 sequences "
                        f"(lengths {lens}), pieces of 2048 tokens with the state carried "
                        f"between calls, bf16 in/out, chunk 64",
            "tokens_per_s": total * steps / t, "ms_per_pass": pass_s * 1e3,
            "calls_per_pass": len(calls), "tokens_per_pass": total,
            "single_launch_tokens_per_s": total * steps / t_single,
            "token_by_token_tokens_per_s": total * steps / t_rec,
            "speedup_over_token_by_token": t_rec / t, "roofline": roof}


def max_over_ranks(values, dist, device):
    """Element-wise max of per-rank timings (the only cross-rank step: each
    rank runs its own pool replica, no data moves between ranks)."""
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def run_gpu(args, rank, world):
    import torch
    from gated_deltanet_recurrent_gb300 import abi, synth
    local = int(os.environ.get("LOCAL_RANK", "0"))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    abi.load_library()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    peak, tc_peak, peak_kind = _peaks()

    b = DecodeBench(torch, abi, synth, device)
    for _ in range(max(3, args.warmup)):
        b.step()
        b.step_two_calls()
    b.timed_e2e(max(3, args.warmup))
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    barrier()
    t_dev, _ = b.timed(b.step, args.steps)
    barrier()
    t_two, t_kernel = b.timed(b.step_two_calls, args.steps, kernel_events=True)
    barrier()
    t_e2e = b.timed_e2e(args.steps)
    barrier()
    t_steady = b.timed_steady(max(args.steps, 64))
    barrier()
    secondary = {}
    sections = set() if args.no_secondary else set(args.sections.split(","))
    if "sweep" in sections:
        secondary["sweep"] = sweep_bench(torch, abi, synth, device, args.sweep_steps)
    if "verify" in sections:
        secondary["verify"] = verify_bench(torch, abi, synth, device, 50, peak)
    if "prefill" in sections:
        secondary["prefill"] = prefill_bench(torch, abi, synth, device, 5, peak, tc_peak)
    if "norm" in sections:
        secondary["norm"] = norm_bench(torch, abi, device, 20, peak)
    if "half" in sections:
        secondary["half_state"] = half_state_bench(torch, abi, synth, device, 50, peak)
    if "small_n" in sections:
        secondary["small_n"] = small_n_bench(torch, abi, synth, device, 50)
    if "in_proj" in sections:
        secondary["in_proj"] = in_proj_bench(torch, abi, synth, device, 20, peak, tc_peak)
    time.sleep(0.2)
    clk = clocks.stop()
    if dist is not None:
        t_dev, t_e2e, t_two, t_kernel = max_over_ranks([t_dev, t_e2e, t_two, t_kernel], dist,
                                                       device)
    if rank != 0:
        return None

    units = b.n * args.steps * world
    # kernels of one headline step, by the library's own form rule
    launches_per_step = abi.gdn_decode_step_conv_launches(b.pool, b.n, torch.bfloat16,
                                                          b.os[0].dtype)
    kernel_avg = t_kernel / args.steps
    achieved = DECODE_KERNEL_BYTES_PER_SLOT * b.n / kernel_avg / 1e9
    line = {
        "metric": METRIC, "value": units / t_dev, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_dev / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; N(0,0.1) states, distributions of the tiny correctness case)",
        "config": {"workload": DECODE_WORKLOAD, "n_slots": 256, "n_active": b.n,
                   "layers": 1, "l2": "flushed between timed steps (512 MiB write, untimed)",
                   "activations": "bf16", "state": "fp32", "parallelism":
                   f"replicas x{world}" if world > 1 else "single GPU"},
        "e2e": {"value": units / t_e2e, "unit": UNIT, "h2d_bytes_per_step": b.h2d,
                "d2h_bytes_per_step": b.d2h,
                "note": "per step: pinned host x|g|beta (one packed buffer, one copy) -> "
                        "device, one-call conv + decode, o -> pinned host; copies on a "
                        "second stream, double-buffered, overlapping the neighbouring "
                        "steps' compute inside the timed regions"},
        "steady_state": {"value": b.n * max(args.steps, 64) * world / t_steady, "unit": UNIT,
                         "ms_per_step": t_steady / max(args.steps, 64) * 1e3,
                         "step_algorithmic_gbs": DECODE_KERNEL_BYTES_PER_SLOT * b.n
                         * max(args.steps, 64) / t_steady / 1e9,
                         "step_hbm_frac": DECODE_KERNEL_BYTES_PER_SLOT * b.n * max(args.steps, 64)
                         / t_steady / 1e9 / peak,
                         "note": "back-to-back one-call steps, no flush, rotating over four "
                                 "disjoint 64-slot sets of the pool (512 MiB of state)"},
        "two_calls": {"value": units / t_two, "unit": UNIT,
                      "ms_per_step": t_two / args.steps * 1e3,
                      "note": "the same step as gdn_conv_silu then gdn_decode_step, "
                              "an event between them"},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"bound": "hbm", "kernel": "decode_bulk_kernel<128, bf16, float, false>",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": _profiled_traffic(),
                     "peak_kind": f"{peak_kind} (HBM copy, burst)",
                     "algorithmic_bytes_per_launch": DECODE_KERNEL_BYTES_PER_SLOT * b.n,
                     "kernel_us": kernel_avg * 1e6,
                     "timed_on": "the decode launch of the two-call step (events between "
                                 "the launches; the one-call step fuses the conv into its "
                                 "own kernel)"},
        "clocks": clk,
    }
    if secondary:
        line["secondary"] = secondary
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return line


def run_reference(args, rank):
    if rank != 0:
        return None
    slots = 8
    dt, units = _oracle_decode_sample(slots, args.steps, args.warmup)
    v = units / dt
    return {"metric": METRIC, "value": v, "unit": UNIT, "impl": "reference", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": DECODE_WORKLOAD, "sample": f"{slots} of the 64 active "
                       "slots per step"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "cpu_baseline": {"value": v, "unit": UNIT, "kind": "oracle",
                             "cores": int(os.environ.get("OMP_NUM_THREADS", "1") or 1),
                             "sample": f"float64 numpy oracle, conv+SiLU + gated delta rule on "
                                       f"{slots} slots per step, {args.steps} steps"}}


def main():
    args = _parse()
    if args.cpu_baseline_child:
        _cpu_baseline_child(args.cpu_seconds)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ.setdefault(v, "1")
        line = run_reference(args, rank)
    else:
        line = run_gpu(args, rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
