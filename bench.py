"""Benchmark of the slot-indexed Gated DeltaNet path on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]

Headline (one JSON line on stdout): decode slot-steps/s for one GDN layer
(32 value heads sharing 16 key heads, K = V = 128, fp32 state, conv_k = 4
over 8192 channels, bf16 activations) on a 256-slot pool with 64 active slot
ids drawn at random.  One step = one gdn_decode_step_conv call: the conv +
SiLU over the 64 new tokens, then the decode step reading q, k, v straight
out of the conv output (its launch overlapping the conv).  L2 is flushed (a
512 MiB write) between timed steps, outside the timed events.

Also in the line: the same metric end to end through the C ABI with inputs
copied from pinned host memory and outputs copied back inside the timed
region (`e2e`), the same step as two calls (`two_calls`: gdn_conv_silu, then
gdn_decode_step), the decode kernel's HBM roofline fraction (timed on the
decode launch of the two-call step), the oracle timed
on the host cores (`cpu_baseline`), SM clocks sampled during timing, and
`secondary` measurements: the 18-layer slot sweep (N = 1 .. 512),
speculative verify (128 slots, T = 4), varlen chunked prefill and the output
gated RMSNorm.

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


def _parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--sweep-steps", type=int, default=128)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--sections", default="sweep,verify,prefill,norm",
                    help="secondary measurements to run (comma list of sweep, verify, prefill, "
                         "norm)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-baseline-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
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


def _cpu_baseline_child(seconds: float):
    # calibrate one step of 8 slots, then run for about `seconds`
    dt, _ = _oracle_decode_sample(8, 1, 0)
    steps = max(1, int(seconds / max(dt, 1e-6)))
    dt, units = _oracle_decode_sample(8, steps, 1)
    print(json.dumps({"value": units / dt, "seconds": dt, "units": units, "steps": steps}))


def _cpu_env():
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    return env


def cpu_baseline(seconds: float):
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-child",
                        "--cpu-seconds", str(seconds)], capture_output=True, text=True,
                       env=_cpu_env(), cwd=ROOT, timeout=600)
    if r.returncode != 0:
        return {"error": r.stderr[-300:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": d["value"], "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"float64 numpy oracle, conv+SiLU then gated delta rule, on 8 of the 64 "
                      f"active slots of the decode workload for {d['steps']} steps "
                      f"({d['units']} slot-steps, {d['seconds']:.1f} s), single thread"}


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
        return d["hbm_gbs"], d.get("bf16_tflops"), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def _profiled_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode source."""
    try:
        text = open(PROFILE_SUMMARY).read()
        sha = hashlib.sha256(open(DECODE_SOURCE, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_sha256_16") != sha:
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class DecodeBench:
    def __init__(self, torch, abi, synth, device):
        self.torch = torch
        self.abi = abi
        wl = synth.decode_workload(seed=1)
        self.shape = s = wl["shape"]
        self.n = n = len(wl["slot_ids"])
        t = lambda a, dt=torch.bfloat16: torch.from_numpy(a).to(device=device, dtype=dt)
        self.pool = abi.Pool.for_shape(s, 1, wl["n_slots"], conv_dtype=torch.bfloat16,
                                       host_checks=False, device=device)
        gen = torch.Generator(device=device).manual_seed(1)
        self.pool.state.normal_(0.0, 0.1, generator=gen)
        lid = torch.from_numpy(wl["slot_ids"]).long().to(device)
        self.pool.state[0, lid] = t(wl["states"], torch.float32)
        self.pool.conv[0, lid] = t(wl["conv_cache"])
        self.ids = torch.from_numpy(wl["slot_ids"]).to(device)
        # x, g and beta of a step are packed into one bf16 buffer (x first, each
        # part 16-byte aligned), so the end-to-end leg stages them with one copy
        nx, ng = n * s.conv_ch, n * s.h_v
        self.inputs = torch.empty(nx + 2 * ng, device=device, dtype=torch.bfloat16)
        self.x = self.inputs[:nx].view(n, s.conv_ch)
        self.g = self.inputs[nx:nx + ng].view(n, s.h_v)
        self.beta = self.inputs[nx + ng:].view(n, s.h_v)
        self.x.copy_(t(wl["x"]))
        self.g.copy_(t(wl["tok"]["g"]))
        self.beta.copy_(t(wl["tok"]["beta"]))
        self.w = t(wl["conv_w"], torch.float32)
        self.y = torch.empty(n, s.conv_ch, device=device, dtype=torch.bfloat16)
        nq = s.h_k * s.dk
        self.q = self.y[:, :nq].view(n, s.h_k, s.dk)
        self.k = self.y[:, nq:2 * nq].view(n, s.h_k, s.dk)
        self.v = self.y[:, 2 * nq:].view(n, s.h_v, s.dv)
        self.o = torch.empty(n, s.h_v, s.dv, device=device)
        self.flush_buf = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=device)
        # pinned host buffers for the end-to-end leg
        self.inputs_h = self.inputs.cpu().pin_memory()
        self.o_h = torch.empty(self.o.shape, dtype=torch.float32).pin_memory()
        self.h2d = self.inputs_h.numel() * self.inputs_h.element_size()
        self.d2h = self.o_h.numel() * self.o_h.element_size()

    def flush(self):
        self.flush_buf.zero_()

    def step(self):
        """The decode step of the layer as one call (conv + SiLU, then the
        decode launch overlapping it)."""
        self.abi.gdn_decode_step_conv(self.pool, 0, self.ids, self.x, self.w, self.y, self.g,
                                      self.beta, self.o)

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

    def step_e2e(self):
        self.inputs.copy_(self.inputs_h, non_blocking=True)
        self.step()
        self.o_h.copy_(self.o, non_blocking=True)

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


def prefill_bench(torch, abi, synth, device, steps):
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
    return {"workload": f"varlen chunked prefill, decode-step layer shape, 8 sequences "
                        f"(lengths {lens}), pieces of 2048 tokens with the state carried "
                        f"between calls, bf16 in/out, chunk 64",
            "tokens_per_s": total * steps / t, "ms_per_pass": t / steps * 1e3,
            "calls_per_pass": len(calls),
            "single_launch_tokens_per_s": total * steps / t_single,
            "token_by_token_tokens_per_s": total * steps / t_rec,
            "speedup_over_token_by_token": t_rec / t}


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
    peak, _, peak_kind = _peaks()

    b = DecodeBench(torch, abi, synth, device)
    for _ in range(max(3, args.warmup)):
        b.step()
        b.step_two_calls()
        b.step_e2e()
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
    t_e2e, _ = b.timed(b.step_e2e, args.steps)
    barrier()
    secondary = {}
    sections = set() if args.no_secondary else set(args.sections.split(","))
    if "sweep" in sections:
        secondary["sweep"] = sweep_bench(torch, abi, synth, device, args.sweep_steps)
    if "verify" in sections:
        secondary["verify"] = verify_bench(torch, abi, synth, device, 50, peak)
    if "prefill" in sections:
        secondary["prefill"] = prefill_bench(torch, abi, synth, device, 5)
    if "norm" in sections:
        secondary["norm"] = norm_bench(torch, abi, device, 20, peak)
    time.sleep(0.2)
    clk = clocks.stop()
    if dist is not None:
        t_dev, t_e2e, t_two, t_kernel = max_over_ranks([t_dev, t_e2e, t_two, t_kernel], dist,
                                                       device)
    if rank != 0:
        return None

    units = b.n * args.steps * world
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
                "note": "pinned host x|g|beta (one packed buffer, one copy) -> device, "
                        "one-call conv + decode, o -> pinned host"},
        "two_calls": {"value": units / t_two, "unit": UNIT,
                      "ms_per_step": t_two / args.steps * 1e3,
                      "note": "the same step as gdn_conv_silu then gdn_decode_step, "
                              "an event between them"},
        "gpu_launches": 2 * args.steps,
        "roofline": {"bound": "hbm", "kernel": "decode_bulk_kernel<128, bf16, float, false>",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": _profiled_traffic(),
                     "peak_kind": f"{peak_kind} (HBM copy, burst)",
                     "algorithmic_bytes_per_launch": DECODE_KERNEL_BYTES_PER_SLOT * b.n,
                     "kernel_us": kernel_avg * 1e6,
                     "timed_on": "the decode launch of the two-call step (events between "
                                 "the launches; the one-call step overlaps them)"},
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
