#!/usr/bin/env python
"""Benchmark of the ragged batched log-probability path on GB300.

One step = the whole hot path over one synthetic batch: ``lp_ragged_plan`` (output
offsets) + ``lp_ragged_compute`` (streaming max / sum-exp / top-k / target gather,
split-row merge). Default workload: decode, B=256 next-token rows of V=128256,
levels=3, no echo. Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle (the only reference that exists for
this path) on the host cores, on the same workload, one bounded sample per step.
Under torchrun every rank runs its own batch (weak scaling, no collective on the
data path); the step time is the max over ranks.
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "logit rows/sec and achieved HBM GB/s (fraction of GB300 peak) for ragged logprobs+top-k"
FALLBACK_HBM_GBS = 6800.0

WORKLOAD_TEXT = {
    "tiny": "tiny: B=4, lengths {3,5,1,7}, V=1000, levels=3, echo {T,F,T,F}, N(0,2) logits with one exact tie",
    "decode": "decode: B=256 next-token rows, V=128256, levels=3, no echo, N(0,3) logits + one +12 spike per row",
    "prefill": "prefill echo: B=8, lengths U[64,2048], V=32000, levels=3, all echo, N(0,2.5) logits",
    "mixed": "mixed ragged: B=64, lengths U[1,512], V=152064, levels=3, echo Bernoulli(0.5), Student-t(3)x2, "
             "1% -inf, 0.1% rows with a duplicated max",
    "wide": "wide top-k: B=32, lengths U[128,1024], V=256000, levels=6, all echo, N(0,1) quantised to 1/16",
}

VARIANT_TEXT = {
    "none": "",
    "temperature": "; per-batch temperatures U[0.25,2] (every 4th exactly 1), logprobs of x/tau",
    "variable": "; VARIABLE logits: only each sequence's last positions present (all for echo, 1-3 otherwise)",
    "vocab8": "; vocab-parallel over 8 shards, one rank's work on one GPU: partials over its 1/8 of the columns "
              "+ merge of the 8 gathered tuple slices (the all-gather between GPUs is not in the step)",
}
SHARDS = 8
# Workloads timed beside the headline one in the same run (per_config), and their steps.
PER_CONFIG = ("decode", "prefill", "mixed", "wide")
PER_CONFIG_STEPS = 200


# --batches N: the workload with N batches drawn from its own distributions (a smaller
# case of the same kernel for ncu captures that must stay within a few GB); None = as named.
SUB_BATCHES = None


def load_batch(config: str, variant: str, dev):
    import workloads
    batch = workloads.make_batch(config, dev, B=SUB_BATCHES, variable_extra=2 if variant == "variable" else None)
    if variant == "temperature":
        batch = workloads.with_temperatures(batch, seed=11)
    return batch


# ncu dram__bytes_read.sum + dram__bytes_write.sum per launch of the row kernel,
# keyed by workload, valid only while the kernels' device code hashes to the recorded value.
NCU_TRAFFIC = {
    "decode": {"source_hash": "14c2f37baacc42df", "kernel": "queue", "bytes_per_launch": 131518976,
               "how": "one-pass launch list (dram__bytes_read.sum + dram__bytes_write.sum), median of the 100 "
                      "lp_ragged_compute launches"},
    "prefill": {"source_hash": "14c2f37baacc42df", "kernel": "warp", "bytes_per_launch": 903248640,
                "how": "--set full capture of one launch (its writes include lines the replay restored)"},
    "mixed": {"source_hash": "14c2f37baacc42df", "kernel": "queue", "bytes_per_launch": 3344303530,
              "how": "one-pass capture of a 12-batch sub-batch (1298 rows) on the row queue, scaled by rows to 5476"},
    "wide": {"source_hash": "14c2f37baacc42df", "kernel": "warp", "bytes_per_launch": 22186875828,
             "how": "one-pass capture of a 3-batch sub-batch (2670 rows), scaled by rows to 21598"},
}


def _code_only(text: str) -> str:
    """The source with // comments and trailing blanks removed (string literals kept), so
    that a comment edit does not void counters taken on the same code."""
    out = []
    for line in text.splitlines():
        in_str, esc, cut = False, False, len(line)
        for i, ch in enumerate(line):
            if in_str:
                if esc:
                    esc = False
                elif ch == "\\":
                    esc = True
                elif ch == '"':
                    in_str = False
            elif ch == '"':
                in_str = True
            elif ch == "/" and line[i + 1:i + 2] == "/":
                cut = i
                break
        code = line[:cut].rstrip()
        if code:
            out.append(code)
    return "\n".join(out)


def kernel_source_hash() -> str:
    """Hash of the kernels' device code (the .cuh sources, comments stripped): the host
    file picks kernels and shapes, the device code decides what one launch moves."""
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "ragged_log_probs_gb300", "csrc", "*.cuh"))):
        with open(f, encoding="utf-8") as fh:
            h.update(os.path.basename(f).encode())
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def algorithmic_bytes(R: int, V: int, W: int, B: int) -> int:
    """Each scored logits row read once, outputs written once, offsets/tokens read."""
    return R * V * 4 + R * W * 8 + (B + 1) * 8 + R * 4


def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampled every 100 ms in the background; rows carry timestamps."""
    FIELDS = ("timestamp,index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()
        if self.path and os.path.exists(self.path):
            os.unlink(self.path)

    def summary(self, t0: float, t1: float):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 11:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[3]), float(parts[4]), parts[7:11]))
            except Exception:
                continue
        inside = [r for r in rows if t0 - 0.15 <= r[0] <= t1 + 0.15]
        window = "timed region"
        if not inside and rows:
            inside = sorted(rows, key=lambda r: abs(r[0] - (t0 + t1) / 2))[:2]
            window = "nearest samples (timed region shorter than the 100 ms sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# ------------------------------------------------------------------------ multi-rank
def combine_over_ranks(values, dist, device="cpu"):
    """Max of each timing over all ranks (each rank times its own batch; the job is as
    slow as its slowest rank). With no process group, the values come back unchanged."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_rows_per_s(rows_per_rank: int, world: int, ms_per_step: float) -> float:
    """Rows of all ranks divided by the (max-over-ranks) step time."""
    return rows_per_rank * world / (ms_per_step / 1e3)


# ------------------------------------------------------------------------ oracle leg
def _oracle_row(args):
    import oracle
    row, t, levels, tau = args
    return oracle.score_row(row, t, levels, tau)[0][0]


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_sample(batch, n_rows: int, seed: int = 0):
    """n scored rows (drawn with replacement once the workload's rows run out), copied
    device->host with their targets: the work items for the oracle."""
    import numpy as np
    import oracle
    off, tokens, sampled, echo = batch.host()
    ioff, tau = batch.host_variant()
    mapping = oracle.output_rows(off, echo, tokens, sampled, input_row_offsets=ioff)
    rng = np.random.default_rng(seed)
    picks = rng.choice(len(mapping), size=n_rows, replace=n_rows > len(mapping))
    cache = {}
    items = []
    for o in picks:
        b, r, t = mapping[o]
        if r not in cache:
            cache[r] = batch.logits[r].cpu().numpy()
        items.append((cache[r], t, batch.levels, 1.0 if tau is None else float(tau[b])))
    return items


def time_oracle(batch, target_cpu_s: float, pool, cores: int, items=None):
    """Time the oracle, as it stands, over a bounded row sample on the host cores."""
    probe = oracle_sample(batch, 1, seed=99)
    t = time.perf_counter()
    _oracle_row(probe[0])
    t_row = max(time.perf_counter() - t, 1e-4)
    n = int(max(cores, min(4000, target_cpu_s / t_row)))
    items = oracle_sample(batch, n, seed=1) if items is None else items
    pool.map(_oracle_row, items[:cores])  # workers import numpy/oracle before timing
    t0 = time.perf_counter()
    pool.map(_oracle_row, items, chunksize=1)
    dt = time.perf_counter() - t0
    return len(items), dt


def time_oracle_one_core(batch, budget_s: float = 2.0, max_rows: int = 64):
    """The same oracle on one core (this process), over a fresh random row sample, for
    about ``budget_s``: the per-core rate beside the pool's."""
    items = oracle_sample(batch, max_rows, seed=2)
    _oracle_row(items[0])  # imports and first-call costs outside the timing
    k, t0 = 0, time.perf_counter()
    for it in items:
        _oracle_row(it)
        k += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return k, time.perf_counter() - t0


# -------------------------------------------------------------------------- our arm
class Workload:
    """One workload on this rank's GPU, ready to time: its inputs (logits rotating over
    enough copies that each step reads HBM), workspace, outputs, and the library calls of
    one step and of one compute launch."""

    def __init__(self, config: str, variant: str, dev):
        import torch

        import ragged_log_probs_gb300 as lp
        self.lp, self.dev, self.config, self.variant = lp, dev, config, variant
        batch = self.batch = load_batch(config, variant, dev)
        self.B, self.T_logits, self.V, self.levels = batch.B, batch.T, batch.V, batch.levels
        self.T = batch.tokens.numel()  # input positions (== T_logits unless VARIABLE logits)
        self.extended = variant in ("temperature", "variable")
        self.sharded = variant == "vocab8"
        self.W = lp.out_per_token(self.levels)
        self.ws = lp.new_workspace(self.B, self.T, self.V, self.levels, dev)
        host = torch.zeros(2, dtype=torch.int32).pin_memory()
        self.out_off = lp.plan(batch.positions_offsets, batch.echo, self.T, self.ws, host_out=host)
        torch.cuda.synchronize()
        self.R = int(host[0])
        if int(host[1]) != 0:
            raise RuntimeError(f"plan status {int(host[1])}")
        self.out_lp = torch.empty((self.R, self.W), dtype=torch.float32, device=dev)
        self.out_tok = torch.empty((self.R, self.W), dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream()
        self.full_logits = batch.logits
        if self.sharded:
            # Rank 0's columns; the gathered buffer holds every shard's tuples (filled once,
            # as the all-gather would), so the merge in each step reads all P slices.
            bounds = [round(i * self.V / SHARDS) for i in range(SHARDS + 1)]
            stride = lp.tuple_bytes(self.levels)
            self.gathered = torch.zeros((SHARDS, self.R * stride), dtype=torch.uint8, device=dev)
            for p_ in range(SHARDS):
                lp.shard_partials(batch.logits[:, bounds[p_]:bounds[p_ + 1]].contiguous(), bounds[p_],
                                  batch.logit_row_offsets, batch.tokens, batch.sampled_tokens, self.out_off,
                                  batch.echo, self.levels, self.gathered[p_], self.R, self.ws)
            self.full_logits = batch.logits[:, bounds[0]:bounds[1]].contiguous()
        props = torch.cuda.get_device_properties(dev)
        self.l2 = int(getattr(props, "L2_cache_size", 0) or (128 << 20))
        self.lbytes = self.full_logits.numel() * 4
        self.n_copies = max(1, math.ceil(3 * self.l2 / self.lbytes))
        self.copies = [self.full_logits] + [self.full_logits.clone() for _ in range(self.n_copies - 1)]

    def launch_compute(self, logits, loff, ioff, tokens, sampled, echo, tau, st=None):
        lp, st = self.lp, (self.stream if st is None else st)
        if self.sharded:
            lp.shard_partials(logits, 0, loff, tokens, sampled, self.out_off, echo, self.levels, self.gathered[0],
                              self.R, self.ws, stream=st)
        elif self.extended:
            lp.compute_ex(logits, loff, tokens, sampled, self.out_off, echo, self.levels, self.out_lp, self.out_tok,
                          self.ws, input_row_offsets=ioff, temperatures=tau, stream=st)
        else:
            lp.compute(logits, loff, tokens, sampled, self.out_off, echo, self.levels, self.out_lp, self.out_tok,
                       self.ws, stream=st)

    def compute_k(self, k, st=None):
        b = self.batch
        self.launch_compute(self.copies[k % self.n_copies], b.logit_row_offsets, b.input_row_offsets, b.tokens,
                            b.sampled_tokens, b.echo, b.temperatures, st)

    def step(self, i, st=None):
        lp, b, st = self.lp, self.batch, (self.stream if st is None else st)
        if self.sharded:
            lp.plan(b.positions_offsets, b.echo, self.T, self.ws, output_row_offsets=self.out_off, stream=st)
            self.compute_k(i, st)
            lp.shard_merge(self.gathered, SHARDS, self.R, self.V, self.out_off, self.levels, self.out_lp,
                           self.out_tok, self.ws, stream=st)
        else:  # plan + reduction in one call (lp_ragged_step)
            lp.step(self.copies[i % self.n_copies], b.logit_row_offsets, b.tokens, b.sampled_tokens, b.echo,
                    self.levels, self.out_off, self.out_lp, self.out_tok, self.ws,
                    input_row_offsets=b.input_row_offsets, temperatures=b.temperatures, stream=st)

    def capture(self, n, body):
        """n calls of body(k, stream) captured in one CUDA graph (launch-bound loops replay
        without host launch overhead; the library's launches carry their programmatic
        dependencies into the graph)."""
        import torch
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream(device=self.dev)
        cs.wait_stream(self.stream)
        with torch.cuda.stream(cs):
            with torch.cuda.graph(g, stream=cs):
                for k in range(n):
                    body(k, cs)
        self.stream.wait_stream(cs)
        return g

    def warm(self, warmup: int):
        """Eager warm-up steps (they also do the library's one-time setup) and the sanity
        gate (parity itself is the tests' job): ids in range, logprobs <= 0."""
        import numpy as np
        import torch
        for i in range(warmup):
            self.step(i)
        torch.cuda.synchronize()
        if self.lp.read_status(self.ws) != 0:
            raise RuntimeError(f"{self.config}: device status set during warm-up")
        tok_np = self.out_tok.cpu().numpy().view(np.uint32)
        lp_np = self.out_lp.cpu().numpy()
        K = self.W - 1
        if np.any(tok_np[:, :K] >= self.V) or np.any(lp_np[~np.isnan(lp_np)] > 1e-4):
            raise RuntimeError(f"{self.config}: output sanity check failed")

    def graphs(self, steps: int, n_ev: int):
        """The timed K steps (plan + compute, inputs rotating) and, for the kernel's own
        duration, n_ev compute launches alone, each captured once in a CUDA graph."""
        import torch
        self.steps, self.n_ev = steps, n_ev
        self.g_steps = self.capture(steps, lambda k, st: self.step(k, st))
        self.g_compute = self.capture(n_ev, lambda k, st: self.compute_k(k, st))
        self.g_steps.replay()
        self.g_compute.replay()
        torch.cuda.synchronize()
        if self.lp.read_status(self.ws) != 0:
            raise RuntimeError(f"{self.config}: device status set during the graph warm-up")

    def time_graph(self, g, n, dist=None):
        """CUDA events on the launching stream around one replay, synchronised (and with a
        barrier under torchrun) on both sides; returns (ms per call, wall start, wall end)."""
        import torch
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        w0 = time.time()
        a.record(self.stream)
        g.replay()
        b.record(self.stream)
        torch.cuda.synchronize()
        w1 = time.time()
        if dist is not None:
            dist.barrier()
        return a.elapsed_time(b) / n, w0, w1

    def algorithmic_bytes(self):
        if self.sharded:  # the partial kernel: its columns read once, one tuple written per row
            return (self.R * self.full_logits.shape[1] * 4 + self.R * self.lp.tuple_bytes(self.levels)
                    + (self.B + 1) * 8 + self.R * 4)
        return algorithmic_bytes(self.R, self.V, self.W, self.B)

    def roofline(self, compute_ms: float) -> dict:
        alg = self.algorithmic_bytes()
        achieved = alg / (compute_ms / 1e3) / 1e9
        peak, peak_src = measured_peak_hbm()
        kind = self.lp.row_kernel(self.T_logits, self.T, self.V, self.levels)  # the library's own choice
        traffic, traffic_how = None, "no ncu capture recorded for this workload and kernel code"
        rec = NCU_TRAFFIC.get(self.config if self.variant == "none" else f"{self.config}/{self.variant}")
        if rec and SUB_BATCHES is None:
            if rec.get("source_hash") != kernel_source_hash():
                traffic_how = "the kernels' device code changed since the recorded ncu capture"
            elif rec.get("kernel") != kind:
                traffic_how = f"the recorded ncu capture is of the other row kernel ({rec.get('kernel')})"
            else:
                traffic, traffic_how = rec["bytes_per_launch"], rec["how"]
        entry = ("lp_ragged_shard_partials" if self.sharded else
                 ("lp_ragged_compute_ex" if self.extended else "lp_ragged_compute"))
        kernel_name = {"warp": f"k_rows ({entry}, warp ranges)", "queue": f"k_rows_cta ({entry}, row queue)"}[kind]
        return {"bound": "hbm", "kernel": kernel_name, "achieved": round(achieved, 1),
                "timing": f"CUDA events around one CUDA-graph replay of {self.n_ev} back-to-back compute launches, "
                          f"same stream, right after the timed steps",
                "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "traffic_source": traffic_how,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                else "fallback 6.8 TB/s", "algorithmic_bytes_per_launch": alg,
                "compute_ms_per_launch": round(compute_ms, 5)}

    def l2_note(self) -> str:
        return (f"inputs larger than L2: {self.n_copies} rotating logits copies of {self.lbytes / 1e6:.0f} MB "
                f"(L2 {self.l2 / 1e6:.0f} MB)")


def gpu_uuid(dev):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


def sub_batch_text() -> str:
    return "" if SUB_BATCHES is None else f" [sub-batch for profiling: {SUB_BATCHES} batches, same distributions]"


def run_ours(args, rank: int, world: int, dist):
    import torch

    import ragged_log_probs_gb300 as lp
    from ragged_log_probs_gb300 import _build

    _build.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = Workload(args.config, args.variant, dev)
    batch, B, T, T_logits, V, levels, W, R = wl.batch, wl.B, wl.T, wl.T_logits, wl.V, wl.levels, wl.W, wl.R
    stream = wl.stream
    wl.warm(args.warmup)
    n_ev = max(20, min(args.steps, 500))
    wl.graphs(args.steps, n_ev)

    sampler = ClockSampler(gpu_uuid(dev))
    sampler.start()
    # untimed settle so the clock samples see the GPU under load
    t_settle = time.perf_counter()
    while time.perf_counter() - t_settle < args.settle_s:
        wl.g_steps.replay()
        torch.cuda.synchronize()
    ms_step, w0, w1 = wl.time_graph(wl.g_steps, args.steps, dist)
    compute_ms, _, _ = wl.time_graph(wl.g_compute, n_ev)
    ms_step, compute_ms = combine_over_ranks([ms_step, compute_ms], dist, dev)
    clocks = sampler.summary(w0, w1)
    status = lp.read_status(wl.ws)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    # End to end through the public API: pinned host inputs -> device, plan+compute, results -> host.
    e2e = None
    if not args.no_e2e:
        full_logits, ws, out_off, out_lp, out_tok = wl.full_logits, wl.ws, wl.out_off, wl.out_lp, wl.out_tok
        h_logits = full_logits.cpu().pin_memory()
        # logits offsets, tokens, sampled, echo, then the variant's inputs (input offsets, temperatures)
        small = [batch.logit_row_offsets, batch.tokens, batch.sampled_tokens, batch.echo]
        small += [t for t in (batch.input_row_offsets, batch.temperatures) if t is not None]
        h_ints = [t.cpu().pin_memory() for t in small]
        d_logits = torch.empty_like(full_logits)
        d_ints = [torch.empty_like(t) for t in small]
        d_ioff = d_ints[4] if batch.input_row_offsets is not None else None
        d_tau = d_ints[-1] if batch.temperatures is not None else None
        h_lp = torch.empty((R, W), dtype=torch.float32).pin_memory()
        h_tok = torch.empty((R, W), dtype=torch.int32).pin_memory()
        h2d = h_logits.numel() * 4 + sum(t.numel() * t.element_size() for t in h_ints)
        d2h = h_lp.numel() * 4 + h_tok.numel() * 4
        k_e2e = int(max(3, min(args.steps, 40e9 // max(h2d, 1))))

        def e2e_step():
            d_logits.copy_(h_logits, non_blocking=True)
            for d, h in zip(d_ints, h_ints):
                d.copy_(h, non_blocking=True)
            if wl.sharded:
                lp.plan(d_ioff if d_ioff is not None else d_ints[0], d_ints[3], T, ws, output_row_offsets=out_off,
                        stream=stream)
                wl.launch_compute(d_logits, d_ints[0], d_ioff, d_ints[1], d_ints[2], d_ints[3], d_tau)
                lp.shard_merge(wl.gathered, SHARDS, R, V, out_off, levels, out_lp, out_tok, ws, stream=stream)
            else:
                lp.step(d_logits, d_ints[0], d_ints[1], d_ints[2], d_ints[3], levels, out_off, out_lp, out_tok, ws,
                        input_row_offsets=d_ioff, temperatures=d_tau, stream=stream)
            h_lp.copy_(out_lp, non_blocking=True)
            h_tok.copy_(out_tok, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        ea.record(stream)
        for _ in range(k_e2e):
            e2e_step()
        eb.record(stream)
        torch.cuda.synchronize()
        e2e_ms = ea.elapsed_time(eb) / k_e2e
        e2e_ms = combine_over_ranks([e2e_ms], dist, dev)[0]
        # The user-facing result objects on the host (top_n = 5 for every batch item, the
        # OpenAI "logprobs=5" case), from the rows copied out by the last e2e step.
        top_n = [min(5, W - 1)] * B
        h_off = out_off.cpu()
        t_asm = time.perf_counter()
        n_asm = 5
        for _ in range(n_asm):
            lp.assemble(h_off, h_lp, h_tok, top_n, V)
        asm_ms = (time.perf_counter() - t_asm) * 1e3 / n_asm
        e2e = {"value": whole_job_rows_per_s(R, world, e2e_ms), "unit": "rows/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms, "steps": k_e2e,
               "host_assembly_ms": round(asm_ms, 3)}
        del h_logits, d_logits

    roofline = wl.roofline(compute_ms)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import multiprocessing as mp
        cores = cpu_cores()
        with mp.get_context("spawn").Pool(cores) as pool:
            n, dt = time_oracle(batch, args.cpu_seconds, pool, cores)
        k1, dt1 = time_oracle_one_core(batch)
        cpu = {"value": n / dt, "unit": "rows/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} scored rows of this workload drawn at random (numpy fp64 oracle, full sort "
                         f"per row), {dt:.1f} s wall over a spawn pool of {cores} processes",
               "one_core": {"value": k1 / dt1, "unit": "rows/s", "cores": 1,
                            "sample": f"{k1} other random rows of this workload in the bench process, "
                                      f"{dt1:.1f} s"}}

    line = {
        "metric": METRIC, "value": whole_job_rows_per_s(R, world, ms_step), "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.config] + VARIANT_TEXT[args.variant] + sub_batch_text(),
                   "name": args.config, "variant": args.variant, "B": B, "T": T, "T_logits": T_logits, "V": V,
                   "levels": levels, "rows_per_gpu": R, "parallelism": f"replicas x{world} (independent batches)",
                   "l2": wl.l2_note(),
                   "launch": "the K timed steps (lp_ragged_step: plan + row kernel; vocab8: plan, partials, merge) "
                             "replayed from one CUDA graph"},
        "hbm_gbs_step": round(wl.algorithmic_bytes() * world / (ms_step / 1e3) / 1e9, 1),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": (3 if wl.sharded else 2) * args.steps, "clocks": clocks,
    }
    if wl.sharded:
        line["config"]["shards"] = SHARDS
        line["config"]["note"] = ("value = rows/s of one rank's step (partials over V/8 columns + merge); the 8 ranks "
                                  "run in parallel, so it is the job's rate less the all-gather, untimed on one GPU")
    del wl, batch
    torch.cuda.empty_cache()

    # The other workloads in the same run, each timed the same way (device timing; the
    # headline alone carries e2e and the oracle's rate), one at a time so that each one's
    # logits are freed before the next is built.
    if args.variant == "none" and not args.no_per_config and SUB_BATCHES is None:
        per = {}
        launches = 0
        for name in PER_CONFIG:
            if name == args.config:
                continue
            w = Workload(name, "none", dev)
            w.warm(args.warmup)
            k = max(3, min(args.steps, PER_CONFIG_STEPS))
            w.graphs(k, max(20, min(k, 100)))
            w.g_steps.replay()
            torch.cuda.synchronize()
            ms_k, a0, a1 = w.time_graph(w.g_steps, k, dist)
            c_ms, _, _ = w.time_graph(w.g_compute, w.n_ev)
            ms_k, c_ms = combine_over_ranks([ms_k, c_ms], dist, dev)
            if lp.read_status(w.ws) != 0:
                raise RuntimeError(f"{name}: device status set in the timed region")
            per[name] = {"workload": WORKLOAD_TEXT[name], "rows_per_gpu": w.R, "steps": k,
                         "value": whole_job_rows_per_s(w.R, world, ms_k), "unit": "rows/s", "ms_per_step": ms_k,
                         "hbm_gbs_step": round(w.algorithmic_bytes() * world / (ms_k / 1e3) / 1e9, 1),
                         "roofline": w.roofline(c_ms), "clocks": sampler.summary(a0, a1), "l2": w.l2_note()}
            launches += 2 * k
            del w
            torch.cuda.empty_cache()
        line["per_config"] = per
        line["gpu_launches_per_config"] = launches
    sampler.stop()
    if rank == 0:
        print(json.dumps(line), flush=True)


# -------------------------------------------------------------------- reference arm
def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    import multiprocessing as mp

    import torch
    import workloads

    cores = cpu_cores()
    with mp.get_context("spawn").Pool(cores) as pool:
        dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
        batch = load_batch(args.config, args.variant, dev)
        probe = oracle_sample(batch, 1, seed=99)
        t = time.perf_counter()
        _oracle_row(probe[0])
        t_row = max(time.perf_counter() - t, 1e-4)
        budget_s = 150.0
        steps_total = args.steps + args.warmup
        per_step = int(max(1, min(cores * 4, budget_s * cores / (t_row * steps_total))))
        items = oracle_sample(batch, per_step * 4, seed=1)
        pool.map(_oracle_row, items[:cores])
        times = []
        for k in range(steps_total):
            work = [items[(k * per_step + j) % len(items)] for j in range(per_step)]
            t0 = time.perf_counter()
            pool.map(_oracle_row, work, chunksize=1)
            if k >= args.warmup:
                times.append(time.perf_counter() - t0)
    ms_step = 1e3 * sum(times) / len(times)
    value = per_step / (ms_step / 1e3)
    sample = (f"{per_step} random scored rows of the workload per step (numpy fp64 oracle, full sort per row) "
              f"over a spawn pool of {cores} processes")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.config] + VARIANT_TEXT[args.variant] + sub_batch_text(),
                   "name": args.config, "variant": args.variant, "B": batch.B, "T": batch.tokens.numel(),
                   "T_logits": batch.T,
                   "V": batch.V, "levels": batch.levels},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="decode", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--variant", default="none", choices=sorted(VARIANT_TEXT),
                    help="input variant: per-batch temperature or VARIABLE logits (lp_ragged_compute_ex)")
    ap.add_argument("--settle-s", type=float, default=1.0)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batches", type=int, default=None,
                    help="profiling aid: the workload with this many batches from its own distributions "
                         "(labelled in config.workload; not a headline number)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the headline workload (no per_config entries for the others)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.batches is not None:
        if args.batches < 1:
            ap.error("--batches must be >= 1")
        global SUB_BATCHES
        SUB_BATCHES = args.batches

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    try:
        run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
