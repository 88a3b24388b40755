"""Benchmark of the Gated MLA decode hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step is one gated MLA decode call (scores, softmax, P.V, split-KV
log-sum-exp merge and sigmoid gate) over the whole synthetic cache of the
workload: B=32 sequences, 96 heads, 8192 cached positions each, bf16
(16.1 GB of keys and values per step, far larger than the 129 MB L2, so no
flush is needed between steps). The metric is KV-read GB/s: the algorithmic
bytes of the cache (every head's full 192+128 features per position) per
step divided by the device time per step.

Under torchrun with N>1 each rank runs its own replica on its own GPU (the
path shards by sequence with no exchange step); value = all ranks' bytes
divided by the slowest rank's time.

`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload on this host's cores (the only reference implementation there is).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import mla_inputs as mi  # noqa: E402
from mla_family_attention_gb300 import accounting as acc  # noqa: E402

METRIC = "MLA decode KV-read GB/s (% HBM peak); prefill attn TFLOP/s (% bf16 peak)"
DEFAULT_WORKLOAD = "decode_b32_h96_t8192"
FALLBACK_HBM_GBS = 6800.0
CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


FALLBACK_BF16_TFLOPS = 1900.0


def peaks(bound="hbm"):
    """(peak, unit, source): HBM copy GB/s, or the dense bf16 TFLOP/s of a
    kernel timed alone (burst), from the measured file if present."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        if bound == "tensor":
            return float(d["bf16_tflops"]), "TFLOP/s", "measured (burst)"
        return float(d["hbm_gbs"]), "GB/s", "measured"
    if bound == "tensor":
        return FALLBACK_BF16_TFLOPS, "TFLOP/s", "fallback"
    return FALLBACK_HBM_GBS, "GB/s", "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 100 ms while the bench runs."""

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def finish(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for r in csv.reader(io.StringIO(out)):
            if len(r) < 10:
                continue
            r = [x.strip() for x in r]
            try:
                ts = time.mktime(time.strptime(r[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(r[2]), float(r[3]), r[4], r[5:]))
            except ValueError:
                continue
        inside = [x for x in rows if self.t0 - 1 <= x[0] <= self.t1 + 1] or rows
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for x in inside for i in range(1, 5)
                          if x[4][i].lower().startswith("active")})
        return {"sm_mhz": statistics.median([x[1] for x in inside]) if inside else None,
                "sm_max_mhz": max([x[2] for x in inside]) if inside else None,
                "reasons": reasons, "samples": len(inside)}


def traffic_for(kernel: str, units=None):
    """DRAM bytes per launch from a committed ncu summary, if the kernel's source
    has not changed since the capture.  The summary records the algorithmic
    units (bytes or flops) of the launch it describes; a launch of the same
    kernel on another workload gets that traffic scaled by its own units
    (these kernels' traffic grows with the work they are given)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path)).get(kernel)
    if not d or d.get("dram_bytes_per_launch") is None:
        return None
    src = os.path.join(ROOT, d["source"])
    if not os.path.exists(src):
        return None
    if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != d["source_sha256_16"]:
        return None
    ref = d.get("algorithmic_per_launch")
    if units is None or not ref:
        return d["dram_bytes_per_launch"]
    return int(round(d["dram_bytes_per_launch"] * units / ref))


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ------------------------------------------------------------------------------------------
def oracle_inputs(dec, n_seq: int):
    """fp64 copies of the first n_seq sequences (all heads): the oracle's inputs."""
    H = dec.H
    npos = sum(dec.lengths[:n_seq])
    return dict(q=dec.q[:n_seq].to("cpu", torch.float64).numpy(),
                k=dec.k[:npos * H * 192].to("cpu", torch.float64).numpy(),
                v=dec.v[:npos * H * 128].to("cpu", torch.float64).numpy(),
                cu_seqlens=dec.cu_seqlens[:n_seq + 1].to("cpu").numpy(),
                gate=dec.gate[:n_seq].to("cpu", torch.float64).numpy(),
                scale=dec.scale)


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _repeat(fn, seconds: float):
    """Run fn until `seconds` of wall time have passed (at least once);
    returns (seconds elapsed, repeats)."""
    reps, t0 = 0, time.perf_counter()
    while True:
        fn()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return el, reps


def _cpu_result(units_per_s, unit_scale, unit, sample, extrapolated=False):
    import oracle
    return {"value": round(units_per_s / unit_scale, 6), "unit": unit,
            "cores": oracle.set_threads(0), "kind": "oracle",
            "sample": sample + (" (extrapolated)" if extrapolated else "")}


def _decode_seq_inputs(dec, b: int, heads: int):
    """fp64 oracle inputs for sequence b of a packed decode cache, first `heads` heads."""
    H, T = dec.H, dec.lengths[b]
    o = int(dec.cu_seqlens[b].item()) * H
    k = dec.k[o * 192:(o + H * T) * 192].view(H, T, 192)[:heads]
    v = dec.v[o * 128:(o + H * T) * 128].view(H, T, 128)[:heads]
    return dict(q=_f64(dec.q[b:b + 1, :heads]), k=_f64(k).reshape(-1), v=_f64(v).reshape(-1),
                cu_seqlens=np.array([0, T], dtype=np.int64),
                gate=None if dec.gate is None else _f64(dec.gate[b:b + 1, :heads * 128]),
                scale=dec.scale)


def run_reference(args, world, rank):
    """Reference arm: the fp64 CPU oracle on this host's cores, one sequence
    (all heads) of the workload per step (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    name = args.workload
    w = mi.WORKLOADS[name]
    lengths = mi.workload_lengths(name)
    n_seq = 1
    dec = mi.make_decode(lengths[:n_seq], w["H"], True, device="cpu", config=w["config"])
    threads = oracle.set_threads(len(os.sched_getaffinity(0)))
    x = oracle_inputs(dec, n_seq)
    for _ in range(args.warmup):
        oracle.mla_decode(**x)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.mla_decode(**x)
    per_step = (time.perf_counter() - t0) / args.steps
    nbytes = acc.decode_kv_bytes(lengths[:n_seq], w["H"])
    value = nbytes / per_step / 1e9
    sample = (f"{n_seq} of {len(lengths)} sequences x {w['H']} heads x {lengths[0]} positions "
              "per step (fp64 inputs prepared once)")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_step * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(name),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(name, B=None):
    w = mi.WORKLOADS[name]
    cfg = {"workload": name if B in (None, w["B"]) else f"{name} (first {B} sequences)",
           "B": B or w["B"], "H": w["H"], "head_dims": "qk 192 (128+64 shared), v 128",
           "gate": bool(w.get("gated", True))}
    if "T" in w:
        cfg["T"] = w["T"]
    if "lo" in w:
        cfg["T_range"] = [w["lo"], w["hi"]]
    if "chunk" in w:
        cfg["chunk"] = w["chunk"]
    small = w["kind"] == "prefill" and w["T"] <= 1024
    cfg["l2"] = ("inputs smaller than L2: step i reads copy i mod N of them (N copies "
                 "together over 4x L2); the N calls are captured once as a CUDA graph and "
                 "replayed back to back; the latency of one call after a 512 MB L2-flushing "
                 "write is reported beside it"
                 if small else "inputs larger than L2 (no flush needed)")
    return cfg


# ------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------
class DecodeWork:
    """Gated MLA decode over a packed cache (rows a1-a6)."""

    def __init__(self, name, dev, batch=0):
        import mla_family_attention_gb300 as mla
        from mla_family_attention_gb300 import _lib
        self.mla, self.lib = mla, _lib
        w = mi.WORKLOADS[name]
        lengths = mi.workload_lengths(name)
        if batch:
            lengths = lengths[:batch]          # smaller case of the same kernel (profiling)
        self.name, self.lengths, self.H, self.B = name, lengths, w["H"], len(lengths)
        self.max_len = max(lengths)
        self.dec = mi.make_decode(lengths, self.H, True, device=dev, config=w["config"])
        self.out = torch.empty((self.B, self.H * 128), dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(mla.workspace_size(_lib.OP_DECODE, self.B, self.H, self.max_len, 0),
                              dtype=torch.uint8, device=dev)
        self.work = acc.decode_kv_bytes(lengths, self.H)
        self.unit, self.bound = "GB/s", "hbm"
        self.launches_per_step = 3
        # (timer op, kernel name, algorithmic bytes per launch)
        self.kernels = [(_lib.OP_DECODE, "decode_partial_kernel", self.work)]

    def step(self, stream):
        d = self.dec
        self.mla.mla_decode(d.q, d.k, d.v, d.cu_seqlens, self.max_len, gate=d.gate, out=self.out,
                            scale=d.scale, ws=self.ws, stream=stream)

    def cpu_sample(self, seconds):
        """The oracle over sequence 0 (all heads when it has at most 8192
        positions, else as many heads as 8192*96 position-heads allow)."""
        import oracle
        oracle.set_threads(len(os.sched_getaffinity(0)))
        T = self.lengths[0]
        heads = min(self.H, max(1, 8192 * self.H // T))
        x = _decode_seq_inputs(self.dec, 0, heads)
        el, reps = _repeat(lambda: oracle.mla_decode(**x), seconds)
        nbytes = T * heads * (192 + 128) * 2 * reps
        return _cpu_result(nbytes / el, 1e9, "GB/s",
                           f"sequence 0 of {self.B} ({T} positions) x {heads} of {self.H} "
                           f"heads, {reps} repeats, {el:.1f} s")

    def e2e(self, dev, stream, world, steps):
        """Same metric through the public API with pinned host buffers: every step
        copies the inputs host->device, runs the call and reads the output back."""
        d = self.dec
        host = {n: getattr(d, n).to("cpu").pin_memory()
                for n in ("q", "k", "v", "gate", "cu_seqlens")}
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        dev_in = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
        out_h = torch.empty((self.B, self.H * 128), dtype=torch.bfloat16).pin_memory()
        out_d = torch.empty_like(out_h, device=dev)
        d2h = out_h.numel() * out_h.element_size()

        def one():
            for n in host:
                dev_in[n].copy_(host[n], non_blocking=True)
            self.mla.mla_decode(dev_in["q"], dev_in["k"], dev_in["v"], dev_in["cu_seqlens"],
                                self.max_len, gate=dev_in["gate"], out=out_d, scale=d.scale,
                                stream=stream)
            out_h.copy_(out_d, non_blocking=True)

        return _time_e2e(one, self.work, dev, world, steps, h2d, d2h)

    def free(self):
        del self.dec, self.out, self.ws


class DsaWork:
    """K3.1 Gated DSA decode: indexer score + top-k, then sparse gated MLA (rows a7-a9)."""

    def __init__(self, name, dev, batch=0):
        import mla_family_attention_gb300 as mla
        from mla_family_attention_gb300 import _lib
        self.mla, self.lib = mla, _lib
        w = mi.WORKLOADS[name]
        lengths = mi.workload_lengths(name)
        if batch:
            lengths = lengths[:batch]
        self.name, self.lengths, self.H, self.B = name, lengths, w["H"], len(lengths)
        self.topk = w["topk"]
        self.max_len = max(lengths)
        self.d = mi.make_dsa(lengths, H=self.H, device=dev, config=w["config"])
        self.cu = mi.cu_from_lengths(lengths).to(dev)
        self.idx = torch.empty((self.B, self.topk), dtype=torch.int32, device=dev)
        self.out = torch.empty((self.B, self.H * 128), dtype=torch.bfloat16, device=dev)
        self.ws_i = torch.empty(mla.workspace_size(_lib.OP_INDEX_TOPK, self.B, 0, self.max_len,
                                                   self.topk), dtype=torch.uint8, device=dev)
        self.ws_s = torch.empty(mla.workspace_size(_lib.OP_SPARSE_DECODE, self.B, self.H, 0,
                                                   self.topk), dtype=torch.uint8, device=dev)
        ib = acc.index_key_bytes(lengths)
        sb = acc.sparse_kv_bytes(lengths, self.H, self.topk)
        self.work = ib + sb
        self.unit, self.bound = "GB/s", "hbm"
        self.launches_per_step = 5      # tiles, score, top-k, sparse partial, merge
        self.kernels = [(_lib.OP_INDEX_TOPK, "dsa_score_kernel", ib),
                        (_lib.OP_SPARSE_DECODE, "decode_partial_kernel<sparse>", sb)]

    def step(self, stream):
        d, m = self.d, self.d.main
        self.mla.dsa_index_topk(d.index_q, d.index_k, d.w, self.cu, self.max_len, self.topk,
                                topk_idx=self.idx, ws=self.ws_i, stream=stream)
        self.mla.dsa_sparse_decode(m.q, m.k, m.v, m.cu_seqlens, self.idx, gate=m.gate,
                                   out=self.out, scale=m.scale, ws=self.ws_s, stream=stream)

    def cpu_sample(self, seconds):
        """Sequence 0: the oracle's index scores and top-k over all its
        positions, then its 96-head sparse gated decode.  The rows the
        selection names are gathered into a compact cache before timing (the
        oracle reads only those rows; copying 8 GB of unselected cache to
        the host would time the copy, not the oracle)."""
        import oracle
        oracle.set_threads(len(os.sched_getaffinity(0)))
        d, m, T, H, K = self.d, self.d.main, self.lengths[0], self.H, self.topk
        iq, ik, w = _f64(d.index_q[:1]), _f64(d.index_k[:T]), _f64(d.w[:1])
        cu = np.array([0, T], dtype=np.int64)
        sel = oracle.dsa_topk(oracle.dsa_index_scores(iq, ik, w, cu), cu, K)[0]
        rows = torch.from_numpy(sel[sel >= 0].astype(np.int64)).to(m.k.device)
        n = int(rows.numel())
        ks = m.k[:H * T * 192].view(H, T, 192).index_select(1, rows)
        vs = m.v[:H * T * 128].view(H, T, 128).index_select(1, rows)
        x = dict(q=_f64(m.q[:1]), k=_f64(ks).reshape(-1), v=_f64(vs).reshape(-1),
                 cu_seqlens=np.array([0, n], dtype=np.int64),
                 idx=np.where(np.arange(K) < n, np.arange(K), -1).astype(np.int32)[None],
                 gate=_f64(m.gate[:1]), scale=m.scale)

        def one():
            s64 = oracle.dsa_index_scores(iq, ik, w, cu)
            oracle.dsa_topk(s64, cu, K)
            oracle.dsa_sparse_decode(**x)

        el, reps = _repeat(one, seconds)
        nbytes = (acc.index_key_bytes([T]) + acc.sparse_kv_bytes([T], H, K)) * reps
        return _cpu_result(nbytes / el, 1e9, "GB/s",
                           f"sequence 0 of {self.B} ({T} positions): index scores, top-{K}, "
                           f"{H}-head sparse decode; {reps} repeats, {el:.1f} s")

    def free(self):
        del self.d, self.idx, self.out, self.ws_i, self.ws_s


class GatherProbeWork:
    """Reference rate for the sparse decode: the same rows of the same cache
    (selected once by the GPU indexer, outside the timed region), gathered
    with plain 16-byte loads and no arithmetic (mla_gather_probe)."""

    def __init__(self, name, dev, batch=0):
        import mla_family_attention_gb300 as mla
        from mla_family_attention_gb300 import _lib
        self.mla, self.lib = mla, _lib
        w = mi.WORKLOADS[name]
        lengths = mi.workload_lengths(name)
        if batch:
            lengths = lengths[:batch]
        self.name, self.lengths, self.H, self.B = name, lengths, w["H"], len(lengths)
        self.topk = w["topk"]
        self.d = mi.make_dsa(lengths, H=self.H, device=dev, config=w["config"])
        cu = mi.cu_from_lengths(lengths).to(dev)
        self.idx = mla.dsa_index_topk(self.d.index_q, self.d.index_k, self.d.w, cu,
                                      max(lengths), self.topk)
        mla.check_device_status()
        self.sink = torch.empty(_lib.load().mla_gather_probe_blocks(), dtype=torch.int32,
                                device=dev)
        self.work = acc.sparse_kv_bytes(lengths, self.H, self.topk)
        self.unit, self.bound = "GB/s", "hbm"
        self.launches_per_step = 1
        self.kernels = [(_lib.OP_GATHER_PROBE, "gather_probe_kernel", self.work)]

    def step(self, stream):
        m = self.d.main
        self.mla.gather_probe(m.k, m.v, m.cu_seqlens, self.idx, self.H, sink=self.sink,
                              stream=stream)

    def free(self):
        del self.d, self.idx, self.sink


class IndexWork:
    """The DSA indexer alone: scores and top-k (rows a7-a8)."""

    def __init__(self, name, dev, batch=0):
        import mla_family_attention_gb300 as mla
        from mla_family_attention_gb300 import _lib
        self.mla, self.lib = mla, _lib
        w = mi.WORKLOADS[name]
        lengths = mi.workload_lengths(name)
        if batch:
            lengths = lengths[:batch]
        self.name, self.lengths, self.H, self.B = name, lengths, w["H"], len(lengths)
        self.topk = w["topk"]
        self.max_len = max(lengths)
        self.d = mi.make_dsa(lengths, H=self.H, device=dev, config=w["config"], with_main=False)
        self.cu = mi.cu_from_lengths(lengths).to(dev)
        self.idx = torch.empty((self.B, self.topk), dtype=torch.int32, device=dev)
        self.ws_i = torch.empty(mla.workspace_size(_lib.OP_INDEX_TOPK, self.B, 0, self.max_len,
                                                   self.topk), dtype=torch.uint8, device=dev)
        self.work = acc.index_key_bytes(lengths)
        self.unit, self.bound = "GB/s", "hbm"
        self.launches_per_step = 3      # tiles, score, top-k
        self.kernels = [(_lib.OP_INDEX_TOPK, "dsa_score_kernel", self.work)]

    def step(self, stream):
        d = self.d
        self.mla.dsa_index_topk(d.index_q, d.index_k, d.w, self.cu, self.max_len, self.topk,
                                topk_idx=self.idx, ws=self.ws_i, stream=stream)

    def cpu_sample(self, seconds):
        """The oracle's index scores and top-k over sequence 0."""
        import oracle
        oracle.set_threads(len(os.sched_getaffinity(0)))
        T = self.lengths[0]
        iq, ik, w = _f64(self.d.index_q[:1]), _f64(self.d.index_k[:T]), _f64(self.d.w[:1])
        cu = np.array([0, T], dtype=np.int64)
        el, reps = _repeat(lambda: oracle.dsa_topk(oracle.dsa_index_scores(iq, ik, w, cu), cu,
                                                   self.topk), seconds)
        return _cpu_result(acc.index_key_bytes([T]) * reps / el, 1e9, "GB/s",
                           f"sequence 0 of {self.B} ({T} positions), {reps} repeats, "
                           f"{el:.1f} s")

    def free(self):
        del self.d, self.idx, self.ws_i


class IndexFp8Work(IndexWork):
    """The DSA indexer over FP8 index keys (132 B per position)."""

    def __init__(self, name, dev, batch=0):
        super().__init__(name, dev, batch)
        mla, _lib = self.mla, self.lib
        self.k8, self.ks = mla.dsa_quantize_index_keys(self.d.index_k)
        self.ws_i = torch.empty(mla.workspace_size(_lib.OP_INDEX_TOPK_FP8, self.B, 0,
                                                   self.max_len, self.topk),
                                dtype=torch.uint8, device=dev)
        self.work = acc.index_key_bytes_fp8(self.lengths)
        self.launches_per_step = 4      # query quantisation, tiles, score, top-k
        self.kernels = [(_lib.OP_INDEX_TOPK_FP8, "dsa_score_kernel<fp8>", self.work)]

    def step(self, stream):
        d = self.d
        self.mla.dsa_index_topk_fp8(d.index_q, self.k8, self.ks, d.w, self.cu, self.max_len,
                                    self.topk, topk_idx=self.idx, ws=self.ws_i, stream=stream)

    def cpu_sample(self, seconds):
        """The oracle's FP8 index scores (query quantisation included) and
        top-k over sequence 0."""
        import oracle
        oracle.set_threads(len(os.sched_getaffinity(0)))
        T = self.lengths[0]
        iq, w = self.d.index_q[:1].cpu(), _f64(self.d.w[:1])
        k8, ks = self.k8[:T].cpu(), self.ks[:T].cpu()
        cu = np.array([0, T], dtype=np.int64)
        el, reps = _repeat(lambda: oracle.dsa_topk(
            oracle.dsa_index_scores_fp8(iq, k8, ks, w, cu), cu, self.topk), seconds)
        return _cpu_result(acc.index_key_bytes_fp8([T]) * reps / el, 1e9, "GB/s",
                           f"sequence 0 of {self.B} ({T} positions), {reps} repeats, "
                           f"{el:.1f} s")

    def free(self):
        del self.k8, self.ks
        super().free()


class PrefillWork:
    """Causal gated MLA prefill (rows a1-a4, a6 on the tensor cores)."""

    def __init__(self, name, dev, batch=0):
        import mla_family_attention_gb300 as mla
        from mla_family_attention_gb300 import _lib
        self.mla, self.lib = mla, _lib
        w = mi.WORKLOADS[name]
        self.name, self.H, self.B, self.T = name, w["H"], w["B"], w["T"]
        self.lengths = [w["T"]] * w["B"]
        self.pf = mi.make_prefill(w["B"], w["H"], w["T"], w["T"], w["gated"], device=dev,
                                  config=w["config"])
        self.out = torch.empty((w["B"], w["T"], w["H"] * 128), dtype=torch.bfloat16, device=dev)
        self.work = acc.prefill_flops(w["B"], w["H"], w["T"], w["T"])
        self.unit, self.bound, self.scale_unit = "TFLOP/s", "tensor", 1e12
        self.launches_per_step = 1
        self.kernels = [(_lib.OP_PREFILL, "mla_prefill_kernel", self.work)]
        in_bytes = sum(t.numel() * t.element_size() for t in
                       (self.pf.q, self.pf.k, self.pf.v) + ((self.pf.gate,) if w["gated"] else ()))
        self.rotating = 0
        self.sets = [(self.pf.q, self.pf.k, self.pf.v, self.pf.gate, self.out)]
        self.i = 0
        if in_bytes < 4 * (129 << 20):
            # a short prompt's 0.5 GFLOP take microseconds: its kernel is read
            # against the I/O floor (inputs read once, outputs written once)
            # at the HBM peak, not against the tensor peak
            io = in_bytes + self.out.numel() * self.out.element_size()
            self.bound = "hbm"
            self.kernels = [(_lib.OP_PREFILL, "mla_prefill_kernel<short>", io, "hbm")]
            # inputs that fit in L2: N copies, together over 4x L2, read in
            # turn, so no step finds its inputs in L2 (one output buffer)
            self.rotating = -(-4 * (129 << 20) // io)
            for _ in range(self.rotating - 1):
                pf = self.pf
                self.sets.append((pf.q.clone(), pf.k.clone(), pf.v.clone(),
                                  None if pf.gate is None else pf.gate.clone(), self.out))

    def step(self, stream):
        q, k, v, g, out = self.sets[self.i % len(self.sets)]
        self.i += 1
        self.mla.mla_prefill(q, k, v, g, out=out, scale=self.pf.scale, stream=stream)

    def cpu_sample(self, seconds):
        """The oracle over the whole prompt when it is short (T <= 1024);
        otherwise over head 0 and the prompt's last 128 query rows, each of
        which sees ~T keys (the rate of that sample stands for the whole)."""
        import oracle
        oracle.set_threads(len(os.sched_getaffinity(0)))
        pf, T = self.pf, self.T
        if T <= 1024:
            x = (_f64(pf.q), _f64(pf.k), _f64(pf.v), None if pf.gate is None else _f64(pf.gate))
            flops, what, ext = self.work, f"the whole prompt ({self.H} heads x {T} rows)", False
        else:
            R = 128
            x = (_f64(pf.q[:, :1, T - R:]), _f64(pf.k[:, :1]), _f64(pf.v[:, :1]),
                 None if pf.gate is None else _f64(pf.gate[:, T - R:, :128]))
            flops, ext = acc.prefill_flops(1, 1, R, T), True
            what = f"head 0 of {self.H}, query rows {T - R}..{T - 1} of {T}"
        el, reps = _repeat(lambda: oracle.mla_prefill(*x, pf.scale), seconds)
        return _cpu_result(flops * reps / el, 1e12, "TFLOP/s",
                           f"{what}, {reps} repeats, {el:.1f} s", ext)

    def free(self):
        del self.pf, self.out, self.sets


class ChunkedPrefillWork:
    """A prompt fed through mla_prefill_chunk in equal chunks (the cache-update
    path): per chunk, an in-place append of its keys and values into a
    fixed-capacity cache, then causal gated prefill over the cache."""

    def __init__(self, name, dev, batch=0):
        import mla_family_attention_gb300 as mla
        from mla_family_attention_gb300 import _lib
        self.mla, self.lib = mla, _lib
        w = mi.WORKLOADS[name]
        B, H, T, c = w["B"], w["H"], w["T"], w["chunk"]
        self.name, self.H, self.B, self.T, self.c = name, H, B, T, c
        self.lengths = [T] * B
        pf = mi.make_prefill(B, H, T, T, w["gated"], device=dev, config=w["config"])
        n = T // c
        sl = [slice(i * c, (i + 1) * c) for i in range(n)]
        self.q = [pf.q[:, :, s].contiguous() for s in sl]
        self.kn = [pf.k[:, :, s].contiguous() for s in sl]
        self.vn = [pf.v[:, :, s].contiguous() for s in sl]
        self.g = [pf.gate[:, s].contiguous() if w["gated"] else None for s in sl]
        self.scale = pf.scale
        del pf
        self.kc = mi.nan_filled((B, H, T, 192), dev)
        self.vc = mi.nan_filled((B, H, T, 128), dev)
        self.out = [torch.empty((B, c, H * 128), dtype=torch.bfloat16, device=dev)
                    for _ in range(n)]
        self.work = sum(acc.prefill_flops(B, H, c, (i + 1) * c) for i in range(n))
        assert self.work == acc.prefill_flops(B, H, T, T)
        self.unit, self.bound, self.scale_unit = "TFLOP/s", "tensor", 1e12
        self.launches_per_step = 2 * n
        self.kernels = [(_lib.OP_PREFILL, "mla_prefill_kernel", self.work // n),
                        (_lib.OP_CACHE_APPEND, "cache_append_kernel",
                         acc.append_bytes(B, H, c), "hbm")]

    def step(self, stream):
        for i in range(len(self.q)):
            self.mla.mla_prefill_chunk(self.q[i], self.kn[i], self.vn[i], self.kc, self.vc,
                                       i * self.c, gate=self.g[i], out=self.out[i],
                                       scale=self.scale, stream=stream)

    def cpu_sample(self, seconds):
        """The oracle's chunked prefill of the last chunk's last 128 query
        rows, head 0, over the cache the earlier chunks filled (the rate of
        that sample stands for the whole prompt)."""
        import oracle
        oracle.set_threads(len(os.sched_getaffinity(0)))
        R, n = 128, len(self.q)
        P = (n - 1) * self.c
        kc = _f64(torch.cat([k[:, :1] for k in self.kn[:-1]], 2))
        vc = _f64(torch.cat([v[:, :1] for v in self.vn[:-1]], 2))
        q = _f64(self.q[-1][:, :1, self.c - R:])
        kn, vn = _f64(self.kn[-1][:, :1]), _f64(self.vn[-1][:, :1])
        g = None if self.g[-1] is None else _f64(self.g[-1][:, self.c - R:, :128])
        el, reps = _repeat(lambda: oracle.mla_prefill_chunk(q, kc, vc, kn, vn, P, g, self.scale),
                           seconds)
        return _cpu_result(acc.prefill_flops(1, 1, R, self.T) * reps / el, 1e12, "TFLOP/s",
                           f"head 0 of {self.H}, last {R} rows of chunk {n - 1} (cache of "
                           f"{P} positions), {reps} repeats, {el:.1f} s", True)

    def free(self):
        del self.q, self.kn, self.vn, self.g, self.kc, self.vc, self.out


class DecodeCachedWork:
    """A decode step over fixed-capacity caches: the current token appended
    at position T-1 of every sequence, then split-KV gated decode over T."""

    def __init__(self, name, dev, batch=0):
        import mla_family_attention_gb300 as mla
        from mla_family_attention_gb300 import _lib
        self.mla, self.lib = mla, _lib
        w = mi.WORKLOADS[name]
        B = batch or w["B"]
        H, T = w["H"], w["T"]
        self.name, self.H, self.B, self.T = name, H, B, T
        self.lengths = [T] * B
        self.cd = mi.make_capacity_decode([T - 1] * B, H, T, w["gated"], device=dev,
                                          config=w["config"])
        self.seqlens = torch.full((B,), T - 1, dtype=torch.int64, device=dev)
        self.out = torch.empty((B, H * 128), dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(mla.workspace_size(_lib.OP_DECODE, B, H, T, 0), dtype=torch.uint8,
                              device=dev)
        self.work = acc.decode_kv_bytes(self.lengths, H)
        self.unit, self.bound = "GB/s", "hbm"
        self.launches_per_step = 4      # append, item prefix, partial, merge
        self.kernels = [(_lib.OP_DECODE, "decode_partial_kernel", self.work),
                        (_lib.OP_CACHE_APPEND, "cache_append_kernel", acc.append_bytes(B, H, 1))]

    def step(self, stream):
        cd = self.cd
        self.mla.mla_decode_cached(cd.q, cd.k_cache, cd.v_cache, self.seqlens, self.T,
                                   k_new=cd.k_new, v_new=cd.v_new, gate=cd.gate, out=self.out,
                                   scale=cd.scale, ws=self.ws, stream=stream)

    def cpu_sample(self, seconds):
        """The oracle's decode step (current token appended) for sequence 0,
        all heads."""
        import oracle
        oracle.set_threads(len(os.sched_getaffinity(0)))
        cd, L = self.cd, self.T - 1
        x = (_f64(cd.q[:1]), _f64(cd.k_cache[:1, :, :L]), _f64(cd.v_cache[:1, :, :L]), [L],
             _f64(cd.k_new[:1]), _f64(cd.v_new[:1]), _f64(cd.gate[:1]), cd.scale)
        el, reps = _repeat(lambda: oracle.mla_decode_cached(*x), seconds)
        return _cpu_result(acc.decode_kv_bytes([self.T], self.H) * reps / el, 1e9, "GB/s",
                           f"sequence 0 of {self.B} ({self.T} positions) x {self.H} heads, "
                           f"{reps} repeats, {el:.1f} s")

    def free(self):
        del self.cd, self.seqlens, self.out, self.ws


class LatentDecodeWork:
    """Gated MLA decode over the absorbed 576-feature latent cache: query
    absorption, tcgen05 attention over the latent, merge with W^V and gate."""

    def __init__(self, name, dev, batch=0):
        import mla_family_attention_gb300 as mla
        from mla_family_attention_gb300 import _lib
        self.mla, self.lib = mla, _lib
        w = mi.WORKLOADS[name]
        lengths = mi.workload_lengths(name)
        if batch:
            lengths = lengths[:batch]
        self.name, self.lengths, self.H, self.B = name, lengths, w["H"], len(lengths)
        self.max_len = max(lengths)
        self.d = mi.make_latent_decode(lengths, self.H, w["gated"], device=dev,
                                       config=w["config"])
        self.out = torch.empty((self.B, self.H * 128), dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(mla.workspace_size(_lib.OP_LATENT_DECODE, self.B, self.H,
                                                 self.max_len, 0), dtype=torch.uint8, device=dev)
        self.work = acc.latent_kv_bytes(lengths)
        self.unit, self.bound = "GB/s", "hbm"
        self.launches_per_step = 5      # absorb, schedule, latent attention, fixup, W^V output
        self.kernels = [(_lib.OP_LATENT_DECODE, "mla_latent_kernel", self.work)]

    def step(self, stream):
        d = self.d
        self.mla.mla_decode_latent(d.q, d.ckv, d.cu_seqlens, self.max_len, d.w_kc, d.w_vc,
                                   gate=d.gate, out=self.out, scale=d.scale, ws=self.ws,
                                   stream=stream)

    CPU_HEADS = 8

    def _cpu_cache(self, T):
        return _f64(self.d.ckv[:T])

    def _cpu_call(self, oracle, q, cache, cu, wk, wv, g):
        return oracle.mla_decode_latent(q, cache, cu, wk, wv, g, self.d.scale)

    def _cpu_bytes(self, T):
        return acc.latent_kv_bytes([T])

    def cpu_sample(self, seconds):
        """The oracle over sequence 0 with 8 of the 96 heads.  The cache bytes
        are shared by all heads while the oracle's work grows with them, so
        the time is scaled by 96/8 (extrapolated)."""
        import oracle
        oracle.set_threads(len(os.sched_getaffinity(0)))
        d, T, hs = self.d, self.lengths[0], self.CPU_HEADS
        q, g = _f64(d.q[:1, :hs]), _f64(d.gate[:1, :hs * 128])
        wk, wv = _f64(d.w_kc[:hs]), _f64(d.w_vc[:hs])
        cache, cu = self._cpu_cache(T), np.array([0, T], dtype=np.int64)
        el, reps = _repeat(lambda: self._cpu_call(oracle, q, cache, cu, wk, wv, g), seconds)
        full = el / reps * self.H / hs
        return _cpu_result(self._cpu_bytes(T) / full, 1e9, "GB/s",
                           f"sequence 0 of {self.B} ({T} positions) x {hs} of {self.H} heads, "
                           f"{reps} repeats, {el:.1f} s, time scaled by {self.H}/{hs}", True)

    def free(self):
        del self.d, self.out, self.ws


class LatentDecodeFp8Work(LatentDecodeWork):
    """The latent decode over 656-byte FP8 records of the same cache."""

    def __init__(self, name, dev, batch=0):
        super().__init__(name, dev, batch)
        self.rec = self.mla.mla_quantize_latent_cache(self.d.ckv)
        self.work = acc.latent_kv_bytes_fp8(self.lengths)
        self.kernels = [(self.lib.OP_LATENT_DECODE, "mla_latent_kernel<fp8>", self.work)]

    def step(self, stream):
        d = self.d
        self.mla.mla_decode_latent_fp8(d.q, self.rec, d.cu_seqlens, self.max_len, d.w_kc, d.w_vc,
                                       gate=d.gate, out=self.out, scale=d.scale, ws=self.ws,
                                       stream=stream)

    def _cpu_cache(self, T):
        return self.rec[:T].cpu()

    def _cpu_call(self, oracle, q, cache, cu, wk, wv, g):
        return oracle.mla_decode_latent_fp8(q, cache, cu, wk, wv, g, self.d.scale)

    def _cpu_bytes(self, T):
        return acc.latent_kv_bytes_fp8([T])

    def free(self):
        del self.rec
        super().free()


class DsaPrefillWork:
    """K3.1 Gated DSA prefill of one prompt: every token's index scores and
    top-k, then every token's gated MLA over its own selection of the latent
    cache (rows f2 and f3 of the scope)."""

    def __init__(self, name, dev, batch=0):
        import mla_family_attention_gb300 as mla
        from mla_family_attention_gb300 import _lib
        self.mla, self.lib = mla, _lib
        w = mi.WORKLOADS[name]
        T, H, K = w["T"], w["H"], w["topk"]
        self.name, self.H, self.B, self.T, self.K = name, H, 1, T, K
        self.lengths = [T]
        self.d = mi.make_dsa_prefill(T, T, H, w["gated"], device=dev, config=w["config"])
        self.idx = torch.empty((T, K), dtype=torch.int32, device=dev)
        self.out = torch.empty((T, H * 128), dtype=torch.bfloat16, device=dev)
        self.ws_i = torch.empty(mla.workspace_size(_lib.OP_PREFILL_INDEX_TOPK, T, 0, T, K),
                                dtype=torch.uint8, device=dev)
        self.ws_a = torch.empty(mla.workspace_size(_lib.OP_SPARSE_PREFILL_LATENT, T, H, T, K),
                                dtype=torch.uint8, device=dev)
        fi = acc.dsa_prefill_index_flops(T, T)
        fa = acc.sparse_latent_attention_flops(T, T, H, K)
        self.work = fi + fa
        self.unit, self.bound, self.scale_unit = "TFLOP/s", "tensor", 1e12
        self.launches_per_step = 7      # score, top-k, absorb, schedule, attention, fixup, out
        # the attention kernel is read against its own flops (the absorption
        # and W^V projection run in the absorb and out kernels)
        self.kernels = [(_lib.OP_LATENT_DECODE, "mla_latent_kernel<gather>",
                         acc.sparse_latent_core_flops(T, T, H, K)),
                        (_lib.OP_PREFILL_INDEX_TOPK, "dsa_prefill_score_kernel", fi)]

    def step(self, stream):
        d = self.d
        self.mla.dsa_prefill_index_topk(d.index_q, d.index_k, d.w, self.K, topk_idx=self.idx,
                                        ws=self.ws_i, stream=stream)
        self.mla.mla_sparse_prefill_latent(d.q, d.ckv, self.idx, d.w_kc, d.w_vc, gate=d.gate,
                                           out=self.out, scale=d.scale, ws=self.ws_a,
                                           stream=stream)

    def cpu_sample(self, seconds):
        """The prompt's last token: the oracle's index scores over its
        T visible positions and its top-k (timed), then its gated MLA over its
        selection with 4 of the 96 heads (timed, scaled by 96/4); flops are the
        token's index flops plus its all-head attention flops (extrapolated)."""
        import oracle
        oracle.set_threads(len(os.sched_getaffinity(0)))
        d, T, K, H, hs = self.d, self.T, self.K, self.H, 4
        i = T - 1
        iq, ik, w = d.index_q[i:i + 1].cpu(), d.index_k.cpu(), d.w[i:i + 1].cpu()
        half = seconds / 2

        def index():
            return oracle.dsa_prefill_topk(oracle.dsa_prefill_index_scores(iq, ik, w), K)

        sel = index()
        el_i, reps_i = _repeat(index, half)
        q, g = _f64(d.q[i:i + 1, :hs]), _f64(d.gate[i:i + 1, :hs * 128])
        ckv, wk, wv = _f64(d.ckv), _f64(d.w_kc[:hs]), _f64(d.w_vc[:hs])
        el_a, reps_a = _repeat(lambda: oracle.dsa_prefill_latent(q, ckv, wk, wv, sel, g, d.scale),
                               half)
        t = el_i / reps_i + el_a / reps_a * H / hs
        flops = (acc.dsa_prefill_index_flops(1, T) +
                 acc.sparse_latent_attention_flops(1, T, H, K))
        return _cpu_result(flops / t, 1e12, "TFLOP/s",
                           f"token {i} of {T}: index + top-{K} ({reps_i} repeats, {el_i:.1f} s), "
                           f"MLA over its selection with {hs} of {H} heads ({reps_a} repeats, "
                           f"{el_a:.1f} s, time scaled by {H}/{hs})", True)

    def free(self):
        del self.d, self.idx, self.out, self.ws_i, self.ws_a


WORK_KINDS = {"decode": DecodeWork, "latent_decode": LatentDecodeWork,
              "dsa_prefill": DsaPrefillWork, "index_fp8": IndexFp8Work,
              "latent_decode_fp8": LatentDecodeFp8Work, "dsa": DsaWork, "index": IndexWork,
              "prefill": PrefillWork, "chunked_prefill": ChunkedPrefillWork,
              "decode_cached": DecodeCachedWork, "gather_probe": GatherProbeWork}


def _time_e2e(one, work, dev, world, steps, h2d, d2h):
    one()
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize(dev)
    el = max_over_ranks((time.perf_counter() - t0) / steps, world)
    barrier(world)
    return {"value": round(work * world / el / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps}


L2_FLUSH_BYTES = 512 << 20   # four times the 129 MB L2
E2E_HOST_LIMIT = 24 << 30    # pinned host copies of the inputs for the end-to-end leg


def time_work(work, steps, warmup, dev, stream, world, sampler=None):
    """CUDA-event time of `steps` steps (after `warmup`), then each dominant
    kernel's own event time over a second run of `steps` steps.  The step
    time is taken with the library's per-kernel events off (an event recorded
    between two kernels keeps the later one from being placed on the SMs
    while the earlier one finishes).  Workloads whose inputs fit in L2
    (work.flush_l2) are timed step by step with a 512 MB write between
    steps, outside the timed events.  Workloads that rotate through copies
    of their inputs (work.rotating: calls of a few microseconds) capture one
    pass over the copies as a CUDA graph and replay it, so the host's
    per-call work does not pace the GPU; the step time is then the graph's
    time over the calls it holds."""
    mla = work.mla
    for _ in range(warmup):
        work.step(stream)
    mla.check_device_status(stream)
    torch.cuda.synchronize(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) \
        if getattr(work, "flush_l2", False) else None
    graph, n_graph = None, 0
    if getattr(work, "rotating", 0):
        n_graph = len(work.sets)
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
            cs = torch.cuda.current_stream(dev)
            for _ in range(n_graph):
                work.step(cs)
        torch.cuda.synchronize(dev)
        graph.replay()
        torch.cuda.synchronize(dev)
        mla.check_device_status(stream)
    reps = max(1, -(-steps // n_graph)) if graph is not None else 0
    use_graph = [graph is not None]

    def region(evs):
        barrier(world)
        torch.cuda.synchronize(dev)
        if use_graph[0]:
            evs[0][0].record(stream)
            for _ in range(reps):
                graph.replay()
            evs[0][1].record(stream)
        elif flush is None:
            evs[0][0].record(stream)
            for _ in range(steps):
                work.step(stream)
            evs[0][1].record(stream)
        else:
            for i in range(steps):
                flush.fill_(i & 0xFF)
                evs[i][0].record(stream)
                work.step(stream)
                evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)

    def events():
        return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(steps if flush is not None else 1)]

    ev = events()
    if sampler:
        sampler.mark_start()
    region(ev)
    if sampler:
        sampler.mark_end()
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev) /
                        (reps * n_graph if use_graph[0] else steps), world)
    if use_graph[0] and work.launches_per_step == 1:
        # one kernel per call: the graph's time per call is that kernel's
        # time (events between the calls would keep the next launch from
        # starting during the previous one's tail, and the host would pace it)
        work.kernel_time_source = "CUDA-graph replay, one kernel per call"
        kd = work.kernels[0]
        return ms, [(kd[1], ms, kd[2], kd[3] if len(kd) > 3 else work.bound)]
    use_graph[0] = False             # the library's per-kernel events: call by call
    mla.timing_enable(True)
    for kd in work.kernels:
        mla.timing_read(kd[0])
    region(events())
    mla.timing_enable(False)
    del flush
    kern = []
    for kd in work.kernels:
        op, kname, units = kd[:3]
        k_ms, n = mla.timing_read(op)
        kern.append((kname, max_over_ranks(k_ms / max(n, 1), world), units,
                     kd[3] if len(kd) > 3 else work.bound))
    mla.check_device_status(stream)
    return ms, kern


def flush_latency(work, dev, stream, calls=20):
    """Median CUDA-event time of one call right after a 512 MB write that
    evicts L2 (the single-call latency of a workload whose inputs fit in L2;
    it includes the launch and the write-back the flush leaves behind)."""
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ts = []
    for i in range(calls):
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        work.step(stream)
        b.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(a.elapsed_time(b))
    work.mla.check_device_status(stream)
    del flush
    return round(float(np.median(ts)), 4)


def _scale(work):
    return getattr(work, "scale_unit", 1e9)


def roofline(work, kern):
    """Roofline object for the dominant (longest) kernel of a step."""
    peak, unit, peak_kind = peaks(work.bound)
    sc = 1e12 if work.bound == "tensor" else 1e9
    kname, k_ms, units, _ = max((k for k in kern if k[3] == work.bound), key=lambda x: x[1])
    achieved = units / (k_ms * 1e-3) / sc
    nominal = 2250.0 if work.bound == "tensor" else 7900.0
    per = "flops" if work.bound == "tensor" else "bytes"
    r = {"bound": work.bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
         "frac": round(achieved / peak, 4), "peak_source": peak_kind,
         f"frac_of_nominal_{int(nominal)}": round(achieved / nominal, 4), "kernel": kname,
         "kernel_ms": round(k_ms, 4), "traffic": traffic_for(kname, units),
         f"algorithmic_{per}_per_launch": units}
    if getattr(work, "kernel_time_source", None):
        r["kernel_time_source"] = work.kernel_time_source
    others = {}
    for kn, km, ku, kb in kern:
        if kn != kname:
            pk, pu, _ = peaks(kb)
            a = ku / (km * 1e-3) / (1e12 if kb == "tensor" else 1e9)
            others[kn] = {"bound": kb, "achieved": round(a, 2), "unit": pu,
                          "frac": round(a / pk, 4), "kernel_ms": round(km, 4),
                          f"algorithmic_{'flops' if kb == 'tensor' else 'bytes'}_per_launch": ku}
    if others:
        r["other_kernels"] = others
    return r


ALSO_FIELDS = ["value", "unit", "ms_per_step", "roofline.frac", "roofline.kernel_ms",
               "cpu_baseline.value", "latency_after_l2_flush_ms"]


def _sig(x, digits=4):
    return None if x is None else float(f"{x:.{digits}g}")


def _compact(entry):
    """The figures of one workload that the one-line summary keeps, in the
    order of ALSO_FIELDS: value, step time, the dominant kernel's roofline
    fraction and time, and the oracle's rate in the same unit."""
    r = entry["roofline"]
    c = entry.get("cpu_baseline") or {}
    return [entry["value"], entry["unit"], entry["ms_per_step"], r["frac"], r["kernel_ms"],
            _sig(c.get("value")), entry.get("latency_after_l2_flush_ms")]


def run_ours(args, world, rank, local):
    """Time the headline workload (full detail in the JSON line), then every
    other workload of the hot path (compact figures in the line's `also`;
    the full per-workload records go to stderr, one JSON object per line)."""
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    name = args.workload
    kind = mi.WORKLOADS[name]["kind"]
    work = WORK_KINDS[kind](name, dev, args.batch)
    sampler = ClockSampler(local)
    ms, kern = time_work(work, args.steps, args.warmup, dev, stream, world, sampler)
    clocks = sampler.finish()
    value = work.work * world / (ms * 1e-3) / _scale(work)
    roof = roofline(work, kern)
    others = roof.pop("other_kernels", None)
    line = {"metric": METRIC, "value": round(value, 2), "unit": work.unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": workload_config(name, work.B), "roofline": roof,
            "gpu_launches": work.launches_per_step * args.steps * world, "clocks": clocks}
    if getattr(work, "rotating", 0):
        line["rotating_input_copies"] = work.rotating
        line["latency_after_l2_flush_ms"] = flush_latency(work, dev, stream)
    if hasattr(work, "e2e"):
        in_bytes = sum(getattr(work.dec, n).numel() * getattr(work.dec, n).element_size()
                       for n in ("q", "k", "v", "gate"))
        if in_bytes <= E2E_HOST_LIMIT:
            line["e2e"] = work.e2e(dev, stream, world, max(3, min(args.steps, args.e2e_steps)))
        else:
            line["e2e"] = {"value": None, "unit": work.unit,
                           "skipped": f"inputs of {in_bytes / 1e9:.0f} GB exceed the "
                                      f"{E2E_HOST_LIMIT / 1e9:.0f} GB pinned host budget"}
    cpu_ok = rank == 0 and world == 1 and not args.no_cpu_baseline
    if cpu_ok and hasattr(work, "cpu_sample"):
        line["cpu_baseline"] = work.cpu_sample(args.cpu_seconds)
    if rank == 0 and others:
        print(json.dumps({"workload": name, "other_kernels": others}), file=sys.stderr,
              flush=True)
    work.free()
    del work
    torch.cuda.empty_cache()
    # the other workloads of the hot path, timed the same way (shorter)
    if not args.only and not args.batch:
        also = {"fields": ALSO_FIELDS}
        for other, w in mi.WORKLOADS.items():
            if other == name or w["kind"] not in WORK_KINDS or w.get("profile_only"):
                continue
            wk = WORK_KINDS[w["kind"]](other, dev)
            k_steps = max(3, min(args.steps, 20))
            ms_o, kern_o = time_work(wk, k_steps, 3, dev, stream, world)
            entry = {"value": round(wk.work * world / (ms_o * 1e-3) / _scale(wk), 2),
                     "unit": wk.unit, "ms_per_step": round(ms_o, 4), "steps": k_steps,
                     "roofline": roofline(wk, kern_o)}
            if getattr(wk, "rotating", 0):
                entry["rotating_input_copies"] = wk.rotating
                entry["latency_after_l2_flush_ms"] = flush_latency(wk, dev, stream)
            if cpu_ok and hasattr(wk, "cpu_sample"):
                entry["cpu_baseline"] = wk.cpu_sample(args.also_cpu_seconds)
            line["gpu_launches"] += wk.launches_per_step * (2 * k_steps + 3) * world
            also[other] = _compact(entry)
            if rank == 0:
                print(json.dumps({"workload": other, **entry}), file=sys.stderr, flush=True)
            wk.free()
            del wk
            torch.cuda.empty_cache()
        line["also"] = also
    if rank == 0:
        print(json.dumps(line, separators=(",", ":")), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=list(mi.WORKLOADS))
    ap.add_argument("--only", action="store_true",
                    help="time only --workload (skip the other workloads' short runs)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="oracle time for the headline workload's cpu_baseline")
    ap.add_argument("--also-cpu-seconds", type=float, default=3.0,
                    help="oracle time for each other workload's cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="use only the first N sequences (small profiling case)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
