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


def oracle_decode_sample(dec, n_seq: int, min_seconds: float):
    """Time the fp64 oracle over the first n_seq sequences (all heads), repeated
    until min_seconds of CPU work; returns (GB/s, seconds, threads, repeats, n_seq)."""
    import oracle
    threads = oracle.set_threads(len(os.sched_getaffinity(0)))
    x = oracle_inputs(dec, n_seq)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.mla_decode(**x)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    nbytes = acc.decode_kv_bytes(dec.lengths[:n_seq], dec.H) * reps
    return nbytes / el / 1e9, el, threads, reps, n_seq


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
    cfg["l2"] = ("inputs smaller than L2: a 512 MB buffer is written between timed steps"
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
        gbs, el, threads, reps, n_seq = oracle_decode_sample(self.dec, 1, seconds)
        return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                "sample": f"{n_seq} of {self.B} sequences x {self.H} heads x "
                          f"{self.lengths[0]} positions, {reps} repeats, {el:.1f} s"}

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

    def free(self):
        del self.d, self.idx, self.out, self.ws_i, self.ws_s


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
        self.flush_l2 = in_bytes < 4 * (129 << 20)

    def step(self, stream):
        pf = self.pf
        self.mla.mla_prefill(pf.q, pf.k, pf.v, pf.gate, out=self.out, scale=pf.scale,
                             stream=stream)

    def free(self):
        del self.pf, self.out


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
        self.kernels = [(_lib.OP_LATENT_DECODE, "mla_latent_kernel<gather>", fa),
                        (_lib.OP_PREFILL_INDEX_TOPK, "dsa_prefill_score_kernel", fi)]

    def step(self, stream):
        d = self.d
        self.mla.dsa_prefill_index_topk(d.index_q, d.index_k, d.w, self.K, topk_idx=self.idx,
                                        ws=self.ws_i, stream=stream)
        self.mla.mla_sparse_prefill_latent(d.q, d.ckv, self.idx, d.w_kc, d.w_vc, gate=d.gate,
                                           out=self.out, scale=d.scale, ws=self.ws_a,
                                           stream=stream)

    def free(self):
        del self.d, self.idx, self.out, self.ws_i, self.ws_a


WORK_KINDS = {"decode": DecodeWork, "latent_decode": LatentDecodeWork,
              "dsa_prefill": DsaPrefillWork, "index_fp8": IndexFp8Work,
              "latent_decode_fp8": LatentDecodeFp8Work, "dsa": DsaWork, "index": IndexWork,
              "prefill": PrefillWork, "chunked_prefill": ChunkedPrefillWork,
              "decode_cached": DecodeCachedWork}


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
    steps, outside the timed events."""
    mla = work.mla
    for _ in range(warmup):
        work.step(stream)
    mla.check_device_status(stream)
    torch.cuda.synchronize(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) \
        if getattr(work, "flush_l2", False) else None

    def region(evs):
        barrier(world)
        torch.cuda.synchronize(dev)
        if flush is None:
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
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev) / steps, world)
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


def _scale(work):
    return getattr(work, "scale_unit", 1e9)


def roofline(work, kern):
    """Roofline object for the dominant (longest) kernel of a step."""
    peak, unit, peak_kind = peaks(work.bound)
    sc = _scale(work)
    kname, k_ms, units, _ = max((k for k in kern if k[3] == work.bound), key=lambda x: x[1])
    achieved = units / (k_ms * 1e-3) / sc
    nominal = 2250.0 if work.bound == "tensor" else 7900.0
    per = "flops" if work.bound == "tensor" else "bytes"
    r = {"bound": work.bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
         "frac": round(achieved / peak, 4), "peak_source": peak_kind,
         f"frac_of_nominal_{int(nominal)}": round(achieved / nominal, 4), "kernel": kname,
         "kernel_ms": round(k_ms, 4), "traffic": traffic_for(kname, units),
         f"algorithmic_{per}_per_launch": units}
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


def run_ours(args, world, rank, local):
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
    line = {"metric": METRIC, "value": round(value, 2), "unit": work.unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": workload_config(name, work.B),
            "roofline": roofline(work, kern),
            "gpu_launches": work.launches_per_step * args.steps * world, "clocks": clocks}
    if hasattr(work, "e2e"):
        in_bytes = sum(getattr(work.dec, n).numel() * getattr(work.dec, n).element_size()
                       for n in ("q", "k", "v", "gate"))
        if in_bytes <= E2E_HOST_LIMIT:
            line["e2e"] = work.e2e(dev, stream, world, max(3, min(args.steps, args.e2e_steps)))
        else:
            line["e2e"] = {"value": None, "unit": work.unit,
                           "skipped": f"inputs of {in_bytes / 1e9:.0f} GB exceed the "
                                      f"{E2E_HOST_LIMIT / 1e9:.0f} GB pinned host budget"}
    if rank == 0 and not args.no_cpu_baseline and hasattr(work, "cpu_sample"):
        line["cpu_baseline"] = work.cpu_sample(args.cpu_seconds)
    work.free()
    del work
    torch.cuda.empty_cache()
    # the other workloads of the hot path, timed the same way (shorter)
    if not args.only and not args.batch:
        also = {}
        for other, w in mi.WORKLOADS.items():
            if other == name or w["kind"] not in WORK_KINDS or w.get("profile_only"):
                continue
            wk = WORK_KINDS[w["kind"]](other, dev)
            k_steps = max(3, min(args.steps, 20))
            ms_o, kern_o = time_work(wk, k_steps, 3, dev, stream, world)
            also[other] = {"value": round(wk.work * world / (ms_o * 1e-3) / _scale(wk), 2),
                           "unit": wk.unit, "ms_per_step": round(ms_o, 4), "steps": k_steps,
                           "roofline": roofline(wk, kern_o)}
            line["gpu_launches"] += wk.launches_per_step * (2 * k_steps + 3) * world
            wk.free()
            del wk
            torch.cuda.empty_cache()
        line["also"] = also
    if rank == 0:
        print(json.dumps(line), flush=True)


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
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
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
