"""Benchmark of the recurrent decode step on GB300.

Default workload: gdn_b64 (GDN decode, B=64, T=1, H=16, HV=32, K=V=128, bf16
q/k/v/out, fp32 pool [256,32,128,128]).  A step is one decode call over the
batch.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl lar|reference]
  python bench.py --sweep      # batch / token curve, one JSON line per point

Timing: W untimed steps, then K steps bracketed by barrier + synchronize and
by one CUDA event pair on the launching stream (the decode kernel is the only
work there, so the average launch duration is the region / K).  When the pool
holds several disjoint batches (gdn_b64: 4 x 64 slots, 512 MiB of state) the
steps rotate over them so no launch finds its state in L2; the other
workloads touch more state than L2 holds.  value = algorithmic bytes of all
ranks' steps / max-over-ranks device time (GB/s).

--impl reference times the fp64 CPU oracle instead (the slow reference arm) on
bounded samples of the same workload; rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "decode state-pool HBM GB/s (% of GB300 peak) and tokens/s at K=V=128"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
# fp32 FMA-pipe peak: 152 SMs x 128 fp32 lanes x 2.07 GHz (maximum SM clock), in
# lane operations (one multiply or fused multiply-add on one fp32 value) per second
ALU_PEAK_OPS = 152 * 128 * 2.07e9
DESCRIPTIONS = {
    "gdn_tiny": "GDN decode B=2 T=1 H=HV=2 K=V=16 fp32",
    "gdn_b64": "GDN decode B=64 T=1 H=16 HV=32 K=V=128, bf16 q/k/v/out, fp32 pool [256,32,128,128]",
    "gdn_b64_bf16": "GDN decode B=64 T=1 H=16 HV=32 K=V=128, bf16 q/k/v/out, bf16 pool [256,32,128,128]",
    "gdn_b64_kv": "GDN decode B=64 T=1 H=16 HV=32 K=V=128, bf16 q/k/v/out, fp32 pool [256,32,128(k),128(v)] "
                  "(state stored untransposed)",
    "gdn_spec_b64": "GDN speculative verify B=64 T=4 H=16 HV=32 K=V=128, per-token pool slots "
                    "(4 per sequence, 320-slot pool), seed = slot of the last accepted token",
    "gdn_mtp_strided": "GDN MTP B=16 T=4 H=16 HV=32 K=V=128, pool = backing[::2] of [256,32,128,128], "
                       "separate write slots (25% -1), all T states cached",
    "kda_b256": "KDA decode B=256 T=1 H=HV=24 K=V=128, in-kernel gate/l2norm/sigmoid, pool [320,24,128,128]",
    "kda_b256_bf16": "KDA decode B=256 T=1 H=HV=24 K=V=128, in-kernel gate/l2norm/sigmoid, bf16 pool [320,24,128,128]",
    "la_b512_bf16": "Lightning-Attention decode B=512 T=1 H=64 K=V=128, packed bf16 QKV, "
                    "bf16 flat pool [640*64,128,128]",
    "gdn_b64_kv_bf16": "GDN decode B=64 T=1 H=16 HV=32 K=V=128, bf16 q/k/v/out, bf16 pool "
                       "[256,32,128(k),128(v)] (state stored untransposed)",
    "gdn_varlen_b64": "GDN variable-length spans N=64 (48 of 1-4 tokens, 16 prefill chunks of 16-128; "
                      "1159 tokens) H=16 HV=32 K=V=128, bf16 q/k/v/out, fp32 pool [256,32,128,128]",
    "gdn_prefill_n16": "GDN chunked prefill, N=16 spans of 256-1024 tokens (11094 tokens) H=16 HV=32 K=V=128, "
                       "bf16 q/k/v/out, fp32 pool [64,32,128,128]",
    "kda_prefill_n16": "KDA chunked prefill, N=16 spans of 256-1024 tokens H=HV=24 K=V=128, raw bf16 q/k/a "
                       "(gate chain, l2 norm, sigmoid in kernel), fp32 pool [64,24,128,128]",
    "la_b512_packed": "Lightning-Attention decode B=512 T=1 H=64 K=V=128, packed bf16 QKV, "
                      "flat pool [640*64,128,128]",
}


# the sources each kernel is built from (the ABI layer included: it sets the launch parameters)
_DECODE_SOURCES = ("decode_kernel.cuh", "decode_kv_kernel.cuh", "decode_gdn.cu", "decode_kda.cu", "decode_la.cu",
                   "decode_params.h", "launch_cache.cpp", "lar_abi.cpp")
_PREFILL_SOURCES = ("prefill.cu", "prefill_tc.cu", "prefill_ws.cu", "prefill_common.cuh", "tc_util.cuh",
                    "decode_kernel.cuh", "decode_params.h", "lar_abi.cpp")


def _code_only(text: str) -> str:
    """C / C++ / CUDA source with its comments removed and its whitespace runs
    collapsed (string and character literals kept), so that a comment edit
    does not count as a kernel change."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            i = text.find("*/", i + 2)
            i = n if i < 0 else i + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(config: str = "gdn_b64") -> str:
    """Hash of the code (comments aside) of the kernels a workload runs (the
    chunked prefill kernels, the decode kernels, or both for a split
    variable-length call); ncu traffic figures are valid only for it."""
    meta = W.make_meta(config) if config in W.CONFIGS else {}
    names = set(_PREFILL_SOURCES if meta.get("prefill") else _DECODE_SOURCES)
    if meta.get("split"):
        names |= set(_PREFILL_SOURCES)
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_attention_recurrent_gb300", "csrc")
    for name in sorted(names):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:12]


def measured_traffic(config: str, steady: bool = False):
    """dram bytes per launch from profiles/dram_traffic.txt (one cold launch) or
    profiles/dram_traffic_steady.txt (back-to-back launches, the L2 left as the
    previous launch left it), if captured on the current kernel."""
    path = os.path.join(ROOT, "profiles", "dram_traffic_steady.txt" if steady else "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(config)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == config and parts[1] == want:
            return int(parts[2])
    return None


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        sel = []
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if ids and device_index < len(ids):
            sel = ["-i", ids[device_index]]
        else:
            try:
                u = str(torch.cuda.get_device_properties(device_index).uuid)
                sel = ["-i", u if u.startswith("GPU-") else "GPU-" + u]
            except Exception:
                sel = ["-i", str(device_index)]
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "50"] + sel

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons, n = [], [], set(), 0
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ts, line in self.lines:
            if not (t0 - 0.06 <= ts <= t1 + 0.06):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            n += 1
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": n}


# ------------------------------------------------------------------ distributed

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ workload on device

def device_inputs(w, dev):
    cu = lambda t: None if t is None else t.to(dev)
    q, k, v = w.qkv_to(dev)    # packed workloads: slices of one fused device buffer
    if w.fused is not None:
        es = q.element_size()
        if not (q.stride() == k.stride() == w.q.stride() and k.data_ptr() == q.data_ptr() + w.K * es
                and v.data_ptr() == q.data_ptr() + 2 * w.K * es):
            raise RuntimeError("packed q/k/v did not reach the device as views of one buffer")
    d = {"q": q, "k": k, "v": v, "pool": w.pool if w.pool.is_cuda else w.pool.to(dev)}
    if w.form == "la":
        d["decay"] = cu(w.decay)
    else:
        d.update(g=cu(w.g), beta=cu(w.beta), A_log=cu(w.A_log), dt_bias=cu(w.dt_bias))
    return d


def inter_shape(w):
    if w.cu_seqlens is not None:
        return (w.v.shape[0], w.HV, w.V, w.K)
    return (w.B, w.T, w.HV, w.V, w.K)


def index_sets(w):
    """Disjoint (read, write) index sets to rotate over, when the pool holds
    several batches (in-place workloads only); else the workload's own set."""
    if w.state_idx is not None:
        return [(w.read_idx, w.write_idx)], 1
    same = w.write_idx is not None and torch.equal(w.read_idx, w.write_idx)
    n = w.P // w.B if same else 1
    if n >= 2:
        n = min(n, 4)
        sets = W.disjoint_index_sets(w.P, w.B, n, seed=1234, index_dtype=w.read_idx.dtype)
        return [(s, s.clone()) for s in sets], n
    return [(w.read_idx, w.write_idx)], 1


# ------------------------------------------------------------------ our arm

def run_lar(args, world, rank, local):
    import linear_attention_recurrent_gb300 as lar

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lar.load()
    w = W.make(args.config, pool_device=dev)
    d = device_inputs(w, dev)
    sets, n_sets = index_sets(w)
    stream = torch.cuda.Stream(device=dev)
    outs, inters, calls = [], [], []
    with torch.cuda.stream(stream):
        for ri, wi in sets:
            out = torch.empty(w.v.shape, dtype=w.out_dtype, device=dev)
            inter = (torch.empty(inter_shape(w), device=dev, dtype=w.inter_dtype)
                     if w.cache_intermediate else None)
            kw = dict(d, read_idx=ri.to(dev), write_idx=None if wi is None else wi.to(dev),
                      out=out, inter=inter)
            if w.cu_seqlens is not None:
                kw.update(cu_seqlens=w.cu_seqlens.to(dev))
            if w.state_idx is not None:
                kw.update(state_idx=w.state_idx.to(dev), write_idx=None, inter=None)
                if w.num_accepted is not None:
                    kw.update(num_accepted=w.num_accepted.to(dev), read_idx=None)
            if w.form != "la":
                kw.update(qk_l2norm=w.qk_l2norm, gate_raw=w.gate_raw, beta_raw=w.beta_raw,
                          state_kv=w.state_kv)
            if w.meta.get("prefill"):
                kw.update(prefill=True)
            calls.append(lar.PreparedCall(w.form, scale=w.scale, stream=stream, **kw))
            outs.append(out)
            inters.append(inter)
    bytes_per_step = w.algorithmic_bytes()
    torch.cuda.synchronize(dev)

    for i in range(args.warmup):
        calls[i % n_sets]()
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    # keep the GPU busy while the sampler spins up, then time exactly K steps
    for i in range(min(args.warmup, 50)):
        calls[i % n_sets]()
    barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        first = torch.cuda.Event(enable_timing=True)
        last = torch.cuda.Event(enable_timing=True)
        hold_stream(stream)
        first.record(stream)
        for i in range(args.steps):
            calls[i % n_sets]()
        last.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(world)
    clocks = sampler.stop(t_wall0, t_wall1)

    total_ms = first.elapsed_time(last)
    # this library's kernels are the only work on `stream` in the timed region, so
    # one call's average duration (back to back, gaps included) is the region / K;
    # a call of one launch makes that the kernel's average launch duration
    mean_launch_ms = total_ms / args.steps
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    gbs = bytes_per_step * args.steps * world / (total_ms * 1e-3) / 1e9
    tokens = w.tokens() * args.steps * world / (total_ms * 1e-3)
    achieved = bytes_per_step / (mean_launch_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()

    e2e = run_e2e(w, d, sets, dev, stream, args) if rank == 0 else None
    cpu = cpu_baseline(w, args) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None

    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; see workloads.py)",
        "config": {"workload": f"{args.config}: {DESCRIPTIONS.get(args.config, args.config)}",
                   "bytes_per_step": bytes_per_step, "tokens_per_step": w.tokens(),
                   "l2": (f"rotating {n_sets} disjoint slot sets "
                          f"({n_sets * w.B * w.HV * w.K * w.V * w.pool.element_size() / 2**20:.0f} MiB of state), "
                          "inputs larger than L2" if n_sets > 1 else "inputs larger than L2"),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   **({"qkv": f"head-dim slices of one fused device buffer, row stride {d['q'].stride()[-2]}"}
                      if w.fused is not None else {})},
        "tokens_per_s": round(tokens, 1),
        "pct_of_8tbs": round(100 * gbs / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_peak": round(100 * gbs / world / peak, 2),
        "roofline": roofline(w, args.config, mean_launch_ms, achieved, peak, peak_kind),
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step(w),
        "clocks": clocks,
    }
    return line


def hold_stream(stream, cycles=1_000_000):
    """Keep `stream` busy (a spin kernel of about 0.5 ms) while the host
    enqueues the timed launches behind it, so the first timed launch does not
    wait for the host: the events then bracket back-to-back device work only."""
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        with torch.cuda.stream(stream):
            sleep(cycles)


# tensor-core rates: the measured dense bf16 GEMM rate x the nominal tf32 / bf16
# ratio (1.1 / 2.25 PFLOP/s): the chunked prefill's products are fp32-accurate,
# reported against the rate of a single tf32 pass
TF32_OVER_BF16 = 1.1 / 2.25
PREFILL_CHUNK = 32


def launches_per_step(w) -> int:
    """Kernels of this library launched per call: a variable-length call
    without a state cache at K = V = 128 launches the chunked kernel for its
    long spans (when its token arrays can hold a span of 16 tokens) and the
    token-by-token kernel for the rest."""
    if w.cu_seqlens is not None and not w.meta.get("prefill") and not w.cache_intermediate and w.K == 128 \
            and w.V == 128 and min(w.B, w.q.shape[0] // 16) > 0:
        return 2
    return 1


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def prefill_tensor_flops(w) -> int:
    """FLOPs of the chunked prefill's tensor-core products per launch, one
    pass (the kernels run each product as several exact-product passes: bf16
    terms or tf32 halves): per 32-token
    chunk of a span and value head, [U | P] = S0^T [K ; Q]^T (GDN, KDA;
    LA: P only), [K ; Q] K^T (GDN; LA: Q K^T; KDA builds it on the CUDA cores),
    O = D M^T and the increment (D o W) K."""
    C, K, V = PREFILL_CHUNK, w.K, w.V
    up = 2 * V * (C if w.form == "la" else 2 * C) * K
    kk = {"gdn": 2 * 2 * C * C * K, "la": 2 * C * C * K, "kda": 0}[w.form]
    per_chunk = up + kk + 2 * V * C * C + 2 * V * K * C
    cu = w.cu_seqlens.to("cpu").long()
    lengths = (cu[1:] - cu[:-1]).clamp(min=0)
    chunks = int(((lengths + C - 1) // C).sum())
    return chunks * w.HV * per_chunk


def roofline(w, config, mean_launch_ms, achieved_gbs, peak_gbs, peak_kind):
    """The bound of the launch: HBM (algorithmic bytes / copy bandwidth) unless
    the fp32 arithmetic of the state update takes longer at the FMA-pipe peak
    (long variable-length spans), in which case the line reports against that.
    The chunked prefill runs its products on the tensor cores and reports
    against the tf32 rate."""
    if w.meta.get("prefill"):
        # GDN / LA with staged bf16 rows run the warp-specialised kernel
        kname = "prefill_tc_kernel" if w.form == "kda" else "prefill_ws_kernel"
    else:
        kname = "decode_kernel"
    kernel = f"{kname}<{w.form}>"
    if launches_per_step(w) == 2:
        # long spans in the chunked kernel, the rest token by token: the figures
        # below cover the call (both launches); traffic sums the two kernels
        chunked = "prefill_tc_kernel" if w.form == "kda" else "prefill_ws_kernel"
        kernel = f"{chunked}<{w.form}> + decode_kernel<{w.form}>"
    base = {"traffic": measured_traffic(config), "traffic_steady": measured_traffic(config, steady=True),
            "kernel": f"{kernel} ({kernel_source_hash(config)})",
            "launches_per_call": launches_per_step(w),
            "mean_launch_us" if launches_per_step(w) == 1 else "mean_call_us": round(mean_launch_ms * 1e3, 3)}
    ops = w.alu_ops()
    if w.meta.get("prefill"):
        flops = prefill_tensor_flops(w)
        bf16, kind = bf16_peak()
        peak = bf16 * TF32_OVER_BF16
        achieved = flops / (mean_launch_ms * 1e-3) / 1e12
        return dict({"bound": "tensor", "achieved": round(achieved, 3), "peak": round(peak, 1),
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{kind} bf16 GEMM rate x nominal tf32/bf16 ratio 1.1/2.25",
                     "flops_per_launch": flops,
                     "passes": ("tf32 x3" if w.form == "kda" else
                                "bf16 x3 ([U | P], increment), bf16 x1 (K K^T), tf32 x3 (O)"),
                     "alu_equivalent": {"achieved": round(ops / (mean_launch_ms * 1e-3) / 1e12, 3),
                                        "unit": "T lane-op/s", "frac": round(ops / (mean_launch_ms * 1e-3) / ALU_PEAK_OPS, 4)},
                     "hbm_frac": round(achieved_gbs / peak_gbs, 4)}, **base)
    t_hbm = w.algorithmic_bytes() / (peak_gbs * 1e9)
    t_alu = ops / ALU_PEAK_OPS
    if t_alu > t_hbm:
        achieved = ops / (mean_launch_ms * 1e-3) / 1e12
        peak = ALU_PEAK_OPS / 1e12
        return dict({"bound": "alu", "achieved": round(achieved, 3), "peak": round(peak, 2),
                     "unit": "T lane-op/s", "frac": round(achieved / peak, 4),
                     "peak_source": "152 SMs x 128 fp32 lanes x 2.07 GHz",
                     "ops_per_launch": ops, "hbm_frac": round(achieved_gbs / peak_gbs, 4)}, **base)
    return dict({"bound": "hbm", "achieved": round(achieved_gbs, 2), "peak": peak_gbs, "unit": "GB/s",
                 "frac": round(achieved_gbs / peak_gbs, 4), "peak_source": f"{peak_kind} copy bandwidth"},
                **base)


def run_e2e(w, d, sets, dev, stream, args):
    """The same metric through the public API with host buffers.  Per step:
    one pinned-host -> device copy of all of the step's inputs (q, k, v, the
    gates and slot indices, packed back to back as a serving loop would stage
    them), one decode call through `PreparedCall`, a device -> host copy of
    the output, and a stream synchronize.  The pool stays resident; the steps
    rotate over the same disjoint slot sets as the device-timed arm, so no step
    finds its state in L2."""
    import linear_attention_recurrent_gb300 as lar

    names = ["q", "k", "v"] + (["decay"] if w.form == "la" else ["g", "beta"])
    out_dev = torch.empty(w.v.shape, dtype=w.out_dtype, device=dev)
    out_host = torch.empty(out_dev.shape, dtype=out_dev.dtype).pin_memory()
    inter = (torch.empty(inter_shape(w), device=dev, dtype=w.inter_dtype)
             if w.cache_intermediate else None)
    staged = []    # per slot set: (pinned host buffer, device buffer, call)
    for ri, wi in sets:
        host_parts = {n: getattr(w, n).contiguous() for n in names if getattr(w, n) is not None}
        if w.state_idx is not None:
            host_parts["state_idx"] = w.state_idx.contiguous()
            if w.num_accepted is not None:
                host_parts["num_accepted"] = w.num_accepted.contiguous()
            else:
                host_parts["read_idx"] = ri.contiguous()
        else:
            host_parts["read_idx"] = ri.contiguous()
            host_parts["write_idx"] = wi.contiguous()
        if w.cu_seqlens is not None:
            host_parts["cu_seqlens"] = w.cu_seqlens.contiguous()
        offs, total = {}, 0
        for n, t in host_parts.items():
            offs[n] = total
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
        dbuf = torch.empty(total, dtype=torch.uint8, device=dev)
        views = {}
        for n, t in host_parts.items():
            nb = t.numel() * t.element_size()
            hbuf[offs[n]:offs[n] + nb].copy_(t.view(-1).view(torch.uint8))
            views[n] = dbuf[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)
        kw = dict(views, pool=d["pool"], out=out_dev, inter=inter)
        if w.form != "la":
            kw.update(A_log=d.get("A_log"), dt_bias=d.get("dt_bias"), qk_l2norm=w.qk_l2norm,
                      gate_raw=w.gate_raw, beta_raw=w.beta_raw, state_kv=w.state_kv)
        if w.meta.get("prefill"):
            kw.update(prefill=True)
        staged.append((hbuf, dbuf, lar.PreparedCall(w.form, scale=w.scale, stream=stream, **kw)))
    h2d = sum(t.numel() * t.element_size() for t in host_parts.values())
    d2h = out_host.numel() * out_host.element_size()
    steps = max(10, min(args.steps, 2000))
    it = [0]

    def step():
        hbuf, dbuf, call = staged[it[0] % len(staged)]
        it[0] += 1
        with torch.cuda.stream(stream):
            dbuf.copy_(hbuf, non_blocking=True)
            call()
            out_host.copy_(out_dev, non_blocking=True)
        stream.synchronize()

    for _ in range(5):
        step()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    dt = (time.perf_counter() - t0) / steps
    return {"value": round(w.algorithmic_bytes() / dt / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(dt * 1e3, 4), "steps": steps,
            "tokens_per_s": round(w.tokens() / dt, 1),
            "note": "wall clock per step, rotating the slot sets: one packed pinned H2D copy of the step's inputs, the "
                    "decode call, D2H of the output, stream sync; the pool stays resident"}


# ------------------------------------------------------------------ oracle timing

def _oracle_step(w, host_pool, batch):
    import oracle
    sel = lambda t: None if t is None else t[batch]
    if w.cu_seqlens is not None:
        # one call per sequence on its own token rows
        fn = {"gdn": oracle.gdn_decode_varlen, "kda": oracle.kda_decode_varlen}[w.form]
        cu = w.cu_seqlens.long()
        for n in torch.as_tensor(batch).view(-1).tolist():
            lo, hi = int(cu[n]), int(cu[n + 1])
            tok = lambda t: None if t is None else t[lo:hi]
            fn(tok(w.q), tok(w.k), tok(w.v), tok(w.g), tok(w.beta), host_pool, torch.tensor([0, hi - lo]),
               w.read_idx[n:n + 1], w.write_idx[n:n + 1], A_log=w.A_log, dt_bias=w.dt_bias,
               qk_l2norm=w.qk_l2norm, gate_raw=w.gate_raw, beta_raw=w.beta_raw, scale=w.scale,
               cache_intermediate=w.cache_intermediate)
        return
    if w.form == "la":
        oracle.la_decode(sel(w.q), sel(w.k), sel(w.v), w.decay, host_pool, sel(w.read_idx),
                         sel(w.write_idx), scale=w.scale, cache_intermediate=w.cache_intermediate)
    elif w.state_idx is not None:
        fn = oracle.gdn_decode_tokens if w.form == "gdn" else oracle.kda_decode_tokens
        fn(sel(w.q), sel(w.k), sel(w.v), sel(w.g), sel(w.beta), host_pool, sel(w.state_idx),
           read_idx=None if w.num_accepted is not None else sel(w.read_idx),
           num_accepted=sel(w.num_accepted), A_log=w.A_log, dt_bias=w.dt_bias,
           qk_l2norm=w.qk_l2norm, gate_raw=w.gate_raw, beta_raw=w.beta_raw, scale=w.scale)
    else:
        fn = oracle.gdn_decode if w.form == "gdn" else oracle.kda_decode
        fn(sel(w.q), sel(w.k), sel(w.v), sel(w.g), sel(w.beta), host_pool, sel(w.read_idx),
           sel(w.write_idx), A_log=w.A_log, dt_bias=w.dt_bias, qk_l2norm=w.qk_l2norm,
           gate_raw=w.gate_raw, beta_raw=w.beta_raw, scale=w.scale,
           cache_intermediate=w.cache_intermediate, layout="kv" if w.state_kv else "vk")


def _host_workload(config):
    """The workload with its pool on the host (the oracle reads it in place)."""
    w = W.make(config, pool_device="cuda" if torch.cuda.is_available() else "cpu")
    if w.backing is not None:
        mult = w.pool.stride(0) // w.backing.stride(0)
        w.backing = w.backing.cpu()
        w.pool = w.backing[::mult]
    else:
        w.pool = w.pool.cpu()
    return w


def _timed_oracle_steps(w, batches, budget_s, executor=None):
    """Whole oracle steps (every entry once per step, split into `batches`,
    run concurrently on `executor` when given) for about `budget_s` seconds.
    Returns (steps, seconds)."""
    reps, t0 = 0, time.perf_counter()
    while True:
        if executor is None:
            for bt in batches:
                _oracle_step(w, w.pool, bt)
        else:
            list(executor.map(lambda bt: _oracle_step(w, w.pool, bt), batches))
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 1000:
            return reps, el


def cpu_baseline(w_dev, args, budget_s=10.0):
    """The oracle as it stands (plain fp64 C loops) on whole steps of the same
    workload: on all host cores (the batch split into one contiguous slice per
    core, the slices run concurrently by threads; the C calls release the
    interpreter lock, and slices touch disjoint pool slots), and on one thread."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    oracle.build()
    w = _host_workload(args.config)
    ncores = max(1, min(os.cpu_count() or 1, w.B))
    slices = [torch.arange(w.B)[i::ncores] for i in range(ncores)]
    with ThreadPoolExecutor(max_workers=ncores) as ex:
        reps, el = _timed_oracle_steps(w, slices, budget_s, ex)
    reps1, el1 = _timed_oracle_steps(w, [torch.arange(w.B)], budget_s / 2)
    per_step = w.algorithmic_bytes()
    return {"value": round(per_step * reps / el / 1e9, 4), "unit": "GB/s", "cores": ncores, "kind": "oracle",
            "sample": f"{reps} whole {args.config} steps ({w.B} entries x {w.HV} heads each) in {el:.1f} s, "
                      f"fp64 C loops, the batch split over {ncores} threads",
            "tokens_per_s": round(w.tokens() * reps / el, 2),
            "single_thread": {"value": round(per_step * reps1 / el1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"{reps1} whole steps in {el1:.1f} s"}}


def sample_bytes(w, n):
    """Algorithmic bytes of the first n entries of a step: their share of the
    state traffic and, with variable-length spans, their share of the per-token
    traffic (their tokens over all tokens)."""
    total = w.algorithmic_bytes()
    if w.cu_seqlens is None:
        return total * n / w.B
    cu = w.cu_seqlens.long()
    unit = w.HV * w.K * w.V * w.pool.element_size()
    ok = lambda t: ((t >= 0) & (t < w.P)).long()
    state = int((ok(w.read_idx.long()) + ok(w.write_idx.long())).sum()) * unit
    state_n = int((ok(w.read_idx[:n].long()) + ok(w.write_idx[:n].long())).sum()) * unit
    tok_frac = int(cu[n] - cu[0]) / max(int(cu[-1] - cu[0]), 1)
    return state_n + (total - state) * tok_frac


def run_reference(args, world, rank):
    """Reference arm: the fp64 CPU oracle, rank 0 only, on bounded samples, the
    sample of each step split over all host cores as in cpu_baseline."""
    if rank != 0:
        return None
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    oracle.build()
    w = _host_workload(args.config)
    ncores = max(1, min(os.cpu_count() or 1, w.B))
    # size each step's sample so warmup + steps stay around a minute
    n_probe = min(8, w.B)
    probe_t0 = time.perf_counter()
    _oracle_step(w, w.pool, torch.arange(n_probe))
    per_entry = max((time.perf_counter() - probe_t0) / n_probe, 1e-6)
    n = max(1, min(w.B, int(60.0 * ncores / ((args.steps + args.warmup) * per_entry))))
    ncores = min(ncores, n)
    slices = [torch.arange(n)[i::ncores] for i in range(ncores)]
    with ThreadPoolExecutor(max_workers=ncores) as ex:
        step = lambda: list(ex.map(lambda bt: _oracle_step(w, w.pool, bt), slices))
        for _ in range(args.warmup):
            step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step()
        el = time.perf_counter() - t0
    bytes_step = sample_bytes(w, n)
    gbs = bytes_step * args.steps / el / 1e9
    sample = (f"{n} of {w.B} entries ({n * w.HV} (entry, head) states) per step, split over "
              f"{ncores} threads; bytes: those of the {n} entries")
    return {"impl": "reference", "metric": METRIC, "value": round(gbs, 5), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.config}: {DESCRIPTIONS.get(args.config, args.config)}",
                       "parallelism": f"{ncores} host threads"},
            "cpu_baseline": {"value": round(gbs, 5), "unit": "GB/s", "cores": ncores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(gbs, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ sweep

SWEEP_POINTS = (
    [("gdn", B, 1) for B in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024)]
    + [("gdn", 64, T) for T in (2, 4, 8)]
    + [("kda", B, 1) for B in (16, 64, 256, 1024)]
    + [("la", B, 1) for B in (16, 64, 512)]
    # variable-length spans (T = tokens per span, every span the same length)
    + [("gdn_varlen", 64, L) for L in (1, 4, 16, 64, 256)]
    + [("gdn_varlen", 8, 1024)]
)
SWEEP_HEADS = {"gdn": (16, 32), "kda": (24, 24), "la": (64, 64), "gdn_varlen": (16, 32)}


def run_sweep(args):
    """GB/s and tokens/s over batch size and token count at K = V = 128 (the
    gdn_b64 / kda_b256 / la_b512 head shapes, no state cache), one JSON line per
    point.  Each point rotates over disjoint slot sets (4 when the pool holds
    them) and times back-to-back launches with one CUDA event pair."""
    import linear_attention_recurrent_gb300 as lar

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lar.load()
    peak, _ = hbm_peak()
    for form, B, T in SWEEP_POINTS:
        H, HV = SWEEP_HEADS[form]
        if form == "gdn_varlen":
            w = W.make_varlen("gdn", [T] * B, H=H, HV=HV, K=128, V=128, P=4 * B, seed=1, pool_device=dev)
        else:
            w = W.make_custom(form, B=B, T=T, H=H, HV=HV, K=128, V=128, P=4 * B, seed=1, pool_device=dev,
                              raw_gates=form == "kda", flat_pool=form == "la")
        d = device_inputs(w, dev)
        sets, n_sets = index_sets(w)
        stream = torch.cuda.Stream(device=dev)
        calls = []
        for ri, wi in sets:
            out = torch.empty(w.v.shape, dtype=w.out_dtype, device=dev)
            kw = dict(d, read_idx=ri.to(dev), write_idx=wi.to(dev), out=out)
            if w.cu_seqlens is not None:
                kw.update(cu_seqlens=w.cu_seqlens.to(dev))
            if w.form != "la":
                kw.update(qk_l2norm=w.qk_l2norm, gate_raw=w.gate_raw, beta_raw=w.beta_raw)
            calls.append(lar.PreparedCall(w.form, scale=w.scale, stream=stream, **kw))
        for i in range(max(args.warmup, 20)):
            calls[i % n_sets]()
        torch.cuda.synchronize(dev)
        launches = max(20, min(5000, int(60e9 / w.algorithmic_bytes())))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(launches):
                calls[i % n_sets]()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) / launches * 1e3
        gbs = w.algorithmic_bytes() / us / 1e3
        print(json.dumps({"sweep": form, "B": B, "T": T, "H": H, "HV": HV, "us": round(us, 2),
                          "GBs": round(gbs, 1), "pct_of_measured_peak": round(100 * gbs / peak, 1),
                          "alu_frac": round(w.alu_ops() / (us * 1e-6) / ALU_PEAK_OPS, 3),
                          "tokens_per_s": round(B * T / us * 1e6), "launches": launches}), flush=True)
        del w, d, calls
        torch.cuda.empty_cache()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--config", default="gdn_b64", choices=W.CONFIGS)
    ap.add_argument("--impl", default="lar", choices=["lar", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="print one line per (form, B, T) point of the batch / token sweep instead")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.sweep:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback exists)")
        run_sweep(args)
        return
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback exists)")
        line = run_lar(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
