"""Decode-step benchmark: quantize the new token + GQA decode attention.

One step = dq_quantize_kv of one new token per sequence (rotation, mean,
grid, codes, packing, 16-bit recent slot) followed by dq_decode_attention over
the whole cache.  The workload is the Llama-3-8B-shaped decode layer: batch 16,
32 query / 8 KV heads, head_dim 128, 8192 cached tokens (4 sink + 128 recent
in bf16, the rest packed), bf16 inputs, seeded synthetic K/V/q.  Each step
re-appends the token at position 8191, so the cache length stays fixed.

Inputs are larger than L2 in aggregate: steps rotate over several copies of
the cache (their total exceeds the L2 size), so no step reads the previous
step's bytes from L2.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead: the slow CPU implementation the GPU results are checked against.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "quantized decode-attn tokens/s & achieved HBM GB/s (% of roofline), 2/3/4-bit"
# the KVQuant-shaped cache with the page's configuration options on: value
# tables per 32 channels, key tables per 128-slot block (a window of 128 recent
# 16-bit tokens holds a block's keys until it is refitted)
NUQ_GROUP_REFIT = W.NUQ.with_(n_recent=128, extra={"lloyd_iters": 8, "outlier_frac": 0.01, "group_size": 32,
                                                   "refit_interval": 128})
CSRC = os.path.join(ROOT, "quantized_decode_attention_gb300", "csrc")
# the sources each attention kernel is compiled from (the traffic record is
# valid only for the exact sources it was captured with)
KERNEL_SRCS = {
    "affine": ["attn_affine.cu", "attn_common.cuh", "common.cuh", "quant_row.cuh"],
    "generic": ["attn.cu", "attn_common.cuh", "common.cuh"],
    "rans": ["attn_rans.cu", "common.cuh"],
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_traffic.json")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--bits", type=int, default=2)
    p.add_argument("--variants", default="3,4", help="other code widths measured in the same run")
    p.add_argument("--copies", type=int, default=0, help="cache copies rotated per step (0 = auto)")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU baseline sample budget")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-nuq", action="store_true", help="skip the KVQuant NUQ cache measurement")
    p.add_argument("--no-dquant", action="store_true", help="skip the D-Quant cache measurement")
    p.add_argument("--qwen", default="32768,131072", help="Qwen3-8B-shaped long-context lengths measured")
    p.add_argument("--no-bf16", action="store_true", help="skip the unquantized 16-bit cache context entry")
    p.add_argument("--profile-attn", action="store_true",
                   help="profiler run: one cache, warmup + steps attention calls, no timing")
    p.add_argument("--profile-batch", type=int, default=4, help="--profile-attn: batch of the D-Quant cache")
    p.add_argument("--profile-kind", default="affine", choices=["affine", "nuq", "nuq_gr", "dquant"],
                   help="--profile-attn cache: the Llama-shaped affine cache at --bits, the KVQuant NUQ cache "
                        "(plain, or with value groups and key refit blocks), or the D-Quant cache")
    return p.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def algorithmic_bytes(w: W.Workload, bits: int, S: int) -> dict:
    """Bytes one decode-attention call must move: packed codes, scale/offset,
    key mean, 16-bit sink/recent slots, q and out."""
    U, d = w.batch * w.n_kv_heads, w.head_dim
    n_raw = min(S, w.n_sink) + min(max(S - w.n_sink, 0), w.n_recent)
    n_q = S - n_raw
    meta = 2 if w.meta_dtype == "f16" else 4
    codes = U * n_q * d * bits // 8 * 2
    metab = U * n_q * 2 * meta * 2
    mean = U * d * 4 if w.mean_k else 0
    raw = U * n_raw * d * 2 * 2
    q = w.batch * w.n_q_heads * d * 4
    out = w.batch * w.n_q_heads * d * 2
    qcomp = w.n_kv_heads * d * d * 4 if w.rot_k == "dense" else 0   # T^-T for the queries
    total = codes + metab + mean + raw + q + out + qcomp
    return {"codes": codes, "meta": metab, "mean": mean, "raw": raw, "q": q, "out": out, "q_comp": qcomp,
            "total": total}


def reduce_max(x: float) -> float:
    """The maximum of x over the ranks of the process group (x itself without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(total_ms: float, steps: int, batch_per_rank: int, world: int):
    """(ms per step, whole-job tokens/s): the slowest rank's time, every rank's tokens."""
    ms_step = reduce_max(total_ms) / steps
    return ms_step, batch_per_rank * world / (ms_step / 1e3)


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def nuq_algorithmic_bytes(w: W.Workload, S: int) -> dict:
    """Bytes one non-uniform decode-attention call must move: key and value
    codes, per-token value tables (one per channel group), per-channel key
    tables (one set per refit block read), the outlier side channels (key CSR
    by token with its row pointers, value entries per token), the 16-bit sinks
    and recent window, q and out."""
    U, d, L = w.batch * w.n_kv_heads, w.head_dim, 1 << w.bits
    n_raw = min(S, w.n_sink) + min(max(S - w.n_sink, 0), w.n_recent)
    n_q = S - n_raw
    frac = w.extra.get("outlier_frac", 0.01)
    kk = int(np.floor(np.float64(np.float32(frac)) * n_q + 0.5))
    kv = int(np.floor(np.float64(np.float32(frac)) * d + 0.5))
    gv = d // (w.extra.get("group_size", 0) or d)
    N = w.extra.get("refit_interval", 0) or 0
    codes = U * n_q * d * w.bits // 8 * 2
    lut = U * n_q * gv * L * 2 + U * (-(-n_q // N) if N else 1) * d * L * 2
    side = U * (d * kk * 4 + (n_q + 1) * 4) + U * n_q * kv * 4
    raw = U * n_raw * d * 2 * 2
    q = w.batch * w.n_q_heads * d * 4
    out = w.batch * w.n_q_heads * d * 2
    total = codes + lut + side + raw + q + out
    return {"codes": codes, "tables": lut, "outliers": side, "raw": raw, "q": q, "out": out, "total": total}


def dquant_algorithmic_bytes(w: W.Workload, S: int) -> dict:
    """Bytes one D-Quant decode-attention call must move: the key and value
    containers and fp16 (s, o) of the quantized tokens, the INT8 window means
    covering them, the 16-bit sinks and recent window, q and out."""
    U, d = w.batch * w.n_kv_heads, w.head_dim
    n = w.n_kv_heads * d
    n_raw = min(S, w.n_sink) + min(max(S - w.n_sink, 0), w.n_recent)
    n_q = S - n_raw
    cont = w.batch * n_q * (w.extra["container_k"] + w.extra["container_v"])
    meta = w.batch * n_q * 8
    mean = w.batch * (-(-n_q // 128)) * (n + 16) if w.mean_k else 0
    raw = U * n_raw * d * 2 * 2
    q = w.batch * w.n_q_heads * d * 4
    out = w.batch * w.n_q_heads * d * 2
    total = cont + meta + mean + raw + q + out
    return {"containers": cont, "meta": meta, "mean": mean, "raw": raw, "q": q, "out": out, "total": total}


class Clocks:
    """SM clocks and clock-event (throttle) reasons of this process's GPU,
    sampled in the background while the measurement runs: through NVML every
    millisecond (ctypes on the driver's libnvidia-ml), else nvidia-smi every
    20 ms.  Each sample carries its host time, so any region's clocks are the
    samples taken inside it (or, for a region shorter than the sampling
    period, the two that bracket it)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, index: int):
        self.index = index
        self.samples = []  # (host time, sm MHz, reason bits or names)
        self.max_mhz = None
        self.proc = None
        self.stop = threading.Event()
        self.source = None

    def _nvml_handle(self):
        import ctypes as C
        import torch
        nv = C.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit")
        pr = torch.cuda.get_device_properties(self.index)
        h = C.c_void_p()
        bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
        if nv.nvmlDeviceGetHandleByPciBusId_v2(bus, C.byref(h)) != 0:
            raise RuntimeError("nvml handle")
        return nv, h

    def __enter__(self):
        try:
            import ctypes as C
            nv, h = self._nvml_handle()
            mx = C.c_uint(0)
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, C.byref(mx)) == 0:  # 1: the SM clock
                self.max_mhz = float(mx.value)
            fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons

            def poll():
                clk, rs = C.c_uint(0), C.c_ulonglong(0)
                while not self.stop.is_set():
                    t = time.perf_counter()
                    if nv.nvmlDeviceGetClockInfo(h, 1, C.byref(clk)) == 0 and fn(h, C.byref(rs)) == 0:
                        self.samples.append((t, float(clk.value), int(rs.value)))
                    time.sleep(0.001)
            self.t = threading.Thread(target=poll, daemon=True)
            self.t.start()
            self.source = "nvml, 1 ms"
        except Exception:
            self._start_smi()
        deadline = time.perf_counter() + 5.0
        while not self.samples and time.perf_counter() < deadline:  # the first sample precedes any region
            time.sleep(0.002)
        return self

    def _start_smi(self):
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            import torch
            pr = torch.cuda.get_device_properties(self.index)
            sel = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        except Exception:
            sel = str(self.index)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", sel, f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

            def read():
                for line in self.proc.stdout:
                    p = [x.strip() for x in line.split(",")]
                    if len(p) >= 6 and p[0].replace(".", "").isdigit():
                        if p[1].replace(".", "").isdigit():
                            self.max_mhz = float(p[1])
                        self.samples.append((time.perf_counter(), float(p[0]),
                                             [names[i] for i in range(4) if p[2 + i].lower() == "active"]))
            self.t = threading.Thread(target=read, daemon=True)
            self.t.start()
            self.source = "nvidia-smi, 20 ms"
        except Exception:
            self.proc = None

    def __exit__(self, *a):
        self.stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()

    def _names(self, r):
        return r if isinstance(r, list) else [n for b, n in self.REASONS.items() if r & b]

    def summary(self, t0: float = None, t1: float = None):
        """Clocks over the host-time window [t0, t1] (all samples if None)."""
        smp = list(self.samples)
        if not smp:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"]}
        how = "inside"
        if t0 is not None:
            inside = [x for x in smp if t0 <= x[0] <= t1]
            if not inside:  # a region shorter than the sampling period: the samples around it
                before = [x for x in smp if x[0] < t0][-1:]
                after = [x for x in smp if x[0] > t1][:1]
                inside, how = before + after, "bracketing"
            smp = inside
        sm = [x[1] for x in smp]
        reasons = sorted({n for x in smp for n in self._names(x[2])})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(smp), "window": how, "source": self.source}


def kernel_sha(kind: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SRCS[kind]:
        h.update(open(os.path.join(CSRC, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kind: str, bits):
    """DRAM bytes per attention launch from the committed ncu capture, or None
    when the kernel's sources differ from the ones captured."""
    key = bits if isinstance(bits, str) else f"{bits}bit"
    kernel_sha = globals()["kernel_sha"](kind)
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        ent = d.get(key)
        if ent and ent.get("src_sha", ent.get("attn_src_sha")) == kernel_sha:
            return ent.get("bytes_per_launch")
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def setup_caches(w, bits, S, k_dev, v_dev, copies):
    import torch
    from quantized_decode_attention_gb300 import KVCache, make_config
    cfg = make_config(batch=w.batch, n_kv_heads=w.n_kv_heads, n_q_heads=w.n_q_heads, head_dim=w.head_dim,
                      max_seq=S, kv_dtype=w.kv_dtype, meta_dtype=w.meta_dtype, out_dtype=w.out_dtype, bits=bits,
                      rot_k=w.rot_k, rot_v=w.rot_v, mean_k=w.mean_k, clip_k=w.clip, clip_v=w.clip,
                      n_sink=w.n_sink, n_recent=w.n_recent)
    base = KVCache.allocate(cfg, zero=False)
    if w.rot_k == "dense":
        T, Qc = W.dense_transform(w)
        base.tensors["k_transform"].view(torch.float32).copy_(torch.from_numpy(T).reshape(-1))
        base.tensors["q_comp"].view(torch.float32).copy_(torch.from_numpy(Qc).reshape(-1))
    base.quantize(k_dev, v_dev, pos0=0)  # the first call also creates the context
    base.check()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record()
    base.quantize(k_dev, v_dev, pos0=0)
    p1.record()
    torch.cuda.synchronize()
    base.check()
    caches = [base]
    for _ in range(copies - 1):
        caches.append(base.clone_shared())
    torch.cuda.synchronize()
    return caches, p0.elapsed_time(p1)


def run_gpu(args, w, bits, S, k_dev, v_dev, q_dev, knew_dev, vnew_dev, rank):
    import torch
    from quantized_decode_attention_gb300 import load
    L2 = torch.cuda.get_device_properties(0).L2_cache_size
    ab = algorithmic_bytes(w, bits, S)
    per_copy = ab["total"]
    copies = args.copies or max(3, int(np.ceil(3 * L2 / per_copy)) + 1)
    caches, prefill_ms = setup_caches(w, bits, S, k_dev, v_dev, copies)
    td = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[w.out_dtype]
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=td, device="cuda")
    stream = torch.cuda.Stream()
    sm_scale = w.head_dim ** -0.5
    pos = S - 1

    def step(c, s):  # append the new token and attend: one fused library call
        c.decode_step(knew_dev, vnew_dev, q_dev, out, S, sm_scale, stream=s.cuda_stream)

    # CUDA graphs: one per cache copy holding [quantize new token, attention],
    # and one holding a step on every copy in turn (replayed for the bulk).
    singles = []
    with torch.cuda.stream(stream):
        for c in caches:
            step(c, stream)  # warm up outside capture
        stream.synchronize()
        for c in caches:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(c, stream)
            singles.append(g)
        macro = torch.cuda.CUDAGraph()
        with torch.cuda.graph(macro, stream=stream):
            for c in caches:
                step(c, stream)
    nc = len(caches)
    clk = Clocks(torch.cuda.current_device()).__enter__()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            singles[i % nc].replay()
        stream.synchronize()
        barrier()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h0 = time.perf_counter()
        t0.record(stream)
        for _ in range(args.steps // nc):
            macro.replay()
        for i in range(args.steps % nc):
            singles[i].replay()
        t1.record(stream)
        stream.synchronize()
        h1 = time.perf_counter()
        torch.cuda.synchronize()
        barrier()
        total_ms = t0.elapsed_time(t1)
        step_clocks = clk.summary(h0, h1)
        # the attention kernel alone, for the roofline: a CUDA graph of
        # back-to-back calls over the rotating cache copies, replayed for about
        # a tenth of a second with events around the replays (so the clock
        # samples fall inside); the average per call is the launch duration
        ng = 8 * nc
        ga = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ga, stream=stream):
            for i in range(ng):
                caches[i % nc].attention(q_dev, out, S, sm_scale, stream=stream.cuda_stream)
        for _ in range(3):
            ga.replay()
        stream.synchronize()
        reps = max(3, int(np.ceil(0.1 / max(1e-6, total_ms / 1e3 / args.steps * ng))))
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h2 = time.perf_counter()
        a0.record(stream)
        for _ in range(reps):
            ga.replay()
        a1.record(stream)
        stream.synchronize()
        h3 = time.perf_counter()
        attn_graph_ms = a0.elapsed_time(a1) / (reps * ng)
        attn_clocks = clk.summary(h2, h3)
        del ga
        # the same calls made one at a time with an event pair around each
        # (context: this adds the per-launch overhead of eager launches); the
        # stream first sleeps so the host can enqueue them ahead of the GPU
        n_attn = min(args.steps, 200)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_attn)]
        torch.cuda._sleep(int(2e8))
        for i in range(n_attn):
            evs[i][0].record(stream)
            caches[i % nc].attention(q_dev, out, S, sm_scale, stream=stream.cuda_stream)
            evs[i][1].record(stream)
        stream.synchronize()
        attn_ms = [a.elapsed_time(b) for a, b in evs]
        # the step's other call alone: quantizing the new token of every sequence
        qevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_attn)]
        torch.cuda._sleep(int(2e8))
        for i in range(n_attn):
            qevs[i][0].record(stream)
            caches[i % nc].quantize(knew_dev, vnew_dev, pos0=pos, stream=stream.cuda_stream)
            qevs[i][1].record(stream)
        stream.synchronize()
        token_ms = [a.elapsed_time(b) for a, b in qevs]
    clk.__exit__(None, None, None)
    torch.cuda.synchronize()
    # e2e: through the public API, host buffers: H2D of q and the new token,
    # both calls, D2H of the output, every step.  The step's inputs sit in one
    # pinned host buffer and move in one copy (q, k, v are views into it).
    nq, nk = q_dev.numel() * 4, knew_dev.numel() * 2
    host = torch.empty(nq + 2 * nk, dtype=torch.uint8).pin_memory()
    host[:nq].copy_(q_dev.cpu().view(torch.uint8).reshape(-1))
    host[nq:nq + nk].copy_(knew_dev.cpu().view(torch.uint8).reshape(-1))
    host[nq + nk:].copy_(vnew_dev.cpu().view(torch.uint8).reshape(-1))
    dev_in = torch.empty(nq + 2 * nk, dtype=torch.uint8, device="cuda")
    q_b = dev_in[:nq].view(torch.float32).view(q_dev.shape)
    k_b = dev_in[nq:nq + nk].view(knew_dev.dtype).view(knew_dev.shape)
    v_b = dev_in[nq + nk:].view(vnew_dev.dtype).view(vnew_dev.shape)
    dev_in.copy_(host)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    n_e2e = min(args.steps, 200)
    with torch.cuda.stream(stream):
        for i in range(3):
            caches[i % nc].quantize(k_b, v_b, pos0=pos, stream=stream.cuda_stream)
        stream.synchronize()
        e_t0, e_t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        wall0 = time.perf_counter()
        e_t0.record(stream)
        for i in range(n_e2e):
            c = caches[i % nc]
            dev_in.copy_(host, non_blocking=True)
            c.decode_step(k_b, v_b, q_b, out, S, sm_scale, stream=stream.cuda_stream)
            out_h.copy_(out, non_blocking=True)
        e_t1.record(stream)
        stream.synchronize()
        wall = time.perf_counter() - wall0
    e2e_ms = max(e_t0.elapsed_time(e_t1), wall * 1e3)
    for c in caches:
        c.check()
    bytes_h2d = host.numel()
    bytes_d2h = out_h.numel() * out_h.element_size()
    res = {
        "total_ms": total_ms, "attn_ms": attn_graph_ms, "attn_ms_eager": statistics.mean(attn_ms),
        "attn_ms_eager_median": statistics.median(attn_ms), "attn_calls": reps * ng,
        "clocks": step_clocks, "attn_clocks": attn_clocks, "copies": nc, "algo": ab, "kernel": "affine",
        "attn_timing": "CUDA graph of back-to-back calls over the cache copies, events around the replays",
        "e2e_tok_s": w.batch * n_e2e / (e2e_ms / 1e3), "h2d": bytes_h2d, "d2h": bytes_d2h,
        "prefill_ms": prefill_ms, "token_ms": statistics.mean(token_ms),
        "prefill_bytes": 2 * k_dev.numel() * k_dev.element_size() + sum(
            t.numel() * t.element_size() for t in caches[0].tensors.values() if t is not None),
    }
    for c in caches[1:]:
        c.detach()
    caches[0].close()
    return res


def run_qwen_long(args, S, rank):
    """Qwen3-8B-shaped long-context decode step at S tokens: dense key transform,
    99.9-percentile clipped 2-bit grid, no 16-bit regions."""
    import torch
    w = W.QWEN_LONG.with_(seq=S)
    k, v = W.make_kv(w)
    q = W.make_q(w)
    kn, vn = W.make_new_token(w)
    dev16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    k_dev, v_dev = dev16(k), dev16(v)
    del k, v
    r = run_gpu(args, w, w.bits, S, k_dev, v_dev, torch.from_numpy(q).cuda(), dev16(kn), dev16(vn), rank)
    del k_dev, v_dev
    torch.cuda.empty_cache()
    return w, r


def run_gpu_nuq(args, w):
    """KVQuant NUQ cache, prefilled: each step is one decode-attention call,
    rotating over cache copies larger than L2 (appends are checked by the tests;
    re-appending at the last position would not change what a step reads)."""
    import torch
    from quantized_decode_attention_gb300 import KVCache, make_config
    S = w.seq
    k, v = W.make_kv(w)
    q = W.make_q(w)
    f16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.float16)
    k_dev, v_dev, q_dev = f16(k), f16(v), torch.from_numpy(q).cuda()
    cfg = make_config(batch=w.batch, n_kv_heads=w.n_kv_heads, n_q_heads=w.n_q_heads, head_dim=w.head_dim,
                      max_seq=S, kv_dtype=w.kv_dtype, out_dtype=w.out_dtype, bits=w.bits, rot_k="none",
                      rot_v="none", mean_k=False, n_sink=w.n_sink, n_recent=w.n_recent, scheme="nuq",
                      lloyd_iters=w.extra.get("lloyd_iters", 8), outlier_frac=w.extra.get("outlier_frac", 0.01),
                      group_size_v=w.extra.get("group_size", 0), refit_k=w.extra.get("refit_interval", 0))
    L2 = torch.cuda.get_device_properties(0).L2_cache_size
    ab = nuq_algorithmic_bytes(w, S)
    copies = args.copies or max(3, int(np.ceil(3 * L2 / ab["total"])) + 1)
    stream = torch.cuda.Stream()
    base = KVCache.allocate(cfg, zero=False)
    with torch.cuda.stream(stream):
        base.quantize(k_dev, v_dev, pos0=0, stream=stream.cuda_stream)  # context and workspace
        stream.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        base.quantize(k_dev, v_dev, pos0=0, stream=stream.cuda_stream)
        p1.record(stream)
        stream.synchronize()
    prefill_ms = p0.elapsed_time(p1)
    base.check()
    caches = [base] + [base.clone_shared() for _ in range(copies - 1)]
    del k_dev, v_dev
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float16, device="cuda")
    sm_scale = w.head_dim ** -0.5
    with torch.cuda.stream(stream):
        for c in caches:
            c.attention(q_dev, out, S, sm_scale, stream=stream.cuda_stream)
        stream.synchronize()
        macro = torch.cuda.CUDAGraph()
        with torch.cuda.graph(macro, stream=stream):
            for c in caches:
                c.attention(q_dev, out, S, sm_scale, stream=stream.cuda_stream)
        nc = len(caches)
        reps = max(1, args.steps // nc)
        for _ in range(max(1, args.warmup // nc)):
            macro.replay()
        stream.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(reps):
            macro.replay()
        t1.record(stream)
        stream.synchronize()
        total_ms = t0.elapsed_time(t1)
        n_attn = min(args.steps, 200)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_attn)]
        torch.cuda._sleep(int(2e8))
        for i in range(n_attn):
            evs[i][0].record(stream)
            caches[i % nc].attention(q_dev, out, S, sm_scale, stream=stream.cuda_stream)
            evs[i][1].record(stream)
        stream.synchronize()
        attn_ms = [a.elapsed_time(b) for a, b in evs]
        # e2e through the public API: q H2D from pinned memory, output D2H
        q_h = q_dev.cpu().pin_memory()
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        q_b = q_dev.clone()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        wall0 = time.perf_counter()
        e0.record(stream)
        for i in range(n_attn):
            q_b.copy_(q_h, non_blocking=True)
            caches[i % nc].attention(q_b, out, S, sm_scale, stream=stream.cuda_stream)
            out_h.copy_(out, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
        e2e_ms = max(e0.elapsed_time(e1), (time.perf_counter() - wall0) * 1e3)
    for c in caches:
        c.check()
    steps = reps * nc
    res = {"total_ms": total_ms, "steps": steps, "attn_ms": total_ms / steps, "attn_ms_eager": statistics.mean(attn_ms),
           "attn_ms_eager_median": statistics.median(attn_ms), "attn_calls": steps,
           "attn_timing": "CUDA graph of back-to-back calls over the cache copies", "algo": ab, "copies": nc,
           "kernel": "generic",
           "prefill_ms": prefill_ms, "e2e_tok_s": w.batch * n_attn / (e2e_ms / 1e3)}
    for c in caches[1:]:
        c.detach()
    caches[0].close()
    return res


def run_gpu_dquant(args, w):
    """D-Quant cache, prefilled: each step is one decode-attention call,
    rotating over cache copies larger than L2.  An append at the last position
    would flush a whole 128-slot window on every step, which real decoding does
    once every 128 tokens, so appends are checked by the tests, not timed here."""
    import torch
    from quantized_decode_attention_gb300 import KVCache, make_config
    S = w.seq
    k, v = W.make_kv(w)
    q = W.make_q(w)
    b16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    k_dev, v_dev, q_dev = b16(k), b16(v), torch.from_numpy(q).cuda()
    del k, v
    e = w.extra
    cfg = make_config(batch=w.batch, n_kv_heads=w.n_kv_heads, n_q_heads=w.n_q_heads, head_dim=w.head_dim,
                      max_seq=S, kv_dtype=w.kv_dtype, out_dtype=w.out_dtype, rot_k=w.rot_k, rot_v=w.rot_v,
                      mean_k=w.mean_k, n_sink=w.n_sink, n_recent=w.n_recent, scheme="rans",
                      levels_k=e["levels_k"], levels_v=e["levels_v"], container_k=e["container_k"],
                      container_v=e["container_v"], rans_alpha=e["alpha"])
    L2 = torch.cuda.get_device_properties(0).L2_cache_size
    ab = dquant_algorithmic_bytes(w, S)
    copies = args.copies or max(3, int(np.ceil(3 * L2 / ab["total"])) + 1)
    stream = torch.cuda.Stream()
    base = KVCache.allocate(cfg, zero=False)
    with torch.cuda.stream(stream):
        base.quantize(k_dev, v_dev, pos0=0, stream=stream.cuda_stream)  # context, scratch
        stream.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        base.quantize(k_dev, v_dev, pos0=0, stream=stream.cuda_stream)
        p1.record(stream)
        stream.synchronize()
    prefill_ms = p0.elapsed_time(p1)
    base.check()
    del k_dev, v_dev
    caches = [base] + [base.clone_shared() for _ in range(copies - 1)]
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    sm_scale = w.head_dim ** -0.5
    nc = len(caches)
    steps = max(nc, min(args.steps, 60))
    with torch.cuda.stream(stream):
        for i in range(max(3, nc)):
            caches[i % nc].attention(q_dev, out, S, sm_scale, stream=stream.cuda_stream)
        stream.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(int(2e8))
        t0.record(stream)
        for i in range(steps):
            evs[i][0].record(stream)
            caches[i % nc].attention(q_dev, out, S, sm_scale, stream=stream.cuda_stream)
            evs[i][1].record(stream)
        t1.record(stream)
        stream.synchronize()
        total_ms = t0.elapsed_time(t1)
        attn_ms = [a.elapsed_time(b) for a, b in evs]
        q_h = q_dev.cpu().pin_memory()
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        q_b = q_dev.clone()
        n_e2e = min(steps, 20)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        wall0 = time.perf_counter()
        e0.record(stream)
        for i in range(n_e2e):
            q_b.copy_(q_h, non_blocking=True)
            caches[i % nc].attention(q_b, out, S, sm_scale, stream=stream.cuda_stream)
            out_h.copy_(out, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
        e2e_ms = max(e0.elapsed_time(e1), (time.perf_counter() - wall0) * 1e3)
    for c in caches:
        c.check()
    res = {"total_ms": total_ms, "steps": steps, "attn_ms": statistics.mean(attn_ms),
           "attn_ms_eager": statistics.mean(attn_ms), "attn_ms_eager_median": statistics.median(attn_ms),
           "attn_calls": steps, "attn_timing": "event pair around each call (calls of milliseconds)", "algo": ab,
           "kernel": "rans",
           "copies": nc, "prefill_ms": prefill_ms, "e2e_tok_s": w.batch * n_e2e / (e2e_ms / 1e3)}
    for c in caches[1:]:
        c.detach()
    caches[0].close()
    return res


def _oracle_unit(args):
    """One (batch, KV head) unit through the oracle, in a worker process: the
    bulk quantize of its first S - 1 tokens (prefill), then the decode step the
    GPU times -- token S - 1 appended on the frozen prefill key mean, and fp64
    decode attention over all S tokens.  Returns the two host times."""
    w1, S, ku, vu, qu = args
    import oracle
    t0 = time.perf_counter()
    qk0 = oracle.quantize_tensor(w1, ku[:, :, :S - 1], True, S - 1)
    qv0 = oracle.quantize_tensor(w1, vu[:, :, :S - 1], False, S - 1)
    t1 = time.perf_counter()
    qk1 = oracle.quantize_tensor(w1, ku[:, :, S - 1:], True, S, mu_frozen=qk0.mu, pos0=S - 1)
    qv1 = oracle.quantize_tensor(w1, vu[:, :, S - 1:], False, S, pos0=S - 1)
    cat = lambda a, b: oracle.QuantTensor(*(np.concatenate([x, y], 2) for x, y in
                                            ((a.codes, b.codes), (a.s, b.s), (a.o, b.o))), a.mu,
                                          np.concatenate([a.xhat, b.xhat], 2))
    oracle.attention(w1, qu, ku, vu, S, cat(qk0, qk1), cat(qv0, qv1))
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def _oracle_warm(_):
    import oracle
    oracle.lib()
    return os.getpid()


_POOL = None


def oracle_pool():
    """Worker processes for the oracle, started with spawn (safe next to CUDA),
    one per host core this process may run on."""
    global _POOL
    if _POOL is None:
        import concurrent.futures as cf
        import multiprocessing as mp
        import oracle
        oracle.build()
        n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        _POOL = (cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn")), n)
        list(_POOL[0].map(_oracle_warm, range(4 * n)))   # start and load every worker before timing
    return _POOL


FEASIBLE_BUDGETS = (1.0, 1.25, 1.5, 1.75, 2.0, 2.25, 2.5, 2.75, 3.0, 3.5, 4.0)


def feasible_alphabet(n: int = 1024, budgets=FEASIBLE_BUDGETS) -> list:
    """D-Quant App. C (Fig. 6 left): the largest number of levels (2..16) whose
    cheapest stream still fits a container of b bits per value of payload plus the
    32-bit state, by the library's own symbol model (dq_kv_sizes refuses an
    infeasible one), against the 2^floor(b) levels of fixed-width coding at that
    rate.  Host only: no kernel runs."""
    from quantized_decode_attention_gb300 import DQError, kv_sizes, make_config
    H = n // 128
    out = []
    for b in budgets:
        C = int(np.ceil((b * n + 32) / 8))
        best = None
        for M in range(2, 17):
            cfg = make_config(batch=1, n_kv_heads=H, n_q_heads=4 * H, head_dim=128, max_seq=256, scheme="rans",
                              rot_k="hadamard", rot_v="none", mean_k=True, levels_k=M, levels_v=2,
                              container_k=C, container_v=C)
            try:
                kv_sizes(cfg)
                best = M
            except DQError:
                pass
        out.append({"payload_bits_per_value": b, "container_bytes": C, "entropy_coded_levels": best,
                    "fixed_width_levels": 2 ** int(b)})
    return out


# D-Quant Sec. 5.4 (Fig. 4) varies one setting at a time around the 8 / 6-level,
# 331 / 231-byte point: the alphabets at that storage, the storage at 8 / 6
# levels, and the key/value split of the same total.  The pages score each
# setting by long-context task accuracy of a trained model; on synthetic data the
# measurable counterpart is how far the decode-attention output moves from exact
# attention over the unquantized tokens.
ABL_LEVELS = ((4, 6), (6, 6), (8, 6), (10, 6), (12, 6), (16, 6), (8, 3), (8, 4), (8, 8), (8, 10), (8, 16))
# key / value containers in the 331 : 231 proportion: about 1.6, 1.96, 2.26, 2.6
# and 3.0 bits per value with the fp16 (s, o) and the INT8 window means
ABL_BUDGETS = ((232, 162), (286, 200), (331, 231), (383, 267), (443, 309))
ABL_KEY_BYTES = (256, 281, 306, 331, 356, 381)  # key container; the value container gets 562 minus it
ABL_PAIR_BYTES = 331 + 231


def exact_attention(q: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, kv_dtype: str) -> np.ndarray:
    """softmax(q K^T / sqrt(d)) V in fp64 over the unquantized 16-bit tokens.
    q [B, Hq, d] fp32; k_bits, v_bits [B, Hkv, S, d] bf16 / fp16 bit patterns;
    query head h reads KV head floor(h Hkv / Hq).  Returns [B, Hq, d] fp64."""
    def f64(bits):
        u = np.ascontiguousarray(bits, dtype=np.uint16)
        if kv_dtype == "bf16":
            return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        return u.view(np.float16).astype(np.float64)
    K, V = f64(k_bits), f64(v_bits)
    B, Hq, d = q.shape
    G = Hq // K.shape[1]
    qg = q.astype(np.float64).reshape(B, K.shape[1], G, d)
    s = np.einsum("bhgd,bhtd->bhgt", qg, K) / np.sqrt(d)
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    p /= p.sum(axis=-1, keepdims=True)
    return np.einsum("bhgt,bhtd->bhgd", p, V).reshape(B, Hq, d)


def dquant_attention_output(w, k_dev, v_dev, q_dev, levels_k, levels_v, ck, cv):
    """The library's fp32 decode-attention output over a D-Quant cache of w's shape,
    prefilled with every token, at the given alphabets and containers; None when
    the symbol model cannot fit a stream into its container."""
    import torch
    from quantized_decode_attention_gb300 import DQError, KVCache, kv_sizes, make_config
    cfg = make_config(batch=w.batch, n_kv_heads=w.n_kv_heads, n_q_heads=w.n_q_heads, head_dim=w.head_dim,
                      max_seq=w.seq, kv_dtype=w.kv_dtype, out_dtype="f32", rot_k=w.rot_k, rot_v=w.rot_v,
                      mean_k=w.mean_k, n_sink=w.n_sink, n_recent=w.n_recent, scheme="rans",
                      levels_k=levels_k, levels_v=levels_v, container_k=ck, container_v=cv,
                      rans_alpha=w.extra["alpha"])
    try:
        kv_sizes(cfg)
    except DQError as e:
        if e.name == "DQ_EINFEASIBLE":
            return None
        raise
    cache = KVCache.allocate(cfg)
    try:
        cache.quantize(k_dev, v_dev, pos0=0)
        out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
        cache.attention(q_dev, out, w.seq)
        torch.cuda.synchronize()
        cache.check()
        return out.cpu().numpy().astype(np.float64)
    finally:
        cache.close()


def dquant_ablation(batch: int = 4, quantized: int = 2048, levels=ABL_LEVELS, budgets=ABL_BUDGETS,
                    key_bytes=ABL_KEY_BYTES) -> dict:
    """D-Quant Sec. 5.4 (Fig. 4) on the D-Quant workload's synthetic tokens (batch
    `batch`, `quantized` quantized tokens plus the 128-token 16-bit window): for each
    setting, the relative L2 distance and the largest absolute difference between
    the library's decode-attention output and exact fp64 attention over the same
    unquantized tokens.  Settings whose streams cannot fit are marked infeasible."""
    import torch
    base = W.DQUANT.with_(batch=batch, seq=quantized + W.DQUANT.n_recent)
    k, v = W.make_kv(base)
    q = W.make_q(base)
    ref = exact_attention(q, k, v, base.kv_dtype)
    dev16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    k_dev, v_dev, q_dev = dev16(k), dev16(v), torch.from_numpy(q).cuda()

    def case(mk, mv, ck, cv):
        e = {**base.extra, "levels_k": mk, "levels_v": mv, "container_k": ck, "container_v": cv}
        row = {"levels_k": mk, "levels_v": mv, "container_k": ck, "container_v": cv,
               "bits_per_value": round(W.dquant_bits_per_value(base.with_(extra=e)), 3)}
        out = dquant_attention_output(base, k_dev, v_dev, q_dev, mk, mv, ck, cv)
        if out is None:
            row["infeasible"] = True
        else:
            row["rel_l2_err"] = float(np.linalg.norm(out - ref) / np.linalg.norm(ref))
            row["max_abs_err"] = float(np.abs(out - ref).max())
        return row

    res = {"workload": f"{base.name}: batch {batch}, {quantized} quantized + {base.n_recent} 16-bit tokens, "
                       f"{base.n_kv_heads} KV heads (1024-value streams)",
           "levels": [case(mk, mv, 331, 231) for mk, mv in levels],
           "budget": [case(8, 6, ck, cv) for ck, cv in budgets],
           "kv_split": [case(8, 6, ck, ABL_PAIR_BYTES - ck) for ck in key_bytes]}
    del k_dev, v_dev, q_dev
    torch.cuda.empty_cache()
    return res


def codes_of_records(rec: np.ndarray, bits: int) -> np.ndarray:
    """Every code held in fixed-stride records (uint8 [..., record bytes]; key
    rows or value pair records), in no particular order.  Records are
    little-endian 32-bit words.  At 2 and 4 bits each 16-bit half holds 16/b
    fields.  At 3 bits, a 2-bit plane of R/16 words comes first (the 2-bit
    layout), then a 1-bit plane: field i of half h keeps its low two bits at
    bit 16h + 2(i mod 8) of plane word i/8, and its high bit at bit
    16h + P(i mod 16) of 1-bit-plane word i/16, P(f) = 2f + 2 for f <= 6, 0 for
    f = 7, 2f - 13 for 8 <= f <= 14, 1 for f = 15."""
    w = np.ascontiguousarray(rec, dtype=np.uint8)
    w = w.reshape(-1, w.shape[-1]).view("<u4").astype(np.int64)
    if bits in (2, 4):
        sh = np.array([16 * h + bits * f for h in (0, 1) for f in range(16 // bits)])
        return ((w[:, :, None] >> sh) & ((1 << bits) - 1)).ravel()
    R = w.shape[1] * 32 // 3                  # codes per record
    i = np.arange(R // 2)
    out = []
    for h in (0, 1):
        lo = (w[:, i >> 3] >> (16 * h + 2 * (i & 7))) & 3
        f = i & 15
        p1 = np.where(f <= 6, 2 * f + 2, np.where(f == 7, 0, np.where(f == 15, 1, 2 * f - 13)))
        hi = (w[:, R // 16 + (i >> 4)] >> (16 * h + p1)) & 1
        out.append(lo | (hi << 2))
    return np.concatenate(out, axis=1).ravel()


def coding_stats(hist: np.ndarray, p: np.ndarray) -> dict:
    """D-Quant Sec. 3 (Table 1) for a symbol histogram over M levels against a model p:
    the empirical entropy H (bits per value), Coding Gain = log2 M - H (what entropy
    coding could save over fixed-width codes) and Normal Gap = CE - H (the extra
    rate of coding with p instead of the empirical frequencies; CE the cross-entropy)."""
    q = np.asarray(hist, dtype=np.float64)
    q = q / q.sum()
    nz = q > 0
    H = float(-(q[nz] * np.log2(q[nz])).sum())
    CE = float(-(q[nz] * np.log2(np.asarray(p, dtype=np.float64)[nz])).sum())
    return {"entropy": H, "coding_gain": float(np.log2(len(q))) - H, "normal_gap": CE - H}


def hadamard_rows(x: np.ndarray) -> np.ndarray:
    """Rows of x times the normalized Sylvester Hadamard matrix, in fp64."""
    d = x.shape[-1]
    Hn = np.array([[1.0]])
    while Hn.shape[0] < d:
        Hn = np.block([[Hn, Hn], [Hn, -Hn]])
    return np.asarray(x, dtype=np.float64) @ (Hn / np.sqrt(d))


def preprocessing_row(tensor: str, name: str, x: np.ndarray, xhat: np.ndarray, codes_buf: np.ndarray,
                      record_bytes: int, p: np.ndarray) -> dict:
    """One row of the Table 1 analogue: x the tokens in the quantizer's space (fp64),
    xhat their dequantized values, codes_buf a cache's whole code buffer (flat
    uint8, records of record_bytes back to back), p the model of the 8 levels."""
    err = x - xhat
    codes = codes_of_records(np.asarray(codes_buf, dtype=np.uint8).reshape(-1, record_bytes), 3)
    row = {"tensor": tensor, "preprocessing": name, "nmse": float((err * err).sum() / (x * x).sum())}
    row.update(coding_stats(np.bincount(codes, minlength=8), p))
    return row


def preprocessing_effect(batch: int = 2, seq: int = 2048) -> dict:
    """D-Quant Sec. 3 (Table 1) on the Llama-shaped synthetic keys (channel means
    and outlier channels) and values: each token's head vector on an 8-level
    min/max grid (the library's 3-bit affine quantizer, fp32 s and o), raw, after
    the Hadamard rotation, and (keys) after also removing the channel mean.  Per
    row: NMSE of the dequantized values (in the quantizer's space, against the
    power of the rotated tokens), the codes' empirical entropy, Coding Gain and
    Normal Gap against the library's analytic order-statistics model for d values."""
    import torch
    from quantized_decode_attention_gb300 import KVCache, make_config, symbol_probs
    if seq % 2:
        raise ValueError("seq must be even (value records hold token pairs)")
    w = W.LLAMA.with_(batch=batch, seq=seq)
    B, H, d = w.batch, w.n_kv_heads, w.head_dim
    k, v = W.make_kv(w)
    p = np.array(symbol_probs(d, 8))
    dev16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    k_dev, v_dev = dev16(k), dev16(v)
    xs = {0: W.bf16_bits_to_f32(k).astype(np.float64), 1: W.bf16_bits_to_f32(v).astype(np.float64)}
    rows = []
    for name, rot, mean, values in (("raw", "none", False, True), ("hadamard", "hadamard", False, True),
                                    ("hadamard+mean", "hadamard", True, False)):
        cfg = make_config(batch=B, n_kv_heads=H, n_q_heads=w.n_q_heads, head_dim=d, max_seq=seq, kv_dtype="bf16",
                          meta_dtype="f32", out_dtype="f32", bits=3, rot_k=rot, rot_v=rot, mean_k=mean,
                          n_sink=0, n_recent=0)
        cache = KVCache.allocate(cfg)
        try:
            cache.quantize(k_dev, v_dev, pos0=0)
            xh = torch.empty((B, H, seq, d), dtype=torch.float32, device="cuda")
            for which in ((0, 1) if values else (0,)):
                cache.dequantize(which, 0, seq, xh)
                torch.cuda.synchronize()
                cache.check()
                x = hadamard_rows(xs[which]) if rot == "hadamard" else xs[which]
                rec = 3 * d // 8 if which == 0 else 3 * d // 4   # key row / value pair record
                n_rec = seq if which == 0 else seq // 2               # records written per unit
                buf = cache.tensors["codes_k" if which == 0 else "codes_v"].cpu().numpy()
                buf = buf.reshape(B * H, -1, rec)[:, :n_rec]          # [unit][slot capacity][record]
                rows.append(preprocessing_row("k" if which == 0 else "v", name, x,
                                              xh.cpu().numpy().astype(np.float64), buf, rec, p))
        finally:
            cache.close()
    del k_dev, v_dev
    torch.cuda.empty_cache()
    return {"workload": f"{w.name}: batch {batch}, {seq} tokens, {H} KV heads, d {d}; 8 levels per token and head",
            "model": [round(x, 6) for x in p.tolist()], "rows": rows}


def grid_ablation(batch: int = 2, seq: int = 2048) -> dict:
    """The grid comparison of "WUSH-KV" (evaluation: the quantizer held fixed,
    relative squared Frobenius reconstruction error, keys and values quantized
    separately, no full-precision windows), with the transform held fixed
    instead: per token and head on the normalized Hadamard rotation, the
    min/max grid, the percentile clip of the pages' serving setting (kappa 0.96
    for keys, 0.92 for values) and the QuEST grid, at 2, 3 and 4 bits, through
    the library (quantize, then dequantize in the rotated space).  Data: the
    Llama-shaped synthetic keys and values, and the Qwen-shaped correlated keys."""
    import torch
    from quantized_decode_attention_gb300 import KVCache, make_config
    out = []
    dev16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    for w0 in (W.LLAMA, W.QWEN_LONG):
        w = w0.with_(batch=batch, seq=seq)
        B, H, d = w.batch, w.n_kv_heads, w.head_dim
        k, v = W.make_kv(w)
        k_dev, v_dev = dev16(k), dev16(v)
        xr = {0: hadamard_rows(W.bf16_bits_to_f32(k).astype(np.float64)),
              1: hadamard_rows(W.bf16_bits_to_f32(v).astype(np.float64))}
        for bits in (2, 3, 4):
            row = {"data": w0.name, "bits": bits}
            for gname, kw in (("minmax", {}), ("clip", {"clip_k": 0.96, "clip_v": 0.92}),
                              ("quest", {"grid_k": "quest"})):
                cfg = make_config(batch=B, n_kv_heads=H, n_q_heads=w.n_q_heads, head_dim=d, max_seq=seq,
                                  kv_dtype="bf16", meta_dtype="f16", out_dtype="f32", bits=bits, rot_k="hadamard",
                                  rot_v="hadamard", mean_k=False, n_sink=0, n_recent=0, **kw)
                cache = KVCache.allocate(cfg)
                try:
                    cache.quantize(k_dev, v_dev, pos0=0)
                    xh = torch.empty((B, H, seq, d), dtype=torch.float32, device="cuda")
                    for which, nm in ((0, "k"), (1, "v")):
                        cache.dequantize(which, 0, seq, xh)
                        torch.cuda.synchronize()
                        e = xh.cpu().numpy().astype(np.float64) - xr[which]
                        row[f"{nm}_{gname}"] = round(float(np.sum(e * e) / np.sum(xr[which] ** 2)), 5)
                    cache.check()
                finally:
                    cache.close()
            out.append(row)
        del k_dev, v_dev
        torch.cuda.empty_cache()
    return {"rows": out, "workload": f"batch {batch}, {seq} tokens, 8 KV heads, d 128; fp16 s and o"}


def drift_statistics(batch: int = 2, seq: int = 1024) -> dict:
    """D-Quant App. C ("drift makes only sparse, local corrections"): the share
    of coded symbols that drift moved off the nearest level of their stream's
    final grid, and the largest move, counted by the library while it encodes
    the D-Quant-shaped synthetic cache (8 / 6 levels in 331 / 231 bytes and at
    1.96 bits per value)."""
    import torch
    from quantized_decode_attention_gb300 import KVCache, make_config
    rows = []
    for D in (W.DQUANT, W.DQUANT_196):
        w = D.with_(batch=batch, seq=seq)
        e = w.extra
        k, v = W.make_kv(w)
        dev16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
        cfg = make_config(batch=w.batch, n_kv_heads=w.n_kv_heads, n_q_heads=w.n_q_heads, head_dim=w.head_dim,
                          max_seq=seq, kv_dtype=w.kv_dtype, out_dtype=w.out_dtype, rot_k=w.rot_k, rot_v=w.rot_v,
                          mean_k=w.mean_k, n_sink=w.n_sink, n_recent=w.n_recent, scheme="rans",
                          levels_k=e["levels_k"], levels_v=e["levels_v"], container_k=e["container_k"],
                          container_v=e["container_v"], rans_alpha=e["alpha"])
        cache = KVCache.allocate(cfg)
        try:
            cache.quantize(dev16(k), dev16(v), pos0=0)
            st = cache.drift_stats()
            cache.check()
        finally:
            cache.close()
        rows.append({"config": f"k{e['levels_k']}x{e['container_k']}-v{e['levels_v']}x{e['container_v']}",
                     "k_changed_frac": round(st["k_changed"] / max(1, st["k_coded"]), 5),
                     "k_max_move": st["k_max_move"],
                     "v_changed_frac": round(st["v_changed"] / max(1, st["v_coded"]), 5),
                     "v_max_move": st["v_max_move"], "symbols": st["k_coded"] + st["v_coded"]})
    return {"rows": rows, "workload": f"batch {batch}, {seq} tokens, 8 KV heads, d 128 (synthetic)"}


def cpu_baseline(w, bits, S, budget_s, k, v, q):
    """The oracle as it stands, timed on this host's cores, one worker process
    per core, a unit (sequence, KV head) per worker at a time: per unit the bulk
    quantize of S - 1 tokens and then the decode step (one-token append + fp64
    attention over S tokens), each timed inside the worker.  A wave's phase time
    is its slowest worker's; as many units as fit the budget, extrapolated to
    the full batch.  Reports decode tokens/s (the step's metric) and bulk
    quantize GB/s (16-bit K and V read + cache bytes written, as on the GPU)."""
    pool, n = oracle_pool()
    wb = w.with_(bits=bits)
    w1 = wb.with_(batch=1, n_kv_heads=1, n_q_heads=w.group)
    units = [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)]
    done, t_quant, t_step = 0, 0.0, 0.0
    t0 = time.perf_counter()
    while done < len(units) and time.perf_counter() - t0 <= budget_s:
        wave = units[done:done + n]
        jobs = [(w1, S, k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], q[b:b + 1, h * w.group:(h + 1) * w.group])
                for (b, h) in wave]
        times = list(pool.map(_oracle_unit, jobs))
        t_quant += max(t[0] for t in times)
        t_step += max(t[1] for t in times)
        done += len(wave)
    scale = len(units) / done
    per_call = t_step * scale
    unit_bytes = 2 * (S - 1) * w.head_dim * 2 + algorithmic_bytes(wb, bits, S)["total"] / len(units)
    qgbs = unit_bytes * done / t_quant / 1e9
    return {"value": w.batch / per_call, "unit": "tokens/s", "cores": n, "kind": "oracle",
            "quantize_gbs": round(qgbs, 3),
            "sample": f"{done} of {len(units)} (sequence, kv-head) units in waves of {n} worker processes; per "
                      f"unit the oracle's bulk quantize of {S - 1} tokens (GB/s: 16-bit K, V read + cache "
                      f"written) and its decode step: token {S - 1} appended on the frozen key mean + fp64 "
                      f"attention over {S} tokens for {w.group} heads; decode time extrapolated to one full call"}


def cfg_of(w: W.Workload, max_seq: int | None = None):
    """The library config of a workload."""
    from quantized_decode_attention_gb300 import make_config
    e = w.extra
    return make_config(batch=w.batch, n_kv_heads=w.n_kv_heads, n_q_heads=w.n_q_heads, head_dim=w.head_dim,
                       max_seq=max_seq or w.seq, kv_dtype=w.kv_dtype, meta_dtype=w.meta_dtype, out_dtype=w.out_dtype,
                       bits=w.bits, rot_k=w.rot_k, rot_v=w.rot_v, mean_k=w.mean_k, clip_k=w.clip, clip_v=w.clip,
                       grid_k=w.grid, n_sink=w.n_sink, n_recent=w.n_recent, scheme=w.scheme,
                       lloyd_iters=e.get("lloyd_iters", 8), outlier_frac=e.get("outlier_frac", 0.01),
                       group_size_v=e.get("group_size", 0), refit_k=e.get("refit_interval", 0),
                       levels_k=e.get("levels_k", 8), levels_v=e.get("levels_v", 6),
                       container_k=e.get("container_k", 331), container_v=e.get("container_v", 231),
                       rans_alpha=e.get("alpha", 1.4))


def profile_attention(args):
    """A short run for a profiler to capture: one cache (the Llama-shaped affine
    cache at args.bits, the KVQuant NUQ cache, or the D-Quant cache at args.profile_batch),
    prefilled once, then args.warmup + args.steps decode-attention calls on one
    stream.  Nothing is timed here."""
    import torch
    import __graft_entry__
    from quantized_decode_attention_gb300 import KVCache
    __graft_entry__.build()
    if args.profile_kind == "affine":
        w = W.LLAMA.with_(bits=args.bits)
    elif args.profile_kind == "nuq":
        w = W.NUQ
    elif args.profile_kind == "nuq_gr":
        w = NUQ_GROUP_REFIT
    else:
        w = W.DQUANT.with_(batch=args.profile_batch)
    S = w.seq
    k, v = W.make_kv(w)
    dt = torch.float16 if w.kv_dtype == "f16" else torch.bfloat16
    dev16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(dt)
    q_dev = torch.from_numpy(W.make_q(w)).cuda()
    cache = KVCache.allocate(cfg_of(w), zero=False)
    cache.quantize(dev16(k), dev16(v), pos0=0)
    torch.cuda.synchronize()
    del k, v
    torch.cuda.empty_cache()  # only the cache stays on the device
    odt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[w.out_dtype]
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=odt, device="cuda")
    for _ in range(args.warmup + args.steps):
        cache.attention(q_dev, out, S, w.head_dim ** -0.5)
    torch.cuda.synchronize()
    cache.check()
    cache.close()
    print(json.dumps({"profile_attn": w.name, "kind": args.profile_kind, "bits": w.bits,
                      "calls": args.warmup + args.steps}))


def main():
    args = parse()
    if args.profile_attn:
        profile_attention(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    w = W.LLAMA.with_(bits=args.bits)
    S = w.seq

    if args.impl == "reference":
        if rank != 0:
            return
        k, v = W.make_kv(w)
        q = W.make_q(w)
        steps = []
        for i in range(args.warmup + args.steps):
            r = cpu_baseline(w, args.bits, S, args.cpu_seconds / max(1, args.steps + args.warmup), k, v, q)
            if i >= args.warmup:
                steps.append(r["value"])
        val = statistics.mean(steps)
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "dtype": "f64",
                "data": "synthetic", "config": {"workload": w.name, "batch": w.batch, "seq_len": S, "bits": args.bits},
                "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": oracle_pool()[1], "kind": "oracle",
                                 "sample": "each step: as many (sequence, kv-head) units as fit its time share, "
                                           "in waves of one worker process per host core; per unit the oracle's "
                                           "decode step (one-token append on the frozen key mean + fp64 "
                                           "attention over the pre-quantized cache), extrapolated to a full "
                                           "decode call"},
                "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "vs_baseline": None}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    import __graft_entry__
    __graft_entry__.build()
    # inputs (seeded), uploaded once; bf16 bit patterns
    k, v = W.make_kv(w)
    q = W.make_q(w)
    kn, vn = W.make_new_token(w)
    dev16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    k_dev, v_dev, q_dev = dev16(k), dev16(v), torch.from_numpy(q).cuda()
    kn_dev, vn_dev = dev16(kn), dev16(vn)
    res = run_gpu(args, w, args.bits, S, k_dev, v_dev, q_dev, kn_dev, vn_dev, rank)
    variants = {}
    for vb in [int(x) for x in args.variants.split(",") if x.strip()]:
        if vb == args.bits:
            continue
        r = run_gpu(args, w.with_(bits=vb), vb, S, k_dev, v_dev, q_dev, kn_dev, vn_dev, rank)
        variants[f"{vb}bit"] = r
    # context: the same decode step over an unquantized bf16 cache (every token a
    # 16-bit slot of the library's own 16-bit path), the pages' "vs BF16" point
    bf16 = None
    if not args.no_bf16:
        wb = W.LLAMA.with_(n_sink=S, n_recent=0, mean_k=False, rot_k="none", rot_v="none")
        bf16 = run_gpu(args, wb, wb.bits, S, k_dev, v_dev, q_dev, kn_dev, vn_dev, rank)
        bf16["kernel"] = "generic"  # every token a 16-bit slot: the older kernel's CTA-wide ring serves it
        torch.cuda.empty_cache()
    del k_dev, v_dev
    nuq = None if args.no_nuq else run_gpu_nuq(args, W.NUQ)
    nuq_gr = None if args.no_nuq else run_gpu_nuq(args, NUQ_GROUP_REFIT)
    dqrs = [] if args.no_dquant else [(D, run_gpu_dquant(args, D)) for D in (W.DQUANT, W.DQUANT_196)]
    qwen = [run_qwen_long(args, int(x), rank) for x in args.qwen.split(",") if x.strip()]

    ms_step, value = aggregate(res["total_ms"], args.steps, w.batch, world)
    peak, peak_kind = peaks()
    def roof(r, bits):
        achieved = r["algo"]["total"] / (r["attn_ms"] / 1e3) / 1e9
        d = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
             "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
             "traffic": traffic_for(r.get("kernel", "affine"), bits), "algorithmic_bytes": r["algo"]["total"],
             "attn_us": round(r["attn_ms"] * 1e3, 2), "calls_timed": r["attn_calls"], "timing": r["attn_timing"],
             "attn_us_eager": round(r["attn_ms_eager"] * 1e3, 2),
             "attn_us_eager_median": round(r["attn_ms_eager_median"] * 1e3, 2)}
        if r.get("attn_clocks"):
            d["clocks"] = r["attn_clocks"]
        return d

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16-mma/f32-acc (bf16 in/out)", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads,
                   "head_dim": w.head_dim, "seq_len": S, "bits": args.bits, "n_sink": w.n_sink,
                   "n_recent": w.n_recent, "parallelism": f"replicas{world}",
                   "l2": f"{res['copies']} cache copies rotated per step (> L2)",
                   "step": "dq_decode_step: append 1 new token/seq + decode attention (one launch), CUDA graph per step"},
        "roofline": roof(res, args.bits),
        "clocks": res["clocks"],
        "e2e": {"value": round(res["e2e_tok_s"], 1), "unit": "tokens/s", "h2d_bytes_per_step": res["h2d"],
                "d2h_bytes_per_step": res["d2h"],
                "how": "eager dq_decode_step calls: one pinned-host H2D copy of q and the new token, output D2H"},
        "gpu_launches": args.steps,
        "quantize": {"token_us": round(res["token_ms"] * 1e3, 2), "prefill_us": round(res["prefill_ms"] * 1e3, 1),
                     "prefill_gbs": round(res["prefill_bytes"] / (res["prefill_ms"] / 1e3) / 1e9, 1),
                     "prefill_bytes": res["prefill_bytes"],
                     "how": "token: dq_quantize_kv of one new token per sequence alone (CUDA events); prefill: "
                            "the whole cache from 16-bit K and V, bytes = inputs read + cache buffers written"},
        "variants": {k2: {"value": round(w.batch / (r["total_ms"] / args.steps / 1e3), 1),
                          "ms_per_step": round(r["total_ms"] / args.steps, 5), "roofline": roof(r, int(k2[0])),
                          "e2e_tok_s": round(r["e2e_tok_s"], 1)} for k2, r in variants.items()},
    }
    if nuq is not None:
        line["variants"][f"{W.NUQ.name}-{W.NUQ.bits}bit"] = {
            "value": round(W.NUQ.batch / (nuq["total_ms"] / nuq["steps"] / 1e3), 1),
            "ms_per_step": round(nuq["total_ms"] / nuq["steps"], 5),
            "roofline": roof(nuq, "nuq"), "e2e_tok_s": round(nuq["e2e_tok_s"], 1),
            "prefill_ms": round(nuq["prefill_ms"], 3),
            "config": {"batch": W.NUQ.batch, "q_heads": W.NUQ.n_q_heads, "kv_heads": W.NUQ.n_kv_heads,
                       "head_dim": W.NUQ.head_dim, "seq_len": W.NUQ.seq, "bits": W.NUQ.bits,
                       "n_sink": W.NUQ.n_sink, "outlier_frac": 0.01, "lloyd_iters": 8,
                       "l2": f"{nuq['copies']} cache copies rotated per step (> L2)",
                       "step": "decode attention over a prefilled cache, CUDA graph over the copies"}}
    if nuq_gr is not None:
        wg = NUQ_GROUP_REFIT
        line["variants"][f"{wg.name}-{wg.bits}bit-group32-refit128"] = {
            "value": round(wg.batch / (nuq_gr["total_ms"] / nuq_gr["steps"] / 1e3), 1),
            "ms_per_step": round(nuq_gr["total_ms"] / nuq_gr["steps"], 5),
            "roofline": roof(nuq_gr, "nuq_g32_r128"), "e2e_tok_s": round(nuq_gr["e2e_tok_s"], 1),
            "prefill_ms": round(nuq_gr["prefill_ms"], 3),
            "config": {"batch": wg.batch, "q_heads": wg.n_q_heads, "kv_heads": wg.n_kv_heads,
                       "head_dim": wg.head_dim, "seq_len": wg.seq, "bits": wg.bits, "n_sink": wg.n_sink,
                       "n_recent": wg.n_recent, "outlier_frac": 0.01, "lloyd_iters": 8,
                       "group_size_v": 32, "refit_interval_k": 128,
                       "l2": f"{nuq_gr['copies']} cache copies rotated per step (> L2)",
                       "step": "decode attention over a prefilled cache (value tables per 32 channels, key "
                               "tables per 128-slot block), CUDA graph over the copies"}}
    for wq, r in qwen:
        line["variants"][f"{wq.name}-s{wq.seq}-{wq.bits}bit"] = {
            "value": round(wq.batch / (r["total_ms"] / args.steps / 1e3), 1),
            "ms_per_step": round(r["total_ms"] / args.steps, 5),
            "roofline": roof(r, f"qwen{wq.seq}"), "e2e_tok_s": round(r["e2e_tok_s"], 1),
            "config": {"batch": wq.batch, "q_heads": wq.n_q_heads, "kv_heads": wq.n_kv_heads,
                       "head_dim": wq.head_dim, "seq_len": wq.seq, "bits": wq.bits, "clip": wq.clip,
                       "key_transform": "dense", "l2": f"{r['copies']} cache copies rotated per step (> L2)",
                       "step": "dq_decode_step: append 1 new token/seq + decode attention, CUDA graph per step"}}
    if bf16 is not None:
        line["variants"]["llama3-8b-decode-bf16-cache"] = {
            "value": round(w.batch / (bf16["total_ms"] / args.steps / 1e3), 1),
            "ms_per_step": round(bf16["total_ms"] / args.steps, 5),
            "roofline": roof(bf16, "bf16"), "e2e_tok_s": round(bf16["e2e_tok_s"], 1),
            "config": {"batch": w.batch, "seq_len": S, "cache": "bf16, unquantized (all tokens 16-bit slots)",
                       "role": "context: the same step without quantization, through the library's 16-bit path"}}
    for D, dqr in dqrs:
        line["variants"][f"{D.name}-k{D.extra['levels_k']}x{D.extra['container_k']}-v{D.extra['levels_v']}x{D.extra['container_v']}"] = {
            "value": round(D.batch / (dqr["total_ms"] / dqr["steps"] / 1e3), 1),
            "ms_per_step": round(dqr["total_ms"] / dqr["steps"], 5),
            "roofline": roof(dqr, "dquant" if D is W.DQUANT else "dquant196"), "e2e_tok_s": round(dqr["e2e_tok_s"], 1),
            "prefill_ms": round(dqr["prefill_ms"], 3),
            "config": {"batch": D.batch, "q_heads": D.n_q_heads, "kv_heads": D.n_kv_heads, "head_dim": D.head_dim,
                       "seq_len": D.seq, "n_recent": D.n_recent, "levels_k": D.extra["levels_k"],
                       "levels_v": D.extra["levels_v"], "container_k": D.extra["container_k"],
                       "container_v": D.extra["container_v"], "bits_per_value": round(W.dquant_bits_per_value(D), 3),
                       "l2": f"{dqr['copies']} cache copies rotated per step (> L2)",
                       "step": "decode attention over a prefilled cache, one call per step"}}
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w, args.bits, S, args.cpu_seconds, k, v, q)
    if rank == 0:
        line["diagnostics"] = {"dquant_feasible_alphabet": feasible_alphabet(),
                               "note": "largest D-Quant alphabet whose cheapest 1024-value stream fits the "
                                       "container, by the library's symbol model, vs fixed-width levels"}
        if not args.no_dquant:
            try:
                abl = dquant_ablation()
            except Exception as e:  # a diagnostic never costs the measurement line
                abl = {"error": f"{type(e).__name__}: {e}"}
            abl["note"] = ("decode-attention output (fp32) against exact fp64 attention over the unquantized "
                           "tokens, one D-Quant setting varied at a time around 8 / 6 levels in 331 / 231 bytes")
            line["diagnostics"]["dquant_ablation"] = abl
        try:
            pre = preprocessing_effect()
        except Exception as e:  # a diagnostic never costs the measurement line
            pre = {"error": f"{type(e).__name__}: {e}"}
        pre["note"] = ("8-level per-token grids of the Llama-shaped synthetic K and V through the library's "
                       "3-bit quantizer: NMSE, entropy, Coding Gain = log2 M - H, Normal Gap = CE - H against "
                       "the analytic order-statistics model")
        line["diagnostics"]["preprocessing"] = pre
        try:
            gab = grid_ablation()
        except Exception as e:  # a diagnostic never costs the measurement line
            gab = {"error": f"{type(e).__name__}: {e}"}
        gab["note"] = ("relative squared reconstruction error of K and V on the Hadamard rotation: min/max grid, "
                       "percentile clip (kappa 0.96 keys / 0.92 values), QuEST grid (s = c_b RMS)")
        line["diagnostics"]["grid_ablation"] = gab
        if not args.no_dquant:
            try:
                dst = drift_statistics()
            except Exception as e:  # a diagnostic never costs the measurement line
                dst = {"error": f"{type(e).__name__}: {e}"}
            dst["note"] = ("symbols moved by drift off the nearest level of their final grid, counted by the library "
                           "while encoding (the page measures 0.75 % of keys and 5.00 % of values on real caches)")
            line["diagnostics"]["drift"] = dst
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
