#!/usr/bin/env python3
"""Benchmark: TP-sharded MLP block tokens/s on one B300, with its roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the path over one batch: the column-parallel linear with
its fused activation, then the row-parallel linear with the in-kernel shard sum
(exactly what tp_mlp_block launches), on synthetic seeded inputs of the
workload's shapes.  Every tensor-parallel shard lives on the one GPU.  With
--gpus N > 1 (under torchrun) each rank runs an independent replica: the path
has no exchange between GPUs, so there is no collective on the data path; the
barrier and the max-over-ranks timing are host bookkeeping.

Printed (rank 0, one JSON line): whole-job tokens/s, the dominant kernel's
achieved TFLOP/s or GB/s against the measured peak, the oracle's CPU
throughput on a bounded sample, the end-to-end number through the public call
with pinned host buffers, SM clocks sampled during the timed region.

--impl reference times the fp64 CPU oracle (the plain implementation the
tests check against) on the same workload, a bounded sample of rows per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TP-sharded MLP block tokens/s on 1 B300; % of HBM or bf16 tensor roofline"
L2_BYTES = 126 * 1024 * 1024

# name -> workload.  Shapes are the Llama-2-70B-sized layers (d_model 8192,
# d_ff 28672; 64 query / 8 KV heads of dim 128) and the small GELU FFN block.
WORKLOADS = {
    "swiglu_ffn_prefill_tp8": dict(kind="ffn", M=4096, d=8192, dff=28672, tp=8, act="swiglu",
                                   bias=False),
    "swiglu_ffn_decode_tp4_b1": dict(kind="ffn", M=1, d=8192, dff=28672, tp=4, act="swiglu",
                                     bias=False),
    "swiglu_ffn_decode_tp4_b8": dict(kind="ffn", M=8, d=8192, dff=28672, tp=4, act="swiglu",
                                     bias=False),
    "swiglu_ffn_decode_tp4_b32": dict(kind="ffn", M=32, d=8192, dff=28672, tp=4, act="swiglu",
                                      bias=False),
    "swiglu_ffn_decode_tp4_b64": dict(kind="ffn", M=64, d=8192, dff=28672, tp=4, act="swiglu",
                                      bias=False),
    "gelu_ffn_tp2": dict(kind="ffn", M=16, d=512, dff=2048, tp=2, act="gelu", bias=True),
    "attn_proj_tp8": dict(kind="attn", M=2048, d=8192, H=64, Hkv=8, hd=128, tp=8),
    # one decoder layer's linear algebra (QKV, O, FFN up, FFN down) per step,
    # replayed from a CUDA graph of tp_layer_forward
    "layer_decode_tp4_b8_graph": dict(kind="layer", M=8, d=8192, H=64, Hkv=8, hd=128,
                                      dff=28672, tp=4, act="swiglu", bias=False),
    # the FFN down projection of the 4096-token prefill, its shard sum done the
    # way a ring all-reduce adds bf16 partials (tp partial GEMMs + ring kernel)
    "row_ring_prefill_tp8": dict(kind="row_ring", M=4096, d=8192, dff=28672, tp=8),
    # d_ff = 28672 is not divisible by 3: tp=3 needs the uneven column split
    # (up projection of the decode FFN, 8 tokens, widths 9558/9557/9557)
    "column_uneven_decode_tp3_b8": dict(kind="uneven", M=8, d=8192, dff=28672, tp=3,
                                        widths=(9558, 9557, 9557)),
    # the decode FFN with e4m3 weights (one byte per weight, one fp32 scale per
    # weight row): the weights it streams are half the bf16 ones
    "swiglu_ffn_decode_tp4_b1_fp8": dict(kind="ffn", M=1, d=8192, dff=28672, tp=4,
                                         act="swiglu", bias=False, fp8=True),
    "swiglu_ffn_decode_tp4_b8_fp8": dict(kind="ffn", M=8, d=8192, dff=28672, tp=4,
                                         act="swiglu", bias=False, fp8=True),
}

# Link bandwidth for the analytic ring all-reduce time of "Tensor parallel
# serving" ("Communication cost"): T = 2 (p - 1) / p * bytes / B.  A stated
# assumption (an NVLink-class per-GPU link), not a measurement: no bytes leave
# the one GPU here.
LINK_GBPS = 900.0


def ring_allreduce_us(p: int, nbytes: float, link_gbps: float = LINK_GBPS) -> float:
    """Time of a ring all-reduce of nbytes over p ranks at link_gbps, in us."""
    if p <= 1:
        return 0.0
    return 2.0 * (p - 1) / p * nbytes / (link_gbps * 1e9) * 1e6
DEFAULT_WORKLOAD = "swiglu_ffn_prefill_tp8"


# ------------------------------------------------------------------ work model
def kernel_work(w):
    """Algorithmic FLOPs and minimum HBM bytes of each kernel launch of one step.

    bf16 operands (2 bytes), fp32 biases, bf16 intermediate h, bf16 output;
    FP8 workloads: one byte per weight plus one fp32 scale per weight row.
    """
    M, d = w["M"], w["d"]
    if w["kind"] == "row_ring":
        dff, tp = w["dff"], w["tp"]
        # partial GEMMs: weights + h + bf16 partials; ring kernel: partials + Y
        flops = 2.0 * M * dff * d
        nbytes = 2.0 * (d * dff + M * dff + tp * M * d) + 2.0 * (tp * M * d + M * d)
        return {"row_ring": (flops, nbytes)}
    if w["kind"] == "uneven":
        return {"column": (2.0 * M * d * w["dff"], 2.0 * (w["dff"] * d + M * d + M * w["dff"]))}
    if w["kind"] == "layer":
        a = kernel_work(dict(w, kind="attn"))
        f = kernel_work(dict(w, kind="ffn"))
        flops = sum(x for x, _ in list(a.values()) + list(f.values()))
        nbytes = sum(y for _, y in list(a.values()) + list(f.values()))
        return {"layer": (flops, nbytes)}
    if w["kind"] == "ffn":
        dff = w["dff"]
        n_w1 = 2 if w["act"] == "swiglu" else 1
        col_flops = 2.0 * M * d * dff * n_w1
        col_bytes = 2.0 * (n_w1 * dff * d + M * d + M * dff) + (4 * dff if w.get("bias") else 0)
        row_flops = 2.0 * M * dff * d
        row_bytes = 2.0 * (d * dff + M * dff + M * d) + (4 * d if w.get("bias") else 0)
        if w.get("fp8"):
            # weights at one byte instead of two; per-row scales (the row split
            # holds one scale per output row in each of its tp shards)
            col_bytes += -1.0 * n_w1 * dff * d + 4.0 * n_w1 * dff
            row_bytes += -1.0 * d * dff + 4.0 * w["tp"] * d
        return {"column": (col_flops, col_bytes), "row": (row_flops, row_bytes)}
    H, Hkv, hd = w["H"], w["Hkv"], w["hd"]
    nq = (H + 2 * Hkv) * hd
    qkv_flops = 2.0 * M * d * nq
    qkv_bytes = 2.0 * (nq * d + M * d + M * nq)
    o_flops = 2.0 * M * H * hd * d
    o_bytes = 2.0 * (d * H * hd + M * H * hd + M * d)
    return {"column": (qkv_flops, qkv_bytes), "row": (o_flops, o_bytes)}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0,
                source="fallback")


def traffic_record(workload):
    """Per-launch DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of the
    dominant kernel from the committed ncu summary -- only while the kernel's
    source file still has the hash it had when the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return {}
    if not rec:
        return {}
    try:
        with open(os.path.join(ROOT, rec["source_file"]), "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return {}
    return rec if h == rec.get("source_sha256_16") else {}


# ------------------------------------------------------------------ clocks
class _Nvml:
    """Read-only NVML queries: the pynvml module when installed, else the same C
    functions of the driver's libnvidia-ml.so.1 through ctypes."""

    CLOCK_SM = 1
    REASON_BITS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20),
                   ("hw_thermal_slowdown", 0x40), ("hw_power_brake_slowdown", 0x80))

    def __init__(self, uuid: str):
        try:
            import pynvml
            pynvml.nvmlInit()
            self._p, self._h = pynvml, pynvml.nvmlDeviceGetHandleByUUID(uuid)
            self.kind = "pynvml"
            return
        except ImportError:
            pass
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByUUID failed")
        self._p, self._lib, self._h, self._ct = None, lib, h, ctypes
        self.kind = "libnvidia-ml (ctypes)"

    def _u32(self, fn, *args):
        v = self._ct.c_uint()
        if fn(self._h, *args, self._ct.byref(v)) != 0:
            raise RuntimeError("nvml query failed")
        return v.value

    def sm_clock(self):
        if self._p:
            return self._p.nvmlDeviceGetClockInfo(self._h, self.CLOCK_SM)
        return self._u32(self._lib.nvmlDeviceGetClockInfo, self.CLOCK_SM)

    def max_sm_clock(self):
        if self._p:
            return self._p.nvmlDeviceGetMaxClockInfo(self._h, self.CLOCK_SM)
        return self._u32(self._lib.nvmlDeviceGetMaxClockInfo, self.CLOCK_SM)

    def reasons(self):
        if self._p:
            r = self._p.nvmlDeviceGetCurrentClocksEventReasons(self._h)
        else:
            v = self._ct.c_ulonglong()
            if self._lib.nvmlDeviceGetCurrentClocksEventReasons(self._h, self._ct.byref(v)) != 0:
                raise RuntimeError("nvml query failed")
            r = v.value
        return {n for n, bit in self.REASON_BITS if r & bit}


class ClockSampler:
    """SM clock and clock-event (throttle) reasons of one GPU, polled through NVML
    every `period_s` on a background thread while the timed region runs (reading
    only: no setting is changed).  Works for timed regions of a few milliseconds."""

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.device_index = device_index
        self.period_s = period_s
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.error = None
        self.kind = None
        self._stop = None
        self._thread = None

    def __enter__(self):
        import threading
        import torch
        try:
            uuid = str(torch.cuda.get_device_properties(self.device_index).uuid)
            if not uuid.startswith("GPU-"):
                uuid = "GPU-" + uuid
            nv = _Nvml(uuid)
            self.kind = nv.kind
            self.max_mhz = nv.max_sm_clock()
        except Exception as e:  # noqa: BLE001 - report, do not fail the benchmark
            self.error = f"nvml unavailable: {type(e).__name__}: {e}"
            return self
        self._stop = threading.Event()

        def poll():
            while True:
                try:
                    self.samples.append(nv.sm_clock())
                    self.reasons |= nv.reasons()
                except Exception as e:  # noqa: BLE001
                    self.error = f"nvml query failed: {type(e).__name__}"
                    return
                if self._stop.wait(self.period_s):
                    return

        self._thread = threading.Thread(target=poll, daemon=True)
        self._thread.start()
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz,
                    "reasons": [self.error or "no samples"]}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples),
                "source": f"{self.kind}, polled every {self.period_s * 1e3:g} ms"}


# ------------------------------------------------------------------ ranks
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def reduce_over_ranks(elapsed_ms: float, tokens: int, world: int):
    """(max elapsed over ranks, total tokens over ranks).  Host bookkeeping only."""
    if world <= 1:
        return elapsed_ms, tokens
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=dev)
    n = torch.tensor([float(tokens)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ our arm
class Path:
    """Sharded weights on the device and the launches of one step."""

    def __init__(self, w, device, seed=20_000):
        import torch
        from tensor_column_linear_gelu_b300 import inputs, tpla
        self.w, self.tpla = w, tpla
        tp = w["tp"]
        if w["kind"] == "ffn":
            f = inputs.ffn(seed, w["M"], w["d"], w["dff"], w["act"], w["bias"], device=device)
            split = "gate_up" if w["act"] == "swiglu" else "column"
            self.w1, self.b1 = tpla.tp_shard_weights(split, tp, f.W1, W_up=f.W_up, b=f.b1)
            self.w2, _ = tpla.tp_shard_weights("row", tp, f.W2)
            self.b2 = f.b2
            if w.get("fp8"):
                # e4m3 codes + row scales replace the bf16 shards
                self.q1, self.s1 = tpla.quantize_shards_fp8(self.w1)
                self.q2, self.s2 = tpla.quantize_shards_fp8(self.w2)
                self.w1 = self.w2 = None
            self.X = f.X
            self.h = torch.empty(w["M"], w["dff"], dtype=torch.bfloat16, device=device)
            self.Y = torch.empty(w["M"], w["d"], dtype=torch.bfloat16, device=device)
            del f
        elif w["kind"] == "row_ring":
            self.h = inputs.normal((w["M"], w["dff"]), 1.0, seed, torch.bfloat16, device)
            W2 = inputs.normal((w["d"], w["dff"]), inputs.WEIGHT_STD, seed + 3, torch.bfloat16,
                               device)
            self.w2, _ = tpla.tp_shard_weights("row", tp, W2)
            del W2
            self.X = self.h
            self.parts_buf = torch.empty(tp, w["M"], w["d"], dtype=torch.bfloat16, device=device)
            self.Y = torch.empty(w["M"], w["d"], dtype=torch.bfloat16, device=device)
        elif w["kind"] == "uneven":
            f = inputs.ffn(seed, w["M"], w["d"], w["dff"], "gelu", False, device=device)
            self.w1, _ = tpla.tp_shard_weights_uneven(w["widths"], f.W1)
            self.X = f.X
            self.Y = torch.empty(w["M"], w["dff"], dtype=torch.bfloat16, device=device)
            del f
        elif w["kind"] == "layer":
            a = inputs.attn(seed, w["M"], w["d"], w["H"], w["Hkv"], w["hd"], device=device)
            f = inputs.ffn(seed + 100, w["M"], w["d"], w["dff"], w["act"], w["bias"],
                           device=device)
            heads = dict(n_heads=w["H"], n_kv_heads=w["Hkv"], head_dim=w["hd"])
            wq, _ = tpla.tp_shard_weights("qkv_heads", tp, a.Wqkv, **heads)
            wo, _ = tpla.tp_shard_weights("row", tp, a.Wo)
            w1, _ = tpla.tp_shard_weights("gate_up", tp, f.W1, W_up=f.W_up)
            w2, _ = tpla.tp_shard_weights("row", tp, f.W2)
            self.X, self.ctx = a.X, a.ctx
            self.layer_kw = dict(X=a.X, wqkv_shards=wq, bqkv_shards=None, ctx=a.ctx,
                                 wo_shards=wo, bo=None, w1_shards=w1, b1_shards=None,
                                 w2_shards=w2, b2=None, ffn_act=w["act"], d_ff=w["dff"], **heads)
            self.graph = tpla.LayerGraph(tp, **self.layer_kw)
            self.Y = self.graph.outputs[3]
            del a, f
        else:
            a = inputs.attn(seed, w["M"], w["d"], w["H"], w["Hkv"], w["hd"], device=device)
            heads = dict(n_heads=w["H"], n_kv_heads=w["Hkv"], head_dim=w["hd"])
            self.w1, _ = tpla.tp_shard_weights("qkv_heads", tp, a.Wqkv, **heads)
            self.w2, _ = tpla.tp_shard_weights("row", tp, a.Wo)
            self.X, self.ctx = a.X, a.ctx
            ws = (w["H"] // tp + 2 * (w["Hkv"] // tp)) * w["hd"]
            self.qkv = torch.empty(tp, w["M"], ws, dtype=torch.bfloat16, device=device)
            self.Y = torch.empty(w["M"], w["d"], dtype=torch.bfloat16, device=device)
            del a
        torch.cuda.synchronize()

    # The FFN step as its two launches: exactly the sequence tp_mlp_block issues
    # (column with fused activation into h, then row with the shard sum), so a
    # CUDA event can sit between them.  The attention step is timed whole.
    def parts(self):
        w, t = self.w, self.tpla
        if w["kind"] == "ffn" and w.get("fp8"):
            def column(s):
                t.column_parallel_linear_fp8(w["tp"], self.X, self.q1, self.s1, self.b1, w["act"],
                                             Y=self.h, N=w["dff"], stream=s)

            def row(s):
                t.row_parallel_linear_fp8(w["tp"], self.h, self.q2, self.s2, self.b2, Y=self.Y,
                                          stream=s)
            return [("column", column), ("row", row)]
        if w["kind"] == "ffn":
            def column(s):
                t.column_parallel_linear(w["tp"], self.X, self.w1, self.b1, w["act"], Y=self.h,
                                         N=w["dff"], stream=s)

            def row(s):
                t.row_parallel_linear(w["tp"], self.h, self.w2, self.b2, Y=self.Y, stream=s)
            return [("column", column), ("row", row)]
        if w["kind"] == "layer":
            return [("layer", lambda s: self.graph.replay())]
        if w["kind"] in ("row_ring", "uneven"):
            return [(w["kind"] if w["kind"] == "row_ring" else "column",
                     lambda s: self.step_public(s))]
        return [("attn_proj", lambda s: self.step_public(s))]

    def step_public(self, s, X=None, Y=None):
        """One step through the public call a user makes."""
        import torch
        w, t = self.w, self.tpla
        X = self.X if X is None else X
        Y = self.Y if Y is None else Y
        if w["kind"] == "row_ring":
            t.row_parallel_linear_ring(w["tp"], X, self.w2, None, wire_dtype=torch.bfloat16,
                                       Y=Y, partials=self.parts_buf, stream=s)
        elif w["kind"] == "uneven":
            t.column_parallel_linear_uneven(w["widths"], X, self.w1, None, "none", Y=Y, stream=s)
        elif w["kind"] == "layer":
            # the graph reads the captured X buffer and writes the captured output
            if X is not self.X:
                self.X.copy_(X, non_blocking=True)
            self.graph.replay()
            if Y is not self.Y:
                Y.copy_(self.Y, non_blocking=True)
        elif w["kind"] == "ffn" and w.get("fp8"):
            t.tp_mlp_block_fp8(w["tp"], X, self.q1, self.s1, self.b1, self.q2, self.s2, self.b2,
                               w["act"], d_ff=w["dff"], h=self.h, Y=Y, stream=s)
        elif w["kind"] == "ffn":
            t.tp_mlp_block(w["tp"], X, self.w1, self.b1, self.w2, self.b2, w["act"],
                           d_ff=w["dff"], h=self.h, Y=Y, stream=s)
        else:
            t.tp_attn_proj(w["tp"], X, self.w1, None, self.ctx, self.w2, None, w["H"], w["Hkv"],
                           w["hd"], qkv_out=self.qkv, Y=Y, stream=s)

    def launches_per_step(self):
        w = self.w
        if w["kind"] == "attn" and w["M"] > 128:
            return 1  # QKV and O share one prefill-GEMM launch
        if w["kind"] == "layer":
            # QKV and O share a launch when both take the prefill GEMM
            return 3 if w["M"] > 128 else 4
        if w["kind"] == "uneven":
            return 1 if w["M"] <= 128 else w["tp"]
        return {"row_ring": w["tp"] + 1}.get(w["kind"], 2)


# Datasheet figures of one B300, for the second denominator of every
# fraction: HBM3e bandwidth, and the dense (no 2:4 sparsity) bf16 tensor peak.
DATASHEET = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0,
             "source": "B300 datasheet: HBM3e 8 TB/s; bf16 dense 2.25 PFLOP/s"}

# Decode-shaped workloads timed in the default run next to the headline one.
KERNEL_TIMING = ("decode-shaped steps (at most 128 tokens): value from K steps with an event "
                 "at each end of the timed region only, kernel_ms and the roofline's avg_ms "
                 "from K further steps with an event around every launch; other steps: one "
                 "timed pass with an event around every launch")
PDL_MAX_TOKENS = 128  # the decode kernels' token limit: their launches overlap
DECODE_EXTRAS = ("swiglu_ffn_decode_tp4_b1", "swiglu_ffn_decode_tp4_b8",
                 "swiglu_ffn_decode_tp4_b32", "swiglu_ffn_decode_tp4_b64",
                 "swiglu_ffn_decode_tp4_b1_fp8", "swiglu_ffn_decode_tp4_b8_fp8")


def measure(args, name, w, dev, world, steps, warmup):
    """Time `steps` steps of workload `w` on device `dev` (after `warmup`
    untimed ones), with CUDA events on the launching stream.  Returns the
    timing, the roofline of the dominant launch and of the whole step, and the
    SM clocks sampled during the timed region.  `path` is returned too, for the
    end-to-end leg."""
    import torch
    from tensor_column_linear_gelu_b300 import tpla
    peaks = load_peaks()
    path = Path(w, dev)
    s = torch.cuda.Stream(device=dev)
    parts = path.parts()
    work = kernel_work(w)
    step_bytes = sum(b for _, b in work.values())
    step_flops = sum(f for f, _ in work.values())
    flush = None
    if step_bytes < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    with torch.cuda.stream(s):
        for _ in range(warmup):
            for _, fn in parts:
                fn(s)
    s.synchronize()
    st = tpla.tp_device_status(s)
    if st != tpla.TP_OK:
        raise RuntimeError(f"{name}: device status after warm-up: {tpla.status_string(st)}")

    K = steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)] for _ in range(K)]
    e_first = torch.cuda.Event(enable_timing=True)
    e_last = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    # Decode-shaped steps (at most 128 tokens: the decode kernels and GEMVs)
    # are chains of programmatic dependent launches, and an event recorded
    # between two launches keeps the second from overlapping the first's
    # tail.  Their timed region has an event at each end only, and a second
    # pass times each launch.  The prefill GEMM is launched in plain stream
    # order: one pass, an event around every launch.
    two_pass = flush is None and w["M"] <= PDL_MAX_TOKENS
    with clocks:
        if two_pass:
            # The timed region: K steps back to back with an event at each end
            # only, so that a launch may overlap its predecessor's tail
            # (programmatic dependent launch) as it does in use.
            with torch.cuda.stream(s):
                e_first.record(s)
                for k in range(K):
                    for _, fn in parts:
                        fn(s)
                e_last.record(s)
            s.synchronize()
            torch.cuda.synchronize()
            barrier(world)
            torch.cuda.synchronize()
        # Per-launch durations (the roofline's kernel): an event around every
        # launch -- K more steps after a two-pass timed region, else the timed
        # region itself (with a flush, the flushes outside the step events).
        with torch.cuda.stream(s):
            for k in range(K):
                if flush is not None:
                    flush.zero_()
                ev[k][0].record(s)
                for j, (_, fn) in enumerate(parts):
                    fn(s)
                    ev[k][j + 1].record(s)
        s.synchronize()
        torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    st = tpla.tp_device_status(s)
    if st != tpla.TP_OK:
        raise RuntimeError(f"{name}: device status after timed region: {tpla.status_string(st)}")

    per_part = {pn: [ev[k][j].elapsed_time(ev[k][j + 1]) for k in range(K)]
                for j, (pn, _) in enumerate(parts)}
    step_ms = [ev[k][0].elapsed_time(ev[k][len(parts)]) for k in range(K)]
    if two_pass:
        elapsed_ms = e_first.elapsed_time(e_last)
    elif flush is None:
        elapsed_ms = ev[0][0].elapsed_time(ev[K - 1][len(parts)])
    else:
        elapsed_ms = sum(step_ms)
    tokens_local = w["M"] * K
    elapsed_max, tokens_all = reduce_over_ranks(elapsed_ms, tokens_local, world)

    # ---------------------------------------------------------- roofline
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if w["kind"] == "ffn":
        avg = {n: sum(v) / len(v) for n, v in per_part.items()}
        dom = max(avg, key=avg.get)
        flops, nbytes = work[dom]
        dur_s = avg[dom] / 1e3
        launches_in_dom = 1
    elif w["kind"] in ("layer", "row_ring", "uneven"):
        dom = next(iter(work))
        flops, nbytes = work[dom]
        dur_s = (sum(per_part[dom]) / K) / 1e3
        launches_in_dom = path.launches_per_step()
    else:
        dom = "attn_proj"
        flops = sum(f for f, _ in work.values())
        nbytes = sum(b for _, b in work.values())
        dur_s = (sum(per_part["attn_proj"]) / K) / 1e3
        launches_in_dom = path.launches_per_step()
    bound = "tensor" if flops / nbytes > ridge else "hbm"
    long_region = elapsed_ms > 1000.0
    step_s = (elapsed_ms / K) / 1e3
    if bound == "tensor":
        peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
        achieved = flops / dur_s / 1e12
        step_achieved = step_flops / step_s / 1e12
        unit = "TFLOP/s"
        peak_kind = ("sustained" if long_region else "burst") + " bf16, " + peaks["source"]
        sheet = DATASHEET["bf16_tflops"]
    else:
        peak = peaks["hbm_gbs"]
        achieved = nbytes / dur_s / 1e9
        step_achieved = step_bytes / step_s / 1e9
        unit = "GB/s"
        peak_kind = "hbm copy, " + peaks["source"]
        sheet = DATASHEET["hbm_gbs"]
    tr = traffic_record(name)
    roofline = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "traffic": tr.get("bytes_per_launch"),
                "kernel": dom, "launches": launches_in_dom,
                "algorithmic_flops": flops, "algorithmic_bytes": nbytes,
                "avg_ms": round(dur_s * 1e3, 4), "peak_kind": peak_kind,
                "datasheet_peak": sheet, "frac_of_datasheet": round(achieved / sheet, 4),
                "step": {"achieved": round(step_achieved, 2), "unit": unit,
                         "frac": round(step_achieved / peak, 4),
                         "frac_of_datasheet": round(step_achieved / sheet, 4),
                         "algorithmic_flops": step_flops, "algorithmic_bytes": step_bytes}}
    if tr.get("bytes_per_launch") is not None:
        roofline["traffic_source"] = tr.get("source")
    return dict(elapsed_max=elapsed_max, tokens_all=tokens_all, roofline=roofline,
                per_part={n: round(sum(v) / len(v), 4) for n, v in per_part.items()},
                clocks=clocks.summary(), flush=flush is not None,
                launches=K * path.launches_per_step(), path=path, stream=s)


def run_ours(args, w, rank, local_rank, world):
    import torch
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    r = measure(args, args.workload, w, dev, world, args.steps, args.warmup)
    r["e2e"] = run_e2e(r.pop("path"), w, r.pop("stream"), args)
    torch.cuda.empty_cache()
    r["cpu"] = None
    if rank == 0 and not args.no_cpu_baseline:
        r["cpu"] = cpu_baseline(w, budget_s=args.cpu_seconds)
    # the decode-shaped workloads, each with its own roofline (HBM-bound)
    r["decode"] = None
    if args.workload == DEFAULT_WORKLOAD and not args.no_decode:
        r["decode"] = {}
        for name in DECODE_EXTRAS:
            wd = WORKLOADS[name]
            d = measure(args, name, wd, dev, world, args.decode_steps, args.warmup)
            d.pop("path")
            d.pop("stream")
            torch.cuda.empty_cache()
            d["value"] = round(d["tokens_all"] / (d["elapsed_max"] / 1e3), 2)
            d["ms_per_step"] = round(d["elapsed_max"] / args.decode_steps, 4)
            d["steps"] = args.decode_steps
            d["kernel_ms"] = d.pop("per_part")
            d["unit"] = "tokens/s"
            d["gpu_launches"] = d.pop("launches")
            for k in ("elapsed_max", "tokens_all", "flush"):
                d.pop(k)
            r["decode"][name] = d
    return r


def run_e2e(path, w, s, args):
    """Same metric through the public call, with each step's input copied in
    from pinned host memory and its result read back to pinned host memory.

    Copies run on their own streams so that step k+1's input copy and step
    k-1's result copy overlap step k's kernels; inputs and outputs are
    double-buffered, and events order each buffer's reuse.  The timed region
    runs from before the first input copy to after the last result copy."""
    import torch
    dev = path.X.device
    Xh = path.X.to("cpu").pin_memory()
    Yh = [torch.empty(path.Y.shape, dtype=path.Y.dtype).pin_memory() for _ in range(2)]
    Xd = [torch.empty_like(path.X) for _ in range(2)]
    Yd = [torch.empty_like(path.Y) for _ in range(2)]
    cin = torch.cuda.Stream(device=dev)
    cout = torch.cuda.Stream(device=dev)
    K = args.steps

    def run(n_steps):
        x_ready = [torch.cuda.Event() for _ in range(2)]
        done = [None, None]     # step k's kernels finished with Xd/Yd[k % 2]
        out_done = [None, None]  # result copy of Yd[k % 2] finished
        for k in range(n_steps):
            b = k % 2
            if done[b] is not None:
                cin.wait_event(done[b])
            with torch.cuda.stream(cin):
                Xd[b].copy_(Xh, non_blocking=True)
                x_ready[b].record(cin)
            s.wait_event(x_ready[b])
            if out_done[b] is not None:
                s.wait_event(out_done[b])
            with torch.cuda.stream(s):
                path.step_public(s, Xd[b], Yd[b])
                done[b] = torch.cuda.Event()
                done[b].record(s)
            cout.wait_event(done[b])
            with torch.cuda.stream(cout):
                Yh[b].copy_(Yd[b], non_blocking=True)
                out_done[b] = torch.cuda.Event()
                out_done[b].record(cout)
        for e in out_done:
            if e is not None:
                s.wait_event(e)

    run(max(1, args.warmup))
    s.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s)
    cin.wait_event(e0)
    run(K)
    e1.record(s)
    s.synchronize()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    return {"value": round(w["M"] * K / (ms / 1e3), 2), "unit": "tokens/s",
            "h2d_bytes_per_step": Xh.numel() * Xh.element_size(),
            "d2h_bytes_per_step": Yh[0].numel() * Yh[0].element_size(),
            "ms_per_step": round(ms / K, 4),
            "overlap": "input copy of step k+1 and result copy of step k-1 on their own "
                       "streams, double-buffered, overlapping step k"}


# ------------------------------------------------------------------ CPU oracle
def oracle_inputs(w, rows, seed=20_000):
    """Host float32 inputs the oracle needs for `rows` sampled rows of the workload
    (the same seeded tensors the GPU arm uses)."""
    import torch
    from tensor_column_linear_gelu_b300 import inputs
    dev = "cuda" if torch.cuda.is_available() else None
    if w["kind"] == "row_ring":
        h = inputs.normal((w["M"], w["dff"]), 1.0, seed, torch.bfloat16, dev)
        W2 = inputs.normal((w["d"], w["dff"]), inputs.WEIGHT_STD, seed + 3, torch.bfloat16, dev)
        a = dict(X=h[rows].float().cpu().numpy(), W2=W2.float().cpu().numpy())
        del h, W2
        return a
    if w["kind"] == "uneven":
        f = inputs.ffn(seed, w["M"], w["d"], w["dff"], "gelu", False, device=dev)
        a = dict(X=f.X[rows].float().cpu().numpy(), W1=f.W1.float().cpu().numpy())
        del f
        return a
    if w["kind"] == "ffn":
        f = inputs.ffn(seed, w["M"], w["d"], w["dff"], w["act"], w["bias"], device=dev)
        a = dict(X=f.X[rows].float().cpu().numpy(), W1=f.W1.float().cpu().numpy(),
                 W1u=None if f.W_up is None else f.W_up.float().cpu().numpy(),
                 W2=f.W2.float().cpu().numpy(),
                 b1=None if f.b1 is None else f.b1.cpu().numpy(),
                 b2=None if f.b2 is None else f.b2.cpu().numpy())
        del f
        if w.get("fp8"):
            # the oracle's own quantization of the same bf16 weights (input
            # preparation, outside the timed oracle step)
            import oracle
            orc = oracle.default()
            a["Q1"], a["S1"] = orc.quantize_rows_fp8(a["W1"])
            a["Q1u"], a["S1u"] = orc.quantize_rows_fp8(a["W1u"])
            a["Q2"], a["S2"] = orc.quantize_row_shards_fp8(w["tp"], a["W2"])
        return a
    at = inputs.attn(seed, w["M"], w["d"], w["H"], w["Hkv"], w["hd"], device=dev)
    a = dict(X=at.X[rows].float().cpu().numpy(), Wqkv=at.Wqkv.float().cpu().numpy(),
             ctx=at.ctx[rows].float().cpu().numpy(), Wo=at.Wo.float().cpu().numpy())
    del at
    if w["kind"] == "layer":
        f = inputs.ffn(seed + 100, w["M"], w["d"], w["dff"], w["act"], w["bias"], device=dev)
        a.update(W1=f.W1.float().cpu().numpy(), W1u=f.W_up.float().cpu().numpy(),
                 W2=f.W2.float().cpu().numpy())
        del f
    return a


def oracle_step(orc, w, a):
    if w["kind"] == "row_ring":
        orc.row_parallel_ring(w["tp"], a["X"], a["W2"], None, "bf16")
        return
    if w["kind"] == "uneven":
        orc.column_parallel_uneven(list(w["widths"]), a["X"], a["W1"])
        return
    if w["kind"] == "ffn" and w.get("fp8"):
        import numpy as np
        h = orc.column_parallel_fp8(w["tp"], a["X"], a["Q1"], a["S1"], None, w["act"],
                                    Qu=a["Q1u"], Su=a["S1u"])
        h = np.vectorize(orc.round_bf16)(h)
        orc.row_parallel_fp8(w["tp"], h, a["Q2"], a["S2"], None)
        return
    if w["kind"] == "ffn":
        orc.mlp_block(w["tp"], a["X"], a["W1"], a["b1"], a["W2"], a["b2"], w["act"], W1u=a["W1u"],
                      round_h=True)
        return
    orc.qkv_proj(w["tp"], a["X"], a["Wqkv"], None, w["H"], w["Hkv"], w["hd"])
    y = orc.o_proj(w["tp"], a["ctx"], a["Wo"], None, w["H"], w["hd"])
    if w["kind"] == "layer":
        # the FFN reads the attention block's output, stored in bf16
        import numpy as np
        y = np.vectorize(orc.round_bf16)(y)
        orc.mlp_block(w["tp"], y, a["W1"], None, a["W2"], None, w["act"], W1u=a["W1u"],
                      round_h=True)


def cpu_baseline(w, budget_s=15.0):
    """The oracle, as it stands, on a bounded sample of the workload's rows: the
    sample grows until one timed run takes at least budget_s / 2 (about
    budget_s of CPU work in all), or covers every row."""
    import oracle
    from tensor_column_linear_gelu_b300 import inputs
    orc = oracle.default()
    n = 1
    while True:
        rows = inputs.sample_rows(w["M"], n, 20_000)
        a = oracle_inputs(w, rows)
        t0 = time.perf_counter()
        oracle_step(orc, w, a)
        t1 = time.perf_counter() - t0
        n = len(rows)
        if t1 >= budget_s / 2 or n >= w["M"]:
            break
        n = int(min(w["M"], max(2 * n, math.ceil(n * 0.6 * budget_s / max(t1, 1e-3)))))
    return {"value": round(n / t1, 4), "unit": "tokens/s", "cores": orc.num_threads(),
            "kind": "oracle",
            "sample": f"{n} of {w['M']} rows of the same workload (fp64 C oracle, OpenMP), "
                      f"{t1:.1f} s"}


def run_reference(args, w, rank, world):
    """--impl reference: the oracle on the host cores, a bounded sample per step."""
    if rank != 0:
        return None
    import oracle
    from tensor_column_linear_gelu_b300 import inputs
    orc = oracle.default()
    rows_per_step = max(1, min(w["M"], args.ref_rows))
    rows = inputs.sample_rows(w["M"], rows_per_step, 20_000)
    a = oracle_inputs(w, rows)
    for _ in range(args.warmup):
        oracle_step(orc, w, a)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(orc, w, a)
    el = time.perf_counter() - t0
    value = rows_per_step * args.steps / el
    sample = f"{rows_per_step} of {w['M']} rows per step (fp64 C oracle, OpenMP)"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload, w, world),
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s",
                             "cores": orc.num_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def workload_config(name, w, world):
    c = {"workload": name}
    c.update({k: v for k, v in w.items() if k != "kind"})
    c["parallelism"] = f"tp{w['tp']} simulated on 1 GPU" + (f", {world} replicas" if world > 1 else "")
    return c


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-rows", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the decode-shaped workloads timed next to the default one")
    ap.add_argument("--decode-steps", type=int, default=50)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    rank, local_rank, world = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local_rank))

    if args.impl == "reference":
        out = run_reference(args, w, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    r = run_ours(args, w, rank, local_rank, world)
    if rank == 0:
        K = args.steps
        value = r["tokens_all"] / (r["elapsed_max"] / 1e3)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(r["elapsed_max"] / K, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 weights x bf16 activations" if w.get("fp8") else "bf16",
            "data": "synthetic",
            "config": dict(workload_config(args.workload, w, world),
                           l2=("L2 flushed between steps (256 MB write)" if r["flush"] else
                               "inputs larger than L2 (weights stream from HBM every step)")),
            "roofline": r["roofline"], "cpu_baseline": r["cpu"], "e2e": r["e2e"],
            "gpu_launches": r["launches"], "clocks": r["clocks"],
            "kernel_ms": r["per_part"],
            "kernel_timing": KERNEL_TIMING,
        }
        if r.get("decode"):
            line["decode"] = r["decode"]
        n_ar = {"ffn": 1, "attn": 1, "layer": 2, "row_ring": 1}.get(w["kind"], 0)
        if n_ar:
            msg = 2.0 * w["M"] * w["d"]  # one bf16 [M, d_model] message per all-reduce
            line["comm_model"] = {
                "ring_allreduce_us_per_step": round(n_ar * ring_allreduce_us(w["tp"], msg), 3),
                "allreduces_per_step": n_ar, "bytes_per_allreduce": msg,
                "link_GBps": LINK_GBPS,
                "note": "analytic 2(p-1)/p*bytes/B for tp devices; nothing is sent here"}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
