#!/usr/bin/env python
"""Benchmark: exact attention on one GB300 through the libfa C ABI.

Headline (one JSON line): forward prefill at B=4, H=32, N=4096, d=128 bf16,
no mask, reported as attention TFLOP/s = 4·B·H·N²·d / time.  The same line
carries, measured in the same process: the long-context forward
(B=1, H=32, N=32768), split-KV decode (B=64, H=32, N_kv=8192, 32 splits,
HBM GB/s and tokens/s) and the training forward + backward (B=2, H=16,
N=8192), each with its fraction of the roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas: (b, h) pairs are independent, there is no exchange
step); rank 0 prints the line with value = all ranks' work / slowest rank.
``--impl reference`` times the float64 CPU oracle on the host cores instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s (4·B·H·N²·d) and % of GB300 BF16 peak; decode HBM GB/s"
UNIT = "TFLOP/s"
PREFILL = dict(B=4, H=32, N=4096, d=128)
LONG = dict(B=1, H=32, N=32768, d=128)
DECODE = dict(B=64, H=32, N=8192, d=128, splits=32)
TRAIN = dict(B=2, H=16, N=8192, d=128)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes per launch from one ncu capture of each kernel (dram__bytes_read.sum +
# dram__bytes_write.sum), keyed by the sha256 of the kernel's sources at capture
# time; a changed kernel reports null until it is captured again.
NCU_TRAFFIC = {
    # the forward kernel at the prefill shape (B=4 H=32 N=4096 d=128), one launch
    "fwd_prefill": {"src": "2909cd273e5e5ee8", "bytes": 402746624 + 114800128},
    # the backward's main kernel at the training shape (B=2 H=16 N=8192 d=128), one launch
    "bwd_train": {"src": "351b9955cd61a286", "bytes": 405801984 + 222792448},
    # the split decode kernel, captured at B=8 (H=32 N_kv=8192 d=128); its traffic is
    # proportional to B, so it is stored here scaled to the B=64 launch
    "decode_split": {"src": "5296948a01a01d33", "bytes": (1073844224 + 6728960) * 8},
}


def fwd_flops(B, H, N, d, Nkv=None):
    return 4.0 * B * H * N * (N if Nkv is None else Nkv) * d


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "io_aware_exact_11_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel, srcs):
    rec = NCU_TRAFFIC.get(kernel)
    if rec and rec["src"] == source_hash(*srcs):
        return rec["bytes"]
    return None


# ------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity for one rank)."""
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.sel = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            self.sel = vis.split(",")[device_index] if vis else str(device_index)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)
        return False

    def summary(self):
        if not getattr(self, "samples", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[1]) for s in self.samples if num(s[1]) is not None]
        mx = [num(s[2]) for s in self.samples if num(s[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[5 + i].lower().startswith("active")})
        sm_sorted = sorted(sm)
        return {"sm_mhz": sm_sorted[len(sm_sorted) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


class SmClockPoller:
    """Reads the SM clock (MHz) through NVML while a timed region runs.

    Reading only: nothing here changes a GPU setting.  If NVML is not
    available the poller returns no samples."""

    NVML_CLOCK_SM = 1

    def __init__(self, device_index: int):
        import ctypes
        self._ct = ctypes
        self.nv = None
        self.h = ctypes.c_void_p()
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0 or nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
                return
            self.nv = nv
        except Exception:
            self.nv = None

    def read(self):
        if self.nv is None:
            return None
        v = self._ct.c_uint()
        if self.nv.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, self._ct.byref(v)) != 0:
            return None
        return float(v.value)

    def poll_until(self, event, samples):
        """Sample until `event` (a recorded torch.cuda.Event) has completed."""
        while not event.query():
            x = self.read()
            if x is not None:
                samples.append(x)
            time.sleep(0.0005)


def median(xs):
    if not xs:
        return None
    s = sorted(xs)
    return s[len(s) // 2]


# --------------------------------------------------------------- CPU oracle
_HEAD = {}


def oracle_sample(budget_s: float, min_blocks: int = 1):
    """The float64 oracle on rows of one prefill head, until ~budget_s elapsed."""
    import numpy as np
    import oracle
    from io_aware_exact_11_gb300 import inputs

    N, d = PREFILL["N"], PREFILL["d"]
    if not _HEAD:
        _HEAD.update({n: inputs.head_as_f64(1, n, 0, 0, N, d) for n in ("q", "k", "v")})
    q, k, v = _HEAD["q"], _HEAD["k"], _HEAD["v"]
    scale = 1 / math.sqrt(d)
    rows_done = 0
    block = 256
    t0 = time.perf_counter()
    while True:
        r0 = rows_done % N
        oracle.attention_rows(q, k, v, scale, np.arange(r0, min(N, r0 + block)))
        rows_done += min(block, N - r0)
        el = time.perf_counter() - t0
        if rows_done >= min_blocks * block and el >= budget_s:
            break
    flops = 4.0 * rows_done * N * d
    return flops / el / 1e12, rows_done, el


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, ws, rank):
    """The oracle as the reference arm: host cores, bounded sample per step."""
    if rank != 0:
        return
    # Keep the whole run to about two minutes whatever --steps/--warmup are.
    per_step = max(0.05, min(2.0, 120.0 / (args.steps + args.warmup / 4)))
    oracle_sample(0.5)  # warm BLAS threads
    for _ in range(args.warmup):
        oracle_sample(per_step / 4)
    vals, rows, secs = [], 0, 0.0
    for _ in range(args.steps):
        v, r, s = oracle_sample(per_step)
        vals.append(v)
        rows += r
        secs += s
    value = 4.0 * rows * PREFILL["N"] * PREFILL["d"] / secs / 1e12
    sample = (f"float64 oracle on query rows of one prefill head (N=4096, d=128, its 4096 rows taken in "
              f"turn and repeated), {rows} rows over {args.steps} steps of ~{per_step:.2f} s")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "prefill forward B=4 H=32 N=4096 d=128 (bounded row sample)", "parallelism": "host"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def run_ours(args, ws, rank, local):
    import torch
    from io_aware_exact_11_gb300 import fa

    if not os.path.exists(fa.LIB_PATH):
        from io_aware_exact_11_gb300 import build
        build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream()
    gen = torch.Generator(device=dev)
    poller = SmClockPoller(local)
    clock_log = {}  # workload -> SM MHz samples taken during its timed region
    peak_mhz = (peaks.get("clocks_under_load") or {}).get("sm_mhz_median")

    sustained = peaks.get("bf16_tflops_sustained")

    def per_clock(tflops, key, scale=1.0):
        """The workload's median SM clock and its TFLOP/s per GHz.  Its fraction
        per clock is taken against the sustained cuBLAS loop, the one peak whose
        clock is known (MEASURED_PEAKS records the median SM clock of that loop);
        `scale` carries a dtype's nominal ratio (2 for FP8)."""
        mhz = median(clock_log.get(key, []))
        out = {"sm_mhz_median": mhz, "sm_samples": len(clock_log.get(key, []))}
        if mhz:
            out["tflops_per_ghz"] = tflops / (mhz / 1e3)
            if peak_mhz and sustained:
                out["frac_of_sustained_peak_per_clock"] = (tflops / mhz) / (scale * float(sustained) / float(peak_mhz))
        return out

    def randn(shape, seed):
        gen.manual_seed(seed * 1000003 + rank)
        return torch.randn(shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)

    def timed(fn, steps, warmup, key=None):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        barrier(ws)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        if key is not None:
            poller.poll_until(e1, clock_log.setdefault(key, []))
        torch.cuda.synchronize()
        barrier(ws)
        return e0.elapsed_time(e1) / 1e3

    peak = float(peaks["bf16_tflops"])
    d = PREFILL["d"]
    if not args.extras_only:
        # ---------------- headline: prefill forward
        B, H, N, d = PREFILL["B"], PREFILL["H"], PREFILL["N"], PREFILL["d"]
        q, k, v = randn((B, H, N, d), 1), randn((B, H, N, d), 2), randn((B, H, N, d), 3)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)

        def step():
            fa.forward(q, k, v, out=o, lse=lse)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        fa.device_status()
        launches0 = fa.launch_count()
        with ClockSampler(local) as clk:
            el = timed(step, args.steps, 0, key="prefill")
        launches = fa.launch_count() - launches0
        fa.device_status()
        el_max = max_over_ranks(el, ws, dev)
        flops = fwd_flops(B, H, N, d)
        value = flops * args.steps * ws / el_max / 1e12
        per_launch = el / args.steps
        achieved = flops / per_launch / 1e12

        # ---------------- e2e: host buffers, copies inside the timed region
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        oh = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        lh = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)

        def e2e_step():
            # The C-ABI host-buffer entry point: q, k, v copied in and o, lse copied
            # out every step, chunk by chunk, overlapped with the forward.
            fa.forward_host(qh, kh, vh, out=oh, lse=lh)

        e2e_steps = max(3, min(args.steps, 20))
        el_e2e = max_over_ranks(timed(e2e_step, e2e_steps, 2), ws, dev)
        h2d = 3 * q.numel() * q.element_size()
        d2h = o.numel() * o.element_size() + lse.numel() * 4
        e2e_value = flops * e2e_steps * ws / el_e2e / 1e12
        del qh, kh, vh, oh, lh

    extra = {}
    extras = set() if args.quick else {x for x in args.extras.split(",") if x}
    if not args.extras_only:
        del q, k, v, o, lse
    if "long" in extras:
        # ---------------- long-context forward
        Bl, Hl, Nl = LONG["B"], LONG["H"], LONG["N"]
        ql, kl, vl = randn((Bl, Hl, Nl, d), 4), randn((Bl, Hl, Nl, d), 5), randn((Bl, Hl, Nl, d), 6)
        ol = torch.empty_like(ql)
        ll = torch.empty((Bl, Hl, Nl), dtype=torch.float32, device=dev)
        n_long = max(2, min(args.steps // 10, 10))
        t_long = timed(lambda: fa.forward(ql, kl, vl, out=ol, lse=ll), n_long, 1, key="long") / n_long
        fl = fwd_flops(Bl, Hl, Nl, d)
        extra["long_forward"] = {"workload": "B=1 H=32 N=32768 d=128 bf16", "tflops": fl / t_long / 1e12,
                                 "ms": t_long * 1e3, "frac_of_bf16_peak": fl / t_long / 1e12 / peak,
                                 **per_clock(fl / t_long / 1e12, "long")}
        del ql, kl, vl, ol, ll

    if "decode" in extras:
        # ---------------- decode
        Bd, Hd, Nd, S = args.decode_batch, DECODE["H"], DECODE["N"], DECODE["splits"]
        qd = randn((Bd, Hd, 1, d), 7)
        kd, vd = randn((Bd, Hd, Nd, d), 8), randn((Bd, Hd, Nd, d), 9)
        od = torch.empty_like(qd)
        ld = torch.empty((Bd, Hd), dtype=torch.float32, device=dev)
        ws_d = torch.empty(fa.decode_workspace_size(Bd, Hd, d, S), dtype=torch.uint8, device=dev)
        n_dec = max(5, min(args.steps, 50))
        t_dec = timed(lambda: fa.decode_splitkv(qd, kd, vd, n_splits=S, out=od, lse=ld, workspace=ws_d),
                      n_dec, 2, key="decode") / n_dec
        kv_bytes = 2.0 * Bd * Hd * Nd * d * 2
        dec_traffic = traffic_for("decode_split", ("fa_decode.cu", "sm103.cuh"))
        extra["decode"] = {"workload": f"B={Bd} H=32 S_q=1 N_kv=8192 d=128 bf16, 32 splits",
                           "hbm_gbs": kv_bytes / t_dec / 1e9, "tokens_per_s": Bd / t_dec, "ms": t_dec * 1e3,
                           "frac_of_hbm_peak": kv_bytes / t_dec / 1e9 / float(peaks["hbm_gbs"]),
                           "bytes_per_step": kv_bytes, "sm_mhz_median": median(clock_log.get("decode", [])),
                           "roofline": {"bound": "hbm", "achieved": kv_bytes / t_dec / 1e9,
                                        "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                                        "frac": kv_bytes / t_dec / 1e9 / float(peaks["hbm_gbs"]),
                                        "kernel": "decode_split_kernel + decode_merge_kernel",
                                        "traffic": None if dec_traffic is None else dec_traffic * Bd / 64}}
        # The same step with the library's own split choice for this shape.
        S_auto = fa.choose_splits(Bd, Hd, Hd, Nd)
        ws_a = torch.empty(fa.decode_workspace_size(Bd, Hd, d, S_auto), dtype=torch.uint8, device=dev)
        t_auto = timed(lambda: fa.decode_splitkv(qd, kd, vd, n_splits=S_auto, out=od, lse=ld, workspace=ws_a),
                       n_dec, 2) / n_dec
        extra["decode"]["library_split_choice"] = {"splits": S_auto, "hbm_gbs": kv_bytes / t_auto / 1e9,
                                                   "tokens_per_s": Bd / t_auto, "ms": t_auto * 1e3}
        del qd, kd, vd, od, ld, ws_d, ws_a

    if "gqa" in extras:
        # ---------------- grouped-query decode, the lab model's 28 query / 4 key-value heads
        # 4 splits: with 4 key/value heads per batch row this already gives 1024 CTAs of 16 key tiles.
        Bg, Hq, Hkv, Ng, S = args.decode_batch, 28, 4, DECODE["N"], 4
        qg = randn((Bg, Hq, 1, d), 21)
        kg, vg = randn((Bg, Hkv, Ng, d), 22), randn((Bg, Hkv, Ng, d), 23)
        og = torch.empty_like(qg)
        lg = torch.empty((Bg, Hq), dtype=torch.float32, device=dev)
        ws_g = torch.empty(fa.decode_workspace_size(Bg, Hq, d, S), dtype=torch.uint8, device=dev)
        n_g = max(5, min(args.steps, 50))
        # K/V (1.07 GB at B=64) is larger than L2, so back-to-back steps stream it from HBM.
        t_g = timed(lambda: fa.decode_splitkv_gqa(qg, kg, vg, n_splits=S, out=og, lse=lg, workspace=ws_g),
                    n_g, 2, key="gqa") / n_g
        kvb = 2.0 * Bg * Hkv * Ng * d * 2
        extra["gqa_decode"] = {"workload": f"B={Bg} Hq=28 Hkv=4 S_q=1 N_kv=8192 d=128 bf16, 4 splits",
                               "hbm_gbs": kvb / t_g / 1e9, "tokens_per_s": Bg / t_g, "ms": t_g * 1e3,
                               "frac_of_hbm_peak": kvb / t_g / 1e9 / float(peaks["hbm_gbs"]),
                               "sm_mhz_median": median(clock_log.get("gqa", []))}
        del qg, kg, vg, og, lg, ws_g

    if "paged" in extras:
        # ---------------- paged cache: pages in shuffled order, every sequence 8192 keys
        for (Hq, Hkv, S, bs) in ((32, 32, 32, 16), (28, 4, 4, 16), (28, 4, 4, 64)):
            Bp, Np = args.decode_batch, DECODE["N"]
            per = Np // bs
            nb = Bp * per
            qp = randn((Bp, Hq, 1, d), 24)
            kp, vp = randn((nb, Hkv, bs, d), 25), randn((nb, Hkv, bs, d), 26)
            gen.manual_seed(27)
            table = torch.randperm(nb, generator=gen, device=dev).to(torch.int32).view(Bp, per)
            lens = torch.full((Bp,), Np, dtype=torch.int32, device=dev)
            op = torch.empty_like(qp)
            lp = torch.empty((Bp, Hq), dtype=torch.float32, device=dev)
            ws_p = torch.empty(fa.decode_workspace_size(Bp, Hq, d, S), dtype=torch.uint8, device=dev)
            n_p = max(5, min(args.steps, 50))
            pkey = f"paged_{Hq}_{Hkv}_{bs}"
            t_p = timed(lambda: fa.decode_paged(qp, kp, vp, table, lens, n_splits=S, out=op, lse=lp, workspace=ws_p),
                        n_p, 2, key=pkey) / n_p
            kvb = 2.0 * Bp * Hkv * Np * d * 2
            extra[f"paged_decode_{Hq}q{Hkv}kv_page{bs}"] = {
                "workload": f"B={Bp} Hq={Hq} Hkv={Hkv} N_kv=8192 d=128 bf16, {bs}-key pages, {S} splits",
                "hbm_gbs": kvb / t_p / 1e9, "tokens_per_s": Bp / t_p, "ms": t_p * 1e3,
                "frac_of_hbm_peak": kvb / t_p / 1e9 / float(peaks["hbm_gbs"]),
                "sm_mhz_median": median(clock_log.get(pkey, []))}
            del qp, kp, vp, table, lens, op, lp, ws_p

    if "train" in extras:
        # ---------------- training forward + backward
        Bt, Ht, Nt = TRAIN["B"], TRAIN["H"], TRAIN["N"]
        qt, kt, vt, dot = (randn((Bt, Ht, Nt, d), s) for s in (10, 11, 12, 13))
        ot = torch.empty_like(qt)
        lt = torch.empty((Bt, Ht, Nt), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(qt), torch.empty_like(kt), torch.empty_like(vt)
        ws_b = torch.empty(fa.backward_workspace_size(Bt, Ht, Nt, d), dtype=torch.uint8, device=dev)
        n_tr = max(3, min(args.steps // 5, 20))
        t_f = timed(lambda: fa.forward(qt, kt, vt, out=ot, lse=lt), n_tr, 1, key="train_fwd") / n_tr
        t_b = timed(lambda: fa.backward(qt, kt, vt, ot, lt, dot, dq=dq, dk=dk, dv=dv, workspace=ws_b),
                    n_tr, 1, key="train_bwd") / n_tr
        ff = fwd_flops(Bt, Ht, Nt, d)
        extra["train"] = {"workload": "B=2 H=16 N=8192 d=128 bf16", "fwd_tflops": ff / t_f / 1e12,
                          "bwd_tflops": 2.5 * ff / t_b / 1e12, "fwd_ms": t_f * 1e3, "bwd_ms": t_b * 1e3,
                          "fwd_frac_of_bf16_peak": ff / t_f / 1e12 / peak,
                          "bwd_frac_of_bf16_peak": 2.5 * ff / t_b / 1e12 / peak,
                          "fwd_clock": per_clock(ff / t_f / 1e12, "train_fwd"),
                          "bwd_clock": per_clock(2.5 * ff / t_b / 1e12, "train_bwd"),
                          "bwd_roofline": {"bound": "tensor", "achieved": 2.5 * ff / t_b / 1e12, "peak": peak,
                                           "unit": "TFLOP/s", "frac": 2.5 * ff / t_b / 1e12 / peak,
                                           "kernel": "time: whole backward (3 kernels); traffic: bwd_main_kernel",
                                           "traffic": traffic_for("bwd_train", ("fa_bwd.cu", "sm103.cuh"))}}
    if "fp8" in extras:
        # ---------------- FP8 (E4M3) forward at the prefill shape; peak = measured bf16 × the nominal 2x
        Bf, Hf, Nf = PREFILL["B"], PREFILL["H"], PREFILL["N"]
        q8, k8, v8 = (randn((Bf, Hf, Nf, d), s).float().to(torch.float8_e4m3fn).view(torch.uint8)
                      for s in (28, 29, 30))
        of = torch.empty((Bf, Hf, Nf, d), dtype=torch.bfloat16, device=dev)
        lf = torch.empty((Bf, Hf, Nf), dtype=torch.float32, device=dev)
        n_f = max(5, min(args.steps, 50))
        t_f8 = timed(lambda: fa.forward_fp8(q8, k8, v8, out=of, lse=lf), n_f, 2, key="fp8") / n_f
        ff8 = fwd_flops(Bf, Hf, Nf, d)
        peak8 = 2.0 * peak
        extra["fp8_prefill_fwd"] = {"workload": "B=4 H=32 N=4096 d=128 E4M3 in, bf16 out",
                                    "tflops": ff8 / t_f8 / 1e12, "ms": t_f8 * 1e3,
                                    **per_clock(ff8 / t_f8 / 1e12, "fp8", 2.0),
                                    "roofline": {"bound": "tensor", "achieved": ff8 / t_f8 / 1e12, "peak": peak8,
                                                 "unit": "TFLOP/s", "frac": ff8 / t_f8 / 1e12 / peak8,
                                                 "peak_source": "measured bf16 burst x 2 (nominal fp8/bf16 ratio)"}}
        del q8, k8, v8, of, lf

    if "d64" in extras:
        # ---------------- head dim 64 at the prefill shape (the other head dim the kernels are built for)
        B6, H6, N6, d6 = PREFILL["B"], PREFILL["H"], PREFILL["N"], 64
        q6, k6, v6 = (randn((B6, H6, N6, d6), s) for s in (31, 32, 33))
        o6 = torch.empty_like(q6)
        l6 = torch.empty((B6, H6, N6), dtype=torch.float32, device=dev)
        n_6 = max(5, min(args.steps, 50))
        t_6 = timed(lambda: fa.forward(q6, k6, v6, out=o6, lse=l6), n_6, 2, key="d64") / n_6
        f6 = fwd_flops(B6, H6, N6, d6)
        extra["d64_prefill_fwd"] = {"workload": "B=4 H=32 N=4096 d=64 bf16", "tflops": f6 / t_6 / 1e12,
                                    "ms": t_6 * 1e3, "frac_of_bf16_peak": f6 / t_6 / 1e12 / peak,
                                    **per_clock(f6 / t_6 / 1e12, "d64")}
        del q6, k6, v6, o6, l6

    if "causal" in extras:
        # ---------------- causal mask: prefill forward and training backward
        Bc, Hc, Nc = PREFILL["B"], PREFILL["H"], PREFILL["N"]
        qc, kc, vc = randn((Bc, Hc, Nc, d), 14), randn((Bc, Hc, Nc, d), 15), randn((Bc, Hc, Nc, d), 16)
        oc = torch.empty_like(qc)
        lc = torch.empty((Bc, Hc, Nc), dtype=torch.float32, device=dev)
        n_c = max(5, min(args.steps, 50))
        t_c = timed(lambda: fa.forward(qc, kc, vc, out=oc, lse=lc, causal=True), n_c, 2, key="causal_fwd") / n_c
        fc = 4.0 * Bc * Hc * d * Nc * (Nc + 1) / 2          # visible (query, key) pairs only
        del qc, kc, vc, oc, lc
        Bt, Ht, Nt = TRAIN["B"], TRAIN["H"], TRAIN["N"]
        qt, kt, vt, dot = (randn((Bt, Ht, Nt, d), s) for s in (17, 18, 19, 20))
        ot = torch.empty_like(qt)
        lt = torch.empty((Bt, Ht, Nt), dtype=torch.float32, device=dev)
        fa.forward(qt, kt, vt, out=ot, lse=lt, causal=True)
        dq, dk, dv = torch.empty_like(qt), torch.empty_like(kt), torch.empty_like(vt)
        ws_b = torch.empty(fa.backward_workspace_size(Bt, Ht, Nt, d), dtype=torch.uint8, device=dev)
        n_tr = max(3, min(args.steps // 5, 20))
        t_cb = timed(lambda: fa.backward(qt, kt, vt, ot, lt, dot, dq=dq, dk=dk, dv=dv, workspace=ws_b, causal=True),
                     n_tr, 1, key="causal_bwd") / n_tr
        fcb = 2.5 * 4.0 * Bt * Ht * d * Nt * (Nt + 1) / 2
        extra["causal"] = {"flop_count": "4·B·H·d·N(N+1)/2 (visible pairs); backward 2.5x that",
                           "prefill_fwd": {"workload": "B=4 H=32 N=4096 d=128 bf16 causal",
                                           "tflops": fc / t_c / 1e12, "ms": t_c * 1e3,
                                           "frac_of_bf16_peak": fc / t_c / 1e12 / peak,
                                           **per_clock(fc / t_c / 1e12, "causal_fwd")},
                           "train_bwd": {"workload": "B=2 H=16 N=8192 d=128 bf16 causal",
                                         "tflops": fcb / t_cb / 1e12, "ms": t_cb * 1e3,
                                         "frac_of_bf16_peak": fcb / t_cb / 1e12 / peak,
                                         **per_clock(fcb / t_cb / 1e12, "causal_bwd")}}
        del qt, kt, vt, dot, ot, lt, dq, dk, dv, ws_b
    fa.device_status()

    if rank != 0:
        return
    if args.extras_only:
        print(json.dumps({"extras_only": True, "extra": extra}), flush=True)
        return
    cpu = None
    if ws == 1 and not args.no_cpu:
        cv, rows, secs = oracle_sample(args.cpu_seconds)
        cpu = {"value": cv, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": f"float64 oracle, {rows} query rows computed in {secs:.1f} s, taking one prefill head's "
                         f"4096 rows (N=4096, d=128) in turn and repeating them"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el_max / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "prefill forward B=4 H=32 N=4096 d=128 bf16, no mask, fp32 accumulation",
                   "B": B, "H": H, "N": N, "d": d, "parallelism": "replicas" if ws > 1 else "single GPU",
                   "l2": "inputs (3 x 128 MiB) larger than the 129 MB L2, no flush",
                   "inputs": "torch.randn (seeded Philox) on the device, rounded to bf16"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_source": f"{peak_src} bf16_tflops (burst)",
                     "per_clock": per_clock(achieved, "prefill"),
                     "kernel": "fwd_kernel<128, false, false>",
                     "traffic": traffic_for("fwd_prefill", ("fa_fwd.cu", "sm103.cuh"))},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
        "extra": extra,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="headline only (no long/decode/train extras)")
    ap.add_argument("--extras-only", action="store_true",
                    help="for profiling: measure only the listed extra workloads (no headline, no contract line)")
    ap.add_argument("--extras", default="long,decode,gqa,paged,train,causal,fp8,d64",
                    help="comma list of extra workloads measured after the headline")
    ap.add_argument("--decode-batch", type=int, default=DECODE["B"],
                    help="decode batch B (64 is the configured workload; smaller only for profiling)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
