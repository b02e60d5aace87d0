"""Benchmark of the GB300 scaled dot-product attention library.

One step = one forward (O and LSE) plus one backward (dQ, dK, dV) of the
LLaMA-style grouped-query causal workload (B=2, Hq=32, Hkv=8, L=S=4096,
E=Ev=128, bf16), inputs already resident in HBM.  Metric: TFLOP/s with the
nominal FLOP counts 4*B*Hq*L*S*E (forward) and 10*B*Hq*L*S*E (backward),
halved for causal.  In the same run a second leg times the memory-bound
split-KV decode (B=16, Hq=32, Hkv=8, one query token, S=32768, bf16) in HBM
GB/s of K and V read once.

Timing: W warm-up steps, then K steps each bracketed by CUDA events on the
launching stream, with a 256 MiB L2 flush between steps outside the events;
a barrier and a device synchronize on both sides of the timed loop; the max
over ranks.  nvidia-smi clocks are sampled during the timed loop.  "e2e" is
the same step through the same calls with host (pinned) buffers: inputs copied
host->device and every output copied device->host inside the timed region, on
copy streams that overlap the copies with the kernels within each step (dO
comes in during the forward, O and LSE go out during the backward).

--impl reference times the float64 CPU oracle (the parity reference, not a
tuned CPU implementation) on a bounded sample of the same workload.

Multi-GPU (torchrun): every rank runs the same per-GPU workload on its own
GPU with no data exchange (weak scaling); value = all ranks' FLOPs / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SDPA fwd/bwd TFLOP/s and % of GB300 bf16 peak; decode HBM GB/s"
MAIN = "gqa_causal_e128"
DECODE = "gqa_decode_s32k"
NOMINAL_BF16_TFLOPS = 2250.0   # dense bf16 tensor rate of the part (context beside the measured peak)
# Dense bf16 tcgen05.mma rate of one SM, measured on GB300 with chains of M=128, N=256,
# K=128 kind::f16 MMAs, one CTA per SM, timed with clock64: 8173-8182 flop per SM clock
# (the 8192 of one 128x256x16 MMA per 128 clocks, less issue gaps).  The computed
# peak is SMs x this rate x SM clock.
TCGEN05_BF16_FLOP_PER_CLK_SM = 8182.0
SUSTAIN_S = 2.0                # seconds of the same step run right after the timed loop, for clock samples
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode leg")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--workload", default=MAIN,
                    choices=["tiny_f32", "tiny_f32_causal", "mha_causal_e64", "gqa_causal_e128", "padded_mask_e128",
                             "padded_seqlen_e128", "gqa_swa_e128", "gqa_causal_dropout_e128"],
                    help="prefill workload of the step (default: the GQA causal E=128 headline workload)")
    ap.add_argument("--phase", choices=["all", "fwd", "bwd", "decode", "paged"], default="all",
                    help="profiling aid: run only the forward loop, the backward loop, or the dense or paged "
                         "decode leg")
    ap.add_argument("--summarize-launches", metavar="CSV",
                    help="print a per-kernel summary of an ncu launch list (gpu__time_duration.sum, --csv) and exit")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    args.steps = max(1, args.steps)
    return args


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained", "sm_max_mhz")}, \
            "measured"
    except Exception:  # noqa: BLE001
        return dict(FALLBACK_PEAKS), "fallback"


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def job_rate(ws, work_per_rank, t_max_ms, unit):
    """Whole-job rate: every rank did `work_per_rank` (flops or bytes) in parallel, the job
    took the slowest rank's time (ms); in `unit` (1e12 for TFLOP/s, 1e9 for GB/s)."""
    return ws * work_per_rank / (t_max_ms * 1e-3) / unit


def reduce_max(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the block runs; mark() notes host times so that
    summary() can keep only the samples taken inside a window (the loops under load)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None
        self.marks = {}
        self.rows = None

    def mark(self, name):
        import datetime
        self.marks[name] = datetime.datetime.now()

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:  # noqa: BLE001
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()

    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def _load(self):
        if self.rows is not None:
            return self.rows
        import datetime
        self.rows = []
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return self.rows
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                    row = {"ts": ts, "sm": float(parts[2]), "smax": float(parts[3])}
                except ValueError:
                    continue
                try:
                    row["w"] = float(parts[4])
                except ValueError:
                    row["w"] = None
                row["reasons"] = {n for n, v in zip(self.REASONS, parts[6:10]) if v.lower().startswith("active")}
                self.rows.append(row)
        os.unlink(self.path)
        return self.rows

    def summary(self, start=None, end=None):
        """Median SM clock, max clock and throttle reasons of the samples between marks
        `start` and `end` (all samples when not given)."""
        rows = self._load()
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        t0 = self.marks.get(start) if start else None
        t1 = self.marks.get(end) if end else None
        sel = [r for r in rows if (t0 is None or r["ts"] >= t0) and (t1 is None or r["ts"] <= t1)]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0, "reasons": ["no samples"]}
        reasons = set().union(*(r["reasons"] for r in sel))
        watts = [r["w"] for r in sel if r["w"] is not None]
        return {"sm_mhz": statistics.median(r["sm"] for r in sel), "sm_max_mhz": max(r["smax"] for r in sel),
                "sm_mhz_min": min(r["sm"] for r in sel), "samples": len(sel),
                "power_w_median": statistics.median(watts) if watts else None, "reasons": sorted(reasons)}


# ------------------------------------------------------------------ helpers
def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "scaled_dot_product_sm_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, sources):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(kernel)
        if ent and ent.get("source_sha") == source_sha(*sources):
            return float(ent["dram_bytes_per_launch"])
    except Exception:  # noqa: BLE001
        pass
    return None


def visible_pairs(w, spec) -> int:
    """(query, key) pairs a banded workload computes, summed over batches and query heads.

    Row i < Lb of batch b sees keys lo(i)..hi(i) with the padding lengths and band
    of the sdpa_options contract (cuDNN "Attention": Padding mask, Diagonal masking
    options); FLOPs are then 4*E (forward) and 10*E (backward) per pair, the same
    per-pair cost as the nominal formulas.
    """
    import numpy as np
    total = 0
    for b in range(w.B):
        Lb = w.L if spec["seq_len_q"] is None else min(spec["seq_len_q"][b], w.L)
        Sb = w.S if spec["seq_len_kv"] is None else min(spec["seq_len_kv"][b], w.S)
        i = np.arange(Lb, dtype=np.int64)
        diag = i + (Sb - Lb if spec["alignment"] == "bottom_right" else 0)
        hi = np.full(Lb, Sb - 1) if spec["right_bound"] is None else np.minimum(Sb - 1, diag + spec["right_bound"])
        lo = np.zeros(Lb, np.int64) if spec["left_bound"] is None else np.maximum(0, diag - spec["left_bound"] + 1)
        total += int(np.maximum(0, hi - lo + 1).sum())
    return total * w.Hq


def computed_peak_tflops(sms: int, mhz: float) -> float:
    """Datasheet-style dense bf16 peak: SMs x measured tcgen05 flop per SM clock x clock."""
    return sms * TCGEN05_BF16_FLOP_PER_CLK_SM * mhz * 1e6 / 1e12


def fp32_alu_peak_tflops(sms: int, mhz: float) -> float:
    """FFMA peak: SMs x 128 fp32 lanes x 2 flops x clock."""
    return sms * 128 * 2 * mhz * 1e6 / 1e12


# ------------------------------------------------------------------ our arm
def run_ours(args, ws, rank, local):
    import torch

    import scaled_dot_product_sm_gb300 as sdpa
    import workloads

    torch.cuda.set_device(local)
    sdpa.build()
    sdpa.load_library()
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count

    w = workloads.get(args.workload)
    q_h, k_h, v_h, dO_h, m_h = workloads.make_inputs(w, seed=0)
    host = [t.pin_memory() for t in (q_h, k_h, v_h, dO_h)] + ([m_h.pin_memory()] if m_h is not None else [])
    q, k, v, dO = (t.to(dev) for t in host[:4])
    mask = host[4].to(dev) if m_h is not None else None
    spec = workloads.make_band(w, seed=0)
    drop = sdpa.Dropout(w.dropout, 0, 0) if w.dropout > 0 else None
    band = None
    if spec is not None:
        lens = [None if spec[n] is None else torch.tensor(spec[n], dtype=torch.int32).pin_memory()
                for n in ("seq_len_q", "seq_len_kv")]
        host += [t for t in lens if t is not None]
        band = sdpa.Band(*[None if t is None else t.to(dev) for t in lens], spec["alignment"], spec["right_bound"],
                         spec["left_bound"])
    scale = w.scale
    stream = torch.cuda.current_stream()
    o = torch.empty(w.B, w.Hq, w.L, w.Ev, dtype=q.dtype, device=dev)
    lse = torch.empty(w.B, w.Hq, w.L, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    bws = torch.empty(max(16, sdpa.backward_workspace_bytes(q, k, v)), dtype=torch.uint8, device=dev)
    fwd_tc = w.dtype == "bf16" and w.E in (64, 128) and w.Ev in (64, 128)
    bwd_tc = w.dtype == "bf16" and w.E == w.Ev and w.E in (64, 128)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def fwd():
        sdpa.sdpa_forward(q, k, v, mask, scale, w.is_causal, w.enable_gqa, out=o, lse=lse, band=band, dropout=drop)

    def bwd():
        sdpa.sdpa_backward(q, k, v, o, dO, lse, mask, scale, w.is_causal, w.enable_gqa, dq=dq, dk=dk, dv=dv,
                           workspace=bws, band=band, dropout=drop)

    if args.phase in ("decode", "paged"):
        return run_decode_only(args, ws, local, dev, peaks, paged=args.phase == "paged")
    fwd_only = args.phase == "fwd"
    if args.phase == "bwd":
        fwd()
        for _ in range(args.warmup + args.steps):
            bwd()
        torch.cuda.synchronize()
        return {"phase": "bwd", "status": sdpa.last_device_status()}
    for _ in range(args.warmup):
        fwd()
        if not fwd_only:
            bwd()
    torch.cuda.synchronize()
    assert sdpa.last_device_status() == 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.mark("timed_start")
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            evs[i][0].record(stream)
            fwd()
            evs[i][1].record(stream)
            if not fwd_only:
                bwd()
            evs[i][2].record(stream)
        torch.cuda.synchronize()
        clk.mark("timed_end")
        barrier(ws)
        t_fwd = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
        t_bwd = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
        # The same step again, back to back for SUSTAIN_S seconds right after the timed loop
        # (outside it), so that the 200 ms clock samples land under this load; its rate is
        # reported beside the timed one.
        n_sus = max(1, int(SUSTAIN_S * 1e3 / max(t_fwd + t_bwd + 0.05, 1e-3)))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for i in range(n_sus):
            flush.fill_(i & 0xFF)
            fwd()
            if not fwd_only:
                bwd()
        s1.record(stream)
        torch.cuda.synchronize()
        clk.mark("sustain_end")
    barrier(ws)
    clocks = clk.summary("timed_start", "sustain_end")
    clocks["samples_in_timed_loop"] = clk.summary("timed_start", "timed_end").get("samples", 0)
    clocks["window"] = (f"the timed loop and {n_sus} more steps of the same work run back to back after it "
                        f"({s0.elapsed_time(s1) / 1e3:.2f} s)")
    t_step = t_fwd + t_bwd
    t_step_max = reduce_max(t_step, ws)
    sustained = {"steps": n_sus, "ms_per_step_incl_flush": round(s0.elapsed_time(s1) / n_sus, 4)}
    if spec is None:
        f_fwd, f_bwd = w.flops("fwd"), w.flops("bwd")
    else:
        pairs = visible_pairs(w, spec)
        f_fwd, f_bwd = 4.0 * w.E * pairs, 10.0 * w.E * pairs
    value = job_rate(ws, f_fwd + f_bwd, t_step_max, 1e12)
    assert sdpa.last_device_status() == 0

    # ---------------------------------------------------------- end to end (host buffers)
    if fwd_only:
        return {"phase": "fwd", "ms": round(t_fwd, 4), "tflops": round(f_fwd / (t_fwd * 1e-3) / 1e12, 2)}
    e2e = None
    if not args.no_e2e:
        out_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (o, lse, dq, dk, dv)]
        h2d = sum(t.numel() * t.element_size() for t in host)
        d2h = sum(t.numel() * t.element_size() for t in out_h)

        dev_in = (q, k, v, dO) + ((mask,) if mask is not None else ()) + tuple(
            t for t in ((band.seq_len_q, band.seq_len_kv) if band is not None else ()) if t is not None)

        # A step as a user of the stream-taking API runs it: the inputs come in on a copy
        # stream and the results go out on another, overlapped with the kernels, and the
        # step ends when the gradients are on the host.  With no dropout or band (whose
        # counters and lengths are per batch) the batch is pipelined per sequence: each
        # sequence's forward and then its backward, its Q, K, V and dO copied in that order,
        # so batch b + 1's inputs land while batch b computes and batch b's gradients leave
        # while batch b + 1 computes.  For the GQA causal E = 128 step this takes 1.49 ms
        # against 1.65 ms with both forwards before both backwards (dO copied after every
        # Q, K, V).  Finer chunks (a sequence's KV-head groups) measured slower on this host
        # link: 2.04 ms per step in four, 3.14 in eight.  No copy crosses a step boundary:
        # the next step's inputs wait for this step's last kernel.
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        per_batch = w.B > 1 and drop is None and band is None
        nb = w.B if per_batch else 1
        bsl = [slice(i, i + 1) for i in range(w.B)] if per_batch else [slice(0, w.B)]
        mb = (lambda t, sl: t[sl]) if (m_h is not None and m_h.shape[0] == w.B) else (lambda t, sl: t)
        bws_c = [bws] if nb == 1 else [torch.empty(max(16, sdpa.backward_workspace_bytes(q[sl], k[sl], v[sl])),
                                                   dtype=torch.uint8, device=dev) for sl in bsl]
        # copied once per step before the batches: the padding lengths, and the mask unless it
        # is sliced per batch below (one broadcast mask serves every batch)
        mask_per_batch = mask is not None and per_batch and m_h.shape[0] == w.B
        extra_in = [(src, dst) for src, dst in list(zip(host, dev_in))[4:] if not (mask_per_batch and dst is mask)]

        def fwd_c(c):
            sl = bsl[c]
            sdpa.sdpa_forward(q[sl], k[sl], v[sl], None if mask is None else mb(mask, sl), scale, w.is_causal,
                              w.enable_gqa, out=o[sl], lse=lse[sl], band=band, dropout=drop)

        def bwd_c(c):
            sl = bsl[c]
            sdpa.sdpa_backward(q[sl], k[sl], v[sl], o[sl], dO[sl], lse[sl], None if mask is None else mb(mask, sl),
                               scale, w.is_causal, w.enable_gqa, dq=dq[sl], dk=dk[sl], dv=dv[sl],
                               workspace=bws_c[c], band=band, dropout=drop)

        def e2e_step():
            s_in.wait_stream(stream)
            ev_f, ev_b = [], []
            with torch.cuda.stream(s_in):
                for src, dst in extra_in:
                    dst.copy_(src, non_blocking=True)
                for c, sl in enumerate(bsl):   # in the order the kernels use them
                    for src, dst in zip(host[:3], (q, k, v)):
                        dst[sl].copy_(src[sl], non_blocking=True)
                    if mask_per_batch:
                        mask[sl].copy_(host[4][sl], non_blocking=True)
                    ev_f.append(torch.cuda.Event())
                    ev_f[-1].record(s_in)
                    dO[sl].copy_(host[3][sl], non_blocking=True)
                    ev_b.append(torch.cuda.Event())
                    ev_b[-1].record(s_in)
            for c, sl in enumerate(bsl):   # each sequence's forward, then its backward
                stream.wait_event(ev_f[c])
                fwd_c(c)
                ev = torch.cuda.Event()
                ev.record(stream)
                s_out.wait_event(ev)
                with torch.cuda.stream(s_out):
                    out_h[0][sl].copy_(o[sl], non_blocking=True)
                    out_h[1][sl].copy_(lse[sl], non_blocking=True)
                stream.wait_event(ev_b[c])
                bwd_c(c)
                ev = torch.cuda.Event()
                ev.record(stream)
                s_out.wait_event(ev)
                with torch.cuda.stream(s_out):
                    for src, dst in zip((dq, dk, dv), out_h[2:]):
                        dst[sl].copy_(src[sl], non_blocking=True)
            stream.wait_stream(s_out)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(ws)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        t_e2e = reduce_max(e0.elapsed_time(e1) / args.steps, ws)
        # the pipelined step's host results against one call over the whole batch: O, LSE,
        # dK, dV bit for bit, dQ up to the order of its fp32 reductions
        fwd()
        bwd()
        torch.cuda.synchronize()
        for name, got, want in zip(("o", "lse", "dq", "dk", "dv"), out_h, (o, lse, dq, dk, dv)):
            want = want.cpu()
            if name == "dq":
                err = float((got.float() - want.float()).norm() / want.float().norm().clamp_min(1e-30))
                ok = err <= 1e-4
            else:
                ok = torch.equal(got.view(torch.int16) if got.dtype == torch.bfloat16 else got,
                                 want.view(torch.int16) if want.dtype == torch.bfloat16 else want)
            if not ok:
                raise RuntimeError(f"e2e step result {name} differs from the whole-batch call")
        e2e = {"value": round(job_rate(ws, f_fwd + f_bwd, t_e2e, 1e12), 2), "unit": "TFLOP/s",
               "ms_per_step": round(t_e2e, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "gpu_launches_per_step": nb * 4, "batches_pipelined": nb}

    # ---------------------------------------------------------- launches and roofline
    bwd_launches = 3   # tensor cores: row stats, main, dQ convert; CUDA cores: pre-pass, dQ, dK/dV
    fwd_launches = 1
    launches = args.steps * (fwd_launches + bwd_launches)
    med_mhz = clocks.get("sm_mhz") or peaks["sm_max_mhz"]
    cpeak_max = computed_peak_tflops(sms, peaks["sm_max_mhz"])
    cpeak_med = computed_peak_tflops(sms, med_mhz)

    def phase(ms, flops, kernel, nl):
        tf = flops / (ms * 1e-3) / 1e12
        return {"ms": round(ms, 4), "tflops": round(tf, 2),
                "frac_of_computed_peak": round(tf / cpeak_max, 4),
                "frac_of_computed_peak_at_median_clock": round(tf / cpeak_med, 4),
                "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                "frac_of_2250_nominal": round(tf / NOMINAL_BF16_TFLOPS, 4),
                "kcycles_at_median_clock": round(ms * med_mhz, 1),
                "kernel": kernel, "launches_per_step": nl}

    phases = {
        "fwd": phase(t_fwd, f_fwd, "fwd_tc_kernel" if fwd_tc else "fwd_simt_kernel", fwd_launches),
        "bwd": phase(t_bwd, f_bwd, "bwd_tc_kernel" if bwd_tc else "bwd_dq_simt_kernel+bwd_dkdv_simt_kernel",
                     bwd_launches),
    }
    computed_peak = {
        "tflops_at_max_clock": round(cpeak_max, 1), "tflops_at_median_clock": round(cpeak_med, 1),
        "sms": sms, "flop_per_clk_per_sm": TCGEN05_BF16_FLOP_PER_CLK_SM, "max_mhz": peaks["sm_max_mhz"],
        "median_mhz": med_mhz,
        "how": "SMs x dense bf16 tcgen05.mma flop per SM clock (measured: chains of M=128, N=256 kind::f16 "
               "MMAs, one CTA per SM, clock64) x SM clock (the part's maximum, and the median sampled under "
               "this load)"}
    if t_fwd >= t_bwd and not fwd_tc:
        achieved = f_fwd / (t_fwd * 1e-3) / 1e12
        pk = fp32_alu_peak_tflops(sms, peaks["sm_max_mhz"])
        roof = {"kernel": "fwd_simt_kernel", "bound": "alu", "achieved": round(achieved, 2), "peak": round(pk, 1),
                "unit": "TFLOP/s", "frac": round(achieved / pk, 4), "traffic": None,
                "peak_source": f"FFMA: {sms} SMs x 128 lanes x 2 x {peaks['sm_max_mhz']:.0f} MHz",
                "algorithmic_per_launch": f_fwd}
    elif t_fwd >= t_bwd:
        achieved = f_fwd / (t_fwd * 1e-3) / 1e12
        roof = {"kernel": "fwd_tc_kernel", "bound": "tensor", "achieved": round(achieved, 2),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16_tflops"], 4),
                "traffic": (traffic_for("fwd_tc_kernel", ["fwd_tc_kernel.cuh", "ptx.cuh", "common.cuh"])
                            if w.name == MAIN else None),
                "peak_source": f"{peak_src} bf16 dense burst",
                "algorithmic_per_launch": f_fwd}
    else:
        achieved = f_bwd / (t_bwd * 1e-3) / 1e12
        if bwd_tc:
            roof = {"kernel": "bwd_tc_kernel", "bound": "tensor", "achieved": round(achieved, 2),
                    "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": round(achieved / peaks["bf16_tflops"], 4),
                    "traffic": (traffic_for("bwd_tc_kernel", ["bwd_tc.cu", "ptx.cuh", "common.cuh"])
                                if w.name == MAIN else None),
                    "peak_source": f"{peak_src} bf16 dense burst", "algorithmic_per_launch": f_bwd}
        else:
            pk = fp32_alu_peak_tflops(sms, peaks["sm_max_mhz"])
            roof = {"kernel": "bwd_dq_simt_kernel+bwd_dkdv_simt_kernel", "bound": "alu",
                    "achieved": round(achieved, 2), "peak": round(pk, 1), "unit": "TFLOP/s",
                    "frac": round(achieved / pk, 4), "traffic": None,
                    "peak_source": f"FFMA: {sms} SMs x 128 lanes x 2 x {peaks['sm_max_mhz']:.0f} MHz",
                    "algorithmic_per_launch": f_bwd}
    roof["duration_ms"] = round(max(t_fwd, t_bwd), 4)
    if roof["bound"] == "tensor":
        roof["frac_of_computed_peak"] = round(roof["achieved"] / cpeak_max, 4)
        roof["frac_of_computed_peak_at_median_clock"] = round(roof["achieved"] / cpeak_med, 4)

    # ---------------------------------------------------------- decode leg
    decode = None
    if not args.no_decode:
        del flush
        wd = workloads.get(DECODE)
        qd_h, kd_h, vd_h, _, _ = workloads.make_inputs(wd, seed=0, with_grad=False)
        qd, kd, vd = qd_h.to(dev), kd_h.to(dev), vd_h.to(dev)
        del qd_h, kd_h, vd_h
        od = torch.empty(wd.B, wd.Hq, 1, wd.Ev, dtype=qd.dtype, device=dev)
        lsed = torch.empty(wd.B, wd.Hq, 1, dtype=torch.float32, device=dev)
        dws = torch.empty(max(16, sdpa.decode_workspace_bytes(qd, kd, vd, 0)), dtype=torch.uint8, device=dev)
        nsplit = sdpa.decode_num_splits(qd, kd, vd)

        def dstep():
            sdpa.sdpa_decode(qd, kd, vd, None, wd.scale, True, 0, out=od, lse=lsed, workspace=dws)

        for _ in range(args.warmup):
            dstep()
        torch.cuda.synchronize()
        dev_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
        barrier(ws)
        torch.cuda.synchronize()
        with ClockSampler(local) as dclk:
            dclk.mark("timed_start")
            for i in range(args.steps):
                dev_evs[i][0].record(stream)
                dstep()
                dev_evs[i][1].record(stream)
            torch.cuda.synchronize()
            dclk.mark("timed_end")
            t_dec1 = sum(a.elapsed_time(b) for a, b in dev_evs) / args.steps
            for _ in range(max(1, int(SUSTAIN_S * 1e3 / max(t_dec1, 1e-3)))):   # clock samples under load
                dstep()
            torch.cuda.synchronize()
            dclk.mark("sustain_end")
        barrier(ws)
        t_dec = reduce_max(t_dec1, ws)
        dclocks = dclk.summary("timed_start", "sustain_end")
        dclocks["samples_in_timed_loop"] = dclk.summary("timed_start", "timed_end").get("samples", 0)
        kv_bytes = (kd.numel() + vd.numel()) * kd.element_size()
        io_bytes = kv_bytes + qd.numel() * 2 + od.numel() * 2 + lsed.numel() * 4
        gbps = job_rate(ws, io_bytes, t_dec, 1e9)
        decode = {"workload": DECODE, "ms": round(t_dec, 4), "gbps": round(gbps, 1),
                  "frac_of_8tbs_nominal": round(gbps / ws / 8000.0, 4),
                  "frac_of_measured_hbm": round(gbps / ws / peaks["hbm_gbs"], 4),
                  "denominators": "headline: the 8 TB/s nominal HBM3e rate; beside it the measured copy "
                                  "(a read+write stream, which runs below what a read-only stream such as "
                                  "this one reaches, so its fraction can pass 1)",
                  "algorithmic_bytes": io_bytes, "splits": nsplit, "launches_per_step": 2,
                  "kernels": ["decode_split_kernel", "decode_merge_kernel"],
                  "traffic": traffic_for("decode_split_kernel", ["decode.cu", "ptx.cuh", "common.cuh"]),
                  "clocks": dclocks,
                  "l2": "inputs (2.1 GB of K/V) larger than L2; no flush"}
        launches += args.steps * 2
        assert sdpa.last_device_status() == 0

        # the same caches as a paged cache: 64-key blocks in shuffled order in one container each
        bsz = 64
        nbs = wd.S // bsz
        perm = torch.randperm(wd.B * nbs, generator=torch.Generator().manual_seed(1)).to(dev)

        kc = paged_container(kd, wd.B, wd.Hkv, wd.S, bsz, perm)
        vc = paged_container(vd, wd.B, wd.Hkv, wd.S, bsz, perm)
        del kd, vd
        table = perm.reshape(wd.B, nbs).to(torch.int32).contiguous()

        def pstep():
            sdpa.sdpa_decode_paged(qd, kc, vc, table, table, wd.S, None, wd.scale, True, 0, out=od, lse=lsed,
                                   workspace=dws)

        for _ in range(args.warmup):
            pstep()
        torch.cuda.synchronize()
        barrier(ws)
        torch.cuda.synchronize()
        for i in range(args.steps):
            dev_evs[i][0].record(stream)
            pstep()
            dev_evs[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        t_pg = reduce_max(sum(a.elapsed_time(b) for a, b in dev_evs) / args.steps, ws)
        gbps_pg = job_rate(ws, io_bytes, t_pg, 1e9)
        decode["paged"] = {"block_size": bsz, "layout": "64-key blocks of every sequence shuffled in one container",
                           "ms": round(t_pg, 4), "gbps": round(gbps_pg, 1),
                           "frac_of_measured_hbm": round(gbps_pg / ws / peaks["hbm_gbs"], 4)}
        launches += args.steps * 2
        assert sdpa.last_device_status() == 0

    # ---------------------------------------------------------- CPU baseline (oracle)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        cpu = cpu_oracle_groups(w, seconds_target=12.0)
        if decode is not None:
            decode["cpu_baseline"] = cpu_oracle_groups(workloads.get(DECODE), seconds_target=8.0)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_step_max, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "L": w.L, "S": w.S, "E": w.E,
                   "Ev": w.Ev, "causal": w.is_causal, "gqa": w.enable_gqa, "scale": w.scale,
                   "mask": w.mask, "band": spec, "dropout": w.dropout,
                   "flops": "visible (query, key) pairs x 4E / 10E" if spec is not None else
                            "4/10 x B*Hq*L*S*E, halved for causal",
                   "step": "forward (O, LSE) + backward (dQ, dK, dV)", "seed": 0,
                   "l2": "256 MiB flush between timed steps, outside the events",
                   "parallelism": f"replicas x{ws} (no exchange)"},
        "phases": phases,
        "computed_peak": computed_peak,
        "sustained": sustained,
        "roofline": roof,
        "decode": decode,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "peaks": {"source": peak_src, **peaks},
        "gpu": props.name, "sms": sms,
    }
    return line


def paged_container(x, B, Hkv, S, bsz, perm):
    """Dense cache [B, Hkv, S, D] as a paged container: its bsz-key blocks in the shuffled order
    `perm` (block b * (S / bsz) + i of the cache goes to container block perm[...])."""
    import torch
    nbs = S // bsz
    blocks = x.reshape(B, Hkv, nbs, bsz, x.shape[3]).permute(0, 2, 1, 3, 4).reshape(B * nbs, Hkv, bsz, x.shape[3])
    c = torch.empty_like(blocks)
    c[perm] = blocks
    return c


def run_decode_only(args, ws, local, dev, peaks, paged=False):
    import torch

    import scaled_dot_product_sm_gb300 as sdpa
    import workloads
    wd = workloads.get(DECODE)
    qd_h, kd_h, vd_h, _, _ = workloads.make_inputs(wd, seed=0, with_grad=False)
    qd, kd, vd = qd_h.to(dev), kd_h.to(dev), vd_h.to(dev)
    od = torch.empty(wd.B, wd.Hq, 1, wd.Ev, dtype=qd.dtype, device=dev)
    lsed = torch.empty(wd.B, wd.Hq, 1, dtype=torch.float32, device=dev)
    dws = torch.empty(max(16, sdpa.decode_workspace_bytes(qd, kd, vd, 0)), dtype=torch.uint8, device=dev)
    if paged:   # 64-key blocks of every sequence shuffled in one container, as in the bench's paged leg
        bsz = 64
        perm = torch.randperm(wd.B * (wd.S // bsz), generator=torch.Generator().manual_seed(1)).to(dev)
        kc = paged_container(kd, wd.B, wd.Hkv, wd.S, bsz, perm)
        vc = paged_container(vd, wd.B, wd.Hkv, wd.S, bsz, perm)
        del kd, vd
        table = perm.reshape(wd.B, wd.S // bsz).to(torch.int32).contiguous()
        for _ in range(args.warmup + args.steps):
            sdpa.sdpa_decode_paged(qd, kc, vc, table, table, wd.S, None, wd.scale, True, 0, out=od, lse=lsed,
                                   workspace=dws)
    else:
        for _ in range(args.warmup + args.steps):
            sdpa.sdpa_decode(qd, kd, vd, None, wd.scale, True, 0, out=od, lse=lsed, workspace=dws)
    torch.cuda.synchronize()
    return {"phase": "paged" if paged else "decode", "status": sdpa.last_device_status()}


# ------------------------------------------------------------------ CPU oracle
def group_work(w, spec, b):
    """Algorithmic work of one KV group (the Hq/Hkv query heads of batch b sharing a KV head):
    forward + backward FLOPs (4E + 10E per visible (query, key) pair), or for a forward-only
    workload the bytes of K and V read once plus Q, O and LSE."""
    G = w.Hq // w.Hkv
    if "bwd" not in w.phases:
        return 2.0 * w.S * (w.E + w.Ev) + G * w.L * (2.0 * (w.E + w.Ev) + 4.0)
    if spec is None:
        one = w.with_(B=1, Hq=G, Hkv=1)
        return one.flops("fwd") + one.flops("bwd")
    sb = dict(spec, **{n: None if spec[n] is None else spec[n][b:b + 1] for n in ("seq_len_q", "seq_len_kv")})
    return 14.0 * w.E * visible_pairs(w.with_(B=1, Hq=G, Hkv=1), sb)


def cpu_oracle_groups(w, seconds_target=12.0):
    """The float64 oracle, as it stands, on whole KV groups of workload w in order (batch-major),
    on the host cores: as many groups as fit in about `seconds_target` seconds, at least one.
    Each KV group is a closed sub-problem (its query heads with all their queries and keys), so
    the whole configuration's time is the sampled time scaled by the work of all groups over
    that of the sampled ones ("extrapolated" unless every group ran)."""
    import oracle
    import workloads
    fwd_only = "bwd" not in w.phases
    q, k, v, dO, mask = workloads.make_inputs(w, seed=0, with_grad=not fwd_only)
    spec = workloads.make_band(w, seed=0)
    band = None if spec is None else oracle.Band(spec["seq_len_q"], spec["seq_len_kv"], spec["alignment"],
                                                 spec["right_bound"], spec["left_bound"])
    drop = oracle.Dropout(w.dropout, 0, 0) if w.dropout > 0 else None
    groups = [(b, kv) for b in range(w.B) for kv in range(w.Hkv)]
    done, t_sum, work = 0, 0.0, 0.0
    for b, kv in groups:
        t0 = time.perf_counter()
        oracle.ref_group(q, k, v, None if fwd_only else dO, b, kv, mask, w.scale, w.is_causal, band=band,
                         dropout=drop)
        t_sum += time.perf_counter() - t0
        work += group_work(w, spec, b)
        done += 1
        if t_sum >= seconds_target:
            break
    total = sum(group_work(w, spec, b) for b, _ in groups)
    unit, scale = ("GB/s", 1e9) if fwd_only else ("TFLOP/s", 1e12)
    what = "forward" if fwd_only else "forward + backward"
    return {"value": round(work / t_sum / scale, 6), "unit": unit, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{w.name}: {done} of {len(groups)} KV groups (b, kv) in batch-major order, each "
                      f"{w.Hq // w.Hkv} query heads with all their queries and keys, {what}, float64 NumPy "
                      f"oracle, BLAS default threads; {t_sum:.2f} s",
            "groups_timed": done, "groups_total": len(groups), "seconds_sampled": round(t_sum, 3),
            "config_seconds": round(t_sum * total / work, 2), "extrapolated": done < len(groups)}


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    import oracle
    import workloads
    w = workloads.get(MAIN)
    q, k, v, dO, _ = workloads.make_inputs(w, seed=0)
    # one query head (b = 0, h = 0) with all its queries and keys, forward + backward: a
    # sample that keeps the run short even where the launcher gives BLAS one thread per rank
    qs, ks, vs, dOs = q[:1, :1], k[:1, :1], v[:1, :1], dO[:1, :1]
    del q, k, v, dO
    flops = w.with_(B=1, Hq=1, Hkv=1).flops("fwd") + w.with_(B=1, Hq=1, Hkv=1).flops("bwd")

    def step():
        oracle.ref_forward(qs, ks, vs, None, w.scale, w.is_causal)
        oracle.ref_backward(qs, ks, vs, dOs, None, w.scale, w.is_causal)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    t = (time.perf_counter() - t0) / args.steps
    value = flops / t / 1e12
    sample = (f"{MAIN}: one query head (b=0, h=0: 1 of {w.B * w.Hq}, all its queries and keys) per step, "
              f"forward + backward, float64 NumPy oracle; BLAS default threads")
    return {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": MAIN, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "L": w.L, "S": w.S, "E": w.E,
                       "Ev": w.Ev, "causal": w.is_causal, "gqa": w.enable_gqa, "seed": 0,
                       "step": "forward + backward of one query head (sample)"},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def summarize_launches(path):
    """Per-kernel launches, total device time and share from an ncu --csv launch list."""
    import collections
    import csv
    scale = {"ns": 1e-3, "nsecond": 1e-3, "us": 1.0, "usecond": 1.0, "ms": 1e3, "msecond": 1e3, "s": 1e6,
             "second": 1e6}
    rows = [r for r in csv.reader(open(path)) if r]
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    h = rows[hi]
    ki, mi, vi, ui = (h.index(x) for x in ("Kernel Name", "Metric Name", "Metric Value", "Metric Unit"))
    agg = collections.defaultdict(lambda: [0, 0.0])
    for r in rows[hi + 1:]:
        if len(r) <= vi or r[mi] != "gpu__time_duration.sum":
            continue
        name = r[ki].split("(")[0].replace("void ", "")
        agg[name][0] += 1
        agg[name][1] += float(r[vi].replace(",", "")) * scale[r[ui]]
    tot = sum(t for _, t in agg.values())
    lines = [f"{'kernel':78s} {'launches':>8s} {'total ms':>10s} {'share':>7s}"]
    for k, (n, t) in sorted(agg.items(), key=lambda x: -x[1][1]):
        lines.append(f"{k[:78]:78s} {n:8d} {t / 1e3:10.3f} {100 * t / tot:6.2f}%")
    return "\n".join(lines)


def main():
    args = parse()
    if args.summarize_launches:
        print(summarize_launches(args.summarize_launches))
        return
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, ws, rank)
    else:
        line = run_ours(args, ws, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
