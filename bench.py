#!/usr/bin/env python
"""MSA forward benchmark on GB300: prefill tokens/s at 128K and decode tokens/s.

One step of the prefill workload is the whole hot path over one 131072-token
sequence (block 128, top-16): msa_index_select then msa_sparse_attn_prefill.
One decode step is 64 sequences x 1 new token over KV caches of 32K-128K:
msa_index_select (Nq = 1) then msa_sparse_attn_decode. Inputs are synthetic
(seeded, generated on the device) and resident in HBM when timing starts.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {msa,reference}]

Prints ONE JSON line on rank 0. Under torchrun every rank runs the same
workload on its own GPU (independent replicas; no collective on the data
path) and `value` is the sum over ranks of tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MSA prefill tokens/s @128K and decode tokens/s (1 GB300) + % of roofline"
L2_NOTE = ("flushed between timed steps (a 512 MB write, then a 512 MB read so that the flush's dirty lines "
           "are written back before the step starts)")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {  # kernel name -> source file (for the ncu traffic freshness check)
    "index_blockmax_table": "index_table.cu", "topk_from_table": "index_table.cu",
    "attn_query_outer": "attn_query_outer.cu", "index_fused_tc": "index_fused_tc.cu",
    "index_topk_table": "index_fused_tc.cu",
    "attn_kv_outer_tc": "attn_kv_outer_tc.cu", "attn_invert": "attn_kv_outer_tc.cu",
    "attn_combine": "attn_kv_outer_tc.cu", "decode_index": "decode.cu", "decode_topk": "decode.cu",
    "decode_attn": "decode.cu", "kl_tile": "attn_kv_outer_tc.cu",
    "kl_combine": "attn_kv_outer_tc.cu", "bwd_tile": "attn_backward.cu", "bwd_dq_combine": "attn_backward.cu",
    "kl_tile_tc": "kl_tc.cu", "bwd_tile_tc": "attn_backward.cu",
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["msa", "reference"], default="msa")
    ap.add_argument("--workload", default="prefill_128k_bs128")
    ap.add_argument("--decode-workload", default="decode_b64")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-kl", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the Bs 64/32 and 1M prefill legs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=0, help="oracle sample rows (0 = auto)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas)
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist

            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        return reduce_scalar(self.pg, x, "max")

    def sum(self, x: float) -> float:
        return reduce_scalar(self.pg, x, "sum")


def reduce_scalar(pg, x: float, op: str) -> float:
    """Max / sum of one float over ranks (identity without a process group)."""
    if pg is None:
        return float(x)
    import torch

    dev = "cuda" if (torch.cuda.is_available() and pg.get_backend() == "nccl") else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX if op == "max" else pg.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# measurement helpers
# ---------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def src_sha(kernel: str) -> str | None:
    f = KERNEL_SOURCES.get(kernel)
    if not f:
        return None
    path = os.path.join(ROOT, "block_sparse_long_select_gb300", "csrc", f)
    if not os.path.exists(path):
        return None
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of that kernel (profiles/*.md line:
    `ncu-traffic <kernel> <workload> <bytes_per_launch> <src sha256[:16]>`)."""
    sha = src_sha(kernel)
    pdir = os.path.join(ROOT, "profiles")
    if not sha or not os.path.isdir(pdir):
        return None
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".md", ".txt")):
            continue
        for line in open(os.path.join(pdir, fn)):
            m = re.match(r"\s*ncu-traffic\s+(\S+)\s+(\S+)\s+([0-9.eE+]+)\s+([0-9a-f]+)", line)
            if m and m.group(1) == kernel and m.group(2) == workload and m.group(4) == sha:
                return float(m.group(3))
    return None


# ---------------------------------------------------------------------------
# algorithmic work (what the method must do, independent of the kernels)
# ---------------------------------------------------------------------------
def attended_keys(sel, q_offset, kv_len, Bs):
    """Sum over (b, i, g) of the number of attended keys (selected blocks
    intersected with j <= pos, j < kv_len)."""
    import torch

    B, Nq, G, K = sel.shape
    dev = sel.device
    pos = (torch.as_tensor(q_offset, device=dev).view(B, 1, 1, 1) +
           torch.arange(Nq, device=dev).view(1, Nq, 1, 1))
    L = torch.as_tensor(kv_len, device=dev).view(B, 1, 1, 1)
    t = sel.long()
    lo = t * Bs
    hi = torch.minimum(torch.minimum(lo + Bs, pos + 1), L)
    n = torch.clamp(hi - lo, min=0) * (t >= 0)
    return int(n.sum().item())


def prefill_work(w, sel, qo, kl):
    pos = qo[:, None].astype(np.int64) + np.arange(w.Nq)[None, :]
    visible = np.minimum(pos + 1, kl[:, None]).sum()
    att = attended_keys(sel, qo, kl, w.Bs)
    # top-K over a block-max table: the candidate maxima t < loc of every row
    # that ranks (more than K visible blocks) read once, the selection written
    loc = pos // w.Bs
    cand = np.where(loc + 1 > w.K, loc, 0).sum()
    return {"index_flops": 2.0 * w.di * w.G * float(visible),
            "attn_flops": 4.0 * w.d * (w.Hq // w.G) * float(att),
            "topk_bytes": 4.0 * w.G * float(cand) + 4.0 * w.K * w.G * w.B * w.Nq,
            "attended_keys": att, "visible_keys": int(visible)}


def decode_work(w, sel, kl):
    att = attended_keys(sel, kl - 1, kl, w.Bs)  # summed over (b, g)
    ik_bytes = float(kl.astype(np.int64).sum()) * w.di * 2
    kv_bytes = float(att) * w.d * 2 * 2
    small = w.B * (w.Hq * w.d * 2 * 2 + w.G * w.di * 2 + w.G * w.K * 4)
    return {"index_bytes": ik_bytes, "attn_bytes": kv_bytes + w.B * w.Hq * w.d * 4, "total_bytes": ik_bytes +
            kv_bytes + small, "index_flops": 2.0 * w.di * w.G * float(kl.sum()),
            "attn_flops": 4.0 * w.d * (w.Hq // w.G) * float(att), "attended_keys": att}


def kl_work(w, work):
    """The KL auxiliary pass recomputes, for every attended key of every
    (query, group), the Hq/G main scores (2 d flops each) and the index score
    (2 di flops): the score half of the attention plus the index dot products
    restricted to the selection."""
    att = work["attended_keys"]
    return {"kl_flops": 2.0 * w.d * (w.Hq // w.G) * float(att) + 2.0 * w.di * float(att)}


def backward_work(w, work):
    """The backward recomputes S and forms dP, then the dV, dK and dQ products:
    five d-long dot products per (token, head, attended key)."""
    return {"bwd_flops": 10.0 * w.d * (w.Hq // w.G) * float(work["attended_keys"])}


def roofline_for(kernel, prof, work, peaks, peak_src, workload, steps, mode="prefill"):
    """Roofline entry of one kernel. achieved = algorithmic work per launch /
    mean launch duration, both from the timed region: the per-step work of the
    step that kernel serves x steps / launches, over the summed CUDA-event
    time of its launches (recorded on its own stream). Prefill kernels are
    contractions (tensor-bound); decode kernels stream their inputs once
    (HBM-bound)."""
    launches, total_ms = prof[kernel]
    per_launch_s = total_ms / 1e3 / launches
    if mode == "decode":
        if "index" in kernel:
            bound, unit, per_step = "hbm", "GB/s", work["index_bytes"]
        elif "attn" in kernel:
            bound, unit, per_step = "hbm", "GB/s", work["attn_bytes"]
        else:
            return None
    elif kernel in ("index_fused_tc", "index_blockmax_table"):
        bound, unit, per_step = "tensor", "TFLOP/s", work["index_flops"]
    elif kernel == "index_topk_table":
        bound, unit, per_step = "hbm", "GB/s", work["topk_bytes"]
    elif kernel in ("attn_kv_outer_tc", "attn_query_outer"):
        bound, unit, per_step = "tensor", "TFLOP/s", work["attn_flops"]
    elif kernel in ("kl_tile", "kl_tile_tc"):
        bound, unit, per_step = "tensor", "TFLOP/s", work["kl_flops"]
    elif kernel in ("bwd_tile", "bwd_tile_tc"):
        bound, unit, per_step = "tensor", "TFLOP/s", work["bwd_flops"]
    else:
        return None
    amount = per_step * steps / launches
    if bound == "tensor":
        # the burst figure: these kernels run inside steps of milliseconds to a
        # fraction of a second, not seconds-long loops under the power cap
        achieved = amount / per_launch_s / 1e12
        peak, peak_name = peaks["bf16_tflops"], "bf16_tflops (burst)"
    else:
        achieved = amount / per_launch_s / 1e9
        peak, peak_name = peaks["hbm_gbs"], "hbm_gbs"
    return {"kernel": kernel, "bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": ncu_traffic(kernel, workload),
            "algorithmic_per_launch": amount, "launches_per_step": launches / steps,
            "launch_ms": round(per_launch_s * 1e3, 4), "peak_source": f"{peak_name} ({peak_src})"}


# ---------------------------------------------------------------------------
# the timed MSA arm
# ---------------------------------------------------------------------------
def run_msa(args, dist):
    import torch

    import block_sparse_long_select_gb300 as msa

    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    msa.load_library()
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)  # > 129 MB L2
    # Read after the flush write: L2 is write-back, so the flush leaves L2 full
    # of dirty lines whose write-back would otherwise fall inside the next
    # step (about 8 % of a decode step). Reading past L2 retires them first
    # and leaves only clean lines of this buffer; the step's inputs stay cold.
    retire = torch.zeros((512 << 20) // 4, dtype=torch.float32, device=dev)

    def time_steps(step, K, W, profile=True):
        for _ in range(W):
            step()
        torch.cuda.synchronize(dev)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        sampler = ClockSampler(dev.index if dev.index is not None else 0)
        dist.barrier()
        torch.cuda.synchronize(dev)
        sampler.start()
        if profile:
            msa.msa_profile_begin()
        t0 = time.perf_counter()
        for s in range(K):
            flush.zero_()  # evict L2 between timed steps (outside the step events)
            retire.sum()  # and write its dirty lines back before the step starts
            starts[s].record(stream)
            step()
            ends[s].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        prof = msa.msa_profile_end() if profile else {}
        dist.barrier()
        clocks = sampler.stop()
        ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        return ms, prof, clocks, wall

    # ----------------------------- prefill -----------------------------
    w = synth.WORKLOADS[args.workload]
    qo_np, kl_np = synth.q_offsets(w), synth.kv_lens(w)
    t = {n: synth.device_tensor(w, n, dev) for n in ("q", "k", "v", "iq", "ik")}
    qo = torch.from_numpy(qo_np).to(dev)
    kl = torch.from_numpy(kl_np).to(dev)
    sel = torch.empty((w.B, w.Nq, w.G, w.K), dtype=torch.int32, device=dev)
    out = torch.empty_like(t["q"])
    ws_i = msa.workspace(msa.msa_workspace_size(msa.MSA_OP_INDEX_SELECT, w.B, w.Nq, w.Nk, w.G, 0, 0, w.di, w.Bs,
                                                w.K, msa.MSA_BF16), dev)
    ws_a = msa.workspace(msa.msa_workspace_size(msa.MSA_OP_PREFILL, w.B, w.Nq, w.Nk, w.G, w.Hq, w.d, 0, w.Bs, w.K,
                                                msa.MSA_BF16), dev)

    def prefill_step():
        msa.msa_index_select(t["iq"], t["ik"], qo, kl, w.Bs, w.K, sel=sel, ws=ws_i)
        msa.msa_sparse_attn_prefill(t["q"], t["k"], t["v"], sel, qo, kl, w.Bs, w.K, out=out, ws=ws_a)

    # the timed pass has no events between kernels (they would serialise the
    # library's overlapped launches); a second pass of the same steps times
    # each kernel with CUDA events for the breakdown and the rooflines
    ms, _, clocks, wall = time_steps(prefill_step, args.steps, args.warmup, profile=False)
    _, prof, _, _ = time_steps(prefill_step, args.steps, 0, profile=True)
    for ws in (ws_i, ws_a):
        st = msa.msa_read_status(ws)
        if st != 0:
            raise RuntimeError(f"device status after prefill: {msa.msa_status_string(st)}")
    work = prefill_work(w, sel, qo_np, kl_np)
    step_ms = float(np.mean(ms))
    tokens = w.B * w.Nq
    max_total_s = dist.max(sum(ms) / 1e3)
    all_tokens = dist.sum(tokens * args.steps)
    value = all_tokens / max_total_s
    launches = sum(v[0] for v in prof.values())
    dom = max(prof, key=lambda k: prof[k][1]) if prof else None
    roof = roofline_for(dom, prof, work, peaks, peak_src, w.name, args.steps) if dom else None
    kernels = {k: {"launches": v[0], "ms_per_step": round(v[1] / args.steps, 4),
                   "share": round(v[1] / max(sum(x[1] for x in prof.values()), 1e-9), 4)} for k, v in prof.items()}
    all_roofs = [r for r in (roofline_for(k, prof, work, peaks, peak_src, w.name, args.steps) for k in prof) if r]

    # ---------------------------- e2e (host buffers) -------------------
    # Every step copies its inputs from pinned host memory and reads its
    # output back, inside the timed region. The copies run on a second
    # stream, pipelined the way a serving loop runs them: the inputs of step
    # s+1 land in the other of two device input sets while step s computes,
    # and the output of step s is read back as soon as step s is done.
    e2e = None
    if not args.no_e2e:
        host = {n: torch.empty(t[n].shape, dtype=t[n].dtype, pin_memory=True) for n in t}
        for n in t:
            host[n].copy_(t[n])
        qo_h, kl_h = qo.cpu().pin_memory(), kl.cpu().pin_memory()
        out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h2d = sum(x.numel() * x.element_size() for x in host.values()) + 2 * qo.numel() * 4
        d2h = out_h.numel() * out_h.element_size()
        sets = [dict(t, qo=qo, kl=kl, out=out),
                dict({n: torch.empty_like(t[n]) for n in t}, qo=torch.empty_like(qo), kl=torch.empty_like(kl),
                     out=torch.empty_like(out))]
        up = torch.cuda.Stream(dev)    # host -> device: the next step's inputs
        down = torch.cuda.Stream(dev)  # device -> host: the finished step's output (both directions at once)

        def copy_in(k):
            for n in t:
                sets[k][n].copy_(host[n], non_blocking=True)
            sets[k]["qo"].copy_(qo_h, non_blocking=True)
            sets[k]["kl"].copy_(kl_h, non_blocking=True)

        def pipeline(nsteps):
            ready = [torch.cuda.Event() for _ in range(2)]    # a set's inputs have landed
            done = [torch.cuda.Event() for _ in range(2)]     # a set's step has finished (its inputs are free)
            drained = [torch.cuda.Event() for _ in range(2)]  # a set's output has been read back
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            t0.record(stream)
            up.wait_event(t0)
            with torch.cuda.stream(up):
                copy_in(0)
                ready[0].record(up)
            for s_ in range(nsteps):
                k = s_ % 2
                S = sets[k]
                stream.wait_event(ready[k])
                if s_ >= 2:
                    stream.wait_event(drained[k])  # step s-2's output in this set has been read back
                msa.msa_index_select(S["iq"], S["ik"], S["qo"], S["kl"], w.Bs, w.K, sel=sel, ws=ws_i)
                msa.msa_sparse_attn_prefill(S["q"], S["k"], S["v"], sel, S["qo"], S["kl"], w.Bs, w.K, out=S["out"],
                                            ws=ws_a)
                done[k].record(stream)
                if s_ + 1 < nsteps:
                    with torch.cuda.stream(up):
                        if s_ >= 1:
                            up.wait_event(done[1 - k])  # step s-1 no longer reads the other set
                        copy_in(1 - k)
                        ready[1 - k].record(up)
                with torch.cuda.stream(down):
                    down.wait_event(done[k])
                    out_h.copy_(S["out"], non_blocking=True)
                    drained[k].record(down)
            stream.wait_stream(up)
            stream.wait_stream(down)
            t1.record(stream)
            torch.cuda.synchronize(dev)
            return t0.elapsed_time(t1)

        pipeline(2)  # warm-up
        n_e = max(8, 2 * args.steps)  # the pipeline fill (first inputs) and drain (last output) spread over the steps
        # three timed runs of the pipelined loop, the median reported (host
        # copies vary from run to run); each run is n_e full steps
        trials = []
        for _ in range(3):
            dist.barrier()
            trials.append(dist.max(pipeline(n_e) / 1e3))
        e_tot = sorted(trials)[1]
        e2e = {"value": round(dist.sum(tokens * n_e) / e_tot, 1), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e_tot * 1e3 / n_e, 4), "steps": n_e,
               "trials_ms_per_step": [round(x * 1e3 / n_e, 4) for x in trials], "statistic": "median of 3 runs",
               "copies": "pinned host buffers; an upload stream copies step s+1's inputs and a download stream reads "
                         "step s-1's output back while step s computes"}
        del host, out_h, sets

    torch.cuda.empty_cache()

    # ------------------------- KL auxiliary forward ---------------------
    # msa_kl_aux_forward over the prefill's selection and lse (one prefill
    # with lse output before the timed region); a step is one KL pass
    kl_leg = bwd_leg = None
    if not (args.no_kl and args.no_backward):
        lse = torch.empty((w.B, w.Nq, w.Hq), dtype=torch.float32, device=dev)
        msa.msa_index_select(t["iq"], t["ik"], qo, kl, w.Bs, w.K, sel=sel, ws=ws_i)
        msa.msa_sparse_attn_prefill(t["q"], t["k"], t["v"], sel, qo, kl, w.Bs, w.K, out=out, lse=lse, ws=ws_a)
    if not args.no_kl:
        klo = torch.empty((w.B, w.Nq, w.G), dtype=torch.float32, device=dev)
        ws_k = msa.workspace(msa.msa_workspace_size(msa.MSA_OP_KL_AUX, w.B, w.Nq, w.Nk, w.G, w.Hq, w.d, w.di, w.Bs,
                                                    w.K, msa.MSA_BF16), dev)

        def kl_step():
            msa.msa_kl_aux_forward(t["q"], t["k"], t["iq"], t["ik"], sel, lse, qo, kl, w.Bs, w.K, kl=klo, ws=ws_k)

        kms, _, kclocks, _ = time_steps(kl_step, args.steps, args.warmup, profile=False)
        _, kprof, _, _ = time_steps(kl_step, args.steps, 0, profile=True)
        st = msa.msa_read_status(ws_k)
        if st != 0:
            raise RuntimeError(f"device status after KL: {msa.msa_status_string(st)}")
        if not bool(torch.isfinite(klo).all()):
            raise RuntimeError("KL auxiliary output not finite")
        kwork = kl_work(w, work)
        k_tot = dist.max(sum(kms) / 1e3)
        kl_leg = {"value": round(dist.sum(tokens * args.steps) / k_tot, 1), "unit": "tokens/s",
                  "ms_per_step": round(float(np.mean(kms)), 4), "steps": args.steps,
                  "what": "msa_kl_aux_forward: KL(head-averaged main distribution || index softmax) over the "
                          "selected keys of every (query, group), from the forward's lse",
                  "roofline": next((roofline_for(k_, kprof, kwork, peaks, peak_src, w.name, args.steps)
                                    for k_ in ("kl_tile_tc", "kl_tile") if k_ in kprof), None),
                  "kernels": {k: {"launches": v[0], "ms_per_step": round(v[1] / args.steps, 4)}
                              for k, v in kprof.items()},
                  "gpu_launches": sum(v[0] for v in kprof.values()), "clocks": kclocks,
                  "kl_flops_per_step": kwork["kl_flops"]}
        del klo, ws_k
    # ------------------------- Main Branch backward ---------------------
    # msa_sparse_attn_backward over the prefill's selection, output and lse
    # with a synthetic output gradient; a step is one backward pass
    if not args.no_backward:
        dout = synth.device_tensor(synth.scaled(w, seed=w.seed + 1000), "q", dev)
        dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
        ws_b = msa.workspace(msa.msa_workspace_size(msa.MSA_OP_BACKWARD, w.B, w.Nq, w.Nk, w.G, w.Hq, w.d, 0, w.Bs,
                                                    w.K, msa.MSA_BF16), dev)

        def bwd_step():
            msa.msa_sparse_attn_backward(t["q"], t["k"], t["v"], out, dout, lse, sel, qo, kl, w.Bs, w.K, dq=dq,
                                         dk=dk, dv=dv, ws=ws_b)

        bms, _, bclocks, _ = time_steps(bwd_step, args.steps, args.warmup, profile=False)
        _, bprof, _, _ = time_steps(bwd_step, args.steps, 0, profile=True)
        st = msa.msa_read_status(ws_b)
        if st != 0:
            raise RuntimeError(f"device status after backward: {msa.msa_status_string(st)}")
        bwork = backward_work(w, work)
        b_tot = dist.max(sum(bms) / 1e3)
        bwd_leg = {"value": round(dist.sum(tokens * args.steps) / b_tot, 1), "unit": "tokens/s",
                   "ms_per_step": round(float(np.mean(bms)), 4), "steps": args.steps,
                   "what": "msa_sparse_attn_backward: dq, dk, dv over the selected blocks from the forward's "
                           "selection, output and lse, synthetic output gradient",
                   "roofline": next((roofline_for(k_, bprof, bwork, peaks, peak_src, w.name, args.steps)
                                     for k_ in ("bwd_tile_tc", "bwd_tile") if k_ in bprof), None),
                   "kernels": {k: {"launches": v[0], "ms_per_step": round(v[1] / args.steps, 4)}
                               for k, v in bprof.items()},
                   "gpu_launches": sum(v[0] for v in bprof.values()), "clocks": bclocks,
                   "bwd_flops_per_step": bwork["bwd_flops"]}
        del dout, dq, dk, dv, ws_b
    if not (args.no_kl and args.no_backward):
        del lse

    del t, out, sel, ws_i, ws_a
    torch.cuda.empty_cache()

    # ---------------- other prefill configurations (one leg each) ----------------
    # the block-size sweep at 128K (Bs 64 with K 32, Bs 32 with K 64) and the
    # 1M-token prefill: the same two calls per step, timed the same way, with
    # the index and attention rooflines of each
    def prefill_leg(name, steps, warmup):
        wl = synth.WORKLOADS[name]
        qo_l, kl_l = synth.q_offsets(wl), synth.kv_lens(wl)
        tl = {n: synth.device_tensor(wl, n, dev) for n in ("q", "k", "v", "iq", "ik")}
        qo_t, kl_t = torch.from_numpy(qo_l).to(dev), torch.from_numpy(kl_l).to(dev)
        sel_l = torch.empty((wl.B, wl.Nq, wl.G, wl.K), dtype=torch.int32, device=dev)
        out_l = torch.empty_like(tl["q"])
        wsi = msa.workspace(msa.msa_workspace_size(msa.MSA_OP_INDEX_SELECT, wl.B, wl.Nq, wl.Nk, wl.G, 0, 0, wl.di,
                                                   wl.Bs, wl.K, msa.MSA_BF16), dev)
        wsa = msa.workspace(msa.msa_workspace_size(msa.MSA_OP_PREFILL, wl.B, wl.Nq, wl.Nk, wl.G, wl.Hq, wl.d, 0,
                                                   wl.Bs, wl.K, msa.MSA_BF16), dev)

        def step_l():
            msa.msa_index_select(tl["iq"], tl["ik"], qo_t, kl_t, wl.Bs, wl.K, sel=sel_l, ws=wsi)
            msa.msa_sparse_attn_prefill(tl["q"], tl["k"], tl["v"], sel_l, qo_t, kl_t, wl.Bs, wl.K, out=out_l,
                                        ws=wsa)

        lms, _, lclocks, _ = time_steps(step_l, steps, warmup, profile=False)
        _, lprof, _, _ = time_steps(step_l, steps, 0, profile=True)
        for ws_ in (wsi, wsa):
            st_ = msa.msa_read_status(ws_)
            if st_ != 0:
                raise RuntimeError(f"device status after {name}: {msa.msa_status_string(st_)}")
        lwork = prefill_work(wl, sel_l, qo_l, kl_l)
        l_tot = dist.max(sum(lms) / 1e3)
        res = {"value": round(dist.sum(wl.B * wl.Nq * steps) / l_tot, 1), "unit": "tokens/s",
               "ms_per_step": round(float(np.mean(lms)), 4), "steps": steps, "warmup": warmup,
               "config": {"workload": wl.name, "batch": wl.B, "seq_len": wl.Nq, "Bs": wl.Bs, "K": wl.K,
                          "hot_blocks": wl.hot},
               "roofline_all": [r for r in (roofline_for(k_, lprof, lwork, peaks, peak_src, wl.name, steps)
                                            for k_ in lprof) if r],
               "kernels": {k_: {"launches": v_[0], "ms_per_step": round(v_[1] / steps, 4)} for k_, v_ in lprof.items()},
               "gpu_launches": sum(v_[0] for v_ in lprof.values()), "clocks": lclocks,
               "work": {"index_flops": lwork["index_flops"], "attn_flops": lwork["attn_flops"],
                        "attended_keys": lwork["attended_keys"]}}
        del tl, sel_l, out_l, wsi, wsa
        torch.cuda.empty_cache()
        return res

    sweep = None
    if not args.no_sweep:
        sweep = {}
        for name, nsteps in (("prefill_128k_bs64", min(args.steps, 10)), ("prefill_128k_bs32", min(args.steps, 10)),
                             ("prefill_1m", 3)):
            sweep[name] = prefill_leg(name, nsteps, args.warmup)

    # ------------------------------ decode -----------------------------
    decode = None
    if not args.no_decode:
        wd = synth.WORKLOADS[args.decode_workload]
        kld_np = synth.kv_lens(wd)
        td = {n: synth.device_tensor(wd, n, dev) for n in ("q", "k", "v", "iq", "ik")}
        qd = td["q"][:, 0]
        kld = torch.from_numpy(kld_np).to(dev)
        qod = kld - 1
        seld = torch.empty((wd.B, 1, wd.G, wd.K), dtype=torch.int32, device=dev)
        outd = torch.empty_like(qd)
        wsd_i = msa.workspace(msa.msa_workspace_size(msa.MSA_OP_INDEX_SELECT, wd.B, 1, wd.Nk, wd.G, 0, 0, wd.di,
                                                     wd.Bs, wd.K, msa.MSA_BF16), dev)
        wsd_a = msa.workspace(msa.msa_workspace_size(msa.MSA_OP_DECODE, wd.B, 1, wd.Nk, wd.G, wd.Hq, wd.d, 0, wd.Bs,
                                                     wd.K, msa.MSA_BF16), dev)

        def decode_step():
            msa.msa_index_select(td["iq"], td["ik"], qod, kld, wd.Bs, wd.K, sel=seld, ws=wsd_i)
            msa.msa_sparse_attn_decode(qd, td["k"], td["v"], seld, kld, wd.Bs, wd.K, out=outd, ws=wsd_a)

        dsteps = max(args.steps, 50)
        dms, _, dclocks, _ = time_steps(decode_step, dsteps, max(args.warmup, 5), profile=False)
        dkms, dprof, _, _ = time_steps(decode_step, dsteps, 0, profile=True)
        for ws in (wsd_i, wsd_a):
            st = msa.msa_read_status(ws)
            if st != 0:
                raise RuntimeError(f"device status after decode: {msa.msa_status_string(st)}")
        dwork = decode_work(wd, seld, kld_np)
        d_tot = dist.max(sum(dms) / 1e3)
        dval = dist.sum(wd.B * dsteps) / d_tot
        dstep_s = float(np.mean(dms)) / 1e3
        step_gbs = dwork["total_bytes"] / dstep_s / 1e9
        ddom = max(dprof, key=lambda k: dprof[k][1]) if dprof else None
        decode = {
            "value": round(dval, 1), "unit": "tokens/s", "ms_per_step": round(float(np.mean(dms)), 4),
            "steps": dsteps, "config": {"workload": wd.name, "batch": wd.B, "kv_len_range": list(wd.kv_len_range),
                                        "Bs": wd.Bs, "K": wd.K, "l2": L2_NOTE},
            "step_roofline": {"bound": "hbm", "achieved": round(step_gbs, 1), "peak": peaks["hbm_gbs"],
                              "unit": "GB/s", "frac": round(step_gbs / peaks["hbm_gbs"], 4),
                              "algorithmic_bytes_per_step": dwork["total_bytes"]},
            "roofline": roofline_for(ddom, dprof, dwork, peaks, peak_src, wd.name, dsteps, "decode") if ddom else None,
            "kernels": {k: {"launches": v[0], "ms_per_step": round(v[1] / dsteps, 4)} for k, v in dprof.items()},
            "gpu_launches": sum(v[0] for v in dprof.values()), "clocks": dclocks,
            "ms_per_step_with_kernel_events": round(float(np.mean(dkms)), 4),
        }
        # streaming decode (msa_decode_step): each step appends one token per
        # sequence to the caches (rows gathered before the timed region), then
        # selects and attends for it; lengths start below the measured ones
        # so that every append fits the cache
        sst = dsteps + 1 + max(args.warmup, 5)
        ks = torch.from_numpy(np.maximum(kld_np - sst, 1).astype(np.int32)).to(dev)
        ar = torch.arange(wd.B, device=dev)
        new_rows = [(td["k"][ar, ks.long() + j].contiguous(), td["v"][ar, ks.long() + j].contiguous(),
                     td["ik"][ar, ks.long() + j].contiguous()) for j in range(sst)]
        iqd = td["iq"][:, 0]
        seld2 = torch.empty((wd.B, wd.G, wd.K), dtype=torch.int32, device=dev)
        wsd_s = msa.workspace(msa.msa_workspace_size(msa.MSA_OP_DECODE_STEP, wd.B, 0, wd.Nk, wd.G, wd.Hq, wd.d, wd.di,
                                                     wd.Bs, wd.K, msa.MSA_BF16), dev)
        cursor = [0]

        def stream_step():
            kn, vn, ikn = new_rows[cursor[0] % sst]
            cursor[0] += 1
            msa.msa_decode_step(qd, kn, vn, iqd, ikn, td["k"], td["v"], td["ik"], ks, wd.Bs, wd.K, sel=seld2,
                                out=outd, ws=wsd_s)

        sms, _, _, _ = time_steps(stream_step, dsteps, max(args.warmup, 5), profile=False)
        st = msa.msa_read_status(wsd_s)
        if st != 0:
            raise RuntimeError(f"device status after streaming decode: {msa.msa_status_string(st)}")
        s_tot = dist.max(sum(sms) / 1e3)
        decode["stream"] = {"value": round(dist.sum(wd.B * dsteps) / s_tot, 1), "unit": "tokens/s",
                            "ms_per_step": round(float(np.mean(sms)), 4), "steps": dsteps,
                            "what": "msa_decode_step: append k/v/index-key rows at kv_len, advance kv_len, "
                                    "select and attend over the grown caches"}
        del td, seld, outd, wsd_i, wsd_a, wsd_s, new_rows
        torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, device-generated)",
        "config": {"workload": w.name, "batch": w.B, "seq_len": w.Nq, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                   "di": w.di, "Bs": w.Bs, "K": w.K, "hot_blocks": w.hot, "parallelism": f"replicas x{dist.world}",
                   "l2": L2_NOTE},
        "roofline": roof, "roofline_all": all_roofs, "kernels": kernels, "gpu_launches": launches,
        "kernel_times": "per-kernel CUDA events on the launching stream, in a second pass of the same steps "
                        "(the timed pass carries no events between kernels)",
        "clocks": clocks, "e2e": e2e, "decode": decode, "kl_aux": kl_leg, "backward": bwd_leg, "prefill_sweep": sweep,
        "work": {"index_flops": work["index_flops"], "attn_flops": work["attn_flops"],
                 "attended_keys": work["attended_keys"]},
        "wall_s_timed_region": round(wall, 3),
    }
    return line


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------
_KV_HOST = {}  # (Nk, Hkv, d) -> zero-filled host K / V of one sequence, reused across calls


def oracle_prefill_rows(w, rows, ik_host):
    """Oracle index select + attention for the listed rows of sequence 0.
    Returns seconds spent inside the oracle (input generation excluded)."""
    import oracle

    rows = np.asarray(rows, np.int32)
    rb = np.zeros(len(rows), np.int32)
    iq = synth.host_rows(w, "iq", 0, rows)
    q = synth.host_rows(w, "q", 0, rows)
    qo, kl = synth.q_offsets(w), synth.kv_lens(w)
    t0 = time.perf_counter()
    sel = oracle.index_select(iq, ik_host, rb, rows, qo, kl, w.Bs, w.K)
    t1 = time.perf_counter()
    key = (w.Nk, w.Hkv, w.d)
    if key not in _KV_HOST:
        _KV_HOST[key] = (np.zeros((1, w.Nk, w.Hkv, w.d), np.float32), np.zeros((1, w.Nk, w.Hkv, w.d), np.float32))
    k, v = _KV_HOST[key]
    row = w.Hkv * w.d
    spans = [(tb * w.Bs, min((tb + 1) * w.Bs, w.Nk)) for tb in sorted(set(int(x) for x in sel.reshape(-1) if x >= 0))]
    for j0, j1 in spans:  # only the selected blocks are filled (the oracle reads no others)
        k[0, j0:j1] = synth.host_range(w, "k", j0 * row, (j1 - j0) * row).reshape(j1 - j0, w.Hkv, w.d)
        v[0, j0:j1] = synth.host_range(w, "v", j0 * row, (j1 - j0) * row).reshape(j1 - j0, w.Hkv, w.d)
    t2 = time.perf_counter()
    oracle.sparse_attn(q, k, v, sel, rb, rows, qo, kl, w.Bs, w.K)
    t3 = time.perf_counter()
    for j0, j1 in spans:  # back to zeros for the next call
        k[0, j0:j1] = 0.0
        v[0, j0:j1] = 0.0
    return (t1 - t0) + (t3 - t2)


def cpu_model() -> str:
    """The host CPU's model name (x86 /proc/cpuinfo, else lscpu, else the machine type)."""
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform

    return platform.machine() or "unknown"


def sample_rows(w, n, offset=0):
    """n query rows evenly spaced over the sequence (their mean cost equals the
    mean cost per token, which grows with position)."""
    step = w.Nq / n
    return np.array([int((k + 0.5) * step) + offset for k in range(n)], np.int32) % w.Nq


def oracle_full_prefill(w):
    """The oracle over every row of a prefill workload (dense host inputs).
    Returns seconds inside the oracle (input generation excluded)."""
    import oracle

    h = {n: synth.host_tensor(w, n) for n in ("q", "k", "v", "iq", "ik")}
    t0 = time.perf_counter()
    oracle.msa_forward(h["q"], h["k"], h["v"], h["iq"], h["ik"], w.Bs, w.K, q_offset=synth.q_offsets(w),
                       kv_len=synth.kv_lens(w))
    return time.perf_counter() - t0


def oracle_full_decode(w):
    """The oracle over every sequence of a decode workload: one batched index
    selection over the whole index-key cache, then attention per sequence on a
    host K/V holding that sequence's selected blocks. Returns oracle seconds."""
    import oracle

    kl = synth.kv_lens(w)
    qo = (kl - 1).astype(np.int32)
    ik = synth.host_tensor(w, "ik")
    iq = synth.host_tensor(w, "iq").reshape(w.B, w.G, w.di)
    q = synth.host_tensor(w, "q").reshape(w.B, w.Hq, w.d)
    rb, ri = np.arange(w.B, dtype=np.int32), np.zeros(w.B, np.int32)
    t0 = time.perf_counter()
    sel = oracle.index_select(iq, ik, rb, ri, qo, kl, w.Bs, w.K)
    secs = time.perf_counter() - t0
    del ik
    row = w.Hkv * w.d
    k = np.zeros((1, w.Nk, w.Hkv, w.d), np.float32)
    v = np.zeros((1, w.Nk, w.Hkv, w.d), np.float32)
    for b in range(w.B):
        spans = [(t * w.Bs, min((t + 1) * w.Bs, w.Nk)) for t in sorted(set(int(x) for x in sel[b].reshape(-1) if x >= 0))]
        for j0, j1 in spans:
            k[0, j0:j1] = synth.host_range(w, "k", (b * w.Nk + j0) * row, (j1 - j0) * row).reshape(j1 - j0, w.Hkv, w.d)
            v[0, j0:j1] = synth.host_range(w, "v", (b * w.Nk + j0) * row, (j1 - j0) * row).reshape(j1 - j0, w.Hkv, w.d)
        t0 = time.perf_counter()
        oracle.sparse_attn(q[b:b + 1], k, v, sel[b:b + 1], np.zeros(1, np.int32), np.zeros(1, np.int32), qo[b:b + 1],
                           kl[b:b + 1], w.Bs, w.K)
        secs += time.perf_counter() - t0
        for j0, j1 in spans:
            k[0, j0:j1] = 0.0
            v[0, j0:j1] = 0.0
    return secs


def cpu_baseline(w, rows_n, full_legs=True):
    """The oracle timed on this host's cores: a row sample of the bench
    workload (the headline CPU figure), and full runs of the tiny fp32, 8K
    prefill and decode workloads."""
    import oracle

    ik = synth.host_tensor(w, "ik")
    rows = sample_rows(w, rows_n)
    secs = oracle_prefill_rows(w, rows, ik)
    del ik
    res = {"value": round(len(rows) / secs, 2), "unit": "tokens/s", "cores": oracle.threads(), "kind": "oracle",
           "cpu_model": cpu_model(),
           "sample": f"{len(rows)} query rows evenly spaced over the {w.Nq}-token sequence, all {w.G} groups / "
                     f"{w.Hq} heads; index select + attention in fp64; tokens/s = rows / oracle seconds",
           "seconds": round(secs, 2)}
    if full_legs:
        full = {}
        for name in ("tiny_fp32", "prefill_8k"):
            wl = synth.WORKLOADS[name]
            sec = oracle_full_prefill(wl)
            full[name] = {"value": round(wl.B * wl.Nq / sec, 2), "unit": "tokens/s", "seconds": round(sec, 3),
                          "rows": wl.B * wl.Nq, "what": "every query row, index select + attention"}
        wd = synth.WORKLOADS["decode_b64"]
        sec = oracle_full_decode(wd)
        full[wd.name] = {"value": round(wd.B / sec, 2), "unit": "tokens/s", "seconds": round(sec, 3), "rows": wd.B,
                         "what": "every sequence's new token, index select over its cache + attention"}
        res["full"] = full
        # sampled rows of the other prefill workloads (the block-size sweep
        # and 1M tokens): evenly spaced rows, so rows / seconds estimates the
        # oracle's tokens/s over the whole sequence
        sampled = {}
        for name, n in (("prefill_128k_bs64", 512), ("prefill_128k_bs32", 512), ("prefill_1m", 16)):
            wl = synth.WORKLOADS[name]
            ikl = synth.host_tensor(wl, "ik")
            rl = sample_rows(wl, n)
            sec = oracle_prefill_rows(wl, rl, ikl)
            del ikl
            sampled[name] = {"value": round(len(rl) / sec, 2), "unit": "tokens/s", "seconds": round(sec, 3),
                             "rows": len(rl), "what": f"{len(rl)} query rows evenly spaced over {wl.Nq} tokens, "
                                                      "index select + attention"}
        _KV_HOST.clear()
        res["sampled"] = sampled
    return res


def run_reference(args, dist):
    """The oracle as the reference arm: each step is a bounded sample of rows."""
    import oracle

    w = synth.WORKLOADS[args.workload]
    ik = synth.host_tensor(w, "ik")
    # enough rows per step that the oracle's row-parallel threads all work
    rows_per_step = 16 * oracle.threads()
    for s in range(args.warmup):
        oracle_prefill_rows(w, sample_rows(w, rows_per_step, offset=s), ik)
    secs = 0.0
    for s in range(args.steps):
        secs += oracle_prefill_rows(w, sample_rows(w, rows_per_step, offset=1000 + s), ik)
    value = rows_per_step * args.steps / secs
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": w.name, "batch": w.B, "seq_len": w.Nq, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                   "di": w.di, "Bs": w.Bs, "K": w.K, "hot_blocks": w.hot, "parallelism": f"replicas x{dist.world}",
                   "l2": "n/a (host)"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": oracle.threads(), "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"{rows_per_step} evenly spaced query rows per step (all groups/heads), "
                                   f"index select + attention in fp64"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    args = parse_args()
    if args.warmup < 3:
        args.warmup = 3
    dist = Dist()
    if args.impl == "reference":
        if dist.rank == 0:
            print(json.dumps(run_reference(args, dist)), flush=True)
        return
    line = run_msa(args, dist)
    if dist.rank == 0:
        if not args.no_cpu_baseline:
            rows = args.cpu_rows or 4096
            line["cpu_baseline"] = cpu_baseline(synth.WORKLOADS[args.workload], rows)
        print(json.dumps(line), flush=True)
    if dist.pg:
        dist.pg.destroy_process_group()


if __name__ == "__main__":
    main()
