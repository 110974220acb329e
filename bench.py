"""Benchmark of the MSA hot path on B300.

One step = one MSA prefill launch over the largest prefill workload, the
Llama-3-70B-shaped attention layer (64/8 heads, d = 128, 131072-token context in
16-token blocks with >= 200 non-contiguous cached segments, 8192-token query chunk),
followed by one MSA decode launch over the batch-64 decode workload (32/8 heads,
contexts 4k-64k split into 2-32 scattered segments), both on inputs resident in HBM.
The plan (host planner) is built and uploaded before timing.

value        = useful prefill TFLOP/s (4 d Hq per visible query/key pair) over the timed
               prefill launches; the decode's algorithmic HBM GB/s is in "decode".
roofline     = prefill kernel vs the measured dense bf16 peak; decode.roofline = decode
               kernel vs the measured HBM copy bandwidth.
prefill_configs = every prefill workload of the metric (the Llama-3-8B-shaped layer with
               an 8192-token context and 2048-token chunk, the 16-session multi-turn
               batch, and the headline one), each timed alone the same way: ms, useful
               TFLOP/s and the fraction of the measured peak.
e2e          = the same metrics with every step's inputs copied from pinned host memory and
               its results read back inside the timed region (the KV pool and the plan
               stay resident: they are the cache).  Copies and kernels run on three
               streams with two buffer sets, as a serving loop would overlap them; the
               serial figure (one stream) is reported beside it.
cpu_baseline = the CPU oracle timed on this host on a bounded sample of the same workload.

`--impl reference` times the CPU oracle as the reference arm (there is no other
implementation of this method to run).
Multi-GPU: replicas only -- each rank runs its own copy of the step with no collective
on the data path; a barrier and a max-reduction of the timings bracket the run.
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

METRIC = "MSA prefill useful TFLOPS (% bf16 TC peak); decode HBM GB/s (% peak), 1 B300"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def code_sha256(text: str) -> str:
    """sha256 of a C++/CUDA source with its comments, trailing blanks and empty lines
    removed: a change to the comments alone leaves it unchanged."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()


TRAFFIC_SOURCES = {
    # the prefill's traffic depends on the kernel and on the planner's schedule
    "prefill": ("msa_prefill.cu", "msa_plan.cpp"),
    "decode": ("msa_decode.cu",),
}


def sources_sha256(name: str) -> str:
    """code_sha256 of the sources a kernel's DRAM traffic depends on, concatenated."""
    csrc = os.path.join(ROOT, "segmented_kv_attention_msa_b300", "csrc")
    return code_sha256("\n".join(open(os.path.join(csrc, f)).read() for f in TRAFFIC_SOURCES[name]))


def kernel_traffic(name: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary (profiles/<name>_traffic.txt or
    profiles/<name>_traffic_<anything>.txt) that was taken on the current code (code_sha256
    of the kernel's sources) and applies to this workload; otherwise None."""
    import glob
    try:
        current = sources_sha256(name)
    except Exception:
        return None
    files = [os.path.join(ROOT, "profiles", f"{name}_traffic.txt")]
    files += sorted(glob.glob(os.path.join(ROOT, "profiles", f"{name}_traffic_*.txt")))
    for summ in files:
        try:
            kv = {}
            for line in open(summ):
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
            if kv.get("code_sha256") == current and kv.get("applies_to") == workload:
                return float(kv["dram_bytes_per_launch"])
        except Exception:
            continue
    return None


def staging(like, device, sets):
    """`sets` byte buffers, each holding one tensor shaped like every tensor of `like`,
    256-byte aligned, back to back (pinned when on the host); returns (buffers, views)
    with views[set][i] a tensor of like[i]'s shape and dtype inside buffers[set]."""
    import torch
    offs, total = [], 0
    for t in like:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    bufs, views = [], []
    for _ in range(sets):
        if str(device) == "cpu":
            buf = torch.empty(total, dtype=torch.uint8).pin_memory()
        else:
            buf = torch.empty(total, dtype=torch.uint8, device=device)
        bufs.append(buf)
        views.append([buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                      for o, t in zip(offs, like)])
    return bufs, views


def staged_equal(buf, like) -> bool:
    """Does the staging buffer `buf` (laid out by staging()) hold exactly `like`'s bytes?"""
    import torch
    off = 0
    for t in like:
        n = t.numel() * t.element_size()
        if not torch.equal(buf[off:off + n].cpu(), t.contiguous().view(torch.uint8).reshape(-1).cpu()):
            return False
        off += (n + 255) // 256 * 256
    return True


def pipelined_e2e(steps, h2d, run, d2h, flush, dev):
    """Milliseconds per step of a stream of `steps` steps, each uploading its inputs
    (h2d), flushing L2 (unless flush is None: inputs larger than L2) and running its
    kernel (run) and reading its results back (d2h).
    Uploads, kernels and read-backs go to three streams; two buffer sets (b = k % 2) let
    step k+1's upload and step k-1's read-back overlap step k's kernel.  A buffer set is
    reused only after the step that last used it is done with it."""
    import torch
    s_in, s_c, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_in, ev_c, ev_out = [], [], []
    torch.cuda.synchronize()
    start.record()
    for s in (s_in, s_c, s_out):
        s.wait_event(start)
    for k in range(steps):
        b = k & 1
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(ev_c[k - 2])    # the kernel of step k-2 has read set b
            h2d(b)
            ev_in.append(torch.cuda.Event())
            ev_in[k].record(s_in)
        with torch.cuda.stream(s_c):
            s_c.wait_event(ev_in[k])
            if k >= 2:
                s_c.wait_event(ev_out[k - 2])   # the results of step k-2 were read back
            if flush is not None:
                flush.fill_(k & 0xFF)
            run(b)
            ev_c.append(torch.cuda.Event())
            ev_c[k].record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_c[k])
            d2h(b)
            ev_out.append(torch.cuda.Event())
            ev_out[k].record(s_out)
    end.record(s_out)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("MSA_BENCH_BACKEND", "nccl")
        dist.init_process_group(backend)
    return world, rank, local


def reduce_max(values, world, device=None):
    """Element-wise max over ranks (used for the per-step timings)."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(per_rank_units, max_seconds):
    """Whole-job throughput: units processed by all ranks / slowest rank's time."""
    return sum(per_rank_units) / max_seconds if max_seconds > 0 else 0.0


# ----------------------------------------------------------------------------- our arm

def run_ours(args, world, rank, local):
    import torch

    import segmented_kv_attention_msa_b300 as msa
    from segmented_kv_attention_msa_b300 import build as B
    from segmented_kv_attention_msa_b300 import workload as W

    if not os.path.exists(msa.LIB_PATH):
        B.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_kind = load_peaks()

    # ---- prefill workload (the metric's configuration) and decode workload
    pl = W.make_layout(args.workload, tiler=msa.chunk_sizes)
    pw = W.make_values(pl, device=dev)
    pplan = msa.Plan.from_layout(pl).upload(dev)
    pst = pplan.stats()
    pout = torch.empty_like(pw.q)
    plse = torch.empty(pw.q.shape[0], pw.q.shape[1], dtype=torch.float32, device=dev)

    do_pf = args.only in (None, "prefill")
    do_dc = args.only in (None, "decode")
    if do_dc:
        dl = W.make_layout(args.decode_workload, decode_batch=args.decode_batch)
        dw = W.make_values(dl, device=dev)
        dplan = msa.Plan.from_layout(dl).upload(dev)
        dst = dplan.stats()
        dout = torch.empty_like(dw.q)
        dlse = torch.empty(dw.q.shape[0], dw.q.shape[1], dtype=torch.float32, device=dev)
    else:
        dl, dw, dplan, dout, dlse = pl, None, pplan, None, None
        dst = {"algorithmic_bytes": 0, "kv_tokens": 0, "num_splits": 0}

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # 256 MB > 126 MB L2

    def step(ev=None):
        if ev is not None:
            ev[0].record()
        if do_pf:
            msa.prefill(pplan, pw.q, pw.k_chunk, pw.v_chunk, pw.k_pool, pw.v_pool, out=pout, lse=plse)
        if ev is not None:
            ev[1].record()
        if do_dc:
            msa.decode(dplan, dw.q, dw.k_pool, dw.v_pool, out=dout, lse=dlse)
        if ev is not None:
            ev[2].record()

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if msa.get_status(pplan) != 0 or (do_dc and msa.get_status(dplan) != 0):
        raise RuntimeError("device error during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        step(evs[k])
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t0
    clocks = sampler.stop()
    if msa.get_status(pplan) != 0 or (do_dc and msa.get_status(dplan) != 0):
        raise RuntimeError("device error during the timed steps")
    pf_ms = [evs[k][0].elapsed_time(evs[k][1]) for k in range(args.steps)]
    dc_ms = [evs[k][1].elapsed_time(evs[k][2]) for k in range(args.steps)]
    pf_mean, dc_mean = statistics.mean(pf_ms), statistics.mean(dc_ms)
    pf_mean, dc_mean = reduce_max([pf_mean, dc_mean], world, dev)

    if not (do_pf and do_dc):
        return _single_kernel_result(args, world, pl, dl, pst, dst, pf_mean, dc_mean, peaks, peak_kind, clocks)
    flops = pst["useful_flops"]
    dbytes = dst["algorithmic_bytes"]
    value = aggregate([flops] * world, pf_mean * 1e-3) / 1e12
    dec_gbs = aggregate([dbytes] * world, dc_mean * 1e-3) / 1e9
    tc_peak = peaks["bf16_tflops"]
    hbm_peak = peaks["hbm_gbs"]
    pf_ach = flops / (pf_mean * 1e-3) / 1e12
    dc_ach = dbytes / (dc_mean * 1e-3) / 1e9

    # ---- end to end: inputs from pinned host memory, results read back, every step
    hq = pw.q.cpu().pin_memory()
    hkc = pw.k_chunk.cpu().pin_memory()
    hvc = pw.v_chunk.cpu().pin_memory()
    hdq = dw.q.cpu().pin_memory()
    h2d_pf = sum(t.numel() * t.element_size() for t in (hq, hkc, hvc))
    d2h_pf = pout.numel() * pout.element_size() + plse.numel() * plse.element_size()
    h2d_dc = hdq.numel() * hdq.element_size()
    d2h_dc = dout.numel() * dout.element_size() + dlse.numel() * dlse.element_size()
    e2e_steps = max(1, min(args.steps, 20))

    # serial: one stream, every copy in line with the kernel (context for the pipelined figure)
    sq = [torch.empty_like(pw.q), torch.empty_like(pw.k_chunk), torch.empty_like(pw.v_chunk)]
    sho = [torch.empty(pout.shape, dtype=pout.dtype).pin_memory(), torch.empty(plse.shape, dtype=plse.dtype).pin_memory()]
    sdq = torch.empty_like(dw.q)
    shd = [torch.empty(dout.shape, dtype=dout.dtype).pin_memory(), torch.empty(dlse.shape, dtype=dlse.dtype).pin_memory()]
    pe = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(e2e_steps)]
    torch.cuda.synchronize()
    for k in range(e2e_steps):
        flush.fill_(k & 0xFF)
        pe[k][0].record()
        for d, h in zip(sq, (hq, hkc, hvc)):
            d.copy_(h, non_blocking=True)
        msa.prefill(pplan, sq[0], sq[1], sq[2], pw.k_pool, pw.v_pool, out=pout, lse=plse)
        sho[0].copy_(pout, non_blocking=True)
        sho[1].copy_(plse, non_blocking=True)
        pe[k][1].record()
        sdq.copy_(hdq, non_blocking=True)
        msa.decode(dplan, sdq, dw.k_pool, dw.v_pool, out=dout, lse=dlse)
        shd[0].copy_(dout, non_blocking=True)
        shd[1].copy_(dlse, non_blocking=True)
        pe[k][2].record()
    torch.cuda.synchronize()
    ser_pf = statistics.mean(pe[k][0].elapsed_time(pe[k][1]) for k in range(e2e_steps))
    ser_dc = statistics.mean(pe[k][1].elapsed_time(pe[k][2]) for k in range(e2e_steps))

    # pipelined: the same per-step copies and launches, on three streams with two buffer
    # sets, so that step k+1's upload and step k-1's read-back overlap step k's kernel.
    # A step's inputs sit in one staging buffer and its results in another, so each
    # direction is one large copy (PCIe moves large copies fastest); the kernels read and
    # write views into those buffers.
    pin_buf, pin_v = staging([pw.q, pw.k_chunk, pw.v_chunk], dev, sets=2)
    host_in, host_in_v = staging([pw.q, pw.k_chunk, pw.v_chunk], "cpu", sets=1)
    for hv, src in zip(host_in_v[0], (pw.q, pw.k_chunk, pw.v_chunk)):
        hv.copy_(src.cpu())
    pres_buf, pres_v = staging([pout, plse], dev, sets=2)
    phost_buf, _ = staging([pout, plse], "cpu", sets=2)

    def pf_h2d(b):
        pin_buf[b].copy_(host_in[0], non_blocking=True)

    def pf_run(b):
        q_, kc_, vc_ = pin_v[b]
        msa.prefill(pplan, q_, kc_, vc_, pw.k_pool, pw.v_pool, out=pres_v[b][0], lse=pres_v[b][1])

    def pf_d2h(b):
        phost_buf[b].copy_(pres_buf[b], non_blocking=True)

    din_buf, din_v = staging([dw.q], dev, sets=2)
    dhost_in, dhost_in_v = staging([dw.q], "cpu", sets=1)
    dhost_in_v[0][0].copy_(dw.q.cpu())
    dres_buf, dres_v = staging([dout, dlse], dev, sets=2)
    dhost_buf, _ = staging([dout, dlse], "cpu", sets=2)

    def dc_h2d(b):
        din_buf[b].copy_(dhost_in[0], non_blocking=True)

    def dc_run(b):
        msa.decode(dplan, din_v[b][0], dw.k_pool, dw.v_pool, out=dres_v[b][0], lse=dres_v[b][1])

    def dc_d2h(b):
        dhost_buf[b].copy_(dres_buf[b], non_blocking=True)

    e2e_pf = pipelined_e2e(e2e_steps, pf_h2d, pf_run, pf_d2h, flush, dev)
    # the decode reads its whole pool every step (far more than L2 holds): no flush needed
    dc_flush = flush if dbytes < 4 * flush.numel() else None
    e2e_dc = pipelined_e2e(e2e_steps, dc_h2d, dc_run, dc_d2h, dc_flush, dev)
    if msa.get_status(pplan) != 0 or msa.get_status(dplan) != 0:
        raise RuntimeError("device error during the end-to-end steps")
    # the results read back by the last pipelined steps are those of the device-timed run
    # (same inputs, deterministic kernels), bit for bit
    last = (e2e_steps - 1) & 1
    for host_buf, like in ((phost_buf[last], (pout, plse)), (dhost_buf[last], (dout, dlse))):
        if not staged_equal(host_buf, like):
            raise RuntimeError("end-to-end results differ from the device-timed run")
    e2e_pf, e2e_dc, ser_pf, ser_dc = reduce_max([e2e_pf, e2e_dc, ser_pf, ser_dc], world, dev)

    append = append_bench(msa, W, pl, pw, dev, flush)
    merge = merge_bench(msa, pl, dev, flush, hbm_peak, peak_kind)
    gather = gather_bench(msa, pplan, pw, dev, flush, hbm_peak, peak_kind)
    configs = {}
    for idx in PREFILL_WORKLOADS:
        if idx == args.workload:
            configs[pl.name] = prefill_entry(pl, pst, pf_mean, tc_peak, peak_kind)
        else:
            configs.update(time_prefill_workload(msa, W, idx, dev, flush, tc_peak, peak_kind, world))
    ablation = None
    if not args.no_ablation:
        al = W.make_layout(2, tiler=msa.chunk_sizes)
        aw = W.make_values(al, device=dev)
        ablation = ablation_bench(msa, W, al, aw, dev, flush)
        del aw

    result = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(pf_mean + dc_mean, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded generator; the paper's datasets are not available)",
        "config": {
            "workload": pl.name, "decode_workload": dl.name,
            "prefill": {"num_heads_q": pl.num_heads_q, "num_heads_kv": pl.num_heads_kv, "head_dim": pl.head_dim,
                        "query_tokens": pl.total_q, "kv_tokens": pst["kv_tokens"],
                        "segments": int(len(pl.segments)), "useful_flops": flops,
                        "kv_tiles": pst["num_kv_tiles"], "tile_pairs": pst["num_tile_pairs"],
                        "partial_pairs": pst["num_partial_pairs"]},
            "decode": {"batch": dl.num_seqs, "num_heads_q": dl.num_heads_q, "num_heads_kv": dl.num_heads_kv,
                       "head_dim": dl.head_dim, "kv_tokens": dst["kv_tokens"], "segments": int(len(dl.segments)),
                       "splits": dst["num_splits"], "algorithmic_bytes": dbytes},
            "l2": "flushed between steps (256 MB write)",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {"bound": "tensor", "achieved": round(pf_ach, 2), "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": round(pf_ach / tc_peak, 4), "traffic": kernel_traffic("prefill", pl.name),
                     "kernel": "msa_prefill_kernel<128>", "peak_source": f"{peak_kind} bf16_tflops (burst)",
                     # the timed steps keep the GPU at its power limit for about a second (see clocks):
                     # the same figure against the cuBLAS throughput measured under that limit
                     "peak_sustained": peaks.get("bf16_tflops_sustained"),
                     "frac_of_sustained": (round(pf_ach / peaks["bf16_tflops_sustained"], 4)
                                           if peaks.get("bf16_tflops_sustained") else None)},
        "decode": {"value": round(dec_gbs, 1), "unit": "GB/s", "ms": round(dc_mean, 4),
                   "roofline": {"bound": "hbm", "achieved": round(dc_ach, 1), "peak": hbm_peak, "unit": "GB/s",
                                "frac": round(dc_ach / hbm_peak, 4),
                                "traffic": kernel_traffic("decode", dl.name),
                                "kernel": "msa_decode_kernel<128,4>", "peak_source": f"{peak_kind} hbm_gbs"},
                   "e2e": {"value": round(dbytes / (e2e_dc * 1e-3) / 1e9, 1), "unit": "GB/s",
                           "h2d_bytes_per_step": h2d_dc, "d2h_bytes_per_step": d2h_dc,
                           "l2": ("flushed before each step" if dc_flush is not None
                                  else "not flushed: each step reads more than L2 holds")}},
        "prefill_ms": round(pf_mean, 4),
        "e2e": {"value": round(flops * world / (e2e_pf * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d_pf, "d2h_bytes_per_step": d2h_pf,
                "prefill_ms": round(e2e_pf, 4), "decode_ms": round(e2e_dc, 4),
                "pipeline": "per step: H2D of its inputs, L2 flush + kernel, D2H of its results; "
                            "3 streams, 2 buffer sets; ms = whole run / steps",
                "serial": {"value": round(flops * world / (ser_pf * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                           "prefill_ms": round(ser_pf, 4), "decode_ms": round(ser_dc, 4)}},
        "prefill_configs": configs,
        "append": append,
        "merge": merge,
        "gather": gather,
        "ablation_per_segment": ablation,
        "clocks": clocks,
        "gpu_launches": 2 * args.steps,
        "wall_s": round(wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(pl, pw, args.cpu_rows)
    return result


PREFILL_WORKLOADS = (2, 3, 5)   # the prefill configurations of the metric (1 is the tiny parity case)


def prefill_entry(pl, pst, ms, tc_peak, peak_kind):
    ach = pst["useful_flops"] / (ms * 1e-3) / 1e12
    return {"ms": round(ms, 4), "useful_tflops": round(ach, 2), "frac": round(ach / tc_peak, 4),
            "peak_source": f"{peak_kind} bf16_tflops (burst)", "useful_flops": pst["useful_flops"],
            "query_tokens": pl.total_q, "kv_tokens": pst["kv_tokens"], "segments": int(len(pl.segments)),
            "traffic": kernel_traffic("prefill", pl.name)}


def time_prefill_workload(msa, W, idx, dev, flush, tc_peak, peak_kind, world, reps: int = 20):
    """One prefill workload timed alone: warm-up, then `reps` launches each after an L2
    flush, CUDA events on the launching stream, mean (max over ranks)."""
    import torch
    lay = W.make_layout(idx, tiler=msa.chunk_sizes)
    wl = W.make_values(lay, device=dev)
    plan = msa.Plan.from_layout(lay).upload(dev)
    out = torch.empty_like(wl.q)
    lse = torch.empty(wl.q.shape[:2], dtype=torch.float32, device=dev)
    for _ in range(3):
        msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool, out=out, lse=lse)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for e0, e1 in ev:
        flush.fill_(9)
        e0.record()
        msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool, out=out, lse=lse)
        e1.record()
    torch.cuda.synchronize()
    if msa.get_status(plan) != 0:
        raise RuntimeError(f"device error in prefill workload {idx}")
    ms = reduce_max([statistics.mean(a.elapsed_time(b) for a, b in ev)], world, dev)[0]
    return {lay.name: prefill_entry(lay, plan.stats(), ms, tc_peak, peak_kind)}


def append_bench(msa, W, pl, pw, dev, flush, reps: int = 20):
    """Write-back of the prefill chunk's K/V into fresh pool blocks (placement planned on the
    host, the copy timed on the device; not part of the step).  Bytes = chunk K and V read
    plus the same written."""
    import numpy as np
    import torch
    n = pl.total_q
    nblk = n // 16 + 2 * pl.num_seqs + 1
    kp = torch.zeros(nblk, pl.num_heads_kv, 16, pl.head_dim, dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    bp = np.zeros(nblk, np.int32)
    bf = np.zeros(nblk, np.int32)
    dst = []
    free = list(range(nblk))
    for s in range(pl.num_seqs):
        qp = pl.q_pos[pl.cu_q[s]:pl.cu_q[s + 1]]
        # a chunk that starts part-way into a block continues a block of its own
        seq_blocks = []
        if len(qp) and qp[0] % 16:
            b = free.pop(0)
            bp[b], bf[b] = qp[0] // 16 * 16, qp[0] % 16
            seq_blocks = [b]
        d, new = msa.append_plan(qp, free, bp, bf, seq_blocks=seq_blocks)
        free = [b for b in free if b not in set(new.tolist())]
        dst.append(d)
    slots = torch.from_numpy(np.concatenate(dst).astype(np.int32)).to(dev)
    for _ in range(3):
        msa.kv_append(slots, pw.k_chunk, pw.v_chunk, kp, vp)
    ts = []
    for _ in range(reps):
        flush.fill_(3)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        msa.kv_append(slots, pw.k_chunk, pw.v_chunk, kp, vp)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    ms = statistics.median(ts)
    nbytes = 2 * 2 * n * pl.num_heads_kv * pl.head_dim * 2
    return {"rows": n, "bytes": nbytes, "us": round(ms * 1e3, 2), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}


def _time_device(run, flush, reps: int = 20):
    """Median CUDA-event time (ms) of run() after 3 warm-up calls, L2 flushed before each."""
    import torch
    for _ in range(3):
        run()
    ts = []
    for _ in range(reps):
        flush.fill_(5)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def merge_bench(msa, pl, dev, flush, hbm_peak, peak_kind):
    """The stand-alone LSE merge (two fp32 partials -> bf16 O and fp32 LSE) at the prefill
    output's shape; not part of the step.  Bytes = both partials and LSEs read, O and LSE
    written."""
    import torch
    rows, heads, d = pl.total_q, pl.num_heads_q, pl.head_dim
    g = torch.Generator(device=dev).manual_seed(20260117)
    o_a = torch.randn(rows, heads, d, generator=g, device=dev)
    o_b = torch.randn(rows, heads, d, generator=g, device=dev)
    l_a = torch.randn(rows, heads, generator=g, device=dev)
    l_b = torch.randn(rows, heads, generator=g, device=dev)
    out = torch.empty(rows, heads, d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(rows, heads, dtype=torch.float32, device=dev)
    ms = _time_device(lambda: msa.merge_lse(o_a, l_a, o_b, l_b, out=out, lse=lse), flush)
    nbytes = rows * heads * (2 * d * 4 + 2 * 4 + d * 2 + 4)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"rows": rows, "heads": heads, "head_dim": d, "bytes": nbytes, "us": round(ms * 1e3, 2),
            "GB/s": round(gbs, 1), "roofline": {"bound": "hbm", "peak": hbm_peak, "frac": round(gbs / hbm_peak, 4),
                                                "peak_source": f"{peak_kind} hbm_gbs"}}


def gather_bench(msa, plan, pw, dev, flush, hbm_peak, peak_kind):
    """The position-order gather of the prefill workload's whole KV context (pool blocks and
    chunk rows, every KV head) into caller buffers; not part of the step.  Bytes = K and V
    read and written once, plus the positions written."""
    import torch
    st = plan.stats()
    n, hkv, d = st["kv_tokens"], plan.num_heads_kv, plan.head_dim
    k = torch.empty(n, hkv, d, dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    pos = torch.empty(n, dtype=torch.int32, device=dev)
    ms = _time_device(lambda: msa.gather(plan, pw.k_chunk, pw.v_chunk, pw.k_pool, pw.v_pool, out=(k, v, pos)),
                      flush)
    nbytes = 2 * (2 * n * hkv * d * 2) + n * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"tokens": n, "bytes": nbytes, "us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
            "roofline": {"bound": "hbm", "peak": hbm_peak, "frac": round(gbs / hbm_peak, 4),
                         "peak_source": f"{peak_kind} hbm_gbs"}}


def ablation_bench(msa, W, pl, pw, dev, flush, reps: int = 10):
    """The many-launch way that one MSA launch replaces: one prefill per cached segment
    (the chunk rows as queries only) plus one over the chunk's own keys, then pairwise
    log-sum-exp merges (msa_merge_lse; the bf16 -> fp32 casts between merges are torch's).
    Same workload, same outputs, timed against one MSA launch; not part of the step."""
    import numpy as np
    import torch
    one = msa.Plan.from_layout(pl).upload(dev)
    one_out = torch.empty_like(pw.q)
    one_lse = torch.empty(pw.q.shape[:2], dtype=torch.float32, device=dev)
    plans = []
    for seg in pl.segments:
        sub = W.Layout(**{**vars(pl), "segments": np.asarray([seg], np.int32)})
        plans.append(msa.Plan.from_layout(sub, chunk_queries_only=True).upload(dev))
    plans.append(msa.Plan.from_layout(W.Layout(**{**vars(pl), "segments": np.zeros((0, 3), np.int32)})).upload(dev))
    outs = [(torch.empty_like(pw.q), torch.empty(pw.q.shape[:2], dtype=torch.float32, device=dev)) for _ in plans]

    def run():
        for pln, (o, l) in zip(plans, outs):
            msa.prefill(pln, pw.q, pw.k_chunk, pw.v_chunk, pw.k_pool, pw.v_pool, out=o, lse=l)

    def merge():
        acc_o, acc_l = outs[0][0].float(), outs[0][1]
        for o, l in outs[1:]:
            mo, ml = msa.merge_lse(acc_o, acc_l, o.float(), l)
            acc_o, acc_l = mo.float(), ml
        return acc_o, acc_l

    def run_one():
        msa.prefill(one, pw.q, pw.k_chunk, pw.v_chunk, pw.k_pool, pw.v_pool, out=one_out, lse=one_lse)

    for _ in range(3):
        run()
        merge()
        run_one()
    t_run, t_merge, t_one = [], [], []
    for _ in range(reps):
        flush.fill_(5)
        e = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        e[0].record()
        run()
        e[1].record()
        merge()
        e[2].record()
        flush.fill_(6)
        e[3].record()
        run_one()
        e[4].record()
        torch.cuda.synchronize()
        t_run.append(e[0].elapsed_time(e[1]))
        t_merge.append(e[1].elapsed_time(e[2]))
        t_one.append(e[3].elapsed_time(e[4]))
    one_ms = statistics.median(t_one)
    for pln in plans:
        if msa.get_status(pln) != 0:
            raise RuntimeError("device error in the per-segment ablation")
    ms_run, ms_merge = statistics.median(t_run), statistics.median(t_merge)
    return {"workload": pl.name, "segments": int(len(pl.segments)), "prefill_launches": len(plans),
            "merges": len(plans) - 1,
            "ms_segment_launches": round(ms_run, 4), "ms_merges": round(ms_merge, 4),
            "ms_total": round(ms_run + ms_merge, 4), "ms_one_msa_launch": round(one_ms, 4),
            "one_launch_speedup": round((ms_run + ms_merge) / one_ms, 3)}


# ----------------------------------------------------------------------------- latency model (Eq. 5)

def latency_model_terms(l1, q1, l2, q2):
    """Regressors of the two-segment prefill latency model, in 16-token blocks.

    The paper's Eq. 5 gives only the marginal cost of recomputing one more block,
    T(l1, q1+1, l2-1, q2) - T(l1, q1, l2, q2) = k5 (l1 + 2 q1) + (k2 - k3 + k5).  The plainest
    T that has exactly that difference (our reading: a request whose first segment is l1
    cached blocks followed by q1 recomputed ones, and whose second segment is l2 cached blocks
    followed by q2 new ones) is T = k0 + k1 l1 + k2 q1 + k3 l2 + k4 q2 + k5 q1 (l1 + q1):
    the quadratic term is the attention of the recomputed blocks over the context before
    them, the linear terms the per-block work."""
    return [1.0, l1, q1, l2, q2, q1 * (l1 + q1)]


def fit_latency_model(samples):
    """Least-squares fit of k0..k5 to [(l1, q1, l2, q2, ms), ...]; returns (k, r2)."""
    import numpy as np
    A = np.array([latency_model_terms(*x[:4]) for x in samples], np.float64)
    y = np.array([x[4] for x in samples], np.float64)
    k, *_ = np.linalg.lstsq(A, y, rcond=None)
    resid = y - A @ k
    r2 = 1.0 - float(resid @ resid) / float(((y - y.mean()) ** 2).sum())
    return k, r2


def two_segment_layout(W, l1, q1, l2, q2, seed):
    """One sequence, blocks of 16: [l1 cached][q1 recomputed][l2 cached][q2 new]; the chunk
    is the q1 + q2 blocks (Llama-3-8B-shaped heads)."""
    import numpy as np
    B = 16
    runs = []
    if l1:
        runs.append((0, l1 * B))
    if l2:
        runs.append(((l1 + q1) * B, l2 * B))
    chunk = np.concatenate([np.arange(l1 * B, (l1 + q1) * B), np.arange((l1 + q1 + l2) * B, (l1 + q1 + l2 + q2) * B)])
    return W.custom_prefill(32, 8, 128, [W.SeqSpec(runs, chunk)], seed=seed, qk_std=1.0 / np.sqrt(128.0))


def run_sweep(args):
    """Cached-ratio sweep (the paper's Fig. 13 measures MSA performance over the cached-token
    ratio; its values are not given) and a fit of the two-segment latency model (Eq. 5) to
    this kernel's timings on one B300.  Prints one JSON line (not the bench line)."""
    import numpy as np
    import torch
    import segmented_kv_attention_msa_b300 as msa
    from segmented_kv_attention_msa_b300 import build as B
    from segmented_kv_attention_msa_b300 import workload as W
    if not os.path.exists(msa.LIB_PATH):
        B.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def time_layout(lay, reps=8):
        wl = W.make_values(lay, device=dev)
        plan = msa.Plan.from_layout(lay).upload(dev)
        out = torch.empty_like(wl.q)
        lse = torch.empty(wl.q.shape[:2], dtype=torch.float32, device=dev)
        for _ in range(3):
            msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool, out=out, lse=lse)
        ts = []
        for _ in range(reps):
            flush.fill_(7)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            msa.prefill(plan, wl.q, wl.k_chunk, wl.v_chunk, wl.k_pool, wl.v_pool, out=out, lse=lse)
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        if msa.get_status(plan) != 0:
            raise RuntimeError("device error in the sweep")
        return statistics.median(ts), plan.stats()["useful_flops"]

    # cached-ratio sweep: 16384-token context of 1024 blocks, a random fraction cached, plus
    # 256 new tokens; the chunk is every evicted block and the new tokens (one launch)
    rng = np.random.default_rng(13)
    sweep = []
    for ratio in (0.0, 0.25, 0.5, 0.75, 0.9):
        cached = rng.random(1024) < ratio
        R = int((~cached).sum()) * 16 + 256
        runs_pool, chunk = W._split_recompute(~cached, 1024 * 16, 256, [R])
        spec = W.SeqSpec(W._cached_runs_tokens(cached) + runs_pool, chunk)
        lay = W.custom_prefill(32, 8, 128, [spec], seed=17, qk_std=1.0 / np.sqrt(128.0))
        ms, fl = time_layout(lay)
        # prefix-only reuse (a prefix cache): the cached blocks before the first evicted one
        # are reused, everything after them is recomputed, in one launch
        f = int(np.argmin(cached)) if not cached.all() else 1024
        pspec = W.SeqSpec([(0, f * 16)] if f else [], np.arange(f * 16, 1024 * 16 + 256))
        ms_pre, _ = time_layout(W.custom_prefill(32, 8, 128, [pspec], seed=17, qk_std=1.0 / np.sqrt(128.0)))
        sweep.append({"cached_ratio": ratio, "cached_blocks": int(cached.sum()), "chunk_tokens": int(lay.total_q),
                      "segments": int(len(lay.segments)), "ms": round(ms, 4), "useful_tflops": round(fl / ms / 1e9, 1),
                      "prefix_only_reused_blocks": f, "prefix_only_ms": round(ms_pre, 4),
                      "speedup_vs_prefix_only": round(ms_pre / ms, 3)})
    base = sweep[0]["ms"]
    for x in sweep:
        x["speedup_vs_full_recompute"] = round(base / x["ms"], 3)

    # latency model: a grid of two-segment requests (in blocks)
    samples = []
    for l1 in (0, 64, 256):
        for q1 in (16, 64, 128):
            for l2 in (0, 64, 256):
                for q2 in (8, 32):
                    lay = two_segment_layout(W, l1, q1, l2, q2, seed=l1 + q1 + l2 + q2)
                    ms, _ = time_layout(lay, reps=5)
                    samples.append((l1, q1, l2, q2, ms))
    k, r2 = fit_latency_model(samples)
    pred = [float(np.dot(latency_model_terms(*x[:4]), k)) for x in samples]
    max_rel = max(abs(pv - x[4]) / x[4] for pv, x in zip(pred, samples))
    res = {"kind": "cached_ratio_sweep_and_latency_model", "gpu": torch.cuda.get_device_name(dev),
           "sweep": sweep,
           "latency_model": {"terms": "T = k0 + k1 l1 + k2 q1 + k3 l2 + k4 q2 + k5 q1 (l1 + q1), blocks of 16, ms",
                             "k": [float(f"{x:.6g}") for x in k], "r2": round(r2, 4), "samples": len(samples),
                             "max_rel_err": round(max_rel, 4),
                             "delta_T_B": "k5 (l1 + 2 q1) + (k2 - k3 + k5)"}}
    print(json.dumps(res), flush=True)


# ----------------------------------------------------------------------------- eviction policy

# Eq. 5 coefficients of the two-segment latency model fitted to this kernel's timings on
# B300 (bench.py --sweep; ms per 16-token block): k5 and k2 - k3 + k5
EVICT_K5 = 3.07463e-6
EVICT_KCONST = 1.10065e-4 - 7.83825e-5 + 3.07463e-6


def modelled_recompute_cost(hit, k5=EVICT_K5, k_const=EVICT_KCONST):
    """Modelled recompute time of one request (ms): Eq. 5's marginal cost
    k5 (l1 + 2 q1) + (k2 - k3 + k5) summed over its recomputed blocks in position order,
    l1 and q1 the cached and recomputed blocks before each."""
    cost, l1, q1 = 0.0, 0, 0
    for h in hit:
        if h:
            l1 += 1
        else:
            cost += k5 * (l1 + 2 * q1) + k_const
            q1 += 1
    return cost


def replay_trace(policy, trace, capacity, k5=EVICT_K5, k_const=EVICT_KCONST):
    """Serve a request trace (time, session, context blocks) through a cache of
    `capacity` blocks managed by `policy` (insert / access / victim).  A request reads
    blocks 0 .. n-1 of its session: cached ones are hits (accessed), the rest are
    recomputed and cached; then the policy evicts until the cache fits again (any block,
    this request's included: its KV has been used).  Returns hit counts and the modelled
    recompute time, with and without the cache."""
    cached = set()
    hits = total = 0
    cost = cost_none = 0.0
    for (now, sess, n) in trace:
        ids = [sess * 65536 + b for b in range(n)]
        hit = [b in cached for b in ids]
        for b, h in zip(ids, hit):
            if h:
                policy.access(b, now)
        for pb, (b, h) in enumerate(zip(ids, hit)):
            if not h:
                policy.insert(b, pb, now)
                cached.add(b)
        while len(cached) > capacity:
            cached.remove(policy.victim(now))
        hits += sum(hit)
        total += n
        cost += modelled_recompute_cost(hit, k5, k_const)
        cost_none += modelled_recompute_cost([False] * n, k5, k_const)
    return {"hits": hits, "blocks": total, "hit_rate": hits / max(1, total), "modelled_ms": cost,
            "modelled_ms_no_cache": cost_none}


def run_evict(args):
    """Eviction policies on a synthetic multi-turn trace (prints its own JSON line): the
    cost-aware policy against LRU and prefix-only at several cache sizes (hit rate and
    modelled recompute time), and the time per eviction of the O(log n) structure against
    the O(n) scan and LRU at 4k-10k cached blocks (the comparison of Fig. 8)."""
    import numpy as np
    import segmented_kv_attention_msa_b300 as msa
    from segmented_kv_attention_msa_b300 import build as B
    from segmented_kv_attention_msa_b300 import workload as W
    if not os.path.exists(msa.LIB_PATH):
        B.build()
    trace = W.multiturn_trace()
    final = {}
    for (_, s, n) in trace:
        final[s] = n
    distinct = sum(final.values())
    res = {"kind": "eviction_policy_synthetic_trace", "trace": {"requests": len(trace), "sessions": len(final),
           "distinct_blocks": distinct, "blocks_read": sum(n for _, _, n in trace), "generator": "workload.multiturn_trace()"},
           "model": {"k5": EVICT_K5, "k_const": EVICT_KCONST, "unit": "ms per 16-token block"},
           "policies": {}}
    for frac in (0.1, 0.2, 0.4):
        cap = int(distinct * frac)
        row = {}
        for name in ("lru", "prefix", "cost"):
            t0 = time.perf_counter()
            r = replay_trace(msa.EvictionPolicy(name), trace, cap)
            r["wall_s"] = round(time.perf_counter() - t0, 2)
            r["hit_rate"] = round(r["hit_rate"], 4)
            r["modelled_ms"] = round(r["modelled_ms"], 1)
            r["modelled_ms_no_cache"] = round(r["modelled_ms_no_cache"], 1)
            row[name] = r
        res["policies"][f"capacity_{int(frac * 100)}pct"] = {"capacity_blocks": cap, **row}
    # time per eviction at n cached blocks: insert n, then alternate evict / insert
    timing = {}
    rng = np.random.default_rng(5)
    for n in (4000, 6000, 8000, 10000):
        row = {}
        for name in ("lru", "cost", "cost_scan"):
            p = msa.EvictionPolicy(name, period=0)
            for b in range(n):
                p.insert(b, int(rng.integers(0, 4096)), float(b % 97))
            reps = 2000
            t0 = time.perf_counter()
            for k in range(reps):
                p.victim(100.0 + k)
                p.insert(n + k, int(rng.integers(0, 4096)), 100.0 + k)
            row[name] = round((time.perf_counter() - t0) / reps * 1e6, 2)
        timing[str(n)] = row
    res["us_per_evict_and_insert"] = timing
    print(json.dumps(res), flush=True)


def _single_kernel_result(args, world, pl, dl, pst, dst, pf_mean, dc_mean, peaks, peak_kind, clocks):
    """Result line of a one-kernel run (--only), used for profiling captures."""
    res = {"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "only": args.only,
           "higher_is_better": True, "scaling": "weak", "dtype": "bf16", "data": "synthetic", "clocks": clocks,
           "gpu_launches": args.steps}
    if args.only == "prefill":
        ach = pst["useful_flops"] / (pf_mean * 1e-3) / 1e12
        res.update({"value": round(ach, 3), "unit": "TFLOP/s", "ms_per_step": round(pf_mean, 4),
                    "config": {"workload": pl.name},
                    "roofline": {"bound": "tensor", "achieved": round(ach, 2), "peak": peaks["bf16_tflops"],
                                 "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 4),
                                 "traffic": kernel_traffic("prefill", pl.name),
                                 "peak_source": f"{peak_kind} bf16_tflops (burst)"}})
    else:
        ach = dst["algorithmic_bytes"] / (dc_mean * 1e-3) / 1e9
        res.update({"value": round(ach, 1), "unit": "GB/s", "ms_per_step": round(dc_mean, 4),
                    "config": {"workload": dl.name},
                    "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                 "frac": round(ach / peaks["hbm_gbs"], 4),
                                 "traffic": kernel_traffic("decode", dl.name),
                                 "peak_source": f"{peak_kind} hbm_gbs"}})
    return res


# ----------------------------------------------------------------------------- the oracle as baseline

def oracle_prefill_sample(pl, arrays, rows):
    from oracle import msa_oracle as O
    t0 = time.perf_counter()
    O.prefill(pl, arrays["q"], arrays["k_chunk"], arrays["v_chunk"], arrays["k_pool"], arrays["v_pool"],
              1.0 / math.sqrt(pl.head_dim), rows=rows)
    return time.perf_counter() - t0


def sample_flops(pl, rows):
    """Useful FLOPs of the sampled query rows (visible pairs x 4 d Hq), counted directly."""
    import numpy as np
    total = 0
    for s in range(pl.num_seqs):
        pos = []
        for (q, f, nb) in pl.segments:
            if q != s:
                continue
            for i in range(nb):
                b = pl.block_table[s, f + i]
                pos.extend(range(int(pl.block_pos[b]), int(pl.block_pos[b]) + int(pl.block_fill[b])))
        pos.extend(pl.q_pos[pl.cu_q[s]:pl.cu_q[s + 1]].tolist())
        pos = np.sort(np.array(pos))
        sel = [r for r in rows if pl.cu_q[s] <= r < pl.cu_q[s + 1]]
        total += int(np.searchsorted(pos, pl.q_pos[sel], side="right").sum())
    return total * pl.num_heads_q * 4 * pl.head_dim


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def sample_rows(pl, n_rows, flop_budget, seed=0):
    """Query rows for a bounded oracle run: `n_rows` random rows if n_rows > 0, else
    random rows until their useful FLOPs reach `flop_budget`."""
    import numpy as np
    rng = np.random.default_rng(seed)
    order = rng.permutation(pl.total_q)
    if n_rows > 0:
        return np.sort(order[:min(n_rows, pl.total_q)])
    take, fl = 0, 0
    while take < len(order) and fl < flop_budget:
        step = max(1, min(len(order) - take, 8))
        fl += sample_flops(pl, np.sort(order[take:take + step]))
        take += step
    return np.sort(order[:take])


def cpu_baseline(pl, pw, n_rows):
    import numpy as np
    arrays = {k: getattr(pw, k).float().cpu().numpy().astype(np.float64)
              for k in ("q", "k_chunk", "v_chunk", "k_pool", "v_pool")}
    rows = sample_rows(pl, n_rows, 6e11)
    secs = oracle_prefill_sample(pl, arrays, rows)
    fl = sample_flops(pl, rows)
    return {"value": round(fl / secs / 1e12, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{len(rows)} of {pl.total_q} query rows of {pl.name}, all {pl.num_heads_q} heads, "
                      f"fp64 numpy ({secs:.2f} s)"}


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle, timed on this host, on a bounded sample per step."""
    if rank != 0:
        return None
    import numpy as np
    from segmented_kv_attention_msa_b300 import workload as W
    pl = W.make_layout(args.workload, tiler=_oracle_tiler())
    pw = W.make_values(pl, device="cpu")
    arrays = {k: getattr(pw, k).float().numpy().astype(np.float64)
              for k in ("q", "k_chunk", "v_chunk", "k_pool", "v_pool")}
    # the whole run stays within a few minutes: about 2.5e12 useful FLOPs over all the timed
    # steps (the oracle does ~0.03 TFLOP/s on 16 cores), at most 1e11 per step
    rows = sample_rows(pl, args.ref_rows, min(1e11, 2.5e12 / max(1, args.steps)))
    for _ in range(args.warmup):
        oracle_prefill_sample(pl, arrays, rows[:8])
    t = [oracle_prefill_sample(pl, arrays, rows) for _ in range(args.steps)]
    fl = sample_flops(pl, rows)
    v = fl / statistics.mean(t) / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.mean(t) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generator)",
        "config": {"workload": pl.name, "sample_rows": len(rows)},
        "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{len(rows)} of {pl.total_q} query rows per step, all heads"},
        "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def _oracle_tiler():
    from oracle import msa_oracle as O
    return O.chunk_sizes


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=5, help="prefill workload (1, 2, 3 or 5)")
    ap.add_argument("--decode-workload", type=int, default=4)
    ap.add_argument("--decode-batch", type=int, default=64,
                    help="sequences of the decode workload (64 = the bench line; fewer for profiling captures)")
    ap.add_argument("--cpu-rows", type=int, default=0,
                    help="query rows of the oracle baseline (0: as many as about 6e11 useful FLOPs)")
    ap.add_argument("--ref-rows", type=int, default=0,
                    help="query rows per reference-arm step (0: as many as about min(1e11, 2.5e12 / steps) "
                         "useful FLOPs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-ablation", action="store_true", help="skip the per-segment launch comparison")
    ap.add_argument("--sweep", action="store_true",
                    help="cached-ratio sweep and latency-model fit (prints its own JSON line, not the bench line)")
    ap.add_argument("--evict", action="store_true",
                    help="eviction policies on a synthetic multi-turn trace (prints its own JSON line; no GPU)")
    ap.add_argument("--only", choices=["prefill", "decode"], default=None,
                    help="time one kernel alone (for profiling captures); not the bench line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.evict:
        run_evict(args)
        return
    world, rank, local = dist_setup()
    if args.sweep:
        if rank == 0:
            run_sweep(args)
        return
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_ours(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
