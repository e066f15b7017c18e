#!/usr/bin/env python3
"""Benchmark: MLA decode over a paged latent KV cache on GB300.

One step = the whole hot path on one batch: the cache write of the batch's new
tokens, the split-KV pass and the LSE merge, with the split count from
mla_num_kv_splits, launched by one mla_plan_run of a plan prepared before the
timed region (``--api calls``: the per-stage entry points mla_cache_write,
mla_decode_splitkv and mla_decode_merge instead; the per-kernel times always
come from a second pass through those, with an event between kernels).  The
default workload is the DeepSeek-style per-shard decode batch (B=64, H=16,
head 576 = 512+64, block 64, seq_lens ~ U{1024..4096}, 64 new tokens).

Prints ONE JSON line (rank 0).  Timing: W warm-up steps, then K steps, each
step bracketed by CUDA events on the launching stream, L2 flushed between steps
by writing a 256 MiB buffer (outside the events); barrier + synchronize on
both sides; the max over ranks.  Multi-GPU (torchrun): every rank runs its own
replica of the batch (no collective on the data path), value = all ranks'
bytes / max time.

``--impl reference`` times the CPU oracle (the plain fp64 restatement of the
method) on the host cores on a bounded sample of the same workload.
``--op lse_merge`` times the cross-shard merge alone; ``--fused-write`` makes
the step's write the fused RMSNorm + rotary write.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 256 << 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def _traffic_record(kernel_src: str, workload: str):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, or None when the kernel source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        with open(kernel_src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        r = rec.get(workload)
        if r and r.get("kernel_sha256") == sha:
            return float(r["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"],
                    "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- multi-rank host logic
def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over all ranks (x itself without a process
    group).  The timed region of the slowest replica sets the job's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step: int, steps: int, world: int, total_ms: float) -> float:
    """Whole-job GB/s: the bytes every replica processed over the slowest
    replica's time (replicas: each of the `world` ranks runs its own batch)."""
    return bytes_per_step * steps * world / (total_ms * 1e-3) / 1e9


# ---------------------------------------------------------------- our arm
# Steps of each record in the ``configs`` list (the headline workload takes
# --steps).
CONFIG_STEPS = 10
# The other workloads, measured after the headline one and reported under
# ``configs``: (workload, num_kv_splits = 1).
OTHER_CONFIGS = (("per_shard", False), ("full_head", False), ("full_head", True),
                 ("fp8_small", False), ("tiny", False))


def _roofline(w, args, workload, deterministic, kv_bytes, flops, s1_ms):
    """Roofline record of the stage-1 kernel: the KV bytes (or, above the
    ridge, the flops) of one launch over its CUDA-event duration, against the
    measured peak."""
    hbm, bf16, src = _peaks()
    R, H = w.kv_lora_rank, w.num_heads
    achieved = kv_bytes / (s1_ms * 1e-3) / 1e9
    # the stage-1 kernel the library picks: a tcgen05 kernel (R = 512 bf16:
    # CTA pairs; R = 256 bf16 or fp8: one CTA) from 64 query vectors per
    # sequence, warp MMA otherwise
    tc = (R == 256 or not w.kv_fp8) and w.rows_per_seq * H > 32 and args.path != 1
    tc = tc or args.path == 2
    kernel_src = ("decode_tc1.cu" if R == 256 else "decode_tc.cu") if tc else "decode_mma.cu"
    traffic = _traffic_record(os.path.join(ROOT, "mla_paged_kv_concat_gb300", "csrc",
                                           kernel_src),
                              workload + ("_s1" if deterministic else ""))
    kname = (("decode_tc1_kernel" if R == 256 else "decode_tc_kernel") if tc
             else "decode_mma_kernel") + " (stage 1)"
    if flops / (bf16 * 1e12) > kv_bytes / (hbm * 1e9):
        # above the ridge (several query rows share each cached row): the
        # contraction's flops against the bf16 tensor peak
        tf = flops / (s1_ms * 1e-3) / 1e12
        return {"bound": "tensor", "kernel": kname, "achieved": round(tf, 1),
                "peak": bf16, "unit": "TFLOP/s", "frac": round(tf / bf16, 4),
                "traffic": traffic,
                "peak_source": f"{src} (MEASURED_PEAKS.json bf16_tflops, burst)",
                "hbm_gbs": round(achieved, 1)}
    return {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1),
            "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
            "traffic": traffic,
            "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs, burst)"}


def run_ours(args, rank, world, local_rank, workload=None, deterministic=None, light=False):
    """One workload's measurement.  light: the per-config record of the
    ``configs`` list (no e2e pass), with its own step count."""
    import torch
    import mla_paged_kv_concat_gb300 as mla
    from mla_paged_kv_concat_gb300 import workloads as W

    workload = args.workload if workload is None else workload
    deterministic = args.deterministic if deterministic is None else deterministic
    steps = min(args.steps, CONFIG_STEPS) if light else args.steps
    warmup = 3 if light else args.warmup
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = mla.load()
    w = W.make(workload)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    S = 1 if deterministic else mla.mla_num_kv_splits(w.max_seq_len, sms)
    R, P, D, H = w.kv_lora_rank, w.rope_dim, w.head_dim, w.num_heads
    rows, seqs = w.num_rows, w.num_seqs
    kvd = mla.MLA_KV_FP8_E4M3 if w.kv_fp8 else mla.MLA_KV_BF16

    # resident device state
    if w.kv_fp8:
        cache = torch.from_numpy(w.kv_cache).to(dev)
    else:
        cache = torch.from_numpy(w.kv_cache.view(np.int16)).view(torch.bfloat16).to(dev)
    nb, bs = w.kv_cache.shape[0], w.block_size
    bstride = bs * D
    q = w.q.to(dev)
    bt = torch.from_numpy(w.block_table).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    kv_c, k_pe = w.kv_c.to(dev), w.k_pe.to(dev)
    slots = torch.from_numpy(w.slot_mapping).to(dev)
    T = slots.numel()
    kv_scale = torch.tensor([w.kv_scale], dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    o = torch.empty(rows, H, R, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(rows, H, dtype=torch.float32, device=dev)
    wsb = mla.mla_decode_workspace_bytes(rows, H, S, R)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def flush_l2():
        # Overwrite L2 with a buffer twice its size, then read the buffer
        # back: the read leaves clean lines, so the timed kernels neither hit
        # their inputs in L2 nor pay for writing back the flush's dirty lines.
        flush.zero_()
        flush.view(torch.int32).sum()
    stream = torch.cuda.current_stream(dev)
    sp = int(stream.cuda_stream)
    maxb = bt.shape[1]

    if args.fused_write:
        # the write fused with RMSNorm of kv_c and the rotary embedding of k_pe
        # (and of q's rope columns when every written token is a query row)
        nr = W.norm_rope_inputs(w, seed=11)
        nr_gamma = nr.gamma.to(dev)
        nr_pos = torch.from_numpy(nr.positions).to(dev)
        nr_table = torch.from_numpy(nr.table).to(dev)
        rot_q = T == rows

    def write(kv_c_t, k_pe_t, slots_t, q_t=None):
        if args.fused_write:
            qp = q_t[:, :, R:] if (rot_q and q_t is not None) else None
            st = lib.mla_norm_rope_cache_write(
                kv_c_t.data_ptr(), kv_c_t.stride(0), k_pe_t.data_ptr(), k_pe_t.stride(0),
                slots_t.data_ptr(), T, R, P, cache.data_ptr(), nb, bs, bstride, kvd,
                kv_scale.data_ptr(), nr_gamma.data_ptr(), nr.eps, nr_pos.data_ptr(),
                nr_table.data_ptr(), nr_table.shape[0],
                qp.data_ptr() if qp is not None else None, qp.stride(0) if qp is not None else 0,
                qp.stride(1) if qp is not None else 0, H if qp is not None else 0,
                err.data_ptr(), sp)
        else:
            st = lib.mla_cache_write(kv_c_t.data_ptr(), kv_c_t.stride(0), k_pe_t.data_ptr(),
                                     k_pe_t.stride(0), slots_t.data_ptr(), T, R, P,
                                     cache.data_ptr(), nb, bs, bstride, kvd,
                                     kv_scale.data_ptr(), err.data_ptr(), sp)
        assert st == 0, st

    def stage1(q_t, bt_t, sl_t, o_t, lse_t):
        st = lib.mla_decode_splitkv(q_t.data_ptr(), q_t.stride(0), q_t.stride(1), rows, H,
                                    cache.data_ptr(), kvd, nb, bs, bstride, R, P,
                                    bt_t.data_ptr(), bt_t.stride(0), maxb, sl_t.data_ptr(),
                                    seqs, w.sm_scale, kv_scale.data_ptr(), S, ws.data_ptr(),
                                    ws.numel(), o_t.data_ptr(), lse_t.data_ptr(),
                                    err.data_ptr(), sp, args.path)
        assert st == 0, st

    def merge(sl_t, o_t, lse_t):
        st = lib.mla_decode_merge(rows, H, R, sl_t.data_ptr(), seqs, bs, maxb, S,
                                  ws.data_ptr(), ws.numel(), o_t.data_ptr(),
                                  lse_t.data_ptr(), sp)
        assert st == 0, st

    launches_per_step = (1 if T else 0) + 1 + (1 if S > 1 else 0)

    def make_plan(q_t, bt_t, sl_t, kv_c_t, k_pe_t, slots_t, o_t=None, lse_t=None):
        """The step as one prepared plan: run() only launches the kernels."""
        nr_args = None
        if args.fused_write:
            nr_args = dict(gamma=nr_gamma, eps=nr.eps, positions=nr_pos,
                           cos_sin_table=nr_table, rotate_q=rot_q)
        return mla.DecodePlan(q_t, cache, bt_t, sl_t, w.sm_scale, S, kv_scale=kv_scale,
                              kv_cache_dtype="fp8" if w.kv_fp8 else None, workspace=ws,
                              out=o if o_t is None else o_t, lse=lse if lse_t is None else lse_t,
                              err_count=err, path=args.path,
                              write=dict(kv_c=kv_c_t, k_pe=k_pe_t, slot_mapping=slots_t),
                              norm_rope=nr_args)

    plan = make_plan(q, bt, sl, kv_c, k_pe, slots) if args.api == "plan" else None

    def step_events():
        # One step bracketed by two events only: an event recorded between
        # two kernels would stop the next one from launching while the
        # previous one drains (programmatic dependent launch).
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e[0].record(stream)
        if plan is not None:
            plan.run(stream)
        else:
            write(kv_c, k_pe, slots, q)
            stage1(q, bt, sl, o, lse)
            merge(sl, o, lse)
        e[1].record(stream)
        return e

    def step_kernel_events():
        # The same step with an event between the kernels, for the per-kernel
        # times (the stage-1 time is the roofline's denominator).
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(stream)
        write(kv_c, k_pe, slots, q)
        e[1].record(stream)
        stage1(q, bt, sl, o, lse)
        e[2].record(stream)
        merge(sl, o, lse)
        e[3].record(stream)
        return e

    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(warmup):
        flush_l2()
        step_events()
        flush_l2()
        step_kernel_events()
    torch.cuda.synchronize(dev)

    evs, kevs = [], []
    with ClockSampler(local_rank) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        for _ in range(steps):
            flush_l2()
            evs.append(step_events())
        torch.cuda.synchronize(dev)
        barrier()
        for _ in range(steps):
            flush_l2()
            kevs.append(step_kernel_events())
        torch.cuda.synchronize(dev)
    t_write = [e[0].elapsed_time(e[1]) for e in kevs]
    t_s1 = [e[1].elapsed_time(e[2]) for e in kevs]
    t_merge = [e[2].elapsed_time(e[3]) for e in kevs]
    t_step = [e[0].elapsed_time(e[1]) for e in evs]
    total_ms = max_over_ranks(float(np.sum(t_step)), dev)
    ms_step = total_ms / steps
    kv_bytes = w.kv_bytes()
    flops = w.flops()
    n_units = world * steps
    value = job_throughput(kv_bytes, steps, world, total_ms)
    hbm, bf16, src = _peaks()
    s1_ms = float(np.mean(t_s1))
    roofline = _roofline(w, args, workload, deterministic, kv_bytes, flops, s1_ms)
    roof_t = max(kv_bytes / (hbm * 1e9), flops / (bf16 * 1e12))
    kernel_ms = {("norm_rope_cache_write" if args.fused_write else "cache_write"):
                 round(float(np.mean(t_write)), 5),
                 "decode_splitkv": round(s1_ms, 5),
                 "decode_merge": round(float(np.mean(t_merge)), 5)}
    if light:
        if rank != 0:
            return None
        return {"workload": workload + ("_s1" if deterministic else ""), "num_kv_splits": S,
                "rows": rows, "heads": H, "kv_tokens": int(w.seq_lens.sum()),
                "kv_bytes": kv_bytes, "steps": steps, "warmup": warmup,
                "ms_per_step": round(ms_step, 5), "value": round(value, 2), "unit": "GB/s",
                "tflops": round(flops * n_units / (total_ms * 1e-3) / 1e12, 2),
                "kernel_ms": kernel_ms, "roofline": roofline,
                "step_roofline_frac": round(roof_t / (ms_step * 1e-3), 4),
                "decode_rows_per_s": round(rows / ((s1_ms + float(np.mean(t_merge))) * 1e-3), 1),
                "gpu_launches": launches_per_step * steps, "clocks": clk.summary()}

    # ---- e2e through the C ABI with host buffers (pinned), copies timed.
    # The step's inputs sit in one pinned host block and go over in one
    # copy; o and lse come back in one copy (separate small copies each pay
    # a few microseconds of fixed cost).
    def carve(buf, specs):
        """Views of `buf` (uint8) for (shape, dtype) specs at 256-byte offsets."""
        out, off = [], 0
        for shape, dt in specs:
            n = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
            out.append(buf[off:off + n].view(dt).view(shape))
            off = (off + n + 255) // 256 * 256
        return out, off

    in_specs = [(tuple(q.shape), q.dtype), (tuple(bt.shape), bt.dtype),
                (tuple(sl.shape), sl.dtype), (tuple(kv_c.shape), kv_c.dtype),
                (tuple(k_pe.shape), k_pe.dtype), (tuple(slots.shape), slots.dtype)]
    out_specs = [(tuple(o.shape), o.dtype), (tuple(lse.shape), lse.dtype)]
    _, in_bytes = carve(torch.empty(1 << 30, dtype=torch.uint8, device="meta"), in_specs)
    _, out_bytes = carve(torch.empty(1 << 30, dtype=torch.uint8, device="meta"), out_specs)
    h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    h_outb = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    d_outb = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
    (h_q, h_bt, h_sl, h_kvc, h_kpe, h_slots), _ = carve(h_in, in_specs)
    (d_q, d_bt, d_sl, d_kvc, d_kpe, d_slots), _ = carve(d_in, in_specs)
    (h_o, h_lse), _ = carve(h_outb, out_specs)
    (d_o, d_lse), _ = carve(d_outb, out_specs)
    h_q.copy_(w.q)
    h_bt.copy_(torch.from_numpy(w.block_table))
    h_sl.copy_(torch.from_numpy(w.seq_lens))
    h_kvc.copy_(w.kv_c)
    h_kpe.copy_(w.k_pe)
    h_slots.copy_(torch.from_numpy(w.slot_mapping))
    h2d = in_bytes
    d2h = out_bytes

    e2e_plan = None
    if args.api == "plan":
        e2e_plan = make_plan(d_q, d_bt, d_sl, d_kvc, d_kpe, d_slots, d_o, d_lse)

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        if e2e_plan is not None:
            e2e_plan.run(stream)
        else:
            write(d_kvc, d_kpe, d_slots, d_q)
            st = lib.mla_decode(d_q.data_ptr(), d_q.stride(0), d_q.stride(1), rows, H,
                                cache.data_ptr(), kvd, nb, bs, bstride, R, P, d_bt.data_ptr(),
                                d_bt.stride(0), maxb, d_sl.data_ptr(), seqs, w.sm_scale,
                                kv_scale.data_ptr(), S, ws.data_ptr(), ws.numel(),
                                d_o.data_ptr(), d_lse.data_ptr(), err.data_ptr(), sp)
            assert st == 0, st
        h_outb.copy_(d_outb, non_blocking=True)

    for _ in range(warmup):
        flush_l2()
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_ms = []
    for _ in range(steps):
        flush_l2()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        e2e_ms.append((a, b))
    torch.cuda.synchronize(dev)
    e2e_serial_total = max_over_ranks(float(sum(a.elapsed_time(b) for a, b in e2e_ms)), dev)
    e2e_serial_value = job_throughput(kv_bytes, steps, world, e2e_serial_total)

    # ---- e2e as a serving loop runs it: step i's inputs go up on one copy
    # stream while step i - 1 computes, results come back on another; two
    # staging sets alternate.  No L2 flush between steps (the loop has no
    # gap for one), so this figure is used only when a step's KV bytes
    # exceed L2.
    e2e_pipe_total = None
    if args.api == "plan":
        sets = []
        for _ in range(2):
            di = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
            do_ = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
            ho = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
            (q_, bt_, sl_, kvc_, kpe_, sl2_), _ = carve(di, in_specs)
            (o_, lse_), _ = carve(do_, out_specs)
            sets.append((di, do_, ho, make_plan(q_, bt_, sl_, kvc_, kpe_, sl2_, o_, lse_)))
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def pipelined(k):
            ev = {(n, i): torch.cuda.Event() for n in ("in", "comp", "out") for i in range(k)}
            for i in range(k):
                di, do_, ho, pl = sets[i % 2]
                if i >= 2:
                    up.wait_event(ev["comp", i - 2])    # its inputs are no longer read
                    stream.wait_event(ev["out", i - 2])  # its outputs have been copied
                with torch.cuda.stream(up):
                    di.copy_(h_in, non_blocking=True)
                    ev["in", i].record(up)
                stream.wait_event(ev["in", i])
                pl.run(stream)
                ev["comp", i].record(stream)
                down.wait_event(ev["comp", i])
                with torch.cuda.stream(down):
                    ho.copy_(do_, non_blocking=True)
                    ev["out", i].record(down)
            stream.wait_event(ev["out", k - 1])

        pipelined(max(warmup, 2))
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        up.wait_stream(stream)
        pipelined(steps)
        b.record(stream)
        torch.cuda.synchronize(dev)
        e2e_pipe_total = max_over_ranks(a.elapsed_time(b), dev)
    l2_bytes = 129e6
    use_pipe = e2e_pipe_total is not None and kv_bytes > l2_bytes
    e2e_total = e2e_pipe_total if use_pipe else e2e_serial_total
    e2e_value = job_throughput(kv_bytes, steps, world, e2e_total)
    if int(err.item()) != 0:
        print(f"warning: device error counter {int(err.item())}", file=sys.stderr)

    if rank != 0:
        return None
    line = {
        "metric": "MLA decode KV GB/s & TFLOPS as % of roofline; decode rows/s at 1 GB300",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if not w.kv_fp8 else "bf16 q / e4m3 cache",
        "data": "synthetic (seeded N(0,1) bf16; NaN-poisoned unused cache memory)",
        "config": {
            "workload": workload + ("_s1" if deterministic else ""), "num_seqs": seqs,
            "rows": rows, "heads": H,
            "kv_lora_rank": R, "rope_dim": P, "block_size": bs,
            "seq_lens": [int(w.seq_lens.min()), int(w.seq_lens.max())],
            "kv_tokens": int(w.seq_lens.sum()), "new_tokens": T, "num_kv_splits": S,
            "parallelism": f"replicas x{world}",
            "write": "RMSNorm + rotary + cache write (fused)" if args.fused_write else "cache write",
            "api": "mla_plan_run (prepared plan)" if args.api == "plan"
                   else "mla_cache_write + mla_decode_splitkv + mla_decode_merge",
            "l2": "flushed between steps (256 MiB write, then read back)",
        },
        "tflops": round(flops * n_units / (total_ms * 1e-3) / 1e12, 2),
        "rows_per_s": round(rows * n_units / (total_ms * 1e-3), 1),
        # decode rows/s over stage 1 + merge (the per-kernel pass), and every
        # byte the step moves (KV, q, o, lse, block table, seq_lens) per step time
        "decode_rows_per_s": round(rows / ((s1_ms + float(np.mean(t_merge))) * 1e-3), 1),
        "all_bytes_gbs": round((kv_bytes + q.numel() * 2 + o.numel() * 2 + lse.numel() * 4
                                + bt.numel() * 4 + sl.numel() * 4) / (ms_step * 1e-3) / 1e9, 1),
        "cache_write_gbs": round(T * D * (2 + (1 if w.kv_fp8 else 2))
                                 / (float(np.mean(t_write)) * 1e-3) / 1e9, 1),
        "step_roofline_frac": round(roof_t / (ms_step * 1e-3), 4),
        "kernel_ms": kernel_ms,
        "roofline": roofline,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_total / steps, 5),
                "mode": ("pipelined: copies of step i+1 overlap step i, no L2 flush "
                         "(a step's KV bytes exceed L2)") if use_pipe else
                        "serial: copy in, step, copy out; L2 flushed between steps",
                "serial_value": round(e2e_serial_value, 2),
                "serial_ms_per_step": round(e2e_serial_total / steps, 5),
                "pipelined_ms_per_step": round(e2e_pipe_total / steps, 5)
                if e2e_pipe_total is not None else None},
        "gpu_launches": launches_per_step * steps,
        "clocks": clk.summary(),
    }
    return line


# ---------------------------------------------------------------- cross-shard merge
def run_lse_merge(args):
    """Time mla_lse_merge alone: G shards' (o, lse) of a decode batch (rows x
    H query vectors, R-wide latent) merged into one.  HBM-bound: it reads
    every part once and writes the result once."""
    import torch
    import mla_paged_kv_concat_gb300 as mla

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lib = mla.load()
    G, rows, H, R = args.parts, args.merge_rows, args.merge_heads, 512
    n = rows * H
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    o_parts = torch.randn(G, rows, H, R, device=dev, generator=gen).to(torch.bfloat16)
    lse_parts = torch.randn(G, rows, H, device=dev, generator=gen) * 4.0
    o = torch.empty(rows, H, R, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(rows, H, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = int(stream.cuda_stream)

    def merge():
        st = lib.mla_lse_merge(o_parts.data_ptr(), o_parts.stride(0), lse_parts.data_ptr(),
                               lse_parts.stride(0), G, rows, H, R, o.data_ptr(),
                               lse.data_ptr(), sp)
        assert st == 0, st

    for _ in range(args.warmup):
        flush.zero_()
        merge()
    torch.cuda.synchronize(dev)
    evs = []
    with ClockSampler(0) as clk:
        for _ in range(args.steps):
            flush.zero_()
            flush.view(torch.int32).sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            merge()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize(dev)
    ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    nbytes = G * n * (R * 2 + 4) + n * (R * 2 + 4)
    achieved = nbytes / (ms * 1e-3) / 1e9
    hbm, _, src = _peaks()
    return {
        "metric": "cross-shard LSE merge GB/s", "value": round(achieved, 1), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 parts, lse ~ 4 N(0,1))",
        "config": {"workload": f"lse_merge G={G} rows={rows} H={H} R={R}",
                   "l2": "flushed between steps (256 MiB write, then read back)"},
        "roofline": {"bound": "hbm", "kernel": "lse_merge_kernel", "achieved": round(achieved, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "traffic": None, "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs, burst)"},
        "gpu_launches": args.steps, "clocks": clk.summary(),
    }


# ---------------------------------------------------------------- oracle timing
# Oracle rows per sample: the cpu_baseline of our arm (about 5-20 s of fp64
# work on 16 cores) and each step of the reference arm (a few seconds at most).
CPU_ROWS = {"tiny": 2, "per_shard": 16, "full_head": 4, "fp8_small": 8, "long_multirow": 2}
REF_ROWS = {"tiny": 2, "per_shard": 4, "full_head": 1, "fp8_small": 4, "long_multirow": 1}


def oracle_sample(w, n_rows: int):
    """Time the oracle (as it stands) on the first n_rows rows of workload w:
    the cache write of the batch's new tokens and the decode of those rows.
    Fewer rows than a sequence holds sample that many of its first sequence's
    rows (each row attends to the whole sequence on its own)."""
    import oracle
    n_rows = max(1, min(n_rows, w.num_rows))
    if n_rows <= w.rows_per_seq:
        n_seqs = 1
    else:
        n_seqs = (n_rows + w.rows_per_seq - 1) // w.rows_per_seq
        n_rows = n_seqs * w.rows_per_seq
    cache = w.kv_cache.copy()
    t0 = time.perf_counter()
    oracle.cache_write(w.kv_c, w.k_pe, w.slot_mapping, cache, block_size=w.block_size,
                       kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim,
                       kv_is_fp8=w.kv_fp8, scale=w.kv_scale)
    oracle.decode(w.q[:n_rows], cache, w.block_table[:n_seqs], w.seq_lens[:n_seqs],
                  block_size=w.block_size, kv_lora_rank=w.kv_lora_rank, rope_dim=w.rope_dim,
                  sm_scale=w.sm_scale, kv_is_fp8=w.kv_fp8, kv_scale=w.kv_scale)
    dt = time.perf_counter() - t0
    kv = int(w.seq_lens[:n_seqs].astype(np.int64).sum()) * w.head_dim * w.kv_elem_bytes()
    return kv / dt / 1e9, dt, n_rows, oracle.max_threads()


def cpu_baseline(workload: str, n_rows):
    from mla_paged_kv_concat_gb300 import workloads as W
    w = W.make(workload)
    n_rows = CPU_ROWS.get(workload, 4) if n_rows is None else n_rows
    gbs, dt, n, cores = oracle_sample(w, n_rows)
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{workload}: cache write of all {w.slot_mapping.size} new tokens + "
                      f"fp64 decode of rows 0..{n - 1} (all {w.num_heads} heads), "
                      f"{dt:.2f} s wall"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from mla_paged_kv_concat_gb300 import workloads as W
    w = W.make(args.workload)
    n_rows = REF_ROWS.get(args.workload, 4) if args.ref_rows is None else args.ref_rows
    vals, dts = [], []
    for i in range(args.warmup + args.steps):
        gbs, dt, n, cores = oracle_sample(w, n_rows)
        if i >= args.warmup:
            vals.append(gbs)
            dts.append(dt)
    value = float(np.mean(vals))
    return {
        "impl": "reference",
        "metric": "MLA decode KV GB/s & TFLOPS as % of roofline; decode rows/s at 1 GB300",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * float(np.mean(dts)), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.workload, "rows_sampled": n},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{args.workload}: rows 0..{n - 1} + the cache write, "
                                   f"per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def relaunch_under_torchrun(n: int) -> None:
    """`--gpus N` without a launcher: start N ranks of this same command under
    torch.distributed.run (one node, rendezvous on 127.0.0.1) and exit with
    their status."""
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr=127.0.0.1", f"--master-port={port}",
           os.path.abspath(__file__)] + sys.argv[1:]
    sys.exit(subprocess.call(cmd))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_multirow",
                    help="the headline workload (default: the largest one-GPU batch)")
    ap.add_argument("--no-configs", action="store_true",
                    help="measure the headline workload only (no configs list)")
    ap.add_argument("--deterministic", action="store_true", help="num_kv_splits = 1")
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 mma.sync, 2 tcgen05")
    ap.add_argument("--cpu-rows", type=int, default=None,
                    help="rows of the workload in the oracle's cpu_baseline sample")
    ap.add_argument("--ref-rows", type=int, default=None,
                    help="rows per step in the --impl reference sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--api", choices=["plan", "calls"], default="plan",
                    help="plan: one prepared mla_plan_run per step; calls: the per-stage "
                         "entry points (mla_cache_write, mla_decode_splitkv, mla_decode_merge)")
    ap.add_argument("--fused-write", action="store_true",
                    help="the step's write also does RMSNorm of kv_c and the rotary embedding")
    ap.add_argument("--op", choices=["decode", "lse_merge"], default="decode",
                    help="lse_merge: time the cross-shard merge alone (one GPU)")
    ap.add_argument("--parts", type=int, default=8, help="--op lse_merge: shards G")
    ap.add_argument("--merge-rows", type=int, default=64, help="--op lse_merge: rows")
    ap.add_argument("--merge-heads", type=int, default=128, help="--op lse_merge: heads")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        relaunch_under_torchrun(args.gpus)
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.op == "lse_merge":
        if rank == 0 and args.impl == "ours":
            print(json.dumps(run_lse_merge(args)), flush=True)
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_ours(args, rank, world, local_rank)
    if not args.no_configs:
        # every other workload, one record each (replicas: each rank runs its
        # own; rank 0 reports)
        import torch
        records = []
        for wl, det in OTHER_CONFIGS:
            if wl == args.workload and det == args.deterministic:
                continue
            torch.cuda.empty_cache()
            records.append(run_ours(args, rank, world, local_rank, workload=wl,
                                    deterministic=det, light=True))
        if line is not None:
            line["configs"] = records
    if line is not None:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_rows)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
