#!/usr/bin/env python3
"""Benchmark of the sparse MLA (DeepSeek Sparse Attention) forward on GB300.

Workload: causal prefill, 4096 query tokens x 128 heads over s_kv = 8192 latent
rows, topk = 2048 indices per token of which 102 are -1 (n_valid = 1946),
Q/KV ~ N(0,1) bf16, sm_scale = 1/sqrt(576).  One step = one forward call over
the whole batch (counting/scheduling kernel, attention kernel, split-token merge).

Prints ONE JSON line (rank 0).  FLOPs per token = 2 * h_q * n_valid * (576 + 512);
``value`` is whole-job TFLOP/s with inputs resident in HBM; ``e2e`` is the same
metric through the public host-buffer entry point dsa_sparse_attn_fwd_host
(pinned host buffers; H2D of the inputs and D2H of out/lse inside every timed
step, pipelined by token chunks of ``--e2e-chunk``); ``roofline`` is the attention kernel
alone (CUDA events recorded around it inside the library call) against the
bound that dominates max(FLOPs / bf16 peak, algorithmic bytes / HBM peak), the
algorithmic bytes being the gathered KV rows plus Q, out, lse and indices;
``cpu_baseline`` is the float64 CPU oracle on a time-bounded sample of the same
tokens.  ``--workload`` selects one of the other input shapes for measurement.

``--impl reference`` times that CPU oracle (the only reference implementation
of this path) on the host cores instead, each step a bounded sample of tokens.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "sparse MLA fwd TFLOPS & % of roofline (h_q=128, topk=2048, 1×GB300)"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 2 * 135_528_448  # twice the GB300 L2


def _flops(indices: torch.Tensor, s_kv: int, h_q: int) -> float:
    nv = ((indices >= 0) & (indices < s_kv)).sum().item()
    return 2.0 * h_q * nv * (576 + 512)


def _alg_bytes(wl) -> float:
    """Algorithmic bytes of one forward: gathered KV rows + Q + out + lse + indices."""
    nv = ((wl.indices >= 0) & (wl.indices < wl.s_kv)).sum().item()
    row = {"bf16": 1152, "fp8": 656, "fp4": 448}[wl.kv_format]
    return nv * row + wl.s_q * wl.h_q * (576 * 2 + 512 * 2 + 4) + wl.indices.numel() * 4


def _compulsory_bytes(wl) -> float:
    """Bytes that must cross HBM once: every distinct KV row that some token selects, Q, out, lse, indices."""
    idx = wl.indices.flatten()
    ok = (idx >= 0) & (idx < wl.s_kv)
    if wl.meta.get("paged"):
        uniq = wl.kv.shape[0]  # upper bound: the whole pool (the translation is not redone here)
    else:
        uniq = int(torch.unique(idx[ok]).numel())
    row = {"bf16": 1152, "fp8": 656, "fp4": 448}[wl.kv_format]
    return uniq * row + wl.s_q * wl.h_q * (576 * 2 + 512 * 2 + 4) + wl.indices.numel() * 4


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json, bf16 burst)"
    return 1900.0, 6800.0, "fallback (1.9 PFLOP/s bf16, 6.8 TB/s)"


class ClockSampler:
    """nvidia-smi samples every 20 ms while the timed region runs, plus the last sample before it (a region
    shorter than the interval is bracketed by the samples just before and after)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "20", "-i", str(gpu_index)], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None

    def _rows(self):
        self.f.flush()
        with open(self.f.name) as g:
            return [r for r in g.read().strip().splitlines() if r.count(",") >= 8]

    def wait_rows(self, n: int, timeout: float = 3.0) -> None:
        """Block until the sampler has written at least n rows (or timeout)."""
        if self.proc is None:
            return
        t0 = time.perf_counter()
        while len(self._rows()) < n and time.perf_counter() - t0 < timeout:
            time.sleep(0.005)

    def mark(self) -> int:
        return len(self._rows()) if self.proc is not None else 0

    def stop(self, first: int = 0):
        """Rows from index `first` on (the caller marks the last row written before its timed region; for a
        region shorter than the sampling interval the rows just before and after bracket it)."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 8][max(0, first - 1):]
        os.unlink(self.f.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


KERNEL_SOURCES = ("dsa_fwd_impl.cuh", "ptx.cuh", "dsa_internal.h", "dsa_fwd.cu", "dsa_fwd_fp8.cu", "dsa_fwd_fp4.cu")


def _kernel_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "sparse_mla_attention_dsa_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _measured_traffic(workload: str):
    """DRAM bytes per launch of the attention kernel from the ncu capture recorded in profiles/, or None when
    there is none for this workload or the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    w = rec.get("workloads", {}).get(workload)
    if w is None or w.get("kernel_sources_sha256", rec.get("kernel_sources_sha256")) != _kernel_sources_sha256():
        return None  # a capture of other kernel sources does not describe the compiled kernel
    return float(w["dram_read_bytes"] + w["dram_write_bytes"])


def cpu_oracle_sample(wl, seconds: float, start_token: int = 0):
    """Run the float64 oracle token by token for about `seconds`; returns (flops, elapsed, n_tokens)."""
    from oracle import dsa_oracle as O
    qb = wl.q.contiguous().view(torch.int16).numpy().view(np.uint16)
    kvr = wl.kv.contiguous().view(torch.int16).numpy().view(np.uint16) if wl.kv_format == "bf16" else wl.kv.numpy()
    idx = wl.indices.numpy()
    if wl.meta.get("paged"):  # the oracle's own translation of logical positions to pool rows
        from oracle import paged as PG
        idx = PG.logical_to_rows(idx, wl.meta["seq_of_token"].numpy(), wl.meta["block_table"].numpy(),
                                 wl.meta["page_size"], wl.kv.shape[0])
    proj = wl.meta.get("w_o") is not None
    if proj:  # the output projection with residual follows the forward
        from oracle import out_proj as OP
        wb = wl.meta["w_o"].contiguous().view(torch.int16).numpy().view(np.uint16)
        xb = wl.meta["x"].contiguous().view(torch.int16).numpy().view(np.uint16)
    flops, n, t0 = 0.0, 0, time.perf_counter()
    t = start_token
    while True:
        o, _ = O.sparse_mla_fwd_sampled(qb, kvr, wl.kv_format, idx, wl.sm_scale, [t % wl.s_q])
        row = idx[t % wl.s_q]
        flops += 2.0 * wl.h_q * int(((row >= 0) & (row < wl.s_kv)).sum()) * 1088
        if proj:
            OP.out_proj_f64(o, wb, xb[t % wl.s_q:t % wl.s_q + 1])
            flops += 2.0 * wb.shape[0] * wb.shape[1]
        n += 1
        t += 1
        if time.perf_counter() - t0 >= seconds or n >= wl.s_q:
            break
    return flops, time.perf_counter() - t0, n


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def max_over_ranks(values, world: int, dev) -> list:
    """Element-wise maximum of per-rank timings over all ranks (the slowest rank sets the job's time); the
    identity for one rank.  Needs an initialised process group when world > 1."""
    if world <= 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def run_reference(args, rank: int, world: int):
    """The CPU oracle as it stands, on this host's cores, each step a bounded token sample (rank 0 only)."""
    from sparse_mla_attention_dsa_gb300 import workloads as W
    if rank != 0:
        return
    wl = W.WORKLOADS[args.workload]() if args.workload != "prefill_causal" else W.prefill_causal()
    for w in range(args.warmup):
        cpu_oracle_sample(wl, 0.0, start_token=w)
    times, flops_all, ntok = [], 0.0, 0
    tok = args.warmup
    for _ in range(args.steps):
        f, dt, n = cpu_oracle_sample(wl, args.ref_step_seconds, start_token=tok)
        tok += n
        times.append(dt)
        flops_all += f
        ntok += n
    total = sum(times)
    value = flops_all / total / 1e12
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": args.workload, "s_q": wl.s_q, "h_q": wl.h_q, "s_kv": wl.s_kv, "topk": wl.topk,
                       "n_valid_per_token": round(flops_all / max(ntok, 1) / (2 * wl.h_q * 1088), 1),
                       "step": f"~{args.ref_step_seconds:g} s token sample"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                             "sample": f"{ntok} tokens of {args.workload} over {args.steps} steps (numpy float64, "
                                       f"BLAS threads = host cores)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gb300(args, rank: int, world: int, local_rank: int):
    from sparse_mla_attention_dsa_gb300 import api, build
    from sparse_mla_attention_dsa_gb300 import workloads as W
    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if args.workload == "prefill_causal":
        wl = W.prefill_causal(seed=2 + rank, s_q=args.s_q, s_kv=args.s_q + 4096)
    else:
        wl = W.WORKLOADS[args.workload]()
    flops = _flops(wl.indices, wl.s_kv, wl.h_q)
    fwd = {"bf16": api.dsa_sparse_attn_fwd, "fp8": api.dsa_sparse_attn_fwd_fp8kv,
           "fp4": api.dsa_sparse_attn_fwd_fp4kv}[wl.kv_format]
    fmt = {"bf16": api.KV_BF16, "fp8": api.KV_FP8, "fp4": api.KV_FP4}[wl.kv_format]
    q, kv, idx = wl.q.to(dev), wl.kv.to(dev), wl.indices.to(dev)
    out = torch.empty((wl.s_q, wl.h_q, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((wl.s_q, wl.h_q), dtype=torch.float32, device=dev)
    ws = torch.empty(api.dsa_sparse_attn_fwd_workspace_size(wl.s_q, wl.h_q, wl.topk, fmt),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    if wl.meta.get("paged"):  # logical positions through a block table over a page pool
        seq, table = wl.meta["seq_of_token"].to(dev), wl.meta["block_table"].to(dev)

        def fwd(q, kv, idx, sm_scale, out, lse, workspace):
            api.dsa_sparse_attn_fwd_paged(q, kv, idx, seq, table, wl.meta["page_size"], sm_scale, out=out, lse=lse,
                                          workspace=workspace)

    proj, pflops = wl.meta.get("w_o") is not None, 0.0
    if proj:  # forward, then y = out . W_o + x through the fused entry point
        w_o, xres = wl.meta["w_o"].to(dev), wl.meta["x"].to(dev)
        y = torch.empty_like(xres)
        ws = torch.empty(api.dsa_sparse_attn_fwd_oproj_workspace_size(wl.s_q, wl.h_q, wl.topk, fmt),
                         dtype=torch.uint8, device=dev)
        pws = torch.empty(api.dsa_out_proj_workspace_size(), dtype=torch.uint8, device=dev)
        pflops = 2.0 * wl.s_q * w_o.shape[0] * w_o.shape[1]

        def fwd(q, kv, idx, sm_scale, out, lse, workspace):
            api.dsa_sparse_attn_fwd_oproj(q, kv, idx, sm_scale, w_o, xres, kv_format=fmt, out=out, lse=lse, y=y,
                                          workspace=workspace)

    def step():
        fwd(q, kv, idx, wl.sm_scale, out=out, lse=lse, workspace=ws)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    api.dsa_read_device_status(ws)
    torch.cuda.synchronize()

    # ---- device-resident timed region (per-step events; L2 flushed between steps, outside the events)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in kev:  # materialise the events before handing them to the library
        a.record(stream)
        b.record(stream)
    sampler = ClockSampler(local_rank)
    sampler.wait_rows(1)  # sampling runs before the region starts
    first_row = sampler.mark()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for i in range(K):
        flush.zero_()
        api.dsa_set_timing_events(kev[i][0], kev[i][1])
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    api.dsa_set_timing_events()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    sampler.wait_rows(first_row + 1)  # at least one sample at or after the region's end
    clocks = sampler.stop(first_row)
    api.dsa_read_device_status(ws)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    kern_ms = [a.elapsed_time(b) for a, b in kev]
    proj_ms = None
    # the same steps with the L2 left warm (no flush between them), for reference
    wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        wev[i][0].record(stream)
        step()
        wev[i][1].record(stream)
    torch.cuda.synchronize()
    warm_ms = max_over_ranks([sum(a.elapsed_time(b) for a, b in wev) / K], world, dev)[0]
    if proj:  # the projection GEMM alone, same flush discipline
        pe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            flush.zero_()
            pe[i][0].record(stream)
            api.dsa_out_proj(out, w_o, xres, y=y, workspace=pws)
            pe[i][1].record(stream)
        torch.cuda.synchronize()
        proj_ms = sum(a.elapsed_time(b) for a, b in pe) / K
    ms = sum(step_ms) / K
    kms = sum(kern_ms) / K
    ms, kms = max_over_ranks([ms, kms], world, dev)
    if proj_ms is not None:
        proj_ms = max_over_ranks([proj_ms], world, dev)[0]

    # ---- end to end through the public API from pinned host buffers
    e2e_ms = float('nan')
    if not args.skip_e2e:
        e2e_ms = _e2e(args, wl, q, kv, idx, out, lse, step, stream, world, dev,
                      {"x": xres, "y": y} if proj else None)

    if rank != 0:
        return
    return _report(args, wl, flops, ms, kms, e2e_ms, clocks, world, proj_ms, pflops, warm_ms)


def _e2e(args, wl, q, kv, idx, out, lse, step, stream, world, dev, extra=None):
    qh, kvh, idxh = wl.q.pin_memory(), wl.kv.pin_memory(), wl.indices.pin_memory()
    outh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lseh = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

    if wl.meta.get("w_o") is not None:
        xh = wl.meta["x"].pin_memory()
        yh = torch.empty(xh.shape, dtype=xh.dtype).pin_memory()

        xd, yd = extra["x"], extra["y"]

        def e2e_step():  # inputs and the residual in, y and lse out; W_o stays resident like model weights
            q.copy_(qh, non_blocking=True)
            kv.copy_(kvh, non_blocking=True)
            idx.copy_(idxh, non_blocking=True)
            xd.copy_(xh, non_blocking=True)
            step()
            yh.copy_(yd, non_blocking=True)
            lseh.copy_(lse, non_blocking=True)
    elif wl.meta.get("paged"):
        def e2e_step():  # the paged entry point takes device buffers: copies around it on one stream
            q.copy_(qh, non_blocking=True)
            kv.copy_(kvh, non_blocking=True)
            idx.copy_(idxh, non_blocking=True)
            step()
            outh.copy_(out, non_blocking=True)
            lseh.copy_(lse, non_blocking=True)
    else:
        from sparse_mla_attention_dsa_gb300 import api
        fmt = {"bf16": api.KV_BF16, "fp8": api.KV_FP8, "fp4": api.KV_FP4}[wl.kv_format]
        chunk = min(args.e2e_chunk, wl.s_q)
        buf = torch.empty(api.dsa_sparse_attn_fwd_host_device_bytes(fmt, wl.s_q, wl.h_q, wl.s_kv, wl.topk, chunk),
                          dtype=torch.uint8, device=dev)

        def e2e_step():  # host buffers in and out; the call pipelines token chunks and returns when done
            api.dsa_sparse_attn_fwd_host(qh, kvh, idxh, wl.sm_scale, kv_format=fmt, out=outh, lse=lseh,
                                         device_buffer=buf, chunk_tokens=chunk, stream=stream)

    for _ in range(max(2, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    KE = max(3, min(args.steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(KE):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / KE], world, dev)[0]

    return e2e_ms


def _report(args, wl, flops, ms, kms, e2e_ms, clocks, world, proj_ms=None, pflops=0.0, warm_ms=None):
    """`flops` are the attention's (the roofline's kernel); `pflops` those of the output projection, if any."""
    from sparse_mla_attention_dsa_gb300 import api
    K = args.steps
    proj = proj_ms is not None
    h2d = wl.q.numel() * 2 + wl.kv.numel() * wl.kv.element_size() + wl.indices.numel() * 4
    d2h = wl.s_q * wl.h_q * (512 * 2 + 4)
    if proj:  # residual in; y and lse out (the attention output stays on the device)
        h2d += wl.meta["x"].numel() * 2
        d2h = wl.s_q * wl.h_q * 4 + wl.meta["x"].numel() * 2
    peak_tf, hbm_gbs, peak_src = _peaks()
    abytes = _alg_bytes(wl)
    t_flops, t_bytes = flops / (peak_tf * 1e12), abytes / (hbm_gbs * 1e9)
    tf_achieved = flops / (kms * 1e-3) / 1e12
    gbs_achieved = abytes / (kms * 1e-3) / 1e9
    if t_bytes >= t_flops:
        roof = {"bound": "hbm", "achieved": gbs_achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": gbs_achieved / hbm_gbs}
    else:
        roof = {"bound": "tensor", "achieved": tf_achieved, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": tf_achieved / peak_tf}
    traffic = args.traffic if args.traffic is not None else _measured_traffic(args.workload)
    if args.s_q is not None and args.workload == "prefill_causal" and args.s_q != 4096 and args.traffic is None:
        traffic = None  # the recorded capture is of the full-size workload
    roof.update({"traffic": traffic, "alg_bytes": abytes, "alg_flops": flops, "peak_source": peak_src,
                 "kernel": "dsa_fwd_kernel<%d>" % {"bf16": 0, "fp8": 1, "fp4": 2}[wl.kv_format],
                 "kernel_ms": kms, "tensor_frac": tf_achieved / peak_tf, "hbm_frac": gbs_achieved / hbm_gbs,
                 "roofline_ms": 1e3 * max(t_flops, t_bytes)})
    cbytes = _compulsory_bytes(wl)
    roof.update({"compulsory_bytes": cbytes, "compulsory_ms": 1e3 * cbytes / (hbm_gbs * 1e9)})
    total = flops + pflops
    value = world * total / (ms * 1e-3) / 1e12
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": args.workload, "s_q": wl.s_q, "h_q": wl.h_q, "s_kv": wl.s_kv, "topk": wl.topk,
                       "n_valid_per_token": round(flops / (2 * wl.h_q * 1088 * wl.s_q), 1), "b_topk": 128,
                       "kv": wl.kv_format,
                       "l2": "flushed before every step (270 MB write, outside the step events)",
                       "parallelism": f"replicas x{world} (tokens are independent)"},
            "roofline": roof,
            "e2e": None if args.skip_e2e else {"value": world * total / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                                               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                                               "ms_per_step": e2e_ms,
                                               "api": "dsa_sparse_attn_fwd_oproj + torch copies" if proj
                                               else "dsa_sparse_attn_fwd_paged + torch copies"
                                               if wl.meta.get("paged") else "dsa_sparse_attn_fwd_host",
                                               "chunk_tokens": None if (proj or wl.meta.get("paged"))
                                               else min(args.e2e_chunk, wl.s_q)},
            "gpu_launches": K * api.dsa_kernels_per_call(),
            "clocks": clocks}
    if warm_ms is not None:
        line["warm_l2"] = {"ms_per_step": warm_ms, "value": world * total / (warm_ms * 1e-3) / 1e12, "unit": UNIT,
                           "note": "the same steps without the L2 flush between them (not the headline)"}
    if proj:
        line["config"]["d_model"] = wl.meta["d_model"]
        line["config"]["step"] = "forward, then y = out . W_o + x (cuBLASLt GEMM, not counted in gpu_launches)"
        line["out_proj"] = {"ms": proj_ms, "tflops": pflops / (proj_ms * 1e-3) / 1e12,
                            "tensor_frac": pflops / (proj_ms * 1e-3) / 1e12 / peak_tf, "flops": pflops,
                            "gemm": f"bf16 M={wl.s_q} K={wl.h_q * 512} N={wl.meta['d_model']}, fp32 accumulate"}
    if not args.no_cpu_baseline:
        f, dt, n = cpu_oracle_sample(wl, args.cpu_seconds)
        line["cpu_baseline"] = {"value": f / dt / 1e12, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                                "sample": f"{n} tokens of {args.workload} ({dt:.1f} s, numpy float64, "
                                          f"BLAS threads = host cores)"}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=2.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--s-q", type=int, default=4096, help="query tokens (4096 = the benchmark workload)")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--e2e-chunk", type=int, default=512,
                    help="query tokens per chunk of the host-buffer pipeline timed as e2e")
    ap.add_argument("--workload", default="prefill_causal",
                    choices=["prefill_causal", "decode_bf16", "decode_fp8", "long_prefill", "decode_paged",
                             "decode_fp4", "prefill_oproj", "tiny"])
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per attention-kernel launch from an ncu capture (null when not given)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_gb300(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
