"""Benchmark: paged MLA decode step on GB300 (one JSON line on rank 0).

A step is one pass of the hot path over one batch: the cache write of the step's new
tokens (B * s_q rows) followed by mla_decode (split scheduler, split-KV decode, LSE
combine). The default workload is the DeepSeek-V3-shaped batch (B=512, s_q=1, H=128,
page 128, seq_lens ~ U[1000, 2000], bf16 cache); --config / --kv / --s_q pick another.

per_config  (N=1) the decode kernel and call timed on each of the other workloads: the
           16-head ragged batch (bf16 and FP8), the 128-head batch with the FP8 cache and
           the long-context FP8 batch at s_q = 1 and 4, each with its roofline

value      decode TFLOP/s of the whole job (algorithmic flops 2*(576+512) per visible
           (row, head, key), summed over ranks) with inputs resident in HBM
e2e        the same metric through the public API with pinned host buffers: every step
           copies q, the new latent/rope rows, slot mapping, block table and seq_lens in
           (one pinned staging buffer, one copy) and reads out and lse back (one copy)
           inside the timed region. Steps are pipelined over two buffer sets: step k's input
           copy (one copy stream) and step k-1's result copy (another) overlap step k-1's
           and step k's decode; serial_ms_per_step is the same with everything on one stream
roofline   the decode kernel (CUDA events the library records on its stream around the
           kernel's launch, in a second pass of the same K steps) against the measured
           HBM copy bandwidth or bf16 tensor peak; call_frac is the same for the whole
           decode call (scheduler + decode + combine) of the timed region
cpu_baseline  the float64 oracle on a bounded sample of the same workload

--impl reference times the oracle itself (the only reference this method has) as the
reference arm. Multi-GPU: one process per GPU (torchrun), each rank an independent
replica with its own sequences (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode TFLOP/s and KV GB/s (bf16 & FP8 KV) at 1 GB300; % of roofline"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--kv", default=None, choices=[None, "bf16", "fp8"])
    ap.add_argument("--s_q", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="the workload's first B sequences only (smaller cases for profiling)")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def make_case(args, rank: int):
    from mla_paged_decode_02_gb300 import synth
    kv = None if args.kv is None else (synth.KV_BF16 if args.kv == "bf16" else synth.KV_FP8_E4M3)
    if args.batch is not None:
        # the same length distribution, seed and shape with a smaller batch
        kw = dict(synth.CONFIGS[args.config])
        name = synth.config_name(args.config, kv, args.s_q) + f"_b{args.batch}"
        kw.pop("name")
        kw["B"] = args.batch
        if isinstance(kw["seq_lens"], list):
            kw["seq_lens"] = kw["seq_lens"][:args.batch]
        if kv is not None:
            kw["kv_dtype"] = kv
        if args.s_q is not None:
            kw["s_q"] = args.s_q
        return synth.make_case(seed=synth.SEED_OF[args.config] + 7919 * rank, name=name, **kw)
    case = synth.make_config(args.config, kv_dtype=kv, s_q=args.s_q)
    if rank:
        kw = dict(synth.CONFIGS[args.config])
        kw.pop("name")
        if kv is not None:
            kw["kv_dtype"] = kv
        if args.s_q is not None:
            kw["s_q"] = args.s_q
        case = synth.make_case(seed=synth.SEED_OF[args.config] + 7919 * rank, name=case.name, **kw)
    return case


def algorithmic(case):
    """Algorithmic flops and bytes of one decode call: 2*(576+512) flops per visible
    (row, head, key); every cache row read once; q read once; out and lse written once."""
    tot = 0
    for L in case.seq_lens:
        for i in range(case.s_q):
            tot += (int(L) - case.s_q + 1 + i) if case.causal else int(L)
    flops = 2.0 * (576 + 512) * case.H * tot
    elem = 2 if case.kv_dtype == 0 else 1
    kv_bytes = float(np.sum(case.seq_lens.astype(np.int64))) * 576 * elem
    q_bytes = case.B * case.s_q * case.H * 576 * 2.0
    out_bytes = case.B * case.s_q * case.H * (512 * 2 + 4.0)
    return flops, kv_bytes, q_bytes, out_bytes


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def _code_only(text: str) -> str:
    """C/CUDA source with comments removed and whitespace collapsed (string literals kept),
    so that an edit of comments alone does not change the hash of the kernel code."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the code (not the comments) of every kernel source file."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_paged_decode_02_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(f.encode() + b"\0")
        h.update(_code_only(open(os.path.join(csrc, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """dram bytes per decode launch from the committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("source_hash") != kernel_source_hash():
        return None
    e = d.get("workloads", {}).get(workload)
    return None if e is None else float(e["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, enabled: bool):
        self.proc = None
        self.index = index
        if enabled:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                     "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except (OSError, ValueError):
                self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def roofline(case, kern_ms, flops, kv_bytes, q_bytes):
    """The decode kernel's roofline: the slower of the flops at the bf16 tensor peak and the
    KV + Q bytes at the HBM copy bandwidth (both measured on this GPU model). With the FP8
    cache the MMAs are E4M3 (twice the bf16 rate) but take q and P as two E4M3 terms each,
    so the algorithmic flops at the bf16 peak equal the issued flops at the E4M3 peak."""
    peaks, peak_kind = load_peaks()
    t = kern_ms * 1e-3
    hbm_t = (kv_bytes + q_bytes) / (peaks["hbm_gbs"] * 1e9)
    tc_t = flops / (peaks["bf16_tflops"] * 1e12)
    if hbm_t >= tc_t:
        roof = {"bound": "hbm", "achieved": (kv_bytes + q_bytes) / t / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops / t / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = ncu_traffic(case.name)
    roof["peak_source"] = f"{peak_kind} ({'hbm_gbs' if roof['bound'] == 'hbm' else 'bf16_tflops'})"
    roof["t_roof_us"] = max(hbm_t, tc_t) * 1e6
    roof["decode_kernel_us"] = kern_ms * 1e3
    return roof, max(hbm_t, tc_t)


PER_CONFIG = [(2, None, None), (3, None, None), (4, "bf16", None), (4, "fp8", None), (5, None, 1), (5, None, 4)]


def measure_config(cfg, kv, s_q, steps, warmup, device):
    """Decode kernel and decode call of one workload (inputs resident, L2 flushed between
    calls when the cache is smaller than three times L2): CUDA events on the stream."""
    import torch
    from mla_paged_decode_02_gb300 import api, synth
    from mla_paged_decode_02_gb300.workload import DeviceWorkload
    kvd = None if kv is None else (synth.KV_BF16 if kv == "bf16" else synth.KV_FP8_E4M3)
    case = synth.make_config(cfg, kv_dtype=kvd, s_q=s_q)
    g = DeviceWorkload(case, device=device)
    flops, kv_bytes, q_bytes, _ = algorithmic(case)
    stream = torch.cuda.current_stream()
    out = torch.empty((case.B, case.s_q, case.H, 512), dtype=torch.bfloat16, device=device)
    lse = torch.empty((case.B, case.s_q, case.H), dtype=torch.float32, device=device)
    flush = torch.empty(int(512e6), dtype=torch.uint8, device=device) if kv_bytes < 3 * 129e6 else None

    def call():
        g.decode(out=out, lse=lse)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    st, bits = api.decode_check(g.workspace)
    if st != 0:
        raise RuntimeError(f"{case.name}: device error word {bits:#x}")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for k in range(steps):
        if flush is not None:
            flush.fill_(k & 0xFF)
        ev[k][0].record(stream)
        call()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    call_ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    for k in range(steps):
        if flush is not None:
            flush.fill_(k & 0xFF)
        if k == 0:
            api.profile_begin(steps)
        call()
    kern_total, n = api.profile_end()
    kern_ms = kern_total / n
    roof, t_roof = roofline(case, kern_ms, flops, kv_bytes, q_bytes)
    roof["decode_call_us"] = call_ms * 1e3
    roof["call_frac"] = t_roof / (call_ms * 1e-3)
    res = {"workload": case.name, "B": case.B, "s_q": case.s_q, "H": case.H, "page_size": case.page_size,
           "kv": "fp8_e4m3" if case.kv_dtype else "bf16", "tokens": int(case.seq_lens.sum()),
           "decode_tflops": round(flops / (kern_ms * 1e-3) / 1e12, 3),
           "kv_gbs": round(kv_bytes / (kern_ms * 1e-3) / 1e9, 1),
           "l2": "flushed between calls" if flush is not None else "inputs larger than L2",
           "roofline": {k: (round(v, 4) if isinstance(v, float) else v) for k, v in roof.items()}}
    del g, flush, out, lse
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, local_rank, world):
    import torch
    from mla_paged_decode_02_gb300 import api
    from mla_paged_decode_02_gb300.workload import DeviceWorkload as GpuCase, bits_to_torch_bf16

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    case = make_case(args, rank)
    g = GpuCase(case, device=device)
    flops, kv_bytes, q_bytes, out_bytes = algorithmic(case)
    stream = torch.cuda.current_stream()

    # the step's new tokens: each sequence's last s_q rows (re-written with the same values)
    step_idx = case.step_tokens()
    lat_d = bits_to_torch_bf16(case.latent_bits[step_idx], device)
    rope_d = bits_to_torch_bf16(case.rope_bits[step_idx], device)
    slots_d = torch.from_numpy(case.slot_mapping[step_idx]).to(device)
    out = torch.empty((case.B, case.s_q, case.H, 512), dtype=torch.bfloat16, device=device)
    lse = torch.empty((case.B, case.s_q, case.H), dtype=torch.float32, device=device)

    def step():
        api.cache_write(lat_d, rope_d, slots_d, g.cache, g.kv_scale)
        api.decode(g.q, g.cache, g.block_table, g.seq_lens, case.softmax_scale, g.kv_scale,
                   max_seq_len=case.max_seq_len, causal=case.causal, out=out, lse=lse,
                   workspace=g.workspace)

    l2_flush = kv_bytes < 3 * 129e6
    flush_buf = torch.empty(int(512e6), dtype=torch.uint8, device=device) if l2_flush else None

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, bits = api.decode_check(g.workspace)
    if st != 0:
        raise RuntimeError(f"device error word after warm-up: status {st} bits {bits:#x}")

    # ---- device-resident timing: K steps, also the decode call alone per step.
    # nvidia-smi needs ~0.3 s to start sampling, longer than K steps take, so the same
    # step loop runs for ~0.5 s before and after the timed region while it samples.
    clocks = ClockSampler(local_rank, not args.no_clocks)

    def soak(seconds):
        if clocks.proc is None:
            return
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            for _ in range(8):
                step()
            torch.cuda.synchronize()

    soak(0.6)
    barrier(world)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    dec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for k in range(args.steps):
        if flush_buf is not None:
            flush_buf.fill_(k & 0xFF)
        ev[k][0].record(stream)
        api.cache_write(lat_d, rope_d, slots_d, g.cache, g.kv_scale)
        dec[k][0].record(stream)
        api.decode(g.q, g.cache, g.block_table, g.seq_lens, case.softmax_scale, g.kv_scale,
                   max_seq_len=case.max_seq_len, causal=case.causal, out=out, lse=lse,
                   workspace=g.workspace)
        dec[k][1].record(stream)
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    soak(0.4)
    clk = clocks.stop()
    # ---- the decode kernel alone: the same K steps again, the library timing its launch
    for k in range(args.steps):
        if flush_buf is not None:
            flush_buf.fill_(k & 0xFF)
        if k == 0:
            api.profile_begin(args.steps)
        step()
    kern_ms_total, kern_n = api.profile_end()
    if kern_n != args.steps:
        raise RuntimeError(f"timed {kern_n} decode kernels, expected {args.steps}")
    kern_ms = kern_ms_total / kern_n
    # ---- the same step through the fused entry point (the scheduler kernel writes the new
    # rows): one launch fewer per step
    def fused_step():
        api.decode_with_cache_write(lat_d, rope_d, slots_d, g.q, g.cache, g.block_table, g.seq_lens,
                                    case.softmax_scale, g.kv_scale, max_seq_len=case.max_seq_len,
                                    causal=case.causal, out=out, lse=lse, workspace=g.workspace)

    for _ in range(args.warmup):
        fused_step()
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for k in range(args.steps):
        if flush_buf is not None:
            flush_buf.fill_(k & 0xFF)
        fev[k][0].record(stream)
        fused_step()
        fev[k][1].record(stream)
    torch.cuda.synchronize()
    st, bits = api.decode_check(g.workspace)
    if st != 0:
        raise RuntimeError(f"device error word after the fused steps: status {st} bits {bits:#x}")
    fused_ms = sum(a.elapsed_time(b) for a, b in fev) / args.steps
    step_ms = sum(a.elapsed_time(b) for a, b in ev)
    dec_ms = sum(a.elapsed_time(b) for a, b in dec) / args.steps
    step_ms_max = max_over_ranks(step_ms, world, device)
    ms_per_step = step_ms_max / args.steps
    total_flops = sum_over_ranks(flops, world, device)
    value = total_flops / (ms_per_step * 1e-3) / 1e12

    # ---- end-to-end through the public API with pinned host buffers. The step's inputs
    # (q, the new latent/rope rows, slot mapping, block table, seq_lens) sit in one pinned
    # staging buffer and go to the device in one copy; out and lse come back in one copy.
    def packed(tensors):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, n

    def views(buf, offs, like):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                for o, t in zip(offs, like)]

    ins_like = [g.q, lat_d, rope_d, slots_d, g.block_table, g.seq_lens]
    in_offs, in_bytes = packed(ins_like)
    h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(in_bytes, dtype=torch.uint8, device=device)
    for hv, t in zip(views(h_in, in_offs, ins_like), ins_like):
        hv.copy_(t.cpu())
    outs_like = [out, lse]
    out_offs, out_bytes = packed(outs_like)
    h_res = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    d_res = torch.empty(out_bytes, dtype=torch.uint8, device=device)
    h2d = sum(t.numel() * t.element_size() for t in ins_like)
    d2h = sum(t.numel() * t.element_size() for t in outs_like)

    def run_on(d_in_i, d_res_i, s):
        d_q, d_lat, d_rope, d_slots, d_bt, d_sl = views(d_in_i, in_offs, ins_like)
        d_out, d_lse = views(d_res_i, out_offs, outs_like)
        api.cache_write(d_lat, d_rope, d_slots, g.cache, g.kv_scale, stream=s)
        api.decode(d_q, g.cache, d_bt, d_sl, case.softmax_scale, g.kv_scale,
                   max_seq_len=case.max_seq_len, causal=case.causal, out=d_out, lse=d_lse,
                   workspace=g.workspace, stream=s)

    def e2e_step():                  # everything in stream order
        d_in.copy_(h_in, non_blocking=True)
        run_on(d_in, d_res, stream)
        h_res.copy_(d_res, non_blocking=True)

    # pipelined: buffer set i = k % 2; the input copy of step k waits until step k-2's
    # decode has read set i, the decode of step k until step k-2's result copy is done
    d_in2 = [d_in, torch.empty(in_bytes, dtype=torch.uint8, device=device)]
    d_res2 = [d_res, torch.empty(out_bytes, dtype=torch.uint8, device=device)]
    h_res2 = [h_res, torch.empty(out_bytes, dtype=torch.uint8).pin_memory()]
    s_h2d, s_d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in", "used", "res", "out")}

    def e2e_pipelined(K):
        for k in range(K):
            i = k & 1
            if k >= 2:
                s_h2d.wait_event(ev["used"][i])
            with torch.cuda.stream(s_h2d):
                d_in2[i].copy_(h_in, non_blocking=True)
            ev["in"][i].record(s_h2d)
            stream.wait_event(ev["in"][i])
            if k >= 2:
                stream.wait_event(ev["out"][i])
            run_on(d_in2[i], d_res2[i], stream)
            ev["used"][i].record(stream)
            ev["res"][i].record(stream)
            s_d2h.wait_event(ev["res"][i])
            with torch.cuda.stream(s_d2h):
                h_res2[i].copy_(d_res2[i], non_blocking=True)
            ev["out"][i].record(s_d2h)
        stream.wait_stream(s_h2d)
        stream.wait_stream(s_d2h)

    def timed(fn, *a):
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn(*a)
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1), world, device) / args.steps

    def check(h):
        h_out, h_lse = views(h, out_offs, outs_like)
        if not (torch.equal(h_out, out.cpu()) and torch.equal(h_lse, lse.cpu())):
            raise RuntimeError("the end-to-end result differs from the device-resident one")

    for _ in range(max(1, args.warmup)):
        e2e_step()
    e2e_serial_ms = timed(lambda: [e2e_step() for _ in range(args.steps)])
    check(h_res)
    e2e_pipelined(max(2, args.warmup))
    e2e_ms = timed(e2e_pipelined, args.steps)
    check(h_res2[(args.steps - 1) & 1])
    e2e_value = total_flops / (e2e_ms * 1e-3) / 1e12

    # ---- roofline of the decode kernel
    roof, t_roof = roofline(case, kern_ms, flops, kv_bytes, q_bytes)
    roof["kernel_timed"] = ("decode_kernel: CUDA events recorded by the library around its launch "
                            "(mla_profile_begin/end), a second pass of the same K steps")
    roof["decode_call_us"] = dec_ms * 1e3
    roof["call_frac"] = t_roof / (dec_ms * 1e-3)

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": case.name, "B": case.B, "s_q": case.s_q, "H": case.H,
                   "page_size": case.page_size, "kv": "fp8_e4m3" if case.kv_dtype else "bf16",
                   "tokens": int(case.seq_lens.sum()), "parallelism": f"dp{world} (replicas)",
                   "l2": "flushed between steps" if l2_flush else "inputs larger than L2"},
        # the decode kernel's rates (as in per_config), and the whole decode call's
        "kv_gbs": round(kv_bytes / (kern_ms * 1e-3) / 1e9, 1),
        "decode_tflops": round(flops / (kern_ms * 1e-3) / 1e12, 3),
        "call_kv_gbs": round(kv_bytes / (dec_ms * 1e-3) / 1e9, 1),
        "call_tflops": round(flops / (dec_ms * 1e-3) / 1e12, 3),
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 5),
                "how": "steps pipelined over two buffer sets and two copy streams",
                "serial_ms_per_step": round(e2e_serial_ms, 5)},
        "roofline": {k: (round(v, 4) if isinstance(v, float) else v) for k, v in roof.items()},
        "gpu_launches": 4 * args.steps,      # cache write, scheduler, decode, combine per step
        "fused_step": {"ms_per_step": round(fused_ms, 5), "launches_per_step": 3,
                       "two_call_ms_per_step": round(ms_per_step, 5), "two_call_launches_per_step": 4,
                       "how": "mla_decode_with_cache_write: extra CTAs of the scheduler's launch write the step's new rows"},
        "clocks": clk,
    }
    if world == 1 and not args.no_per_config:
        del g
        torch.cuda.empty_cache()
        from mla_paged_decode_02_gb300 import synth
        kvd = lambda kv: None if kv is None else (synth.KV_BF16 if kv == "bf16" else synth.KV_FP8_E4M3)
        line["per_config"] = [measure_config(c, kv, sq, max(args.steps, 10), max(args.warmup, 3), device)
                              for c, kv, sq in PER_CONFIG
                              if synth.config_name(c, kvd(kv), sq) != case.name]
    return line, case


def cpu_baseline(case, min_s: float = 10.0, budget_s: float = 25.0):
    """The oracle as it stands on this host's cores, over a bounded sample: sequences of
    the workload in order (all their rows), repeated from the start if one pass is shorter
    than `min_s`, stopping after `budget_s`."""
    from oracle import mla_oracle as O
    cache = O.cache_write(case.empty_cache(), case.latent_bits, case.rope_bits, case.slot_mapping,
                          case.page_size, case.kv_dtype, case.kv_scale)
    done_flops, t_used, nb = 0.0, 0.0, 0
    t_start = time.perf_counter()
    while True:
        b = nb % case.B
        rows = [(b, i, h) for i in range(case.s_q) for h in range(case.H)]
        t0 = time.perf_counter()
        O.mla_decode(case.q_bits, cache, case.block_table, case.seq_lens, case.page_size,
                     case.softmax_scale, case.kv_dtype, case.kv_scale, case.causal, rows=rows)
        t_used += time.perf_counter() - t0
        done_flops += O.flops([case.seq_lens[b]], case.s_q, case.H, case.causal)
        nb += 1
        elapsed = time.perf_counter() - t_start
        if elapsed > budget_s or (elapsed > min_s and nb % case.B == 0) or (elapsed > min_s and nb > case.B):
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": done_flops / t_used / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{nb} sequence decodes (sequences 0..{min(nb, case.B) - 1} of {case.B} of "
                      f"{case.name} in order, repeated; all s_q*H rows each), float64 numpy, {t_used:.1f} s"}


def run_reference(args, rank, world):
    """Reference arm: the float64 oracle, timed on the host cores, rank 0 only."""
    if rank != 0:
        return None
    from oracle import mla_oracle as O
    case = make_case(args, 0)
    cache = O.cache_write(case.empty_cache(), case.latent_bits, case.rope_bits, case.slot_mapping,
                          case.page_size, case.kv_dtype, case.kv_scale)
    per_step = max(1, min(case.B, 2))

    def step(k):
        bs = [(k * per_step + j) % case.B for j in range(per_step)]
        rows = [(b, i, h) for b in bs for i in range(case.s_q) for h in range(case.H)]
        O.mla_decode(case.q_bits, cache, case.block_table, case.seq_lens, case.page_size,
                     case.softmax_scale, case.kv_dtype, case.kv_scale, case.causal, rows=rows)
        return sum(O.flops([case.seq_lens[b]], case.s_q, case.H, case.causal) for b in bs)

    for k in range(args.warmup):
        step(k)
    fl, t0 = 0.0, time.perf_counter()
    for k in range(args.steps):
        fl += step(args.warmup + k)
    dt = time.perf_counter() - t0
    value = fl / dt / 1e12
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": case.name},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} sequences of {case.name} per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    rank, local_rank, world = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
    else:
        line, case = run_ours(args, rank, local_rank, world)
        if rank == 0:
            if not args.no_cpu_baseline and world == 1:
                line["cpu_baseline"] = cpu_baseline(case)
            print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
