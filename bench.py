#!/usr/bin/env python3
"""Sparse MLA decode benchmark on GB300: query-tokens/s and fraction of the roofline.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one smla_decode call over one batch of the workload (all query
tokens: gather, dequant, QK, softmax, PV, split merge), inputs resident in HBM.
L2 is flushed (a 512 MiB write) between timed steps, outside the timed
events. Under torchrun (N > 1) every rank decodes its own batch of the same
shape (independent replicas, weak scaling); the JSON line reports the total
tokens of all ranks over the slowest rank's time.

--impl reference times the float64 CPU oracle (the reference arm) on a bounded
sample of the same workload on the host cores.
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

# The CPU oracle runs with one BLAS thread, so its reported core count is exact.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

# The largest configuration the throughput target is quoted on: MTP decode, 64 requests x 4
# query tokens with independent top-k sets, 128 heads, 4k-128k contexts, per-head sink.
DEFAULT_WORKLOAD = W.WORKLOADS[3].name
METRIC = "sparse-MLA decode query-tokens/s"
E2E_VARIANTS = 4  # index sets the end-to-end loop cycles through
L2_FLUSH_BYTES = 512 << 20


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", 0.0)) or None,
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one step's launches of the
# kernel (two when the last partial wave runs as a second launch), from one ncu capture of this
# bench's own command on the named workload at full size (a one-pass metric set: nothing is
# saved or replayed), with the SHA-256 (first 16 hex digits) of that kernel's sources at capture
# time. A capture of an older kernel (the hash differs) is not reported.
TRAFFIC = {
    ("fp8_mtp_T256_H128_K2048_ctx4k-128k_sink", "decode_hg_kernel"): (429726464, "4f0b0b30b45adc0e"),
    ("fp8_T128_H128_K2048_ctx64k_sink", "decode_hg_kernel"): (231280128, "4f0b0b30b45adc0e"),
    ("fp8_T32_H64_K2048_ctx1k-32k", "decode_hg_kernel"): (51805440, "4f0b0b30b45adc0e"),
    ("fp8_T256_H16_K2048_ctx8k-128k_pad20", "decode_mma_kernel"): (333995520, "8d7176b8a678685a"),
    ("fp8tensor_mtp_T256_H128_K2048_ctx4k-128k_sink", "decode_hg_f8_kernel"): (341052160, "0889268099627afb"),
    ("store_fp8_ds_rows65536_P64_pos131072", "pack_kernel"): (111933184, "e75a497c2046fc9b"),
}
KERNEL_SOURCES = {
    "decode_hg_kernel": ("common.cuh", "kernels.h", "tcgen05.cuh", "decode_hg.cu", "tensor_maps.cu"),
    "decode_mma_kernel": ("common.cuh", "kernels.h", "decode_mma.cu"),
    "pack_kernel": ("common.cuh", "kernels.h", "cache_kernels.cu"),
    "decode_hg_f8_kernel": ("common.cuh", "kernels.h", "tcgen05.cuh", "decode_hg_f8.cu", "tensor_maps.cu"),
}


def kernel_sources_sha(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "sparse_mla_decode_smla_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    rec = TRAFFIC.get((workload, kernel))
    if rec is None or rec[1] != kernel_sources_sha(kernel):
        return None
    return rec[0]


def algorithmic_work(problem) -> tuple[int, int, int]:
    """(valid indices, KV-row bytes, FLOPs) of one decode of the whole batch."""
    valid = int((problem.topk >= 0).sum().item())
    w = problem.w
    return valid, valid * w.row_bytes, valid * w.num_heads * 2 * (576 + 512)


def workload_config(problem, valid: int, num_splits: int, world: int) -> dict:
    """The `config` object of both arms' JSON lines (identical for the same workload)."""
    w = problem.w
    return {"workload": w.name, "tokens": w.num_tokens, "heads": w.num_heads,
            "topk": w.topk, "valid_indices": valid, "kv_format": w.kv_format,
            "kv_row_bytes": w.row_bytes, "page_size": w.page_size,
            "num_pages": problem.num_pages, "sink": w.sink,
            "l2": "flushed between timed steps (512 MiB write, outside the events)",
            "num_splits": num_splits or "auto", "parallelism": f"replicas x{world}"}


def roofline(valid_bytes, flops, seconds, peaks) -> dict:
    """The bound of whichever side takes longer at its peak; peaks["tensor"] names the tensor
    peak used (the measured bf16 one unless an 8-bit path scales it)."""
    t_hbm = valid_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        achieved = valid_bytes / seconds / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                "peak_source": peaks["source"] + " hbm_gbs (burst)"}
    achieved = flops / seconds / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops"], "traffic": None,
            "peak_source": peaks["source"] + " " + peaks.get("tensor", "bf16_tflops (burst)")}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except FileNotFoundError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            self.proc.wait(timeout=5)

    def summary(self) -> dict:
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(ms_local: float, tokens_per_rank: int, world: int, device) -> tuple[float, float]:
    """(slowest rank's ms per step, whole-job query-tokens/s): every rank decodes its own
    batch of `tokens_per_rank` tokens, so the job's rate is all ranks' tokens over the
    slowest rank's step time."""
    ms_max = reduce_max(ms_local, world, device)
    return ms_max, world * tokens_per_rank / (ms_max * 1e-3)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------------------ oracle arm


def run_oracle_sample(problem, budget_s: float, wall_limit_s: float | None = None,
                      max_tokens: int | None = None, q_e4m3=None, q_scale=None):
    """Time the float64 oracle's decode, as it stands, on whole query tokens.

    The oracle's cache rows for a few requests at a time are packed first, outside the
    timed region, as the GPU side's cache is packed before its timed steps. Returns
    (tokens, seconds of oracle decode) once the decode time reaches budget_s, the wall
    time reaches wall_limit_s (default 4 x budget_s) or max_tokens tokens are done; at
    least one token is timed.
    """
    from oracle.workload_oracle import OracleCache, oracle_decode
    w = problem.w
    T = w.num_tokens
    order = list(dict.fromkeys(list(range(0, T, max(1, T // 64))) + list(range(T))))
    wall_limit = 4.0 * budget_s if wall_limit_s is None else wall_limit_s
    wall0 = time.perf_counter()
    done, el = 0, 0.0
    for i in range(0, len(order), 4):
        batch = order[i:i + 4]
        cache = OracleCache(problem, [t // w.next_n for t in batch])
        for t in batch:
            t0 = time.perf_counter()
            oracle_decode(problem, tokens=[t], cache=cache, q_e4m3=q_e4m3, q_scale=q_scale)
            el += time.perf_counter() - t0
            done += 1
            if (el >= budget_s or time.perf_counter() - wall0 >= wall_limit
                    or (max_tokens is not None and done >= max_tokens)):
                return done, el
    return done, el


def workload_from_args(args) -> W.Workload:
    w = W.BY_NAME[args.workload]
    if args.ctx_hi:
        w = W.small_variant(w, num_requests=args.requests or w.num_requests,
                            ctx_lo=min(args.ctx_lo or w.ctx_lo, args.ctx_hi), ctx_hi=args.ctx_hi,
                            topk=w.topk, tail_pad=w.tail_pad, name_suffix=f"ctx<={args.ctx_hi}")
    return w


def reference_arm(args):
    """The float64 oracle on the host cores, on the GPU arm's workload and metric.

    A step is one query token of the workload decoded by the oracle (its cache rows packed
    beforehand, untimed). Steps stop once the oracle's decode time reaches
    --ref-budget-seconds (or after --steps tokens); the line reports the steps timed.
    """
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    w = workload_from_args(args)
    problem = W.make_problem(w, device="cpu")
    if args.warmup > 0:  # one untimed token
        run_oracle_sample(problem, budget_s=0.0)
    n, el = run_oracle_sample(problem, budget_s=args.ref_budget_seconds,
                              wall_limit_s=4.0 * args.ref_budget_seconds, max_tokens=max(1, args.steps))
    value = n / el if el > 0 else float("nan")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "query-tokens/s",
            "n_gpus": 1, "steps": n, "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / n, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(problem, algorithmic_work(problem)[0], args.num_splits, world),
            "cpu_baseline": {"value": value, "unit": "query-tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{n} query tokens of {w.name}, one per step, oracle decode "
                                       f"time {el:.1f} s (cache rows packed beforehand, untimed), "
                                       f"numpy float64, 1 BLAS thread"},
            "e2e": {"value": value, "unit": "query-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------ GPU arm


def decode_launches(smla, desc, num_sms) -> int:
    """Kernel launches of one smla_decode call, from the library's own plan: one or two
    decode launches (the second when the last partial wave runs as two splits per item),
    plus the merge kernel when the split partials go through the workspace."""
    p = smla.plan_launches(desc, num_sms)
    return p.num_launches + (1 if p.merge == smla.SMLA_MERGE_KERNEL else 0)


def gpu_arm(args):
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import sparse_mla_decode_smla_gb300 as smla
    from sparse_mla_decode_smla_gb300.runner import DeviceDecode

    w = workload_from_args(args)
    problem = W.make_problem(w, seed=W.SEED_BASE + w.seed_offset + 1000 * rank, device=dev)
    dd = DeviceDecode(problem, num_splits=args.num_splits, device=dev)
    q8 = None
    if args.q_fp8:  # E4M3 q with a per-tensor scale: the FP8-operand kernel
        if w.kv_format != "fp8_tensor" or w.num_heads < 64:
            raise SystemExit("--q-fp8 needs a per-tensor FP8 workload with 64 or more heads")
        q8 = W.q_to_e4m3(problem.q).to(dev).contiguous()
        dd.q = q8
        dd.desc.q_format, dd.desc.q_scale = smla.SMLA_Q_FP8_E4M3, W.Q_SCALE_FP8
        dd.kernel_name = "decode_hg_f8_kernel"
    valid, kv_bytes, flops = algorithmic_work(problem)
    launches_per_step = decode_launches(smla, dd.desc, torch.cuda.get_device_properties(dev).multi_processor_count)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        dd.run()
    torch.cuda.synchronize(dev)

    def events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:  # create the CUDA events now, so the library can record into them
            e.record(stream)
        return evs

    starts, ends = events(args.steps), events(args.steps)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize(dev)
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            dd.run()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        wall = time.perf_counter() - wall0
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(step_ms) / len(step_ms)

    # the decode kernel alone, in a second pass of as many steps: the library records
    # these events right around the decode kernel (the split merge, when there is one,
    # follows it). Kept out of the pass above, where events between the two kernels
    # would stop the merge's launch from overlapping the decode kernel's tail.
    k_starts, k_ends = events(args.steps), events(args.steps)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        flush.fill_(float(i))
        smla.set_kernel_events(k_starts[i], k_ends[i])
        dd.run()
    smla.set_kernel_events()
    torch.cuda.synchronize(dev)
    kernel_ms = sum(s.elapsed_time(e) for s, e in zip(k_starts, k_ends)) / args.steps
    ms_max, value = aggregate(ms, w.num_tokens, world, dev)

    # End to end through the public API: pinned host inputs -> decode -> host outputs, as a
    # serving loop runs it. A step's inputs (q, top-k indices, page table) travel in one
    # host-to-device copy and its results (out, LSE) in one device-to-host copy, each side one
    # pinned buffer laid out like a device staging buffer whose views the decode call reads and
    # writes in place. Three streams overlap step i's decode with step i+1's input copy and step
    # i-1's output copy (two device buffers on each side, ordered by events). Consecutive steps
    # take different index sets over the same pool (E2E_VARIANTS of them), so no step finds the
    # previous one's rows in L2; the span timed runs from the first input copy to the last
    # output copy.
    def layout(parts):
        offs, off = [], 0
        for t in parts:
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, off

    def view(buf, off, like):
        return buf[off:off + like.numel() * like.element_size()].view(like.dtype).view(like.shape)

    in_parts = [dd.q, dd.topk, dd.page_table]
    in_offs, h2d = layout(in_parts)
    out_parts = [dd.out, dd.lse]
    out_offs, d2h = layout(out_parts)
    e2e_steps = args.e2e_steps
    variants = [dd.topk] + ([v.to(dev) for v in W.make_topk_variants(problem, E2E_VARIANTS - 1)] if e2e_steps else [])
    h_in = []
    for v in variants:
        hb = torch.empty(h2d, dtype=torch.uint8).pin_memory()
        for t, off in zip([dd.q, v, dd.page_table], in_offs):
            view(hb, off, t).copy_(t.cpu())
        h_in.append(hb)
    d_in = [torch.empty(h2d, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_out = [torch.empty(d2h, dtype=torch.uint8, device=dev) for _ in range(2)]
    h_out = [torch.empty(d2h, dtype=torch.uint8).pin_memory() for _ in range(2)]
    # the decode's views of each slot's buffers, made once
    in_views = [[view(d_in[k], off, t) for t, off in zip(in_parts, in_offs)] for k in range(2)]
    out_views = [[view(d_out[k], off, t) for t, off in zip(out_parts, out_offs)] for k in range(2)]
    s_h2d, s_cmp, s_d2h = (torch.cuda.Stream(dev) for _ in range(3))
    e_in = [torch.cuda.Event() for _ in range(2)]
    e_dec = [torch.cuda.Event() for _ in range(2)]
    e_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        k = i % 2
        with torch.cuda.stream(s_h2d):
            if i >= 2:
                s_h2d.wait_event(e_dec[k])  # decode i-2 has read this input buffer
            d_in[k].copy_(h_in[i % len(h_in)], non_blocking=True)
            e_in[k].record(s_h2d)
        s_cmp.wait_event(e_in[k])
        if i >= 2:
            s_cmp.wait_event(e_out[k])  # step i-2's results have left this output buffer
        dd.q, dd.topk, dd.page_table = in_views[k]
        dd.out, dd.lse = out_views[k]
        dd.run(s_cmp)
        e_dec[k].record(s_cmp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(e_dec[k])
            h_out[k].copy_(d_out[k], non_blocking=True)
            e_out[k].record(s_d2h)

    for i in range(3 if e2e_steps else 0):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e_ms = [float("nan")]
    copy_ms = {}
    if e2e_steps:  # each direction's copy alone, for reference
        for name, st, dst, src in (("h2d_ms", s_h2d, d_in[0], h_in[0]), ("d2h_ms", s_d2h, h_out[0], d_out[0])):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(st)
            with torch.cuda.stream(st):
                dst.copy_(src, non_blocking=True)
            c1.record(st)
            c1.synchronize()
            copy_ms[name] = c0.elapsed_time(c1)
    if e2e_steps:
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        a.record(s_h2d)
        for i in range(e2e_steps):
            e2e_step(i)
        z.record(s_d2h)
        z.synchronize()
        e_ms = [a.elapsed_time(z) / e2e_steps]
    e2e_ms = reduce_max(sum(e_ms) / len(e_ms), world, dev)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    peaks = measured_peaks()
    if args.q_fp8:  # E4M3 operands: the measured bf16 peak times the nominal fp8 / bf16 ratio of 2
        peaks = dict(peaks, bf16_tflops=2 * peaks["bf16_tflops"],
                     bf16_tflops_sustained=(2 * peaks["bf16_tflops_sustained"]
                                            if peaks.get("bf16_tflops_sustained") else None),
                     tensor="bf16_tflops (burst) x 2 (fp8)")
    rl = roofline(kv_bytes, flops, kernel_ms * 1e-3, peaks)
    rl["kernel"] = dd.kernel_name
    rl["kernel_ms"] = kernel_ms
    rl["traffic"] = args.traffic if args.traffic is not None else recorded_traffic(w.name, dd.kernel_name)
    step_rl = roofline(kv_bytes, flops, ms * 1e-3, peaks)
    line = {
        "metric": METRIC, "value": value, "unit": "query-tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if args.q_fp8 else "f16", "data": "synthetic",
        "config": dict(workload_config(problem, valid, args.num_splits, world),
                       **({"q": "e4m3", "q_scale": W.Q_SCALE_FP8} if args.q_fp8 else {})),
        "roofline": rl,
        "roofline_step_frac": step_rl["frac"],
        "roofline_sustained_frac": (rl["achieved"] / peaks["bf16_tflops_sustained"]
                                    if rl["bound"] == "tensor" and peaks.get("bf16_tflops_sustained")
                                    else None),
        "algorithmic": {"kv_bytes": kv_bytes, "flops": flops},
        "e2e": {"value": world * w.num_tokens / (e2e_ms * 1e-3), "unit": "query-tokens/s",
                "method": f"pipelined: copy in, decode and copy out of consecutive steps overlap on three streams; "
                          f"{E2E_VARIANTS} index sets in turn, no L2 flush",
                **{k: round(v, 4) for k, v in copy_ms.items()},
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "wall_s": wall,
    }
    if args.cpu_baseline_seconds > 0 and world == 1:
        cpu_problem = problem
        n, el = run_oracle_sample(cpu_problem, budget_s=args.cpu_baseline_seconds,
                                  q_e4m3=None if q8 is None else q8.cpu(), q_scale=W.Q_SCALE_FP8)
        line["cpu_baseline"] = {"value": n / el, "unit": "query-tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"{n} of {w.num_tokens} query tokens of {w.name}, oracle "
                                          f"decode time {el:.1f} s (cache rows packed beforehand, "
                                          f"untimed), numpy float64, 1 BLAS thread"}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# ------------------------------------------------------------------------------ indexer arm


def indexer_work(problem, ix) -> dict:
    """Algorithmic work of one indexer pass (logits + top-k) over a batch."""
    w = problem.w
    ctx = ix.ctx.cpu().tolist()
    vis = [max(0, ctx[t // w.next_n] - w.next_n + 1 + t % w.next_n) for t in range(w.num_tokens)]
    key_bytes = sum(max(0, c) for c in ctx) * (W.INDEX_DIM + 4)  # each request's keys, read once
    io_bytes = w.num_tokens * ix.heads * (W.INDEX_DIM + 4) + w.num_tokens * w.topk * 4
    flops = sum(vis) * ix.heads * W.INDEX_DIM * 2
    return {"key_bytes": key_bytes, "bytes": key_bytes + io_bytes, "flops": flops,
            "logit_bytes": sum(vis) * 4, "visible": sum(vis)}


def run_indexer_oracle_sample(problem, ix, budget_s: float):
    """The float64 indexer oracle (logits + top-k) on whole query tokens, until budget_s."""
    from oracle import indexer_oracle as IX
    w = problem.w
    pt = problem.page_table.cpu().numpy()
    q = ix.q.cpu().numpy()
    wt = ix.weights.cpu().double().numpy()
    ctx = ix.ctx.cpu().numpy()
    done, el = 0, 0.0
    for t in range(0, w.num_tokens, max(1, w.num_tokens // 32)):
        r, i = divmod(t, w.next_n)
        n = IX.visible_len(ctx[r], w.next_n, i)
        npg = -(-n // w.page_size)
        cache = {int(pg): ix.cache[int(pg)].cpu().numpy() for pg in pt[r][:npg]}
        t0 = time.perf_counter()
        keys, sc = IX.request_keys(cache, pt[r], n, w.page_size)
        IX.topk_set(IX.logits_of_token(q[t], wt[t], keys, sc), w.topk)
        el += time.perf_counter() - t0
        done += 1
        if el >= budget_s:
            break
    return done, el


def indexer_arm(args):
    """The indexer (smla_indexer_logits + smla_indexer_topk) on the batch shape of a decode workload."""
    import sparse_mla_decode_smla_gb300 as smla
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = workload_from_args(args)
    problem = W.make_problem(w, device=dev)
    ix = W.make_indexer_inputs(problem, device=dev)
    stride = w.page_table_stride * w.page_size
    desc = smla.make_indexer_desc(w.num_requests, w.next_n, ix.heads, w.page_size, problem.num_pages,
                                  w.page_table_stride, stride, w.topk)
    pt = problem.page_table.to(device=dev, dtype=torch.int32).contiguous()
    logits = torch.empty((w.num_tokens, stride), dtype=torch.float32, device=dev)
    topk = torch.empty((w.num_tokens, w.topk), dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    work = indexer_work(problem, ix)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        smla.indexer_logits(desc, ix.q, ix.weights, ix.cache, pt, ix.ctx, logits, err)
        if ev:
            ev[1].record(stream)
        smla.indexer_topk(desc, logits, ix.ctx, topk)
        if ev:
            ev[2].record(stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with ClockSampler(0) as clk:
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            flush.fill_(float(i))
            step(evs[i])
        torch.cuda.synchronize(dev)
    lg_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    tk_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    ms = lg_ms + tk_ms
    assert err.item() == 0, f"indexer error word {err.item()}"
    peaks = measured_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]  # the measured bf16 peak x the nominal fp8 / bf16 ratio of 2
    t_hbm = work["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = work["flops"] / (fp8_peak * 1e12)
    if t_hbm >= t_tc:
        ach = work["bytes"] / (lg_ms * 1e-3) / 1e9
        rl = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
              "frac": ach / peaks["hbm_gbs"], "peak_source": peaks["source"] + " hbm_gbs (burst)"}
    else:
        ach = work["flops"] / (lg_ms * 1e-3) / 1e12
        rl = {"bound": "tensor", "achieved": ach, "peak": fp8_peak, "unit": "TFLOP/s",
              "frac": ach / fp8_peak, "peak_source": peaks["source"] + " bf16_tflops (burst) x 2 (fp8)"}
    rl.update({"kernel": "indexer_logits_kernel", "kernel_ms": lg_ms, "traffic": None})
    line = {"metric": "indexer query-tokens/s", "value": w.num_tokens / (ms * 1e-3), "unit": "query-tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": w.name, "op": "indexer", "tokens": w.num_tokens, "next_n": w.next_n,
                       "index_heads": ix.heads, "topk": w.topk, "visible_slots": work["visible"],
                       "l2": "flushed between timed steps (512 MiB write, outside the events)"},
            "roofline": rl, "kernels_ms": {"indexer_logits_kernel": lg_ms, "indexer_topk_kernel": tk_ms},
            "algorithmic": work, "gpu_launches": 2 * args.steps, "clocks": clk.summary()}
    if args.cpu_baseline_seconds > 0:
        n, el = run_indexer_oracle_sample(problem, ix, args.cpu_baseline_seconds)
        line["cpu_baseline"] = {"value": n / el, "unit": "query-tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"{n} of {w.num_tokens} query tokens, indexer oracle (logits + top-k) "
                                          f"time {el:.1f} s, numpy float64, 1 BLAS thread"}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------ fused-store arm


def store_work(n: int, row_bytes: int) -> dict:
    """Algorithmic bytes of one fused store of n rows: the bf16 latent and RoPE (1152 B), the
    position and slot (16 B) and the row's cos/sin (256 B) read, the packed row written."""
    per_row = 2 * 576 + 16 + 64 * 4 + row_bytes
    return {"bytes_per_row": per_row, "bytes": n * per_row + 1024, "rows": n}


def store_arm(args):
    """smla_store_kv_normed (RMSNorm + RoPE + quantise on write) over one prefill chunk of rows."""
    import numpy as np
    import sparse_mla_decode_smla_gb300 as smla
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n, P, max_pos = args.store_rows, 64, 131072
    fmt = {"fp8_ds": (smla.SMLA_KV_FP8_DS, 656), "fp8_tensor": (smla.SMLA_KV_FP8_TENSOR, 576),
           "bf16": (smla.SMLA_KV_BF16, 1152)}[args.store_format]
    x = W.make_store_inputs(n, 7, max_position=max_pos, device=dev)
    x.positions = torch.arange(n, dtype=torch.int64, device=dev)  # a chunk's consecutive positions
    pages = -(-n // P)
    perm = torch.randperm(pages, generator=torch.Generator().manual_seed(8)).to(dev)
    slots = perm.repeat_interleave(P)[:n] * P + torch.arange(n, device=dev) % P
    kv = torch.zeros((pages * P, fmt[1]), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    kv_scale = 2.0 ** -4

    def step():
        smla.store_kv_normed(fmt[0], x.latent, x.rope, x.weight, 1e-6, x.positions, x.cos_sin, slots, kv,
                             pages * P, kv_scale=kv_scale, error_word=err)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(0) as clk:
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            flush.fill_(float(i))
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    assert err.item() == 0, f"store error word {err.item()}"
    peaks = measured_peaks()
    work = store_work(n, fmt[1])
    ach = work["bytes"] / (ms * 1e-3) / 1e9
    rl = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
          "frac": ach / peaks["hbm_gbs"], "kernel": "pack_kernel (normed)", "kernel_ms": ms,
          "traffic": recorded_traffic(f"store_{args.store_format}_rows{n}_P{P}_pos{max_pos}", "pack_kernel"),
          "peak_source": peaks["source"] + " hbm_gbs (burst)"}
    line = {"metric": "fused cache-store rows/s", "value": n / (ms * 1e-3), "unit": "rows/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"store_{args.store_format}_rows{n}_P{P}_pos{max_pos}", "op": "store",
                       "rows": n, "kv_format": args.store_format, "row_bytes": fmt[1],
                       "positions": "consecutive from 0", "slots": "shuffled pages of 64",
                       "l2": "flushed between timed steps (512 MiB write, outside the events)"},
            "roofline": rl, "algorithmic": work, "gpu_launches": args.steps, "clocks": clk.summary()}
    if args.cpu_baseline_seconds > 0:
        import oracle as O
        host = {k: getattr(x, k).cpu() for k in ("latent", "rope", "weight", "positions", "cos_sin")}
        bits = {k: host[k].view(torch.int16).numpy().view(np.uint16) for k in ("latent", "rope", "weight")}
        cs = host["cos_sin"].double().numpy()
        done, el, chunk = 0, 0.0, 1024
        while el < args.cpu_baseline_seconds and done < n:
            lo, hi = done, min(n, done + chunk)
            c = cs[host["positions"][lo:hi].numpy()]
            t0 = time.perf_counter()
            O.store_normed_rows(bits["latent"][lo:hi], bits["rope"][lo:hi], bits["weight"], 1e-6, c[:, :32],
                                c[:, 32:], args.store_format, O.SCALE_POW2, kv_scale)
            el += time.perf_counter() - t0
            done = hi
        line["cpu_baseline"] = {"value": done / el, "unit": "rows/s", "cores": 1, "kind": "oracle",
                                "sample": f"{done} of {n} rows, fused-store oracle, numpy float64, 1 BLAS thread, "
                                          f"{el:.1f} s"}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=[w.name for w in W.WORKLOADS + W.EXTRA_WORKLOADS])
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--op", default="decode", choices=["decode", "indexer", "store"],
                    help="decode (the hot path, default), the indexer that produces its top-k indices, "
                         "or the fused cache store (RMSNorm + RoPE + quantise on write)")
    ap.add_argument("--store-rows", type=int, default=65536, help="--op store: rows per call")
    ap.add_argument("--store-format", default="fp8_ds", choices=["fp8_ds", "fp8_tensor", "bf16"])
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--q-fp8", action="store_true",
                    help="E4M3 q against a per-tensor FP8 workload (the FP8-operand tensor-core kernel)")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=15.0)
    ap.add_argument("--ref-budget-seconds", type=float, default=60.0,
                    help="reference arm: oracle decode time of all timed steps together")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--ctx-lo", type=int, default=0, help="smaller variant (profiling): context range low")
    ap.add_argument("--ctx-hi", type=int, default=0, help="smaller variant (profiling): context range high")
    ap.add_argument("--requests", type=int, default=0, help="smaller variant (profiling): requests")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the decode kernel from an ncu capture, if current")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return reference_arm(args)
    if args.op == "indexer":
        return indexer_arm(args)
    if args.op == "store":
        return store_arm(args)
    return gpu_arm(args)


if __name__ == "__main__":
    sys.exit(main())
