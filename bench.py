"""Throughput benchmark for libmla_prefill (one JSON line on rank 0).

A step is one pass of the whole path on one batch: the prefill plan followed
by the ragged paged MLA attention, on the DeepSeek-V3-shaped workload (B=8,
new lengths U[512,4096], no prior cache, H=128, q_depth 192, depth 128,
k_rope 64 paged with P=128, causal, bf16).  Inputs are resident in HBM and
larger than L2 (about 2.1 GB per batch), so no flush is needed between steps.

Metric: causal-effective TFLOP/s = H * 2 * (192 + 128) * sum_b A_b per step,
A_b = n_b * prior_b + n_b (n_b + 1) / 2 (the visible (query, key) pairs), over
the device time of the timed steps.  Under torchrun every rank runs its own
batch (weak scaling, no data-path collective); the step time is the maximum
over ranks.

--mode chunked times chunked execution instead of the full-context call: the
plan, then all its buffer rows of buffer_token_size tokens in one
mla_prefill_ragged_chunked call (the K buffer of row r being rows
r*T .. r*T+T-1 of the batch-order packed K/V); --combine fold / merge time one
mla_prefill_ragged_chunk per row instead, folded in place or followed by
mla_prefill_merge.  Same metric, same work.

--mode contiguous times mla_prefill_ragged_contiguous: the same K_rope rows laid
out contiguously (row = K row) instead of paged.

--impl reference times the CPU oracle instead (float64, the machine's host
cores) on a bounded sample of the same workload.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time
from dataclasses import replace

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "MLA prefill causal-effective TFLOP/s and % of GB300 tensor peak, 1 GPU"
WORKLOAD = "deepseek_v3_bf16"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic of one attention launch per workload, from the ncu captures
# summarised in profiles/; valid only while the kernel source is unchanged.
ATTENTION_TRAFFIC = {"source_sha1": "a4fea7fad2f013099c92a0be7b2506f181e00ea7",
                     "bytes_per_launch": {"deepseek_v3_bf16": 2401581568, "fp8_e4m3": 3197671424}}


def causal_flops(w):
    pairs = 0
    for b in range(w.batch):
        n, prior = int(w.n[b]), int(w.prior[b])
        pairs += n * prior + n * (n + 1) // 2 if w.spec.mask == "causal" else n * (n + prior)
    return w.heads * 2 * (192 + 128) * pairs


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


def source_sha1():
    with open(os.path.join(ROOT, "mla_ragged_paged_gb300", "csrc", "attention.cu"), "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()


class Ticker:
    """Labelled segments of the timed steps: tick(label) records an event on
    the stream that ends the previous segment and starts `label` (None ends
    without starting one); totals() sums each label's event-timed spans."""

    def __init__(self, stream):
        self.stream = stream
        self.marks = []

    def tick(self, label):
        e = torch.cuda.Event(enable_timing=True)
        e.record(self.stream)
        self.marks.append((label, e))

    def totals(self):
        out = {}
        for (label, e0), (_, e1) in zip(self.marks, self.marks[1:]):
            if label is not None:
                out[label] = out.get(label, 0.0) + e0.elapsed_time(e1)
        return out


class ClockSampler:
    """nvidia-smi clocks and throttle reasons while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        rows = []
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:7], float(parts[7])))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        loaded = [r for r in rows if r[3] > 50] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[2]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(loaded)}


def dist_setup():
    """Process group from the torchrun environment: NCCL with one GPU per rank,
    gloo where no GPU is present (the CPU reference arm, host-side tests)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return world, rank, local


def dist_max(x, world):
    """Maximum of x over the ranks (the step time of a weak-scaling run)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_sum(x, world):
    """Sum of x over the ranks (work units every rank processed)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def rank_spec(spec, rank):
    """Every rank runs its own batch of the same shape (weak scaling): the
    workload's seed is offset by the rank."""
    return spec if rank == 0 else replace(spec, seed=spec.seed + 1000 * rank)


_ORACLE_OUT = {}


def oracle_sample(w, rows, heads):
    """Time the oracle on the last `rows` query rows of the longest sequence
    of `w` for the given heads; returns (causal-effective flops, seconds, text).
    The output array is allocated once, outside the timed region."""
    from oracle import attention as oatt
    out = _ORACLE_OUT.get(id(w))
    if out is None:
        out = _ORACLE_OUT[id(w)] = np.zeros((w.total_q, w.heads, 128), dtype=np.float64)
    b = int(np.argmax(w.n))
    n, prior = int(w.n[b]), int(w.prior[b])
    rows = int(min(n, max(1, rows)))
    heads = [h % w.heads for h in heads]
    sel = np.arange(n - rows, n)
    t0 = time.perf_counter()
    oatt.reference(w, heads=heads, rows={b: sel}, out=out)
    dt = time.perf_counter() - t0
    pairs = int(sum(prior + i + 1 for i in sel)) if w.spec.mask == "causal" else rows * (n + prior)
    text = (f"sequence {b} (n={n}, prior={prior}), {len(heads)} head(s) from {heads[0]}, "
            f"last {rows} query rows")
    return 2 * (192 + 128) * pairs * len(heads), dt, text


def oracle_shape_for(w, budget_s):
    """(rows, head count) for which one oracle_sample call takes about budget_s."""
    n = int(w.n.max())
    _, dt, _ = oracle_sample(w, 256, [0])
    per_head = dt * n / 256.0
    if per_head >= budget_s:
        return max(1, int(256 * budget_s / max(dt, 1e-4))), 1
    return n, int(min(w.heads, max(1, budget_s // max(per_head, 1e-4))))


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, world, rank):
    """The CPU oracle on host cores; under torchrun only rank 0 runs it."""
    if rank != 0:
        return
    spec = workloads.config(args.workload)
    w = workloads.generate(spec)
    ktok = spec.dtype == "fp8" and args.k_scales == "token"
    if ktok:
        w = workloads.per_token_k(w)
    per_step = max(0.05, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    rows, nh = oracle_shape_for(w, per_step)
    for i in range(args.warmup):
        oracle_sample(w, rows, [i + k for k in range(nh)])
    tot_f, tot_t, sample = 0, 0.0, ""
    for i in range(args.steps):
        f, dt, sample = oracle_sample(w, rows, [args.warmup + i + k for k in range(nh)])
        tot_f += f
        tot_t += dt
    value = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{spec.name}: {spec.description}",
                       "sample_per_step": "query rows of one (sequence, head)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": host_cores(),
                             "kind": "oracle", "sample": f"per step: {sample}"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    if spec.dtype == "fp8":
        line["config"]["k_scales"] = ("one K_nope scale per K row (re-quantised per row)" if ktok
                                      else "per-tensor K_nope scale")
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # 1000 steps: about 1.6 s timed on the default workload, so the clock
    # sampler (every 100 ms) sees the GPU under load a dozen times.
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD, choices=[c.name for c in workloads.CONFIGS],
                    help="workload to time (default: the DeepSeek-V3-shaped bf16 batch)")
    ap.add_argument("--combine", default=None, choices=["single", "fold", "merge"],
                    help="chunked mode: all buffer rows in one mla_prefill_ragged_chunked call (default); "
                         "chunked / latent modes: one call per row, folding every row into the output in place "
                         "(MLA_CHUNK_ACCUMULATE), or write per-row outputs and run mla_prefill_merge")
    ap.add_argument("--mode", default="full", choices=["full", "chunked", "contiguous", "latent", "split"],
                    help="full-context attention call (paged K_rope); one call per plan buffer row "
                         "plus the merge; the full-context call on a contiguous K_rope; or the "
                         "latent-cache path (per row: gather fused with the K/V up-projection, attention; fold or merge); "
                         "or Q split into q_nope and a bf16 q_rope")
    ap.add_argument("--k-scales", default="tensor", choices=["tensor", "token"],
                    help="fp8 workloads: one K_nope scale per tensor, or one per K row (the "
                         "workload's K_nope re-quantised row by row)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import mla_ragged_paged_gb300 as pkg
    from mla_ragged_paged_gb300 import binding
    # One rank compiles (if the library is stale); the others wait for it.
    if local == 0:
        pkg.build()
    barrier(world)
    if local != 0:
        pkg.build()          # up to date by now: returns at once
    binding.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    spec = workloads.config(args.workload)
    fp8 = spec.dtype == "fp8"
    w = workloads.generate(rank_spec(spec, rank))
    ktok = fp8 and args.k_scales == "token"
    if args.k_scales == "token" and not fp8:
        ap.error("--k-scales token needs an fp8 workload")
    if ktok:
        w = workloads.per_token_k(w)
    F = causal_flops(w)
    d = workloads.device_inputs(w, device=dev)
    contiguous = args.mode == "contiguous"
    latent = args.mode == "latent"
    split = args.mode == "split"
    if split:
        # q_nope = Q[..., :128] (bf16, or the e4m3 codes); q_rope = Q[..., 128:]
        # as bf16 real values (fp8: the rope codes times q_scale, rounded).
        if fp8:
            rope = w.q.view(torch.float8_e4m3fn)[..., 128:].to(torch.float32) * w.q_scale
            d["q_rope"] = rope.to(torch.bfloat16).to(dev)
            d["q_nope"] = w.q[..., :128].contiguous().to(dev)
        else:
            d["q_nope"] = w.q[..., :128].contiguous().to(dev)
            d["q_rope"] = w.q[..., 128:].contiguous().to(dev)
        del d["q"]
    if latent:
        assert not fp8, "the latent-cache path is bf16"
        lpool, w_uk, w_uv = workloads.latent_cache(w)
        d["latent_pool"], d["w_uk"], d["w_uv"] = lpool.to(dev), w_uk.to(dev), w_uv.to(dev)
        del d["k_nope"], d["v"], d["k_rope_pool"]
    if contiguous:
        rows, rsc = workloads.contiguous_rope(w)
        d["k_rope_contig"] = rows[:, spec.rope_col:spec.rope_col + 64].contiguous().to(dev)
        del d["k_rope_pool"], d["page_table"]
        if fp8:
            d["k_rope_scales"] = rsc.to(dev)
    in_bytes = sum(t.numel() * t.element_size() for t in d.values())
    Tq, H, B = w.total_q, w.heads, w.batch
    T = spec.buffer_token_size
    R = (w.total_k + T - 1) // T
    out = torch.empty((Tq, H, 128), dtype=torch.bfloat16, device=dev)
    # fp8: converted K_rope rows per pool slot, or per K row (contiguous
    # K_rope, per-token K scales).
    ws = binding.alloc_workspace(B, dev, fp8_pool_slots=(w.total_k if contiguous or ktok
                                                         else w.num_pages * w.page_size) if fp8 else None)
    scales = {k: d.get(k) for k in ("q_scale", "k_scale", "v_scale", "k_rope_scales")}
    plan_out = (torch.empty((R, B + 1), dtype=torch.int32, device=dev),
                torch.empty((R, B), dtype=torch.int32, device=dev),
                torch.empty((R,), dtype=torch.int32, device=dev),
                torch.empty((1,), dtype=torch.int32, device=dev))
    stream = torch.cuda.current_stream(dev)
    chunked = args.mode in ("chunked", "latent")
    combine = args.combine or ("single" if args.mode == "chunked" else "fold")
    if latent and combine == "single":
        ap.error("--combine single applies to --mode chunked")
    single = chunked and combine == "single"
    fold = chunked and combine == "fold"
    scratch = binding.chunked_scratch(R, Tq, H, dev) if chunked and combine == "merge" else None
    lse_buf = torch.empty((Tq, H), dtype=torch.float32, device=dev) if fold else None
    lbuf = binding.LatentRowBuffers(T, H, dev) if latent else None

    def attention(inp, o, tk=None):
        """The attention part of a step; `tk` (a Ticker) labels its segments."""
        tick = tk.tick if tk is not None else (lambda label: None)
        tick("attn")
        if split:
            binding.prefill_ragged_split(o, inp["q_nope"], inp["q_rope"], inp["k_nope"], inp["v"],
                                         inp["k_rope_pool"], inp["page_table"], inp["row_offsets"],
                                         inp["cache_lens"], w.scale, binding.MLA_MASK_CAUSAL, ws,
                                         stream=stream, **scales)
            return
        if contiguous:
            binding.prefill_ragged_contiguous(o, inp["q"], inp["k_nope"], inp["v"], inp["k_rope_contig"],
                                              inp["row_offsets"], inp["cache_lens"], w.scale,
                                              binding.MLA_MASK_CAUSAL, ws, stream=stream, **scales)
            return
        if not chunked:
            binding.prefill_ragged(o, inp["q"], inp["k_nope"], inp["v"], inp["k_rope_pool"],
                                   inp["page_table"], inp["row_offsets"], inp["cache_lens"], w.scale,
                                   binding.MLA_MASK_CAUSAL, ws, stream=stream, **scales)
            return
        if single:
            # Every buffer row of the plan in one call; the rows' K buffers
            # are the packed K/V, stacked T rows apart.
            binding.prefill_ragged_chunked(o, inp["q"], inp["k_nope"], inp["v"], inp["k_rope_pool"],
                                           inp["page_table"], inp["row_offsets"], inp["cache_lens"],
                                           plan_out[0], plan_out[1], plan_out[3], T, w.scale,
                                           binding.MLA_MASK_CAUSAL, ws, stream=stream, **scales)
            return
        flags = binding.MLA_CHUNK_ACCUMULATE if fold else 0
        for r in range(R):
            lo, hi = r * T, min((r + 1) * T, w.total_k)
            o_r, l_r = (o, lse_buf) if fold else (scratch[0][r], scratch[1][r])
            if latent:
                # The row's K_nope and V projected from its gathered latent
                # rows (one launch), then its attention with K_rope read from
                # the latent cache through the page table.
                n = hi - lo
                tick("gemm")
                kn, vv = lbuf.k_nope[:n], lbuf.v[:n]
                binding.gather_up_project(kn, vv, inp["latent_pool"], inp["w_uk"], inp["w_uv"],
                                          inp["page_table"], plan_out[0][r], plan_out[1][r], stream=stream)
                tick("attn")
                binding.prefill_ragged_chunk(o_r, l_r, inp["q"], kn, vv,
                                             binding.latent_rope_pages(inp["latent_pool"]), inp["page_table"],
                                             inp["row_offsets"], inp["cache_lens"], plan_out[0][r],
                                             plan_out[1][r], w.scale, binding.MLA_MASK_CAUSAL, ws,
                                             stream=stream, flags=flags)
                continue
            row_scales = dict(scales, k_scale=scales["k_scale"][lo:hi]) if ktok else scales
            binding.prefill_ragged_chunk(o_r, l_r, inp["q"], inp["k_nope"][lo:hi], inp["v"][lo:hi],
                                         inp["k_rope_pool"], inp["page_table"], inp["row_offsets"],
                                         inp["cache_lens"], plan_out[0][r], plan_out[1][r], w.scale,
                                         binding.MLA_MASK_CAUSAL, ws, stream=stream, flags=flags,
                                         **row_scales)
        if combine == "merge":
            tick("merge")
            binding.merge(o, scratch[0], scratch[1], inp["row_offsets"], plan_out[0], stream=stream)

    def step(inp, o):
        binding.plan(inp["row_offsets"], inp["cache_lens"], T, R, stream=stream, out=plan_out)
        attention(inp, o)

    for _ in range(args.warmup):
        step(d, out)
    assert binding.device_status(ws) == 0, "device status after warm-up"

    # Device-resident timing: labelled segments of every step (events on the
    # launching stream) and the whole timed region.
    tk = Ticker(stream)
    barrier(world)
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            tk.tick("plan")
            binding.plan(d["row_offsets"], d["cache_lens"], T, R, stream=stream, out=plan_out)
            attention(d, out, tk)
            tk.tick(None)
        t_end.record(stream)
        barrier(world)
    total_ms = dist_max(t_start.elapsed_time(t_end), world)
    # Every rank's batch is drawn with its own seed: the whole job's work is
    # the sum of the ranks' causal-effective flops.
    F_all = dist_sum(float(F), world)
    # Attention-kernel span (the per-row calls in chunked mode) and merge span.
    seg = {k: v / args.steps for k, v in tk.totals().items()}   # ms per step per segment
    attn_ms = seg["attn"]
    merge_ms = seg.get("merge")
    assert binding.device_status(ws) == 0, "device status after timed steps"
    clocks = clk.summary()

    # End to end through the public API: pinned host inputs -> device, plan +
    # attention, output -> pinned host, every step.
    h = workloads.device_inputs(w, device="cpu", pin=True)
    if latent:
        for k in ("latent_pool", "w_uk", "w_uv"):
            h[k] = d[k].cpu().pin_memory()
    if split:
        for k in ("q_nope", "q_rope"):
            h[k] = d[k].cpu().pin_memory()
    if contiguous:
        h["k_rope_contig"] = d["k_rope_contig"].cpu().pin_memory()
        if fp8:
            h["k_rope_scales"] = d["k_rope_scales"].cpu().pin_memory()
    keys = (["q_nope", "q_rope"] if split else ["q"]) + ["row_offsets", "cache_lens"]
    if latent:
        keys += ["latent_pool", "page_table", "w_uk", "w_uv"]
    else:
        keys += ["k_nope", "v"] + (["k_rope_contig"] if contiguous else ["k_rope_pool", "page_table"])
    if fp8:
        keys += ["q_scale", "k_scale", "v_scale", "k_rope_scales"]
    # Two device buffer sets: step i copies its inputs in on an H2D stream,
    # runs on the compute stream and copies its output out on a D2H stream,
    # so the copies of steps i+1 and i-1 overlap step i.
    sets = [{k: torch.empty_like(d[k]) for k in keys} for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    hosts = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(h[k].numel() * h[k].element_size() for k in keys)
    d2h = hosts[0].numel() * hosts[0].element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in", "done", "out")}

    def e2e_steps(n):
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev["done"][b])       # step i-2 no longer reads set b
                for k in keys:
                    sets[b][k].copy_(h[k], non_blocking=True)
                ev["in"][b].record(s_in)
            stream.wait_event(ev["in"][b])
            if i >= 2:
                stream.wait_event(ev["out"][b])          # output of step i-2 copied out
            if fp8:
                scales.update({k: sets[b][k] for k in ("q_scale", "k_scale", "v_scale", "k_rope_scales")})
            step(sets[b], outs[b])
            ev["done"][b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["done"][b])
                hosts[b].copy_(outs[b], non_blocking=True)
                ev["out"][b].record(s_out)

    e2e_steps(2)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    e2e_steps(args.e2e_steps)
    s_out.wait_stream(stream)
    s_out.wait_stream(s_in)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = dist_max(e0.elapsed_time(e1), world)

    # The host link's own rate: the same per-step input copies, pinned host ->
    # device, one cudaMemcpyAsync per tensor on the copy stream, no compute
    # beside them (best of three).
    link_ms = None
    for _ in range(3):
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s_in):
            c0.record(s_in)
            for k in keys:
                sets[0][k].copy_(h[k], non_blocking=True)
            c1.record(s_in)
        torch.cuda.synchronize(dev)
        t = c0.elapsed_time(c1)
        link_ms = t if link_ms is None else min(link_ms, t)
    link_gbs = h2d / (link_ms * 1e-3) / 1e9
    e2e_h2d_gbs = h2d * args.e2e_steps / (e2e_ms * 1e-3) / 1e9

    peaks, peak_src = load_peaks()
    # fp8 UMMAs run at twice the bf16 rate (nominal 4.5 vs 2.25 PFLOP/s dense).
    peak = peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)
    achieved = F / (attn_ms * 1e-3) / 1e12
    traffic = None
    if ATTENTION_TRAFFIC["source_sha1"] == source_sha1() and args.mode == "full":
        traffic = ATTENTION_TRAFFIC["bytes_per_launch"].get(spec.name + (" per-token K" if ktok else ""))
    merge_roofline = None
    if combine == "merge" and chunked:
        # Algorithmic merge bytes: per (token, head), 256 + 4 bytes read from
        # each row holding keys of its sequence, 256 bytes written.
        G = np.concatenate([[0], np.cumsum(w.n + w.prior)])
        rows_b = (np.minimum(-(-G[1:] // T), R) - G[:-1] // T) * ((w.n + w.prior) > 0)
        mbytes = H * int(sum(int(w.n[b]) * (int(rows_b[b]) * 260 + 256) for b in range(B)))
        m_gbs = mbytes / (merge_ms * 1e-3) / 1e9
        merge_roofline = {"bound": "hbm", "achieved": m_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                          "frac": m_gbs / peaks["hbm_gbs"], "bytes_per_launch": mbytes,
                          "ms": merge_ms, "kernel": "merge_kernel"}
    latent_roofline = None
    if latent:
        # Gather + up-projection: two GEMMs [S, 512] x [512, H*128] per step,
        # one launch per buffer row.
        gflop = 2 * 2 * w.total_k * 512 * H * 128
        g_tf = gflop / (seg["gemm"] * 1e-3) / 1e12
        latent_roofline = {"bound": "tensor", "achieved": g_tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                           "frac": g_tf / peaks["bf16_tflops"], "ms": seg["gemm"],
                           "flop_per_step": gflop, "kernel": "up_project_kernel (gather fused, tcgen05)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not latent:
        # About 10-30 s of host work: size from a short probe, then widen the
        # head sample once if the first run came in under 10 s.
        rows, nh = oracle_shape_for(w, 15.0)
        f, dt, sample = oracle_sample(w, rows, list(range(nh)))
        if dt < 10.0 and nh < w.heads:
            nh = min(w.heads, int(nh * 15.0 / max(dt, 0.1)) + 1)
            f, dt, sample = oracle_sample(w, rows, list(range(nh)))
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
               "sample": sample + f"; {dt:.1f} s of float64 numpy on the host"}

    # This library's kernels per step.
    if latent:
        launches_per_step = 1 + 3 * R          # plan; per row gather + up-projection, scheduler, attention
    elif chunked and not single:
        launches_per_step = 1 + R * (3 if fp8 else 2)
    else:
        launches_per_step = 4 if fp8 else 3    # plan, scheduler, (fp8: K_rope conversion), attention
    if chunked and combine == "merge":
        launches_per_step += 1                 # merge
    merge_txt = " + mla_prefill_merge" if combine == "merge" else ""
    if rank == 0:
        value = F_all * args.steps / (total_ms * 1e-3) / 1e12
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3" if fp8 else "bf16",
            "data": "synthetic",
            "config": {"workload": f"{spec.name}: {spec.description}", "global_batch": B * world,
                       "total_q_tokens": Tq, "heads": H, "causal_effective_tflop_per_step": F_all / 1e12,
                       "parallelism": f"dp{world} (independent batches)" if world > 1 else "none",
                       "l2": f"inputs ({in_bytes / 1e9:.2f} GB) larger than L2; no flush",
                       "step": ("mla_prefill_plan + %d x (mla_gather_up_project + "
                                "mla_prefill_ragged_chunk, K_rope from the latent cache) (T=%d)%s" % (R, T, merge_txt))
                               if latent else
                               ("mla_prefill_plan + mla_prefill_ragged_chunked over its %d rows (T=%d)" % (R, T))
                               if single else
                               ("mla_prefill_plan + %d x mla_prefill_ragged_chunk (T=%d)%s"
                                % (R, T, merge_txt)) if chunked else
                               ("mla_prefill_plan + mla_prefill_ragged_contiguous (K_rope [S_k, 64], not paged)"
                                if contiguous else "mla_prefill_plan + mla_prefill_ragged_split (q_nope + bf16 q_rope)"
                                if split else "mla_prefill_plan + mla_prefill_ragged")},
            "pct_of_peak": 100.0 * value / world / peak,
            "clocks": clocks,
            "e2e": {"value": F_all * args.e2e_steps / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "h2d_gbs": e2e_h2d_gbs, "link_gbs": link_gbs, "h2d_frac_of_link": e2e_h2d_gbs / link_gbs,
                    "link_measure": "the step's input copies alone, pinned host to device, best of 3",
                    "pipelining": "two buffer sets: H2D of step i+1 and D2H of step i-1 overlap step i"},
            "gpu_launches": launches_per_step * args.steps,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                         "kernel": ("mla_attention_kernel over %d buffer rows (+ their scheduler launches)" % R)
                                   if chunked and not single else
                                   "mla_attention_kernel (+ its 1-CTA scheduler launch in the span)",
                         "peak_source": f"{peak_src} bf16_tflops (burst)" + (" x 2 (fp8/bf16 nominal ratio)" if fp8 else "")},
            "cpu_baseline": cpu,
        }
        if fp8:
            line["config"]["k_scales"] = ("one K_nope scale per K row (re-quantised per row)" if ktok
                                          else "per-tensor K_nope scale")
        if chunked:
            line["config"]["combine"] = {"single": "all rows in one mla_prefill_ragged_chunked call",
                                         "fold": "one call per row, in-place fold (MLA_CHUNK_ACCUMULATE)",
                                         "merge": "one call per row + mla_prefill_merge"}[combine]
        if merge_roofline is not None:
            line["roofline_merge"] = merge_roofline
        if latent:
            line["roofline_gemm"] = latent_roofline
            line["segments_ms"] = seg
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
