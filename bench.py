"""Benchmark: one paged decode step (store_kvcache of the step's new K/V rows,
then decode attention) on synthetic inputs, timed with CUDA events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0). ``value`` is microseconds per step (store +
decode, inputs resident in HBM, L2 flushed between steps); ``roofline``
reports the decode launch's KV-read bandwidth against the measured HBM copy
peak; ``e2e`` repeats the step through host buffers (pinned H2D of the step's
inputs and D2H of its output inside the timed region); ``cpu_baseline`` times
the fp64 CPU oracle on a bounded sample of the same step and scales it to a
full step. ``--impl reference`` times only that oracle (the reference arm).
With N > 1 (torchrun) every rank runs its own replica of the step on its own
GPU: the path has no cross-GPU exchange.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_255_gb300 import inputs  # noqa: E402

METRIC = "paged-decode µs/step and KV-read GB/s (fraction of GB300 HBM peak)"
DEFAULT_WORKLOAD = "qwen3_0_6b"
L2_FLUSH_BYTES = 512 << 20       # > 2x the 129 MB L2
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PREFILL_METRIC = "paged-prefill µs/step and attention TFLOP/s (fraction of GB300 bf16 tensor peak)"
PROFILE_FILE = os.path.join(ROOT, "profiles", "decode_traffic.txt")
KERNEL_SOURCES = ["paged_kv_cache_255_gb300/csrc/decode.cu", "paged_kv_cache_255_gb300/csrc/common.cuh"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks(key="hbm_gbs"):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS}[key], "fallback"


def ncu_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on this workload with the current kernel source."""
    try:
        text = open(PROFILE_FILE).read()
    except OSError:
        return None
    want = kernel_hash()
    for m in re.finditer(r"^traffic\s+workload=(\S+)\s+kernel_hash=(\S+)\s+bytes_per_launch=(\d+)",
                         text, re.M):
        if m.group(1) == workload and m.group(2) == want:
            return int(m.group(3))
    return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the GPU is busy."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu=timestamp,{','.join(self.FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "20", "-i", str(index)],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def wait_first_sample(self, timeout_s: float = 5.0):
        """nvidia-smi's start-up can stall the GPU for a moment: start the
        sampler before the warm-up and wait for its first line, so that the
        start never falls in a timed region."""
        if self.proc is None:
            return
        t0 = time.time()
        while time.time() - t0 < timeout_s:
            self.fh.flush()
            try:
                if os.path.getsize(self.path) > 0:
                    return
            except OSError:
                return
            time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 1 + len(self.FIELDS):
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, f in enumerate(flags)
                          if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons, "samples": len(rows)}


def dist_setup(n_gpus):
    if n_gpus <= 1 and "RANK" not in os.environ:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", n_gpus))
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(wl):
    s = wl.spec
    return {"workload": s.name, "num_seqs": wl.num_seqs, "num_q_heads": s.num_q_heads,
            "num_kv_heads": s.num_kv_heads, "head_dim": s.head_dim, "block_size": s.block_size,
            "num_blocks": wl.num_blocks, "store_rows": int(wl.slot_mapping.shape[0]),
            "context_tokens": int(wl.context_lens.astype(np.int64).sum()),
            "max_context_len": wl.max_context_len, "seed": wl.seed,
            "l2": "flushed between steps (512 MiB write)"}


def oracle_sample(wl, target_s: float, host=None):
    """Time the fp64 oracle on a bounded sample of the step and scale to a full
    step. Returns (us_per_step, threads, sample description)."""
    import oracle
    O = oracle.get()
    threads = O.num_threads()
    if host is None:
        host = (wl.q.cpu(), wl.k_cache.cpu(), wl.v_cache.cpu(), wl.k_new.cpu(), wl.v_new.cpu())
    q, kc, vc, kn, vn = host
    t_store = 0.0
    if wl.slot_mapping.shape[0]:
        kc = oracle._bits(kc).copy()            # private pools for the in-place store (untimed)
        vc = oracle._bits(vc).copy()
        t0 = time.perf_counter()
        O.store_kvcache_into(kn, vn, kc, vc, wl.slot_mapping)
        t_store = time.perf_counter() - t0
    S, Hq = wl.num_seqs, wl.spec.num_q_heads
    work_all = float(wl.context_lens.astype(np.float64).sum()) * Hq
    rng = np.random.Generator(np.random.PCG64(123))
    order = rng.permutation(S * Hq)
    done_pairs, done_work, elapsed, passes = 0, 0.0, 0.0, 0
    batch = max(threads, 8)
    # random (sequence, head) outputs, in growing batches, until target_s of
    # oracle time; a workload smaller than that is repeated whole
    while elapsed < target_s:
        pos = done_pairs % (S * Hq)
        idx = order[pos:pos + batch]
        pairs = np.stack([idx // Hq, idx % Hq], 1).astype(np.int32)
        t0 = time.perf_counter()
        O.decode_pairs(q, kc, vc, wl.block_tables, wl.context_lens, wl.scale, pairs, threads=0)
        elapsed += time.perf_counter() - t0
        done_pairs += len(idx)
        done_work += float(wl.context_lens[idx // Hq].astype(np.float64).sum())
        batch = min(batch * 2, 4096)
    decode_s = elapsed * (work_all / max(done_work, 1.0))
    us = (t_store + decode_s) * 1e6
    sample = (f"oracle store of all {int(wl.slot_mapping.shape[0])} rows + decode of "
              f"{done_pairs} (seq, q-head) outputs drawn at random with repeats (one step "
              f"has {S * Hq}), {elapsed:.1f} s of oracle time, scaled by context tokens "
              f"to one full step")
    return us, threads, sample


def workload_spec(args):
    spec = inputs.SPECS[args.workload]
    if args.num_seqs:
        spec = inputs.scaled(spec, num_seqs=args.num_seqs, name=f"{spec.name}_s{args.num_seqs}")
    return spec


def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = inputs.generate(workload_spec(args), seed=0,
                         device="cuda" if torch.cuda.is_available() else "cpu")
    host = (wl.q.cpu(), wl.k_cache.cpu(), wl.v_cache.cpu(), wl.k_new.cpu(), wl.v_new.cpu())
    # the whole run (warm-up and timed steps) takes about --ref-seconds of oracle time
    per_step = max(0.05, args.ref_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(wl, per_step, host)
    vals = []
    for _ in range(args.steps):
        us, threads, sample = oracle_sample(wl, per_step, host)
        vals.append(us)
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "us/step",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(wl),
            "cpu_baseline": {"value": v, "unit": "us/step", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gpu(args, rank, world, local):
    from paged_kv_cache_255_gb300 import pagedattn as pa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = inputs.generate(workload_spec(args), seed=0, device=dev)
    S, Hq, Hkv, D = wl.num_seqs, wl.spec.num_q_heads, wl.spec.num_kv_heads, wl.spec.head_dim
    q = wl.q
    k_cache, v_cache = wl.k_cache, wl.v_cache
    HM = args.layout == "head_major"
    if HM:          # the same values in a [NB, Hkv, bs, D] pool
        k_cache = k_cache.permute(0, 2, 1, 3).contiguous()
        v_cache = v_cache.permute(0, 2, 1, 3).contiguous()
        if args.q_len > 1:
            raise SystemExit("--q-len > 1 runs on the token-major layout only")
    k_new, v_new = wl.k_new, wl.v_new
    slots = torch.from_numpy(wl.slot_mapping).to(dev)
    bt = torch.from_numpy(wl.block_tables).to(dev)
    cl = torch.from_numpy(wl.context_lens).to(dev)
    Q = args.q_len
    if Q > 1:
        # Q query tokens per sequence (speculative verification)
        gq = torch.Generator(device=dev)
        gq.manual_seed(1)
        q = torch.randn((S, Q, Hq, D), generator=gq, device=dev).to(torch.bfloat16)
    out = torch.empty_like(q)
    ws = pa.workspace_for(Hq, Hkv, D, 0, dev)

    def decode_call(q_, bt_, cl_):
        if Q > 1:
            return pa.decode_multi(q_, k_cache, v_cache, bt_, cl_, wl.scale, out=out)
        return pa.decode(q_, k_cache, v_cache, bt_, cl_, wl.scale, out=out, workspace=ws,
                         head_major=HM)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    has_store = slots.shape[0] > 0

    def step():
        if has_store:
            pa.store_kvcache(k_new, v_new, k_cache, v_cache, slots, head_major=HM)
        decode_call(q, bt, cl)

    # ---- device-resident timing: store then decode back to back, as a user
    # issues them (the decode launch may overlap the store's tail)
    clocks = ClockSampler(local)
    clocks.wait_first_sample()
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    step_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    ms = max_over_ranks(sum(step_ms) / len(step_ms), world)

    # ---- the same steps with an event between store and decode, for the
    # per-call split and the decode launch's own bandwidth (roofline)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        if has_store:
            pa.store_kvcache(k_new, v_new, k_cache, v_cache, slots, head_major=HM)
        ev[i][1].record(stream)
        decode_call(q, bt, cl)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    store_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    dec_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    dec_avg = max_over_ranks(sum(dec_ms) / len(dec_ms), world)
    store_avg = max_over_ranks(sum(store_ms) / len(store_ms), world)

    # ---- warm: the same steps without the L2 flush between them (inputs that
    # fit L2 then stay there; informative, not the reported value). A short
    # spin on the GPU before each step stands in for the flush kernel's other
    # role: the host queues the step while it runs, so the events do not time
    # the host's launch calls.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        torch.cuda._sleep(100_000)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    warm_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    warm_avg = max_over_ranks(sum(warm_ms) / len(warm_ms), world)

    # ---- end to end through host buffers: the step's inputs are packed in one
    # pinned staging buffer, copied in one transfer, and the output read back
    host_inputs = [q, k_new, v_new, slots, bt, cl]
    offs, total = [], 0
    for t in host_inputs:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_stage = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    for t, o in zip(host_inputs, offs):
        n = t.numel() * t.element_size()
        h_stage[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
    d_stage = torch.empty(total, dtype=torch.uint8, device=dev)
    views = [d_stage[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
             for t, o in zip(host_inputs, offs)]
    dq, dk, dv, ds, dbt, dcl = views
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_inputs)
    d2h = hout.numel() * hout.element_size()

    def e2e_step():
        d_stage.copy_(h_stage, non_blocking=True)
        if has_store:
            pa.store_kvcache(dk, dv, k_cache, v_cache, ds, head_major=HM)
        decode_call(dq, dbt, dcl)
        hout.copy_(out, non_blocking=True)

    for _ in range(args.warmup):
        flush.zero_()
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(args.steps):
        flush.zero_()
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        e2e_step()
        b_.record(stream)
        b_.synchronize()
        e2e_ms.append(a_.elapsed_time(b_))
    e2e = max_over_ranks(sum(e2e_ms) / len(e2e_ms), world)
    torch.cuda.synchronize()
    if not torch.equal(hout.view(torch.int16), out.cpu().view(torch.int16)):
        raise SystemExit("e2e output differs from the device-resident output")

    # ---- the same two steps replayed from CUDA graphs (one launch per step)
    def time_replay(g):
        for _ in range(args.warmup):
            flush.zero_()
            g.replay()
        torch.cuda.synchronize()
        t = []
        for _ in range(args.steps):
            flush.zero_()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            g.replay()
            b_.record(stream)
            b_.synchronize()
            t.append(a_.elapsed_time(b_))
        return max_over_ranks(sum(t) / len(t), world)

    def time_graphs():
        g_dev = pa.DecodeStepGraph(q, k_cache, v_cache, bt, cl, wl.scale, k_new=k_new, v_new=v_new,
                                   slot_mapping=slots if has_store else None, out=out,
                                   head_major=HM)
        graph_ms = time_replay(g_dev)
        g_e2e = pa.DecodeStepGraph(dq, k_cache, v_cache, dbt, dcl, wl.scale, k_new=dk, v_new=dv,
                                   slot_mapping=ds if has_store else None, out=out,
                                   host_stage=h_stage, device_stage=d_stage, host_out=hout,
                                   head_major=HM)
        graph_e2e_ms = time_replay(g_e2e)
        torch.cuda.synchronize()
        if not torch.equal(hout.view(torch.int16), out.cpu().view(torch.int16)):
            raise SystemExit("graph e2e output differs from the device-resident output")
        return graph_ms, graph_e2e_ms

    graph_ms = graph_e2e_ms = float("nan")
    if Q == 1:
        graph_ms, graph_e2e_ms = time_graphs()

    if rank != 0:
        return
    kv_bytes = wl.kv_bytes()
    peak, peak_src = measured_peaks()
    achieved = kv_bytes / (dec_avg * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": ms * 1e3, "unit": "us/step", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": dict(workload_config(wl), q_len=Q, layout=args.layout),
        "store_us": store_avg * 1e3, "decode_us": dec_avg * 1e3,
        "median_us_per_step": statistics.median(step_ms) * 1e3,
        "warm_us_per_step": warm_avg * 1e3,
        # store bandwidth: K and V rows read and written, plus the slots read
        "store_gbs": (4 * int((wl.slot_mapping >= 0).sum()) * Hkv * D * 2 + 8 * int(wl.slot_mapping.shape[0]))
                     / (store_avg * 1e-3) / 1e9 if has_store and store_avg > 0 else None,
        "kv_read_gbs": achieved, "hbm_frac": achieved / peak,
        "unique_kv_read_gbs": wl.unique_kv_bytes() / (dec_avg * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": ncu_traffic(wl.spec.name) if Q == 1 and not HM else None,
                     "kernel": "pa_decode (decode + combine launches)",
                     "algorithmic_bytes": kv_bytes, "peak_source": f"{peak_src} hbm_gbs"},
        "e2e": {"value": e2e * 1e3, "unit": "us/step", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "graph": {"us_per_step": graph_ms * 1e3 if Q == 1 else None,
                  "e2e_us_per_step": graph_e2e_ms * 1e3 if Q == 1 else None,
                  "note": "store + decode (and, for e2e, the H2D and D2H copies) captured "
                          "in one CUDA graph, one replay per step"},
        "gpu_launches": args.steps * (3 if has_store else 2),
        "timing": "value: store + decode back to back per step; store_us / decode_us: a "
                  "second pass with an event between the two calls",
        "clocks": clk,
    }
    if not args.no_cpu_baseline and world >= 1:
        us, threads, sample = oracle_sample(wl, args.cpu_seconds)
        line["cpu_baseline"] = {"value": us, "unit": "us/step", "cores": threads,
                                "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)


def prefill_flops(pb) -> int:
    """Algorithmic FLOPs of one prefill launch: per causal (row, key) pair and
    query head, a 128-long dot product for the score and a 128-long
    multiply-add of V, 2 * 128 FLOPs each."""
    return 4 * pb.wl.spec.head_dim * pb.wl.spec.num_q_heads * pb.causal_pairs()


def prefill_config(pb, chunk):
    c = workload_config(pb.wl)
    c.update(store_rows=int(pb.slot_mapping.shape[0]), query_rows=int(pb.query_start_loc[-1]),
             max_query_len=pb.max_query_len, chunk="whole prompt" if chunk is None else chunk,
             causal_pairs=pb.causal_pairs())
    return c


def prefill_oracle_sample(pb, target_s: float, host=None):
    """Time the fp64 oracle on random rows of the prefill step (each row as a
    one-row chunk of its sequence cut at its causal limit) and scale by causal
    (row, key) pairs to the whole step, plus the oracle store of all chunk rows.
    Returns (us_per_step, threads, sample description)."""
    import oracle
    O = oracle.get()
    threads = O.num_threads()
    if host is None:
        host = (pb.wl.k_cache, pb.wl.v_cache)
    kc, vc = oracle._bits(host[0]).copy(), oracle._bits(host[1]).copy()
    t0 = time.perf_counter()
    O.store_kvcache_into(pb.k_new, pb.v_new, kc, vc, pb.slot_mapping)
    t_store = time.perf_counter() - t0
    qsl = pb.query_start_loc
    T = int(qsl[-1])
    seq_of = np.searchsorted(qsl, np.arange(T), side="right") - 1
    n = np.diff(qsl)[seq_of]
    cut = (pb.wl.context_lens[seq_of].astype(np.int64) - n + (np.arange(T) - qsl[seq_of]) + 1)
    rng = np.random.Generator(np.random.PCG64(321))
    order = rng.permutation(T)
    done, done_pairs, elapsed, batch = 0, 0, 0.0, max(threads, 4)
    while elapsed < target_s:
        idx = order[done % T:done % T + batch]
        t0 = time.perf_counter()
        O.prefill(pb.q[torch.from_numpy(idx)], kc, vc, pb.wl.block_tables[seq_of[idx]],
                  cut[idx].astype(np.int32), np.arange(len(idx) + 1, dtype=np.int32),
                  pb.wl.scale)
        elapsed += time.perf_counter() - t0
        done += len(idx)
        done_pairs += int(cut[idx].sum())
        batch = min(batch * 2, 1024)
    us = (t_store + elapsed * pb.causal_pairs() / max(done_pairs, 1)) * 1e6
    sample = (f"oracle store of all {T} chunk rows + {done} random query rows (all "
              f"{pb.wl.spec.num_q_heads} heads) out of {T} ({elapsed:.1f} s of oracle time), "
              f"scaled by causal (row, key) pairs to one full step")
    return us, threads, sample


def prefill_spec(args):
    spec, chunk = inputs.PREFILL_SPECS[args.workload]
    if args.num_seqs:
        spec = inputs.scaled(spec, num_seqs=args.num_seqs, name=f"{spec.name}_s{args.num_seqs}")
    return spec, chunk


def run_reference_prefill(args, rank, world):
    if rank != 0:
        return
    spec, chunk = prefill_spec(args)
    pb = inputs.prefill_batch(spec, seed=0, chunk=chunk)
    per_step = max(0.05, args.ref_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        prefill_oracle_sample(pb, per_step)
    vals = []
    for _ in range(args.steps):
        us, threads, sample = prefill_oracle_sample(pb, per_step)
        vals.append(us)
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": PREFILL_METRIC, "value": v, "unit": "us/step",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": prefill_config(pb, chunk),
            "cpu_baseline": {"value": v, "unit": "us/step", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gpu_prefill(args, rank, world, local):
    """One prefill step: store of every chunk row's K/V, then paged prefill."""
    from paged_kv_cache_255_gb300 import pagedattn as pa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec, chunk = prefill_spec(args)
    pb = inputs.prefill_batch(spec, seed=0, chunk=chunk)
    wl = pb.wl
    k_cache, v_cache = wl.k_cache.to(dev), wl.v_cache.to(dev)
    HM = args.layout == "head_major"
    if HM:          # the same values in a [NB, Hkv, bs, D] pool
        k_cache = k_cache.permute(0, 2, 1, 3).contiguous()
        v_cache = v_cache.permute(0, 2, 1, 3).contiguous()
    host_inputs = [pb.q, pb.k_new, pb.v_new, torch.from_numpy(pb.slot_mapping),
                   torch.from_numpy(wl.block_tables), torch.from_numpy(wl.context_lens),
                   torch.from_numpy(pb.query_start_loc)]
    q, k_new, v_new, slots, bt, cl, qsl = [t.to(dev) for t in host_inputs]
    out = torch.empty_like(q)
    mql = pb.max_query_len
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(q_, kn_, vn_, sl_, bt_, cl_, qsl_):
        pa.store_kvcache(kn_, vn_, k_cache, v_cache, sl_, head_major=HM)
        pa.prefill(q_, k_cache, v_cache, bt_, cl_, qsl_, wl.scale, max_query_len=mql, out=out,
                   head_major=HM)

    clocks = ClockSampler(local)
    clocks.wait_first_sample()
    for _ in range(args.warmup):
        flush.zero_()
        step(q, k_new, v_new, slots, bt, cl, qsl)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        pa.store_kvcache(k_new, v_new, k_cache, v_cache, slots, head_major=HM)
        ev[i][1].record(stream)
        pa.prefill(q, k_cache, v_cache, bt, cl, qsl, wl.scale, max_query_len=mql, out=out,
                   head_major=HM)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    step_ms = max_over_ranks(statistics.mean(e[0].elapsed_time(e[2]) for e in ev), world)
    store_ms = max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in ev), world)
    pf_ms = max_over_ranks(statistics.mean(e[1].elapsed_time(e[2]) for e in ev), world)

    # end to end: pinned host inputs packed in one staging buffer, one H2D,
    # the step, the output read back
    offs, total = [], 0
    for t in host_inputs:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_stage = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    for t, o in zip(host_inputs, offs):
        nb = t.numel() * t.element_size()
        h_stage[o:o + nb].copy_(t.contiguous().view(-1).view(torch.uint8))
    d_stage = torch.empty(total, dtype=torch.uint8, device=dev)
    views = [d_stage[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
             for t, o in zip(host_inputs, offs)]
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_inputs)
    d2h = hout.numel() * hout.element_size()

    def e2e_step():
        d_stage.copy_(h_stage, non_blocking=True)
        step(*views)
        hout.copy_(out, non_blocking=True)

    for _ in range(args.warmup):
        flush.zero_()
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(args.steps):
        flush.zero_()
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        e2e_step()
        b_.record(stream)
        b_.synchronize()
        e2e_ms.append(a_.elapsed_time(b_))
    e2e = max_over_ranks(statistics.mean(e2e_ms), world)
    torch.cuda.synchronize()
    if not torch.equal(hout.view(torch.int16), out.cpu().view(torch.int16)):
        raise SystemExit("e2e output differs from the device-resident output")
    if rank != 0:
        return
    flops = prefill_flops(pb)
    peak, peak_src = measured_peaks("bf16_tflops")
    achieved = flops / (pf_ms * 1e-3) / 1e12
    line = {
        "metric": PREFILL_METRIC, "value": step_ms * 1e3, "unit": "us/step", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": dict(prefill_config(pb, chunk), layout=args.layout),
        "store_us": store_ms * 1e3, "prefill_us": pf_ms * 1e3,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None, "kernel": "pa_prefill",
                     "algorithmic_flops": flops,
                     "peak_source": f"{peak_src} bf16_tflops (burst)"},
        "e2e": {"value": e2e * 1e3, "unit": "us/step", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * 2,
        "timing": "value: store + prefill per step, events between the two calls",
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        us, threads, sample = prefill_oracle_sample(pb, args.cpu_seconds)
        line["cpu_baseline"] = {"value": us, "unit": "us/step", "cores": threads,
                                "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(inputs.SPECS) + sorted(inputs.PREFILL_SPECS),
                    help="a decode step, or a prefill step (%s)" % ", ".join(inputs.PREFILL_SPECS))
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="run a copy of the workload with this many sequences (profiling)")
    ap.add_argument("--q-len", type=int, default=1,
                    help="query tokens per sequence (speculative verification); 1 = decode")
    ap.add_argument("--layout", default="token_major", choices=["token_major", "head_major"],
                    help="KV pool layout: [NB, bs, Hkv, D] or [NB, Hkv, bs, D]")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_setup(args.gpus)
    prefill = args.workload in inputs.PREFILL_SPECS
    if args.impl == "reference":
        (run_reference_prefill if prefill else run_reference)(args, rank, world)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA device")
        (run_gpu_prefill if prefill else run_gpu)(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
