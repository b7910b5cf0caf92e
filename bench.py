"""Benchmark: one paged decode step (store_kvcache of the step's new K/V rows,
then decode attention) on synthetic inputs, timed with CUDA events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0). ``value`` is microseconds per step (store +
decode, inputs resident in HBM) on the headline workload: the skewed
long-context decode step (8 sequences of 32k-131k tokens among 120 short
ones, 32 q / 8 KV heads), the largest of the decode steps. Its 2.3 GB of K/V
reads are 18x the L2, so its steps run back to back (inputs larger than L2);
steps that read less than 8x the L2 are preceded by an L2 flush (a 512 MiB
write). ``l2_alt`` repeats each decode step in the other mode: the large
steps flushed, the others warm (no flush: inputs near or below the L2 size
then partly stay in it, so it gives no DRAM fraction).
``roofline`` reports the decode launch's KV-read bandwidth against the
measured HBM copy peak; ``e2e`` repeats the step through host buffers (pinned
H2D of the step's inputs and D2H of its output inside the timed region);
``cpu_baseline`` times the fp64 CPU oracle on the whole step, on one thread
and on all host cores. ``workloads`` holds the other decode steps and the two
prefill steps, each timed the same way (store + call; the prefill steps
always with the L2 flushed) with its own roofline fraction. ``--impl reference`` times only the
oracle (the reference arm). With N > 1 (torchrun) every rank runs its own
replica of the step on its own GPU: the path has no cross-GPU exchange.
"""
from __future__ import annotations

import argparse
import dataclasses
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_255_gb300 import inputs  # noqa: E402

METRIC = "paged-decode µs/step and KV-read GB/s (fraction of GB300 HBM peak)"
DEFAULT_WORKLOAD = "long_context"
# decode and prefill steps measured beside the headline (sub-records): name ->
# (workload, query tokens per sequence, pool layout)
SUB_DECODE = {
    "large_batch": ("large_batch", 1, "token_major"),
    "qwen3_0_6b": ("qwen3_0_6b", 1, "token_major"),
    "qwen3_0_6b_bs256": ("qwen3_0_6b_bs256", 1, "token_major"),
    "prefix_shared": ("prefix_shared", 1, "token_major"),
    "tiny": ("tiny", 1, "token_major"),
    # multi-token decode: 4 new tokens per sequence (speculative verification)
    "qwen3_0_6b_q4": ("qwen3_0_6b", 4, "token_major"),
    # the headline step on a head-major pool [NB, Hkv, bs, D]
    "long_context_head_major": ("long_context", 1, "head_major"),
}
SUB_PREFILL = ["chunked_8b", "qwen3_0_6b_prompts"]
L2_BYTES = 129_000_000           # GB300 L2
L2_FLUSH_BYTES = 512 << 20       # > 2x the L2
# A decode step whose K/V reads are at least this many times the L2 runs its
# timed steps back to back (inputs larger than L2: each step streams them
# through L2 many times over, so nothing of one step is left for the next);
# smaller steps get the L2 flush before each step. The flush is a write, and
# the lines it leaves dirty are written back to HBM during the next step.
LARGE_INPUT_FACTOR = 8
L2_FLUSHED = "flushed between steps (512 MiB write)"
# GPU spin before a step that is not preceded by the flush (about 100 us at
# 2 GHz, as long as the flush): the host queues the step meanwhile, so the
# events do not time the host's launch calls
SPIN_CYCLES = 200_000
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# comparison kernels selectable with --variant: name -> pagedattn flag
VARIANTS = {"decode_simt": "VARIANT_DECODE_SIMT", "prefill_mma": "VARIANT_PREFILL_MMA"}
PREFILL_METRIC = "paged-prefill µs/step and attention TFLOP/s (fraction of GB300 bf16 tensor peak)"
PROFILE_FILE = os.path.join(ROOT, "profiles", "decode_traffic.txt")
KERNEL_SOURCES = ["paged_kv_cache_255_gb300/csrc/decode.cu", "paged_kv_cache_255_gb300/csrc/common.cuh"]
PREFILL_SOURCES = ["paged_kv_cache_255_gb300/csrc/prefill_tc.cu",
                   "paged_kv_cache_255_gb300/csrc/tcgen05.cuh",
                   "paged_kv_cache_255_gb300/csrc/common.cuh"]
# a whole oracle step is timed unless one all-cores step would take longer
# than this; then a sample of the step's outputs is timed and scaled
FULL_STEP_LIMIT_S = 30.0


def kernel_hash(sources=KERNEL_SOURCES) -> str:
    """Hash of a kernel's code, by default the decode kernel's (comments and
    whitespace removed, so that an edited comment does not invalidate
    counters taken on the same code)."""
    h = hashlib.sha256()
    for p in sources:
        with open(os.path.join(ROOT, p)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def measured_peaks(key="hbm_gbs"):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS}[key], "fallback"


def ncu_traffic(workload: str, sources=KERNEL_SOURCES):
    """DRAM bytes per launch of the kernel built from `sources` (the decode
    kernel by default) from the committed ncu summary, if it was taken on this
    workload key with the current kernel source."""
    try:
        text = open(PROFILE_FILE).read()
    except OSError:
        return None
    want = kernel_hash(sources)
    for m in re.finditer(r"^traffic\s+workload=(\S+)\s+kernel_hash=(\S+)\s+bytes_per_launch=(\d+)",
                         text, re.M):
        if m.group(1) == workload and m.group(2) == want:
            return int(m.group(3))
    return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the GPU is busy."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "utilization.gpu",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

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
                rows.append((float(parts[1]), float(parts[2]), float(parts[4]), parts[5:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "samples_under_load": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        # samples taken while a kernel was running; the median clock is taken
        # over those when there are any
        busy = [r for r in rows if r[2] > 0]
        use = busy or rows
        reasons = sorted({names[i] for _, _, _, flags in use for i, f in enumerate(flags)
                          if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in use),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons, "samples": len(rows),
                "samples_under_load": len(busy)}


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


def large_inputs(wl) -> bool:
    """The decode step's distinct K/V bytes (a shared prefix counted once) are
    at least LARGE_INPUT_FACTOR times the L2."""
    return wl.unique_kv_bytes() >= LARGE_INPUT_FACTOR * L2_BYTES


def l2_note(wl) -> str:
    if large_inputs(wl):
        return (f"not flushed: inputs larger than L2 (the step reads "
                f"{wl.unique_kv_bytes() / L2_BYTES:.0f}x the 129 MB L2 in distinct K/V bytes)")
    return L2_FLUSHED


def between_steps(flush):
    """Queue what precedes each timed step: the L2 flush, or (flush None) a
    GPU spin of about the same length."""
    if flush is None:
        torch.cuda._sleep(SPIN_CYCLES)
    else:
        flush.zero_()


def workload_config(wl, q_len=1, layout="token_major"):
    s = wl.spec
    return {"workload": s.name, "num_seqs": wl.num_seqs, "num_q_heads": s.num_q_heads,
            "num_kv_heads": s.num_kv_heads, "head_dim": s.head_dim, "block_size": s.block_size,
            "num_blocks": wl.num_blocks, "store_rows": int(wl.slot_mapping.shape[0]),
            "context_tokens": int(wl.context_lens.astype(np.int64).sum()),
            "max_context_len": wl.max_context_len, "seed": wl.seed, "l2": l2_note(wl),
            "q_len": q_len, "layout": layout}


# ---------------------------------------------------------------------------
# the fp64 oracle on the host cores (cpu_baseline and the reference arm)

def host_copies(wl):
    return (wl.q.cpu(), wl.k_cache.cpu(), wl.v_cache.cpu(), wl.k_new.cpu(), wl.v_new.cpu())


def oracle_full_step(wl, host, threads: int):
    """One whole decode step on the oracle: the store of every new row into
    private copies of the pools (the copies are not timed), then every
    (sequence, query head) output. Returns (seconds, threads used)."""
    import oracle
    O = oracle.get()
    q, kc, vc, kn, vn = host
    kb, vb = oracle._bits(kc), oracle._bits(vc)
    t_store = 0.0
    if wl.slot_mapping.shape[0]:
        kb, vb = kb.copy(), vb.copy()
        t0 = time.perf_counter()
        O.store_kvcache_into(kn, vn, kb, vb, wl.slot_mapping)
        t_store = time.perf_counter() - t0
    t0 = time.perf_counter()
    O.decode(q, kb, vb, wl.block_tables, wl.context_lens, wl.scale, threads=threads)
    return t_store + time.perf_counter() - t0, (threads if threads > 0 else O.num_threads())


def oracle_sampled_step(wl, host, target_s: float, threads: int):
    """A bounded sample for steps too big to time whole: random (sequence,
    head) outputs until target_s of oracle time, scaled by context tokens to
    the whole step; the store is timed whole. Returns (seconds, threads, pairs)."""
    import oracle
    O = oracle.get()
    q, kc, vc, kn, vn = host
    kb, vb = oracle._bits(kc), oracle._bits(vc)
    t_store = 0.0
    if wl.slot_mapping.shape[0]:
        kb, vb = kb.copy(), vb.copy()
        t0 = time.perf_counter()
        O.store_kvcache_into(kn, vn, kb, vb, wl.slot_mapping)
        t_store = time.perf_counter() - t0
    S, Hq = wl.num_seqs, wl.spec.num_q_heads
    work_all = float(wl.context_lens.astype(np.float64).sum()) * Hq
    order = np.random.Generator(np.random.PCG64(123)).permutation(S * Hq)
    done, work, elapsed, batch = 0, 0.0, 0.0, 64
    while elapsed < target_s and done < S * Hq:
        idx = order[done:done + batch]
        pairs = np.stack([idx // Hq, idx % Hq], 1).astype(np.int32)
        t0 = time.perf_counter()
        O.decode_pairs(q, kb, vb, wl.block_tables, wl.context_lens, wl.scale, pairs,
                       threads=threads)
        elapsed += time.perf_counter() - t0
        done += len(idx)
        work += float(wl.context_lens[idx // Hq].astype(np.float64).sum())
        batch = min(batch * 2, 4096)
    used = threads if threads > 0 else O.num_threads()
    return t_store + elapsed * work_all / max(work, 1.0), used, done


def cpu_baseline(wl, host=None):
    """The oracle timed on the whole step, on one thread and on all host
    cores (median of three all-cores steps)."""
    if host is None:
        host = host_copies(wl)
    t_all = [oracle_full_step(wl, host, 0) for _ in range(3)]
    all_s, cores = statistics.median(t for t, _ in t_all), t_all[0][1]
    S, Hq = wl.num_seqs, wl.spec.num_q_heads
    what = (f"full step: oracle store of all {int(wl.slot_mapping.shape[0])} new rows + all "
            f"{S * Hq} (sequence, query head) outputs")
    if all_s * cores <= FULL_STEP_LIMIT_S:
        one_s, _ = oracle_full_step(wl, host, 1)
        one_what = what
    else:      # one thread would take too long: time a sample of the step
        one_s, _, n = oracle_sampled_step(wl, host, 15.0, 1)
        one_what = (f"store of all rows + {n} random (sequence, query head) outputs of "
                    f"{S * Hq}, scaled by context tokens to the full step")
    return {"value": all_s * 1e6, "unit": "us/step", "cores": cores, "kind": "oracle",
            "sample": what,
            "all_cores": {"value": all_s * 1e6, "cores": cores, "sample": what},
            "single_thread": {"value": one_s * 1e6, "cores": 1, "sample": one_what}}


def workload_spec(args, name=None):
    spec = inputs.SPECS[name or args.workload]
    if args.num_seqs:
        spec = inputs.scaled(spec, num_seqs=args.num_seqs, name=f"{spec.name}_s{args.num_seqs}")
    return spec


def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = inputs.generate(workload_spec(args), seed=0,
                         device="cuda" if torch.cuda.is_available() else "cpu")
    host = host_copies(wl)
    # each step is one whole oracle step on all host cores, unless that would
    # take the run past --ref-seconds; then each step times a sample
    t_first, threads = oracle_full_step(wl, host, 0)
    budget = max(0.05, args.ref_seconds / max(1, args.steps + args.warmup))
    whole = t_first <= max(budget, FULL_STEP_LIMIT_S / max(1, args.steps + args.warmup))
    S, Hq = wl.num_seqs, wl.spec.num_q_heads

    def one():
        if whole:
            t, _ = oracle_full_step(wl, host, 0)
            return t, (f"full step: oracle store of all {int(wl.slot_mapping.shape[0])} new "
                       f"rows + all {S * Hq} (sequence, query head) outputs")
        t, _, n = oracle_sampled_step(wl, host, budget, 0)
        return t, (f"oracle store of all rows + {n} random (sequence, query head) outputs of "
                   f"{S * Hq}, scaled by context tokens to the full step")

    for _ in range(max(0, args.warmup - 1)):
        one()
    vals, sample = [], ""
    for _ in range(args.steps):
        t, sample = one()
        vals.append(t * 1e6)
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "us/step",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(wl, args.q_len, args.layout),
            "cpu_baseline": {"value": v, "unit": "us/step", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm: decode steps

class DecodeStep:
    """Device buffers and calls of one decode step (store, then decode)."""

    def __init__(self, wl, dev, layout="token_major", q_len=1):
        from paged_kv_cache_255_gb300 import pagedattn as pa
        self.pa, self.wl, self.dev = pa, wl, dev
        s = wl.spec
        self.HM = layout == "head_major"
        self.Q = q_len
        self.k_cache, self.v_cache = wl.k_cache, wl.v_cache
        if self.HM:          # the same values in a [NB, Hkv, bs, D] pool
            self.k_cache = self.k_cache.permute(0, 2, 1, 3).contiguous()
            self.v_cache = self.v_cache.permute(0, 2, 1, 3).contiguous()
            if q_len > 1:
                raise SystemExit("--q-len > 1 runs on the token-major layout only")
        self.q = wl.q
        if q_len > 1:
            # q_len query tokens per sequence (speculative verification)
            gq = torch.Generator(device=dev)
            gq.manual_seed(1)
            self.q = torch.randn((wl.num_seqs, q_len, s.num_q_heads, s.head_dim), generator=gq,
                                 device=dev).to(torch.bfloat16)
        self.k_new, self.v_new = wl.k_new, wl.v_new
        self.slots = torch.from_numpy(wl.slot_mapping).to(dev)
        self.bt = torch.from_numpy(wl.block_tables).to(dev)
        self.cl = torch.from_numpy(wl.context_lens).to(dev)
        self.out = torch.empty_like(self.q)
        self.ws = pa.workspace_for(s.num_q_heads, s.num_kv_heads, s.head_dim, 0, dev)
        self.has_store = self.slots.shape[0] > 0

    def store(self, kn=None, vn=None, sl=None):
        if self.has_store:
            self.pa.store_kvcache(self.k_new if kn is None else kn, self.v_new if vn is None else vn,
                                  self.k_cache, self.v_cache, self.slots if sl is None else sl,
                                  head_major=self.HM)

    def decode(self, q=None, bt=None, cl=None):
        q = self.q if q is None else q
        bt = self.bt if bt is None else bt
        cl = self.cl if cl is None else cl
        if self.Q > 1:
            return self.pa.decode_multi(q, self.k_cache, self.v_cache, bt, cl, self.wl.scale,
                                        out=self.out)
        return self.pa.decode(q, self.k_cache, self.v_cache, bt, cl, self.wl.scale, out=self.out,
                              workspace=self.ws, head_major=self.HM)

    def step(self, kn=None, vn=None, sl=None, q=None, bt=None, cl=None):
        """Store + decode in one call (pa_decode_step; decode alone when the
        step stores nothing)."""
        if not self.has_store or self.Q > 1:
            self.store(kn, vn, sl)
            return self.decode(q, bt, cl)
        return self.pa.decode_step(self.k_new if kn is None else kn,
                                   self.v_new if vn is None else vn,
                                   self.slots if sl is None else sl, self.q if q is None else q,
                                   self.k_cache, self.v_cache, self.bt if bt is None else bt,
                                   self.cl if cl is None else cl, self.wl.scale, out=self.out,
                                   workspace=self.ws, head_major=self.HM)

    def launches_per_step(self):
        return 3 if self.has_store else 2


def time_decode(st: DecodeStep, flush, stream, steps, warmup, world):
    """Store + decode per step, each step preceded by the L2 flush (or, with
    flush None, by a GPU spin): one pass through the one-call step (the step
    time) and one with an event between separate store and decode calls (the
    split). Returns milliseconds (max over ranks) and the step times."""
    for _ in range(warmup):
        between_steps(flush)
        st.step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        between_steps(flush)
        ev[i][0].record(stream)
        st.step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    ms = max_over_ranks(sum(step_ms) / len(step_ms), world)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        between_steps(flush)
        ev[i][0].record(stream)
        st.store()
        ev[i][1].record(stream)
        st.decode()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    store_ms = [e[0].elapsed_time(e[1]) for e in ev]
    dec_ms = [e[1].elapsed_time(e[2]) for e in ev]
    return {"ms": ms, "step_ms": step_ms,
            "decode_ms": max_over_ranks(sum(dec_ms) / len(dec_ms), world),
            "store_ms": max_over_ranks(sum(store_ms) / len(store_ms), world)}


def traffic_key(st: DecodeStep) -> str:
    """Workload key of a decode step's line in the traffic summary."""
    return (st.wl.spec.name + ("_head_major" if st.HM else "")
            + (f"_q{st.Q}" if st.Q > 1 else ""))


def decode_rates(st: DecodeStep, t):
    """Bandwidth figures of a timed decode step."""
    wl = st.wl
    s = wl.spec
    kv_bytes = wl.kv_bytes()
    peak, peak_src = measured_peaks()
    dec_s = t["decode_ms"] * 1e-3
    achieved = kv_bytes / dec_s / 1e9
    n_valid = int((wl.slot_mapping >= 0).sum())
    store_bytes = 4 * n_valid * s.num_kv_heads * s.head_dim * 2 + 8 * int(wl.slot_mapping.shape[0])
    return {
        "us_per_step": t["ms"] * 1e3, "store_us": t["store_ms"] * 1e3,
        "decode_us": t["decode_ms"] * 1e3,
        "median_us_per_step": statistics.median(t["step_ms"]) * 1e3,
        # store bandwidth: K and V rows read and written, plus the slots read
        "store_gbs": store_bytes / (t["store_ms"] * 1e-3) / 1e9
        if st.has_store and t["store_ms"] > 0 else None,
        "kv_read_gbs": achieved, "hbm_frac": achieved / peak,
        "unique_kv_read_gbs": wl.unique_kv_bytes() / dec_s / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": ncu_traffic(traffic_key(st)),
                     "kernel": "pa_decode (decode + combine launches)",
                     "algorithmic_bytes": kv_bytes, "peak_source": f"{peak_src} hbm_gbs"},
    }


def l2_alt_record(st: DecodeStep, t, flushed: bool):
    """The step timed in the other L2 mode than its own (see l2_note)."""
    r = decode_rates(st, t)
    return {"l2": L2_FLUSHED if flushed else
            "not flushed (inputs at or below a few times the L2 partly stay there)",
            "us_per_step": r["us_per_step"], "decode_us": r["decode_us"],
            "hbm_frac": r["hbm_frac"] if flushed else None}


def decode_sub_record(name, args, dev, flush, stream, world):
    workload, q_len, layout = SUB_DECODE[name]
    wl = inputs.generate(workload_spec(args, workload), seed=0, device=dev)
    st = DecodeStep(wl, dev, layout, q_len)
    big = large_inputs(wl)
    t = time_decode(st, None if big else flush, stream, args.steps, args.warmup, world)
    rec = {"config": workload_config(wl, q_len, layout), **decode_rates(st, t),
           "gpu_launches": args.steps * st.launches_per_step()}
    # the other L2 mode beside it: flushed for large inputs, warm for the rest
    rec["l2_alt"] = l2_alt_record(
        st, time_decode(st, flush if big else None, stream, args.steps, args.warmup, world), big)
    del st, wl
    torch.cuda.empty_cache()
    return rec


def run_gpu(args, rank, world, local):
    from paged_kv_cache_255_gb300 import pagedattn as pa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = inputs.generate(workload_spec(args), seed=0, device=dev)
    st = DecodeStep(wl, dev, args.layout, args.q_len)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # the clock sampler runs from before the first warm-up step to after the
    # last timed pass (sub-records included)
    clocks = ClockSampler(local)
    clocks.wait_first_sample()

    # ---- device-resident timing: store then decode back to back, as a user
    # issues them (the decode launch may overlap the store's tail). A step
    # whose inputs are many times the L2 runs without the flush (l2_note);
    # every other pass below takes the same mode.
    fl = None if large_inputs(wl) else flush
    t = time_decode(st, fl, stream, args.steps, args.warmup, world)
    # ---- the same in the other mode: flushed for large inputs, else warm
    # (not flushed; informative, not the reported value)
    t_alt = time_decode(st, flush if fl is None else None, stream, args.steps, args.warmup,
                        world)

    # ---- end to end through host buffers: the step's inputs are packed in one
    # pinned staging buffer, copied in one transfer, and the output read back
    host_inputs = [st.q, st.k_new, st.v_new, st.slots, st.bt, st.cl]
    offs, total = [], 0
    for x in host_inputs:
        offs.append(total)
        total += (x.numel() * x.element_size() + 255) // 256 * 256
    h_stage = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    for x, o in zip(host_inputs, offs):
        n = x.numel() * x.element_size()
        h_stage[o:o + n].copy_(x.contiguous().view(-1).view(torch.uint8).cpu())
    d_stage = torch.empty(total, dtype=torch.uint8, device=dev)
    views = [d_stage[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape)
             for x, o in zip(host_inputs, offs)]
    dq, dk, dv, ds, dbt, dcl = views
    hout = torch.empty(st.out.shape, dtype=st.out.dtype, pin_memory=True)
    h2d = sum(x.numel() * x.element_size() for x in host_inputs)
    d2h = hout.numel() * hout.element_size()

    def e2e_step():
        d_stage.copy_(h_stage, non_blocking=True)
        st.step(dk, dv, ds, dq, dbt, dcl)
        hout.copy_(st.out, non_blocking=True)

    for _ in range(args.warmup):
        between_steps(fl)
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(args.steps):
        between_steps(fl)
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        e2e_step()
        b_.record(stream)
        b_.synchronize()
        e2e_ms.append(a_.elapsed_time(b_))
    e2e = max_over_ranks(sum(e2e_ms) / len(e2e_ms), world)
    torch.cuda.synchronize()
    if not torch.equal(hout.view(torch.int16), st.out.cpu().view(torch.int16)):
        raise SystemExit("e2e output differs from the device-resident output")

    # ---- the same two steps replayed from CUDA graphs (one launch per step)
    def time_replay(g):
        for _ in range(args.warmup):
            between_steps(fl)
            g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(args.steps):
            between_steps(fl)
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            g.replay()
            b_.record(stream)
            b_.synchronize()
            ts.append(a_.elapsed_time(b_))
        return max_over_ranks(sum(ts) / len(ts), world)

    graph_ms = graph_e2e_ms = float("nan")
    if st.Q == 1:
        sl = st.slots if st.has_store else None
        g_dev = pa.DecodeStepGraph(st.q, st.k_cache, st.v_cache, st.bt, st.cl, wl.scale,
                                   k_new=st.k_new, v_new=st.v_new, slot_mapping=sl, out=st.out,
                                   head_major=st.HM)
        graph_ms = time_replay(g_dev)
        g_e2e = pa.DecodeStepGraph(dq, st.k_cache, st.v_cache, dbt, dcl, wl.scale, k_new=dk,
                                   v_new=dv, slot_mapping=ds if st.has_store else None,
                                   out=st.out, host_stage=h_stage, device_stage=d_stage,
                                   host_out=hout, head_major=st.HM)
        graph_e2e_ms = time_replay(g_e2e)
        torch.cuda.synchronize()
        if not torch.equal(hout.view(torch.int16), st.out.cpu().view(torch.int16)):
            raise SystemExit("graph e2e output differs from the device-resident output")
        del g_dev, g_e2e

    host = host_copies(wl) if rank == 0 and not args.no_cpu_baseline else None
    # the step's structure (lengths, tables, slots) for the CPU baseline; its
    # values are in the host copies, and the device pools are freed below
    wl_struct = dataclasses.replace(wl, q=None, k_new=None, v_new=None, k_cache=None,
                                    v_cache=None)
    rates = decode_rates(st, t)
    alt_rec = l2_alt_record(st, t_alt, fl is None)
    config = workload_config(wl, st.Q, args.layout)
    launches = args.steps * st.launches_per_step()
    del st, wl, views, dq, dk, dv, ds, dbt, dcl, d_stage
    torch.cuda.empty_cache()

    # ---- the other decode steps and the prefill steps, timed the same way
    subs = {}
    if not args.no_sub_records:
        for name, (workload, q_len, layout) in SUB_DECODE.items():
            if (workload, q_len, layout) != (args.workload, args.q_len, args.layout):
                subs[name] = decode_sub_record(name, args, dev, flush, stream, world)
        for name in SUB_PREFILL:
            subs[name] = prefill_sub_record(name, args, dev, flush, stream, world)
    clk = clocks.stop()

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": rates["us_per_step"], "unit": "us/step", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t["ms"],
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config,
        **{k: v for k, v in rates.items() if k != "us_per_step"},
        "l2_alt": alt_rec,
        "e2e": {"value": e2e * 1e3, "unit": "us/step", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "graph": {"us_per_step": graph_ms * 1e3 if args.q_len == 1 else None,
                  "e2e_us_per_step": graph_e2e_ms * 1e3 if args.q_len == 1 else None,
                  "note": "store + decode (and, for e2e, the H2D and D2H copies) captured "
                          "in one CUDA graph, one replay per step"},
        "gpu_launches": launches,
        "timing": "value: one pa_decode_step call (store, then decode) per step; store_us / "
                  "decode_us: a second pass with separate store and decode calls and an event "
                  "between them; config.l2: what precedes each timed step; l2_alt: the same "
                  "two passes in the other L2 mode; workloads: the same on each other step",
        "clocks": clk,
        "workloads": subs,
    }
    if args.variant:
        line["kernel_variant"] = args.variant
    if host is not None:
        line["cpu_baseline"] = cpu_baseline(wl_struct, host)
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm: prefill steps

def prefill_flops(pb) -> int:
    """Algorithmic FLOPs of one prefill launch: per causal (row, key) pair and
    query head, a 128-long dot product for the score and a 128-long
    multiply-add of V, 2 * 128 FLOPs each."""
    return 4 * pb.wl.spec.head_dim * pb.wl.spec.num_q_heads * pb.causal_pairs()


def prefill_config(pb, chunk, layout="token_major"):
    c = workload_config(pb.wl, 1, layout)
    c.pop("q_len")
    c["l2"] = L2_FLUSHED
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


def prefill_spec(args, name=None):
    spec, chunk = inputs.PREFILL_SPECS[name or args.workload]
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
            "data": "synthetic", "config": prefill_config(pb, chunk, args.layout),
            "cpu_baseline": {"value": v, "unit": "us/step", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


class PrefillStep:
    """Device buffers and calls of one prefill step (store of the chunk rows,
    then paged prefill)."""

    def __init__(self, pb, dev, layout="token_major"):
        from paged_kv_cache_255_gb300 import pagedattn as pa
        self.pa, self.pb = pa, pb
        wl = pb.wl
        self.k_cache, self.v_cache = wl.k_cache.to(dev), wl.v_cache.to(dev)
        self.HM = layout == "head_major"
        if self.HM:          # the same values in a [NB, Hkv, bs, D] pool
            self.k_cache = self.k_cache.permute(0, 2, 1, 3).contiguous()
            self.v_cache = self.v_cache.permute(0, 2, 1, 3).contiguous()
        self.host_inputs = [pb.q, pb.k_new, pb.v_new, torch.from_numpy(pb.slot_mapping),
                            torch.from_numpy(wl.block_tables), torch.from_numpy(wl.context_lens),
                            torch.from_numpy(pb.query_start_loc)]
        self.args = [t.to(dev) for t in self.host_inputs]
        self.out = torch.empty_like(self.args[0])
        self.mql = pb.max_query_len

    def store(self, kn, vn, sl):
        self.pa.store_kvcache(kn, vn, self.k_cache, self.v_cache, sl, head_major=self.HM)

    def prefill(self, q, bt, cl, qsl):
        self.pa.prefill(q, self.k_cache, self.v_cache, bt, cl, qsl, self.pb.wl.scale,
                        max_query_len=self.mql, out=self.out, head_major=self.HM)

    def step(self, q, kn, vn, sl, bt, cl, qsl):
        self.store(kn, vn, sl)
        self.prefill(q, bt, cl, qsl)


def time_prefill(ps: PrefillStep, flush, stream, steps, warmup, world):
    q, kn, vn, sl, bt, cl, qsl = ps.args
    for _ in range(warmup):
        flush.zero_()
        ps.step(*ps.args)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(stream)
        ps.store(kn, vn, sl)
        ev[i][1].record(stream)
        ps.prefill(q, bt, cl, qsl)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return {"ms": max_over_ranks(statistics.mean(e[0].elapsed_time(e[2]) for e in ev), world),
            "store_ms": max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in ev), world),
            "prefill_ms": max_over_ranks(statistics.mean(e[1].elapsed_time(e[2]) for e in ev), world)}


def prefill_rates(pb, t):
    flops = prefill_flops(pb)
    peak, peak_src = measured_peaks("bf16_tflops")
    achieved = flops / (t["prefill_ms"] * 1e-3) / 1e12
    return {"us_per_step": t["ms"] * 1e3, "store_us": t["store_ms"] * 1e3,
            "prefill_us": t["prefill_ms"] * 1e3,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak,
                         "traffic": ncu_traffic("prefill_" + pb.wl.spec.name, PREFILL_SOURCES),
                         "kernel": "pa_prefill",
                         "algorithmic_flops": flops,
                         "peak_source": f"{peak_src} bf16_tflops (burst)"}}


def prefill_sub_record(name, args, dev, flush, stream, world):
    spec, chunk = prefill_spec(args, name)
    pb = inputs.prefill_batch(spec, seed=0, chunk=chunk)
    ps = PrefillStep(pb, dev)
    steps = max(3, min(args.steps, 10))
    t = time_prefill(ps, flush, stream, steps, args.warmup, world)
    rec = {"metric": PREFILL_METRIC, "config": prefill_config(pb, chunk), "steps": steps,
           **prefill_rates(pb, t), "gpu_launches": steps * 2}
    del ps, pb
    torch.cuda.empty_cache()
    return rec


def run_gpu_prefill(args, rank, world, local):
    """One prefill step: store of every chunk row's K/V, then paged prefill."""
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec, chunk = prefill_spec(args)
    pb = inputs.prefill_batch(spec, seed=0, chunk=chunk)
    ps = PrefillStep(pb, dev, args.layout)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    clocks = ClockSampler(local)
    clocks.wait_first_sample()
    t = time_prefill(ps, flush, stream, args.steps, args.warmup, world)

    # end to end: pinned host inputs packed in one staging buffer, one H2D,
    # the step, the output read back
    host_inputs = ps.host_inputs
    offs, total = [], 0
    for x in host_inputs:
        offs.append(total)
        total += (x.numel() * x.element_size() + 255) // 256 * 256
    h_stage = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    for x, o in zip(host_inputs, offs):
        nb = x.numel() * x.element_size()
        h_stage[o:o + nb].copy_(x.contiguous().view(-1).view(torch.uint8))
    d_stage = torch.empty(total, dtype=torch.uint8, device=dev)
    views = [d_stage[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape)
             for x, o in zip(host_inputs, offs)]
    hout = torch.empty(ps.out.shape, dtype=ps.out.dtype, pin_memory=True)
    h2d = sum(x.numel() * x.element_size() for x in host_inputs)
    d2h = hout.numel() * hout.element_size()

    def e2e_step():
        d_stage.copy_(h_stage, non_blocking=True)
        ps.step(*views)
        hout.copy_(ps.out, non_blocking=True)

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
    clk = clocks.stop()
    if not torch.equal(hout.view(torch.int16), ps.out.cpu().view(torch.int16)):
        raise SystemExit("e2e output differs from the device-resident output")
    if rank != 0:
        return
    rates = prefill_rates(pb, t)
    line = {
        "metric": PREFILL_METRIC, "value": rates["us_per_step"], "unit": "us/step",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t["ms"],
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": prefill_config(pb, chunk, args.layout),
        **{k: v for k, v in rates.items() if k != "us_per_step"},
        "e2e": {"value": e2e * 1e3, "unit": "us/step", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * 2,
        "timing": "value: store + prefill per step, events between the two calls",
        "clocks": clk,
    }
    if args.variant:
        line["kernel_variant"] = args.variant
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
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="oracle time of the prefill CPU baseline's sample")
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub-records", action="store_true",
                    help="time the chosen workload only (profiling runs)")
    ap.add_argument("--variant", choices=sorted(VARIANTS),
                    help="run a comparison kernel the library keeps for tests instead of the "
                         "product kernel (profiling runs; the line then names it)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.variant and (args.impl != "native" or not torch.cuda.is_available()):
        ap.error("--variant selects a GPU kernel")
    rank, world, local = dist_setup(args.gpus)
    if args.variant:
        from paged_kv_cache_255_gb300 import pagedattn as pa
        pa.debug_kernel_variant(getattr(pa, VARIANTS[args.variant]))
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
