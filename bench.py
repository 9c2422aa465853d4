"""Benchmark of one paged-KV attention step (index build + cache write +
paged attention) on synthetic workloads shaped like the pages' examples.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--decode-workload NAME|none] [--impl ours|reference]

Prints one JSON line.  A step is the whole path over one batch: the three
C-ABI calls on inputs already resident in HBM -- pa_prepare_and_write (the
index build and the cache write in one launch) and pa_attention -- captured
once into a CUDA graph and replayed once per step (``eager`` reports the same
calls launched one by one; ``three_calls`` the step as pa_prepare_inputs,
pa_cache_write and pa_attention).  The L2 is flushed (a 256 MB write) between timed steps,
outside the timed events.  ``e2e`` repeats the step through the same public
calls with the step's inputs copied from pinned host memory and the output
copied back inside the timed region.

The default workload is the mixed chunked-prefill step (one 5000-token
chunk at 2048 computed plus 200 decodes), so one line carries both
kernels' rooflines: ``roofline`` for the split-K kernel on the decode-class
requests (HBM) and ``roofline_prefill`` for the tensor-core kernel on the
chunk (bf16 tensor peak).  ``decode_workload`` adds the attention call of
the 256-request decode batch, timed alone, with its own HBM roofline.

Under torchrun every rank runs an independent replica (its own pool and
requests, seeded by rank): the path has no exchange step.  Timing is the max
over ranks; ``value`` is the tokens all ranks processed per second.

``--impl reference`` times the CPU oracle (the reference arm here) on a
bounded sample of the same workload, on the host cores.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import threading
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "paged-attn step tokens/s"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="mixed", choices=sorted(workloads.NAMED))
    ap.add_argument("--decode-workload", default="decode",
                    choices=sorted(workloads.NAMED) + ["none"],
                    help="a decode-only workload whose attention call is also timed alone, "
                         "with its HBM roofline (main arm, one GPU)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica_workload(name: str, rank: int):
    """Every rank runs an independent replica of the workload: the same shape
    with its own seed (rank 0 keeps the workload's default seed)."""
    return workloads.named(name, None if rank == 0 else 1000 + rank)


def reduce_over_ranks(x: float, op: str, dist, device) -> float:
    """max or sum of a host scalar over all ranks (no-op on one rank)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def kv_bytes(w) -> tuple[int, int]:
    """Algorithmic bytes of one attention call: K/V context read (logical and
    unique-physical), plus q read, out write and the block-table entries."""
    elt = 2
    extra = (w.num_tokens * w.num_q_heads * w.head_dim * elt * 2
             + int(np.ceil(w.context_lens / w.block_size).sum()) * 4)
    logical = w.kv_read_bytes() + extra
    unique = w.kv_unique_bytes() + extra
    return logical, unique


def load_peaks():
    """(hbm GB/s, bf16 TFLOP/s burst, source) from MEASURED_PEAKS.json."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


TENSOR_PATH_MIN_TOKENS = 17   # requests with more query tokens run on the tensor-core kernel


def causal_flops(w, mask) -> int:
    """4*D*Hq per visible (query, key) pair: QK^T and PV, causal-exact."""
    n = w.num_scheduled_tokens.astype(np.int64)[mask]
    c = w.num_computed_tokens.astype(np.int64)[mask]
    pairs = int((n * c + n * (n + 1) // 2).sum())
    return 4 * w.head_dim * w.num_q_heads * pairs


def sub_batch(w, mask, q, bt_dev, qsl_host, sl_host, dev):
    """The requests selected by `mask` as a batch of their own (inputs for
    pa_attention), built outside any timed region."""
    import torch
    reqs = np.nonzero(mask)[0]
    toks = np.concatenate([np.arange(qsl_host[r], qsl_host[r + 1]) for r in reqs])
    n = (qsl_host[reqs + 1] - qsl_host[reqs]).astype(np.int32)
    qsl = torch.from_numpy(np.concatenate([[0], np.cumsum(n)]).astype(np.int32)).to(dev)
    sl = torch.from_numpy(sl_host[reqs].astype(np.int32)).to(dev)
    qs = q.index_select(0, torch.from_numpy(toks).to(dev)).contiguous()
    bts = bt_dev.index_select(0, torch.from_numpy(reqs).to(dev)).contiguous()
    return qs, qsl, sl, bts, int(n.max()), int(sl_host[reqs].max())


KERNEL_SOURCES = {
    "paged_decode_kernel": ("decode.cu", "decode_fp16.cu", "pa_internal.cuh"),
    "paged_prefill_kernel": ("prefill.cu", "pa_internal.cuh"),
    "cache_write_kernel": ("cache_write.cu", "pa_internal.cuh"),
    "prepare_write_kernel": ("prep_write.cu", "pa_internal.cuh"),
}


# The prefill-class requests of a workload timed alone form a batch of their
# own; for the mixed step that batch is the `chunk` workload's shape (one
# 5000-token chunk at 2048, 32/8, D 128), whose ncu summary gives its traffic.
# (Inside the mixed step's own launches, under ncu, the kernels run one after
# another, so the first tensor-core grid would take every item itself.)
PREFILL_ALONE = {"mixed": "chunk"}


def kernel_source_hash(kernel: str = "paged_decode_kernel") -> str:
    """Hash of a kernel's sources with comments and blank space removed: a
    comment edit does not change the kernel the profile measured."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "paged_kv_attention_prepare_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str = "paged_decode_kernel"):
    """DRAM bytes per launch of a kernel from a committed ncu summary
    (``profiles/<kernel>_<workload>.txt`` or ``.md``), if it was taken on the
    current kernel source."""
    for ext in (".txt", ".md"):
        path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}{ext}")
        try:
            text = open(path).read()
        except OSError:
            continue
        m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
        hm = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
        if not m or not hm or hm.group(1) != kernel_source_hash(kernel):
            return None
        return float(m.group(1))
    return None


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled during the timed
    region.  Reads NVML directly (every 20 ms, from a thread; read-only
    queries), else falls back to ``nvidia-smi -lms 200``."""

    # nvmlClocksEventReasons bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, uuid: str | None = None):
        self.index, self.uuid = index, uuid
        self.proc = None
        self.samples = []          # (sm_mhz, reasons bitmask)
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None

    def _open_nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            u = self.uuid if self.uuid.startswith("GPU-") else "GPU-" + self.uuid
            ok = lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0
        if not ok:
            ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index),
                                                   ctypes.byref(h)) == 0
        if not ok:
            lib.nvmlShutdown()
            return False
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # 1 = SM clock
            self.max_mhz = float(mx.value)
        self._nvml, self._handle = lib, h
        return True

    def _poll(self):
        import ctypes
        lib, h = self._nvml, self._handle
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                r = rs.value if get_reasons(h, ctypes.byref(rs)) == 0 else 0
                self.samples.append((float(clk.value), int(r)))
            self._stop.wait(0.02)

    def __enter__(self):
        if self._open_nvml():
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
            self._nvml.nvmlShutdown()
            return
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            names = [0x8, 0x40, 0x20, 0x4]
            for line in out.splitlines():
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm, self.max_mhz = float(parts[1]), float(parts[2])
                except ValueError:
                    continue
                bits = sum(b for b, v in zip(names, parts[5:9]) if v.lower() == "active")
                self.samples.append((sm, bits))

    def summary(self):
        if not self.samples:
            return None
        reasons = set()
        for _, bits in self.samples:
            reasons |= {n for b, n in self.REASONS.items() if bits & b}
        return {"sm_mhz": float(np.median([c for c, _ in self.samples])),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(self.samples),
                "source": "nvml" if self._nvml is not None else "nvidia-smi"}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline, and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(w, vals_host, seconds: float, threads: int = 0):
    """Time the oracle on a bounded sample: the full index build and cache
    write, and attention for a growing random subset of tokens until about
    ``seconds`` of CPU work, on ``threads`` host threads (0: every core).
    Returns (tokens/s for the whole step, threads, description, phase times:
    seconds for the index build, the cache write, and attention scaled to
    the step)."""
    import oracle
    nthreads = threads if threads > 0 else oracle.num_cpus()
    t0 = time.perf_counter()
    idx = oracle.prepare_inputs(w.num_scheduled_tokens, w.num_computed_tokens, w.block_table,
                                w.block_size, w.num_tokens, w.num_blocks)
    t1 = time.perf_counter()
    fp8 = w.kv_cache_dtype == "fp8_e4m3"
    if fp8:
        kc, vc, _ = oracle.cache_write_fp8(vals_host["key"], vals_host["value"],
                                           vals_host["key_cache"], vals_host["value_cache"],
                                           idx["slot_mapping"], w.num_kv_heads, w.head_dim,
                                           w.block_size, w.num_blocks, w.dtype, w.k_scale,
                                           w.v_scale)
    else:
        kc, vc, _ = oracle.cache_write(vals_host["key"], vals_host["value"],
                                       vals_host["key_cache"], vals_host["value_cache"],
                                       idx["slot_mapping"], w.num_kv_heads, w.head_dim,
                                       w.block_size, w.num_blocks)
    t2 = time.perf_counter()
    rng = np.random.default_rng(0)
    n, spent, done = max(1, nthreads), 0.0, 0
    order = rng.permutation(w.num_tokens)
    while done < w.num_tokens and spent < seconds:
        take = np.sort(order[done:done + n])
        a = time.perf_counter()
        oracle.attention(vals_host["q"], kc, vc, w.block_table, idx["query_start_loc"],
                         idx["seq_lens"], w.num_q_heads, w.num_kv_heads, w.head_dim,
                         w.block_size, w.num_blocks, w.scale, w.dtype, tokens=take,
                         num_threads=nthreads, kv_cache_dtype=w.kv_cache_dtype,
                         k_scale=w.k_scale, v_scale=w.v_scale)
        spent += time.perf_counter() - a
        done += len(take)
        n = min(n * 2, w.num_tokens - done) if spent < seconds / 4 else n
    per_token = spent / done
    step_s = (t1 - t0) + (t2 - t1) + per_token * w.num_tokens
    desc = (f"index build + cache write on all {w.num_tokens} tokens; attention on {done} "
            f"random tokens ({spent:.1f} s), scaled to the step's {w.num_tokens} tokens")
    phases = {"prep_s": t1 - t0, "write_s": t2 - t1, "attention_s": per_token * w.num_tokens,
              "attention_tokens_sampled": int(done)}
    return w.num_tokens / step_s, nthreads, desc, phases


def cpu_baseline(w, vals_host, seconds: float) -> dict:
    """The oracle on every host core (``value``) and on one thread, each on a
    bounded sample of the step, with per-phase times."""
    v, threads, desc, phases = oracle_sample(w, vals_host, seconds)
    v1, _, desc1, phases1 = oracle_sample(w, vals_host, max(1.0, seconds / 4), threads=1)
    return {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc,
            "phases": phases,
            "single_thread": {"value": v1, "unit": UNIT, "cores": 1, "sample": desc1,
                              "phases": phases1}}


def host_values(vals):
    return {k: v.detach().cpu() for k, v in vals.items()}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = workloads.named(args.workload)
    vals = host_values(workloads.make_values(w, 1, device="cpu"))
    budget = max(2.0, min(args.cpu_seconds, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, vals, budget / 4)
    vals_s, threads, desc, phases = [], 0, "", {}
    for _ in range(args.steps):
        v, threads, desc, phases = oracle_sample(w, vals, budget)
        vals_s.append(v)
    value = float(np.median(vals_s))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * w.num_tokens / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "num_reqs": w.num_reqs, "num_tokens": w.num_tokens},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": desc, "phases": phases},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# The CUDA path
# ---------------------------------------------------------------------------

def attention_alone(name, args, pa, dev, stream, flush, hbm_peak, peak_kind):
    """Another workload's attention call timed alone: its index build and
    cache write run first (untimed), then pa_attention on its whole batch is
    timed with CUDA events, the L2 flushed before each launch.  Returns the
    workload's name, the call's time and its HBM roofline."""
    import torch
    w = workloads.named(name)
    vals = workloads.make_values(w, 1, device=dev)
    i32 = torch.int32
    R, T = w.num_reqs, w.num_tokens
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    nst, nct, bt = up(w.num_scheduled_tokens), up(w.num_computed_tokens), up(w.block_table)
    req, pos, slot = (torch.empty(T, dtype=i32, device=dev) for _ in range(3))
    qsl = torch.empty(R + 1, dtype=i32, device=dev)
    sl, li = torch.empty(R, dtype=i32, device=dev), torch.empty(R, dtype=i32, device=dev)
    ks, vs = vals.get("k_scale"), vals.get("v_scale")
    kc, vc = vals["key_cache"], vals["value_cache"]
    pa.pa_prepare_inputs(nst, nct, bt, w.block_size, T, w.num_blocks, req, pos, slot, qsl, sl, li)
    pa.pa_cache_write(vals["key"], vals["value"], kc, vc, slot, k_scale=ks, v_scale=vs)
    out = torch.empty_like(vals["q"])
    ws_bytes = pa.pa_attention_workspace_size(R, T, w.max_query_len, w.max_seq_len,
                                              w.num_q_heads, w.num_kv_heads, w.head_dim)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    # host-side values settled before the timed launches (shares_blocks scans
    # the block table on the host)
    shared, max_q, max_seq, q = w.shares_blocks, w.max_query_len, w.max_seq_len, vals["q"]
    evs = []
    for k in range(max(args.warmup, 1) + args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pa.pa_attention(q, kc, vc, bt, qsl, sl, max_q, max_seq, w.scale, out, ws, k_scale=ks,
                        v_scale=vs, shared_blocks=shared)
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    status, detail = pa.pa_get_status()
    if status != pa.PA_OK:
        raise RuntimeError(f"device checks failed ({name}): {pa.check_bits(detail)}")
    times_ms = [a.elapsed_time(b) for a, b in evs[max(args.warmup, 1):]]
    secs = float(np.mean(times_ms)) / 1e3
    logical, unique = kv_bytes(w)
    alg = unique if shared else logical
    achieved = alg / secs / 1e9
    line = {"workload": w.name, "num_reqs": R, "num_tokens": T, "attn_us": secs * 1e6,
            "attn_us_min_max": [min(times_ms) * 1e3, max(times_ms) * 1e3],
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": recorded_traffic(name),
                         "kernel": "pa_attention (paged_decode_kernel + merge_kernel)",
                         "algorithmic_bytes_per_launch": alg, "avg_launch_us": secs * 1e6,
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                         "frac_of_8TBps": achieved / 8000.0}}
    del vals, kc, vc, out, ws
    torch.cuda.empty_cache()
    return line


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from paged_kv_attention_prepare_gb300.builder import build
    build()
    import paged_kv_attention_prepare_gb300 as pa

    dev = torch.device("cuda", local)
    w = replica_workload(args.workload, rank)
    vals = workloads.make_values(w, 1 + rank, device=dev)
    i32 = torch.int32
    R, T = w.num_reqs, w.num_tokens
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    nst, nct, bt = up(w.num_scheduled_tokens), up(w.num_computed_tokens), up(w.block_table)
    req, pos, slot = (torch.empty(T, dtype=i32, device=dev) for _ in range(3))
    qsl = torch.empty(R + 1, dtype=i32, device=dev)
    sl, li = torch.empty(R, dtype=i32, device=dev), torch.empty(R, dtype=i32, device=dev)
    q, key, value = vals["q"], vals["key"], vals["value"]
    kc, vc = vals["key_cache"], vals["value_cache"]
    ks, vs = vals.get("k_scale"), vals.get("v_scale")   # FP8 pools only
    # an engine that shares blocks across requests (copy-on-write forks,
    # prefix caching) says so: PA_ATTN_SHARED_BLOCKS
    shared = w.shares_blocks
    max_q, max_seq = w.max_query_len, w.max_seq_len   # settled before any timed region
    out = torch.empty_like(q)
    ws_bytes = pa.pa_attention_workspace_size(R, T, w.max_query_len, w.max_seq_len,
                                              w.num_q_heads, w.num_kv_heads, w.head_dim)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # The step: the index build and the cache write in one launch
    # (pa_prepare_and_write), then attention; ``fused=False`` runs the three
    # calls of the boundary one after another (reported as three_calls).
    def step(nst=nst, nct=nct, bt=bt, q=q, key=key, value=value, timed=True, fused=True):
        if fused:   # the index build and the cache write as one launch
            pa.pa_prepare_and_write(nst, nct, bt, w.block_size, T, w.num_blocks, req, pos, slot,
                                    qsl, sl, li, key, value, kc, vc, k_scale=ks, v_scale=vs)
        else:
            pa.pa_prepare_inputs(nst, nct, bt, w.block_size, T, w.num_blocks, req, pos, slot,
                                 qsl, sl, li)
            pa.pa_cache_write(key, value, kc, vc, slot, k_scale=ks, v_scale=vs)
        if timed:
            a0.record(stream)
        pa.pa_attention(q, kc, vc, bt, qsl, sl, max_q, max_seq, w.scale, out, ws,
                        k_scale=ks, v_scale=vs, shared_blocks=shared)
        if timed:
            a1.record(stream)

    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(max(args.warmup, 0)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    status, detail = pa.pa_get_status()
    if status != pa.PA_OK:
        raise RuntimeError(f"device checks failed during warm-up: {pa.check_bits(detail)}")

    # ---- the step captured once into a CUDA graph (the three calls, same
    # buffers); the launches of one replay are counted at capture
    graph, graph_error = None, None
    pa.pa_launch_count()
    try:
        gstream = torch.cuda.Stream(dev)
        gstream.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gstream):
            step(timed=False)
        torch.cuda.synchronize()
    except RuntimeError as exc:  # capture refused: report it, time the calls eagerly
        graph, graph_error = None, str(exc).splitlines()[0]
    launches_per_replay = pa.pa_launch_count()

    # ---- timed regions: device-resident inputs.  (1) the calls launched one
    # by one (per-step events also bracket the attention call); (2) graph
    # replays, the headline when the capture succeeded.
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    g_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    uuid = str(getattr(torch.cuda.get_device_properties(dev), "uuid", "") or "") or None
    with ClockSampler(local, uuid) as clocks:
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        pa.pa_launch_count()
        for k in range(args.steps):
            flush.zero_()
            s0, s1, b0, b1 = ev[k]
            s0.record(stream)
            a0, a1 = b0, b1
            step()
            s1.record(stream)
        torch.cuda.synchronize()
        eager_launches = pa.pa_launch_count()
        if dist is not None:
            dist.barrier()
        if graph is not None:
            for _ in range(max(args.warmup, 1)):
                flush.zero_()
                graph.replay()
            if dist is not None:
                dist.barrier()
            torch.cuda.synchronize()
            for k in range(args.steps):
                flush.zero_()
                g_ev[k][0].record(stream)
                graph.replay()
                g_ev[k][1].record(stream)
            torch.cuda.synchronize()
            if dist is not None:
                dist.barrier()
    # ---- the same step as the boundary's three calls (pa_prepare_inputs,
    # pa_cache_write, pa_attention), captured and replayed the same way
    three_line = None
    try:
        fgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(fgraph, stream=gstream):
            step(timed=False, fused=False)
        torch.cuda.synchronize()
        for _ in range(max(args.warmup, 1)):
            flush.zero_()
            fgraph.replay()
        f_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        for k in range(args.steps):
            flush.zero_()
            f_ev[k][0].record(stream)
            fgraph.replay()
            f_ev[k][1].record(stream)
        torch.cuda.synchronize()
        f_ms = reduce_over_ranks(float(np.sum([x.elapsed_time(y) for x, y in f_ev])), "max", dist,
                                 dev) / args.steps
        three_line = {"ms_per_step": f_ms,
                      "value": reduce_over_ranks(T, "sum", dist, dev) / (f_ms / 1e3), "unit": UNIT,
                      "what": "pa_prepare_inputs + pa_cache_write + pa_attention as one graph"}
        del fgraph
    except (RuntimeError, pa.PAError) as exc:
        three_line = {"error": str(exc).splitlines()[0]}
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    attn_ms = [e[2].elapsed_time(e[3]) for e in ev]
    eager_ms = reduce_over_ranks(float(np.sum(step_ms)), "max", dist, dev) / args.steps
    all_tokens = reduce_over_ranks(T, "sum", dist, dev)
    if graph is not None:
        graph_ms = reduce_over_ranks(float(np.sum([x.elapsed_time(y) for x, y in g_ev])), "max",
                                     dist, dev) / args.steps
        ms_per_step, launches = graph_ms, launches_per_replay * args.steps
        del graph
    else:
        graph_ms, ms_per_step, launches = None, eager_ms, eager_launches
    value = all_tokens / (ms_per_step / 1e3)
    status, detail = pa.pa_get_status()
    if status != pa.PA_OK:
        raise RuntimeError(f"device checks failed in the timed region: {pa.check_bits(detail)}")

    # ---- the index build alone: the plain call vs. the extended one (token-id
    # gather from a device or page-locked host token buffer, discard mask)
    def time_calls(fn, reps):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for k in range(max(args.warmup, 1) + reps):
            flush.zero_()
            if k >= max(args.warmup, 1):
                evs[k - max(args.warmup, 1)][0].record(stream)
            fn()
            if k >= max(args.warmup, 1):
                evs[k - max(args.warmup, 1)][1].record(stream)
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in evs])) * 1e3

    tok_buf = workloads.make_token_buffer(w, 1 + rank)
    tok_dev = torch.from_numpy(tok_buf).to(dev)
    tok_host = torch.from_numpy(tok_buf).pin_memory()
    totals = up(workloads.make_request_totals(w, 1 + rank))
    tok_idx = torch.empty(T, dtype=torch.int64, device=dev)
    in_ids = torch.empty(T, dtype=i32, device=dev)
    discard = torch.empty(R, dtype=torch.uint8, device=dev)

    def prep_ex(ids):
        pa.pa_prepare_inputs_ex(nst, nct, bt, w.block_size, T, w.num_blocks, req, pos, slot, qsl,
                                sl, li, token_ids=ids, token_indices=tok_idx, input_ids=in_ids,
                                request_num_tokens=totals, discard_request_mask=discard)

    prep_us = {
        "pa_prepare_inputs": time_calls(
            lambda: pa.pa_prepare_inputs(nst, nct, bt, w.block_size, T, w.num_blocks, req, pos,
                                         slot, qsl, sl, li), args.steps),
        "pa_prepare_inputs_ex_device_tokens": time_calls(lambda: prep_ex(tok_dev), args.steps),
        "pa_prepare_inputs_ex_host_tokens": time_calls(lambda: prep_ex(tok_host), args.steps),
    }
    del tok_dev, tok_host

    # ---- the cache write alone: the step's new K/V rows into their slots
    # (read and write, plus the slot indices)
    write_elt = 1 if w.kv_cache_dtype == "fp8_e4m3" else 2
    write_bytes = T * 2 * w.num_kv_heads * w.head_dim * (2 + write_elt) + 4 * T
    write_us = time_calls(lambda: pa.pa_cache_write(vals["key"], vals["value"], kc, vc, slot,
                                                    k_scale=ks, v_scale=vs), args.steps)
    cache_write = {"us": write_us, "bytes": int(write_bytes),
                   "GBps": write_bytes / (write_us * 1e-6) / 1e9,
                   "note": "launch-bound below ~10 MB of rows"}

    # ---- end to end: inputs from pinned host memory, output back to host.
    # Every step copies its inputs host -> device and reads its output back,
    # through the same public calls.  When the step's KV bytes exceed the L2
    # many times over, steps are pipelined the way an engine runs them: the
    # next step's inputs are copied (second stream, double-buffered) while the
    # current step computes, and the L2 is not flushed (the inputs are larger
    # than L2).  Otherwise steps run one after another with the L2 flushed
    # between them, outside the timed events.
    host_in = {"nst": w.num_scheduled_tokens, "nct": w.num_computed_tokens, "bt": w.block_table}
    pinned = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in host_in.items()}
    for k in ("q", "key", "value"):
        pinned[k] = vals[k].cpu().contiguous().pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    d2h = out_host.numel() * out_host.element_size()
    pipelined = w.kv_unique_bytes() > 2 * L2_FLUSH_BYTES
    nbuf = 2 if pipelined else 1
    dev_in = [{k: torch.empty_like(v, device=dev) for k, v in pinned.items()} for _ in range(nbuf)]
    outs = [out] + [torch.empty_like(out) for _ in range(nbuf - 1)]
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(nbuf)]
    computed = [torch.cuda.Event() for _ in range(nbuf)]

    def e2e_compute(b):
        d = dev_in[b]
        pa.pa_prepare_and_write(d["nst"], d["nct"], d["bt"], w.block_size, T, w.num_blocks, req,
                                pos, slot, qsl, sl, li, d["key"], d["value"], kc, vc, k_scale=ks,
                                v_scale=vs)
        pa.pa_attention(d["q"], kc, vc, d["bt"], qsl, sl, max_q, max_seq,
                        w.scale, outs[b], ws, k_scale=ks, v_scale=vs, shared_blocks=shared)

    def e2e_h2d(b):
        with torch.cuda.stream(copy_stream):
            for k in pinned:
                dev_in[b][k].copy_(pinned[k], non_blocking=True)
            copied[b].record(copy_stream)

    def e2e_run(nsteps, t_start=None, t_end=None):
        """nsteps pipelined steps: H2D(k+1) overlaps step k; D2H(k) follows it."""
        if t_start is not None:
            t_start.record(copy_stream)
        e2e_h2d(0)
        for k in range(nsteps):
            b = k % nbuf
            if k + 1 < nsteps:
                e2e_h2d((k + 1) % nbuf)   # queued after D2H(k - 1): buffer (k+1)%2 is free
            stream.wait_event(copied[b])
            e2e_compute(b)
            computed[b].record(stream)
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(computed[b])
                out_host.copy_(outs[b], non_blocking=True)
        if t_end is not None:
            t_end.record(copy_stream)

    if pipelined:
        e2e_run(max(args.warmup, 1))
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_run(args.steps, t_a, t_b)
        torch.cuda.synchronize()
        e2e_ms = reduce_over_ranks(t_a.elapsed_time(t_b), "max", dist, dev)
        e2e_mode = "pipelined: next step's inputs copied during this step; inputs larger than L2"
    else:
        def e2e_step():
            e2e_h2d(0)
            stream.wait_event(copied[0])
            e2e_compute(0)
            out_host.copy_(out, non_blocking=True)

        for _ in range(max(args.warmup, 1)):
            flush.zero_()
            e2e_step()
        torch.cuda.synchronize()
        e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        for k in range(args.steps):
            flush.zero_()
            e2e_ev[k][0].record(stream)
            e2e_step()
            e2e_ev[k][1].record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_over_ranks(float(np.sum([a.elapsed_time(b) for a, b in e2e_ev])), "max",
                                   dist, dev)
        e2e_mode = "serial: copy in, step, copy out; L2 flushed between steps"
    if dist is not None:
        dist.barrier()
    status, detail = pa.pa_get_status()
    if status != pa.PA_OK:
        raise RuntimeError(f"device checks failed: {pa.check_bits(detail)}")

    # ---- rooflines.  The attention call is timed live above; when the batch
    # mixes both request classes, each class is also timed alone (as a batch
    # of its own, same kernels) so each kernel gets its own roofline.
    hbm_peak, tf_peak, peak_kind = load_peaks()
    long_mask = w.num_scheduled_tokens >= TENSOR_PATH_MIN_TOKENS
    short_mask = ~long_mask
    qsl_host = np.concatenate([[0], np.cumsum(w.num_scheduled_tokens)]).astype(np.int64)
    sl_host = w.context_lens.astype(np.int64)

    def time_sub(mask):
        qs, qsl_s, sl_s, bt_s, mq, ms = sub_batch(w, mask, q, bt, qsl_host, sl_host, dev)
        os_ = torch.empty_like(qs)
        evs = []
        for k in range(max(args.warmup, 1) + args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            pa.pa_attention(qs, kc, vc, bt_s, qsl_s, sl_s, mq, ms, w.scale, os_, ws, k_scale=ks,
                            v_scale=vs, shared_blocks=shared)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in evs[max(args.warmup, 1):]])) / 1e3

    logical, unique = kv_bytes(w)
    if long_mask.any() and short_mask.any():
        decode_s = time_sub(short_mask)
        cache_elt = 1 if w.kv_cache_dtype == "fp8_e4m3" else 2
        alg = (int(sl_host[short_mask].sum()) * 2 * w.num_kv_heads * w.head_dim * cache_elt
               + int(short_mask.sum()) * w.num_q_heads * w.head_dim * 4)
        what = "decode-class requests alone (paged_decode_kernel + merge_kernel)"
    else:
        decode_s = float(np.mean(attn_ms)) / 1e3
        alg = unique if args.workload == "shared_prefix" else logical
        what = "pa_attention (paged_decode_kernel + merge_kernel)"
    roofline = None
    if short_mask.any():
        achieved = alg / decode_s / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved / hbm_peak, "traffic": recorded_traffic(args.workload),
                    "kernel": what, "algorithmic_bytes_per_launch": alg,
                    "avg_launch_us": decode_s * 1e6,
                    "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                    "frac_of_8TBps": achieved / 8000.0}
        if args.workload == "shared_prefix":
            roofline["effective_logical_GBps"] = logical / decode_s / 1e9
    roofline_prefill = None
    if long_mask.any():
        pre_s = time_sub(long_mask) if short_mask.any() else float(np.mean(attn_ms)) / 1e3
        flops = causal_flops(w, long_mask)
        achieved = flops / pre_s / 1e12
        roofline_prefill = {"bound": "tensor", "achieved": achieved, "peak": tf_peak,
                            "unit": "TFLOP/s", "frac": achieved / tf_peak,
                            "traffic": recorded_traffic(PREFILL_ALONE.get(args.workload, args.workload),
                                                        "paged_prefill_kernel"),
                            "kernel": "pa_attention on the prefill-class requests alone: "
                                      "paged_prefill_kernel (tcgen05)" +
                                      (", after widen_v_kernel (V to f16 once per call)"
                                       if (w.dtype == "bf16" and w.head_dim == 128
                                           and w.kv_cache_dtype != "fp8_e4m3") else ""),
                            "flops_per_launch": flops,
                            "avg_launch_us": pre_s * 1e6,
                            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json bf16_tflops, "
                                           "burst; fp16 runs at the same dense rate)"}
        if roofline is None:
            roofline = roofline_prefill

    # ---- whole-block operations on this workload's pools (run last: they
    # overwrite blocks): copy-on-write copies and new-block zeroing of up to
    # 4096 blocks, timed alone; algorithmic bytes = read + written.
    block_ops = None
    n_ops = min(4096, w.num_blocks // 2)
    if n_ops > 0:
        perm = np.random.default_rng(77 + rank).permutation(w.num_blocks).astype(np.int32)
        src_b, dst_b = up(perm[:n_ops]), up(perm[n_ops:2 * n_ops])
        block_bytes = w.block_size * w.num_kv_heads * w.head_dim * kc.element_size()
        copy_us = time_calls(lambda: pa.pa_copy_blocks(kc, vc, src_b, dst_b), args.steps)
        zero_us = time_calls(lambda: pa.pa_zero_blocks(kc, vc, dst_b), args.steps)
        copy_bytes = 2 * 2 * n_ops * block_bytes
        zero_bytes = 2 * n_ops * block_bytes
        block_ops = {
            "blocks": n_ops, "block_bytes": block_bytes,
            "copy_blocks": {"us": copy_us, "bytes": copy_bytes,
                            "GBps": copy_bytes / copy_us / 1e3,
                            "frac": copy_bytes / copy_us / 1e3 / hbm_peak},
            "zero_blocks": {"us": zero_us, "bytes": zero_bytes,
                            "GBps": zero_bytes / zero_us / 1e3,
                            "frac": zero_bytes / zero_us / 1e3 / hbm_peak},
            "peak": hbm_peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"}
        status, detail = pa.pa_get_status()
        if status != pa.PA_OK:
            raise RuntimeError(f"device checks failed in block ops: {pa.check_bits(detail)}")

    decode_line = None
    if world == 1 and args.decode_workload not in ("none", args.workload):
        decode_line = attention_alone(args.decode_workload, args, pa, dev, stream, flush,
                                      hbm_peak, peak_kind)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, host_values(vals), args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "num_reqs": R, "num_tokens": T,
                       "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
                       "head_dim": w.head_dim, "block_size": w.block_size,
                       "kv_bytes": w.kv_read_bytes(), "parallelism": f"replicas x{world}",
                       "l2": "flushed between steps (256 MB write outside the timed events)",
                       "shared_blocks_flag": bool(shared)},
            "roofline": roofline,
            "roofline_prefill": roofline_prefill,
            "decode_workload": decode_line,
            "cpu_baseline": cpu,
            "e2e": {"value": all_tokens / (e2e_ms / args.steps / 1e3), "unit": UNIT,
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "mode": e2e_mode},
            "gpu_launches": int(launches),
            "clocks": clocks.summary(),
            "attn_us_per_step": float(np.mean(attn_ms)) * 1e3,
            "prep_us": prep_us,
            "cache_write": cache_write,
            "block_ops": block_ops,
            "launch": ("cuda_graph: pa_prepare_and_write + pa_attention captured once, one "
                       "replay per step"
                       if graph_ms is not None else f"eager (graph capture failed: {graph_error})"),
            "three_calls": three_line,
            "eager": {"ms_per_step": eager_ms, "value": all_tokens / (eager_ms / 1e3),
                      "unit": UNIT, "gpu_launches": int(eager_launches),
                      "what": "pa_prepare_and_write + pa_attention launched one by one per step"},
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
