"""Benchmark of the transform-coded KV cache hot path on B300.

One step = one pass of the whole hot path over one batch of the Llama-3.1-8B-shaped decode workload
(32 query / 8 KV heads, d = 128, batch 1, 32768 cached tokens, 2.75 bits per element): kv_encode appends
the new token's key and value to the packed cache (rotation, quantisation, packing) and kv_attend_decode
runs decode attention of the 32 query heads over the packed cache (q rotation, split-K over the context,
merge, inverse rotation). The cache grows by one token per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-workloads]

Prints one JSON line. value = algorithmic bytes of a step (packed K/V records read, q read, output written,
appended token in and records out) / device time of the step, in GB/s; L2 is flushed (a 2 x L2 buffer is
written) before every timed step and the flush is outside the timed events. The line's "workloads" object
holds the other workloads, measured the same way: the 131072-token layer at 1.33 bits, the Qwen2.5-7B-shaped
batch at 2, 3 and 4 bits, the 32-layer prefill stack (encode throughput, calibration time, one decode per
layer), the headline layer in 256-token pages (one layer, and four layers in one launch, with the query's rotary
embedding in the kernel), and the token-axis allocation on the headline layer (token weights, kept tokens, record
compaction, decode at the retained length). --impl reference times the CPU oracle (test infrastructure) on full steps of the headline workload,
its KV heads spread over spawned processes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "llama_decode_32k"   # the headline workload
BITS = 2.75
DESCRIPTION = {"llama_decode_32k": "llama3.1-8b layer decode", "qwen_batched_8k": "qwen2.5-7b batched layer decode",
               "llama_long_128k": "llama3.1-8b long-context layer decode",
               "llama_prefill_32l": "llama3.1-8b 32-layer prefill stack"}
METRIC = "decode_attn_packed_kv_hbm_gbs"
UNIT = "GB/s"
# the decode kernel and the device headers it is built from: the recorded traffic is valid while they are unchanged
KERNEL_SRCS = [os.path.join(ROOT, "transform_coded_kv_02_b300", "csrc", f)
               for f in ("kvtc_decode.cuh", "kvtc_codec.cuh", "kvtc_ptx.cuh")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_llama32k_traffic.md")
# the line's other decode workloads: (workload, bits per element)
EXTRA_DECODE = [("llama_long_128k", 1.33), ("qwen_batched_8k", 2.0), ("qwen_batched_8k", 3.0),
                ("qwen_batched_8k", 4.0)]


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="the headline workload only")
    ap.add_argument("--cpu-steps", type=int, default=4, help="full oracle steps timed for the CPU baseline")
    return ap.parse_args(argv)


# ------------------------------------------------------------------------------------------------------
# workload arithmetic
# ------------------------------------------------------------------------------------------------------
def record_words(bits: float, d: int = 128) -> int:
    return int(math.floor(bits * d / 32 + 1e-9))


def step_bytes(T_ctx: int, w, rk: int, rv: int) -> int:
    """Algorithmic bytes of one step at context length T_ctx (after the append): records read, q read, output
    written, the appended token read and its records written."""
    B, Hkv, Hq, d = w.B, w.Hkv, w.Hq, w.d
    packed = B * Hkv * T_ctx * 4 * (rk + rv)
    q_out = B * Hq * d * 2 + B * Hq * d * 4
    append = B * Hkv * d * 2 * 2 + B * Hkv * 4 * (rk + rv)
    return packed + q_out + append


def decode_bytes(T_ctx: int, w, rk: int, rv: int) -> int:
    B, Hkv, Hq, d = w.B, w.Hkv, w.Hq, w.d
    return B * Hkv * T_ctx * 4 * (rk + rv) + B * Hq * d * 2 + B * Hq * d * 4


def bf16_decode_bytes(T_ctx: int, w) -> int:
    B, Hkv, Hq, d = w.B, w.Hkv, w.Hq, w.d
    return B * Hkv * T_ctx * d * 2 * 2 + B * Hq * d * 2 + B * Hq * d * 4


def encode_bytes(token_heads: int, d: int, rk: int, rv: int) -> int:
    """Prefill encode of token_heads (token, KV head) pairs: the bf16 key and value read, both records written."""
    return token_heads * (2 * d * 2 + 4 * (rk + rv))


def workload_name(w, bits: float, rk_w: int, rv_w: int, steps: bool = True) -> str:
    calib = "per-sequence calibration, " if w.calib == "own_prefix" else ""
    grow = " growing by 1 per step" if steps else ""
    work = ", append-encode + decode per step" if steps else ", one decode query per sequence"
    return (f"{DESCRIPTION[w.name]}: {w.Hq} q / {w.Hkv} kv heads, d={w.d}, batch {w.B}, {w.T} cached tokens{grow}, "
            f"{calib}{bits} bits/elem (K {rk_w} + V {rv_w} words/token){work}")


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over the ranks (the job's time is its slowest rank's); x itself when world == 1."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank: float, seconds: float, world: int) -> float:
    """Whole-job throughput: every rank processes the same amount of work (its own layer), and the job takes
    the slowest rank's time."""
    return world * bytes_per_rank / seconds / 1e9


# ------------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, flags in rows for n, fl in zip(names, flags) if fl.lower() == "active"})
        sm = [r[0] for r in rows]
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(r[1] for r in rows)), "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------------------------------------------
# helpers
# ------------------------------------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SRCS:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """Per-launch DRAM bytes of the decode kernel from the committed ncu summary, if it was taken on the
    current kernel source (the summary records the source hash)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    text = open(TRAFFIC_FILE).read()
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    t = re.search(r"traffic_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    if not h or not t or h.group(1) != kernel_source_hash():
        return None
    return float(t.group(1))


def bf16_tensor(np_bits, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(np_bits).view(np.int16)).to(dev).view(torch.bfloat16)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def make_workload(n_new: int, layer: int = 0, name: str = WORKLOAD):
    """Synthetic layer with T + n_new tokens: the first T are prefilled, the rest appended one per step. Rank r
    of a multi-GPU run takes layer r of the model: its own data, the same shapes."""
    from transform_coded_kv_02_b300 import synth
    w = synth.WORKLOADS[name]
    return w, synth.make_layer(w, layer=layer, T=w.T + n_new, steps=n_new)


# ------------------------------------------------------------------------------------------------------
# the CPU oracle on the host cores (the baseline leg and the reference arm)
# ------------------------------------------------------------------------------------------------------
def _oracle_worker(conn, heads, T, bits, scale):
    """One process: the oracle's calibration and the records of its KV heads' first T tokens, then full steps on
    request. Step i appends token T + i of each head (the oracle's encode of that key and value) and decodes
    query i of the head's query heads over its T + i + 1 records."""
    from oracle import kvtc_oracle as O
    from transform_coded_kv_02_b300 import synth
    state = []
    for hp in heads:
        pk, pv = O.calibrate(hp["ck"], hp["cv"], hp["cq"], bits, bits)
        kf, vf = synth.as_float(hp["k"]), synth.as_float(hp["v"])
        rk, rv = O.encode(kf, pk), O.encode(vf, pv)
        state.append((pk, pv, kf, vf, rk, rv, synth.as_float(hp["q"])))
    conn.send("ready")
    while True:
        i = conn.recv()
        if i is None:
            break
        for pk, pv, kf, vf, rk, rv, q in state:
            O.encode(kf[T + i:T + i + 1], pk)
            O.encode(vf[T + i:T + i + 1], pv)
            O.attend_decode(q[i], rk, rv, pk, pv, T + i + 1, scale)
        conn.send(i)
    conn.close()


class OracleHeads:
    """The oracle as it stands on full steps of a workload: its (sequence, KV head) units spread over up to
    max_procs spawned processes of one BLAS thread each, every process holding its units' records; step(i)
    runs step i on every unit and returns the step's wall time."""

    def __init__(self, w, L, bits, max_procs):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        units = [(b, h) for b in range(w.B) for h in range(w.Hkv)]
        self.n_proc = max(1, min(max_procs, len(units)))
        g = w.g
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"  # inherited by the spawned processes
        self.conns, self.procs = [], []
        for p_i in range(self.n_proc):
            heads = []
            for b, h in units[p_i::self.n_proc]:
                si = b * w.Hkv + h if L.per_seq_params else h
                heads.append({"k": L.k[b, h], "v": L.v[b, h], "ck": L.calib_k[si], "cv": L.calib_v[si],
                              "cq": L.calib_q[si], "q": L.q[:, b, h * g:(h + 1) * g]})
            parent, child = ctx.Pipe()
            p = ctx.Process(target=_oracle_worker, args=(child, heads, w.T, bits, 1.0 / math.sqrt(w.d)), daemon=True)
            p.start()
            child.close()
            self.conns.append(parent)
            self.procs.append(p)
        for c in self.conns:
            if c.recv() != "ready":
                raise RuntimeError("oracle process failed to start")

    def step(self, i: int) -> float:
        t0 = time.perf_counter()
        for c in self.conns:
            c.send(i)
        for c in self.conns:
            c.recv()
        return time.perf_counter() - t0

    def close(self):
        for c in self.conns:
            try:
                c.send(None)
            except (BrokenPipeError, OSError):
                pass
        for p in self.procs:
            p.join(timeout=30)


def time_oracle(w, L, bits, first: int, warmup: int, steps: int):
    """Full oracle steps first .. first + warmup + steps - 1 of the workload (tokens appended one per step after
    the first T); the last `steps` are timed. Returns (per-step seconds, processes used)."""
    runner = OracleHeads(w, L, bits, host_cores())
    try:
        for i in range(warmup):
            runner.step(first + i)
        ts = [runner.step(first + warmup + j) for j in range(steps)]
    finally:
        runner.close()
    return ts, runner.n_proc


def cpu_baseline(w, L, bits, n_steps):
    """The oracle on full steps of the headline workload, on the host cores (one untimed step first)."""
    ts, n_proc = time_oracle(w, L, bits, 0, 1, n_steps)
    secs = float(np.sum(ts))
    rw = record_words(bits)
    nbytes = sum(step_bytes(w.T + 2 + j, w, rw, rw) for j in range(n_steps))
    return {"value": nbytes / secs / 1e9, "unit": UNIT, "cores": n_proc, "kind": "oracle",
            "ms_per_step": secs / n_steps * 1e3,
            "sample": f"{n_steps} full steps of the workload (append-encode + decode of all {w.B * w.Hkv} KV heads "
                      f"over {w.T}+ cached records), {n_proc} processes of one thread each on {host_cores()} host "
                      f"cores, {secs:.1f} s timed"}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle on full steps of the headline workload, each step timed whole."""
    if rank != 0:
        return None
    K, W = args.steps, args.warmup
    w, L = make_workload(K + W + 1)
    ts, n_proc = time_oracle(w, L, BITS, 0, W, K)
    rw = record_words(BITS)
    nbytes = sum(step_bytes(w.T + W + j + 1, w, rw, rw) for j in range(K))
    secs = float(np.sum(ts))
    value = nbytes / secs / 1e9
    sample = (f"every step whole: append-encode + decode of all {w.Hkv} KV heads over {w.T}+ cached records, "
              f"{n_proc} processes of one thread each on {host_cores()} host cores")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": K, "warmup": W,
            "ms_per_step": secs / K * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": workload_name(w, BITS, rw, rw), "l2": "n/a (host)", "parallelism": "single host"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": n_proc, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return line


# ------------------------------------------------------------------------------------------------------
# the CUDA path
# ------------------------------------------------------------------------------------------------------
class Gpu:
    """Device, stream, L2 flush and the event timing every measurement uses."""

    def __init__(self, local_rank):
        import torch
        self.torch = torch
        torch.cuda.set_device(local_rank)
        self.dev = torch.device("cuda", local_rank)
        self.stream = torch.cuda.current_stream(self.dev)
        self.cap = torch.cuda.Stream(self.dev)
        l2 = torch.cuda.get_device_properties(self.dev).L2_cache_size
        self.flush_buf = torch.empty(2 * l2 // 4 + 1024, dtype=torch.int32, device=self.dev)

    def flush_l2(self):
        self.flush_buf.fill_(1)

    def timed(self, items):
        """items: list of lists of zero-argument callables (graph replays). Before each item L2 is flushed;
        events bracket every callable. A sleep kernel first gives the host a head start. Returns seconds
        [n_items, n_callables]."""
        torch = self.torch
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(it) + 1)] for it in items]
        torch.cuda._sleep(int(4e7))
        for it, ev in zip(items, evs):
            self.flush_l2()
            ev[0].record(self.stream)
            for c, e in zip(it, ev[1:]):
                c()
                e.record(self.stream)
        torch.cuda.synchronize()
        return np.array([[ev[k].elapsed_time(ev[k + 1]) * 1e-3 for k in range(len(ev) - 1)] for ev in evs])

    def graph(self, fn):
        g = self.torch.cuda.CUDAGraph()
        with self.torch.cuda.graph(g, stream=self.cap, capture_error_mode="relaxed"):
            fn()
        return g


class Layer:
    """One workload layer on the device: calibrated parameters, the packed caches, the prefill tokens, and the
    appended tokens and decode queries of n_new steps."""

    def __init__(self, gpu, w, L, bits, n_new):
        from transform_coded_kv_02_b300 import kvtc
        torch = gpu.torch
        self.gpu, self.w, self.bits, self.kvtc = gpu, w, bits, kvtc
        dev = gpu.dev
        B, Hkv, Hq, d, T = w.B, w.Hkv, w.Hq, w.d, w.T
        self.T_cap = (T + n_new + 15) // 16 * 16
        t0 = time.perf_counter()
        self.P = kvtc.kv_calibrate(list(zip(L.calib_k, L.calib_v, L.calib_q)), bits, bits)
        self.calibrate_s = time.perf_counter() - t0
        self.P.upload()
        self.rk_w, self.rv_w = self.P.record_words(0), self.P.record_words(1)
        self.rec_k = torch.zeros((B, Hkv, self.T_cap, self.rk_w), dtype=torch.int32, device=dev)
        self.rec_v = torch.zeros((B, Hkv, self.T_cap // 2, 2 * self.rv_w), dtype=torch.int32, device=dev)
        self.cache = kvtc.make_cache(self.rec_k, self.rec_v, B, Hkv, self.T_cap, L.per_seq_params)
        self.k_all = bf16_tensor(L.k, dev)                    # [B, Hkv, T + n_new, d]
        self.v_all = bf16_tensor(L.v, dev)
        self.k_pre = self.k_all[:, :, :T].contiguous()
        self.v_pre = self.v_all[:, :, :T].contiguous()
        self.k_new = self.k_all[:, :, T:].permute(2, 0, 1, 3).contiguous()  # [n_new, B, Hkv, d]
        self.v_new = self.v_all[:, :, T:].permute(2, 0, 1, 3).contiguous()
        self.q_all = bf16_tensor(L.q, dev)                    # [n_new, B, Hq, d]
        self.pos_all = (T + torch.arange(n_new, dtype=torch.int64, device=dev)).repeat_interleave(B).view(n_new, B)
        self.seq_all = (self.pos_all + 1).to(torch.int32)
        self.out = torch.zeros((B, Hq, d), dtype=torch.float32, device=dev)
        # zero-filled before first use: the decode's arrival counters live here
        self.ws = torch.zeros(kvtc.kv_decode_workspace_bytes(self.P, B, Hkv, Hq, self.T_cap), dtype=torch.uint8,
                              device=dev)
        self.scale = 1.0 / math.sqrt(d)
        self.pos0 = torch.zeros(B, dtype=torch.int64, device=dev)

    def check(self):
        assert self.kvtc.kv_check_status() == self.kvtc.KV_OK, self.kvtc.kv_last_error()

    def prefill(self):
        self.kvtc.kv_encode(self.P, self.cache, self.k_pre, self.v_pre, self.kvtc.KV_DTYPE_BF16, self.w.B, self.w.T,
                            self.pos0)

    def time_prefill(self, reps=5):
        """Prefill encode of the whole context, seconds (median of reps; L2 flushed before each)."""
        torch = self.gpu.torch
        ts = []
        for _ in range(reps + 1):
            self.gpu.flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(1_000_000)  # the host's tensor-map setup and launch happen while this runs
            e0.record(self.gpu.stream)
            self.prefill()
            e1.record(self.gpu.stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e-3)
        self.check()
        return float(np.median(ts[1:]))

    def append(self, i):
        self.kvtc.kv_encode(self.P, self.cache, self.k_new[i], self.v_new[i], self.kvtc.KV_DTYPE_BF16, self.w.B, 1,
                            self.pos_all[i])

    def decode(self, i):
        self.kvtc.kv_attend_decode(self.P, self.cache, self.q_all[i], self.w.B, self.w.Hq, self.seq_all[i],
                                   self.scale, self.out, self.ws)

    def time_bf16(self, steps):
        """The uncompressed bf16 flash-decode comparator over the same tokens and queries: per-call seconds."""
        torch, w, dev = self.gpu.torch, self.w, self.gpu.dev
        kb = torch.zeros((w.B, w.Hkv, self.T_cap, w.d), dtype=torch.bfloat16, device=dev)
        vb = torch.zeros((w.B, w.Hkv, self.T_cap, w.d), dtype=torch.bfloat16, device=dev)
        kb[:, :, :self.k_all.shape[2]] = self.k_all
        vb[:, :, :self.v_all.shape[2]] = self.v_all
        ws_b = torch.zeros(self.kvtc.kv_decode_bf16_workspace_bytes(w.B, w.Hkv, w.Hq, self.T_cap),
                           dtype=torch.uint8, device=dev)
        out_b = torch.zeros_like(self.out)
        gs = [self.gpu.graph(lambda i=i: self.kvtc.kv_attend_decode_bf16(
            kb, vb, w.B, w.Hkv, w.Hq, self.T_cap, self.q_all[i], self.seq_all[i], self.scale, out_b, ws_b))
            for i in steps]
        torch.cuda.synchronize()
        self.gpu.timed([[g.replay] for g in gs[:3]])
        t = self.gpu.timed([[g.replay] for g in gs])[:, 0]
        self.check()
        return t

    def time_e2e(self, steps):
        """End to end through the C ABI with host buffers, as a serving loop runs it: each step's new key, value
        and query go over from one pinned host buffer in one copy, the append and the decode run, and the output
        comes back into the step's own pinned host slot. The host enqueues the steps without waiting for the
        device (L2 flushed before each step, outside its events); each step is timed by events on the stream.
        A second pass waits for every step on the host and times it by the host clock. Returns (per-step seconds
        on the device, per-step host seconds of the waiting pass, bytes in, bytes out per step)."""
        torch, dev = self.gpu.torch, self.gpu.dev
        n_new = self.k_new.shape[0]
        nk, nq = self.k_new[0].numel(), self.q_all[0].numel()
        in_h = torch.cat([self.k_new.reshape(n_new, -1), self.v_new.reshape(n_new, -1),
                          self.q_all.reshape(n_new, -1)], dim=1).cpu().pin_memory()
        in_d = torch.empty_like(in_h[0], device=dev)
        k_d = in_d[:nk].view(self.k_new.shape[1:])
        v_d = in_d[nk:2 * nk].view(self.v_new.shape[1:])
        q_d = in_d[2 * nk:2 * nk + nq].view(self.q_all.shape[1:])
        out_h = torch.empty((n_new,) + tuple(self.out.shape), dtype=torch.float32).pin_memory()
        sid = self.gpu.stream.cuda_stream
        kv = self.kvtc

        def one_step(i):
            in_d.copy_(in_h[i], non_blocking=True)
            kv.kv_encode(self.P, self.cache, k_d, v_d, kv.KV_DTYPE_BF16, self.w.B, 1, self.pos_all[i], stream=sid)
            kv.kv_attend_decode(self.P, self.cache, q_d, self.w.B, self.w.Hq, self.seq_all[i], self.scale, self.out,
                                self.ws, stream=sid)
            out_h[i].copy_(self.out, non_blocking=True)

        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in steps]
        torch.cuda.synchronize()
        torch.cuda._sleep(int(2e7))
        for i, (e0, e1) in zip(steps, evs):
            self.gpu.flush_l2()
            e0.record(self.gpu.stream)
            one_step(i)
            e1.record(self.gpu.stream)
        torch.cuda.synchronize()
        te = np.array([e0.elapsed_time(e1) * 1e-3 for e0, e1 in evs])
        ts = []
        for i in steps:
            self.gpu.flush_l2()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            one_step(i)
            torch.cuda.synchronize()
            ts.append(time.perf_counter() - t0)
        self.check()
        ref = self.out.cpu()
        assert torch.equal(out_h[steps[-1]], ref), "the output read back differs from the device's"
        return te, np.array(ts), (k_d.numel() + v_d.numel() + q_d.numel()) * 2, self.out.numel() * 4


def decode_workload(gpu, name, bits, L, n_new, peak):
    """One decode workload at one bit budget: calibration (timed on the host), prefill encode (timed), every
    appended token encoded, then the decode call on its own over contexts T + 5 .. T + n_new (graph replays, L2
    flushed before each), the bf16 comparator over the same tokens and queries, and the end-to-end figure."""
    from transform_coded_kv_02_b300 import synth
    w = synth.WORKLOADS[name]
    lay = Layer(gpu, w, L, bits, n_new)
    t_pre = lay.time_prefill(3)
    lay.prefill()
    for i in range(n_new):  # every appended token is in the cache: decode i reads T + i + 1 tokens
        lay.append(i)
    steps = list(range(4, n_new))
    gs = [gpu.graph(lambda i=i: lay.decode(i)) for i in range(n_new)]
    gpu.torch.cuda.synchronize()
    gpu.timed([[g.replay] for g in gs[:4]])
    t = gpu.timed([[gs[i].replay] for i in steps])[:, 0]
    lay.check()
    del gs
    dec_bytes = float(np.mean([decode_bytes(w.T + i + 1, w, lay.rk_w, lay.rv_w) for i in steps]))
    dec = float(np.mean(t))
    t_b = lay.time_bf16(steps)
    b_avg = float(np.mean(t_b))
    b_bytes = float(np.mean([bf16_decode_bytes(w.T + i + 1, w) for i in steps]))
    e_steps = steps[:8]
    te, ts, h2d, d2h = lay.time_e2e(e_steps)
    e2e_bytes = float(np.mean([step_bytes(w.T + i + 1, w, lay.rk_w, lay.rv_w) for i in e_steps]))
    pre_tok = w.B * w.Hkv * w.T
    achieved = dec_bytes / dec / 1e9
    entry = {"workload": workload_name(w, bits, lay.rk_w, lay.rv_w, steps=False),
             "decode": {"avg_us": dec * 1e6, "p10_us": float(np.percentile(t, 10)) * 1e6,
                        "p90_us": float(np.percentile(t, 90)) * 1e6, "calls": len(steps),
                        "tokens_per_s": w.B / dec},
             "roofline": {"bound": "hbm", "kernel": "kv_attend_decode (decode_kernel)", "achieved": achieved,
                          "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                          "algorithmic_bytes_per_launch": dec_bytes},
             "bf16_flash_decode": {"avg_us": b_avg * 1e6, "gbs": b_bytes / b_avg / 1e9,
                                   "frac": b_bytes / b_avg / 1e9 / peak, "speedup_packed_vs_bf16": b_avg / dec},
             "e2e": {"value": e2e_bytes / float(np.mean(te)) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
                     "d2h_bytes_per_step": d2h, "step_us": float(np.mean(te)) * 1e6,
                     "host_waits_each_step_us": float(np.median(ts)) * 1e6},
             "prefill_encode": {"token_heads": pre_tok, "seconds": t_pre, "token_heads_per_s": pre_tok / t_pre,
                                "gbs": encode_bytes(pre_tok, w.d, lay.rk_w, lay.rv_w) / t_pre / 1e9},
             "kv_calibrate_s": lay.calibrate_s, "parameter_sets": len(L.calib_k)}
    del lay
    return entry


def prefill_stack(gpu, peak):
    """The 32-layer prefill stack. Per layer: tokens drawn on the device (4 sequences x 8 KV heads x 65536 bf16
    tokens), kv_calibrate on the 4096-token calibration slice (host, timed), kv_encode of every token (timed on
    the device, L2 flushed before), then one decode step over the whole context (timed)."""
    from transform_coded_kv_02_b300 import kvtc, synth
    torch, dev = gpu.torch, gpu.dev
    w = synth.WORKLOADS["llama_prefill_32l"]
    B, Hkv, Hq, T, d = w.B, w.Hkv, w.Hq, w.T, w.d
    enc_t, dec_t, cal_t = [], [], []
    rk_w = rv_w = None
    for layer in range(w.layers):
        Ld = synth.make_layer_device(w, layer, dev)
        t0 = time.perf_counter()
        P = kvtc.kv_calibrate(list(zip(Ld.calib_k, Ld.calib_v, Ld.calib_q)), BITS, BITS)
        cal_t.append(time.perf_counter() - t0)
        P.upload()
        rk_w, rv_w = P.record_words(0), P.record_words(1)
        rk = torch.zeros((B, Hkv, T, rk_w), dtype=torch.int32, device=dev)
        rv = torch.zeros((B, Hkv, T // 2, 2 * rv_w), dtype=torch.int32, device=dev)
        cache = kvtc.make_cache(rk, rv, B, Hkv, T, False)
        pos0 = torch.zeros(B, dtype=torch.int64, device=dev)
        q = bf16_tensor(Ld.q[0], dev)
        sl = torch.full((B,), T, dtype=torch.int32, device=dev)
        out = torch.zeros((B, Hq, d), dtype=torch.float32, device=dev)
        ws = torch.zeros(kvtc.kv_decode_workspace_bytes(P, B, Hkv, Hq, T), dtype=torch.uint8, device=dev)
        gpu.flush_l2()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        torch.cuda._sleep(1_000_000)
        e[0].record(gpu.stream)
        kvtc.kv_encode(P, cache, Ld.k, Ld.v, kvtc.KV_DTYPE_BF16, B, T, pos0)
        e[1].record(gpu.stream)
        kvtc.kv_attend_decode(P, cache, q, B, Hq, sl, 1.0 / math.sqrt(d), out, ws)
        e[2].record(gpu.stream)
        torch.cuda.synchronize()
        assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
        assert bool(torch.isfinite(out).all())
        enc_t.append(e[0].elapsed_time(e[1]) * 1e-3)
        dec_t.append(e[1].elapsed_time(e[2]) * 1e-3)
        del Ld, rk, rv, cache, ws, P
    tok = w.layers * B * Hkv * T
    secs = float(np.sum(enc_t))
    gbs = encode_bytes(tok, d, rk_w, rv_w) / secs / 1e9
    return {"workload": f"{DESCRIPTION[w.name]}: {w.layers} layers x batch {B} x {T} tokens x {Hkv} kv heads, d={d}, "
                        f"bf16, {BITS} bits/elem (K {rk_w} + V {rv_w} words/token), calibration on the {w.n_calib}-"
                        f"token prefix of sequence 0 of each layer",
            "encode": {"token_heads": tok, "seconds": secs, "token_heads_per_s": tok / secs,
                       "tokens_per_s": w.layers * B * T / secs, "gbs": gbs, "frac_of_hbm": gbs / peak,
                       "per_layer_us": float(np.mean(enc_t)) * 1e6},
            "kv_calibrate_s_per_layer": float(np.mean(cal_t)),
            "decode_per_layer_us": float(np.mean(dec_t)) * 1e6}


def paged_workload(gpu, w, L, peak, page=256, n_layers=4, rope_base=500000.0):
    """The headline layer's prefill in pages of `page` tokens scattered over the pool, the query's rotary embedding
    applied in the decode kernel; decode calls of one layer and of n_layers layers in one launch (the layer's
    records and parameters repeated per layer), graph replays with L2 flushed before each."""
    from transform_coded_kv_02_b300 import kvtc
    torch, dev = gpu.torch, gpu.dev
    B, Hkv, Hq, d, T = w.B, w.Hkv, w.Hq, w.d, w.T
    P = kvtc.kv_calibrate(list(zip(L.calib_k, L.calib_v, L.calib_q)) * n_layers, BITS, BITS)
    P.set_rope(rope_base).upload()
    rk_w, rv_w = P.record_words(0), P.record_words(1)
    max_pages = (T + page - 1) // page
    Z = n_layers * B
    n_pages = Z * max_pages
    bt_np = np.random.default_rng(7).permutation(n_pages).astype(np.int32).reshape(Z, max_pages)
    bt = torch.from_numpy(bt_np).to(dev)
    kp = torch.zeros((n_pages, Hkv, page, rk_w), dtype=torch.int32, device=dev)
    vp = torch.zeros((n_pages, Hkv, page // 2, 2 * rv_w), dtype=torch.int32, device=dev)
    k = bf16_tensor(L.k[:, :, :T], dev)
    v = bf16_tensor(L.v[:, :, :T], dev)
    kl = k.unsqueeze(0).expand(n_layers, *k.shape).contiguous()
    vl = v.unsqueeze(0).expand(n_layers, *v.shape).contiguous()
    c_all = kvtc.make_paged_cache(kp, vp, n_pages, page, Hkv, B, n_layers, max_pages, bt, False, 0)
    kvtc.kv_encode_paged(P, c_all, kl, vl, kvtc.KV_DTYPE_BF16, T, torch.zeros(B, dtype=torch.int64, device=dev))
    del kl, vl
    c_one = kvtc.make_paged_cache(kp, vp, n_pages, page, Hkv, B, 1, max_pages, bt, False, 0)
    q = bf16_tensor(L.q[0], dev)
    ql = q.unsqueeze(0).expand(n_layers, *q.shape).contiguous()
    seq = torch.full((B,), T, dtype=torch.int32, device=dev)
    qpos = torch.full((B,), T - 1, dtype=torch.int32, device=dev)
    out = torch.zeros((n_layers, B, Hq, d), dtype=torch.float32, device=dev)
    scale = 1.0 / math.sqrt(d)
    ws1 = torch.zeros(kvtc.kv_decode_paged_workspace_bytes(P, c_one, Hq), dtype=torch.uint8, device=dev)
    wsn = torch.zeros(kvtc.kv_decode_paged_workspace_bytes(P, c_all, Hq), dtype=torch.uint8, device=dev)
    g1 = gpu.graph(lambda: kvtc.kv_attend_decode_paged(P, c_one, ql[0], Hq, seq, qpos, scale, out[0], ws1))
    gn = gpu.graph(lambda: kvtc.kv_attend_decode_paged(P, c_all, ql, Hq, seq, qpos, scale, out, wsn))
    torch.cuda.synchronize()
    gpu.timed([[g1.replay], [gn.replay]])
    t1 = gpu.timed([[g1.replay] for _ in range(24)])[:, 0]
    tn = gpu.timed([[gn.replay] for _ in range(24)])[:, 0]
    assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
    assert bool(torch.isfinite(out).all())
    lb = decode_bytes(T, w, rk_w, rv_w)
    a1, an = float(np.mean(t1)), float(np.mean(tn))
    del g1, gn
    return {"workload": f"{workload_name(w, BITS, rk_w, rv_w, steps=False)}, {page}-token pages in random pool order, "
                        f"query rotary embedding (base {rope_base:g}) in the kernel",
            "decode_one_layer": {"avg_us": a1 * 1e6, "gbs": lb / a1 / 1e9, "frac": lb / a1 / 1e9 / peak},
            f"decode_{n_layers}_layers_one_launch": {"avg_us": an * 1e6, "gbs": n_layers * lb / an / 1e9,
                                                    "frac": n_layers * lb / an / 1e9 / peak,
                                                    "us_per_layer": an / n_layers * 1e6},
            "algorithmic_bytes_per_layer": lb}


def token_axis_workload(gpu, w, L, peak, full_decode_us, W=32, keep_frac=0.25):
    """Token-axis allocation on the headline layer after its prefill: token weights from W observation queries per
    query head (two tensor-core passes over the bf16 keys), the kept tokens (keep_frac of the context), record
    compaction, then the decode over the kept tokens; each call timed on its own (graph replays, L2 flushed)."""
    from transform_coded_kv_02_b300 import kvtc
    torch, dev = gpu.torch, gpu.dev
    B, Hkv, Hq, d, T = w.B, w.Hkv, w.Hq, w.d, w.T
    W = min(W, L.q.shape[0], 128 // (Hq // Hkv))
    P = kvtc.kv_calibrate(list(zip(L.calib_k, L.calib_v, L.calib_q)), BITS, BITS).upload()
    rk_w, rv_w = P.record_words(0), P.record_words(1)
    T_cap = (T + 15) // 16 * 16
    k = bf16_tensor(L.k[:, :, :T], dev)
    v = bf16_tensor(L.v[:, :, :T], dev)
    q_obs = bf16_tensor(np.ascontiguousarray(np.transpose(L.q[:W], (1, 2, 0, 3))), dev)
    rk = torch.zeros((B, Hkv, T_cap, rk_w), dtype=torch.int32, device=dev)
    rv = torch.zeros((B, Hkv, T_cap // 2, 2 * rv_w), dtype=torch.int32, device=dev)
    src = kvtc.make_cache(rk, rv, B, Hkv, T_cap)
    kvtc.kv_encode(P, src, k, v, kvtc.KV_DTYPE_BF16, B, T, torch.zeros(B, dtype=torch.int64, device=dev))
    keep = int(keep_frac * T)
    lam = torch.zeros((B, Hkv, T), dtype=torch.float32, device=dev)
    wsw = torch.empty(kvtc.kv_token_weights_workspace_bytes(B, Hkv, T), dtype=torch.uint8, device=dev)
    idx = torch.zeros((B, Hkv, keep), dtype=torch.int32, device=dev)
    ck = torch.zeros((B, Hkv, T_cap, rk_w), dtype=torch.int32, device=dev)
    cv = torch.zeros((B, Hkv, T_cap // 2, 2 * rv_w), dtype=torch.int32, device=dev)
    dst = kvtc.make_cache(ck, cv, B, Hkv, T_cap)
    scale = 1.0 / math.sqrt(d)
    q = bf16_tensor(L.q[W % L.q.shape[0]], dev)
    seq = torch.full((B,), keep, dtype=torch.int32, device=dev)
    out = torch.zeros((B, Hq, d), dtype=torch.float32, device=dev)
    wsd = torch.zeros(kvtc.kv_decode_workspace_bytes(P, B, Hkv, Hq, T_cap), dtype=torch.uint8, device=dev)
    calls = {"weights": lambda: kvtc.kv_token_weights(q_obs, W, k, B, Hkv, Hq, T, scale, lam, wsw),
             "select": lambda: kvtc.kv_token_select(lam, B, Hkv, T, keep, idx),
             "compact": lambda: kvtc.kv_cache_compact(P, src, dst, B, idx, keep),
             "decode": lambda: kvtc.kv_attend_decode(P, dst, q, B, Hq, seq, scale, out, wsd)}
    graphs = {n: gpu.graph(f) for n, f in calls.items()}
    torch.cuda.synchronize()
    order = ["weights", "select", "compact", "decode"]
    gpu.timed([[graphs[n].replay for n in order]])
    t = gpu.timed([[graphs[n].replay for n in order] for _ in range(12)])
    assert kvtc.kv_check_status() == kvtc.KV_OK, kvtc.kv_last_error()
    assert bool(torch.isfinite(out).all())
    avg = {n: float(np.mean(t[:, i])) for i, n in enumerate(order)}
    bh = B * Hkv
    w_bytes = 2 * bh * T * d * 2 + B * Hq * W * d * 2 + bh * T * 4          # keys read twice, queries, weights out
    s_bytes = 5 * bh * T * 4 + bh * keep * 4                                  # 4 radix rounds and the output pass
    c_bytes = 2 * bh * keep * (rk_w + rv_w) * 4 + bh * keep * 4               # kept records in and out, indices
    d_bytes = decode_bytes(keep, w, rk_w, rv_w)
    del graphs
    return {"workload": f"{workload_name(w, BITS, rk_w, rv_w, steps=False)}: {W} observation queries per query "
                        f"head, {keep} of {T} tokens kept per KV head ({keep_frac:g})",
            "token_weights": {"avg_us": avg["weights"] * 1e6, "gbs": w_bytes / avg["weights"] / 1e9,
                              "bound": "hbm (keys read in each of two passes)"},
            "token_select": {"avg_us": avg["select"] * 1e6, "gbs": s_bytes / avg["select"] / 1e9},
            "compact": {"avg_us": avg["compact"] * 1e6, "gbs": c_bytes / avg["compact"] / 1e9},
            "decode_kept": {"avg_us": avg["decode"] * 1e6, "gbs": d_bytes / avg["decode"] / 1e9,
                            "frac": d_bytes / avg["decode"] / 1e9 / peak,
                            "speedup_vs_full_context": full_decode_us / (avg["decode"] * 1e6)}}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    gpu = Gpu(local_rank)
    K, W = args.steps, args.warmup
    n_new = K + W
    w, L = make_workload(n_new, layer=rank)
    lay = Layer(gpu, w, L, BITS, n_new)
    B, d, T = w.B, w.d, w.T
    rk_w, rv_w = lay.rk_w, lay.rv_w
    peak, peak_kind = measured_peaks()

    # prefill encode (reported beside the step metric)
    enc_t = lay.time_prefill(5)
    enc_tok = B * w.Hkv * T
    lay.prefill()

    # one CUDA graph per step holding the append and the decode (pointers of step i baked in), so that the
    # timed loop is one host call per step and the device never waits on the host; separate append-only and
    # decode-only graphs time the two calls on their own (the decode one for the roofline figure)
    g_step = [gpu.graph(lambda i=i: (lay.append(i), lay.decode(i))) for i in range(n_new)]
    g_enc = [gpu.graph(lambda i=i: lay.append(i)) for i in range(n_new)]
    g_dec = [gpu.graph(lambda i=i: lay.decode(i)) for i in range(n_new)]
    torch.cuda.synchronize()
    gpu.timed([[g_step[i].replay] for i in range(W)])
    lay.check()

    clocks = ClockSampler(local_rank) if rank == 0 else None
    if clocks:
        clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    t_step = gpu.timed([[g_step[W + j].replay] for j in range(K)])[:, 0]
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    lay.check()
    # the two calls on their own, over the same steps (the appends rewrite the same records)
    t_dec = gpu.timed([[g_dec[W + j].replay] for j in range(K)])[:, 0]
    t_app = gpu.timed([[g_enc[W + j].replay] for j in range(K)])[:, 0]
    lay.check()
    del g_step, g_enc, g_dec
    total = max_over_ranks(float(np.sum(t_step)), world, gpu.dev)
    ctx = [T + W + j + 1 for j in range(K)]
    value = job_gbs(sum(step_bytes(c, w, rk_w, rv_w) for c in ctx), total, world)
    dec_bytes_avg = float(np.mean([decode_bytes(c, w, rk_w, rv_w) for c in ctx]))
    dec_avg = float(np.mean(t_dec))
    achieved = dec_bytes_avg / dec_avg / 1e9

    nb = list(range(W, W + min(K, 64)))
    t_b = lay.time_bf16(nb)
    bf16_avg = float(np.mean(t_b))
    bf16_bytes = float(np.mean([bf16_decode_bytes(T + i + 1, w) for i in nb]))
    dec_same = float(np.mean(t_dec[:len(nb)]))
    te, ts, h2d, d2h = lay.time_e2e(nb)
    e2e_bytes = float(np.mean([step_bytes(T + i + 1, w, rk_w, rv_w) for i in nb]))
    e2e_val = job_gbs(e2e_bytes, max_over_ranks(float(np.mean(te)), world, gpu.dev), world)
    del lay

    workloads = None
    if not args.no_workloads:
        from transform_coded_kv_02_b300 import synth
        workloads = {}
        held = {}
        for name, bits in EXTRA_DECODE:
            if name not in held:
                wx = synth.WORKLOADS[name]
                held = {name: synth.make_layer(wx, layer=rank, T=wx.T + 28, steps=28)}  # one layer held at a time
            workloads[f"{name}@{bits}"] = decode_workload(gpu, name, bits, held[name], 28, peak)
        del held
        workloads["llama_prefill_32l@2.75"] = prefill_stack(gpu, peak)
        workloads["llama_decode_32k_paged@2.75"] = paged_workload(gpu, w, L, peak)
        workloads["llama_decode_32k_token_axis@2.75"] = token_axis_workload(gpu, w, L, peak, dec_avg * 1e6)

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        if n_new < args.cpu_steps + 1:
            w, L = make_workload(args.cpu_steps + 1)
        cpu = cpu_baseline(w, L, BITS, args.cpu_steps)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": total / K * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u32-packed codes, f16 mma / f32 accumulate", "data": "synthetic",
        "config": {"workload": workload_name(w, BITS, rk_w, rv_w),
                   "l2": "flushed before every timed step (2 x L2 buffer written, outside the timed events)",
                   "parallelism": "replicas" if world > 1 else "single gpu"},
        "roofline": {"bound": "hbm", "kernel": "kv_attend_decode (decode_kernel)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "frac_of_nominal_8tbs": achieved / 8000.0,
                     "traffic": recorded_traffic(), "algorithmic_bytes_per_launch": dec_bytes_avg,
                     "avg_launch_us": dec_avg * 1e6},
        "decode": {"tokens_per_s": B / dec_avg, "avg_us": dec_avg * 1e6,
                   "p10_us": float(np.percentile(t_dec, 10)) * 1e6, "p90_us": float(np.percentile(t_dec, 90)) * 1e6},
        "append_encode": {"avg_us": float(np.mean(t_app)) * 1e6},
        "bf16_flash_decode": {"avg_us": bf16_avg * 1e6, "gbs": bf16_bytes / bf16_avg / 1e9,
                              "frac": bf16_bytes / bf16_avg / 1e9 / peak,
                              "speedup_packed_vs_bf16": bf16_avg / dec_same},
        "prefill_encode": {"token_heads": enc_tok, "seconds": enc_t, "token_heads_per_s": enc_tok / enc_t,
                           "gbs": encode_bytes(enc_tok, d, rk_w, rv_w) / enc_t / 1e9},
        "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "step_us": float(np.mean(te)) * 1e6, "host_waits_each_step_us": float(np.median(ts)) * 1e6,
                "how": "kv_encode + kv_attend_decode through the C ABI, step inputs copied from pinned host memory "
                       "and the output read back every step, steps enqueued without host waits, per-step events"},
        "gpu_launches": 2 * K,
        "wall_s_timed_loop_with_flushes": wall,
        "step_us": {"avg": float(np.mean(t_step)) * 1e6, "p10": float(np.percentile(t_step, 10)) * 1e6,
                    "p90": float(np.percentile(t_step, 90)) * 1e6},
        "clocks": clk,
        "cpu_baseline": cpu,
        "workloads": workloads,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
