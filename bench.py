"""Benchmark: one transformer block's streamed QKV projection + packed-INT4-K/V
attention on the H3 Ref2VA-sized workload (N = 152,263 tokens, hidden 7168,
56 heads x 128), on synthetic seeded inputs.

One step = streamed_qkv_proj (x . W^T on the tensor cores, Q kept BF16 and
rotated, K / V rotated, group-scaled (32) and packed to INT4) followed by
packed_kv_attention (Q against the packed K/V, output written over Q).

Prints one JSON line (rank 0).  `value` is block TFLOP/s:
(2 N C 3C + 4 N^2 C) / step time, over all ranks.  Every rank runs an
independent block (its own seed): the work per GPU is fixed (weak scaling)
and no data crosses ranks; only the timings are reduced (max).

Besides the device-timed block the line carries: the same block end to end
through the public calls with x coming from and the output going to pinned
host memory (e2e), the two-phase form that never holds Q or the output whole
on the device (e2e_two_phase), the two-phase form with the packed K/V store
itself in host memory, streamed back chunk by chunk into a key-chunked
attention (e2e_host_staged), the standalone rotate + quantise + pack kernel
and its inverse on K/V [262,144, 2 x 7168] (kernels.pack), the peak memory
against materialising the BF16 QKV, and the CPU oracle's time on a sample
(cpu_baseline).  Each end-to-end leg records its own SM clocks and the rate
its copies got from the host link (host_link, CUDA events around each copy):
that rate differs from box to box and over time, and the legs depend on it.

--impl reference times the CPU oracle (the plain C reference implementation
of the same computation) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

E2E_IN_CHUNK = 16384   # tokens per host-to-device chunk of x in the end-to-end step
E2E_OUT_CHUNK = 19456  # query rows per attention launch in the end-to-end step (38 CTA pairs)
E2E_EARLY_QUERY_CHUNKS = 1  # query chunks of the end-to-end step attended while x is still arriving
E2E_KV_CHUNK = 16384   # keys per host-staged chunk of the packed store
E2E_STEPS, E2E_WARMUP = 10, 2  # end-to-end steps timed (at most --steps), after these untimed ones
PACK_N = 262144        # the standalone pack / unpack record: K/V [N, 2 x 7168], group 32
METRIC = "block TFLOP/s + tokens/s (QKV GEMM + INT4-KV attn) at N=152,263; peak GiB"
GiB = 2.0 ** 30


def flops(n: int, C: int, causal: bool = False) -> tuple[float, float]:
    """(projection FLOPs, attention FLOPs) of one block; causal: row i sees i + 1 keys."""
    return 2.0 * n * C * 3 * C, (2.0 * n * (n + 1) * C if causal else 4.0 * n * n * C)


ATTENTION_SOURCES = ("attention.cu", "ptx.cuh", "quant.cuh", "internal.h")


def code_text(text):
    """C/CUDA source without comments, whitespace runs collapsed to one space."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def attention_code_sha256():
    """sha256 of the attention kernel's sources with comments and whitespace runs
    removed: the key under which DRAM counters of an ncu capture stay valid."""
    import hashlib
    h = hashlib.sha256()
    for name in ATTENTION_SOURCES:
        with open(os.path.join(ROOT, "serving_tcgen05_streamed_gb300", "csrc", name)) as f:
            h.update((name + "\0" + code_text(f.read()) + "\0").encode())
    return h.hexdigest()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


class LinkMeter:
    """Times each host<->device copy of an end-to-end leg with a pair of CUDA
    events on the copy's own stream (recorded after any wait the stream was
    given, so only the copy itself is timed), and reports the rate the host
    link delivered in each direction over the timed steps."""

    def __init__(self):
        self.pending = []
        self.reset()

    def reset(self):
        self.pending.clear()
        self.bytes = {"h2d": 0, "d2h": 0}
        self.ms = {"h2d": 0.0, "d2h": 0.0}

    def copy(self, dst, src, s, kind: str):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            a.record(s)
            dst.copy_(src, non_blocking=True)
            b.record(s)
        self.pending.append((kind, a, b, dst.numel() * dst.element_size()))

    def collect(self):  # after a synchronize
        for kind, a, b, nb in self.pending:
            self.ms[kind] += a.elapsed_time(b)
            self.bytes[kind] += nb
        self.pending.clear()

    def record(self) -> dict:
        return {k + "_gbs": (self.bytes[k] / (self.ms[k] * 1e6) if self.ms[k] > 0 else None) for k in ("h2d", "d2h")}


def dist_setup(gpus: int, backend: str = "nccl"):
    """One process per GPU (torchrun): returns (world, rank, local_rank).
    Every rank runs its own independent block; the process group is used only
    for barriers and for the max of the per-rank times."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float) -> float:
    """The largest of the ranks' values (the job takes as long as its slowest rank)."""
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def timed_leg(step, steps: int, world: int, device_index: int, meter: LinkMeter | None = None):
    """Runs E2E_WARMUP untimed steps, then `steps` timed ones (wall clock, each
    step ends synchronised), sampling the SM clock over the timed region; the
    meter, if any, keeps the copies of the timed steps only.
    Returns (seconds per step, max over ranks; clock record)."""
    for _ in range(E2E_WARMUP):
        step()
    torch.cuda.synchronize()
    if meter is not None:
        meter.reset()
    barrier(world)
    sampler = ClockSampler(device_index)
    sampler.start()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    secs = (time.perf_counter() - t0) / steps
    clocks = sampler.stop()
    if meter is not None:
        meter.collect()
    return max_over_ranks(world, secs), clocks


def query_chunks(n: int, tail: int = 2048) -> list[tuple[int, int]]:
    """Query-row chunks of the end-to-end legs: E2E_OUT_CHUNK rows each, then
    the rest in halving pieces (multiples of 256 rows) down to at most `tail`
    rows, so that the copy of the last chunk's output, which no attention
    overlaps, stays small.  Returns (first row, rows) pairs tiling [0, n)."""
    out, s0 = [], 0
    while s0 < n:
        rest = n - s0
        if rest >= 2 * E2E_OUT_CHUNK:
            ln = E2E_OUT_CHUNK
        elif rest <= tail:
            ln = rest
        else:
            ln = min(E2E_OUT_CHUNK, (rest // 2 + 255) // 256 * 256)
        out.append((s0, ln))
        s0 += ln
    return out


def job_value(world: int, rank_ms_total: float, steps: int, flops_per_block: float) -> tuple[float, float]:
    """(ms per step, whole-job TFLOP/s): every rank runs one block per step, the
    step time is the slowest rank's."""
    total = max_over_ranks(world, rank_ms_total)
    ms = total / steps
    return ms, world * flops_per_block / (ms * 1e-3) / 1e12


# --------------------------------------------------------------------------- CPU oracle (reference arm / baseline)
def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or "unknown"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


class CpuOracleSample:
    """The CPU oracle on a bounded sample of the block: the projection of
    token rows and the attention of query rows (all heads, all N keys).  Both
    are exact per row, so the time per row extrapolates to the whole block.
    Inputs come from the seeded generators (generated once, on the GPU when
    there is one, and copied to the host)."""

    def __init__(self, wl, seed: int, proj_rows: int, attn_rows: int):
        import oracle
        from serving_tcgen05_streamed_gb300 import inputs

        self.wl = wl
        n, C = wl.n, wl.hidden
        heads = C // 128
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        as_u16 = lambda t: t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
        x, w, qn, kn = inputs.block_inputs(wl, device=dev)
        rows = inputs.sample_rows(n, proj_rows, seed=seed).numpy()
        self.xb = as_u16(x[torch.as_tensor(rows, device=dev)])
        self.wb = as_u16(w)
        self.qn = None if qn is None else qn.cpu().numpy()
        self.kn = None if kn is None else kn.cpu().numpy()
        del x, w
        cap = ((n + 127) // 128) * 128
        kc, vc, ks, vs = inputs.random_packed_kv(heads, n, cap, 32, 4, seed=seed, device=dev)
        self.kc, self.vc, self.ks, self.vs = kc.cpu().numpy(), vc.cpu().numpy(), as_u16(ks), as_u16(vs)
        del kc, vc, ks, vs
        self.q = as_u16(inputs.random_q(attn_rows, C, seed=seed))
        oracle.build()
        self.cores = oracle.threads()

    def describe(self, proj_rows: int, attn_rows: int) -> str:
        return (f"{proj_rows} projection rows + {attn_rows} attention query rows ({self.wl.heads} heads x "
                f"{self.wl.n} keys); time per row extrapolated to N={self.wl.n}")

    def time_rows(self, proj_rows: int, attn_rows: int, threads: int | None = None):
        """Seconds per projection row and per attention query row, on `threads`
        OpenMP threads (default: all)."""
        import oracle
        oracle.set_threads(threads or self.cores)
        try:
            t0 = time.perf_counter()
            oracle.qkv_proj(self.xb[:proj_rows], self.wb, q_norm_w=self.qn, k_norm_w=self.kn)
            t_proj = (time.perf_counter() - t0) / proj_rows
            t0 = time.perf_counter()
            oracle.attention(self.q[:attn_rows], self.kc, self.vc, self.ks, self.vs, n_kv=self.wl.n)
            t_attn = (time.perf_counter() - t0) / attn_rows
        finally:
            oracle.set_threads(self.cores)
        return t_proj, t_attn

    def run(self, proj_rows: int, attn_rows: int, threads: int | None = None) -> float:
        """Extrapolated block seconds."""
        t_proj, t_attn = self.time_rows(proj_rows, attn_rows, threads)
        return (t_proj + t_attn) * self.wl.n


def run_reference(args, wl, world, rank):
    if rank != 0:
        return
    cpu = CpuOracleSample(wl, seed=100, proj_rows=args.ref_proj_rows, attn_rows=args.ref_attn_rows)
    secs = []
    for i in range(args.warmup + args.steps):
        t = cpu.run(args.ref_proj_rows, args.ref_attn_rows)
        if i >= args.warmup:
            secs.append(t)
    t_block = sum(secs) / len(secs)
    v = sum(flops(wl.n, wl.hidden)) / t_block / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_block * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 (fp64 accumulation)", "data": "synthetic (seeded generators)",
        "config": {"workload": wl.name, "n_tokens": wl.n, "hidden": wl.hidden, "heads": wl.heads, "group": 32,
                   "kv_bits": 4},
        "tokens_per_s": wl.n / t_block,
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cpu.cores, "kind": "oracle",
                         "sample": cpu.describe(args.ref_proj_rows, args.ref_attn_rows) + " (extrapolated)",
                         "cpu_model": cpu_model()},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(wl, fp: float, fa: float, proj_rows: int, attn_rows: int, single_proj_rows: int,
                 single_attn_rows: int) -> dict:
    """The oracle on the host cores: all cores on the CPU-baseline plan's sample
    (projection rows + query rows, per-row times extrapolated to the block),
    and one core on a smaller sample."""
    n = wl.n
    sample = CpuOracleSample(wl, seed=7, proj_rows=max(proj_rows, single_proj_rows),
                             attn_rows=max(attn_rows, single_attn_rows))
    tp, ta = sample.time_rows(proj_rows, attn_rows)
    tp1, ta1 = sample.time_rows(single_proj_rows, single_attn_rows, threads=1)
    return {"value": (fp + fa) / ((tp + ta) * n) / 1e12, "unit": "TFLOP/s", "cores": sample.cores, "kind": "oracle",
            "sample": sample.describe(proj_rows, attn_rows) + " (extrapolated)",
            "cpu_model": cpu_model(),
            "s_per_projection_row": tp, "s_per_query_row": ta, "block_s_extrapolated": (tp + ta) * n,
            "single_core": {"value": (fp + fa) / ((tp1 + ta1) * n) / 1e12, "unit": "TFLOP/s", "cores": 1,
                            "sample": sample.describe(single_proj_rows, single_attn_rows) + " (extrapolated)",
                            "s_per_projection_row": tp1, "s_per_query_row": ta1,
                            "block_s_extrapolated": (tp1 + ta1) * n}}


# --------------------------------------------------------------------------- GPU arm
def peak_memory(wl, x, w, qn, kn, kvq):
    """Peak bytes allocated by one streamed block (ours) and by the
    materialise-BF16-QKV-then-quantise path, above the resident inputs."""
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    q, store = kvq.streamed_qkv_proj(x, w, group=32, chunk_tokens=wl.chunk_tokens, q_norm_w=qn, k_norm_w=kn)
    kvq.packed_kv_attention(q, store, out=q)
    torch.cuda.synchronize()
    ours = torch.cuda.max_memory_allocated() - base
    del q, store
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    qkv = x @ w.t()  # [N, 3C] BF16 materialised (cuBLAS)
    C = wl.hidden
    store = kvq.kv_rotate_quant_pack(qkv[:, C:], C, 32, 4)
    torch.cuda.synchronize()
    mat = torch.cuda.max_memory_allocated() - base
    del qkv, store
    torch.cuda.synchronize()
    return ours / GiB, mat / GiB


def run_gpu(args, wl, world, rank, local):
    import serving_tcgen05_streamed_gb300 as kvq
    from serving_tcgen05_streamed_gb300 import inputs

    kvq.load()
    n, C = wl.n, wl.hidden
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    x, w, qn, kn = inputs.block_inputs(wl, device=dev)
    if world > 1:  # independent problems per rank
        x = x.roll(rank * 7, dims=0)
    causal = args.workload == "causal"
    wl_label = (wl.name + (", causal attention" if causal else "") + (", RoPE 128 in the projection" if args.rope else "")
                + (", text and audio query rows routed to an INT8 store of every key" if args.route_av else ""))
    rope = None
    if args.rope:  # split-half RoPE table of Q and K: token position t, frequencies 10000^(-2i/128)
        pos = torch.arange(n, dtype=torch.float64, device=dev)[:, None]
        ang = pos * (10000.0 ** (-2.0 * torch.arange(64, dtype=torch.float64, device=dev) / 128))[None, :]
        rope = torch.stack([torch.cos(ang), torch.sin(ang)], dim=-1).to(torch.float32).contiguous()
    fp, fa = flops(n, C, causal)

    mixed = wl is inputs.MIXED
    if mixed:  # INT8 for the conditioning ranges, rotated INT4 for the generated video
        stores = [kvq.PackedKV.empty(seg_n, C, 32, bits, dev) for _, seg_n, bits in inputs.MIXED_SEGMENTS]
        peak_ours = peak_mat = None
    else:
        peak_ours, peak_mat = peak_memory(wl, x, w, qn, kn, kvq)
        stores = [kvq.PackedKV.empty(n, C, 32, 4, dev)]
    store = stores[0]
    q = torch.empty((n, C), dtype=torch.bfloat16, device=dev)
    route = bool(args.route_av) and mixed
    fine = kvq.PackedKV.empty(n, C, 32, 8, dev) if route else None  # INT8 K/V of every key for the routed rows
    # query rows routed to the fine store: the text and audio segments
    routed_segs, start_ = [], 0
    for name_, seg_n, _ in (inputs.MIXED_SEGMENTS if mixed else ()):
        routed_segs.append((start_, seg_n, route and name_ in ("text", "audio")))
        start_ += seg_n

    def attend_rows(qc, s0):
        """Attention of query rows s0 .. s0+len(qc)-1, output over qc."""
        if mixed and not route:
            kvq.packed_kv_attention_mixed(qc, stores, out=qc, stream=stream)
        elif mixed:
            for a, ln_, to_fine in routed_segs:
                lo, hi = max(a, s0), min(a + ln_, s0 + qc.shape[0])
                if lo >= hi:
                    continue
                part = qc[lo - s0:hi - s0]
                kvq.packed_kv_attention_mixed(part, [fine] if to_fine else stores, out=part, stream=stream)
        elif causal:
            kvq.packed_kv_attention_causal(qc, store, q_pos0=s0, out=qc, stream=stream)
        else:
            kvq.packed_kv_attention(qc, store, out=qc, stream=stream)

    def project_fine(xc, s0, ln):
        if route:
            kvq.streamed_qkv_proj_ex(xc, w, [fine.rows(s0, ln)], rope[s0:s0 + ln] if rope is not None else None,
                                     sections=kvq.SECTION_KV, group=32, chunk_tokens=wl.chunk_tokens, q_norm_w=qn,
                                     k_norm_w=kn, stream=stream)

    def project(xin):
        if rope is not None:
            kvq.streamed_qkv_proj_ex(xin, w, stores, rope, group=32, chunk_tokens=wl.chunk_tokens, q_norm_w=qn,
                                       k_norm_w=kn, q_out=q, stream=stream)
        elif mixed:
            kvq.streamed_qkv_proj_mixed(xin, w, stores, group=32, chunk_tokens=wl.chunk_tokens, q_norm_w=qn,
                                        k_norm_w=kn, q_out=q, stream=stream)
        else:
            kvq.streamed_qkv_proj(xin, w, group=32, chunk_tokens=wl.chunk_tokens, q_norm_w=qn, k_norm_w=kn, q_out=q,
                                  store=store, stream=stream)
        project_fine(xin, 0, n)

    def attend():
        attend_rows(q, 0)

    def step():
        ev_p0.record(stream)
        project(x)
        ev_a0.record(stream)
        attend()
        ev_a1.record(stream)

    ev_p0, ev_a0, ev_a1 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert kvq.device_status() == kvq.KVQ_OK

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    attn_ms, proj_ms = [], []
    for i in range(args.steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
        ends[i].synchronize()
        attn_ms.append(ev_a0.elapsed_time(ev_a1))
        proj_ms.append(ev_p0.elapsed_time(ev_a0))
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_per_step, value = job_value(world, sum(step_ms), args.steps, fp + fa)
    assert kvq.device_status() == kvq.KVQ_OK

    # ------------------------------------------------------------ end to end: host buffers in and out
    # Each step copies x in from pinned host memory and the attention output back.
    # The copies run on their own stream and overlap the kernels: x goes in by token
    # chunks, each chunk projected (through a row window of the store) as soon as it
    # has landed; the attention runs by query chunks, each chunk's output copied back
    # while the next is computed.  The projection gives the one-call bits (rows are
    # independent) and so do the query chunks attended in one call; the first query
    # chunk, attended key range by key range while x arrives (below), differs from
    # them by the rounding of the log-sum-exp merges, within the attention's bar.
    x_host = x.cpu().pin_memory()
    out_host = torch.empty((n, C), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x)
    copy = torch.cuda.Stream(device=dev)
    in_chunks = [(s0, min(E2E_IN_CHUNK, n - s0)) for s0 in range(0, n, E2E_IN_CHUNK)]
    out_chunks = query_chunks(n)

    def windows(s0, length):  # the stores' rows of tokens s0 .. s0+length-1, in order
        out, start = [], 0
        for st_ in stores:
            a, b = max(s0, start), min(s0 + length, start + st_.n)
            if a < b:
                out.append(st_.rows(a - start, b - a))
            start += st_.n
        return out

    # While x is still arriving, the first query chunks (their own rows already
    # projected) attend each newly projected key range through the key-chunk call,
    # carrying a log-sum-exp state; their last call, once every x chunk is in, writes
    # their output.  On a slow host link this fills the time the projection would wait
    # for x.  The other query chunks then attend all keys in one call each.  Not for
    # the causal and the routed blocks (key-chunk calls are unmasked, one store set).
    early = out_chunks[:E2E_EARLY_QUERY_CHUNKS] if not causal and not route else []
    early_rows = early[-1][0] + early[-1][1] if early else 0
    early_states = [kvq.partial_state(ln, C, dev) for _, ln in early]

    def e2e_step():
        landed = []
        for s0, ln in in_chunks:
            link.copy(x_dev[s0:s0 + ln], x_host[s0:s0 + ln], copy, "h2d")
            ev = torch.cuda.Event()
            ev.record(copy)
            landed.append(ev)
        done = 0  # keys the early query chunks have attended
        for i, ((s0, ln), ev) in enumerate(zip(in_chunks, landed)):
            stream.wait_event(ev)
            if rope is not None:
                kvq.streamed_qkv_proj_ex(x_dev[s0:s0 + ln], w, windows(s0, ln), rope[s0:s0 + ln], group=32,
                                           chunk_tokens=wl.chunk_tokens, q_norm_w=qn, k_norm_w=kn, q_out=q[s0:s0 + ln],
                                           stream=stream)
            else:
                kvq.streamed_qkv_proj_mixed(x_dev[s0:s0 + ln], w, windows(s0, ln), group=32,
                                            chunk_tokens=wl.chunk_tokens, q_norm_w=qn, k_norm_w=kn,
                                            q_out=q[s0:s0 + ln], stream=stream)
            project_fine(x_dev[s0:s0 + ln], s0, ln)
            avail = s0 + ln  # keys projected so far
            if early and avail >= early_rows and i + 1 < len(in_chunks):
                for (e0, el), (oa, la) in zip(early, early_states):
                    kvq.packed_kv_attention_partial(q[e0:e0 + el], windows(done, avail - done), state=(oa, la),
                                                    merge=done > 0, stream=stream)
                done = avail
        for (e0, el), (oa, la) in zip(early, early_states):
            qc = q[e0:e0 + el]
            kvq.packed_kv_attention_partial(qc, windows(done, n - done), state=(oa, la), merge=done > 0, final=True,
                                            out=qc, stream=stream)
            ev = torch.cuda.Event()
            ev.record(stream)
            copy.wait_event(ev)
            link.copy(out_host[e0:e0 + el], qc, copy, "d2h")
        for s0, ln in out_chunks[len(early):]:
            qc = q[s0:s0 + ln]
            attend_rows(qc, s0)
            ev = torch.cuda.Event()
            ev.record(stream)
            copy.wait_event(ev)
            link.copy(out_host[s0:s0 + ln], qc, copy, "d2h")
        torch.cuda.synchronize()

    e2e_steps = max(1, min(args.steps, E2E_STEPS))
    link = LinkMeter()
    e2e_s, e2e_clocks = timed_leg(e2e_step, e2e_steps, world, local, link)
    e2e_link = link.record()
    e2e_val = world * (fp + fa) / e2e_s / 1e12

    # ------------------------------------------------------------ end to end, two phases (no full Q or output on device)
    # Phase 1 projects K/V only, by token chunks of x landing from the host; phase 2
    # brings x in again by query chunks, recomputes their Q only and attends, each
    # output chunk going back to the host.  Device memory: W, the packed store and
    # two chunk buffers of each kind.  Same FLOPs as the one-call path (the
    # projection's sections split its columns).
    del x_dev
    torch.cuda.synchronize()
    mem0 = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    xb = [torch.empty((E2E_IN_CHUNK, C), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    xq = [torch.empty((E2E_OUT_CHUNK, C), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    qb = [torch.empty((E2E_OUT_CHUNK, C), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in1", "p1", "in2", "qp", "attn", "out")}

    def e2e_two_phase_step():
        for i, (s0, ln) in enumerate(in_chunks):
            b = i % 2
            copy.wait_event(ev["p1"][b])  # chunk i-2's projection has read xb[b]
            link.copy(xb[b][:ln], x_host[s0:s0 + ln], copy, "h2d")
            ev["in1"][b].record(copy)
            stream.wait_event(ev["in1"][b])
            kvq.streamed_qkv_proj_ex(xb[b][:ln], w, windows(s0, ln), rope[s0:s0 + ln] if rope is not None else None,
                                     sections=kvq.SECTION_KV, group=32, chunk_tokens=wl.chunk_tokens, q_norm_w=qn,
                                     k_norm_w=kn, stream=stream)
            project_fine(xb[b][:ln], s0, ln)
            ev["p1"][b].record(stream)
        for i, (s0, ln) in enumerate(out_chunks):
            b = i % 2
            if i == 0:
                link.copy(xq[0][:ln], x_host[s0:s0 + ln], copy, "h2d")
                ev["in2"][0].record(copy)
            stream.wait_event(ev["in2"][b])
            stream.wait_event(ev["out"][b])  # chunk i-2's output has left qb[b]
            qc = kvq.streamed_qkv_proj_ex(xq[b][:ln], w, None, rope[s0:s0 + ln] if rope is not None else None,
                                          sections=kvq.SECTION_Q, group=32, chunk_tokens=wl.chunk_tokens, q_norm_w=qn,
                                          k_norm_w=kn, q_out=qb[b][:ln], stream=stream)
            ev["qp"][b].record(stream)
            attend_rows(qc, s0)
            ev["attn"][b].record(stream)
            if i + 1 < len(out_chunks):  # next chunk's x, once the projection of chunk i-1 has read xq[1-b]
                s1, l1 = out_chunks[i + 1]
                copy.wait_event(ev["qp"][1 - b])
                link.copy(xq[1 - b][:l1], x_host[s1:s1 + l1], copy, "h2d")
                ev["in2"][1 - b].record(copy)
            copy.wait_event(ev["attn"][b])
            link.copy(out_host[s0:s0 + ln], qc, copy, "d2h")
            ev["out"][b].record(copy)
        torch.cuda.synchronize()

    link = LinkMeter()
    e2e2_s, e2e2_clocks = timed_leg(e2e_two_phase_step, e2e_steps, world, local, link)
    e2e2_link = link.record()
    peak2_gib = (torch.cuda.max_memory_allocated(dev) - mem0) / GiB
    # device memory the step holds beyond what stays resident across steps (W, norms, table)
    resident_gib = (sum(st_.nbytes() for st_ in stores) + (fine.nbytes() if route else 0)) / GiB
    assert kvq.device_status() == kvq.KVQ_OK

    # ------------------------------------------------------------ end to end, packed store staged in host memory
    # vram_lab.py's streamed block plans K/V kept in host memory and streamed to the
    # device block by block.  Phase 1 projects K/V only, by token chunks of x from
    # the host, into a device chunk store whose rows go to pinned host memory, one
    # contiguous buffer per key chunk.  Phase 2 brings x in again by query chunks,
    # recomputes their Q and attends the host-staged store key chunk by key chunk
    # (copied in on the copy stream, two device buffers), merging each chunk into a
    # carried log-sum-exp state; the last chunk writes the output over Q, which goes
    # back to the host.  The device holds W, chunk buffers and the state only: the
    # footprint does not grow with N.
    hs = None
    if not args.no_host_staged and not mixed and not causal and rope is None:
        hs = host_staged_leg(kvq, wl, w, qn, kn, x_host, out_host, stream, copy, dev, world, e2e_steps,
                             out_chunks)
        hs["value"] = world * (fp + fa) / hs.pop("seconds") / 1e12
        assert kvq.device_status() == kvq.KVQ_OK

    pack = None
    if not args.no_pack_record and rank == 0:
        pack = pack_record(kvq, dev, warmup=3, steps=10)

    # ------------------------------------------------------------ roofline of the dominant kernel (attention)
    peaks, peak_kind = load_peaks()
    attn_avg_ms = sum(attn_ms) / len(attn_ms)
    proj_avg_ms = sum(proj_ms) / len(proj_ms)
    attn_tflops = fa / (attn_avg_ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    traffic = None  # DRAM bytes per launch from an ncu capture of the same attention code, else null
    tp = os.path.join(ROOT, "profiles", "attention_traffic.json")
    if os.path.exists(tp):
        with open(tp) as f:
            rec = json.load(f)
        if rec.get("code_sha256") == attention_code_sha256() and rec.get("workload") == wl_label:
            traffic = rec.get("bytes_per_launch")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not mixed and not causal and rope is None:
        del x_host, out_host
        cpu = cpu_baseline(wl, fp, fa, args.cpu_proj_rows, args.cpu_attn_rows, args.cpu_single_proj_rows,
                           args.cpu_single_attn_rows)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 GEMM / fp16 attention operands, fp32 accumulate",
            "data": "synthetic (seeded generators; random-init weights of the H3 block shape)",
            "config": {"workload": wl_label, "n_tokens": n, "hidden": C,
                       "heads": wl.heads, "group": 32, "causal": causal, "rope": rope is not None,
                       "route_av": route,
                       "kv_bits": "8/4 by token range" if mixed else 4, "chunk_tokens": wl.chunk_tokens,
                       "qk_rmsnorm": True,
                       "l2": f"inputs larger than L2 (x {n * C * 2 / GiB:.2f} GiB, packed K/V "
                             f"{sum(st.nbytes() for st in stores) / GiB:.2f} GiB)",
                       "parallelism": f"independent blocks x{world}"},
            "tokens_per_s": world * n / (ms_per_step * 1e-3),
            "kernel_ms": {"qkv_proj": proj_avg_ms, "attention": attn_avg_ms},
            "kernel_tflops": {"qkv_proj": fp / (proj_avg_ms * 1e-3) / 1e12, "attention": attn_tflops},
            "peak_gib": peak_ours, "peak_gib_materialise_bf16_qkv": peak_mat,
            "peak_ratio": peak_ours / peak_mat if peak_mat else None,
            "kv_store": [{"tokens": st.n, "bits": st.bits} for st in stores],
            "roofline": {"kernel": "packed_kv_attention", "bound": "tensor", "achieved": attn_tflops,
                         "peak": peak, "unit": "TFLOP/s", "frac": attn_tflops / peak, "traffic": traffic,
                         "peak_source": f"{peak_kind} bf16 sustained (fp16 dense rate = bf16 dense rate)"},
            "clocks": clocks,
            "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": int(x.numel() * 2),
                    "d2h_bytes_per_step": int(n * C * 2), "ms_per_step": e2e_s * 1e3, "clocks": e2e_clocks,
                    "host_link": e2e_link,
                    "note": "x copied in from pinned host memory and the attention output copied back each step, "
                            "on a copy stream overlapping the kernels (token chunks in, query chunks out); the "
                            f"first {len(early)} query chunks attend each key range as it is projected (key-chunk "
                            "calls with a log-sum-exp state), the rest attend all keys at once; W stays resident"},
            "e2e_two_phase": {"value": world * (fp + fa) / e2e2_s / 1e12, "unit": "TFLOP/s",
                              "ms_per_step": e2e2_s * 1e3, "clocks": e2e2_clocks, "host_link": e2e2_link,
                              "device_gib": resident_gib + peak2_gib,
                              "device_gib_materialise_bf16_qkv": peak_mat,
                              "h2d_bytes_per_step": int(2 * x.numel() * 2), "d2h_bytes_per_step": int(n * C * 2),
                              "note": "phase 1: K/V only by token chunks of x from the host; phase 2: x again by "
                                      "query chunks, Q only recomputed, attention, output chunk back to the host; "
                                      "device_gib = packed store + chunk buffers (x, Q and output never held in "
                                      "full), W excluded as in the peak comparison"},
            "e2e_host_staged": hs,
            "kernels": {"pack": pack} if pack else None,
            # per step: the projection (and, routed, the fine store's K/V section) and the attention calls
            "gpu_launches": ((2 + len(routed_segs)) if route else 2) * args.steps,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def host_staged_leg(kvq, wl, w, qn, kn, x_host, out_host, stream, copy, dev, world, steps, out_chunks):
    """The block end to end with the packed K/V store in pinned host memory (see
    the comment at its call).  Returns seconds per step, device memory and the
    bytes copied each way."""
    n, C = wl.n, wl.hidden
    heads = C // 128
    kv_chunks = [(s0, min(E2E_KV_CHUNK, n - s0)) for s0 in range(0, n, E2E_KV_CHUNK)]
    assert E2E_KV_CHUNK <= E2E_IN_CHUNK  # phase 1 lands x by key chunks in the x chunk buffers
    torch.cuda.synchronize()
    mem0 = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)

    def host_chunk():
        return kvq.PackedKV(
            torch.empty((heads, E2E_KV_CHUNK, 64), dtype=torch.uint8, pin_memory=True),
            torch.empty((heads, E2E_KV_CHUNK, 64), dtype=torch.uint8, pin_memory=True),
            torch.empty((heads, E2E_KV_CHUNK, 4), dtype=torch.float16, pin_memory=True),
            torch.empty((heads, E2E_KV_CHUNK, 4), dtype=torch.float16, pin_memory=True), E2E_KV_CHUNK, 4, 32)

    host_kv = [host_chunk() for _ in kv_chunks]
    kv_dev = [kvq.PackedKV.empty(E2E_KV_CHUNK, C, 32, 4, dev) for _ in range(2)]
    xb = [torch.empty((E2E_IN_CHUNK, C), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    xq = [torch.empty((E2E_OUT_CHUNK, C), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    qb = [torch.empty((E2E_OUT_CHUNK, C), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    o_acc, lse_acc = kvq.partial_state(E2E_OUT_CHUNK, C, dev)
    # device-to-host copies get a stream of their own: on the copy stream, a chunk's
    # store or output waiting for its kernel would hold up the next x chunk or key
    # chunk queued behind it
    copy_out = torch.cuda.Stream(device=dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in1", "p1", "kvout", "in2", "qp", "kvin", "attn",
                                                              "out")}
    parts = lambda st: (st.k_codes, st.v_codes, st.k_scales, st.v_scales)  # noqa: E731

    def one_step():
        for i, (s0, ln) in enumerate(kv_chunks):  # phase 1: K/V of every token, to the host
            b = i % 2
            copy.wait_event(ev["p1"][b])
            link.copy(xb[b][:ln], x_host[s0:s0 + ln], copy, "h2d")
            ev["in1"][b].record(copy)
            stream.wait_event(ev["in1"][b])
            stream.wait_event(ev["kvout"][b])  # the chunk store of chunk i-2 has gone to the host
            kvq.streamed_qkv_proj_ex(xb[b][:ln], w, [kv_dev[b].rows(0, ln)], sections=kvq.SECTION_KV, group=32,
                                     chunk_tokens=wl.chunk_tokens, q_norm_w=qn, k_norm_w=kn, stream=stream)
            ev["p1"][b].record(stream)
            copy_out.wait_event(ev["p1"][b])
            for d, s_ in zip(parts(host_kv[i]), parts(kv_dev[b])):
                link.copy(d, s_, copy_out, "d2h")
            ev["kvout"][b].record(copy_out)
        copy.wait_stream(copy_out)  # the key chunks go back to the device buffers only once they have all left
        kc = 0
        for i, (s0, ln) in enumerate(out_chunks):  # phase 2: Q per query chunk, the store streamed in
            b = i % 2
            if i == 0:
                link.copy(xq[0][:ln], x_host[s0:s0 + ln], copy, "h2d")
                ev["in2"][0].record(copy)
            stream.wait_event(ev["in2"][b])
            stream.wait_event(ev["out"][b])
            qc = kvq.streamed_qkv_proj_ex(xq[b][:ln], w, None, sections=kvq.SECTION_Q, group=32,
                                          chunk_tokens=wl.chunk_tokens, q_norm_w=qn, k_norm_w=kn,
                                          q_out=qb[b][:ln], stream=stream)
            ev["qp"][b].record(stream)
            if i + 1 < len(out_chunks):  # next chunk's x, once the projection of chunk i-1 has read it
                s1, l1 = out_chunks[i + 1]
                copy.wait_event(ev["qp"][1 - b])
                link.copy(xq[1 - b][:l1], x_host[s1:s1 + l1], copy, "h2d")
                ev["in2"][1 - b].record(copy)
            state = (o_acc[:ln], lse_acc[:ln])
            for j, (k0, kl) in enumerate(kv_chunks):
                kb = kc % 2
                kc += 1
                copy.wait_event(ev["attn"][kb])  # the attention that last read this buffer has run
                for d, s_ in zip(parts(kv_dev[kb]), parts(host_kv[j])):
                    link.copy(d, s_, copy, "h2d")
                ev["kvin"][kb].record(copy)
                stream.wait_event(ev["kvin"][kb])
                last = j == len(kv_chunks) - 1
                kvq.packed_kv_attention_partial(qc, [kv_dev[kb].rows(0, kl)], state=state, merge=j > 0, final=last,
                                                out=qc if last else None, stream=stream)
                ev["attn"][kb].record(stream)
            copy_out.wait_event(ev["attn"][(kc - 1) % 2])
            link.copy(out_host[s0:s0 + ln], qc, copy_out, "d2h")
            ev["out"][b].record(copy_out)
        torch.cuda.synchronize()

    link = LinkMeter()
    secs, clocks = timed_leg(one_step, steps, world, torch.cuda.current_device(), link)
    peak = (torch.cuda.max_memory_allocated(dev) - mem0) / GiB
    store_bytes = sum(t.numel() * t.element_size() for st in host_kv for t in parts(st))
    return {"unit": "TFLOP/s", "ms_per_step": secs * 1e3, "seconds": secs, "clocks": clocks,
            "host_link": link.record(),
            "device_gib": peak, "host_store_gib": store_bytes / GiB,
            "h2d_bytes_per_step": int(2 * n * C * 2 + len(out_chunks) * store_bytes),
            "d2h_bytes_per_step": int(store_bytes + n * C * 2),
            "key_chunk": E2E_KV_CHUNK, "query_chunk": E2E_OUT_CHUNK,
            "note": "packed K/V in pinned host memory, one buffer per key chunk of "
                    f"{E2E_KV_CHUNK}; phase 1 projects K/V by token chunks and sends them to the host; phase 2 "
                    "recomputes Q per query chunk and attends the store chunk by chunk (packed_kv_attention_partial, "
                    "log-sum-exp state), each chunk copied in while the previous one is attended; device_gib = "
                    "chunk buffers + state, W excluded"}


def pack_record(kvq, dev, warmup: int, steps: int) -> dict:
    """kv_rotate_quant_pack and kv_unpack on K/V [PACK_N, 2 x 7168] BF16, group
    32, INT4: median CUDA-event time over `steps` launches, L2 flushed (a 512 MiB
    write) before each, against the measured HBM copy bandwidth."""
    from serving_tcgen05_streamed_gb300 import inputs
    C, g = 7168, 32
    peaks, kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    kv = inputs.sweep_kv(PACK_N, C, seed=0, device=dev)
    store = kvq.PackedKV.empty(PACK_N, C, g, 4, dev)
    out = torch.empty_like(kv)
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    nbytes = PACK_N * (2 * C * 2 + 2 * (C // 2 + (C // g) * 2))  # BF16 K/V + INT4 codes + fp16 scales
    rec = {"n": PACK_N, "hidden": C, "group": g, "bits": 4, "bytes_per_launch": nbytes, "peak_gbs": hbm,
           "peak_source": f"{kind} hbm copy", "l2": "flushed before every launch"}
    for name, fn in (("kv_rotate_quant_pack", lambda: kvq.kv_rotate_quant_pack(kv, C, g, 4, out=store)),
                     ("kv_unpack", lambda: kvq.kv_unpack(store, C, out=out))):
        ts = []
        for i in range(warmup + steps):
            flush.fill_(i & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            if i >= warmup:
                ts.append(a.elapsed_time(b))
        ms = statistics.median(ts)
        gbs = nbytes / (ms * 1e-3) / 1e9
        rec[name] = {"ms": ms, "gbs": gbs, "frac": gbs / hbm}
    assert kvq.device_status() == kvq.KVQ_OK
    del kv, store, out, flush
    torch.cuda.empty_cache()
    return rec


def run_sweep(args):
    """Bandwidth of the standalone rotate + quantise + pack kernel and of its
    inverse over the sweep sizes (K/V BF16 [N, 2 x 7168], groups 32/64/128),
    against the measured HBM copy bandwidth.  L2 is flushed (a 512 MiB write)
    before every timed launch."""
    import serving_tcgen05_streamed_gb300 as kvq
    from serving_tcgen05_streamed_gb300 import inputs
    kvq.load()
    torch.cuda.set_device(0)
    C = 7168
    peaks, kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device="cuda")
    rows = []
    sizes = args.sweep_n or inputs.SWEEP_N
    groups = args.sweep_groups or inputs.SWEEP_GROUPS
    for n in sizes:
        kv = inputs.sweep_kv(n, C, seed=0, device="cuda")
        for g in groups:
            store = kvq.PackedKV.empty(n, C, g, 4, "cuda")
            out = torch.empty_like(kv)
            res = {}
            for name, fn in (("pack", lambda: kvq.kv_rotate_quant_pack(kv, C, g, 4, out=store)),
                             ("unpack", lambda: kvq.kv_unpack(store, C, out=out))):
                ts = []
                for i in range(args.warmup + args.steps):
                    flush.fill_(i & 0xFF)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    fn()
                    b.record()
                    b.synchronize()
                    if i >= args.warmup:
                        ts.append(a.elapsed_time(b))
                ms = statistics.median(ts)
                nbytes = n * (2 * C * 2 + 2 * (C // 2 + (C // g) * 2))  # BF16 K/V + INT4 codes + fp16 scales
                res[name] = {"ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9}
            rows.append({"n": n, "group": g, "bytes": nbytes, "pack_ms": res["pack"]["ms"],
                         "pack_gbs": res["pack"]["gbs"], "unpack_ms": res["unpack"]["ms"],
                         "unpack_gbs": res["unpack"]["gbs"]})
            del store, out
        del kv
    assert kvq.device_status() == kvq.KVQ_OK
    best = max(rows, key=lambda r: r["pack_gbs"])
    big = max(rows, key=lambda r: (r["n"], r["group"] == 32))
    print(json.dumps({
        "metric": "kv_rotate_quant_pack bandwidth (BF16 K/V -> rotated INT4 + fp16 scales)", "value": big["pack_gbs"],
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
        "dtype": "bf16 in, int4 + fp16 out", "data": "synthetic: N(0,1) with 1% Student-t (nu=3) channels",
        "config": {"workload": "K/V [N, 2x7168] sweep", "l2": "flushed before every launch"},
        "roofline": {"kernel": "kv_rotate_quant_pack", "bound": "hbm", "achieved": big["pack_gbs"], "peak": hbm,
                     "unit": "GB/s", "frac": big["pack_gbs"] / hbm, "peak_source": f"{kind} hbm copy",
                     "at": {"n": big["n"], "group": big["group"]}},
        "best": best, "sweep": rows}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--ref-proj-rows", type=int, default=128,
                    help="reference arm: projection rows of the oracle per step")
    ap.add_argument("--ref-attn-rows", type=int, default=32,
                    help="reference arm: attention query rows of the oracle per step")
    ap.add_argument("--cpu-proj-rows", type=int, default=1024,
                    help="cpu_baseline (all cores): projection rows")
    ap.add_argument("--cpu-attn-rows", type=int, default=256,
                    help="cpu_baseline (all cores): attention query rows")
    ap.add_argument("--cpu-single-proj-rows", type=int, default=32,
                    help="cpu_baseline (one core): projection rows")
    ap.add_argument("--cpu-single-attn-rows", type=int, default=4,
                    help="cpu_baseline (one core): attention query rows")
    ap.add_argument("--no-pack-record", action="store_true",
                    help="skip the standalone pack / unpack record")
    ap.add_argument("--no-host-staged", action="store_true",
                    help="skip the end-to-end leg with the packed store in host memory")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=("h3_ref2va", "mid", "mixed", "causal", "sweep"), default="h3_ref2va",
                    help="h3_ref2va: N=152,263 (the benchmark); mid: N=16,384 at the same width (profiling); "
                         "mixed: N=217,088 with INT8 conditioning ranges; causal: the N=152,263 block with causal "
                         "attention; sweep: pack/unpack bandwidth")
    ap.add_argument("--route-av", action="store_true",
                    help="mixed workload: text and audio query rows attend an INT8 store of every key")
    ap.add_argument("--rope", action="store_true",
                    help="split-half RoPE (rot_dim 128) of Q and K in the projection epilogue")
    ap.add_argument("--sweep-n", type=int, nargs="+", default=None,
                    help="sweep: token counts to run (default: 4,096 ... 262,144)")
    ap.add_argument("--sweep-groups", type=int, nargs="+", default=None, choices=(32, 64, 128),
                    help="sweep: group sizes to run (default: 32 64 128)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    from serving_tcgen05_streamed_gb300 import inputs
    if args.workload == "sweep":
        run_sweep(args)
        return
    wl = {"h3_ref2va": inputs.H3_REF2VA, "mid": inputs.MID, "mixed": inputs.MIXED,
          "causal": inputs.H3_REF2VA}[args.workload]
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, wl, int(os.environ.get("WORLD_SIZE", "1")), rank)
        return
    world, rank, local = dist_setup(args.gpus)
    run_gpu(args, wl, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
