#!/usr/bin/env python
"""Benchmark: tokens/s through the batched multi-LoRA projections, and roofline fraction.

One step = one pass of the whole hot path over one batch: the segment build (tokens grouped
by adapter) plus the forward of every projection slot of the workload (LoRA delta: paged
shrink and expand fused; tcgen05 base GEMM with the fused delta epilogue), the q, k and v
slots of a layer, which read the same input, in one lora_linear_forward_group call and o in
one lora_linear_forward call.  Adapters are resident
(loading is set-up, not timed).  Default workload: the largest one, the Llama-13B-shaped layer
stack (H=5120, 40 layers x q/k/v/o = 160 projections, 256 adapters of rank 8..64, a mixed batch
of 448 decode tokens and 4 prefill requests of 512 tokens, Zipf(1.0) request->adapter, pool of
2^22 pages with 30% KV pages).  Other workloads with --config 1..5.

Timing (our arm): the steps are captured into CUDA graphs with a 256 MB L2 flush between
steps and CUDA events around every step and every kernel (events inside the graph, so host
launch latency is excluded); steps are replayed in chunks; W untimed warm-up steps first.
`value` = tokens x steps / summed step time (max over ranks).  `e2e` = the same metric
through the public API with pinned host buffers: per step the H2D copy of the token ids and
activations, the library calls, and the D2H copy of every slot's output (for steps that copy
more than 32 MB, on two copy streams, each call waiting only for its own input, so that they
overlap the calls).

--impl reference times the CPU oracle (fp64, the definition of the layer) on a bounded
sample of the same workload; there is no other reference implementation of this path.
Multi-GPU: every rank runs its own replica of the batch (independent problems, no collective
on the data path); timing is the max over ranks.  `--gpus N` with N > 1 outside torchrun
re-launches this script under torch.distributed.run with N processes; inside torchrun N must
equal WORLD_SIZE.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20
GRAPH_CHUNK = 32


# ------------------------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, use_cuda):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if use_cuda else "gloo")
    return dist if world > 1 else None


def max_over_ranks(value: float, dist, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: str):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.idx), "-lms", "200"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9 or not (t0 <= ts <= t1):
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, f in enumerate(flags) if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def source_digest(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def committed_traffic(kernel_file, config_key):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source still matches."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        entry = json.load(open(path))[f"{os.path.basename(kernel_file)}:config{config_key}"]
    except (KeyError, ValueError):
        return None
    if entry.get("source_sha") != source_digest(kernel_file):
        return None
    return entry.get("dram_bytes_per_launch")


# ------------------------------------------------------------------------------- workload bytes / flops
def gemm_launch_groups(wl):
    """The slots each base-GEMM launch of a step covers (the library's rule, restated): a group
    call runs one grouped launch (split-K for batches of <= 256 tokens, persistent otherwise); a
    single slot has its own launch."""
    return [list(g) for g in wl.slot_groups()]


def algorithmic(wl):
    """Algorithmic bytes and flops of one step (every slot), and of one base-GEMM and one
    LoRA-delta launch (averages over the step's launches of each kind).

    Base GEMM launch: W of each of its slots once, x once, y of each slot once.  LoRA-delta
    launch over a group of slots that read the same x: the x rows of the tokens that carry LoRA,
    once, then for every slot of the group each used adapter's A and B pages once and the fp32
    delta rows it writes.  The delta is an intermediate of this implementation's two-kernel
    split; the step total does not count it.
    """
    H, T, S = wl.H, wl.T, wl.n_slots
    used = np.unique(wl.token_adapter[wl.token_adapter >= 0])
    lora_pages = int(2 * wl.ranks[used].astype(np.int64).sum()) * S            # A and B, once per slot
    sum_r = int(wl.ranks[wl.token_adapter[wl.token_adapter >= 0]].astype(np.int64).sum())
    step_bytes = S * H * H * 2 + wl.n_inputs * T * H * 2 + S * T * H * 2 + lora_pages * H * 2
    step_flops = S * (2 * T * H * H + 4 * H * sum_r)
    launches = gemm_launch_groups(wl)
    gemm_bytes = sum(len(g) * (H * H * 2 + T * H * 2) + T * H * 2 for g in launches) // len(launches)
    gemm_flops = S * 2 * T * H * H // len(launches)
    t_lora = int((wl.token_adapter >= 0).sum())
    n_groups = len(wl.slot_groups())
    delta_step = n_groups * t_lora * H * 2 + S * ((lora_pages // S) * H * 2 + t_lora * H * 4)
    delta_bytes = delta_step // n_groups
    return dict(step_bytes=step_bytes, step_flops=step_flops, gemm_bytes=gemm_bytes, gemm_flops=gemm_flops,
                delta_bytes=delta_bytes, gemm_bytes_step=gemm_bytes * len(launches), gemm_flops_step=S * 2 * T * H * H,
                delta_bytes_step=delta_step,
                lora_page_bytes=lora_pages * H * 2, distinct_adapters=int(used.size), sum_rank=sum_r)


def gemm_kernel_names(wl, n_sm):
    """The base-GEMM kernels of a step, one name per distinct kernel ("a + b")."""
    names = []
    for g in gemm_launch_groups(wl):
        split = wl.T <= 256 and (wl.H // 64) % 2 == 0
        if len(g) > 1 and split:
            ks = [f"gemm_lora_group_splitk<{4 if (wl.H // 64) % 4 == 0 else 2}>"]
        else:
            ks = gemm_kernel_name(wl.H, wl.T, n_sm, len(g))
        for k in ks:
            if k not in names:
                names.append(k)
    return " + ".join(names)


def gemm_kernel_name(H, T, n_sm, n_slots=1):
    """The base-GEMM kernel the library launches for n_slots slots of T tokens (its tile choice,
    restated): one slot of <= 256 tokens splits K over a cluster; larger batches walk their tiles
    with persistent CTAs (one slot: when there are more tiles than SMs), of 256 features
    (gemm_lora_persistent<2>) when 1.5 x their waves is below the waves of 128-feature tiles."""
    if T <= 256 and n_slots == 1:
        return ["gemm_lora_kernel"]
    m_tiles = (H + 127) // 128
    n_tiles = (T + 255) // 256
    want = (3 * n_sm // 4 + m_tiles - 1) // m_tiles
    if n_tiles < want:
        n_tiles = min(want, (T + 31) // 32)
    bn = min(256, ((T + n_tiles - 1) // n_tiles + 31) // 32 * 32)
    n_tiles = (T + bn - 1) // bn
    if n_slots == 1 and m_tiles * n_tiles <= n_sm:
        return ["gemm_lora_kernel"]
    mh = 1
    if bn == 256:
        w1 = -(-n_slots * m_tiles * n_tiles // n_sm)
        w2 = -(-n_slots * ((H + 255) // 256) * n_tiles // n_sm)
        mh = 2 if 3 * w2 < 2 * w1 else 1
    return [f"gemm_lora_persistent<{mh}>"]


# ------------------------------------------------------------------------------- our arm
def stack_layers(layers):
    """Spec overrides that cut the layer stack to its first `layers` layers (the same batch, adapters
    and ranks; a pool scaled to the layers' pages): every projection launch is the full stack's."""
    spec = workloads.SPECS[5]
    return {"layers": layers, "n_slots": 4 * layers,
            "pool_pages": -(-spec.pool_pages * layers // spec.layers)}


class Harness:
    def __init__(self, key, device, overrides=None):
        import torch
        import adapter_gemm_lora_gb300 as L
        from adapter_gemm_lora_gb300 import build as B
        B.build()
        self.L, self.torch = L, torch
        self.wl = wl = workloads.make(key, **(overrides or {}))
        self.key = key
        H, S, T = wl.H, wl.n_slots, wl.T
        self.dev = device
        to_dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).to(device).view(torch.bfloat16)  # noqa
        self.pool_t = torch.full((wl.spec.pool_pages, H), float("nan"), dtype=torch.bfloat16, device=device)
        self.pool = L.lora_pool_create(self.pool_t, wl.spec.pool_pages, H, S, wl.spec.n_adapters, wl.page_order)
        L.lora_pool_reserve(self.pool, wl.kv_pages)
        for a in range(wl.spec.n_adapters):
            r = int(wl.ranks[a])
            L.lora_adapter_load(self.pool, a, r, [wl.A(a, s) for s in range(S)], [wl.B(a, s) for s in range(S)], S)
        self.x = [to_dev(wl.x(i)) for i in range(wl.n_inputs)]
        self.W = [to_dev(wl.W(s)) for s in range(S)]
        self.y = [torch.empty((T, H), dtype=torch.bfloat16, device=device) for _ in range(S)]
        self.ta = torch.from_numpy(wl.token_adapter).to(device)
        # Per layer, q, k and v read the same input: one group call covers the three slots.
        self.groups = wl.slot_groups()
        max_group = max(len(g) for g in self.groups)
        nbytes = L.lora_segments_size_group(self.pool, T, max_group)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.seg = L.lora_segments_init_group(self.pool, self.ws, nbytes, T, max_group)
        self.flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        # A step whose inputs are larger than the L2 evicts them itself: no flush is needed, and a
        # write-flush would leave dirty lines whose write-back lands inside the next timed step.
        self.step_bytes = algorithmic(wl)["step_bytes"]
        self.flush = self.step_bytes <= L2_BYTES
        torch.cuda.synchronize()

    def forward_all(self, xs, stream):
        """Every slot of the workload: one group call per run of slots sharing an input."""
        L, wl = self.L, self.wl
        for g in self.groups:
            x = xs[wl.slot_input(g[0])]
            if len(g) == 1:
                L.lora_linear_forward(self.pool, self.seg, g[0], x, self.W[g[0]], self.y[g[0]], None, stream=stream)
            else:
                L.lora_linear_forward_group(self.pool, self.seg, g, x, [self.W[s] for s in g], [self.y[s] for s in g],
                                            None, stream=stream)

    def step(self, stream):
        self.L.lora_segments_build(self.pool, self.ta, self.wl.T, self.seg, stream=stream)
        self.forward_all(self.x, stream)

    def capture(self, n_steps, stream):
        """A graph of n_steps steps, each bracketed by events (and preceded by an L2 flush when the
        step's inputs fit in twice the L2)."""
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
               for _ in range(n_steps)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            for i in range(n_steps):
                if self.flush:
                    self.flush_buf.zero_()
                evs[i][0].record()
                self.step(torch.cuda.current_stream().cuda_stream)
                evs[i][1].record()
        return g, evs

    def run_timed(self, steps, warmup, dist):
        torch, L = self.torch, self.L
        stream = torch.cuda.Stream(device=self.dev)
        with torch.cuda.stream(stream):
            for _ in range(max(warmup, 1)):                 # eager warm-up (also sets kernel attributes)
                self.flush_buf.zero_()
                self.step(stream.cuda_stream)
        torch.cuda.synchronize()
        chunk = min(GRAPH_CHUNK, steps)
        L.lora_profile_read(self.pool, reset=True)
        g_full, ev_full = self.capture(chunk, stream)
        counts = L.lora_profile_read(self.pool, reset=True)    # launches made during the capture
        launches_per_graph = {k: v["launches"] for k, v in counts.items()}
        rem = steps % chunk
        g_rem, ev_rem = self.capture(rem, stream) if rem else (None, [])
        torch.cuda.synchronize()
        for _ in range(max(1, warmup // chunk)):          # graph warm-up
            g_full.replay()
        torch.cuda.synchronize()
        self.soak(g_full, 1.0)
        n_full = steps // chunk
        step_ms = []
        barrier(dist)
        torch.cuda.synchronize()
        t0 = time.time()
        for _ in range(n_full):
            g_full.replay()
            torch.cuda.synchronize()
            step_ms += [a.elapsed_time(b) for a, b in ev_full]
        if g_rem is not None:
            g_rem.replay()
            torch.cuda.synchronize()
            step_ms += [a.elapsed_time(b) for a, b in ev_rem]
        torch.cuda.synchronize()
        barrier(dist)
        t1 = time.time()
        assert len(step_ms) == steps
        L.lora_status(self.pool, stream=stream.cuda_stream)
        kern_ms, sets = self.kernel_times(stream, chunk)
        per_step = {k: launches_per_graph[k] // chunk for k in L.KINDS}
        launches = {k: per_step[k] * steps for k in L.KINDS}
        return dict(step_ms=step_ms, kern_ms=kern_ms, kern_sets=sets, launches=launches,
                    launches_per_graph=launches_per_graph, launches_per_step=per_step, t0=t0, t1=t1)

    def kernel_times(self, stream, n_steps):
        """Per-kernel device times of n_steps more steps, right after the timed region.

        Events around every kernel (the library records them on the launching stream) would sit
        between the kernels of a graph and undo their programmatic-launch overlap, so these steps
        are launched directly, behind a short GPU sleep: every launch is queued before the GPU
        reaches it and the events bracket device execution only.  Kernel launches here carry no
        programmatic-launch attribute (the library drops it while profiling).
        """
        torch, L = self.torch, self.L
        L.lora_profile_read(self.pool, reset=True)
        L.lora_profile_enable(self.pool, True)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(2e8))                     # ~0.1 s head start for the host
            for _ in range(n_steps):
                if self.flush:
                    self.flush_buf.zero_()
                self.step(stream.cuda_stream)
        torch.cuda.synchronize()
        rec = L.lora_profile_read(self.pool, reset=True)
        L.lora_profile_enable(self.pool, False)
        return {k: v["ms"] for k, v in rec.items()}, 1

    def soak(self, graph, seconds):
        """Untimed replays right before the timed region so the clock sampler sees the loaded GPU."""
        end = time.time() + seconds
        while time.time() < end:
            graph.replay()
            self.torch.cuda.synchronize()

    def run_e2e(self, steps):
        """Public-API path with pinned host buffers, copies inside the timed region.  When a step
        copies more than 32 MB, the token ids and every input go host -> device on one copy
        stream, in order; each projection group waits only for its own input on the compute
        stream, and its outputs go device -> host on a second copy stream as soon as the group is
        done, so copies overlap compute.  Smaller steps run copies and calls on one stream (the
        events of the overlap cost more than they hide there)."""
        torch, L, wl = self.torch, self.L, self.wl
        H, T, S = wl.H, wl.T, wl.n_slots
        h2d = T * 4 + wl.n_inputs * T * H * 2
        d2h = S * T * H * 2
        overlap = h2d + d2h > (32 << 20)
        stream = torch.cuda.Stream(device=self.dev)
        s_in = torch.cuda.Stream(device=self.dev)
        s_out = torch.cuda.Stream(device=self.dev)
        h_ta = torch.from_numpy(wl.token_adapter.copy()).pin_memory()
        h_x = [torch.from_numpy(np.ascontiguousarray(wl.x(i)).view(np.int16)).view(torch.bfloat16).pin_memory()
               for i in range(wl.n_inputs)]
        h_y = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(S)]
        d_ta = torch.empty_like(self.ta)
        d_x = [torch.empty((T, H), dtype=torch.bfloat16, device=self.dev) for _ in range(wl.n_inputs)]
        times = []
        if not overlap:
            with torch.cuda.stream(stream):
                for it in range(steps + 2):
                    if self.flush:
                        self.flush_buf.zero_()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    d_ta.copy_(h_ta, non_blocking=True)
                    for i in range(wl.n_inputs):
                        d_x[i].copy_(h_x[i], non_blocking=True)
                    L.lora_segments_build(self.pool, d_ta, T, self.seg, stream=stream.cuda_stream)
                    self.forward_all(d_x, stream.cuda_stream)
                    for s_ in range(S):
                        h_y[s_].copy_(self.y[s_], non_blocking=True)
                    e1.record()
                    e1.synchronize()
                    if it >= 2:
                        times.append(e0.elapsed_time(e1))
            return times, h2d, d2h, "one stream"
        for it in range(steps + 2):
            with torch.cuda.stream(stream):
                if self.flush:
                    self.flush_buf.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
            s_in.wait_stream(stream)
            with torch.cuda.stream(s_in):
                d_ta.copy_(h_ta, non_blocking=True)
                ev_ta = torch.cuda.Event()
                ev_ta.record()
                ev_x = []
                for i in range(wl.n_inputs):
                    d_x[i].copy_(h_x[i], non_blocking=True)
                    ev_x.append(torch.cuda.Event())
                    ev_x[-1].record()
            stream.wait_event(ev_ta)
            L.lora_segments_build(self.pool, d_ta, T, self.seg, stream=stream.cuda_stream)
            for g in self.groups:
                i = wl.slot_input(g[0])
                stream.wait_event(ev_x[i])
                x = d_x[i]
                if len(g) == 1:
                    L.lora_linear_forward(self.pool, self.seg, g[0], x, self.W[g[0]], self.y[g[0]], None,
                                          stream=stream.cuda_stream)
                else:
                    L.lora_linear_forward_group(self.pool, self.seg, g, x, [self.W[s] for s in g],
                                                [self.y[s] for s in g], None, stream=stream.cuda_stream)
                ev_g = torch.cuda.Event()
                ev_g.record(stream)
                s_out.wait_event(ev_g)
                with torch.cuda.stream(s_out):
                    for s_ in g:
                        h_y[s_].copy_(self.y[s_], non_blocking=True)
            stream.wait_stream(s_out)
            e1.record(stream)
            e1.synchronize()
            if it >= 2:
                times.append(e0.elapsed_time(e1))
        return times, h2d, d2h, "two copy streams overlapping the calls"


def attention_leg(L, H, device, n_req=256, ctx=(128, 2048), head_dim=128, calls=30, seed=7):
    """Paged decode attention over KV pages of a unified pool (the pool's second consumer): one new
    token per request at one layer, contexts uniform in `ctx` (seeded), KV pages taken by
    lora_kv_grow in a seeded page order.  HBM roofline: every cached K and V page row is read
    once (2 x context x H x 2 bytes per request) plus q and out.  Inputs (GBs of KV) are far
    larger than L2, so no flush is needed between calls."""
    import torch
    rng = np.random.default_rng(seed)
    lens = rng.integers(ctx[0], ctx[1] + 1, size=n_req)
    num_pages = int(2 * lens.sum()) + 64
    pool_t = torch.empty((num_pages, H), dtype=torch.bfloat16, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    pool_t.normal_(generator=g)
    pool = L.lora_pool_create(pool_t, num_pages, H, 1, 1, rng.permutation(num_pages))
    try:
        for r, n in enumerate(lens):
            L.lora_kv_grow(pool, r, int(n), 1)
        max_len = int(lens.max())
        table = torch.empty((n_req, max_len, 1, 2), dtype=torch.int32, device=device)
        seq = torch.empty(n_req, dtype=torch.int32, device=device)
        L.lora_kv_batch_table(pool, np.arange(n_req), max_len, table, seq)
        q = torch.randn((n_req, H), generator=g, device=device).to(torch.bfloat16)
        out = torch.empty_like(q)
        n_heads = H // head_dim
        stream = torch.cuda.current_stream(device).cuda_stream
        for _ in range(3):
            L.lora_attention_decode(pool, n_req, table, seq, max_len, 1, 0, q, out, n_heads, stream=stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(calls):
            L.lora_attention_decode(pool, n_req, table, seq, max_len, 1, 0, q, out, n_heads, stream=stream)
        e1.record()
        torch.cuda.synchronize()
        L.lora_status(pool)
        us = e0.elapsed_time(e1) * 1e3 / calls
        nbytes = int(2 * lens.sum()) * H * 2 + 2 * n_req * H * 2
        peaks = load_peaks()
        gbs = nbytes / (us * 1e-6) / 1e9
        kernel = "attention_heads_kernel"
        return {"kernel": kernel, "requests": n_req, "H": H, "head_dim": head_dim,
                "context": f"uniform [{ctx[0]}, {ctx[1]}], mean {lens.mean():.0f}", "us_per_call": round(us, 2),
                "algorithmic_bytes": nbytes, "achieved_gbs": round(gbs, 1), "peak_gbs": peaks["hbm_gbs"],
                "frac": round(gbs / peaks["hbm_gbs"], 4), "bound": "hbm"}
    finally:
        L.lora_pool_destroy(pool)
        del pool_t
        torch.cuda.empty_cache()


def prefetch_leg(device, n_steps=256, loads=(0, 16, 64, 256)):
    """Adapter loads overlapped with compute ("S-LoRA, in depth", "Scheduling": pinned host memory and
    a copy stream let the next batch's adapters load while the current batch computes; "Fewer
    Expert Transfers Without Changing Routing", Eq. (1): a step costs c + rho tau with blocking
    copies, and at best max(c, rho tau) when they overlap compute).

    On the decode workload (one layer's q/k/v/o, 256 tokens): c = the step alone (graph replay);
    tau = one packed load of the largest adapter the batch does not use (pinned host memory,
    lora_adapter_load_packed on a copy stream) alone; then n_steps steps replayed on the compute
    stream while the copy stream loads and unloads that adapter `m` times (rho = m / n_steps).
    The load kernel reads host memory with SM threads, so it also takes SMs from the steps."""
    import torch
    h = Harness(2, device)
    L, wl = h.L, h.wl
    S = wl.n_slots
    used = set(int(a) for a in wl.token_adapter if a >= 0)
    spare = max((a for a in range(wl.spec.n_adapters) if a not in used), key=lambda a: int(wl.ranks[a]))
    r = int(wl.ranks[spare])
    A = [wl.A(spare, s) for s in range(S)]
    B = [wl.B(spare, s) for s in range(S)]
    nbytes = L.lora_adapter_packed_size(h.pool, r)
    buf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    L.lora_adapter_pack(h.pool, r, A, B, buf, nbytes)
    compute = torch.cuda.Stream(device=device)
    copy = torch.cuda.Stream(device=device)
    L.lora_adapter_unload(h.pool, spare, stream=compute.cuda_stream)
    with torch.cuda.stream(compute):
        for _ in range(5):
            h.step(compute.cuda_stream)
    chunk = 32
    g, g_events = h.capture(chunk, compute)       # the graph records these events: keep them alive
    torch.cuda.synchronize()

    def cycle(n):
        for _ in range(n):
            L.lora_adapter_load_packed(h.pool, spare, r, buf, nbytes, S, copy_stream=copy.cuda_stream)
            L.lora_adapter_unload(h.pool, spare, stream=copy.cuda_stream)

    cycle(3)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(copy)
    cycle(32)
    e1.record(copy)
    torch.cuda.synchronize()
    tau = e0.elapsed_time(e1) / 32
    rows = []
    for m in loads:
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0 = torch.cuda.Event(enable_timing=True)
        c0.record(compute)
        k0.record(copy)
        with torch.cuda.stream(compute):
            for _ in range(n_steps // chunk):
                g.replay()
        c1.record(compute)
        cycle(m)
        torch.cuda.synchronize()
        c_ms = c0.elapsed_time(c1) / n_steps
        rows.append({"loads": m, "rho": round(m / n_steps, 4), "step_ms": round(c_ms, 5)})
    c = rows[0]["step_ms"]
    for row in rows:
        rt = row["rho"] * tau
        row["blocking_model_ms"] = round(c + rt, 5)
        row["overlap_model_ms"] = round(max(c, rt), 5)
    L.lora_status(h.pool)
    del g, g_events
    L.lora_pool_destroy(h.pool)
    return {"workload": wl.spec.name, "adapter_rank": r, "adapter_bytes": int(2 * r * S * wl.H * 2),
            "tau_ms": round(tau, 5), "c_ms": c, "rows": rows,
            "note": "steps replayed on the compute stream while the copy stream loads and unloads one packed "
                    "adapter m times; tau includes the unload"}


def default_steps(key):
    return {1: 2000, 2: 8000, 3: 400, 4: 2000, 5: 40}[key]


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world, True)
    device = torch.device("cuda", local)
    key = args.config
    steps = args.steps if args.steps is not None else default_steps(key)
    overrides = stack_layers(args.layers) if key == 5 and args.layers else None
    h = Harness(key, device, overrides)
    wl = h.wl
    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = visible.split(",")[local] if visible else str(local)
    clocks = ClockSampler(smi_index).start()
    res = h.run_timed(steps, args.warmup, dist)
    clocks.stop()
    e2e_times, h2d, d2h, e2e_copies = h.run_e2e(min(steps, 200 if key != 5 else 10))
    attention = attention_leg(h.L, wl.H, device) if not args.no_attention else None
    prefetch = prefetch_leg(device) if args.prefetch else None
    total_ms = sum(res["step_ms"])
    total_ms_max = max_over_ranks(total_ms, dist, device)
    T = wl.T
    value = world * T * steps / (total_ms_max / 1e3)
    e2e_ms = max_over_ranks(statistics.mean(e2e_times), dist, device)
    peaks = load_peaks()
    alg = algorithmic(wl)
    ms_per_step = total_ms_max / steps
    per_launch_ms = {k: res["kern_ms"][k] / max(1, res["launches_per_graph"][k]) for k in ("gemm", "delta")}
    shares = {k: v / max(1e-12, sum(res["kern_ms"].values())) for k, v in res["kern_ms"].items()}
    # The roofline object describes the kernel kind with the largest share of device time: the
    # base GEMM (its roof follows the workload's arithmetic intensity) or the LoRA delta (HBM).
    # A kind runs as several kernels in one step (a grouped launch for q/k/v, one for o):
    # its figures are per-launch averages, algorithmic bytes and time alike (the step's totals
    # divided by the kernel launches the library counted; x is counted once per call).
    dominant = "delta" if res["kern_ms"]["delta"] > res["kern_ms"]["gemm"] else "gemm"
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    launch_ms = per_launch_ms[dominant]
    if dominant == "gemm":
        kernel_file = os.path.join(ROOT, "adapter_gemm_lora_gb300", "csrc", "gemm_tcgen05.cu")
        kernel_name = gemm_kernel_names(wl, torch.cuda.get_device_properties(device).multi_processor_count)
        hbm_bound = alg["gemm_flops"] / alg["gemm_bytes"] < ridge
        n_launch = max(1, res["launches_per_step"]["gemm"])
        alg_bytes, alg_flops = alg["gemm_bytes_step"] // n_launch, alg["gemm_flops_step"] // n_launch
    else:
        kernel_file = os.path.join(ROOT, "adapter_gemm_lora_gb300", "csrc", "lora_gather.cu")
        kernel_name = "lora_delta_kernel"
        hbm_bound = True
        alg_bytes, alg_flops = alg["delta_bytes"], None
    traffic = committed_traffic(kernel_file, key)
    if hbm_bound:
        achieved = alg_bytes / (launch_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic}
    else:
        achieved = alg_flops / (launch_ms / 1e3) / 1e12
        pk = peaks["bf16_tflops"]            # burst: each launch is timed alone, well under a second
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk, "unit": "TFLOP/s",
                "frac": round(achieved / pk, 4), "traffic": traffic,
                "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4)}
    roof.update({"kernel": kernel_name, "peak_source": peaks["source"], "avg_launch_us": round(launch_ms * 1e3, 2),
                 "algorithmic_per_launch": alg_bytes if roof["bound"] == "hbm" else alg_flops,
                 "per_launch_us": {k: round(v * 1e3, 2) for k, v in per_launch_ms.items()}})
    step_s = ms_per_step / 1e3
    t_hbm = alg["step_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = alg["step_flops"] / (peaks["bf16_tflops"] * 1e12)
    step_roof = {"bound": "hbm" if t_hbm >= t_tc else "tensor", "roofline_us": round(max(t_hbm, t_tc) * 1e6, 2),
                 "measured_us": round(step_s * 1e6, 2), "frac": round(max(t_hbm, t_tc) / step_s, 4),
                 "algorithmic_bytes": alg["step_bytes"], "algorithmic_flops": alg["step_flops"],
                 "achieved_gbs": round(alg["step_bytes"] / step_s / 1e9, 1),
                 "achieved_tflops": round(alg["step_flops"] / step_s / 1e12, 1)}
    line = {
        "metric": "tokens/s through batched multi-LoRA projections",
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights and adapters)",
        "config": {"workload": wl.spec.name, "description": wl.spec.description, "H": wl.H, "T": T,
                   "slots": wl.n_slots, "layers": wl.spec.layers, "adapters_resident": wl.spec.n_adapters,
                   "distinct_adapters_in_batch": alg["distinct_adapters"], "pool_pages": wl.spec.pool_pages,
                   "parallelism": f"replicas x{world}",
                   "l2": ("flushed (256 MB write) before every step" if h.flush else
                          f"inputs larger than L2: a step reads {alg['step_bytes'] / 1e6:.0f} MB (L2: 129 MB)"),
                   "timing": "CUDA graph replay, events per step inside the graph; per-kernel times from "
                             f"{GRAPH_CHUNK} more steps launched behind a GPU sleep with events around every kernel"},
        "roofline": roof,
        "step_roofline": step_roof,
        "kernel_share": {k: round(v, 4) for k, v in shares.items() if res["kern_ms"][k] > 0},
        "gpu_launches": int(sum(res["launches"].values())),
        "gpu_launches_per_step": res["launches_per_step"],
        "e2e": {"value": round(world * T / (e2e_ms / 1e3), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "path": f"eager public API calls, pinned host buffers, copies on {e2e_copies}"},
        "clocks": clocks.summary(res["t0"] - 1.5, res["t1"]),
    }
    if attention is not None:
        line["attention_decode"] = attention
    if prefetch is not None:
        line["adapter_prefetch"] = prefetch
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, seconds=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------------------------- oracle (CPU)
def oracle_scene(wl, slots, tokens):
    """The oracle's pool for the given slots (its own bookkeeping and placement)."""
    import oracle as O

    class Sparse(dict):
        def __setitem__(self, k, v):
            super().__setitem__(int(k), np.asarray(v, np.uint16).copy())

        def __getitem__(self, idx):
            idx = np.asarray(idx)
            return np.stack([dict.__getitem__(self, int(i)) for i in idx.reshape(-1)]).reshape(idx.shape + (wl.H,))

    model = O.PoolModel(wl.spec.pool_pages, wl.n_slots, wl.spec.n_adapters, wl.page_order)
    model.reserve(wl.kv_pages)
    pool = Sparse()
    used = set(int(a) for a in wl.token_adapter[tokens] if a >= 0)
    for a in range(wl.spec.n_adapters):
        _, tab = model.load(a, int(wl.ranks[a]), [True] * wl.n_slots)
        if a in used:
            O.place_adapter(pool, tab, [wl.A(a, s) if s in slots else None for s in range(wl.n_slots)],
                            [wl.B(a, s) if s in slots else None for s in range(wl.n_slots)])
    return model, pool


def oracle_cores():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def oracle_sample(wl, seconds):
    """Tokens and slots of a bounded oracle sample: every slot for small stacks, else 4 slots."""
    rng = np.random.default_rng(1234)
    slots = list(range(wl.n_slots)) if wl.n_slots <= 4 else [0, 1, 2, 3]
    n_tok = min(wl.T, 64)
    tokens = np.sort(rng.choice(wl.T, size=n_tok, replace=False))
    return slots, tokens


def cpu_baseline(wl, seconds=15.0):
    slots, tokens = oracle_sample(wl, seconds)
    model, pool = oracle_scene(wl, set(slots), tokens)
    xs = {i: wl.x(i) for i in {wl.slot_input(s) for s in slots}}
    Ws = {s: wl.W(s) for s in slots}
    import oracle as O
    t0 = time.time()
    reps = 0
    while True:
        for s in slots:
            O.linear_forward(pool, model.tables, wl.token_adapter, s, xs[wl.slot_input(s)], Ws[s], tokens=tokens)
        reps += 1
        if time.time() - t0 >= seconds or reps >= 1000:
            break
    el = time.time() - t0
    # tokens through the whole stack per second: each sampled token passed len(slots) of n_slots slots
    value = reps * len(tokens) * (len(slots) / wl.n_slots) / el
    return {"value": round(value, 3), "unit": "tokens/s", "cores": oracle_cores(), "kind": "oracle",
            "sample": f"{len(tokens)} of {wl.T} tokens through {len(slots)} of {wl.n_slots} slots, "
                      f"repeated {reps}x over {el:.1f} s (fp64 NumPy, per-token page-table gathers)"}


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    key = args.config
    wl = workloads.make(key)
    steps = args.steps if args.steps is not None else 10
    per_step = max(0.5, min(6.0, 150.0 / max(1, steps + args.warmup)))
    slots, tokens = oracle_sample(wl, per_step)
    model, pool = oracle_scene(wl, set(slots), tokens)
    xs = {i: wl.x(i) for i in {wl.slot_input(s) for s in slots}}
    Ws = {s: wl.W(s) for s in slots}
    import oracle as O

    def one():
        for s in slots:
            O.linear_forward(pool, model.tables, wl.token_adapter, s, xs[wl.slot_input(s)], Ws[s], tokens=tokens)
    for _ in range(args.warmup):
        one()
    times = []
    for _ in range(steps):
        t0 = time.time()
        one()
        times.append(time.time() - t0)
    tot = sum(times)
    value = steps * len(tokens) * (len(slots) / wl.n_slots) / tot
    line = {"impl": "reference", "metric": "tokens/s through batched multi-LoRA projections", "value": round(value, 3),
            "unit": "tokens/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": round(tot / steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": wl.spec.name, "description": wl.spec.description, "H": wl.H, "T": wl.T,
                       "slots": wl.n_slots},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": oracle_cores(), "kind": "oracle",
                             "sample": f"{len(tokens)} of {wl.T} tokens through {len(slots)} of {wl.n_slots} "
                                       f"slots per step"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def relaunch_under_torchrun(n, argv):
    """Run this script as n ranks (one process per GPU) on this node and return their status."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def check_world(gpus, argv):
    """None when this process is one rank of a run of `gpus` ranks; otherwise the exit status of a
    relaunch (or an error when torchrun started a different number of ranks)."""
    if gpus < 1:
        raise SystemExit(f"--gpus must be >= 1, got {gpus}")
    world = os.environ.get("WORLD_SIZE")
    if world is None:
        return relaunch_under_torchrun(gpus, argv) if gpus > 1 else None
    if int(world) != gpus:
        raise SystemExit(f"--gpus {gpus} but torchrun started WORLD_SIZE={world} ranks")
    return None


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-attention", action="store_true", help="skip the paged decode attention leg")
    ap.add_argument("--layers", type=int, default=0,
                    help="layer stack only: keep its first N layers (profiling a stack-shaped step)")
    ap.add_argument("--prefetch", action="store_true",
                    help="also measure decode steps with adapter loads on a copy stream")
    ap.add_argument("--eager-steps", type=int, default=0,
                    help="for profilers: run this many untimed eager steps of the workload and exit")
    ap.add_argument("--attention-only", action="store_true",
                    help="for profilers: run the attention leg alone (no workload) and print its figures")
    ap.add_argument("--attention-requests", type=int, default=256)
    ap.add_argument("--attention-h", type=int, default=0, help="attention leg hidden size (default: the workload's)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    rc = check_world(args.gpus, argv)
    if rc is not None:
        raise SystemExit(rc)
    if args.attention_only or args.eager_steps > 0:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


def run_profile_case(args):
    """Small, untimed runs for a profiler to capture: the workload's steps launched eagerly (one
    segment build and every slot's projections per step), or the attention leg alone."""
    import torch
    device = torch.device("cuda", 0)
    if args.attention_only:
        import adapter_gemm_lora_gb300 as L
        from adapter_gemm_lora_gb300 import build as B
        B.build()
        H = args.attention_h or workloads.SPECS[args.config].H
        print(json.dumps(attention_leg(L, H, device, n_req=args.attention_requests, calls=2)), flush=True)
        return
    overrides = stack_layers(args.layers) if args.config == 5 and args.layers else None
    h = Harness(args.config, device, overrides)
    stream = torch.cuda.current_stream(device).cuda_stream
    for _ in range(args.eager_steps):
        h.step(stream)
    torch.cuda.synchronize()
    h.L.lora_status(h.pool)
    print(json.dumps({"profile_case": h.wl.spec.name, "steps": args.eager_steps, "T": h.wl.T, "H": h.wl.H,
                      "pool_gb": round(h.pool_t.numel() * 2 / 1e9, 2)}), flush=True)


if __name__ == "__main__":
    main()
