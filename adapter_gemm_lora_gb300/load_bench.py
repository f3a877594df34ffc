"""Adapter load time on this GPU: synchronous loads against packed loads on a copy stream.

"S-LoRA, in depth", "Scheduling": a 32 MiB adapter (rank 16, q/k/v/o over 32 layers of a 4096-wide
model) over a link of ~20 GB/s takes ~1.6 ms, a noticeable share of a decode step; "What to do
next" asks for adapter load time as a metric.  "Fewer Expert Transfers Without Changing Routing"
(Table 1) measures the same copy time per expert on five GPUs.  This tool times, for such
adapters in a pool on the current GPU:
  - lora_adapter_load: host repacking into page rows, a pageable host-to-device copy, the page
    scatter and the table upload, then a stream synchronisation (wall clock);
  - lora_adapter_pack (host only, done once per adapter) and lora_adapter_load_packed: one kernel
    on a copy stream reading the packed rows from pinned host memory into the pages (CUDA events
    on the copy stream, and the host time of the call).

    python -m adapter_gemm_lora_gb300.load_bench [--rank 16] [--slots 128] [--adapters 6]

prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import statistics
import time

import numpy as np


def main(argv=None):
    import torch

    import adapter_gemm_lora_gb300 as L
    from adapter_gemm_lora_gb300 import build
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--H", type=int, default=4096)
    ap.add_argument("--rank", type=int, default=16)
    ap.add_argument("--slots", type=int, default=128)
    ap.add_argument("--adapters", type=int, default=6)
    args = ap.parse_args(argv)
    build.build()
    H, r, S, n = args.H, args.rank, args.slots, args.adapters
    need = 2 * r * S
    num_pages = 2 * need * n + 16
    rng = np.random.default_rng(0)
    A = [rng.integers(0, 1 << 15, size=(H, r), dtype=np.uint16) for _ in range(S)]
    B = [rng.integers(0, 1 << 15, size=(r, H), dtype=np.uint16) for _ in range(S)]
    pool_t = torch.zeros((num_pages, H), dtype=torch.bfloat16, device="cuda")
    pool = L.lora_pool_create(pool_t, num_pages, H, S, 2 * n)
    copy = torch.cuda.Stream()
    out = {"tool": "load_bench", "H": H, "rank": r, "slots": S, "adapter_MiB": need * H * 2 / 2**20,
           "gpu": torch.cuda.get_device_name(0)}
    try:
        sync_ms, tables = [], {}
        for a in range(n):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            tables[a] = L.lora_adapter_load(pool, a, r, A, B, S)
            sync_ms.append((time.perf_counter() - t0) * 1e3)
        nbytes = L.lora_adapter_packed_size(pool, r)
        bufs = [torch.empty(nbytes, dtype=torch.uint8).pin_memory() for _ in range(n)]
        pack_ms, call_ms, dev_ms = [], [], []
        for i in range(n):
            t0 = time.perf_counter()
            L.lora_adapter_pack(pool, r, A, B, bufs[i], nbytes)
            pack_ms.append((time.perf_counter() - t0) * 1e3)
        for i in range(n):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(copy)
            t0 = time.perf_counter()
            tables[n + i] = L.lora_adapter_load_packed(pool, n + i, r, bufs[i], nbytes, S, copy_stream=copy)
            call_ms.append((time.perf_counter() - t0) * 1e3)
            e1.record(copy)
            e1.synchronize()
            dev_ms.append(e0.elapsed_time(e1))
        L.lora_status(pool)
        for i in range(n):                    # packed and synchronous loads hold the same rows
            a_pages = torch.from_numpy(tables[i].reshape(-1).astype(np.int64)).cuda()
            b_pages = torch.from_numpy(tables[n + i].reshape(-1).astype(np.int64)).cuda()
            assert torch.equal(pool_t[a_pages].view(torch.int16), pool_t[b_pages].view(torch.int16))
        med = statistics.median
        out.update({
            "sync_load_ms": round(med(sync_ms[1:] or sync_ms), 3),
            "pack_host_ms": round(med(pack_ms), 3),
            "packed_load_call_ms": round(med(call_ms), 3),
            "packed_load_device_ms": round(med(dev_ms[1:] or dev_ms), 3),
            "packed_load_GBps": round(need * H * 2 / (med(dev_ms[1:] or dev_ms) / 1e3) / 1e9, 1),
        })
    finally:
        L.lora_pool_destroy(pool)
    print(json.dumps(out), flush=True)
    return out


if __name__ == "__main__":
    main()
