"""Eviction-rule simulation on the library's own pool bookkeeping (CPU only, planning pools).

Capacity planning for the unified pool ("S-LoRA, in depth", "What to do next": measure how many
adapters must be resident and what adapter loads cost).  A seeded stream of requests, each for
one adapter (Zipf popularity over N adapters with mixed ranks), is served one request at a time
through a pool that holds a fixed number of pages: lora_adapter_ensure, then
lora_adapter_release.  For every eviction rule of lora_pool_set_eviction it counts the adapter
loads and the bytes they move, and for the farthest-future rule it sweeps the lookahead k, as
"Fewer Expert Transfers Without Changing Routing" does for expert caches (section "Limited
foresight": the share of the gap between LRU and the full-foresight rule that k requests of
foresight recover).  Per-step cost follows that page's Equation (1): c + rho * tau with blocking
copies, approaching max(c, rho * tau) when copies overlap compute.

    python -m adapter_gemm_lora_gb300.eviction_sim [--adapters 2000] [--alpha 0.5] ...

prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import time

import numpy as np

RANKS = (8, 16, 32, 64)


def simulate(L, stream, ranks, pool_pages, n_slots, policy, lookahead=0, window=4096):
    """Serve `stream` through a planning pool; returns (loads, pages loaded)."""
    n_ad = len(ranks)
    pool = L.lora_pool_create(None, pool_pages, 64, n_slots, n_ad)
    stream = np.ascontiguousarray(stream, dtype=np.int32)
    loads = pages = 0
    try:
        for i in range(stream.size):
            a = int(stream[i])
            if policy == L.LORA_EVICT_FARTHEST:
                L.lora_pool_set_eviction(pool, policy, stream[i + 1:i + 1 + window], lookahead)
            elif i == 0:
                L.lora_pool_set_eviction(pool, policy)
            _, loaded, _ = L.lora_adapter_ensure(pool, a, int(ranks[a]), None, None, n_slots, n_ad, planning=True)
            if loaded:
                loads += 1
                pages += 2 * int(ranks[a]) * n_slots
            L.lora_adapter_release(pool, a)
    finally:
        L.lora_pool_destroy(pool)
    return loads, pages


def main(argv=None):
    import adapter_gemm_lora_gb300 as L
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--adapters", type=int, default=2000)
    ap.add_argument("--alpha", type=float, default=0.5, help="Zipf exponent of adapter popularity")
    ap.add_argument("--requests", type=int, default=20000)
    ap.add_argument("--resident-share", type=float, default=0.25,
                    help="pool pages as a share of all adapters' pages")
    ap.add_argument("--H", type=int, default=4096)
    ap.add_argument("--slots", type=int, default=128, help="projection slots (32 layers x q/k/v/o)")
    ap.add_argument("--seed", type=int, default=4)
    ap.add_argument("--lookaheads", default="1,2,4,8,16,32,64,0")
    args = ap.parse_args(argv)
    L.library()
    rng = np.random.default_rng(args.seed)
    ranks = rng.choice(RANKS, size=args.adapters)
    p = 1.0 / np.arange(1, args.adapters + 1) ** args.alpha
    popularity = rng.permutation(args.adapters)          # popularity rank -> adapter id
    stream = popularity[rng.choice(args.adapters, size=args.requests, p=p / p.sum())]
    pool_pages = int(args.resident_share * 2 * int(ranks.sum()) * args.slots)
    page_bytes = 2 * args.H
    out = {"tool": "eviction_sim", "adapters": args.adapters, "alpha": args.alpha, "requests": args.requests,
           "pool_pages": pool_pages, "resident_share": args.resident_share, "slots": args.slots, "H": args.H,
           "seed": args.seed, "policies": {}}
    t0 = time.time()
    names = {L.LORA_EVICT_LOAD_ORDER: "load_order", L.LORA_EVICT_LRU: "lru"}
    for pol, name in names.items():
        loads, pages = simulate(L, stream, ranks, pool_pages, args.slots, pol)
        out["policies"][name] = {"loads_per_request": round(loads / args.requests, 4),
                                 "MB_per_request": round(pages * page_bytes / args.requests / 1e6, 3)}
    lru = out["policies"]["lru"]["loads_per_request"]
    ks = [int(k) for k in args.lookaheads.split(",")]
    full = None
    sweep = {}
    for k in sorted(ks, key=lambda k: (k <= 0, k)):
        loads, pages = simulate(L, stream, ranks, pool_pages, args.slots, L.LORA_EVICT_FARTHEST, lookahead=k)
        sweep[k] = (loads / args.requests, pages * page_bytes / args.requests / 1e6)
        if k <= 0:
            full = sweep[k][0]
    for k, (lpr, mb) in sweep.items():
        rec = {"loads_per_request": round(lpr, 4), "MB_per_request": round(mb, 3)}
        if full is not None and lru > full:
            rec["gap_recovered"] = round((lru - lpr) / (lru - full), 3)
        out["policies"][f"farthest_k{k}" if k > 0 else "farthest_full_window"] = rec
    out["seconds"] = round(time.time() - t0, 1)
    print(json.dumps(out), flush=True)
    return out


if __name__ == "__main__":
    main()
