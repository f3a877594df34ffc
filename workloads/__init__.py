"""Seeded synthetic workloads for the multi-adapter LoRA projection.

This module only *draws* inputs: adapter ranks, the request -> adapter map,
prompt lengths, the pool's free-list order, the KV-filler share, and the
tensors x, W, A and B (drawn in fp32, stored as bf16 bit patterns).  It holds
none of the method's arithmetic, so both the oracle and the CUDA path can be
fed from it without sharing any computation.

The five workloads follow the seeded configurations of the S-LoRA study
("S-LoRA, in depth", section "What the paper measured ..."): synthetic traffic
in which a few adapters are popular and most are rarely used, represented by a
finite Zipf law over the adapter set.  No dataset and no trained weight is
used; random weights stand in for Llama-shaped projections.

Drawing order.  One ``numpy.random.default_rng(seed)`` draws the batch
structure in a fixed order: ranks, request -> adapter, prompt lengths, page
permutation.  Each tensor then comes from its own child generator
``default_rng([seed, TAG, i, j])`` so that any slot or adapter can be
regenerated alone (the full-size workloads hold tens of GB of adapter weights
and are generated lazily, one adapter or slot at a time).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Tuple

import numpy as np

# Tags of the per-tensor child generators.
_TAG_X, _TAG_W, _TAG_A, _TAG_B = 11, 12, 13, 14

RANK_CHOICES = (8, 16, 32, 64)


def to_bf16_bits(values_f32: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return uint16 bits.

    The draws are finite normals, so no NaN/Inf handling is needed.
    """
    u = np.ascontiguousarray(values_f32, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


@dataclass(frozen=True)
class Spec:
    """Static description of one seeded workload."""
    key: int
    name: str
    H: int
    n_slots: int
    n_adapters: int
    pool_pages: int
    kv_fill: float                       # share of the pool reserved as KV filler before adapters load
    assign: str                          # "uniform" | "zipf" | "perm"
    zipf_alpha: float = 0.0
    fixed_ranks: Optional[Tuple[int, ...]] = None
    n_decode: int = 0                    # requests with one token each
    prefill_lens: Optional[Tuple[int, ...]] = None   # fixed prompt lengths
    prefill_uniform: Optional[Tuple[int, int, int]] = None  # (n_req, lo, hi) inclusive
    tokens_per_req: int = 1              # for decode-style requests
    layers: int = 1                      # q/k/v/o layers (n_slots = 4 * layers) or 1 for a single slot

    @property
    def description(self) -> str:
        return _DESCRIPTIONS[self.key]


_DESCRIPTIONS = {
    1: "tiny single projection: H=256, one 256x256 W, 4 adapters r={8,8,16,16}, 8 req x 4 tok, uniform",
    2: "decode: H=4096 q/k/v/o, 256 req x 1 tok, 64 adapters r~U{8,16,32,64}, Zipf(1.0), pool 2^18, 50% KV",
    3: "prefill: H=4096 q/k/v/o, 16 req, len U[128,1024], 16 adapters, one per request, pool 2^18, 50% KV",
    4: "many adapters: H=4096 q/k/v/o, 1024 req x 1 tok, 2000 adapters, Zipf(0.5), pool 2^20, 50% KV",
    5: "layer stack: H=5120, 40 layers x q/k/v/o, 256 adapters, Zipf(1.0), 448 decode + 4x512 prefill, pool 2^22, 30% KV",
}

SPECS = {
    1: Spec(1, "tiny", H=256, n_slots=1, n_adapters=4, pool_pages=1024, kv_fill=0.0,
            assign="uniform", fixed_ranks=(8, 8, 16, 16), n_decode=8, tokens_per_req=4),
    2: Spec(2, "decode", H=4096, n_slots=4, n_adapters=64, pool_pages=1 << 18, kv_fill=0.5,
            assign="zipf", zipf_alpha=1.0, n_decode=256, layers=1),
    3: Spec(3, "prefill", H=4096, n_slots=4, n_adapters=16, pool_pages=1 << 18, kv_fill=0.5,
            assign="perm", prefill_uniform=(16, 128, 1024), layers=1),
    4: Spec(4, "many", H=4096, n_slots=4, n_adapters=2000, pool_pages=1 << 20, kv_fill=0.5,
            assign="zipf", zipf_alpha=0.5, n_decode=1024, layers=1),
    5: Spec(5, "stack", H=5120, n_slots=160, n_adapters=256, pool_pages=1 << 22, kv_fill=0.3,
            assign="zipf", zipf_alpha=1.0, n_decode=448, prefill_lens=(512, 512, 512, 512), layers=40),
}


@dataclass
class Workload:
    """One seeded draw of a workload: batch structure plus lazily drawn tensors."""
    spec: Spec
    seed: int
    ranks: np.ndarray              # int32 [n_adapters]
    req_adapter: np.ndarray        # int32 [n_req]
    req_len: np.ndarray            # int32 [n_req]
    token_adapter: np.ndarray      # int32 [T]; -1 = no adapter
    page_order: np.ndarray         # int64 [pool_pages]: free-list order handed to the pool
    kv_pages: int                  # pages reserved as KV filler before the adapters load
    _cache: dict = field(default_factory=dict, repr=False)

    # ---- shapes -----------------------------------------------------------
    @property
    def H(self) -> int:
        return self.spec.H

    @property
    def T(self) -> int:
        return int(self.token_adapter.shape[0])

    @property
    def n_slots(self) -> int:
        return self.spec.n_slots

    def slot_input(self, slot: int) -> int:
        """Index of the activation a projection slot reads.

        q, k and v of a layer read the same x_l; o reads an independent x'_l;
        each layer has its own inputs (no chaining through un-normalised layers).
        """
        if self.spec.n_slots == 1:
            return 0
        layer, proj = divmod(slot, 4)
        return 2 * layer + (1 if proj == 3 else 0)

    def slot_groups(self):
        """Runs of consecutive slots that read the same input: [[q, k, v], [o], ...] per layer."""
        groups = []
        for slot in range(self.n_slots):
            if groups and self.slot_input(groups[-1][-1]) == self.slot_input(slot):
                groups[-1].append(slot)
            else:
                groups.append([slot])
        return groups

    @property
    def n_inputs(self) -> int:
        return 1 if self.spec.n_slots == 1 else 2 * (self.spec.n_slots // 4)

    # ---- tensors (bf16 bit patterns, uint16) ------------------------------
    def _normal(self, tag: int, i: int, j: int, shape, std: float) -> np.ndarray:
        g = np.random.default_rng([self.seed, tag, i, j])
        v = g.standard_normal(size=shape, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        return to_bf16_bits(v)

    def x(self, inp: int) -> np.ndarray:
        """Activation ``inp``: bf16 [T, H], x ~ N(0, 1)."""
        return self._normal(_TAG_X, inp, 0, (self.T, self.H), 1.0)

    def W(self, slot: int) -> np.ndarray:
        """Base weight of ``slot`` in nn.Linear layout W_t[out, in]: bf16 [H, H], N(0, 1/H)."""
        return self._normal(_TAG_W, slot, 0, (self.H, self.H), 1.0 / np.sqrt(self.H))

    def A(self, adapter: int, slot: int) -> np.ndarray:
        """LoRA down-projection of ``adapter`` on ``slot``: bf16 [H, r], N(0, 1/H)."""
        r = int(self.ranks[adapter])
        return self._normal(_TAG_A, adapter, slot, (self.H, r), 1.0 / np.sqrt(self.H))

    def B(self, adapter: int, slot: int) -> np.ndarray:
        """LoRA up-projection of ``adapter`` on ``slot``: bf16 [r, H], N(0, 1/r)."""
        r = int(self.ranks[adapter])
        return self._normal(_TAG_B, adapter, slot, (r, self.H), 1.0 / np.sqrt(r))

    # ---- accounting -------------------------------------------------------
    def adapter_pages(self) -> int:
        """Pages all adapters take: 2 * r per slot (A and B are r vectors each)."""
        return int(2 * self.ranks.astype(np.int64).sum() * self.n_slots)


def _zipf_probs(n: int, alpha: float) -> np.ndarray:
    k = np.arange(1, n + 1, dtype=np.float64)
    p = k ** (-alpha)
    return p / p.sum()


def make(key: int, seed: Optional[int] = None, **overrides) -> Workload:
    """Draw workload ``key`` (1..5) with ``seed`` (default: the key itself).

    ``overrides`` replace Spec fields (used by tests for small variants, e.g.
    ``pool_pages`` or ``kv_fill``).
    """
    spec = SPECS[key]
    if overrides:
        spec = Spec(**{**spec.__dict__, **overrides})
    seed = key if seed is None else seed
    rng = np.random.default_rng(seed)

    # 1. ranks
    if spec.fixed_ranks is not None:
        ranks = np.array(spec.fixed_ranks, dtype=np.int32)
    else:
        ranks = rng.choice(np.array(RANK_CHOICES, dtype=np.int32), size=spec.n_adapters)
    ranks = ranks.astype(np.int32)

    # 2. requests and their adapters
    if spec.prefill_uniform is not None:
        n_pre = spec.prefill_uniform[0]
    elif spec.prefill_lens is not None:
        n_pre = len(spec.prefill_lens)
    else:
        n_pre = 0
    n_req = spec.n_decode + n_pre
    if spec.assign == "uniform":
        req_adapter = rng.integers(0, spec.n_adapters, size=n_req)
    elif spec.assign == "perm":
        req_adapter = rng.permutation(spec.n_adapters)[:n_req]
    elif spec.assign == "zipf":
        popularity = rng.choice(spec.n_adapters, size=n_req, p=_zipf_probs(spec.n_adapters, spec.zipf_alpha))
        rank_to_id = rng.permutation(spec.n_adapters)
        req_adapter = rank_to_id[popularity]
    else:
        raise ValueError(spec.assign)
    req_adapter = req_adapter.astype(np.int32)

    # 3. prompt lengths: decode requests first, then prefill requests
    lens = [spec.tokens_per_req] * spec.n_decode
    if spec.prefill_uniform is not None:
        _, lo, hi = spec.prefill_uniform
        lens += list(rng.integers(lo, hi + 1, size=n_pre))
    elif spec.prefill_lens is not None:
        lens += list(spec.prefill_lens)
    req_len = np.array(lens, dtype=np.int32)
    token_adapter = np.repeat(req_adapter, req_len).astype(np.int32)

    # 4. page permutation: the free list order handed to the pool
    page_order = rng.permutation(spec.pool_pages).astype(np.int64)
    kv_pages = int(spec.kv_fill * spec.pool_pages)

    return Workload(spec=spec, seed=seed, ranks=ranks, req_adapter=req_adapter, req_len=req_len,
                    token_adapter=token_adapter, page_order=page_order, kv_pages=kv_pages)


def small(H: int, T: int, n_adapters: int, ranks, seed: int, n_slots: int = 1,
          pool_pages: Optional[int] = None, kv_fill: float = 0.25,
          none_share: float = 0.0) -> Workload:
    """A small custom workload for parity edge cases (ragged T, odd ranks, no-adapter tokens).

    Tokens get adapters uniformly; a share ``none_share`` of them gets -1 (no adapter).
    """
    rng = np.random.default_rng(seed)
    ranks = np.array(ranks, dtype=np.int32)
    assert ranks.shape[0] == n_adapters
    token_adapter = rng.integers(0, n_adapters, size=T).astype(np.int32)
    if none_share > 0:
        token_adapter[rng.random(T) < none_share] = -1
    need = int(2 * ranks.astype(np.int64).sum() * n_slots)
    if pool_pages is None:
        pool_pages = int((need + 16) / max(1e-9, 1.0 - kv_fill)) + 8
    page_order = rng.permutation(pool_pages).astype(np.int64)
    spec = Spec(0, "small", H=H, n_slots=n_slots, n_adapters=n_adapters, pool_pages=pool_pages,
                kv_fill=kv_fill, assign="uniform", n_decode=T)
    return Workload(spec=spec, seed=seed, ranks=ranks, req_adapter=token_adapter.copy(),
                    req_len=np.ones(T, dtype=np.int32), token_adapter=token_adapter,
                    page_order=page_order, kv_pages=int(kv_fill * pool_pages))


def small_prefill(H: int, req_lens, n_adapters: int, ranks, seed: int, n_slots: int = 1,
                  kv_fill: float = 0.25, none_reqs=(), n_decode: int = 0) -> Workload:
    """A small prefill-shaped workload: `n_decode` one-token requests with uniform adapters, then
    one request per entry of `req_lens`, all of whose tokens carry that request's adapter (drawn
    uniformly; requests listed in `none_reqs` carry none, -1)."""
    rng = np.random.default_rng(seed)
    ranks = np.array(ranks, dtype=np.int32)
    assert ranks.shape[0] == n_adapters
    lens = np.array([1] * n_decode + list(req_lens), dtype=np.int32)
    req_adapter = rng.integers(0, n_adapters, size=lens.size).astype(np.int32)
    for i in none_reqs:
        req_adapter[n_decode + i] = -1
    token_adapter = np.repeat(req_adapter, lens).astype(np.int32)
    T = int(lens.sum())
    need = int(2 * ranks.astype(np.int64).sum() * n_slots)
    pool_pages = int((need + 16) / max(1e-9, 1.0 - kv_fill)) + 8
    page_order = rng.permutation(pool_pages).astype(np.int64)
    spec = Spec(0, "small_prefill", H=H, n_slots=n_slots, n_adapters=n_adapters, pool_pages=pool_pages,
                kv_fill=kv_fill, assign="uniform", n_decode=T)
    return Workload(spec=spec, seed=seed, ranks=ranks, req_adapter=req_adapter, req_len=lens,
                    token_adapter=token_adapter, page_order=page_order, kv_pages=int(kv_fill * pool_pages))
