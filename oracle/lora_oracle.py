"""CPU oracle for the unmerged multi-adapter LoRA linear layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The product path
(the CUDA library and its Python binding) never calls it, and this module
imports nothing from the product.

What it computes, and where the pages fix it
--------------------------------------------
* "S-LoRA, in depth", section "Merge or keep adapters separate": a LoRA
  adapter turns W (h x h) into W + AB with A (h x r) and B (r x h); for one
  token with activation x the layer output is xW + (xA)B.  The unmerged form
  keeps W shared and adds the per-token low-rank term.  ``linear_forward`` is
  that definition written out in fp64, token by token.
* Same page, section "Unified paging: adapters and KV cache in one pool": a
  page holds one vector of length H; a rank-r A or B takes r pages, because
  each is r vectors of length h.  Reading: page j of A holds column j of A;
  page j of B holds row j of B.  The oracle reads A and B *through the page
  table out of the pool array*, so a gather mistake on the GPU shows up here.
* Same section, the pool sketch: pages come from one free list shared with KV
  cache; an adapter needs rank * 2 * projections * layers pages; a request for
  more pages than are free fails and leaves the pool as it was.
  ``PoolModel`` restates that bookkeeping (pop from the end of the free list,
  released pages appended back), with the fixes noted on the class.
* Batching by adapter: tokens are grouped by adapter id with a stable order
  ("segments"); the pages name no algorithm for this, so the oracle takes the
  plainest definition: a stable ascending sort by adapter id, no-adapter
  tokens (id -1) first and outside every segment.

Precision: inputs are bf16 bit patterns; every product and sum here is fp64.
The GPU keeps bf16 inputs, accumulates in fp32 and rounds y once to bf16.

Parity pins (tests/test_oracle_pins.py) tie each function to something other
than itself: the merged/unmerged identity, the B = 0 special case, brute-force
loops on tiny inputs, placement and batch-composition invariance, recognisable
adapters, and the page arithmetic of the worked example on the same page.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

# Status codes mirrored by value from the C boundary (the oracle does not link it).
OK = 0
EINVAL = -1
ENOPAGES = -2
EUNKNOWN_ADAPTER = -3
ERANK = -4
EEXIST = -5
EBUSY = -8

MAX_RANK = 64

# Eviction rules for idle adapters.
EVICT_LOAD_ORDER = 0      # the pool sketch: the adapter loaded earliest
EVICT_LRU = 1             # least recently used (loaded, ensured or acquired)
EVICT_FARTHEST = 2        # next use farthest in the known future; beyond the lookahead, LRU


def bf16_to_f64(bits) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to fp64 exactly."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Pool bookkeeping ("Unified paging" section: one free list, one page = one H-vector)
# ---------------------------------------------------------------------------
class PoolModel:
    """Host bookkeeping of a unified page pool.

    Follows the sketch's semantics: ``free`` is a list of page ids and pages
    are taken with ``pop()`` from its end; pages given back are appended.
    Adapters carry the sketch's count of active requests: ``ensure`` gives a
    resident adapter one more, or loads a new one with one (making room by
    evicting idle adapters, those with no active request, in the order they
    were loaded); ``evict_idle`` is the sketch's eviction on its own.
    Differences from the sketch, each a fix rather than a new rule:
      * a failed request (too few free pages) changes nothing, and an eviction
        that could not free enough pages evicts nothing;
      * requests end with an explicit ``release`` (the sketch never decrements
        its count, so its idle-adapter eviction could never fire); ``load``
        makes a resident, idle adapter and ``unload`` refuses a busy one;
      * KV/filler pages are reserved and released by explicit page lists
        (the sketch's ``grow_kv`` per request).
    Page tables: for an adapter of rank r over ``n_slots`` projection slots,
    ``table[slot, 0, j]`` is the page of column j of A and ``table[slot, 1, j]``
    the page of row j of B.  Pages are taken in that order (slot-major, A then
    B, j ascending); a slot without LoRA gets -1 and takes no page.
    """

    def __init__(self, num_pages: int, n_slots: int, max_adapters: int,
                 page_order: Optional[Sequence[int]] = None):
        self.num_pages = int(num_pages)
        self.n_slots = int(n_slots)
        self.max_adapters = int(max_adapters)
        self.free: List[int] = list(range(num_pages)) if page_order is None else [int(p) for p in page_order]
        self.reserved: set = set()
        self.tables: Dict[int, np.ndarray] = {}
        self.ranks: Dict[int, int] = {}
        self.refs: Dict[int, int] = {}          # active requests per resident adapter, in load order
        # eviction rule ("Fewer Expert Transfers...", section "A better eviction rule cuts transfers
        # without changing routing" and appendix "Limited foresight"): which idle adapter goes first
        self.policy = EVICT_LOAD_ORDER
        self.future: List[int] = []             # upcoming adapter requests, in order
        self.lookahead = 0                      # requests of `future` looked at (<= 0: all)
        self.clock = 0
        self.last_use: Dict[int, int] = {}
        self.kv: Dict[int, List[int]] = {}      # request -> its KV pages, in the order taken
        self.kv_layers: Dict[int, int] = {}

    @staticmethod
    def pages_for_adapter(rank: int, layers: int, projections: int) -> int:
        """Pages one adapter takes: A and B are ``rank`` vectors each, per projection and layer."""
        return rank * 2 * projections * layers

    def reserve(self, n: int):
        if n < 0:
            return EINVAL, None
        if n > len(self.free):
            return ENOPAGES, None
        ids = [self.free.pop() for _ in range(n)]
        self.reserved.update(ids)
        return OK, ids

    def release(self, ids: Sequence[int]) -> int:
        ids = [int(i) for i in ids]
        if len(set(ids)) != len(ids) or any(i not in self.reserved for i in ids):
            return EINVAL
        for i in ids:
            self.reserved.discard(i)
        self.free.extend(ids)
        return OK

    def load(self, adapter: int, rank: int, present: Sequence[bool]):
        if not (0 <= adapter < self.max_adapters) or len(present) != self.n_slots:
            return EINVAL, None
        if not (1 <= rank <= MAX_RANK):
            return ERANK, None
        if adapter in self.tables:
            return EEXIST, None
        need = 2 * rank * sum(1 for p in present if p)
        if need > len(self.free):
            return ENOPAGES, None
        table = np.full((self.n_slots, 2, rank), -1, dtype=np.int64)
        for s in range(self.n_slots):
            if not present[s]:
                continue
            for half in (0, 1):
                for j in range(rank):
                    table[s, half, j] = self.free.pop()
        self.tables[adapter] = table
        self.ranks[adapter] = rank
        self.refs[adapter] = 0
        self._touch(adapter)
        return OK, table

    def unload(self, adapter: int) -> int:
        if adapter not in self.tables:
            return EUNKNOWN_ADAPTER
        if self.refs[adapter] > 0:
            return EBUSY
        self._drop(adapter)
        return OK

    def _drop(self, adapter: int) -> None:
        table = self.tables.pop(adapter)
        self.ranks.pop(adapter)
        self.refs.pop(adapter)
        self.last_use.pop(adapter, None)
        self.free.extend(int(p) for p in table.reshape(-1) if p >= 0)

    # ---- adapter lifecycle: the sketch's adapter_refs, ensure_adapter, evict_idle_adapters ----
    def acquire(self, adapter: int) -> int:
        if adapter not in self.tables:
            return EUNKNOWN_ADAPTER
        self.refs[adapter] += 1
        self._touch(adapter)
        return OK

    def _touch(self, adapter: int) -> None:
        self.clock += 1
        self.last_use[adapter] = self.clock

    def set_eviction(self, policy: int, future: Sequence[int] = (), lookahead: int = 0) -> int:
        if policy not in (EVICT_LOAD_ORDER, EVICT_LRU, EVICT_FARTHEST):
            return EINVAL
        self.policy = policy
        self.future = [int(a) for a in future]
        self.lookahead = int(lookahead)
        return OK

    def eviction_order(self) -> List[int]:
        """Idle resident adapters, the first to evict first."""
        idle = [a for a, n in self.refs.items() if n == 0]          # load order
        if self.policy == EVICT_LRU:
            return sorted(idle, key=lambda a: self.last_use[a])
        if self.policy == EVICT_FARTHEST:
            horizon = self.future if self.lookahead <= 0 else self.future[:self.lookahead]
            nxt = {}
            for i, a in enumerate(horizon):
                nxt.setdefault(a, i)
            beyond = [a for a in idle if a not in nxt]
            seen = [a for a in idle if a in nxt]
            # never used within the horizon: all equal, least recently used first; then the
            # rest, next use farthest first
            return sorted(beyond, key=lambda a: self.last_use[a]) + sorted(seen, key=lambda a: -nxt[a])
        return idle

    def release_adapter(self, adapter: int) -> int:
        if adapter not in self.tables:
            return EUNKNOWN_ADAPTER
        if self.refs[adapter] == 0:
            return EINVAL
        self.refs[adapter] -= 1
        return OK

    def evict_idle(self, need: int):
        """Evict idle adapters, oldest load first, until at least ``need`` pages are free.
        Returns (status, evicted ids).  If evicting every idle adapter would still leave fewer
        than ``need`` pages free, nothing is evicted (ENOPAGES)."""
        if need < 0:
            return EINVAL, []
        idle = self.eviction_order()
        freeable = sum(int((self.tables[a] >= 0).sum()) for a in idle)
        if len(self.free) + freeable < need:
            return ENOPAGES, []
        evicted = []
        for a in idle:
            if len(self.free) >= need:
                break
            self._drop(a)
            evicted.append(a)
        return OK, evicted

    def ensure(self, adapter: int, rank: int, present: Sequence[bool]):
        """The sketch's ensure_adapter.  Returns (status, table, loaded, evicted): a resident
        adapter gets one more active request (its factors are not looked at; a different rank
        is ERANK: the rank is part of the adapter); otherwise idle adapters are evicted to make
        room and the adapter is loaded with one request."""
        if adapter in self.tables:
            if rank != self.ranks[adapter]:
                return ERANK, None, False, []
            self.refs[adapter] += 1
            self._touch(adapter)
            return OK, self.tables[adapter], False, []
        if not (0 <= adapter < self.max_adapters) or len(present) != self.n_slots:
            return EINVAL, None, False, []
        if not (1 <= rank <= MAX_RANK):
            return ERANK, None, False, []
        need = 2 * rank * sum(1 for p in present if p)
        st, evicted = self.evict_idle(need)
        if st != OK:
            return st, None, False, []
        st, table = self.load(adapter, rank, present)
        assert st == OK
        self.refs[adapter] = 1
        return OK, table, True, evicted

    # ---- KV cache pages per request: the sketch's grow_kv ----
    def kv_grow(self, request: int, n_tokens: int, layers: int):
        """Pages for n_tokens new tokens of a request: each token takes 2 * layers pages (per
        layer ascending, its K vector then its V vector), popped from the shared free list.  Too
        few free pages: ENOPAGES, nothing taken (the sketch's "caller must preempt or abort").
        A request keeps the layer count of its first growth."""
        if n_tokens < 0 or layers < 1 or (request in self.kv_layers and self.kv_layers[request] != layers):
            return EINVAL, None
        need = 2 * layers * n_tokens
        if need > len(self.free):
            return ENOPAGES, None
        ids = [self.free.pop() for _ in range(need)]
        self.kv.setdefault(request, []).extend(ids)
        self.kv_layers[request] = layers
        return OK, ids

    def kv_free(self, request: int) -> int:
        """A finished request gives all its KV pages back, in the order they were taken."""
        if request not in self.kv:
            return EINVAL
        self.free.extend(self.kv.pop(request))
        self.kv_layers.pop(request)
        return OK

    def kv_table(self, request: int, layer: int) -> np.ndarray:
        """int [tokens, 2]: the (K page, V page) of every cached token of the request at a layer."""
        L = self.kv_layers[request]
        ids = np.asarray(self.kv[request], dtype=np.int64).reshape(-1, L, 2)
        return ids[:, layer, :]

    def stats(self) -> dict:
        adapter_pages = sum(int((t >= 0).sum()) for t in self.tables.values())
        kv_pages = sum(len(v) for v in self.kv.values())
        return {"free": len(self.free), "adapter": adapter_pages, "reserved": len(self.reserved) + kv_pages,
                "resident_adapters": len(self.tables)}


# ---------------------------------------------------------------------------
# Segments: tokens grouped by adapter id (stable)
# ---------------------------------------------------------------------------
def segments(token_adapter) -> tuple:
    """Group tokens by adapter.

    Returns (perm, seg_off, seg_adapter):
      perm        int32 [T]: stable ascending sort of token indices by adapter id;
                  tokens with id -1 come first;
      seg_off     int32 [S+1]: segment s covers perm[seg_off[s]:seg_off[s+1]];
                  seg_off[0] = number of no-adapter tokens, seg_off[S] = T;
      seg_adapter int32 [S]: adapter id of segment s, ascending; adapters
                  with no token get no segment.
    """
    ta = np.asarray(token_adapter, dtype=np.int64)
    perm = np.argsort(ta, kind="stable")
    keys = ta[perm]
    n_none = int((ta < 0).sum())
    body = keys[n_none:]
    if body.size == 0:
        return perm.astype(np.int32), np.array([n_none], dtype=np.int32), np.zeros(0, dtype=np.int32)
    starts = np.flatnonzero(np.r_[True, body[1:] != body[:-1]])
    seg_off = np.r_[starts + n_none, ta.size].astype(np.int32)
    seg_adapter = body[starts].astype(np.int32)
    return perm.astype(np.int32), seg_off, seg_adapter


# ---------------------------------------------------------------------------
# The unmerged forward: y_t = x_t W + (x_t A_{a(t)}) B_{a(t)}
# ---------------------------------------------------------------------------
def place_adapter(pool_bits: np.ndarray, table: np.ndarray, A_list, B_list) -> None:
    """Write one adapter's factors into the pool through its page table (in place).

    ``A_list[slot]`` is bf16 bits [H, r] (or None: no LoRA on that slot) and
    ``B_list[slot]`` bf16 bits [r, H].  Page ``table[slot, 0, j]`` receives
    column j of A and page ``table[slot, 1, j]`` row j of B: the only vectors
    of length H the two factors have.
    """
    for s, (A, B) in enumerate(zip(A_list, B_list)):
        if A is None:
            continue
        r = A.shape[1]
        for j in range(r):
            pool_bits[table[s, 0, j]] = A[:, j]
            pool_bits[table[s, 1, j]] = B[j, :]


def gather_adapter(pool_bits: np.ndarray, table_slot: np.ndarray):
    """Read one adapter's (A, B) on one slot out of the pool through its page table.

    ``table_slot`` is int [2, r]: row 0 = pages of A's columns, row 1 = pages of B's rows.
    Returns A (H x r) and B (r x H) in fp64.
    """
    A = bf16_to_f64(pool_bits[table_slot[0]]).T      # page j -> column j of A
    B = bf16_to_f64(pool_bits[table_slot[1]])        # page j -> row j of B
    return A, B


def linear_forward(pool_bits: np.ndarray, tables: Dict[int, np.ndarray], token_adapter,
                   slot: int, x_bits: np.ndarray, Wt_bits: np.ndarray,
                   tokens: Optional[Sequence[int]] = None):
    """Oracle forward of one projection slot.

    pool_bits     uint16 [num_pages, H]: the pool's contents (bf16 bits);
    tables        adapter id -> int [n_slots, 2, r] page table (-1 = slot without LoRA);
    token_adapter int [T]: adapter id per token, -1 = none;
    x_bits        uint16 [T, H]: activations;
    Wt_bits       uint16 [H, H]: base weight in nn.Linear layout W_t[out, in], so W = W_t^T;
    tokens        optional subset of token indices to evaluate (sampled checks at full size).

    Returns (y, delta) in fp64, rows in the order of ``tokens`` (all tokens by default):
    y = x W + delta, delta_t = (x_t A) B for the token's adapter, 0 for none.
    """
    ta = np.asarray(token_adapter, dtype=np.int64)
    idx = np.arange(ta.size) if tokens is None else np.asarray(tokens, dtype=np.int64)
    x = bf16_to_f64(x_bits[idx])
    W = bf16_to_f64(Wt_bits).T
    base = x @ W
    delta = np.zeros_like(base)
    for row, t in enumerate(idx):
        a = int(ta[t])
        if a < 0:
            continue
        tab = tables[a][slot]
        if tab[0, 0] < 0:            # this adapter carries no LoRA on this slot
            continue
        A, B = gather_adapter(pool_bits, tab)
        delta[row] = (x[row] @ A) @ B
    return base + delta, delta


def merged_forward(x_bits: np.ndarray, Wt_bits: np.ndarray, A_bits: np.ndarray, B_bits: np.ndarray) -> np.ndarray:
    """The merged form x (W + A B) of one adapter, fp64 ("Merge or keep adapters separate")."""
    x = bf16_to_f64(x_bits)
    W = bf16_to_f64(Wt_bits).T
    return x @ (W + bf16_to_f64(A_bits) @ bf16_to_f64(B_bits))


def bf16_round(values: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 (ties to even), returned as fp64.

    Used only to state expectations for exactly representable cases; it goes
    through fp32 first, which is exact for the small integers those cases use.
    """
    f = np.asarray(values, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return bf16_to_f64(u.astype(np.uint16))


# ---------------------------------------------------------------------------
# Decode attention over KV pages of the same pool
# ---------------------------------------------------------------------------
def attention_decode(pool_bits: np.ndarray, kv_tables: Sequence[np.ndarray], q_bits: np.ndarray,
                     n_heads: int) -> np.ndarray:
    """One layer's attention for one new token per request, reading K and V out of the pool.

    "S-LoRA, in depth", "Unified paging": a KV cache tensor for a sequence of length S takes S
    pages, one H-vector each, and one token holds a K and a V vector per layer; the pool serves
    them from the same free list as adapter pages.  The pages give no attention formula; this
    is the plain scaled dot-product attention of a decode step.  For request i, its cached
    tokens j (K_j = pool[kv_tables[i][j, 0]], V_j = pool[kv_tables[i][j, 1]]) and each head h of
    width d = H / n_heads:
        s_j = q_h . K_{j,h} / sqrt(d),   p = softmax_j(s),   out_h = sum_j p_j V_{j,h}
    q_bits: uint16 [n_req, H] bf16 bits.  Returns fp64 [n_req, H].  A request with no cached
    token gets zeros.
    """
    q_all = bf16_to_f64(q_bits)
    n_req, H = q_all.shape
    d = H // n_heads
    out = np.zeros((n_req, H))
    for i in range(n_req):
        tab = np.asarray(kv_tables[i], dtype=np.int64)
        if tab.shape[0] == 0:
            continue
        K = bf16_to_f64(pool_bits[tab[:, 0]])
        V = bf16_to_f64(pool_bits[tab[:, 1]])
        for h in range(n_heads):
            cols = slice(h * d, (h + 1) * d)
            s = np.array([float(np.dot(q_all[i, cols], K[j, cols])) for j in range(tab.shape[0])]) / np.sqrt(d)
            w = np.exp(s - s.max())
            w /= w.sum()
            out[i, cols] = w @ V[:, cols]
    return out
