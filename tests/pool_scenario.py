"""Drive a pool-lifecycle scenario (tests/golden/pool_lifecycle_scenario.json or a random one)
through either the oracle's PoolModel or the library's planning pool, recording what each step
returns, so both can be compared with the fixture and with each other."""
from __future__ import annotations

import numpy as np

import oracle as O


class OracleDriver:
    def __init__(self, num_pages, n_slots, max_adapters, page_order=None, model_cls=O.PoolModel):
        self.m = model_cls(num_pages, n_slots, max_adapters, page_order)
        self.n_slots = n_slots

    def ensure(self, a, r):
        st, tab, loaded, ev = self.m.ensure(a, r, [True] * self.n_slots)
        return st, (None if tab is None else np.asarray(tab).tolist()), loaded, list(ev)

    def release_adapter(self, a):
        return self.m.release_adapter(a)

    def acquire(self, a):
        return self.m.acquire(a)

    def reserve(self, n):
        st, ids = self.m.reserve(n)
        return st, ids

    def release_pages(self, ids):
        return self.m.release(ids)

    def unload(self, a):
        return self.m.unload(a)

    def evict_idle(self, need):
        return self.m.evict_idle(need)

    def set_eviction(self, policy, future=(), lookahead=0):
        return self.m.set_eviction(policy, future, lookahead)

    def kv_grow(self, req, n, layers):
        st, ids = self.m.kv_grow(req, n, layers)
        return st, ids

    def kv_free(self, req):
        return self.m.kv_free(req)

    def kv_table(self, req, layer):
        return self.m.kv_table(req, layer).tolist() if req in self.m.kv else None

    def refs(self, a):
        return self.m.refs.get(a, -1)

    def resident(self):
        return sorted(self.m.tables)

    def stats(self):
        return self.m.stats()


class LibraryDriver:
    """The same operations on the C library's planning pool (host bookkeeping only)."""

    def __init__(self, L, num_pages, n_slots, max_adapters, page_order=None):
        self.L = L
        self.n_slots, self.max_adapters = n_slots, max_adapters
        self.p = L.lora_pool_create(None, num_pages, 64, n_slots, max_adapters,
                                    None if page_order is None else np.asarray(page_order, dtype=np.int64))

    def _call(self, fn, *args):
        try:
            return self.L.LORA_OK, fn(*args)
        except self.L.LoraError as e:
            return e.code, None

    def ensure(self, a, r):
        st, out = self._call(self.L.lora_adapter_ensure, self.p, a, r, None, None, self.n_slots, self.max_adapters,
                             None, True)
        if st != self.L.LORA_OK:
            return st, None, False, []
        tab, loaded, ev = out
        return st, tab.tolist(), loaded, ev

    def release_adapter(self, a):
        return self._call(self.L.lora_adapter_release, self.p, a)[0]

    def acquire(self, a):
        return self._call(self.L.lora_adapter_acquire, self.p, a)[0]

    def reserve(self, n):
        st, ids = self._call(self.L.lora_pool_reserve, self.p, n)
        return st, (None if ids is None else [int(i) for i in ids])

    def release_pages(self, ids):
        return self._call(self.L.lora_pool_release, self.p, ids)[0]

    def unload(self, a):
        return self._call(self.L.lora_adapter_unload, self.p, a, None, True)[0]

    def evict_idle(self, need):
        st, ev = self._call(self.L.lora_pool_evict_idle, self.p, need, self.max_adapters, None, True)
        return st, ([] if ev is None else ev)

    def set_eviction(self, policy, future=(), lookahead=0):
        return self._call(self.L.lora_pool_set_eviction, self.p, policy, list(future), lookahead)[0]

    def kv_grow(self, req, n, layers):
        return self._call(self.L.lora_kv_grow, self.p, req, n, layers)

    def kv_free(self, req):
        return self._call(self.L.lora_kv_free, self.p, req)[0]

    def kv_table(self, req, layer):
        if self.L.lora_kv_length(self.p, req) < 0:
            return None
        return self.L.lora_kv_table(self.p, req, layer).tolist()

    def refs(self, a):
        return self.L.lora_adapter_refs(self.p, a)

    def resident(self):
        return [a for a in range(self.max_adapters) if self.L.lora_adapter_refs(self.p, a) >= 0]

    def stats(self):
        s = self.L.lora_pool_stats(self.p)
        return {"free": s["free"], "adapter": s["adapter"], "reserved": s["reserved"],
                "resident_adapters": s["resident_adapters"]}

    def close(self):
        self.L.lora_pool_destroy(self.p)


def run_golden(driver, steps):
    """Run the fixture's steps; return a list of mismatch messages (empty when every expected
    field holds)."""
    bad = []
    for i, st in enumerate(steps):
        op = st["op"]
        if op == "ensure":
            got, tab, loaded, ev = driver.ensure(st["adapter"], st["rank"])
            if got != st["status"]:
                bad.append(f"step {i}: ensure status {got} != {st['status']}")
                continue
            if "loaded" in st and loaded != st["loaded"]:
                bad.append(f"step {i}: loaded {loaded} != {st['loaded']}")
            if "table" in st and (tab is None or [row for row in tab[0]] != st["table"]):
                bad.append(f"step {i}: table {tab} != {st['table']}")
            if "evicted" in st and got == 0 and ev != st["evicted"]:
                bad.append(f"step {i}: evicted {ev} != {st['evicted']}")
        elif op == "reserve":
            got, ids = driver.reserve(st["n"])
            if got != st["status"] or ("ids" in st and ids != st["ids"]):
                bad.append(f"step {i}: reserve {got} {ids}")
        elif op == "release_adapter":
            got = driver.release_adapter(st["adapter"])
            if got != st["status"]:
                bad.append(f"step {i}: release status {got} != {st['status']}")
        elif op == "unload":
            got = driver.unload(st["adapter"])
            if got != st["status"]:
                bad.append(f"step {i}: unload status {got} != {st['status']}")
        elif op == "evict_idle":
            got, ev = driver.evict_idle(st["need"])
            if got != st["status"] or ev != st["evicted"]:
                bad.append(f"step {i}: evict_idle {got} {ev}")
        elif op == "stats":
            s = driver.stats()
            for k in ("free", "adapter", "reserved", "resident_adapters"):
                if s[k] != st[k]:
                    bad.append(f"step {i}: stats {k} {s[k]} != {st[k]}")
            continue
        else:
            raise ValueError(op)
        if "refs" in st and driver.refs(st["adapter"]) != st["refs"]:
            bad.append(f"step {i}: refs {driver.refs(st['adapter'])} != {st['refs']}")
        if "free" in st and driver.stats()["free"] != st["free"]:
            bad.append(f"step {i}: free {driver.stats()['free']} != {st['free']}")
        if "resident" in st and driver.resident() != st["resident"]:
            bad.append(f"step {i}: resident {driver.resident()} != {st['resident']}")
    return bad


def random_ops(seed, n_ops, max_adapters):
    """A seeded sequence of lifecycle operations over a small pool (ranks 1..8)."""
    rng = np.random.default_rng(seed)
    ranks = rng.integers(1, 9, size=max_adapters)
    ops = []
    for _ in range(n_ops):
        k = rng.integers(0, 100)
        a = int(rng.integers(0, max_adapters))
        if k < 35:
            ops.append(("ensure", a, int(ranks[a])))
        elif k < 60:
            ops.append(("release_adapter", a))
        elif k < 67:
            ops.append(("acquire", a))
        elif k < 75:
            ops.append(("reserve", int(rng.integers(0, 12))))
        elif k < 82:
            ops.append(("release_reserved",))
        elif k < 88:
            ops.append(("unload", a))
        elif k < 93:
            ops.append(("evict_idle", int(rng.integers(0, 80))))
        elif k < 96:
            req = int(rng.integers(0, 4))
            if rng.random() < 0.7:
                ops.append(("kv_grow", req, int(rng.integers(0, 4)), 1 + req % 2 + int(rng.random() < 0.05)))
            else:
                ops.append(("kv_free", req))
        else:
            fut = rng.integers(0, max_adapters, size=int(rng.integers(0, 20))).tolist()
            ops.append(("set_eviction", int(rng.integers(0, 3)), fut, int(rng.integers(-1, 8))))
    return ops


def apply_op(driver, op, reserved_lists):
    """Apply one random op; return a comparable record of its outcome."""
    kind = op[0]
    if kind == "ensure":
        return ("ensure",) + tuple(map(_freeze, driver.ensure(op[1], op[2])))
    if kind == "release_adapter":
        return ("release_adapter", driver.release_adapter(op[1]))
    if kind == "acquire":
        return ("acquire", driver.acquire(op[1]))
    if kind == "reserve":
        st, ids = driver.reserve(op[1])
        if st == 0:
            reserved_lists.append(ids)
        return ("reserve", st, _freeze(ids))
    if kind == "release_reserved":
        if not reserved_lists:
            return ("release_reserved", None)
        ids = reserved_lists.pop(0)
        return ("release_reserved", driver.release_pages(ids))
    if kind == "unload":
        return ("unload", driver.unload(op[1]))
    if kind == "evict_idle":
        st, ev = driver.evict_idle(op[1])
        return ("evict_idle", st, tuple(ev))
    if kind == "set_eviction":
        return ("set_eviction", driver.set_eviction(op[1], op[2], op[3]))
    if kind == "kv_grow":
        st, ids = driver.kv_grow(op[1], op[2], op[3])
        return ("kv_grow", st, _freeze(ids), _freeze(driver.kv_table(op[1], 0)))
    if kind == "kv_free":
        return ("kv_free", driver.kv_free(op[1]))
    raise ValueError(kind)


def _freeze(v):
    if isinstance(v, list):
        return tuple(_freeze(x) for x in v)
    return v


def cache_loads(driver_factory, stream, capacity, policy, lookahead=0, foresight=True):
    """Serve a request stream one request at a time through a pool that holds `capacity`
    adapters of rank 1 (one slot): ensure the adapter, then end its request.  Returns the number
    of loads.  With the farthest-future rule the pool is told the requests after the current one
    (none when `foresight` is False)."""
    d = driver_factory(capacity * 2)
    loads = 0
    for i, a in enumerate(stream):
        d.set_eviction(policy, list(stream[i + 1:]) if foresight else [], lookahead)
        st, tab, loaded, ev = d.ensure(int(a), 1)
        assert st == 0, (i, a, st)
        loads += int(loaded)
        assert d.release_adapter(int(a)) == 0
    return loads


def min_loads(stream, capacity):
    """Fewest loads any eviction choice can give (exhaustive search over cache contents)."""
    from functools import lru_cache
    stream = tuple(int(a) for a in stream)

    @lru_cache(maxsize=None)
    def best(i, cache):
        if i == len(stream):
            return 0
        a = stream[i]
        if a in cache:
            return best(i + 1, cache)
        if len(cache) < capacity:
            return 1 + best(i + 1, tuple(sorted(cache + (a,))))
        return 1 + min(best(i + 1, tuple(sorted([c for c in cache if c != v] + [a]))) for v in cache)
    return best(0, ())
