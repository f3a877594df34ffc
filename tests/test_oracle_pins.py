"""The oracle against what the pages and the mathematics fix (CPU only)."""
import json
import os

import numpy as np
import pytest

import oracle as O
import workloads
from pins import ALL_PINS, build_scene

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin_holds(pin):
    ok, msg = pin(O)
    assert ok, msg


def test_worked_example_page_arithmetic():
    """'Unified paging' worked example: adapter and KV sizes in pages and bytes."""
    g = json.load(open(os.path.join(GOLDEN, "pool_worked_example.json")))
    H, L, nb = g["hidden"], g["layers"], g["bytes_per_value"]
    kv_vectors = 2 * L                                       # K and V per layer
    assert kv_vectors == g["kv_vectors_per_token"]
    assert kv_vectors * H * nb == g["kv_bytes_per_token"]
    assert g["adapter_rank"] * 2 * g["projections"] == g["adapter_vectors_per_layer"]
    pages = O.PoolModel.pages_for_adapter(g["adapter_rank"], L, g["projections"])
    assert pages == g["adapter_vectors"]
    assert pages * H * nb == g["adapter_bytes"]
    assert g["adapter_bytes"] // g["kv_bytes_per_token"] == g["kv_tokens_per_adapter"]
    assert round(g["context_tokens"] / g["kv_tokens_per_adapter"]) == g["adapters_per_context_about"]
    total_gib = g["adapters"] * g["adapter_bytes"] / 2**30
    assert abs(total_gib - g["adapters_total_gib_about"]) < 1.0


def test_pool_enopages_exactly_at_boundary_and_unchanged():
    pool = O.PoolModel(100, n_slots=2, max_adapters=8, page_order=np.random.default_rng(0).permutation(100))
    assert pool.reserve(36)[0] == O.OK                       # 64 left
    assert pool.load(0, 16, [True, True])[0] == O.OK          # 64 pages -> 0 left
    before = (list(pool.free), dict(pool.ranks))
    assert pool.load(1, 1, [True, False])[0] == O.ENOPAGES    # needs 2, has 0
    assert (list(pool.free), dict(pool.ranks)) == before
    assert pool.unload(0) == O.OK
    st, tab = pool.load(1, 16, [True, True])                 # exactly 64 again
    assert st == O.OK and len(pool.free) == 0
    assert pool.load(2, 1, [True, False])[0] == O.ENOPAGES


def test_pool_errors_and_stats():
    pool = O.PoolModel(64, n_slots=3, max_adapters=4)
    assert pool.load(0, 0, [True] * 3)[0] == O.ERANK
    assert pool.load(0, 65, [True] * 3)[0] == O.ERANK
    assert pool.load(4, 8, [True] * 3)[0] == O.EINVAL
    assert pool.load(-1, 8, [True] * 3)[0] == O.EINVAL
    assert pool.load(1, 8, [True, False, True])[0] == O.OK
    assert pool.load(1, 8, [True] * 3)[0] == O.EEXIST
    assert pool.unload(2) == O.EUNKNOWN_ADAPTER
    st, ids = pool.reserve(5)
    assert pool.release(ids + [ids[0]]) == O.EINVAL           # duplicate
    assert pool.stats() == {"free": 64 - 32 - 5, "adapter": 32, "reserved": 5, "resident_adapters": 1}
    assert pool.release(ids) == O.OK
    assert pool.tables[1][1].min() == -1 and pool.tables[1][0].min() >= 0


def test_free_list_pops_from_end_in_table_order():
    order = np.array([5, 9, 2, 7, 1, 0, 3, 8, 4, 6])
    pool = O.PoolModel(10, n_slots=2, max_adapters=2, page_order=order)
    st, tab = pool.load(0, 2, [True, True])
    assert st == O.OK
    # slot 0: A pages then B pages, then slot 1; each taken from the end of the list
    assert tab.reshape(-1).tolist() == [6, 4, 8, 3, 0, 1, 7, 2]


def test_init_statistics_unit_variance():
    """With x~N(0,1), W,A~N(0,1/H), B~N(0,1/r): x W and the delta have variance near 1."""
    sc = build_scene(O, H=256, ranks=[16], T=64, seed=21, none_share=0.0)
    y, delta = O.linear_forward(sc["pool_bits"], sc["pool"].tables, sc["ta"], 0, sc["x"], sc["Wt"][0])
    base = y - delta
    assert 0.7 < base.var() < 1.3
    assert 0.6 < delta.var() < 1.4


def test_workload_structure():
    w2 = workloads.make(2)
    assert w2.T == 256 and w2.ranks.shape == (64,) and set(np.unique(w2.ranks)) <= {8, 16, 32, 64}
    w3 = workloads.make(3)
    assert len(set(w3.req_adapter.tolist())) == 16 and 16 * 128 <= w3.T <= 16 * 1024
    w1 = workloads.make(1)
    assert w1.T == 32 and w1.ranks.tolist() == [8, 8, 16, 16]
    for k in (1, 2, 3, 4, 5):
        w = workloads.make(k)
        assert w.adapter_pages() + w.kv_pages <= w.spec.pool_pages
    # lazily drawn tensors are reproducible one by one
    assert np.array_equal(w2.A(3, 1), workloads.make(2).A(3, 1))


def test_bf16_round_ties_to_even():
    vals = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 256.0, -3.5])
    got = O.bf16_round(vals)
    assert got.tolist() == [1.0, 1.0, 1.0 + 2**-6, 256.0, -3.5]


def test_pool_lifecycle_golden_scenario():
    """The pool sketch's adapter lifecycle ("Unified paging"), worked out by hand on 40 pages:
    page ids taken, active-request counts, eviction order and failures."""
    from pool_scenario import OracleDriver, run_golden
    g = json.load(open(os.path.join(GOLDEN, "pool_lifecycle_scenario.json")))
    d = OracleDriver(g["pool"]["num_pages"], g["pool"]["n_slots"], g["pool"]["max_adapters"])
    assert run_golden(d, g["steps"]) == []


def test_pool_lifecycle_invariants():
    """Random lifecycle sequences (adapters, reserved and KV pages): every page is in exactly one
    place, only idle adapters are evicted, a successful ensure leaves the adapter resident with
    an active request, and a failed ensure or eviction changes nothing."""
    from pool_scenario import OracleDriver, apply_op, random_ops
    n_pages, n_ad = 96, 10
    for seed in range(20):
        d = OracleDriver(n_pages, 2, n_ad, page_order=np.random.default_rng(seed).permutation(n_pages))
        reserved = []
        for op in random_ops(seed, 300, n_ad):
            refs_before = dict(d.m.refs)
            free_before = list(d.m.free)
            rec = apply_op(d, op, reserved)
            pages = [int(p) for t in d.m.tables.values() for p in t.reshape(-1) if p >= 0]
            kv = [p for ids in d.m.kv.values() for p in ids]
            owned = pages + kv + list(d.m.reserved)
            assert len(owned) == len(set(owned)), "a page has two owners"
            assert not set(owned) & set(d.m.free)
            assert len(owned) + len(d.m.free) == n_pages
            if rec[0] in ("ensure", "evict_idle"):
                for a in rec[-1]:
                    assert refs_before.get(a) == 0, f"busy adapter {a} evicted"
                if rec[1] == O.ENOPAGES:
                    assert d.m.refs == refs_before and d.m.free == free_before
            if rec[0] == "ensure" and rec[1] == O.OK:
                assert d.m.refs[op[1]] >= 1


def _cache_driver(model_cls=O.PoolModel, n_ad=16):
    from pool_scenario import OracleDriver
    return lambda pages: OracleDriver(pages, 1, n_ad, model_cls=model_cls)


def _letters(stream):
    return [ord(c) - ord("A") for c in stream]


def eviction_pin_failures(model_cls=O.PoolModel):
    """The eviction rules against what fixes them; returns a list of failures (empty = pinned).
    (1) the introduction's two-slot sequences under LRU; (2) Belady: one request at a time,
    farthest-future eviction gives the fewest loads any schedule can (exhaustive search);
    (3) LRU never beats that minimum; (4) the farthest-future rule told nothing is LRU."""
    from pool_scenario import cache_loads, min_loads
    bad = []
    g = json.load(open(os.path.join(GOLDEN, "eviction_toy_sequences.json")))
    for case in g["cases"]:
        got = cache_loads(_cache_driver(model_cls), _letters(case["stream"]), g["capacity"], O.EVICT_LRU)
        if got != case["loads"]:
            bad.append(f"toy {case['stream']}: {got} loads != {case['loads']}")
    rng = np.random.default_rng(7)
    for trial in range(120):
        n = int(rng.integers(2, 7))
        cap = int(rng.integers(1, n))
        stream = rng.integers(0, n, size=int(rng.integers(1, 13))).tolist()
        opt = min_loads(stream, cap)
        ff = cache_loads(_cache_driver(model_cls), stream, cap, O.EVICT_FARTHEST)
        lru = cache_loads(_cache_driver(model_cls), stream, cap, O.EVICT_LRU)
        blind = cache_loads(_cache_driver(model_cls), stream, cap, O.EVICT_FARTHEST, foresight=False)
        if ff != opt:
            bad.append(f"farthest-future {ff} != optimum {opt} on {stream} (capacity {cap})")
        if lru < opt:
            bad.append(f"LRU {lru} below the optimum {opt} on {stream}")
        if blind != lru:
            bad.append(f"farthest-future without foresight {blind} != LRU {lru} on {stream}")
    return bad


def test_eviction_rules_pinned():
    assert eviction_pin_failures() == []


def test_lookahead_window():
    """The farthest-future rule with a horizon of k requests: k = 0 or a horizon past the end of
    the stream is the full rule; a horizon of 1 can only see the next request."""
    from pool_scenario import cache_loads
    rng = np.random.default_rng(11)
    for trial in range(40):
        stream = rng.integers(0, 6, size=30).tolist()
        full = cache_loads(_cache_driver(), stream, 3, O.EVICT_FARTHEST)
        assert cache_loads(_cache_driver(), stream, 3, O.EVICT_FARTHEST, lookahead=100) == full
        assert cache_loads(_cache_driver(), stream, 3, O.EVICT_FARTHEST, lookahead=1) >= full


# ---- decode attention over pool pages, and the KV pages it reads -----------------------------
def _bits(values):
    return workloads.to_bf16_bits(np.asarray(values, dtype=np.float32))


def attention_pin_failures(attention=None):
    """Decode attention against closed forms; returns failures (empty = pinned)."""
    attention = attention or O.attention_decode
    bad = []
    # two heads of width 4, two cached tokens with hand-picked vectors: the scores are 1, 0 (head
    # 0) and 1, -1 (head 1) after the 1/sqrt(4) scale, so the weights are sigmoids of 1 and 2
    H = 8
    pool = np.zeros((6, H), np.uint16)
    pool[2] = _bits([2, 0, 0, 0, 0, 1, 0, 0])     # K of token 0
    pool[5] = _bits([0, 0, 0, 0, 0, -1, 0, 0])    # K of token 1
    pool[0] = _bits([1, 1, 1, 1, 4, 0, 0, 0])     # V of token 0
    pool[3] = _bits([3, 3, 3, 3, 0, 4, 0, 0])     # V of token 1
    q = _bits([[1, 0, 0, 0, 0, 2, 0, 0]])
    out = attention(pool, [np.array([[2, 0], [5, 3]])], q, 2)[0]
    a = 1 / (1 + np.exp(-1.0))
    b = 1 / (1 + np.exp(-2.0))
    want = np.array([a + 3 * (1 - a)] * 4 + [4 * b, 4 * (1 - b), 0, 0])
    if not np.allclose(out, want, rtol=0, atol=1e-12):
        bad.append(f"two-token closed form: {out} != {want}")
    # one cached token: the output is its V, whatever q and K are
    rng = np.random.default_rng(3)
    H, nh = 64, 4
    pool = _bits(rng.standard_normal((10, H)))
    q = _bits(rng.standard_normal((1, H)))
    out = attention(pool, [np.array([[7, 2]])], q, nh)[0]
    if not np.array_equal(out, O.bf16_to_f64(pool[2])):
        bad.append("one cached token does not return its V")
    # identical keys: uniform weights, the output is the mean of the V rows
    tab = np.array([[7, 1], [7, 4], [7, 9]])
    out = attention(pool, [tab], q, nh)[0]
    if not np.allclose(out, O.bf16_to_f64(pool[[1, 4, 9]]).mean(axis=0), rtol=0, atol=1e-12):
        bad.append("identical keys do not average V")
    # a head sees only its own columns: changing K and q outside head 0 leaves head 0 unchanged
    tab = np.array([[0, 1], [3, 4], [5, 6]])
    q2 = q.copy()
    q2[0, 16:] = _bits(rng.standard_normal(H - 16))
    pool2 = pool.copy()
    pool2[[0, 3, 5], 16:] = _bits(rng.standard_normal((3, H - 16)))
    o1 = attention(pool, [tab], q, nh)[0, :16]
    o2 = attention(pool2, [tab], q2, nh)[0, :16]
    if not np.allclose(o1, o2, rtol=0, atol=1e-12):
        bad.append("heads are not independent")
    return bad


def test_attention_decode_pinned():
    assert attention_pin_failures() == []


def test_attention_invariant_to_token_order_and_page_placement():
    rng = np.random.default_rng(5)
    H, nh, n = 128, 8, 9
    pool = workloads.to_bf16_bits(rng.standard_normal((40, H)).astype(np.float32))
    q = workloads.to_bf16_bits(rng.standard_normal((2, H)).astype(np.float32))
    tabs = [rng.choice(40, size=(n, 2), replace=False), rng.choice(40, size=(4, 2), replace=False)]
    base = O.attention_decode(pool, tabs, q, nh)
    perm = rng.permutation(n)
    assert np.allclose(O.attention_decode(pool, [tabs[0][perm], tabs[1]], q, nh), base, rtol=0, atol=1e-12)
    moved = np.full_like(pool, 0x7FC0)
    new_ids = rng.permutation(40)                       # every page moved to another id
    moved[new_ids] = pool
    assert np.array_equal(O.attention_decode(moved, [new_ids[t] for t in tabs], q, nh), base)


def test_kv_pages_per_token_and_order():
    """The sketch's grow_kv: 2 pages per layer per token (the worked example: 64 for 32 layers),
    popped from the end of the shared free list, K then V per layer; a failed growth takes nothing."""
    g = json.load(open(os.path.join(GOLDEN, "pool_worked_example.json")))
    m = O.PoolModel(200, 1, 4)
    st, ids = m.kv_grow(9, 1, g["layers"])
    assert st == O.OK and len(ids) == g["kv_vectors_per_token"]
    m = O.PoolModel(20, 1, 4)                           # free list 0..19, popped from the end
    assert m.kv_grow(7, 2, 2) == (O.OK, [19, 18, 17, 16, 15, 14, 13, 12])
    assert m.kv_table(7, 1).tolist() == [[17, 16], [13, 12]]      # layer 1: (K, V) per token
    assert m.kv_grow(7, 1, 3)[0] == O.EINVAL            # layer count fixed by the first growth
    assert m.kv_grow(8, 4, 2)[0] == O.ENOPAGES and len(m.free) == 12   # 16 pages asked, 12 free
    assert m.kv_free(7) == O.OK and m.free[-8:] == [19, 18, 17, 16, 15, 14, 13, 12]
    assert m.kv_free(7) == O.EINVAL


def test_workload_generator_scales_give_unit_variance():
    """Sanity, not parity, on the generator the benchmark and the GPU tests draw from (the test
    above uses the pins' own draws): with x ~ N(0,1), W, A ~ N(0, 1/H), B ~ N(0, 1/r), an
    element of xW has variance H * 1 * (1/H) = 1 and an element of the LoRA delta (xA)B has
    variance r * (H * 1/H) * (1/r) = 1.  A standard deviation of 1/H in place of 1/sqrt(H)
    would give 1/H."""
    H, T = 512, 96
    wl = workloads.small(H=H, T=T, n_adapters=4, ranks=[8, 16, 32, 64], seed=17, none_share=0.0)
    model = O.PoolModel(wl.spec.pool_pages, 1, 4, wl.page_order)
    pool = np.full((wl.spec.pool_pages, H), 0x7FC0, np.uint16)
    for a in range(4):
        st, tab = model.load(a, int(wl.ranks[a]), [True])
        O.place_adapter(pool, tab, [wl.A(a, 0)], [wl.B(a, 0)])
    y, delta = O.linear_forward(pool, model.tables, wl.token_adapter, 0, wl.x(0), wl.W(0))
    base = y - delta
    assert 0.85 < base.var() < 1.15, base.var()
    assert 0.8 < delta.var() < 1.2, delta.var()
    assert abs(base.mean()) < 0.05 and abs(delta.mean()) < 0.05
