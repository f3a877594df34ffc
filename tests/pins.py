"""Pin checks for the oracle, written against an oracle-like namespace.

Each ``pin_*`` function takes ``O`` (the oracle module, or a copy of it with a
planted mistake) and returns (ok, message).  test_oracle_pins.py runs them on
the real oracle (all must hold); test_oracle_mutations.py runs them on mutants
(each mutant must break at least one).

None of these re-types the oracle's formula: each compares it with something
fixed independently: the merged form x(W + AB) computed from the matrices
(never through pages), scalar loops, exact special cases, invariances, or the
pages' worked example.
"""
from __future__ import annotations

import numpy as np

from workloads import to_bf16_bits


def _rand_bits(rng, shape, std=1.0):
    return to_bf16_bits((rng.standard_normal(shape) * std).astype(np.float32))


def build_scene(O, H, ranks, T, n_slots=1, seed=0, kv_fill=0.3, page_order_seed=None, none_share=0.25,
                token_adapter=None, zero_B=()):
    """Small scene: pool + page tables + inputs, placed through the oracle's own pool model."""
    rng = np.random.default_rng(seed)
    n_ad = len(ranks)
    need = 2 * int(sum(ranks)) * n_slots
    num_pages = int((need + 8) / (1 - kv_fill)) + 4
    order_rng = np.random.default_rng(seed if page_order_seed is None else page_order_seed)
    page_order = order_rng.permutation(num_pages)
    pool = O.PoolModel(num_pages, n_slots, max_adapters=n_ad + 2, page_order=page_order)
    st, _ = pool.reserve(int(kv_fill * num_pages))
    assert st == O.OK
    pool_bits = np.full((num_pages, H), 0x7FC0, dtype=np.uint16)        # NaN-poisoned
    mats = {}
    for a, r in enumerate(ranks):
        A = [_rand_bits(rng, (H, r), 1 / np.sqrt(H)) for _ in range(n_slots)]
        if a in zero_B:
            B = [np.zeros((r, H), dtype=np.uint16) for _ in range(n_slots)]
        else:
            B = [_rand_bits(rng, (r, H), 1 / np.sqrt(r)) for _ in range(n_slots)]
        st, table = pool.load(a, r, [True] * n_slots)
        assert st == O.OK
        O.place_adapter(pool_bits, table, A, B)
        mats[a] = (A, B)
    if token_adapter is None:
        token_adapter = rng.integers(0, n_ad, size=T)
        token_adapter[rng.random(T) < none_share] = -1
    token_adapter = np.asarray(token_adapter, dtype=np.int32)
    x = _rand_bits(rng, (T, H))
    Wt = [_rand_bits(rng, (H, H), 1 / np.sqrt(H)) for _ in range(n_slots)]
    return dict(pool=pool, pool_bits=pool_bits, mats=mats, ta=token_adapter, x=x, Wt=Wt, H=H)


def _f(bits):
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def pin_merged_identity(O):
    """x(W + A B) from the matrices == the unmerged forward through the pool, per token."""
    sc = build_scene(O, H=64, ranks=[8, 3, 16, 1], T=12, n_slots=2, seed=1)
    for slot in range(2):
        y, _ = O.linear_forward(sc["pool_bits"], sc["pool"].tables, sc["ta"], slot, sc["x"], sc["Wt"][slot])
        for t, a in enumerate(sc["ta"]):
            if a < 0:
                ref = _f(sc["x"][t:t + 1]) @ _f(sc["Wt"][slot]).T
            else:
                A, B = sc["mats"][int(a)]
                ref = O.merged_forward(sc["x"][t:t + 1], sc["Wt"][slot], A[slot], B[slot])
            err = np.max(np.abs(y[t] - ref[0])) / (1 + np.max(np.abs(ref)))
            if not err < 1e-12:
                return False, f"slot {slot} token {t}: merged/unmerged differ by {err:.3e}"
    return True, ""


def pin_zero_B(O):
    """An adapter with B = 0, and a token with no adapter, give exactly x W."""
    sc = build_scene(O, H=32, ranks=[4, 8], T=8, seed=2, zero_B=(1,), token_adapter=[0, 1, -1, 1, 0, -1, 1, 1])
    y, delta = O.linear_forward(sc["pool_bits"], sc["pool"].tables, sc["ta"], 0, sc["x"], sc["Wt"][0])
    base = _f(sc["x"]) @ _f(sc["Wt"][0]).T
    for t, a in enumerate(sc["ta"]):
        if a in (1, -1):
            if not (np.array_equal(y[t], base[t]) and not np.any(delta[t])):
                return False, f"token {t} (adapter {a}) is not exactly x W"
        elif not np.any(delta[t]):
            return False, f"token {t}: adapter 0 gave no delta"
    return True, ""


def pin_brute_force(O):
    """Scalar triple loops on tiny inputs (matrices, not pages) == the oracle."""
    for H, ranks, T, seed in ((16, [1, 2], 5, 3), (32, [8, 2, 1], 8, 4), (64, [8], 3, 5)):
        sc = build_scene(O, H=H, ranks=ranks, T=T, seed=seed, none_share=0.2)
        y, _ = O.linear_forward(sc["pool_bits"], sc["pool"].tables, sc["ta"], 0, sc["x"], sc["Wt"][0])
        x, Wt = _f(sc["x"]), _f(sc["Wt"][0])
        for t in range(T):
            a = int(sc["ta"][t])
            for n in range(H):
                acc = 0.0
                for k in range(H):
                    acc += x[t, k] * Wt[n, k]
                if a >= 0:
                    A, B = (_f(m[0]) for m in sc["mats"][a])
                    r = A.shape[1]
                    for j in range(r):
                        s = 0.0
                        for k in range(H):
                            s += x[t, k] * A[k, j]
                        acc += s * B[j, n]
                if abs(acc - y[t, n]) > 1e-12 * (1 + abs(acc)):
                    return False, f"H={H} t={t} n={n}: loop {acc!r} vs oracle {y[t, n]!r}"
    return True, ""


def pin_placement_invariance(O):
    """Different page permutations and KV-filler shares give bitwise the same outputs."""
    outs = []
    for order_seed, kv in ((10, 0.0), (11, 0.5), (12, 0.8)):
        sc = build_scene(O, H=64, ranks=[8, 16, 4], T=10, seed=6, page_order_seed=order_seed, kv_fill=kv)
        y, _ = O.linear_forward(sc["pool_bits"], sc["pool"].tables, sc["ta"], 0, sc["x"], sc["Wt"][0])
        outs.append(y)
    for y in outs[1:]:
        if not np.array_equal(y, outs[0]):
            return False, "output depends on page placement"
    return True, ""


def pin_batch_invariance(O):
    """Token t's output does not depend on the other tokens of the batch."""
    sc = build_scene(O, H=64, ranks=[8, 16, 4], T=16, seed=7)
    y, _ = O.linear_forward(sc["pool_bits"], sc["pool"].tables, sc["ta"], 0, sc["x"], sc["Wt"][0])
    rng = np.random.default_rng(8)
    for t in range(16):
        sub = rng.permutation(16)[:5]
        if t not in sub:
            sub[0] = t
        y2, _ = O.linear_forward(sc["pool_bits"], sc["pool"].tables, sc["ta"][sub], 0, sc["x"][sub], sc["Wt"][0])
        row = int(np.flatnonzero(sub == t)[0])
        if np.max(np.abs(y2[row] - y[t])) > 1e-12 * (1 + np.max(np.abs(y[t]))):
            return False, f"token {t} changes with batch composition"
    return True, ""


def pin_recognisable(O):
    """Adapter a's A reads coordinate c_a of x; its B writes (a+1) at column d_a.

    So token t's delta is exactly x_t[c_a] * (a + 1) at column d_a and 0
    elsewhere: it names the adapter and the pages that were used.
    """
    H, n_ad, T = 32, 5, 20
    rng = np.random.default_rng(9)
    ranks = [1, 2, 3, 2, 1]
    num_pages = 64
    pool = O.PoolModel(num_pages, 2, max_adapters=n_ad, page_order=rng.permutation(num_pages))
    pool.reserve(9)
    pool_bits = np.full((num_pages, H), 0x7FC0, dtype=np.uint16)
    one = to_bf16_bits(np.ones(1, np.float32))[0]
    spec = {}
    for a, r in enumerate(ranks):
        As, Bs = [], []
        for slot in range(2):
            c, d = (3 * a + slot) % H, (7 * a + 2 * slot + 1) % H
            A = np.zeros((H, r), np.uint16)
            A[c, 0] = one                                   # only column 0 is live
            B = np.zeros((r, H), np.uint16)
            B[0, d] = to_bf16_bits(np.array([a + 1], np.float32))[0]
            if r > 1:
                B[1:, (d + 5) % H] = to_bf16_bits(np.array([100.0], np.float32))[0]   # multiplied by s_j = 0
            As.append(A)
            Bs.append(B)
            spec[(a, slot)] = (c, d)
        st, table = pool.load(a, r, [True, True])
        O.place_adapter(pool_bits, table, As, Bs)
    ta = rng.integers(-1, n_ad, size=T).astype(np.int32)
    x = to_bf16_bits(rng.integers(-8, 9, size=(T, H)).astype(np.float32))
    Wt = np.zeros((H, H), np.uint16)
    for slot in range(2):
        _, delta = O.linear_forward(pool_bits, pool.tables, ta, slot, x, Wt)
        for t in range(T):
            want = np.zeros(H)
            a = int(ta[t])
            if a >= 0:
                c, d = spec[(a, slot)]
                want[d] = _f(x[t, c]) * (a + 1)
            if not np.array_equal(delta[t], want):
                return False, f"slot {slot} token {t}: delta does not identify adapter {a}"
    return True, ""


def pin_segments_bruteforce(O):
    """Stable grouping by adapter == an explicit bucket walk, on several batch shapes."""
    rng = np.random.default_rng(12)
    cases = [rng.integers(-1, 6, size=40), np.full(9, -1), np.arange(17)[::-1].copy(), np.full(13, 4),
             rng.integers(0, 3, size=1), np.zeros(0, dtype=np.int64)]
    for ta in cases:
        perm, off, sa = O.segments(ta)
        want_perm = [t for t in range(len(ta)) if ta[t] < 0]
        want_off, want_sa = [len(want_perm)], []
        for a in sorted(set(int(v) for v in ta if v >= 0)):
            want_perm += [t for t in range(len(ta)) if ta[t] == a]
            want_off.append(len(want_perm))
            want_sa.append(a)
        if list(perm) != want_perm or list(off) != want_off or list(sa) != want_sa:
            return False, f"segments differ for {list(ta)}"
    return True, ""


ALL_PINS = [pin_merged_identity, pin_zero_B, pin_brute_force, pin_placement_invariance,
            pin_batch_invariance, pin_recognisable, pin_segments_bruteforce]
