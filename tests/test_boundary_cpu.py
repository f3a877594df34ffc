"""The C boundary without a GPU: the library loads, exports every declared entry point, and
its host page bookkeeping (planning pools) matches the oracle's pool model exactly."""
import json
import os
import re
import subprocess

import numpy as np
import pytest

import oracle as O
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from adapter_gemm_lora_gb300 import build
    build.build()
    import adapter_gemm_lora_gb300 as lib
    lib.library()
    return lib


def _declared():
    text = open(os.path.join(ROOT, "include", "lora.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(L):
    declared = _declared()
    assert declared == sorted(L.EXPORTED)
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (lora_[a-z_]+)", out))
    assert set(declared) <= exported, set(declared) - exported


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "lora.h"\nint main(void){lora_pool_stats_t s; (void)s; return LORA_OK;}\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-c", str(src),
                        "-o", str(tmp_path / "t.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def _mirror_ops(L, num_pages, n_slots, max_adapters, order, ops):
    """Apply the same operations to a planning pool and to the oracle's model; compare everything."""
    pool = L.lora_pool_create(None, num_pages, 64, n_slots, max_adapters, order)
    model = O.PoolModel(num_pages, n_slots, max_adapters, order)
    try:
        for op in ops:
            kind = op[0]
            if kind == "reserve":
                st, ids = model.reserve(op[1])
                try:
                    got = L.lora_pool_reserve(pool, op[1])
                    assert st == O.OK and got.tolist() == ids
                except L.LoraError as e:
                    assert e.code == st
            elif kind == "release":
                st = model.release(op[1])
                try:
                    L.lora_pool_release(pool, op[1])
                    assert st == O.OK
                except L.LoraError as e:
                    assert e.code == st
            elif kind == "load":
                _, aid, rank, present = op
                st, tab = model.load(aid, rank, present)
                A = [np.zeros(1, np.uint16) if p else None for p in present]
                try:
                    got = L.lora_adapter_load(pool, aid, rank, A, None, n_slots, planning=True)
                    assert st == O.OK, f"library loaded, oracle said {st}"
                    assert np.array_equal(got.astype(np.int64), tab)
                except L.LoraError as e:
                    assert e.code == st, (e, st)
            elif kind == "unload":
                st = model.unload(op[1])
                try:
                    L.lora_adapter_unload(pool, op[1], planning=True)
                    assert st == O.OK
                except L.LoraError as e:
                    assert e.code == st
            s = L.lora_pool_stats(pool)
            ms = model.stats()
            assert (s["free"], s["adapter"], s["reserved"], s["resident_adapters"]) == \
                (ms["free"], ms["adapter"], ms["reserved"], ms["resident_adapters"])
    finally:
        L.lora_pool_destroy(pool)


def test_pool_matches_oracle_random_ops(L):
    rng = np.random.default_rng(5)
    n_slots, max_ad, num_pages = 3, 12, 500
    ops, reserved = [], []
    for _ in range(400):
        k = rng.integers(0, 5)
        if k == 0:
            ops.append(("reserve", int(rng.integers(0, 40))))
        elif k == 1 and ops:
            ops.append(("release", [int(v) for v in rng.choice(num_pages, size=rng.integers(1, 4), replace=False)]))
        elif k in (2, 3):
            present = [bool(v) for v in rng.random(n_slots) < 0.8]
            ops.append(("load", int(rng.integers(-1, max_ad + 1)), int(rng.integers(0, 66)), present))
        else:
            ops.append(("unload", int(rng.integers(-1, max_ad + 1))))
    _mirror_ops(L, num_pages, n_slots, max_ad, rng.permutation(num_pages), ops)


def test_release_exactly_reserved(L):
    rng = np.random.default_rng(6)
    order = rng.permutation(64)
    pool = L.lora_pool_create(None, 64, 64, 1, 4, order)
    model = O.PoolModel(64, 1, 4, order)
    ids = L.lora_pool_reserve(pool, 10)
    _, mids = model.reserve(10)
    assert ids.tolist() == mids
    with pytest.raises(L.LoraError) as e:
        L.lora_pool_release(pool, [int(ids[0]), int(ids[0])])
    assert e.value.code == L.LORA_EINVAL
    L.lora_pool_release(pool, ids[::-1])
    model.release(list(ids[::-1]))
    t = L.lora_adapter_load(pool, 0, 7, None, None, 1, planning=True)
    _, mt = model.load(0, 7, [True])
    assert np.array_equal(t.astype(np.int64), mt)
    L.lora_pool_destroy(pool)


def test_enopages_at_boundary_leaves_pool_unchanged(L):
    pool = L.lora_pool_create(None, 100, 64, 2, 8)
    L.lora_pool_reserve(pool, 36)
    L.lora_adapter_load(pool, 0, 16, None, None, 2, planning=True)        # 64 pages: exactly what is left
    before = L.lora_pool_stats(pool)
    with pytest.raises(L.LoraError) as e:
        L.lora_adapter_load(pool, 1, 1, [np.zeros(1, np.uint16), None], None, 2, planning=True)
    assert e.value.code == L.LORA_ENOPAGES
    assert L.lora_pool_stats(pool) == before
    with pytest.raises(L.LoraError) as e:
        L.lora_pool_reserve(pool, 1)
    assert e.value.code == L.LORA_ENOPAGES
    L.lora_pool_destroy(pool)


def test_worked_example_capacity_plan(L):
    """A planning pool sized like the worked example: 2,000 rank-16 adapters on q/k/v/o over
    32 layers take 2000 * 4096 pages of 4096 values (about 62 GiB at 2 bytes per value)."""
    slots = 4 * 32
    pool = L.lora_pool_create(None, 2000 * 4096, 4096, slots, 2000)
    for a in range(2000):
        L.lora_adapter_load(pool, a, 16, None, None, slots, planning=True)
    s = L.lora_pool_stats(pool)
    assert s["adapter"] == 2000 * O.PoolModel.pages_for_adapter(16, 32, 4) and s["free"] == 0
    assert abs(s["adapter"] * 4096 * 2 / 2**30 - 62.5) < 1e-9
    with pytest.raises(L.LoraError):
        L.lora_adapter_load(pool, 1999, 16, None, None, slots, planning=True)   # already loaded
    L.lora_pool_destroy(pool)


@pytest.mark.parametrize("args,code", [
    ((None, 0, 64, 1, 1), -1), ((None, 10, 63, 1, 1), -1), ((None, 10, 64, 0, 1), -1),
    ((None, 10, 64, 1, 0), -1), ((None, 10, 64, 1, 16385), -1), ((None, 10, 32768, 1, 1), -1)])
def test_pool_create_rejects_bad_geometry(L, args, code):
    with pytest.raises(L.LoraError) as e:
        L.lora_pool_create(*args)
    assert e.value.code == code and e.value.message


def test_page_order_must_be_permutation(L):
    with pytest.raises(L.LoraError):
        L.lora_pool_create(None, 4, 64, 1, 1, np.array([0, 1, 1, 3]))


def test_workload_tables_match_oracle_config2(L):
    """Placing config 2's 64 adapters after 50% KV filler gives the oracle's page tables."""
    w = workloads.make(2)
    pool = L.lora_pool_create(None, w.spec.pool_pages, w.H, w.n_slots, w.spec.n_adapters, w.page_order)
    model = O.PoolModel(w.spec.pool_pages, w.n_slots, w.spec.n_adapters, w.page_order)
    assert L.lora_pool_reserve(pool, w.kv_pages).tolist() == model.reserve(w.kv_pages)[1]
    for a in range(w.spec.n_adapters):
        t = L.lora_adapter_load(pool, a, int(w.ranks[a]), None, None, w.n_slots, planning=True)
        assert np.array_equal(t.astype(np.int64), model.load(a, int(w.ranks[a]), [True] * w.n_slots)[1])
    L.lora_pool_destroy(pool)


def test_device_calls_rejected_on_planning_pool(L):
    pool = L.lora_pool_create(None, 10, 64, 1, 1)
    seg = L.lora_segments()
    with pytest.raises(L.LoraError) as e:
        L.lora_linear_forward(pool, seg, 0, 16, 16, 32, stream=0)
    assert e.value.code == L.LORA_EINVAL
    assert L.lora_segments_size(pool, 100) > 100 * 64 * 4
    L.lora_pool_destroy(pool)


def test_group_workspace_sizes_and_argument_checks(L):
    """A group workspace holds one fp32 delta buffer and one split-K scratch area per slot; bad
    group sizes are refused."""
    H, T = 128, 300
    pool = L.lora_pool_create(None, 10, H, 4, 1)
    one = L.lora_segments_size(pool, T)
    assert L.lora_segments_size_group(pool, T, 1) == one
    # fp32 delta + split-K scratch (3 tiles of 256 tokens) + the fused tiles' s (512 bf16 per token;
    # batches of more than 256 tokens)
    per_slot = T * H * 4 + 3 * 256 * H * 4 + T * 512 * 2
    for g in (2, 3, 4):
        assert L.lora_segments_size_group(pool, T, g) - one == (g - 1) * per_slot
    for g in (0, L.LORA_MAX_GROUP + 1):
        with pytest.raises(L.LoraError) as e:
            L.lora_segments_size_group(pool, T, g)
        assert e.value.code == L.LORA_EINVAL
    seg = L.lora_segments()
    seg.delta_slots = 2
    with pytest.raises(L.LoraError) as e:                 # planning pool: no device calls
        L.lora_linear_forward_group(pool, seg, [0, 1], 16, [16, 16], [32, 48], stream=0)
    assert e.value.code == L.LORA_EINVAL
    L.lora_pool_destroy(pool)


def test_pool_lifecycle_golden_scenario_library(L):
    """The C pool's adapter lifecycle on the hand-worked scenario of the pool sketch."""
    from pool_scenario import LibraryDriver, run_golden
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "pool_lifecycle_scenario.json")))
    d = LibraryDriver(L, g["pool"]["num_pages"], g["pool"]["n_slots"], g["pool"]["max_adapters"])
    try:
        assert run_golden(d, g["steps"]) == []
    finally:
        d.close()


@pytest.mark.parametrize("seed", range(8))
def test_pool_lifecycle_matches_oracle(L, seed):
    """Random ensure / acquire / release / reserve / unload / evict sequences: statuses, page
    tables, evicted ids, active-request counts and page accounting bit-exact with the oracle."""
    from pool_scenario import LibraryDriver, OracleDriver, apply_op, random_ops
    n_pages, n_slots, n_ad = 120, 2, 12
    order = np.random.default_rng(100 + seed).permutation(n_pages)
    lib = LibraryDriver(L, n_pages, n_slots, n_ad, page_order=order)
    ora = OracleDriver(n_pages, n_slots, n_ad, page_order=order)
    try:
        res_l, res_o = [], []
        for i, op in enumerate(random_ops(seed, 400, n_ad)):
            a, b = apply_op(lib, op, res_l), apply_op(ora, op, res_o)
            assert a == b, f"op {i} {op}: library {a} vs oracle {b}"
            assert lib.stats() == ora.stats(), f"op {i} {op}"
            assert [lib.refs(k) for k in range(n_ad)] == [ora.refs(k) for k in range(n_ad)], f"op {i} {op}"
    finally:
        lib.close()


def test_pool_lifecycle_errors(L):
    pool = L.lora_pool_create(None, 64, 64, 1, 4)
    try:
        with pytest.raises(L.LoraError) as e:
            L.lora_adapter_acquire(pool, 1)
        assert e.value.code == L.LORA_EUNKNOWN_ADAPTER
        L.lora_adapter_load(pool, 1, 4, None, None, 1, planning=True)
        assert L.lora_adapter_refs(pool, 1) == 0 and L.lora_adapter_refs(pool, 2) == -1
        with pytest.raises(L.LoraError) as e:
            L.lora_adapter_release(pool, 1)                  # idle: nothing to release
        assert e.value.code == L.LORA_EINVAL
        tab, loaded, ev = L.lora_adapter_ensure(pool, 1, 4, None, None, 1, 4, planning=True)
        assert not loaded and ev == [] and L.lora_adapter_refs(pool, 1) == 1
        with pytest.raises(L.LoraError) as e:
            L.lora_adapter_ensure(pool, 1, 8, None, None, 1, 4, planning=True)   # resident with rank 4
        assert e.value.code == L.LORA_ERANK
        with pytest.raises(L.LoraError) as e:
            L.lora_adapter_unload(pool, 1, planning=True)
        assert e.value.code == L.LORA_EBUSY
        with pytest.raises(L.LoraError) as e:
            L.lora_pool_evict_idle(pool, 100, 4, planning=True)
        assert e.value.code == L.LORA_ENOPAGES
        with pytest.raises(L.LoraError) as e:
            L.lora_adapter_ensure(pool, 4, 4, None, None, 1, 4, planning=True)    # id out of range
        assert e.value.code == L.LORA_EINVAL
    finally:
        L.lora_pool_destroy(pool)


@pytest.mark.parametrize("policy", [0, 1, 2])
def test_eviction_rules_match_oracle_on_request_streams(L, policy):
    """Seeded Zipf request streams served one at a time through a pool of 24 adapters' pages:
    the C pool loads exactly the adapters the oracle loads, under each eviction rule."""
    from pool_scenario import LibraryDriver, OracleDriver
    rng = np.random.default_rng(30 + policy)
    n_ad, cap = 60, 24
    p = 1.0 / np.arange(1, n_ad + 1) ** 0.8
    stream = rng.choice(n_ad, size=400, p=p / p.sum()).tolist()
    lib = LibraryDriver(L, cap * 2, 1, n_ad)
    ora = OracleDriver(cap * 2, 1, n_ad)
    try:
        for i, a in enumerate(stream):
            fut = stream[i + 1:]
            for d in (lib, ora):
                assert d.set_eviction(policy, fut, 16 if policy == 2 else 0) == 0
            got, want = lib.ensure(a, 1), ora.ensure(a, 1)
            assert got[0] == 0 and got == want, f"request {i} ({a}): {got} vs {want}"
            assert lib.release_adapter(a) == ora.release_adapter(a) == 0
    finally:
        lib.close()


def test_set_eviction_rejects_bad_arguments(L):
    pool = L.lora_pool_create(None, 8, 64, 1, 2)
    try:
        with pytest.raises(L.LoraError) as e:
            L.lora_pool_set_eviction(pool, 3)
        assert e.value.code == L.LORA_EINVAL
    finally:
        L.lora_pool_destroy(pool)


def test_eviction_sim_tool_runs(L):
    """The capacity-planning simulation runs on the library's planning pools and reports loads
    between the number of distinct adapters requested and the number of requests."""
    from adapter_gemm_lora_gb300 import eviction_sim
    out = eviction_sim.main(["--adapters", "40", "--requests", "300", "--slots", "4", "--lookaheads", "2,0"])
    assert set(out["policies"]) == {"load_order", "lru", "farthest_k2", "farthest_full_window"}
    for rec in out["policies"].values():
        assert 0 < rec["loads_per_request"] <= 1


def test_packed_adapter_rows_follow_the_page_order(L):
    """lora_adapter_pack (host only) writes A's columns and B's rows per slot in the order the
    pool takes pages: the packed rows equal the oracle's pool read through its page table."""
    H, S, r = 128, 3, 5
    pool = L.lora_pool_create(None, 64, H, S, 2)
    try:
        rng = np.random.default_rng(12)
        A = [rng.integers(0, 2**16, size=(H, r), dtype=np.uint16), None, rng.integers(0, 2**16, size=(H, r), dtype=np.uint16)]
        B = [rng.integers(0, 2**16, size=(r, H), dtype=np.uint16), None, rng.integers(0, 2**16, size=(r, H), dtype=np.uint16)]
        present = [a is not None for a in A]
        nbytes = L.lora_adapter_packed_size(pool, r, present, S)
        need = 2 * r * 2
        header = -(-need * 4 // 256) * 256 + -(-S * 128 * 4 // 256) * 256
        assert nbytes == header + need * H * 2
        need_all = 2 * r * S                                  # every slot present
        assert L.lora_adapter_packed_size(pool, r) == \
            -(-need_all * 4 // 256) * 256 + -(-S * 128 * 4 // 256) * 256 + need_all * H * 2
        buf = np.zeros(nbytes, dtype=np.uint8)
        L.lora_adapter_pack(pool, r, A, B, buf, nbytes)
        rows = buf[header:].view(np.uint16).reshape(need, H)
        model = O.PoolModel(64, S, 2)
        st, tab = model.load(0, r, present)
        opool = np.zeros((64, H), np.uint16)
        O.place_adapter(opool, tab, A, B)
        order = [int(p) for s in range(S) for half in (0, 1) for p in tab[s, half] if p >= 0]
        assert np.array_equal(rows, opool[order])
        with pytest.raises(L.LoraError) as e:
            L.lora_adapter_pack(pool, r, A, B, buf, nbytes - 1)
        assert e.value.code == L.LORA_EINVAL
        with pytest.raises(L.LoraError) as e:                 # planning pool: no device
            L.lora_adapter_load_packed(pool, 0, r, buf, nbytes, S, present=present, copy_stream=0)
        assert e.value.code == L.LORA_EINVAL
    finally:
        L.lora_pool_destroy(pool)


def test_kv_pages_match_oracle_and_release_refuses_them(L):
    from pool_scenario import LibraryDriver, OracleDriver
    lib, ora = LibraryDriver(L, 40, 1, 4), OracleDriver(40, 1, 4)
    try:
        for d in (lib, ora):
            assert d.kv_grow(7, 2, 2) == (0, [39, 38, 37, 36, 35, 34, 33, 32])
            assert d.kv_table(7, 1) == [[37, 36], [33, 32]]
            assert d.kv_grow(7, 1, 3)[0] == O.EINVAL
            assert d.kv_grow(8, 9, 2)[0] == O.ENOPAGES        # 36 asked, 32 free
        assert L.lora_kv_length(lib.p, 7) == 2 and L.lora_kv_length(lib.p, 8) == -1
        assert lib.stats() == ora.stats()
        with pytest.raises(L.LoraError) as e:                # KV pages are not reserved pages
            L.lora_pool_release(lib.p, [39])
        assert e.value.code == L.LORA_EINVAL
        for d in (lib, ora):
            assert d.kv_free(7) == 0 and d.kv_free(7) == O.EINVAL
        assert lib.stats() == ora.stats()
    finally:
        lib.close()


def test_packing_a_large_adapter_across_threads(L):
    """An adapter above 8 MiB is repacked by several host threads; every page row is still
    column j of A or row j of B of its slot, slots in order (slots without LoRA skipped)."""
    H, S, r = 2048, 40, 32
    pool = L.lora_pool_create(None, 16, H, S, 1)
    try:
        rng = np.random.default_rng(21)
        A = [None if s % 7 == 3 else rng.integers(0, 2**16, size=(H, r), dtype=np.uint16) for s in range(S)]
        B = [None if a is None else rng.integers(0, 2**16, size=(r, H), dtype=np.uint16) for a in A]
        present = [a is not None for a in A]
        nbytes = L.lora_adapter_packed_size(pool, r, present, S)
        n_rows = 2 * r * sum(present)
        assert n_rows * H * 2 > 8 << 20
        buf = np.zeros(nbytes, dtype=np.uint8)
        L.lora_adapter_pack(pool, r, A, B, buf, nbytes)
        rows = buf[nbytes - n_rows * H * 2:].view(np.uint16).reshape(-1, 2, r, H)
        want = np.stack([np.stack([a.T, b]) for a, b in zip(A, B) if a is not None])
        assert np.array_equal(rows, want)
    finally:
        L.lora_pool_destroy(pool)


def test_noalloc_scratch_holds_a_workspace_at_its_limits(L):
    """The allocation-free entry point carves an ordinary segment workspace out of its static
    array: at its token and hidden-size limits, with the largest adapter table, the workspace
    must fit (the constants here are the header's)."""
    hdr = open(os.path.join(ROOT, "include", "lora.h")).read()
    consts = {k: int(eval(v)) for k, v in re.findall(r"#define (LORA_NOALLOC_\w+)\s+(\([^)]*\)|\d+)", hdr)}
    assert consts == {"LORA_NOALLOC_MAX_TOKENS": L.LORA_NOALLOC_MAX_TOKENS, "LORA_NOALLOC_MAX_H": L.LORA_NOALLOC_MAX_H,
                      "LORA_NOALLOC_SCRATCH_BYTES": L.LORA_NOALLOC_SCRATCH_BYTES}
    pool = L.lora_pool_create(None, 1 << 20, L.LORA_NOALLOC_MAX_H, 4, L.LORA_MAX_ADAPTERS)
    try:
        need = L.lora_segments_size(pool, L.LORA_NOALLOC_MAX_TOKENS)
        H, T = L.LORA_NOALLOC_MAX_H, L.LORA_NOALLOC_MAX_TOKENS
        # fp32 delta (T x H) and split-K partial sums (3 tiles of T columns) dominate
        assert need >= 4 * T * H + 3 * 4 * T * H
        assert need <= L.LORA_NOALLOC_SCRATCH_BYTES
    finally:
        L.lora_pool_destroy(pool)


def test_segments_struct_layout_matches_the_header(L, tmp_path):
    """The binding's ctypes mirror of lora_segments has the C struct's size and field offsets."""
    import ctypes
    fields = [f for f, _ in L.lora_segments._fields_]
    body = "".join(f'printf("%s %zu\\n", "{f}", offsetof(lora_segments, {f}));' for f in fields)
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "lora.h"\n'
                   'int main(void){' + body + 'printf("size %zu\\n", sizeof(lora_segments)); return 0;}\n')
    exe = tmp_path / "layout"
    r = subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True).stdout.splitlines())
    for f in fields:
        assert int(out[f]) == getattr(L.lora_segments, f).offset, f
    assert int(out["size"]) == ctypes.sizeof(L.lora_segments)
