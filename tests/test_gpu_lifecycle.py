"""The unified pool's adapter lifecycle on a device pool, through the C boundary (GB300 only).

"S-LoRA, in depth", "Unified paging": adapters and KV cache share one free list; an adapter with
no active request left can be evicted and its pages reused.  Adapters here become resident by
lora_adapter_ensure; one is released and evicted while a batch that uses it is still queued on
the stream; a new adapter is loaded into the reclaimed pages.  Every output is checked against
the oracle, whose pool follows its own bookkeeping (PoolModel.ensure / evict) and placement."""
import numpy as np
import pytest

import oracle as O
import workloads
from helpers import bits_to_torch, check_close, torch_to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from adapter_gemm_lora_gb300 import build
    build.build()
    import adapter_gemm_lora_gb300 as lib
    lib.library()
    return lib


def test_evict_and_reload_in_stream_order(L):
    import torch
    H, T, n_ad = 256, 96, 6
    ranks = [8, 16, 64, 4, 32, 8]
    wl = workloads.small(H=H, T=T, n_adapters=n_ad, ranks=ranks, seed=321, kv_fill=0.0)
    num_pages = 200                                  # room for adapters 0..3 (184 pages), not more
    order = np.random.default_rng(5).permutation(num_pages)
    pool_t = torch.full((num_pages, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    pool = L.lora_pool_create(pool_t, num_pages, H, 1, n_ad, order)
    model = O.PoolModel(num_pages, 1, n_ad, order)
    opool = np.full((num_pages, H), 0x7FC0, np.uint16)
    x, W = wl.x(0), wl.W(0)
    x_t, W_t = bits_to_torch(x), bits_to_torch(W)
    rng = np.random.default_rng(9)

    def ensure(a):
        A, B = [wl.A(a, 0)], [wl.B(a, 0)]
        tab, loaded, ev = L.lora_adapter_ensure(pool, a, ranks[a], A, B, 1, n_ad)
        st, mtab, mloaded, mev = model.ensure(a, ranks[a], [True])
        assert st == O.OK and loaded == mloaded and ev == list(mev)
        assert np.array_equal(tab.astype(np.int64), mtab), f"page table of adapter {a}"
        if loaded:
            O.place_adapter(opool, mtab, A, B)
        return ev

    def batch(ids):
        ta = rng.choice(np.array(ids, dtype=np.int32), size=T).astype(np.int32)
        nbytes = L.lora_segments_size(pool, T)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        seg = L.lora_segments_init(pool, ws, nbytes, T)
        ta_t = torch.from_numpy(ta).cuda()
        L.lora_segments_build(pool, ta_t, T, seg)
        y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        d = torch.empty((T, H), dtype=torch.float32, device="cuda")
        L.lora_linear_forward(pool, seg, 0, x_t, W_t, y, d)
        return ta, (ws, ta_t, seg), y, d

    try:
        for a in range(4):
            assert ensure(a) == []
        # batch 1 (adapters 0..3) is queued; its oracle reference is taken before any page changes
        ta1, keep1, y1, d1 = batch([-1, 0, 1, 2, 3])
        ref1 = O.linear_forward(opool, {k: v.copy() for k, v in model.tables.items()}, ta1, 0, x, W)
        # adapter 2's requests end; adapter 4 needs 64 pages with 16 free: adapter 2 (128 pages, the
        # only idle one) is evicted and adapter 4 is written into its pages, all behind batch 1
        pages2 = set(model.tables[2].reshape(-1).tolist())
        L.lora_adapter_release(pool, 2)
        assert model.release_adapter(2) == O.OK
        assert ensure(4) == [2]
        assert set(model.tables[4].reshape(-1).tolist()) <= pages2      # adapter 4 sits in adapter 2's pages
        torch.cuda.synchronize()
        L.lora_status(pool)
        check_close(torch_to_bits(y1), d1.cpu().numpy(), ref1[0], ref1[1], "batch queued before the eviction")
        # batch 2 uses the new adapter
        ta2, keep2, y2, d2 = batch([-1, 0, 1, 3, 4])
        torch.cuda.synchronize()
        L.lora_status(pool)
        ref2 = O.linear_forward(opool, model.tables, ta2, 0, x, W)
        check_close(torch_to_bits(y2), d2.cpu().numpy(), ref2[0], ref2[1], "adapter in reclaimed pages")
        # batch 3 still names the evicted adapter: device error, and those tokens get no delta
        ta3, keep3, y3, d3 = batch([0, 2, 4])
        torch.cuda.synchronize()
        with pytest.raises(L.LoraError) as e:
            L.lora_status(pool)
        assert e.value.code == L.LORA_EDEVICE
        ref3 = O.linear_forward(opool, model.tables, np.where(ta3 == 2, -1, ta3), 0, x, W)
        check_close(torch_to_bits(y3), d3.cpu().numpy(), ref3[0], ref3[1], "evicted adapter treated as none")
        s = L.lora_pool_stats(pool)
        ms = model.stats()
        assert (s["free"], s["adapter"], s["resident_adapters"]) == (ms["free"], ms["adapter"], ms["resident_adapters"])
        assert [L.lora_adapter_refs(pool, a) for a in range(n_ad)] == [model.refs.get(a, -1) for a in range(n_ad)]
    finally:
        L.lora_pool_destroy(pool)


def test_packed_loads_on_a_copy_stream(L):
    """Adapters packed into pinned host memory and loaded on a copy stream ("Scheduling":
    prefetch on a separate stream from pinned memory) give the same pages, page contents and
    outputs, bit for bit, as synchronous loads; a packed load into the pages of an adapter just
    unloaded behind a queued batch leaves that batch's result intact."""
    import torch
    H, T, S = 512, 80, 2
    ranks = [8, 64, 16, 3, 32, 40]
    n_ad = len(ranks)
    wl = workloads.small(H=H, T=T, n_adapters=n_ad, ranks=ranks, seed=77, n_slots=S, kv_fill=0.0)
    present = {a: [True, a % 2 == 0] for a in range(n_ad)}          # odd adapters carry no LoRA on slot 1
    pages = {a: 2 * ranks[a] * sum(present[a]) for a in range(n_ad)}
    num_pages = sum(pages[a] for a in range(5)) + 8
    order = np.random.default_rng(78).permutation(num_pages)
    pool_ts = [torch.full((num_pages, H), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    p_sync = L.lora_pool_create(pool_ts[0], num_pages, H, S, n_ad, order)
    p_pack = L.lora_pool_create(pool_ts[1], num_pages, H, S, n_ad, order)
    model = O.PoolModel(num_pages, S, n_ad, order)
    opool = np.full((num_pages, H), 0x7FC0, np.uint16)
    copy = torch.cuda.Stream()
    bufs = {}

    def factors(a):
        return ([wl.A(a, s) if present[a][s] else None for s in range(S)],
                [wl.B(a, s) if present[a][s] else None for s in range(S)])

    def load_packed(a):
        A, B = factors(a)
        nbytes = L.lora_adapter_packed_size(p_pack, ranks[a], present[a], S)
        buf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        L.lora_adapter_pack(p_pack, ranks[a], A, B, buf, nbytes)
        bufs[a] = buf                                   # kept until the copy stream has passed the load
        tab = L.lora_adapter_load_packed(p_pack, a, ranks[a], buf, nbytes, S, present=present[a], copy_stream=copy)
        st, mtab = model.load(a, ranks[a], present[a])
        assert st == O.OK and np.array_equal(tab.astype(np.int64), mtab), f"page table of adapter {a}"
        O.place_adapter(opool, mtab, A, B)

    def forward(pool, ta, slot):
        nbytes = L.lora_segments_size(pool, T)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        seg = L.lora_segments_init(pool, ws, nbytes, T)
        ta_t = torch.from_numpy(ta).cuda()
        L.lora_segments_build(pool, ta_t, T, seg)
        y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        d = torch.empty((T, H), dtype=torch.float32, device="cuda")
        L.lora_linear_forward(pool, seg, slot, bits_to_torch(wl.x(slot)), bits_to_torch(wl.W(slot)), y, d)
        return y, d, (ws, ta_t)

    try:
        for a in range(5):
            A, B = factors(a)
            L.lora_adapter_load(p_sync, a, ranks[a], A, B, S)
            load_packed(a)
        cur = torch.cuda.current_stream()
        for a in range(5):
            L.lora_adapter_wait(p_pack, a, cur)
        rng = np.random.default_rng(79)
        ta = rng.choice(np.array([-1, 0, 1, 2, 3, 4], dtype=np.int32), size=T).astype(np.int32)
        for slot in range(S):
            ys, ds, _ = forward(p_sync, ta, slot)
            yp, dp, _ = forward(p_pack, ta, slot)
            torch.cuda.synchronize()
            assert np.array_equal(torch_to_bits(ys), torch_to_bits(yp)), f"slot {slot}: y differs"
            assert np.array_equal(ds.cpu().numpy(), dp.cpu().numpy()), f"slot {slot}: delta differs"
            ref = O.linear_forward(opool, model.tables, ta, slot, wl.x(slot), wl.W(slot))
            check_close(torch_to_bits(yp), dp.cpu().numpy(), ref[0], ref[1], f"packed loads, slot {slot}")
        used = np.array(sorted(p for t in model.tables.values() for p in t.reshape(-1) if p >= 0))
        assert torch.equal(pool_ts[0][used], pool_ts[1][used])
        # a batch that uses adapter 1 is queued; adapter 1 is unloaded behind it and adapter 5 is
        # loaded into its pages on the copy stream
        tb = rng.choice(np.array([0, 1, 2], dtype=np.int32), size=T).astype(np.int32)
        yb, db, keep = forward(p_pack, tb, 0)
        refb = O.linear_forward(opool, {k: v.copy() for k, v in model.tables.items()}, tb, 0, wl.x(0), wl.W(0))
        pages1 = set(model.tables[1].reshape(-1).tolist()) - {-1}
        L.lora_adapter_unload(p_pack, 1)
        assert model.unload(1) == O.OK
        load_packed(5)
        assert set(model.tables[5].reshape(-1).tolist()) - {-1} <= pages1
        torch.cuda.synchronize()
        L.lora_status(p_pack)
        check_close(torch_to_bits(yb), db.cpu().numpy(), refb[0], refb[1], "batch queued before the page reuse")
        L.lora_adapter_wait(p_pack, 5, cur)
        tc = rng.choice(np.array([-1, 0, 5], dtype=np.int32), size=T).astype(np.int32)
        yc, dc, _ = forward(p_pack, tc, 0)
        torch.cuda.synchronize()
        refc = O.linear_forward(opool, model.tables, tc, 0, wl.x(0), wl.W(0))
        check_close(torch_to_bits(yc), dc.cpu().numpy(), refc[0], refc[1], "adapter packed into reclaimed pages")
        L.lora_status(p_pack)
    finally:
        L.lora_pool_destroy(p_sync)
        L.lora_pool_destroy(p_pack)
