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
