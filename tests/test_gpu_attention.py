"""Paged decode attention over KV pages of the unified pool, against the oracle (GB300 only).

The KV pages come from lora_kv_grow on a device pool (mirrored by the oracle's PoolModel.kv_grow),
their rows are written through the pages, free pages hold NaN, and lora_attention_decode's
output is compared with oracle.attention_decode, element by element, within the library's
tolerance |gpu - oracle| <= 1e-2 (1 + |oracle|)."""
import numpy as np
import pytest

import oracle as O
import workloads
from helpers import bits_to_torch, torch_to_bits

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


def _scene(L, H, layers, lengths, seed):
    import torch
    rng = np.random.default_rng(seed)
    need = 2 * layers * sum(lengths)
    num_pages = need + 64
    order = rng.permutation(num_pages)
    pool_t = torch.full((num_pages, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    pool = L.lora_pool_create(pool_t, num_pages, H, 1, 1, order)
    model = O.PoolModel(num_pages, 1, 1, order)
    opool = np.full((num_pages, H), 0x7FC0, np.uint16)
    for r, n in enumerate(lengths):
        ids = L.lora_kv_grow(pool, 100 + r, n, layers)
        st, mids = model.kv_grow(100 + r, n, layers)
        assert st == O.OK and ids == mids
        rows = workloads.to_bf16_bits(rng.standard_normal((len(ids), H)).astype(np.float32))
        opool[ids] = rows
        if ids:
            idx = torch.tensor(ids, dtype=torch.long, device="cuda")
            pool_t[idx] = bits_to_torch(rows)
    return pool, pool_t, model, opool, rng


@pytest.mark.parametrize("H,n_heads,layers,lengths", [
    (256, 2, 2, [1, 5, 0, 33, 7]),        # D = 128, an empty request, ragged lengths
    (512, 8, 1, [64, 3, 17]),            # D = 64
    (1024, 8, 3, [129, 1, 40, 2, 96, 11]),
    (2048, 16, 1, [300, 0, 1, 77]),       # two head groups
    (4096, 64, 2, [50, 3, 200]),          # D = 64, eight head groups
    (8192, 64, 1, [40, 7, 129]),          # D = 128, eight head groups
    (8192, 128, 1, [33, 5]),              # D = 64, sixteen head groups
    (640, 5, 1, [17, 9, 24]),             # a group of five heads: three warps idle
])
def test_attention_decode_matches_oracle(L, H, n_heads, layers, lengths):
    import torch
    pool, pool_t, model, opool, rng = _scene(L, H, layers, lengths, seed=H + layers)
    n_req, max_len = len(lengths), max(lengths) + 3
    table = torch.empty((n_req, max_len, layers, 2), dtype=torch.int32, device="cuda")
    seq = torch.empty(n_req, dtype=torch.int32, device="cuda")
    try:
        L.lora_kv_batch_table(pool, [100 + r for r in range(n_req)], max_len, table, seq)
        assert seq.cpu().tolist() == lengths
        q_bits = workloads.to_bf16_bits(rng.standard_normal((n_req, H)).astype(np.float32))
        for layer in range(layers):
            out = torch.empty((n_req, H), dtype=torch.bfloat16, device="cuda")
            L.lora_attention_decode(pool, n_req, table, seq, max_len, layers, layer, bits_to_torch(q_bits), out,
                                    n_heads)
            torch.cuda.synchronize()
            L.lora_status(pool)
            want = O.attention_decode(opool, [model.kv_table(100 + r, layer) for r in range(n_req)], q_bits, n_heads)
            got = O.bf16_to_f64(torch_to_bits(out))
            bad = np.abs(got - want) > 1e-2 * (1 + np.abs(want))
            assert not bad.any(), f"layer {layer}: {int(bad.sum())} elements out of tolerance"
    finally:
        L.lora_pool_destroy(pool)


@pytest.mark.parametrize("H,n_heads", [(256, 2), (8192, 128)])
def test_attention_decode_bad_page_sets_the_error_word(L, H, n_heads):
    import torch
    pool, pool_t, model, opool, rng = _scene(L, H, 1, [4], seed=5)
    table = torch.empty((1, 4, 1, 2), dtype=torch.int32, device="cuda")
    seq = torch.empty(1, dtype=torch.int32, device="cuda")
    try:
        L.lora_kv_batch_table(pool, [100], 4, table, seq)
        table[0, 2, 0, 0] = 1 << 30                        # a page id outside the pool: skipped, reported
        q_bits = workloads.to_bf16_bits(rng.standard_normal((1, H)).astype(np.float32))
        out = torch.empty((1, H), dtype=torch.bfloat16, device="cuda")
        L.lora_attention_decode(pool, 1, table, seq, 4, 1, 0, bits_to_torch(q_bits), out, n_heads)
        torch.cuda.synchronize()
        with pytest.raises(L.LoraError) as e:
            L.lora_status(pool)
        assert e.value.code == L.LORA_EDEVICE
        tab = model.kv_table(100, 0)
        want = O.attention_decode(opool, [tab[[0, 1, 3]]], q_bits, n_heads)     # the bad token left out
        got = O.bf16_to_f64(torch_to_bits(out))
        assert np.all(np.abs(got - want) <= 1e-2 * (1 + np.abs(want)))
    finally:
        L.lora_pool_destroy(pool)
