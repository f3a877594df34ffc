"""The five seeded workloads at full size, in the launch configuration the benchmark times
(one segment build, then lora_linear_forward per projection slot), checked against the
oracle on sampled outputs (GB300 only)."""
import numpy as np
import pytest

import oracle as O
import workloads
from helpers import DeviceScene, bits_to_torch, check_close, torch_to_bits

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


def _sample_tokens(wl, n, seed):
    """Random tokens plus each request's first and last token (segment edges, ragged tails)."""
    rng = np.random.default_rng(seed)
    ends = np.cumsum(wl.req_len)
    edges = np.r_[0, ends[:-1], ends - 1]
    pick = rng.choice(wl.T, size=min(n, wl.T), replace=False)
    return np.unique(np.r_[pick, edges[: 2 * n]]).astype(np.int64)


@pytest.mark.parametrize("key,slots,n_tok", [
    (2, None, None),               # all 4 slots, all 256 tokens
    (3, [0, 3], 96),
    (4, [1, 3], 160),
    (5, [0, 1, 2, 3, 82, 159], 64),
])
def test_config_full_size(L, key, slots, n_tok):
    import torch
    wl = workloads.make(key)
    check_slots = list(range(wl.n_slots)) if slots is None else slots
    sc = DeviceScene(L, wl, oracle_slots=set(check_slots), dense_oracle=False)
    sc.segments(wl.token_adapter)
    perm, off, sa = sc.read_segments()
    w = O.segments(wl.token_adapter)
    assert np.array_equal(perm, w[0]) and np.array_equal(off, w[1]) and np.array_equal(sa, w[2])
    tokens = None if n_tok is None else _sample_tokens(wl, n_tok, key)
    xs = {}
    outs = {}
    for slot in range(wl.n_slots):         # every slot runs, as in the timed step
        i = wl.slot_input(slot)
        if i not in xs:
            xs = {i: (wl.x(i), None)}
            xs[i] = (xs[i][0], bits_to_torch(xs[i][0]))
        W_bits = wl.W(slot)
        y, d = sc.forward(slot, xs[i][1], bits_to_torch(W_bits), with_delta=slot in check_slots)
        if slot in check_slots:
            outs[slot] = (torch_to_bits(y), d.cpu().numpy(), xs[i][0], W_bits)
        del y, d
    torch.cuda.synchronize()
    L.lora_status(sc.pool)
    for slot, (y_bits, d, x_bits, W_bits) in outs.items():
        y_ref, d_ref = sc.oracle(wl.token_adapter, slot, x_bits, W_bits, tokens=tokens)
        if tokens is not None:
            y_bits, d = y_bits[tokens], d[tokens]
        check_close(y_bits, d, y_ref, d_ref, f"config {key} slot {slot}")
    sc.close()
