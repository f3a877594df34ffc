"""The five seeded workloads at full size, in the launch configuration the benchmark times
(one segment build, then per layer one lora_linear_forward_group call for the q, k and v
slots, which read the same input, and one lora_linear_forward call for o), checked against
the oracle on sampled outputs (GB300 only)."""
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
    groups = wl.slot_groups()
    sc.segments(wl.token_adapter, max_group=max(len(g) for g in groups))
    perm, off, sa = sc.read_segments()
    w = O.segments(wl.token_adapter)
    assert np.array_equal(perm, w[0]) and np.array_equal(off, w[1]) and np.array_equal(sa, w[2])
    tokens = None if n_tok is None else _sample_tokens(wl, n_tok, key)
    outs = {}
    for group in groups:                   # every slot runs, as in the timed step
        x_bits = wl.x(wl.slot_input(group[0]))
        x_t = bits_to_torch(x_bits)
        W_bits = [wl.W(slot) for slot in group]
        checked = any(slot in check_slots for slot in group)
        if len(group) > 1:
            ys, ds = sc.forward_group(group, x_t, [bits_to_torch(b) for b in W_bits], with_delta=checked)
        else:
            y, d = sc.forward(group[0], x_t, bits_to_torch(W_bits[0]), with_delta=checked)
            ys, ds = [y], [d]
        for i, slot in enumerate(group):
            if slot in check_slots:
                outs[slot] = (torch_to_bits(ys[i]), ds[i].cpu().numpy(), x_bits, W_bits[i])
        del ys, ds, x_t
    torch.cuda.synchronize()
    L.lora_status(sc.pool)
    for slot, (y_bits, d, x_bits, W_bits) in outs.items():
        y_ref, d_ref = sc.oracle(wl.token_adapter, slot, x_bits, W_bits, tokens=tokens)
        if tokens is not None:
            y_bits, d = y_bits[tokens], d[tokens]
        check_close(y_bits, d, y_ref, d_ref, f"config {key} slot {slot}")
    sc.close()
