"""The allocation-free entry point against the ordinary one (GB300 only).

lora_linear_forward_noalloc serves callers that cannot allocate device memory: a plugin
whose host runtime owns all device memory, code recording a CUDA graph while stream capture
forbids cudaMalloc, a latency-critical loop that must not synchronise the device.  It keeps
its scratch in a static device array instead of a caller workspace.  This file checks, through
the C boundary, that two calls in a row give what lora_segments_build + lora_linear_forward
give, within the parity tolerance, and that oversized calls are refused.  It is collected
last and builds everything it needs itself, so it also passes alone in a fresh process.
"""
import numpy as np
import pytest

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


def _bf16(t):
    import oracle as O
    return O.bf16_to_f64(torch_to_bits(t))


def test_noalloc_matches_workspace_path_two_calls(L):
    import torch
    H, n_slots = 1024, 2
    wl = workloads.small(H=H, T=128, n_adapters=6, ranks=[8, 16, 32, 64, 3, 1], seed=404, n_slots=n_slots,
                         none_share=0.2)
    sc = DeviceScene(L, wl)
    calls = [(wl.token_adapter, 0, wl.x(0)), (wl.token_adapter[:77][::-1].copy(), 1, wl.x(1)[:77])]
    for ta, slot, x_bits in calls:                       # two calls in a row, different batches and slots
        T = len(ta)
        x = bits_to_torch(x_bits)
        W = bits_to_torch(wl.W(slot))
        sc.segments(ta)
        y_ref, _ = sc.forward(slot, x, W, with_delta=False)
        ta_dev = torch.from_numpy(np.asarray(ta, dtype=np.int32)).cuda()
        y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        L.lora_linear_forward_noalloc(sc.pool, ta_dev, T, slot, x, W, y)
        torch.cuda.synchronize()
        a, b = _bf16(y), _bf16(y_ref)
        assert np.all(np.abs(a - b) <= 1e-2 * (1 + np.abs(b)))
        y_or, _ = sc.oracle(ta, slot, x_bits, wl.W(slot))
        check_close(torch_to_bits(y), None, y_or, None, f"noalloc slot {slot}")
    L.lora_status(sc.pool)
    sc.close()


def test_noalloc_at_its_size_limits(L):
    """128 tokens at H = 8192, the largest call the static array is sized for, twice in a row."""
    import torch
    H, T = L.LORA_NOALLOC_MAX_H, L.LORA_NOALLOC_MAX_TOKENS
    wl = workloads.small(H=H, T=T, n_adapters=3, ranks=[64, 8, 33], seed=406, n_slots=1, none_share=0.1)
    sc = DeviceScene(L, wl)
    x = bits_to_torch(wl.x(0))
    W = bits_to_torch(wl.W(0))
    sc.segments(wl.token_adapter)
    y_ref, _ = sc.forward(0, x, W, with_delta=False)
    ta_dev = torch.from_numpy(np.asarray(wl.token_adapter, dtype=np.int32)).cuda()
    ys = []
    for _ in range(2):
        y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        L.lora_linear_forward_noalloc(sc.pool, ta_dev, T, 0, x, W, y)
        ys.append(y)
    torch.cuda.synchronize()
    b = _bf16(y_ref)
    for y in ys:
        a = _bf16(y)
        assert np.all(np.abs(a - b) <= 1e-2 * (1 + np.abs(b)))
    tokens = np.arange(0, T, 7)
    y_or, _ = sc.oracle(wl.token_adapter, 0, wl.x(0), wl.W(0), tokens=tokens)
    check_close(torch_to_bits(ys[1])[tokens], None, y_or, None, "noalloc at the limits")
    L.lora_status(sc.pool)
    sc.close()


def test_noalloc_rejects_sizes_beyond_its_limit(L):
    import torch
    wl = workloads.small(H=256, T=4, n_adapters=1, ranks=[4], seed=405)
    sc = DeviceScene(L, wl)
    T = L.LORA_NOALLOC_MAX_TOKENS + 1
    ta = torch.full((T,), -1, dtype=torch.int32, device="cuda")
    x = torch.zeros((T, 256), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(L.LoraError) as e:
        L.lora_linear_forward_noalloc(sc.pool, ta, T, 0, x, W, y)
    assert e.value.code == L.LORA_EINVAL and "limit" in e.value.message
    sc.close()
