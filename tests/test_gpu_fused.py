"""Prefill-shaped batches: 256-token tiles with at most 4 adapters take their LoRA term inside
the base GEMM (GB300 only, through the C boundary).

The tile plan the segment build writes is integer work and is checked bit for bit against a
plain restatement here; the outputs are checked against the oracle (y, and the LoRA term read
through delta_dbg, which the library then computes with the GEMM's own LoRA extension), and
the invariances of the unfused path are checked again on the fused one.
"""
import numpy as np
import pytest

import oracle as O
import workloads
from helpers import DeviceScene, bits_to_torch, check_close, torch_to_bits

pytestmark = pytest.mark.gpu

TILE = 256


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


def plan_reference(ta, units, perm):
    """Per 256-token tile: its distinct adapter ids ascending, or None for more than 4; the fused
    (tile, position) entries in tile order; the work units holding a token of an unfused tile."""
    n_tiles = (len(ta) + TILE - 1) // TILE
    plan = []
    for i in range(n_tiles):
        ids = sorted({int(a) for a in ta[i * TILE:(i + 1) * TILE] if a >= 0})
        plan.append(ids if len(ids) <= 4 else None)
    entries = [4 * i + b for i, ids in enumerate(plan) if ids is not None for b in range(len(ids))]
    rest = []
    for u in units:
        fused = [plan[perm[u[2] + k] // TILE] is not None for k in range(u[3])]
        if not all(fused):                 # holds a token of an unfused tile; bit 8: also fused tokens
            rest.append((u[0], u[1], u[2], u[3] | (256 if any(fused) else 0)))
    return plan, entries, rest


def read_plan(sc):
    import torch
    torch.cuda.synchronize()
    seg = sc.seg
    n_tiles = (seg.T + TILE - 1) // TILE
    raw = sc.read_i32(seg.tile_plan, 8 * n_tiles).reshape(n_tiles, 8)
    plan = [None if r[0] < 0 else [int(v) for v in r[1:1 + r[0]]] for r in raw]
    n_e = int(sc.read_i32(seg.n_entries, 1)[0])
    entries = sc.read_i32(seg.entries, n_e).tolist()
    n_r = int(sc.read_i32(seg.n_units_rest, 1)[0])
    rest = [tuple(u) for u in sc.read_i32(seg.units_rest, 4 * n_r).reshape(n_r, 4)]
    return plan, entries, rest


@pytest.mark.parametrize("case", ["prefill", "mixed", "decode_like", "ragged", "none_requests"])
def test_tile_plan_bit_exact(L, case):
    rng = np.random.default_rng(len(case))
    n_ad = 12
    ranks = [(8, 16, 32, 64, 5, 40)[a % 6] for a in range(n_ad)]
    if case == "prefill":
        wl = workloads.small_prefill(64, rng.integers(60, 700, size=9), n_ad, ranks, seed=3)
    elif case == "mixed":
        wl = workloads.small_prefill(64, [512, 300, 700], n_ad, ranks, seed=4, n_decode=300)
    elif case == "decode_like":
        wl = workloads.small(H=64, T=1500, n_adapters=n_ad, ranks=ranks, seed=5, none_share=0.1)
    elif case == "ragged":
        wl = workloads.small_prefill(64, [257, 1, 255, 3, 513], n_ad, ranks, seed=6, n_decode=7)
    else:
        wl = workloads.small_prefill(64, [400, 300, 200, 600], n_ad, ranks, seed=7, none_reqs=(1, 3))
    sc = DeviceScene(L, wl)
    sc.segments(wl.token_adapter)
    perm, _, _ = sc.read_segments()
    units = sc.read_units()
    got = read_plan(sc)
    want = plan_reference(wl.token_adapter, units, perm)
    assert got[0] == want[0], "tile plan"
    assert got[1] == want[1], "fused entries"
    assert got[2] == want[2], "units of the unfused tiles"
    if case == "decode_like":
        assert all(p is None for p in got[0]) and len(got[2]) == len(units)
    sc.close()


FUSED = [
    # H, request lengths, decode tokens in front, ranks, slots called as a group
    (2048, [700, 380, 1100, 420], 0, [8, 16, 33, 64, 1, 24], [0]),          # one slot: 176 tiles, persistent
    (2048, [300, 520, 260, 900, 640], 0, [64, 8, 16, 32], [0, 1, 2]),      # group of three slots
    (1024, [1500, 1200, 2000, 640], 300, [16, 64, 8, 40, 3], [0, 1]),     # a decode prefix: unfused tiles too
    (4096, [700, 1000], 0, [64, 16], [0, 1, 2, 3]),                       # group of four, K of 64 blocks
    (1344, [1500, 2000, 1500], 0, [16, 64, 8], [0, 1, 2]),               # 256-feature tiles, ragged last one
    (5120, [512, 512, 512, 512], 448, [8, 16, 32, 64], [0]),            # one slot, a decode prefix, 128-feature tiles
]


@pytest.mark.parametrize("H,lens,n_decode,ranks,slots", FUSED)
def test_fused_parity(L, H, lens, n_decode, ranks, slots):
    n_slots = max(slots) + 1
    wl = workloads.small_prefill(H, lens, len(ranks), ranks, seed=H + sum(lens), n_slots=n_slots,
                                 none_reqs=(1,), n_decode=n_decode)
    # the last slot carries no LoRA for odd adapters: a projection without adapter pages
    present = (lambda a: [True] * (n_slots - 1) + [a % 2 == 0]) if n_slots > 1 else None
    sc = DeviceScene(L, wl, present=present)
    sc.segments(wl.token_adapter, max_group=len(slots))
    plan, _, _ = read_plan(sc)
    assert any(p is not None for p in plan)
    x_bits = wl.x(0)
    x_t = bits_to_torch(x_bits)
    W_ts = [bits_to_torch(wl.W(s)) for s in slots]
    if len(slots) == 1:
        y, d = sc.forward(slots[0], x_t, W_ts[0])
        ys, ds = [y], [d]
    else:
        ys, ds = sc.forward_group(slots, x_t, W_ts)
    L.lora_status(sc.pool)
    tokens = np.unique(np.r_[np.arange(0, wl.T, 5), np.cumsum(wl.req_len) - 1])
    for i, slot in enumerate(slots):
        y_ref, d_ref = sc.oracle(wl.token_adapter, slot, x_bits, wl.W(slot), tokens=tokens)
        check_close(torch_to_bits(ys[i])[tokens], ds[i].cpu().numpy()[tokens], y_ref, d_ref,
                    f"fused H={H} slot {slot}")
    # without delta_dbg (the timed path): the same y
    if len(slots) == 1:
        ys2 = [sc.forward(slots[0], x_t, W_ts[0], with_delta=False)[0]]
    else:
        ys2, _ = sc.forward_group(slots, x_t, W_ts, with_delta=False)
    for i in range(len(slots)):
        assert np.array_equal(torch_to_bits(ys2[i]), torch_to_bits(ys[i]))
    sc.close()


def test_fused_group_bitwise_equals_single_slot_calls(L):
    H, slots = 2048, [0, 1, 2]
    wl = workloads.small_prefill(H, [600, 700, 480, 820], 5, [8, 64, 16, 32, 24], seed=31, n_slots=3, n_decode=40)
    sc = DeviceScene(L, wl)
    sc.segments(wl.token_adapter, max_group=3)
    x_t = bits_to_torch(wl.x(0))
    W_ts = [bits_to_torch(wl.W(s)) for s in slots]
    ys, ds = sc.forward_group(slots, x_t, W_ts)
    for i, slot in enumerate(slots):
        y1, d1 = sc.forward(slot, x_t, W_ts[i])
        assert np.array_equal(torch_to_bits(ys[i]), torch_to_bits(y1)), f"slot {slot}: y differs"
        assert np.array_equal(ds[i].cpu().numpy(), d1.cpu().numpy()), f"slot {slot}: delta differs"
    sc.close()


def _int_bits(rng, shape, lo, hi):
    return workloads.to_bf16_bits(rng.integers(lo, hi + 1, size=shape).astype(np.float32))


def test_fused_exact_small_integers_bit_exact(L):
    """Small-integer x, W, A, B on fused tiles: s is an exact small integer (hi = s, lo = 0), every
    product and sum is exact, so y and the LoRA term equal the oracle bit for bit."""
    rng = np.random.default_rng(177)
    H = 2048
    ranks = [1, 4, 8, 13, 64]
    wl = workloads.small_prefill(H, [700, 500, 900, 500], len(ranks), ranks, seed=178, none_reqs=(2,))
    T = wl.T
    x = _int_bits(rng, (T, H), -1, 1)
    W = np.zeros((H, H), np.uint16)
    W[np.arange(H), (np.arange(H) * 7) % H] = _int_bits(rng, (H,), -3, 3)
    mats = {a: (_int_bits(rng, (H, r), -1, 1) * (rng.random((H, r)) < 0.004),
                _int_bits(rng, (r, H), -2, 2) * (rng.random((r, H)) < 0.04)) for a, r in enumerate(ranks)}
    wl.A = lambda a, s: mats[a][0].astype(np.uint16)
    wl.B = lambda a, s: mats[a][1].astype(np.uint16)
    sc = DeviceScene(L, wl)
    sc.segments(wl.token_adapter)
    plan, _, _ = read_plan(sc)
    assert all(p is not None for p in plan)
    y, d = sc.forward(0, bits_to_torch(x), bits_to_torch(W))
    y_ref, d_ref = sc.oracle(wl.token_adapter, 0, x, W)
    assert np.abs(y_ref).max() <= 256 and np.array_equal(y_ref, np.round(y_ref))
    got = O.bf16_to_f64(torch_to_bits(y))
    assert np.array_equal(got, y_ref), f"{int((got != y_ref).sum())} elements differ"
    assert np.array_equal(d.cpu().numpy().astype(np.float64), d_ref)
    sc.close()


def test_fused_zero_B_adapter_bitwise_equals_no_adapter(L):
    """On fused tiles an adapter whose B is zero gives bitwise the y of no adapter (+0 and -0 equal)."""
    H = 2048
    wl = workloads.small_prefill(H, [800, 700, 600, 500], 2, [16, 64], seed=190)
    wl.B = (lambda orig: (lambda a, s: np.zeros_like(orig(a, s)) if a == 1 else orig(a, s)))(wl.B)
    sc = DeviceScene(L, wl)
    x, W = wl.x(0), wl.W(0)
    ta = np.where(np.arange(wl.T) % 3 == 0, 1, 0).astype(np.int32)
    sc.segments(ta)
    y1, _ = sc.forward(0, bits_to_torch(x), bits_to_torch(W), with_delta=False)
    sc.segments(np.where(ta == 1, -1, ta).astype(np.int32))
    y0, _ = sc.forward(0, bits_to_torch(x), bits_to_torch(W), with_delta=False)
    a, b = O.bf16_to_f64(torch_to_bits(y1)), O.bf16_to_f64(torch_to_bits(y0))
    assert np.array_equal(a, b)
    sc.close()


def test_fused_batch_composition_bitwise(L):
    """On fused tiles a token's y and LoRA term do not depend on the other tokens: the same
    requests in another order (other tile neighbours, other tile slots) give the same bits."""
    H = 2048
    lens = [300, 700, 450, 380, 900]
    wl = workloads.small_prefill(H, lens, 5, [8, 64, 16, 33, 24], seed=200, none_reqs=(3,))
    sc = DeviceScene(L, wl)
    x, W = wl.x(0), wl.W(0)
    sc.segments(wl.token_adapter)
    y_a, d_a = sc.forward(0, bits_to_torch(x), bits_to_torch(W))
    starts = np.r_[0, np.cumsum(lens)[:-1]]
    order = [4, 2, 0, 3, 1]
    idx = np.concatenate([np.arange(starts[r], starts[r] + lens[r]) for r in order])
    sc.segments(wl.token_adapter[idx])
    plan, _, _ = read_plan(sc)
    assert all(p is not None for p in plan)
    y_b, d_b = sc.forward(0, bits_to_torch(x[idx]), bits_to_torch(W))
    assert np.array_equal(torch_to_bits(y_b), torch_to_bits(y_a)[idx])
    assert np.array_equal(d_b.cpu().numpy(), d_a.cpu().numpy()[idx])
    sc.close()
