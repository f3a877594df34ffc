"""CUDA path vs the oracle, element by element, through the C boundary (GB300 only)."""
import zlib

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


def _run_slot(sc, ta, slot, x_bits, W_bits, tokens=None):
    x_t, W_t = bits_to_torch(x_bits), bits_to_torch(W_bits)
    y, d = sc.forward(slot, x_t, W_t)
    y_bits, d_np = torch_to_bits(y), d.cpu().numpy()
    y_ref, d_ref = sc.oracle(ta, slot, x_bits, W_bits, tokens=tokens)
    if tokens is not None:
        y_bits, d_np = y_bits[tokens], d_np[tokens]
    return y_bits, d_np, y_ref, d_ref


# ---------------------------------------------------------------------------- segments
@pytest.mark.parametrize("case", ["random", "all_none", "all_distinct", "single", "one_token", "empty", "long",
                                  "chunk_exact", "chunk_plus_one"])
def test_segments_bit_exact(L, case):
    rng = np.random.default_rng(zlib.crc32(case.encode()))
    n_ad = 40
    ta = {"random": lambda: rng.integers(-1, n_ad, size=777),
          "all_none": lambda: np.full(100, -1),
          "all_distinct": lambda: rng.permutation(n_ad),
          "single": lambda: np.full(300, 7),
          "one_token": lambda: np.array([5]),
          "empty": lambda: np.zeros(0, dtype=np.int64),
          "long": lambda: rng.integers(-1, n_ad, size=5000),
          # the build handles 1,024 tokens per chunk and keeps the first chunk's keys in registers
          "chunk_exact": lambda: rng.integers(-1, n_ad, size=1024),
          "chunk_plus_one": lambda: rng.integers(-1, n_ad, size=1025)}[case]().astype(np.int32)
    ranks = [(3, 12, 24, 64, 8, 40, 17, 9)[a % 8] for a in range(n_ad)]     # every rank class
    wl = workloads.small(H=64, T=max(len(ta), 1), n_adapters=n_ad, ranks=ranks, seed=1)
    sc = DeviceScene(L, wl)
    sc.segments(ta)
    perm, off, sa = sc.read_segments()
    w_perm, w_off, w_sa = O.segments(ta)
    assert np.array_equal(perm, w_perm)
    assert np.array_equal(off, w_off)
    assert np.array_equal(sa, w_sa)
    # the work list: every segment cut into runs of <= 16 tokens, listed by rank class
    # (33..64, 17..32, 9..16, 1..8), then adapter id, then offset
    want = []
    for s in range(len(w_sa)):
        a, lo, hi = int(w_sa[s]), int(w_off[s]), int(w_off[s + 1])
        r = int(wl.ranks[a])
        cls = 0 if r > 32 else 1 if r > 16 else 2 if r > 8 else 3
        want += [(cls, a, b, r, min(16, hi - b)) for b in range(lo, hi, 16)]
    want = np.array([(a, r, b, n) for _, a, b, r, n in sorted(want)], dtype=np.int32).reshape(-1, 4)
    assert np.array_equal(sc.read_units(), want)
    L.lora_status(sc.pool)
    sc.close()


def test_segments_at_the_adapter_id_limit_after_a_small_pool(L):
    """The segment build keys its shared-memory histogram by adapter id, so a pool with
    max_adapters = LORA_MAX_ADAPTERS needs 2 x 16,385 int32 of dynamic shared memory: a build on a
    small pool first, then one on a pool at the limit (ids up to 16,383), both bit-exact."""
    for n_ad, loaded in ((40, [0, 3, 39]), (L.LORA_MAX_ADAPTERS, [0, 7, 5000, L.LORA_MAX_ADAPTERS - 1])):
        rng = np.random.default_rng(n_ad)
        wl = workloads.small(H=64, T=600, n_adapters=n_ad, ranks=[8] * n_ad, seed=9)
        sc = DeviceScene(L, wl, adapters=loaded)
        ta = rng.choice(np.array(loaded + [-1], dtype=np.int32), size=600)
        sc.segments(ta)
        perm, off, sa = sc.read_segments()
        w_perm, w_off, w_sa = O.segments(ta)
        assert np.array_equal(perm, w_perm) and np.array_equal(off, w_off) and np.array_equal(sa, w_sa)
        L.lora_status(sc.pool)
        sc.close()


def test_unknown_adapter_raises_device_error_and_is_treated_as_none(L):
    wl = workloads.small(H=128, T=16, n_adapters=4, ranks=[4, 8, 2, 16], seed=3)
    sc = DeviceScene(L, wl, adapters=[0, 1, 3])          # adapter 2 never loaded
    ta = np.array([0, 2, 1, 3, -1, 2, 0, 1, 3, 3, -1, 0, 1, 2, 0, 3], dtype=np.int32)
    sc.segments(ta)
    with pytest.raises(L.LoraError) as e:
        L.lora_status(sc.pool)
    assert e.value.code == L.LORA_EDEVICE and "unknown adapter" in e.value.message
    ta_eff = np.where(ta == 2, -1, ta)
    perm, off, sa = sc.read_segments()
    w = O.segments(ta_eff)
    assert np.array_equal(perm, w[0]) and np.array_equal(off, w[1]) and np.array_equal(sa, w[2])
    x, W = wl.x(0), wl.W(0)
    y, d, y_ref, d_ref = _run_slot(sc, ta_eff, 0, x, W)
    check_close(y, d, y_ref, d_ref, "unknown->none")
    L.lora_status(sc.pool)                               # cleared by the previous read
    sc.close()


def test_out_of_range_adapter_ids_are_flagged_and_treated_as_none(L):
    """Ids below -1 or at and above max_adapters: the error word is raised, the tokens take no
    LoRA term, and the segments are those of the batch with those ids replaced by -1 (in the
    first 1,024-token chunk and after it)."""
    wl = workloads.small(H=128, T=1100, n_adapters=4, ranks=[4, 8, 2, 16], seed=5)
    sc = DeviceScene(L, wl)
    rng = np.random.default_rng(17)
    ta = rng.integers(-1, 4, size=1100).astype(np.int32)
    bad = np.array([3, 100, 517, 1023, 1024, 1099])
    ta[bad] = np.array([4, -2, 1 << 30, -(1 << 31), 5, 4], dtype=np.int32)
    sc.segments(ta)
    with pytest.raises(L.LoraError) as e:
        L.lora_status(sc.pool)
    assert e.value.code == L.LORA_EDEVICE and "unknown adapter" in e.value.message
    ta_eff = ta.copy()
    ta_eff[bad] = -1
    perm, off, sa = sc.read_segments()
    w = O.segments(ta_eff)
    assert np.array_equal(perm, w[0]) and np.array_equal(off, w[1]) and np.array_equal(sa, w[2])
    L.lora_status(sc.pool)
    sc.close()


# ---------------------------------------------------------------------------- small parity
SMALL = [
    # H, T, ranks, n_slots, none_share
    (64, 1, [1], 1, 0.0),
    (64, 7, [1, 2, 8], 1, 0.2),
    (128, 33, [8, 16, 64, 3], 2, 0.25),
    (192, 100, [64, 64, 5], 1, 0.1),
    (256, 32, [8, 8, 16, 16], 1, 0.0),
    (256, 257, [8, 16, 32, 64, 1, 7], 3, 0.3),
    (384, 300, [16, 40], 1, 0.5),
    (512, 520, [64, 8, 33, 17, 2, 9, 12, 63], 2, 0.15),
    (1024, 96, [32, 64, 8, 16], 4, 0.2),
    (2048, 256, [64, 8, 16, 32, 1], 1, 0.2),     # base GEMM splits K over a cluster of 4
    (1216, 64, [16, 64, 3], 2, 0.3),            # uneven 2-way K split, ragged last feature tile
    (2048, 2600, [16, 64, 8, 32], 1, 0.2),      # persistent GEMM, 176 tiles, ragged last token tile
    (1024, 9700, [8, 16, 64], 1, 0.1),          # persistent GEMM, 304 tiles over two waves
]


@pytest.mark.parametrize("H,T,ranks,n_slots,none_share", SMALL)
def test_small_parity(L, H, T, ranks, n_slots, none_share):
    wl = workloads.small(H=H, T=T, n_adapters=len(ranks), ranks=ranks, seed=H + T, n_slots=n_slots,
                         none_share=none_share)
    # the last slot carries no LoRA for odd adapters: a projection without adapter pages
    present = (lambda a: [True] * (n_slots - 1) + [a % 2 == 0]) if n_slots > 1 else None
    sc = DeviceScene(L, wl, present=present)
    sc.segments(wl.token_adapter)
    for slot in range(n_slots):
        y, d, y_ref, d_ref = _run_slot(sc, wl.token_adapter, slot, wl.x(slot % 2), wl.W(slot))
        check_close(y, d, y_ref, d_ref, f"H={H} T={T} slot={slot}")
    L.lora_status(sc.pool)
    sc.close()


GROUP = [
    # H, T, ranks, n_slots, none_share, slots of the group call
    (256, 257, [8, 16, 32, 64, 1, 7], 4, 0.3, [2, 0, 3]),
    (2048, 256, [64, 8, 16, 32, 1], 4, 0.2, [0, 1, 2]),      # decode shape: split-K base GEMM
    (512, 33, [3, 64], 4, 0.0, [3, 1, 0, 2]),
    (1024, 1, [16], 2, 0.0, [1]),
    (384, 700, [8, 40, 64, 17], 3, 0.25, [1, 2]),            # several units per adapter
    (384, 100, [8, 64, 5], 3, 0.3, [0, 2, 1]),               # K split over 2 CTAs (6 blocks of 64)
    (4096, 200, [64, 32, 16, 8, 64, 16], 4, 0.1, [0, 1, 2]),  # 96 tiles: several per cluster
    (1024, 2600, [16, 64, 8, 33], 3, 0.2, [0, 1, 2]),         # persistent group vs single-tile launches
    (1344, 5000, [16, 64, 8], 3, 0.2, [0, 1, 2]),             # 256-feature tiles, the last one 64 features
    (512, 700, [8, 64, 24], 2, 0.25, [1, 0]),                 # persistent group, 32-token tiles, 4 K chunks a stage
    (192, 100, [8, 16, 64], 3, 0.2, [2, 0, 1]),               # K of 3 blocks: no split, persistent group
]


@pytest.mark.parametrize("H,T,ranks,n_slots,none_share,slots", GROUP)
def test_group_forward_bitwise_equals_single_slot_calls(L, H, T, ranks, n_slots, none_share, slots):
    """Slots that share x in one lora_linear_forward_group call give bit for bit what one
    lora_linear_forward call per slot gives, and both meet the oracle's tolerance.  Batches of
    <= 256 tokens take the grouped persistent split-K GEMM there and the single-slot split-K
    GEMM here; larger batches one persistent launch over every slot's tiles there."""
    wl = workloads.small(H=H, T=T, n_adapters=len(ranks), ranks=ranks, seed=7 * H + T, n_slots=n_slots,
                         none_share=none_share)
    present = (lambda a: [True] * (n_slots - 1) + [a % 2 == 0]) if n_slots > 1 else None
    sc = DeviceScene(L, wl, present=present)
    sc.segments(wl.token_adapter, max_group=len(slots))
    x_bits = wl.x(0)
    x_t = bits_to_torch(x_bits)
    W_ts = [bits_to_torch(wl.W(s)) for s in slots]
    for _ in range(2):                                    # the second call reuses the scratch
        ys, ds = sc.forward_group(slots, x_t, W_ts)
    for i, slot in enumerate(slots):
        y1, d1 = sc.forward(slot, x_t, W_ts[i])
        assert np.array_equal(torch_to_bits(ys[i]), torch_to_bits(y1)), f"slot {slot}: y differs from a single call"
        assert np.array_equal(ds[i].cpu().numpy().view(np.uint32), d1.cpu().numpy().view(np.uint32)), \
            f"slot {slot}: delta differs from a single call"
        y_ref, d_ref = sc.oracle(wl.token_adapter, slot, x_bits, wl.W(slot))
        check_close(torch_to_bits(ys[i]), ds[i].cpu().numpy(), y_ref, d_ref, f"group H={H} T={T} slot={slot}")
    # without delta_dbg the deltas live in the workspace's scratch: same outputs
    ys2, _ = sc.forward_group(slots, x_t, W_ts, with_delta=False)
    for i in range(len(slots)):
        assert np.array_equal(torch_to_bits(ys2[i]), torch_to_bits(ys[i]))
    L.lora_status(sc.pool)
    sc.close()


def test_group_forward_argument_errors(L):
    import torch
    wl = workloads.small(H=64, T=4, n_adapters=1, ranks=[2], seed=83, n_slots=3)
    sc = DeviceScene(L, wl)
    sc.segments(wl.token_adapter, max_group=2)
    x = bits_to_torch(wl.x(0))
    W = bits_to_torch(wl.W(0))
    y = [torch.empty_like(x) for _ in range(3)]
    cases = [([0, 1, 2], [W] * 3, y),                    # more slots than the workspace's delta scratch
             ([1, 1], [W] * 2, y[:2]),                    # a slot listed twice
             ([0, 3], [W] * 2, y[:2]),                    # slot out of range
             ([0, 1], [W] * 2, [y[0], y[0]]),             # two slots share one y
             ([0, 1], [W] * 2, [y[0], x])]                # y aliases x
    for slots, Ws, ys in cases:
        with pytest.raises(L.LoraError) as e:
            L.lora_linear_forward_group(sc.pool, sc.seg, slots, x, Ws, ys)
        assert e.value.code == L.LORA_EINVAL, slots
    sc.close()


def test_config1_all_tokens(L):
    wl = workloads.make(1)
    sc = DeviceScene(L, wl)
    sc.segments(wl.token_adapter)
    perm, off, sa = sc.read_segments()
    w = O.segments(wl.token_adapter)
    assert np.array_equal(perm, w[0]) and np.array_equal(off, w[1]) and np.array_equal(sa, w[2])
    y, d, y_ref, d_ref = _run_slot(sc, wl.token_adapter, 0, wl.x(0), wl.W(0))
    check_close(y, d, y_ref, d_ref, "config 1")
    L.lora_status(sc.pool)
    sc.close()


# ---------------------------------------------------------------------------- exact cases
def _int_bits(rng, shape, lo, hi):
    from workloads import to_bf16_bits
    return to_bf16_bits(rng.integers(lo, hi + 1, size=shape).astype(np.float32))


def test_exact_small_integers_bit_exact(L):
    """Small-integer x, W, A, B: every product and partial sum is exact in fp32 and the
    result fits bf16 exactly, so the GPU must equal the oracle bit for bit."""
    import torch
    rng = np.random.default_rng(77)
    H, T, n_ad = 256, 70, 5
    ranks = [1, 4, 8, 13, 64]
    wl = workloads.small(H=H, T=T, n_adapters=n_ad, ranks=ranks, seed=78, none_share=0.2)
    x = _int_bits(rng, (T, H), -1, 1)
    W = np.zeros((H, H), np.uint16)
    W[np.arange(H), (np.arange(H) * 7) % H] = _int_bits(rng, (H,), -3, 3)    # one non-zero per row
    mats = {a: (_int_bits(rng, (H, r), -1, 1) * (rng.random((H, r)) < 0.05),
                _int_bits(rng, (r, H), -2, 2) * (rng.random((r, H)) < 0.25)) for a, r in enumerate(ranks)}
    wl.A = lambda a, s: mats[a][0].astype(np.uint16)
    wl.B = lambda a, s: mats[a][1].astype(np.uint16)
    sc = DeviceScene(L, wl)
    sc.segments(wl.token_adapter)
    y, d = sc.forward(0, bits_to_torch(x), bits_to_torch(W))
    y_ref, d_ref = sc.oracle(wl.token_adapter, 0, x, W)
    assert np.abs(y_ref).max() <= 256 and np.array_equal(y_ref, np.round(y_ref))
    got = O.bf16_to_f64(torch_to_bits(y))
    assert np.array_equal(got, y_ref), f"{int((got != y_ref).sum())} elements differ"
    assert np.array_equal(d.cpu().numpy().astype(np.float64), d_ref)
    sc.close()


def test_zero_B_adapter_bitwise_equals_no_adapter(L):
    """An adapter whose B is zero gives bitwise the same y as no adapter (+0 and -0 equal)."""
    H, T = 512, 64
    wl = workloads.small(H=H, T=T, n_adapters=2, ranks=[16, 32], seed=90, none_share=0.0)
    wl.B = (lambda orig: (lambda a, s: np.zeros_like(orig(a, s)) if a == 1 else orig(a, s)))(wl.B)
    sc = DeviceScene(L, wl)
    x, W = wl.x(0), wl.W(0)
    ta = np.where(np.arange(T) % 2 == 0, 1, 0).astype(np.int32)
    sc.segments(ta)
    y1, _ = sc.forward(0, bits_to_torch(x), bits_to_torch(W))
    sc.segments(np.where(ta == 1, -1, ta).astype(np.int32))
    y0, _ = sc.forward(0, bits_to_torch(x), bits_to_torch(W))
    a, b = O.bf16_to_f64(torch_to_bits(y1)), O.bf16_to_f64(torch_to_bits(y0))
    assert np.array_equal(a, b)
    y_ref, _ = sc.oracle(ta, 0, x, W)
    check_close(torch_to_bits(y1), None, y_ref, None, "B=0")
    sc.close()


def test_placement_invariance_bitwise(L):
    """Different page permutations and KV-filler shares give bitwise identical outputs."""
    outs = []
    for order_seed, kv in ((1, 0.0), (2, 0.5), (3, 0.9)):
        wl = workloads.small(H=256, T=50, n_adapters=6, ranks=[8, 16, 32, 64, 3, 1], seed=55, kv_fill=kv,
                             none_share=0.1)
        wl.page_order = np.random.default_rng(order_seed).permutation(wl.spec.pool_pages)
        sc = DeviceScene(L, wl)
        sc.segments(wl.token_adapter)
        y, d = sc.forward(0, bits_to_torch(wl.x(0)), bits_to_torch(wl.W(0)))
        outs.append((torch_to_bits(y), d.cpu().numpy()))
        sc.close()
    for y, d in outs[1:]:
        assert np.array_equal(y, outs[0][0]) and np.array_equal(d, outs[0][1])


def test_batch_composition(L):
    """A token's output does not depend on the other tokens: bitwise for the LoRA delta,
    within tolerance for y (the base GEMM's tile shape follows T)."""
    H = 256
    wl = workloads.small(H=H, T=200, n_adapters=5, ranks=[8, 16, 32, 64, 4], seed=60, none_share=0.2)
    sc = DeviceScene(L, wl)
    x, W = wl.x(0), wl.W(0)
    sc.segments(wl.token_adapter)
    y_all, d_all = sc.forward(0, bits_to_torch(x), bits_to_torch(W))
    y_all, d_all = O.bf16_to_f64(torch_to_bits(y_all)), d_all.cpu().numpy()
    sub = np.random.default_rng(61).choice(200, size=37, replace=False)
    sc.segments(wl.token_adapter[sub])
    y_s, d_s = sc.forward(0, bits_to_torch(x[sub]), bits_to_torch(W))
    assert np.array_equal(d_s.cpu().numpy(), d_all[sub])
    y_s = O.bf16_to_f64(torch_to_bits(y_s))
    assert np.all(np.abs(y_s - y_all[sub]) <= 1e-2 * (1 + np.abs(y_all[sub])))
    sc.close()


def test_reruns_bitwise_identical(L):
    wl = workloads.make(1)
    sc = DeviceScene(L, wl)
    sc.segments(wl.token_adapter)
    x_t, W_t = bits_to_torch(wl.x(0)), bits_to_torch(wl.W(0))
    runs = [sc.forward(0, x_t, W_t) for _ in range(3)]
    for y, d in runs[1:]:
        assert np.array_equal(torch_to_bits(y), torch_to_bits(runs[0][0]))
        assert np.array_equal(d.cpu().numpy(), runs[0][1].cpu().numpy())
    sc.close()


def test_recognisable_adapters_on_gpu(L):
    """Each adapter's A reads one coordinate of x and its B writes (a+1) at one column:
    every token's delta names the adapter whose pages were used."""
    H, T, n_ad = 128, 40, 7
    wl = workloads.small(H=H, T=T, n_adapters=n_ad, ranks=[1, 2, 3, 4, 5, 6, 7], seed=70, none_share=0.2, n_slots=2)
    from workloads import to_bf16_bits
    one = to_bf16_bits(np.ones(1, np.float32))[0]

    def A(a, s):
        m = np.zeros((H, int(wl.ranks[a])), np.uint16)
        m[(5 * a + s) % H, 0] = one
        return m

    def B(a, s):
        m = np.zeros((int(wl.ranks[a]), H), np.uint16)
        m[0, (11 * a + 3 * s + 1) % H] = to_bf16_bits(np.array([a + 1], np.float32))[0]
        return m
    wl.A, wl.B = A, B
    sc = DeviceScene(L, wl)
    sc.segments(wl.token_adapter)
    x = wl.x(0)
    xf = O.bf16_to_f64(x)
    for slot in range(2):
        _, d = sc.forward(slot, bits_to_torch(x), bits_to_torch(np.zeros((H, H), np.uint16)))
        d = d.cpu().numpy()
        for t, a in enumerate(wl.token_adapter):
            want = np.zeros(H)
            if a >= 0:
                want[(11 * a + 3 * slot + 1) % H] = np.float32(xf[t, (5 * a + slot) % H]) * (a + 1)
            assert np.array_equal(d[t].astype(np.float64), want), (slot, t, a)
    sc.close()


def test_nan_poisoned_free_pages_never_reach_output(L):
    wl = workloads.small(H=256, T=64, n_adapters=3, ranks=[64, 8, 16], seed=80, kv_fill=0.7)
    sc = DeviceScene(L, wl)
    sc.segments(wl.token_adapter)
    y, d = sc.forward(0, bits_to_torch(wl.x(0)), bits_to_torch(wl.W(0)))
    assert bool(y.float().isfinite().all()) and bool(d.isfinite().all())
    sc.close()


def test_unload_then_reload_other_adapter(L):
    wl = workloads.small(H=128, T=30, n_adapters=3, ranks=[8, 16, 4], seed=81)
    sc = DeviceScene(L, wl, adapters=[0, 1])
    L.lora_adapter_unload(sc.pool, 0)
    assert sc.model.unload(0) == O.OK
    del sc.tables[0]
    r = int(wl.ranks[2])
    tab = L.lora_adapter_load(sc.pool, 2, r, [wl.A(2, 0)], [wl.B(2, 0)], 1)
    st, mtab = sc.model.load(2, r, [True])
    assert np.array_equal(tab.astype(np.int64), mtab)
    O.place_adapter(sc.opool, mtab, [wl.A(2, 0)], [wl.B(2, 0)])
    sc.tables[2] = mtab
    ta = np.array([t % 3 for t in range(30)], dtype=np.int32)
    ta[ta == 0] = -1
    sc.segments(ta)
    y, d, y_ref, d_ref = _run_slot(sc, ta, 0, wl.x(0), wl.W(0))
    check_close(y, d, y_ref, d_ref, "reload")
    sc.close()


def test_forward_argument_errors(L):
    import torch
    wl = workloads.small(H=64, T=4, n_adapters=1, ranks=[2], seed=82)
    sc = DeviceScene(L, wl)
    sc.segments(wl.token_adapter)
    x = bits_to_torch(wl.x(0))
    W = bits_to_torch(wl.W(0))
    with pytest.raises(L.LoraError) as e:
        L.lora_linear_forward(sc.pool, sc.seg, 1, x, W, torch.empty_like(x))       # slot out of range
    assert e.value.code == L.LORA_EINVAL
    with pytest.raises(L.LoraError):
        L.lora_linear_forward(sc.pool, sc.seg, 0, x, W, x)                         # y aliases x
    with pytest.raises(L.LoraError):
        L.lora_segments_build(sc.pool, sc.ta_t, 5, sc.seg)                         # T > T_max
    sc.close()
