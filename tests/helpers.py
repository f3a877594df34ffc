"""Test-side harness: device scenes built from seeded workloads, and the oracle's view of them.

The oracle's pool is built by the oracle's own bookkeeping (PoolModel) and placement
(place_adapter) from the generator's arrays; nothing the CUDA path writes is fed back
into it.  Device outputs are only compared against it.
"""
from __future__ import annotations

import numpy as np

import oracle as O


class SparsePool:
    """Array-like pool for the oracle at full size: only written pages are stored; the
    rest read as bf16 NaN (the device pool's poison value)."""

    NAN = np.uint16(0x7FC0)

    def __init__(self, num_pages, H):
        self.num_pages, self.H = num_pages, H
        self.rows = {}

    def __setitem__(self, idx, row):
        self.rows[int(idx)] = np.asarray(row, dtype=np.uint16).copy()

    def __getitem__(self, idx):
        idx = np.asarray(idx)
        out = np.full(idx.shape + (self.H,), self.NAN, dtype=np.uint16)
        for pos, p in np.ndenumerate(idx):
            r = self.rows.get(int(p))
            if r is not None:
                out[pos] = r
        return out


def bits_to_torch(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def torch_to_bits(t):
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceScene:
    """A pool on the device with a workload's adapters loaded, mirrored by the oracle."""

    def __init__(self, L, wl, adapters=None, present=None, dense_oracle=None, stream=None, check_tables=True,
                 oracle_slots=None):
        import torch
        self.L, self.wl = L, wl
        self.H, self.n_slots = wl.H, wl.n_slots
        self.num_pages = wl.spec.pool_pages
        self.max_adapters = wl.spec.n_adapters
        self.pool_t = torch.full((self.num_pages, self.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        self.pool = L.lora_pool_create(self.pool_t, self.num_pages, self.H, self.n_slots, self.max_adapters,
                                       wl.page_order)
        self.model = O.PoolModel(self.num_pages, self.n_slots, self.max_adapters, wl.page_order)
        if dense_oracle is None:
            dense_oracle = self.num_pages * self.H <= (1 << 26)
        self.opool = np.full((self.num_pages, self.H), 0x7FC0, np.uint16) if dense_oracle else \
            SparsePool(self.num_pages, self.H)
        kv = L.lora_pool_reserve(self.pool, wl.kv_pages)
        _, mkv = self.model.reserve(wl.kv_pages)
        assert kv.tolist() == mkv
        self.tables = {}
        adapters = range(wl.spec.n_adapters) if adapters is None else adapters
        for a in adapters:
            r = int(wl.ranks[a])
            pres = [True] * self.n_slots if present is None else present(a)
            A = [wl.A(a, s) if pres[s] else None for s in range(self.n_slots)]
            B = [wl.B(a, s) if pres[s] else None for s in range(self.n_slots)]
            tab = L.lora_adapter_load(self.pool, a, r, A, B, self.n_slots, stream=stream)
            st, mtab = self.model.load(a, r, pres)
            assert st == O.OK
            if check_tables:
                assert np.array_equal(tab.astype(np.int64), mtab), f"page table of adapter {a} differs"
            if oracle_slots is None:
                O.place_adapter(self.opool, mtab, A, B)
            else:   # mirror only the slots the test samples
                O.place_adapter(self.opool, mtab, [A[s] if s in oracle_slots else None for s in range(self.n_slots)],
                                [B[s] if s in oracle_slots else None for s in range(self.n_slots)])
            self.tables[a] = mtab
        self.ws = None

    def segments(self, token_adapter, stream=None, max_group=1):
        import torch
        T = len(token_adapter)
        T_max = max(T, 1)
        nbytes = self.L.lora_segments_size_group(self.pool, T_max, max_group)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.seg = self.L.lora_segments_init_group(self.pool, self.ws, nbytes, T_max, max_group)
        self.ta_t = torch.from_numpy(np.asarray(token_adapter, dtype=np.int32)).cuda()
        self.L.lora_segments_build(self.pool, self.ta_t, T, self.seg, stream=stream)
        return self.seg

    def read_i32(self, ptr, n):
        import torch
        off = ptr - self.ws.data_ptr()
        return self.ws[off:off + 4 * n].view(torch.int32).cpu().numpy()

    def read_segments(self):
        import torch
        torch.cuda.synchronize()
        T = self.seg.T
        n_seg = int(self.read_i32(self.seg.n_seg, 1)[0])
        return (self.read_i32(self.seg.perm, T), self.read_i32(self.seg.seg_off, n_seg + 1),
                self.read_i32(self.seg.seg_adapter, n_seg))

    def read_units(self):
        """The LoRA-delta work list of the last build: int32 [U][4] (adapter, rank, first, count)."""
        import torch
        torch.cuda.synchronize()
        n_units = int(self.read_i32(self.seg.n_units, 1)[0])
        return self.read_i32(self.seg.units, 4 * n_units).reshape(n_units, 4)

    def forward(self, slot, x_t, W_t, with_delta=True, stream=None):
        import torch
        T = x_t.shape[0]
        y = torch.empty((T, self.H), dtype=torch.bfloat16, device="cuda")
        d = torch.empty((T, self.H), dtype=torch.float32, device="cuda") if with_delta else None
        self.L.lora_linear_forward(self.pool, self.seg, slot, x_t, W_t, y, d, stream=stream)
        return y, d

    def forward_group(self, slots, x_t, W_ts, with_delta=True, stream=None):
        """lora_linear_forward_group over `slots` (one shared x); returns lists of y and delta."""
        import torch
        T = x_t.shape[0]
        ys = [torch.empty((T, self.H), dtype=torch.bfloat16, device="cuda") for _ in slots]
        ds = [torch.empty((T, self.H), dtype=torch.float32, device="cuda") for _ in slots] if with_delta else None
        self.L.lora_linear_forward_group(self.pool, self.seg, slots, x_t, W_ts, ys, ds, stream=stream)
        return ys, ds

    def oracle(self, token_adapter, slot, x_bits, W_bits, tokens=None):
        return O.linear_forward(self.opool, self.tables, token_adapter, slot, x_bits, W_bits, tokens=tokens)

    def close(self):
        self.L.lora_pool_destroy(self.pool)


def bf16_f64(bits):
    return O.bf16_to_f64(bits)


def check_close(y_gpu_bits, d_gpu, y_ref, d_ref, tag=""):
    """The stated tolerance: |gpu - oracle| <= 1e-2 (1 + |oracle|) per element on y;
    relative L2 <= 5e-3 on the LoRA delta (read as fp32 from delta_dbg)."""
    y = bf16_f64(y_gpu_bits)
    bad = np.abs(y - y_ref) > 1e-2 * (1 + np.abs(y_ref))
    assert not bad.any(), f"{tag}: {int(bad.sum())} y elements out of tolerance; worst at " \
                          f"{np.unravel_index(np.argmax(np.abs(y - y_ref)), y.shape)}"
    if d_gpu is not None:
        d = np.asarray(d_gpu, dtype=np.float64)
        assert np.isfinite(d).all(), f"{tag}: non-finite delta"
        num = np.linalg.norm(d - d_ref)
        den = np.linalg.norm(d_ref)
        if den > 0:
            assert num / den <= 5e-3, f"{tag}: delta relative L2 {num / den:.3e}"
        else:
            assert num == 0, f"{tag}: delta should be zero"
        badd = np.abs(d - d_ref) > 1e-2 * (1 + np.abs(d_ref))
        assert not badd.any(), f"{tag}: {int(badd.sum())} delta elements out of tolerance"
