"""Plant plausible mistakes in a copy of the oracle; the pins must catch each one (CPU only)."""
import types

import numpy as np
import pytest

import oracle as O
from oracle import lora_oracle as L
from pins import ALL_PINS


def _forward(mut):
    """The oracle's forward with one planted mistake, selected by ``mut``."""
    def linear_forward(pool_bits, tables, token_adapter, slot, x_bits, Wt_bits, tokens=None):
        ta = np.asarray(token_adapter, dtype=np.int64)
        idx = np.arange(ta.size) if tokens is None else np.asarray(tokens, dtype=np.int64)
        x = L.bf16_to_f64(x_bits[idx])
        W = L.bf16_to_f64(Wt_bits) if mut == "W_not_transposed" else L.bf16_to_f64(Wt_bits).T
        base = x @ W
        delta = np.zeros_like(base)
        for row, t in enumerate(idx):
            a = int(ta[t])
            if a < 0:
                continue
            if mut == "neighbour_adapter":
                a = (a + 1) % len(tables)
            tab = tables[a][0 if mut == "slot_ignored" else slot]
            if tab[0, 0] < 0:
                continue
            if mut == "A_B_pages_swapped":
                A, B = L.bf16_to_f64(pool_bits[tab[1]]).T, L.bf16_to_f64(pool_bits[tab[0]])
            elif mut == "A_pages_reversed":
                A, B = L.bf16_to_f64(pool_bits[tab[0][::-1]]).T, L.bf16_to_f64(pool_bits[tab[1]])
            else:
                A, B = L.gather_adapter(pool_bits, tab)
            if mut == "last_rank_dropped":
                A, B = A[:, :-1], B[:-1]
            delta[row] = (x[row] @ A) @ B
        if mut == "lora_dropped":
            delta[:] = 0
        if mut == "lora_sign":
            return base - delta, -delta
        return base + delta, delta
    return linear_forward


def _segments_unstable(token_adapter):
    ta = np.asarray(token_adapter, dtype=np.int64)
    perm, off, sa = L.segments(ta)
    perm = perm.copy()
    for s in range(len(sa)):
        perm[off[s]:off[s + 1]] = perm[off[s]:off[s + 1]][::-1]     # ties in descending token order
    return perm, off, sa


def _segments_none_last(token_adapter):
    ta = np.asarray(token_adapter, dtype=np.int64)
    key = np.where(ta < 0, np.iinfo(np.int64).max, ta)
    perm = np.argsort(key, kind="stable")
    perm2, off, sa = L.segments(ta)
    return perm.astype(np.int32), off, sa


def _place_swapped(pool_bits, table, A_list, B_list):
    for s, (A, B) in enumerate(zip(A_list, B_list)):
        if A is None:
            continue
        for j in range(A.shape[1]):
            pool_bits[table[s, 1, j]] = A[:, j]
            pool_bits[table[s, 0, j]] = B[j, :]


class _PoolFrontPop(L.PoolModel):
    def load(self, adapter, rank, present):
        self.free.reverse()
        try:
            return super().load(adapter, rank, present)
        finally:
            self.free.reverse()


MUTANTS = {
    "lora_dropped": dict(linear_forward=_forward("lora_dropped")),
    "lora_sign": dict(linear_forward=_forward("lora_sign")),
    "W_not_transposed": dict(linear_forward=_forward("W_not_transposed")),
    "A_B_pages_swapped": dict(linear_forward=_forward("A_B_pages_swapped")),
    "A_pages_reversed": dict(linear_forward=_forward("A_pages_reversed")),
    "last_rank_dropped": dict(linear_forward=_forward("last_rank_dropped")),
    "slot_ignored": dict(linear_forward=_forward("slot_ignored")),
    "neighbour_adapter": dict(linear_forward=_forward("neighbour_adapter")),
    "segments_unstable": dict(segments=_segments_unstable),
    "segments_none_last": dict(segments=_segments_none_last),
    "place_swapped": dict(place_adapter=_place_swapped),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    mutant = types.SimpleNamespace(**{k: getattr(O, k) for k in dir(O) if not k.startswith("_")})
    for k, v in MUTANTS[name].items():
        setattr(mutant, k, v)
    failed = [p.__name__ for p in ALL_PINS if not p(mutant)[0]]
    assert failed, f"no pin caught mutant {name}"


def test_front_pop_changes_tables_but_not_outputs():
    """Popping from the wrong end is invisible to the forward (placement invariance) but
    changes the page tables, which the GPU parity tests compare bit-exactly."""
    a = L.PoolModel(20, 1, 2, page_order=np.arange(20))
    b = _PoolFrontPop(20, 1, 2, page_order=np.arange(20))
    assert not np.array_equal(a.load(0, 3, [True])[1], b.load(0, 3, [True])[1])


# ---- pool lifecycle: plausible mistakes in the sketch's bookkeeping, caught by the hand-worked
# scenario of tests/golden/pool_lifecycle_scenario.json
class _NewestFirst(O.PoolModel):
    def evict_idle(self, need):
        saved = self.refs
        self.refs = dict(reversed(list(saved.items())))
        try:
            return super().evict_idle(need)
        finally:
            self.refs = {a: n for a, n in saved.items() if a in self.tables}


class _EvictsBusy(O.PoolModel):
    def evict_idle(self, need):
        saved = dict(self.refs)
        self.refs = {a: 0 for a in self.refs}
        st, ev = super().evict_idle(need)
        self.refs = {a: n for a, n in saved.items() if a in self.tables}
        return st, ev


class _EvictsThenFails(O.PoolModel):          # the sketch taken literally: evictions stand on failure
    def evict_idle(self, need):
        for a in [a for a, n in self.refs.items() if n == 0]:
            if len(self.free) >= need:
                break
            self._drop(a)
        return (O.OK if len(self.free) >= need else O.ENOPAGES), []


class _PagesBackReversed(O.PoolModel):
    def _drop(self, adapter):
        table = self.tables.pop(adapter)
        self.ranks.pop(adapter)
        self.refs.pop(adapter)
        self.free.extend(int(p) for p in table.reshape(-1)[::-1] if p >= 0)


class _ResidentNotCounted(O.PoolModel):
    def ensure(self, adapter, rank, present):
        if adapter in self.tables:
            return O.OK, self.tables[adapter], False, []
        return super().ensure(adapter, rank, present)


@pytest.mark.parametrize("cls", [_NewestFirst, _EvictsBusy, _EvictsThenFails, _PagesBackReversed, _ResidentNotCounted],
                         ids=lambda c: c.__name__)
def test_lifecycle_mutation_is_caught(cls):
    import json
    import os
    from pool_scenario import OracleDriver, run_golden
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pool_lifecycle_scenario.json")))
    d = OracleDriver(g["pool"]["num_pages"], g["pool"]["n_slots"], g["pool"]["max_adapters"], model_cls=cls)
    assert run_golden(d, g["steps"]) != [], f"{cls.__name__} passes the scenario"


# ---- eviction rules: plausible mistakes, caught by the eviction pins (toy sequences, Belady's
# optimum by exhaustive search, the rule without foresight reducing to LRU)
class _NearestFutureFirst(O.PoolModel):
    def eviction_order(self):
        if self.policy != O.EVICT_FARTHEST:
            return super().eviction_order()
        return list(reversed(super().eviction_order()))


class _UnrequestedLast(O.PoolModel):
    def eviction_order(self):
        order = super().eviction_order()
        if self.policy != O.EVICT_FARTHEST:
            return order
        horizon = self.future if self.lookahead <= 0 else self.future[:self.lookahead]
        return [a for a in order if a in horizon] + [a for a in order if a not in horizon]


class _MostRecentlyUsed(O.PoolModel):
    def eviction_order(self):
        if self.policy != O.EVICT_LRU:
            return super().eviction_order()
        return sorted(super().eviction_order(), key=lambda a: -self.last_use[a])


class _LoadOrderForLru(O.PoolModel):
    def eviction_order(self):
        if self.policy == O.EVICT_LRU:
            return [a for a, n in self.refs.items() if n == 0]
        return super().eviction_order()


@pytest.mark.parametrize("cls", [_NearestFutureFirst, _UnrequestedLast, _MostRecentlyUsed, _LoadOrderForLru],
                         ids=lambda c: c.__name__)
def test_eviction_mutation_is_caught(cls):
    from test_oracle_pins import eviction_pin_failures
    assert eviction_pin_failures(cls) != [], f"{cls.__name__} passes the eviction pins"


# ---- decode attention: plausible mistakes, caught by the attention pins
def _attention(mut):
    def attention_decode(pool_bits, kv_tables, q_bits, n_heads):
        q_all = L.bf16_to_f64(q_bits)
        n_req, H = q_all.shape
        d = H // n_heads
        out = np.zeros((n_req, H))
        for i in range(n_req):
            tab = np.asarray(kv_tables[i], dtype=np.int64)
            k_col, v_col = (1, 0) if mut == "K_V_swapped" else (0, 1)
            K, V = L.bf16_to_f64(pool_bits[tab[:, k_col]]), L.bf16_to_f64(pool_bits[tab[:, v_col]])
            for h in range(n_heads):
                cols = slice(h, H, n_heads) if mut == "heads_interleaved" else slice(h * d, (h + 1) * d)
                qs = slice(None) if mut == "scores_over_all_heads" else cols
                s = K[:, qs] @ q_all[i, qs]
                if mut != "no_scale":
                    s = s / np.sqrt(d)
                w = np.exp(s - s.max())
                out[i, cols] = (w / w.sum()) @ V[:, cols]
        return out
    return attention_decode


@pytest.mark.parametrize("mut", ["no_scale", "scores_over_all_heads", "K_V_swapped", "heads_interleaved"])
def test_attention_mutation_is_caught(mut):
    from test_oracle_pins import attention_pin_failures
    assert attention_pin_failures(_attention(mut)) != [], f"{mut} passes the attention pins"


def test_attention_restatement_passes():
    """The same restatement without a planted mistake passes, so the pins are what catch them."""
    from test_oracle_pins import attention_pin_failures
    assert attention_pin_failures(_attention("none")) == []
