"""LoRA-aware tensor parallelism on CPU ranks (gloo, world sizes 2 and 4): every rank's output of
the column-parallel (q/k/v) and row-parallel (o) schedules equals the oracle's unpartitioned layer
(its columns F_i, or all of it), for a batch with several adapters of ragged ranks and tokens
without an adapter.  The per-rank products are plain fp64 here; the schedule and the partition
arithmetic are the library's."""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from adapter_gemm_lora_gb300 import tp  # noqa: E402

_WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import numpy as np
import torch
import torch.distributed as dist
import oracle as O
import workloads
from adapter_gemm_lora_gb300 import tp

dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
H, ranks = {H}, {ranks}
wl = workloads.small(H=H, T={T}, n_adapters=len(ranks), ranks=ranks, seed={seed}, none_share=0.2)
ta = wl.token_adapter
f64 = lambda b: torch.from_numpy(O.bf16_to_f64(b))
x = f64(wl.x(0))
W = f64(wl.W(0))
A = {{a: f64(wl.A(a, 0)) for a in range(len(ranks))}}
B = {{a: f64(wl.B(a, 0)) for a in range(len(ranks))}}
r_of = {{a: int(r) for a, r in enumerate(ranks)}}

class Local:
    # fp64 products; each token uses its own adapter's shard, none for -1
    def base(self, x, W):
        return x @ W.T
    def shrink(self, x, ta, A):
        w = max(v.shape[1] for v in A.values())
        s = torch.zeros((x.shape[0], w), dtype=x.dtype)
        for a, Aa in A.items():
            rows = torch.from_numpy(np.nonzero(ta == a)[0])
            s[rows, :Aa.shape[1]] = x[rows] @ Aa
        return s
    def expand(self, s, ta, B):
        out = torch.zeros((s.shape[0], next(iter(B.values())).shape[1]), dtype=s.dtype)
        for a, Ba in B.items():
            rows = torch.from_numpy(np.nonzero(ta == a)[0])
            out[rows] = s[rows, :Ba.shape[0]] @ Ba
        return out

# the oracle's layer: x W^T + (x A) B per token, read through its page tables
model = O.PoolModel(wl.spec.pool_pages, 1, len(ranks), wl.page_order)
opool = np.full((wl.spec.pool_pages, H), 0x7FC0, np.uint16)
for a in range(len(ranks)):
    _, tab = model.load(a, int(ranks[a]), [True])
    O.place_adapter(opool, tab, [wl.A(a, 0)], [wl.B(a, 0)])
y_ref, _ = O.linear_forward(opool, model.tables, ta, 0, wl.x(0), wl.W(0))

W_i, A_i, B_i = tp.shard_column(W, A, B, world, rank)
y_i = tp.column_parallel_forward(x, ta, W_i, A_i, B_i, r_of, Local())
f0, f1 = tp.split_range(H, world, rank)
err_c = float(np.abs(y_i.numpy() - y_ref[:, f0:f1]).max())

k0, k1 = tp.split_range(H, world, rank)
W_r, A_r, B_r = tp.shard_row(W, A, B, world, rank)
y = tp.row_parallel_forward(x[:, k0:k1].contiguous(), ta, W_r, A_r, B_r, H, Local())
err_r = float(np.abs(y.numpy() - y_ref).max())
assert err_c < 1e-9 and err_r < 1e-9, (rank, err_c, err_r)
print("rank", rank, "ok", err_c, err_r)
dist.destroy_process_group()
"""


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


@pytest.mark.parametrize("world,H,ranks,T", [(2, 128, [8, 16, 3, 64], 37), (4, 256, [5, 16, 64, 1, 33], 50)])
def test_lora_tensor_parallel_matches_the_oracle(tmp_path, world, H, ranks, T):
    script = tmp_path / "worker.py"
    script.write_text(_WORKER.format(root=ROOT, H=H, ranks=ranks, T=T, seed=H + T))
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                   OMP_NUM_THREADS="1")
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.STDOUT, text=True))
    outs = [p.communicate(timeout=240)[0] for p in procs]
    for r, (p, out) in enumerate(zip(procs, outs)):
        assert p.returncode == 0, f"rank {r}:\n{out}"
        assert f"rank {r} ok" in out


def test_split_arithmetic_and_communication_count():
    assert tp.split_sizes(10, 4) == [3, 3, 2, 2] and sum(tp.split_sizes(1, 4)) == 1
    assert [tp.split_range(10, 4, i) for i in range(4)] == [(0, 3), (3, 6), (6, 8), (8, 10)]
    # the page's example: rank 16 against H = 4096, below 1 % of the base's communication
    c = tp.comm_elements(T=1, H=4096, r=16, world=8)
    assert c["ratio"] == pytest.approx(5 * 16 / (2 * 4096)) and c["ratio"] < 0.01
