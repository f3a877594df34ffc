"""LoRA-aware tensor parallelism for the unmerged multi-adapter layer.

"S-LoRA, in depth", section "Tensor parallelism for adapters": the base model is split the
Megatron way (q, k and v column-parallel, o row-parallel), and every adapter is split to match,
so that the extra communication is a few [T, r] tensors beside the base's [T, H] all-reduce.
For a batch whose token t carries adapter a(t) of rank r_a (or none, -1):

  column-parallel projection (q, k, v), rank i of N owning output features F_i:
      W_i = W[F_i, :]          A_i(a) = A_a[:, R_i(a)]          B_i(a) = B_a[:, F_i]
      s_i[t] = x_t A_i(a(t))              the token's shrink over the rank's columns of its A
      s[t]   = all_gather_i(s_i[t])       [T, r_a(t)] reassembled column block by column block
      y_i[t] = x_t W_i^T + s[t] B_i(a(t)) [T, |F_i|], stays sharded by output feature

  row-parallel projection (o), rank i owning input features K_i (x arrives sharded, x_i = x[:, K_i]):
      W_i = W[:, K_i]          A_i(a) = A_a[K_i, :]             B_i(a) = B_a[:, F_i]
      s[t]   = all_reduce_i(x_i,t A_i(a(t)))     [T, r_max]
      p_i[t] = x_i,t W_i^T, plus s[t] B_i(a(t)) added into its columns F_i
      y      = all_reduce_i(p_i)          [T, H], the base's own all-reduce, shared

Per layer that is 3 all-gathers and one all-reduce of [T, r], 5 (N-1) T r / N elements a rank
receives, against the base's 2 (N-1) T H / N (the page's rank-16, H=4096 example: under 1 %).
R_i(a) and F_i are contiguous near-equal splits (the first n mod N ranks take one more).

This module holds the partition arithmetic and the collective schedule (torch.distributed: NCCL
between GPUs, gloo between CPU ranks).  The per-rank products come from a `local` object with
base(x, W) = x W^T, shrink(x, token_adapter, A) and expand(s, token_adapter, B) (A and B: dicts
adapter -> factor shard; each token uses its own adapter's, none for -1), so that the schedule
runs over whichever kernels compute them.
"""
from __future__ import annotations

from typing import Dict, List, Tuple


def split_sizes(n: int, world: int) -> List[int]:
    """Near-equal contiguous split of n items over `world` ranks (the first n % world get one more)."""
    base, extra = divmod(n, world)
    return [base + (1 if i < extra else 0) for i in range(world)]


def split_range(n: int, world: int, rank: int) -> Tuple[int, int]:
    sizes = split_sizes(n, world)
    lo = sum(sizes[:rank])
    return lo, lo + sizes[rank]


def shard_column(W, A: Dict, B: Dict, world: int, rank: int):
    """Rank `rank`'s shards for a column-parallel projection (W in nn.Linear layout [out][in];
    A[a] is [H_in, r_a], B[a] is [r_a, H_out])."""
    f0, f1 = split_range(W.shape[0], world, rank)
    A_i, B_i = {}, {}
    for a in A:
        r0, r1 = split_range(A[a].shape[1], world, rank)
        A_i[a] = A[a][:, r0:r1]
        B_i[a] = B[a][:, f0:f1]
    return W[f0:f1, :], A_i, B_i


def shard_row(W, A: Dict, B: Dict, world: int, rank: int):
    """Rank `rank`'s shards for a row-parallel projection: W columns K_i, A rows K_i, B columns F_i."""
    k0, k1 = split_range(W.shape[1], world, rank)
    f0, f1 = split_range(W.shape[0], world, rank)
    return W[:, k0:k1], {a: A[a][k0:k1, :] for a in A}, {a: B[a][:, f0:f1] for a in B}


def gather_shrink(s_i, token_adapter, ranks: Dict[int, int], group=None):
    """The full [T, r_max] shrink from every rank's column block: rank j holds, for token t,
    columns R_j(a(t)) of x_t A_a(t) in its first |R_j(a(t))| columns."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    r_max = max(ranks.values()) if ranks else 0
    width = -(-r_max // world)                    # the widest block any rank holds
    pad = torch.zeros((s_i.shape[0], width), dtype=s_i.dtype, device=s_i.device)
    pad[:, :min(width, s_i.shape[1])] = s_i[:, :width]
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad, group=group)
    s = torch.zeros((s_i.shape[0], r_max), dtype=s_i.dtype, device=s_i.device)
    ta = torch.as_tensor(token_adapter, device=s_i.device)
    for a, r in ranks.items():
        rows = (ta == a).nonzero(as_tuple=True)[0]
        if rows.numel() == 0:
            continue
        for j in range(world):
            c0, c1 = split_range(r, world, j)
            s[rows, c0:c1] = parts[j][rows, :c1 - c0]
    return s


def column_parallel_forward(x, token_adapter, W_i, A_i: Dict, B_i: Dict, ranks: Dict[int, int], local, group=None):
    """y_i = x W_i^T + (x A_a) B_i(a) per token on this rank: one all-gather of the shrink."""
    s_i = local.shrink(x, token_adapter, A_i)
    s = gather_shrink(s_i, token_adapter, ranks, group)
    return local.base(x, W_i) + local.expand(s, token_adapter, B_i)


def row_parallel_forward(x_i, token_adapter, W_i, A_i: Dict, B_i: Dict, H_out: int, local, group=None):
    """y = sum_i x_i W_i^T + (sum_i x_i A_i) B per token, on every rank: one all-reduce of the
    shrink, and the base's all-reduce of [T, H_out] carrying each rank's columns of the LoRA term."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    s = local.shrink(x_i, token_adapter, A_i)
    dist.all_reduce(s, group=group)
    p = local.base(x_i, W_i)
    f0, f1 = split_range(H_out, world, rank)
    p[:, f0:f1] += local.expand(s, token_adapter, B_i)
    dist.all_reduce(p, group=group)
    return p


def comm_elements(T: int, H: int, r: int, world: int) -> dict:
    """Elements a rank receives per layer (q, k, v column-parallel; o row-parallel), counting an
    all-reduce as a reduce-scatter plus an all-gather: the LoRA terms against the base's."""
    n = world
    lora = 3 * (n - 1) * T * r / n + 2 * (n - 1) * T * r / n
    base = 2 * (n - 1) * T * H / n
    return {"lora": lora, "base": base, "ratio": lora / base if base else 0.0}
