"""Multi-rank token mapping (UniEP page, section 2.2, Algorithm 1) on CPU
ranks: world_size-2 gloo processes exchange their expert counts, and the
global addresses they assign must (1) be unique and fill every owner's
receive buffer exactly, and (2) equal the single-GPU mapping of the
concatenated batch (rank 0's tokens first) re-expressed per owner.  The
local stable ranks come from the oracle's permutation (test
infrastructure), and so do the cross-rank bases: on CPU ranks there is no
device for the library's moe_rank_bases, so the test restates its
definition (the GPU test checks the library's bases against the same
restatement)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from combine_fp32_softmax_gb300 import ep


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def bases_restated(all_counts, rank, owners):
    """Algorithm 1's cross-rank base of every expert for `rank`: the rows of
    the lower experts of the same owner, plus the lower ranks' slots to it."""
    G, E = all_counts.shape
    per_expert = all_counts.sum(dim=0).tolist()
    start, run = [0] * E, {}
    for e in range(E):
        start[e] = run.get(owners[e], 0)
        run[owners[e]] = start[e] + per_expert[e]
    lower = all_counts[:rank].sum(dim=0).tolist() if rank > 0 else [0] * E
    return torch.tensor([start[e] + lower[e] for e in range(E)], dtype=torch.int64)


def receive_rows_restated(all_counts, owners, G):
    per_expert = all_counts.sum(dim=0).tolist()
    return [sum(per_expert[e] for e in range(len(owners)) if owners[e] == o) for o in range(G)]


def _local_sel(rank, T, E, k, seed=0):
    g = torch.Generator().manual_seed(seed * 100 + rank)
    z = torch.randn(T, E, generator=g)
    from oracle import moe_oracle as O
    return O.route(z.numpy(), k).sel


def _global_addresses(rank, G, T, E, k, all_counts):
    from oracle import moe_oracle as O
    sel = _local_sel(rank, T, E, k)
    perm = O.permute(sel, E)  # local stable order: row r of expert e has local rank r - offsets[e]
    owners = ep.owner_of(E, G)
    base = bases_restated(all_counts, rank, owners)
    flat = sel.reshape(-1)
    local_rank = perm.dest - perm.offsets[flat]
    addr = base.numpy()[flat] + local_rank
    own = np.array(owners)[flat]
    return own, addr


def _worker(rank, G, port, T, E, k, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=G)
    sel = _local_sel(rank, T, E, k)
    counts = torch.bincount(torch.from_numpy(sel.reshape(-1)), minlength=E)
    all_counts = ep.all_gather_counts(counts)
    own, addr = _global_addresses(rank, G, T, E, k, all_counts)
    q.put((rank, own.tolist(), addr.tolist(), all_counts.tolist()))
    dist.destroy_process_group()


@pytest.mark.parametrize("E,k", [(8, 2), (6, 3)])
def test_two_rank_mapping_matches_single_gpu_mapping(E, k):
    G, T = 2, 50
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, G, port, T, E, k, q)) for r in range(G)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    all_counts = torch.tensor(res[0][3])
    owners = ep.owner_of(E, G)
    sizes = receive_rows_restated(all_counts, owners, G)
    # (1) every owner's buffer is filled exactly once
    for o in range(G):
        got = sorted(a for r in range(G) for ow, a in zip(res[r][1], res[r][2]) if ow == o)
        assert got == list(range(sizes[o]))
    # (2) equal to the single-rank mapping of the concatenated batch
    from oracle import moe_oracle as O
    sel = np.concatenate([_local_sel(r, T, E, k) for r in range(G)])
    perm = O.permute(sel, E)
    first_row_of_owner = [min([perm.offsets[e] for e in range(E) if owners[e] == o], default=0) for o in range(G)]
    flat = sel.reshape(-1)
    want = perm.dest - np.array(first_row_of_owner)[np.array(owners)[flat]]
    got = np.concatenate([np.array(res[r][2]) for r in range(G)])
    assert np.array_equal(got, want)


def test_one_rank_reduces_to_offsets():
    E, T, k = 7, 40, 3
    sel = _local_sel(0, T, E, k)
    counts = torch.bincount(torch.from_numpy(sel.reshape(-1)), minlength=E)
    base = bases_restated(counts[None].to(torch.int64), 0, ep.owner_of(E, 1))
    from oracle import moe_oracle as O
    assert base.tolist() == O.permute(sel, E).offsets[:-1].tolist()
