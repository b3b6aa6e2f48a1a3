"""Multi-rank token mapping through the library (GPU): G ranks are played
one after another on one GPU (no rank waits on another), their counts are
combined on the host as the all-gather would, and the addresses the
library assigns must equal the single-GPU mapping of the concatenated
batch, re-expressed inside each expert owner's receive buffer."""
import numpy as np
import pytest
import torch

from combine_fp32_softmax_gb300 import ep, moe
from combine_fp32_softmax_gb300.configs import MoEConfig
from combine_fp32_softmax_gb300.inputs import make_logits
from tests.gpu_util import DEV, device_error
from tests.test_ep_mapping import bases_restated, receive_rows_restated

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("G,E,k", [(2, 8, 2), (3, 64, 6), (4, 32, 4)])
def test_multi_rank_addresses_match_concatenated_batch(G, E, k):
    T = 1000
    cfgs = [MoEConfig(f"rank{r}", T, 64, 64, E, k) for r in range(G)]
    ws = moe.alloc_workspace(cfgs[0], DEV)
    sels, counts = [], []
    for r in range(G):
        z = make_logits(cfgs[r], seed=100 + r).to(DEV)
        idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
        w = torch.empty(T, k, dtype=torch.float32, device=DEV)
        moe.moe_route(cfgs[r], z, idx, w, ws)
        c = torch.empty(E, dtype=torch.int32, device=DEV)
        off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
        dest = torch.empty(T * k, dtype=torch.int32, device=DEV)
        moe.moe_token_addresses(cfgs[r], idx, None, c, off, dest, ws)
        sels.append(idx)
        counts.append(c.cpu().to(torch.int64))
    all_counts = torch.stack(counts)
    owners = ep.owner_of(E, G)
    got = []
    for r in range(G):
        rb, rows = ep.rank_bases(all_counts.to(DEV), r, owners)
        assert rb.cpu().tolist() == bases_restated(all_counts, r, owners).tolist()
        assert rows.cpu().tolist() == receive_rows_restated(all_counts, owners, G)
        c = torch.empty(E, dtype=torch.int32, device=DEV)
        off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
        dest = torch.empty(T * k, dtype=torch.int32, device=DEV)
        moe.moe_token_addresses(cfgs[r], sels[r], rb, c, off, dest, ws)
        got.append(dest.cpu().numpy())
    assert device_error(ws) == (0, 0)
    # single-GPU mapping of the concatenated batch
    cat = MoEConfig("cat", G * T, 64, 64, E, k)
    wsc = moe.alloc_workspace(cat, DEV)
    R = G * T * k
    t = {n: torch.empty(s, dtype=torch.int32, device=DEV) for n, s in
         [("counts", E), ("offsets", E + 1), ("dest", R), ("row_token", R), ("row_slot", R)]}
    moe.moe_dispatch(cat, torch.cat(sels), None, t["counts"], t["offsets"], t["dest"], t["row_token"],
                     t["row_slot"], None, wsc)
    offsets = t["offsets"].cpu().numpy()
    first = [min([offsets[e] for e in range(E) if owners[e] == o], default=0) for o in range(G)]
    flat = torch.cat(sels).cpu().numpy().reshape(-1)
    want = t["dest"].cpu().numpy() - np.array(first)[np.array(owners)[flat]]
    assert np.array_equal(np.concatenate(got), want)


def test_rank_bases_single_rank_and_owner_clamp():
    """One rank: the bases are the exclusive prefix sums of the counts (the
    single-GPU offsets) and one owner receives every row.  Owner indices
    outside [0, G) are clamped into range, so the bases equal those of the
    clamped owner table."""
    E = 40
    g = torch.Generator().manual_seed(3)
    counts = torch.randint(0, 50, (1, E), generator=g, dtype=torch.int32)
    base, rows = ep.rank_bases(counts.to(DEV), 0, [0] * E)
    want = torch.cumsum(counts[0], 0) - counts[0]
    assert base.cpu().tolist() == want.tolist()
    assert rows.cpu().tolist() == [int(counts.sum())]
    G = 3
    all_counts = torch.randint(0, 50, (G, E), generator=g, dtype=torch.int32)
    wild = [(-2 if e % 7 == 0 else (5 if e % 5 == 0 else e % G)) for e in range(E)]
    clamped = [min(max(o, 0), G - 1) for o in wild]
    for r in range(G):
        b1, r1 = ep.rank_bases(all_counts.to(DEV), r, wild)
        b2, r2 = ep.rank_bases(all_counts.to(DEV), r, clamped)
        assert torch.equal(b1, b2) and torch.equal(r1, r2)
        assert b1.cpu().tolist() == bases_restated(all_counts.to(torch.int64), r, clamped).tolist()
