"""The allocation-free Reindex entry point (csa2_index_score_topk_reindex_noalloc) against the
workspace-taking one and against the oracle.

Some callers cannot give the library device memory beyond their inputs and outputs (a plugin
inside another engine that only hands over its buffers, or a process that reserved all device
memory up front); for them the library keeps its Reindex scratch in a fixed 4 MiB device array.
This test calls both entry points through the C ABI on the same inputs, twice in a row with
different queries (the fixed array keeps the previous call's contents), and requires identical
selections, which must also pass the oracle's Top-K check.  The cases cover the shapes where the
two could part ways: more than 1,024 queries, a pool of more than 2,048 blocks (the workspace
version then selects with its two-kernel path, this one with one CTA per query) and bf16 keys of
dimension 64.  It lives in its own file, collected last, and passes alone or after the others.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp4_kv_top_csa2_b300 import csa2 as c
    return c


def _keys(g, n, dtype):
    x = torch.randn(n, 128 if dtype == 1 else 64, generator=g)
    return x.to(torch.float8_e4m3fn).view(torch.uint8) if dtype == 1 else x.to(torch.bfloat16)


def _case(seed, lengths, q_per_seq, n_pool, dtype, Hi):
    g = torch.Generator().manual_seed(seed)
    k = _keys(g, sum(lengths), dtype)
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int64)
    q_seq, vis, pools = [], [], []
    for b, L in enumerate(lengths):
        for i in range(q_per_seq):
            v = L - i  # queries of one sequence see slightly different prefixes
            nb = (v + 7) // 8
            ids = torch.sort(torch.randperm(nb, generator=g)[: min(nb, n_pool)]).values
            pools.append(torch.cat([ids, torch.full((n_pool - ids.numel(),), -1)]))
            q_seq.append(b)
            vis.append(v)
    return (k, cu, torch.tensor(q_seq, dtype=torch.int32), torch.tensor(vis, dtype=torch.int32),
            torch.stack(pools).to(torch.int32))


def _queries(seed, nq, dtype, Hi):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(nq, Hi, 128 if dtype == 1 else 64, generator=g)
    q = x.to(torch.float8_e4m3fn).view(torch.uint8) if dtype == 1 else x.to(torch.bfloat16)
    return q, torch.rand(nq, Hi, generator=g)


def _np(t):
    t = t.cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


@pytest.mark.parametrize("lengths,q_per_seq,n_pool,topk,dtype,Hi", [
    ([70000, 30001, 16000], 1, 2048, 2048, 1, 8),  # the decoder's pool, three sequences
    ([50000], 1100, 16, 100, 1, 8),                 # more than 1,024 queries
    ([40000], 1, 4096, 2048, 1, 8),                 # a pool of more than 2,048 blocks
    ([9000, 5003], 2, 512, 512, 0, 4),              # bf16 keys of dimension 64
])
def test_noalloc_reindex_matches_workspace_version_twice(csa2, lengths, q_per_seq, n_pool, topk,
                                                         dtype, Hi):
    k, cu, q_seq, vis, pool = _case(3, lengths, q_per_seq, n_pool, dtype, Hi)
    nq = q_seq.numel()
    max_vis = int(vis.max())
    dk, dcu, dseq, dvis, dpool = (t.cuda() for t in (k, cu, q_seq, vis, pool))
    ws = csa2.workspace(csa2.csa2_index_score_topk_workspace_size(nq, max_vis, n_pool, topk))
    check = sorted({0, nq // 2, nq - 1})
    for call in range(2):
        q, w = _queries(100 + call, nq, dtype, Hi)
        dq, dw = q.cuda(), w.cuda()
        ref = torch.empty((nq, topk), dtype=torch.int32, device="cuda")
        got = torch.full((nq, topk), -7, dtype=torch.int32, device="cuda")
        csa2.csa2_index_score_topk(dq, dtype, dw, dk, dcu, dseq, dvis, max_vis, topk, ref,
                                   cand_blocks=dpool, ws=ws)
        csa2.csa2_index_score_topk_reindex_noalloc(dq, dtype, dw, dk, dcu, dseq, dvis, max_vis,
                                                   topk, got, dpool)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"call {call}"
        assert (ref[:, 0] >= 0).all()
        orc = oracle.index_score_topk(_np(q), dtype, w.numpy(), _np(k), cu.numpy(),
                                      q_seq.numpy(), vis.numpy(), topk,
                                      cand_blocks=pool.numpy(), queries=check)
        g = got.cpu().numpy()
        for n in check:
            check_topk(g[n], orc[n], topk, f"call {call} query {n}")


def test_noalloc_rejects_requests_beyond_its_scratch(csa2):
    k, cu, q_seq, vis, pool = _case(4, [20000], 1, 2048, 1, 8)
    nq = 65  # 65 * 2048 * 8 slots > 1,048,576
    q, w = _queries(5, nq, 1, 8)
    big_pool = pool.expand(nq, -1).contiguous().cuda()
    out = torch.empty((nq, 64), dtype=torch.int32, device="cuda")
    with pytest.raises(csa2.Csa2Error) as ei:
        csa2.csa2_index_score_topk_reindex_noalloc(
            q.cuda(), csa2.CSA2_E4M3, w.cuda(), k.cuda(), cu.cuda(),
            torch.zeros(nq, dtype=torch.int32, device="cuda"),
            vis.expand(nq).contiguous().cuda(), 20000, 64, out, big_pool)
    assert ei.value.status == -4
