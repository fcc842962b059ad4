"""The allocation-free Reindex entry point (csa2_index_score_topk_reindex_noalloc) against the
workspace-taking one.

Some callers cannot give the library device memory beyond their inputs and outputs (a plugin
inside another engine that only hands over its buffers, or a process that reserved all device
memory up front); for them the library keeps its Reindex scratch in a fixed 4 MiB device array.
This test calls both entry points through the C ABI on the same inputs, twice in a row with
different queries (the fixed array keeps the previous call's contents), and requires identical
selections.  It lives in its own file, collected last, and passes alone or after the others.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp4_kv_top_csa2_b300 import csa2 as c
    return c


def _inputs(seed, lengths, n_pool):
    g = torch.Generator().manual_seed(seed)
    n = sum(lengths)
    k = torch.randn(n, 128, generator=g).to(torch.float8_e4m3fn).view(torch.uint8).cuda()
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int64).cuda()
    vis = torch.tensor(lengths, dtype=torch.int32).cuda()
    pools = []
    for L in lengths:  # ascending distinct block ids, -1 padded
        nb = (L + 7) // 8
        ids = torch.sort(torch.randperm(nb, generator=g)[: min(nb, n_pool)]).values
        pools.append(torch.cat([ids, torch.full((n_pool - ids.numel(),), -1)]))
    pool = torch.stack(pools).to(torch.int32).cuda()
    return k, cu, vis, pool


def _queries(seed, nq):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(nq, 8, 128, generator=g).to(torch.float8_e4m3fn).view(torch.uint8).cuda()
    w = torch.rand(nq, 8, generator=g).cuda()
    return q, w


def test_noalloc_reindex_matches_workspace_version_twice(csa2):
    lengths = [70000, 30001, 16000]
    n_pool, topk = 2048, 2048
    k, cu, vis, pool = _inputs(3, lengths, n_pool)
    nq = len(lengths)
    q_seq = torch.arange(nq, dtype=torch.int32, device="cuda")
    max_vis = max(lengths)
    ws = csa2.workspace(csa2.csa2_index_score_topk_workspace_size(nq, max_vis, n_pool, topk))
    for call in range(2):
        q, w = _queries(100 + call, nq)
        ref = torch.empty((nq, topk), dtype=torch.int32, device="cuda")
        got = torch.full((nq, topk), -7, dtype=torch.int32, device="cuda")
        csa2.csa2_index_score_topk(q, csa2.CSA2_E4M3, w, k, cu, q_seq, vis, max_vis, topk, ref,
                                   cand_blocks=pool, ws=ws)
        csa2.csa2_index_score_topk_reindex_noalloc(q, csa2.CSA2_E4M3, w, k, cu, q_seq, vis,
                                                   max_vis, topk, got, pool)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"call {call}"
        assert (ref[:, 0] >= 0).all()


def test_noalloc_rejects_requests_beyond_its_scratch(csa2):
    k, cu, vis, pool = _inputs(4, [20000], 2048)
    nq = 65  # 65 * 2048 * 8 slots > 1,048,576
    q, w = _queries(5, nq)
    big_pool = pool.expand(nq, -1).contiguous()
    out = torch.empty((nq, 64), dtype=torch.int32, device="cuda")
    with pytest.raises(csa2.Csa2Error) as ei:
        csa2.csa2_index_score_topk_reindex_noalloc(
            q, csa2.CSA2_E4M3, w, k, cu, torch.zeros(nq, dtype=torch.int32, device="cuda"),
            vis.expand(nq).contiguous(), 20000, 64, out, big_pool)
    assert ei.value.status == -4
