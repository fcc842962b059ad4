"""GPU-vs-oracle parity of each C-ABI call on small inputs that still span several tiles and a
ragged tail, plus the degenerate cases (empty inputs, fewer candidates than K, empty slots)."""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import check_attn, check_topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp4_kv_top_csa2_b300 import csa2 as c
    return c


def _bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _kv(n, seed):
    g = torch.Generator().manual_seed(seed)
    sigma = 10.0 ** (torch.rand(512, generator=g) * 2 - 1)
    return (torch.randn(n, 512, generator=g) * sigma).to(torch.bfloat16)


# ------------------------------------------------------------------------------------------------
# FP4 quantisation: bit-exact
# ------------------------------------------------------------------------------------------------
def _edge_rows():
    rows = []
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for k in range(-12, 12, 3):  # every E2M1 midpoint at scale 2^k (amax = 6 * 2^k)
        for sign in (1, -1):
            r = np.zeros(512)
            for g in range(32):
                v = np.array(mids + [6.0] + mids[::-1] + [0.0]) * 2.0 ** k * sign
                r[16 * g:16 * g + 16] = np.roll(v, g)
            rows.append(r)
    tiny = np.zeros(512)
    tiny[::16] = 2.0 ** -11
    tiny[1::16] = -(2.0 ** -20)
    rows.append(tiny)
    sub = np.zeros(512)
    for g in range(32):  # scales across the E4M3 subnormal range
        sub[16 * g:16 * g + 16] = np.linspace(-1, 1, 16) * 6 * 2.0 ** (-14 + g / 4)
    rows.append(sub)
    big = np.zeros(512)
    big[::2] = 3.0e38
    big[1::2] = -1e30
    rows.append(big)
    z = np.zeros(512)
    z[::3] = -0.0
    rows.append(z)
    inf = np.linspace(-5.0, 5.0, 512)  # groups holding an infinity saturate (scale 448, code 7)
    inf[3], inf[16 + 9], inf[32], inf[33] = np.inf, -np.inf, np.inf, -np.inf
    rows.append(inf)
    return torch.tensor(np.array(rows), dtype=torch.float32).to(torch.bfloat16)


@pytest.mark.parametrize("n", [1, 7, 1000])
def test_kv_quant_bit_exact(csa2, n):
    x = torch.cat([_kv(n, n), _edge_rows()])
    codes = torch.empty((x.shape[0], 256), dtype=torch.uint8, device="cuda")
    sf = torch.empty((x.shape[0], 32), dtype=torch.uint8, device="cuda")
    csa2.csa2_kv_quant_fp4(x.cuda(), codes, sf)
    rc, rs = oracle.kv_quant_fp4(_bits(x))
    assert np.array_equal(sf.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_kv_quant_scattered_rows_and_empty(csa2):
    x = _kv(37, 2)
    out_rows = torch.randperm(100, generator=torch.Generator().manual_seed(0))[:37]
    codes = torch.zeros((100, 256), dtype=torch.uint8, device="cuda")
    sf = torch.zeros((100, 32), dtype=torch.uint8, device="cuda")
    csa2.csa2_kv_quant_fp4(x.cuda(), codes, sf, out_rows=out_rows.cuda())
    rc, rs = oracle.kv_quant_fp4(_bits(x))
    c, s = codes.cpu().numpy(), sf.cpu().numpy()
    assert np.array_equal(c[out_rows.numpy()], rc) and np.array_equal(s[out_rows.numpy()], rs)
    untouched = np.setdiff1d(np.arange(100), out_rows.numpy())
    assert not c[untouched].any() and not s[untouched].any()
    csa2.csa2_kv_quant_fp4(x[:0].cuda(), codes, sf)  # n_rows = 0 is a no-op


# ------------------------------------------------------------------------------------------------
# Indexer score + Top-K, pool
# ------------------------------------------------------------------------------------------------
def _index_case(lengths, dtype, Hi, seed, dup=0.0):
    g = torch.Generator().manual_seed(seed)
    Di = 64 if dtype == 0 else 128
    n = sum(lengths)
    kf = torch.randn(n, Di, generator=g)
    if dup:
        m = int(dup * n)
        dst = torch.randperm(n, generator=g)[:m]
        src = (torch.rand(m, generator=g) * n).long()
        kf[dst] = kf[src] + 1e-3 * torch.randn(m, Di, generator=g)
    qf = torch.randn(len(lengths), Hi, Di, generator=g)
    if dtype == 0:
        k, q = kf.to(torch.bfloat16), qf.to(torch.bfloat16)
        kn, qn = _bits(k), _bits(q)
    else:
        k = kf.to(torch.float8_e4m3fn).view(torch.uint8)
        q = qf.to(torch.float8_e4m3fn).view(torch.uint8)
        kn, qn = k.numpy(), q.numpy()
    w = torch.rand(len(lengths), Hi, generator=g)
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int64)
    return k, q, w, cu, kn, qn


def _pool_ws(csa2, bm, n_pool):
    return csa2.workspace(csa2.csa2_hier_candidate_pool_workspace_size(bm.shape[0], bm.shape[1],
                                                                       n_pool))


def _run_index(csa2, k, q, w, cu, vis, dtype, topk, cand=None, bm=None):
    nq = q.shape[0]
    max_vis = int(max(vis)) if len(vis) else 0
    out = torch.empty((nq, topk), dtype=torch.int32, device="cuda")
    ncand = 0 if cand is None else cand.shape[1]
    ws = csa2.workspace(csa2.csa2_index_score_topk_workspace_size(nq, max_vis, ncand, topk))
    csa2.csa2_index_score_topk(q.cuda(), dtype, w.cuda(), k.cuda(), cu.cuda(),
                               torch.arange(nq, dtype=torch.int32, device="cuda"),
                               torch.tensor(vis, dtype=torch.int32, device="cuda"), max_vis, topk,
                               out, cand_blocks=None if cand is None else cand.cuda(),
                               out_block_max=bm, ws=ws)
    return out.cpu().numpy()


@pytest.mark.parametrize("dtype,Hi,lengths,topk,dup", [
    (1, 8, [5, 3001, 20000], 2048, 0.0),
    (1, 8, [9000, 40000], 100, 0.1),
    (1, 8, [17000], 1, 0.1),
    (1, 8, [20000, 4100], 4096, 0.0),  # largest topk
    (0, 4, [4096, 700], 512, 0.0),
    (1, 16, [3000], 3000, 0.0),
])
def test_full_topk_and_block_max(csa2, dtype, Hi, lengths, topk, dup):
    k, q, w, cu, kn, qn = _index_case(lengths, dtype, Hi, sum(lengths) + topk, dup)
    vis = list(lengths)
    nb = (max(vis) + 7) // 8
    bm = torch.full((len(vis), nb), float("nan"), device="cuda")
    got = _run_index(csa2, k, q, w, cu, vis, dtype, topk, bm=bm)
    ref = oracle.index_score_topk(qn, dtype, w.numpy(), kn, cu.numpy(), np.arange(len(vis)),
                                  np.array(vis), topk)
    bmh = bm.cpu().numpy()
    for n in range(len(vis)):
        check_topk(got[n], ref[n], topk, f"query {n}")
        nbn = (vis[n] + 7) // 8
        np.testing.assert_allclose(bmh[n, :nbn], ref[n]["bm"], rtol=2e-6, atol=1e-6)


@pytest.mark.parametrize("dtype,Hi,lengths", [(1, 8, [5, 3001, 20000]), (0, 4, [4096, 700]),
                                              (1, 8, [1 << 17])])
def test_block_max_call_equals_full_selection_block_max(csa2, dtype, Hi, lengths):
    """csa2_index_block_max writes the block maxima csa2_index_score_topk writes (bit for bit),
    which are the oracle's within the fp32 accumulation band."""
    k, q, w, cu, kn, qn = _index_case(lengths, dtype, Hi, 7 + sum(lengths))
    vis = list(lengths)
    nq, max_vis = len(vis), max(vis)
    nb = (max_vis + 7) // 8
    bm1 = torch.full((nq, nb), float("nan"), device="cuda")
    _run_index(csa2, k, q, w, cu, vis, dtype, 64, bm=bm1)
    bm2 = torch.full((nq, nb), float("nan"), device="cuda")
    csa2.csa2_index_block_max(q.cuda(), dtype, w.cuda(), k.cuda(), cu.cuda(),
                              torch.arange(nq, dtype=torch.int32, device="cuda"),
                              torch.tensor(vis, dtype=torch.int32, device="cuda"), max_vis, bm2)
    ref = oracle.index_score_topk(qn, dtype, w.numpy(), kn, cu.numpy(), np.arange(nq),
                                  np.array(vis), 1)
    for n in range(nq):
        nbn = (vis[n] + 7) // 8
        assert torch.equal(bm1[n, :nbn], bm2[n, :nbn])
        np.testing.assert_allclose(bm2[n, :nbn].cpu().numpy(), ref[n]["bm"], rtol=2e-6, atol=1e-6)


def test_full_short_and_empty_visibility(csa2):
    k, q, w, cu, kn, qn = _index_case([1000, 1000, 1000], 1, 8, 5)
    vis = [0, 3, 999]  # nothing visible / fewer candidates than K / ragged
    got = _run_index(csa2, k, q, w, cu, vis, 1, 64)
    ref = oracle.index_score_topk(qn, 1, w.numpy(), kn, cu.numpy(), np.arange(3), np.array(vis), 64)
    assert np.all(got[0] == -1)
    for n in (1, 2):
        check_topk(got[n], ref[n], 64, f"query {n}")


def test_pool_and_reindex(csa2):
    lengths = [30000, 16384 * 2 + 5]
    k, q, w, cu, kn, qn = _index_case(lengths, 1, 8, 11, dup=0.05)
    vis = lengths
    nb = (max(vis) + 7) // 8
    bm = torch.empty((2, nb), device="cuda")
    _run_index(csa2, k, q, w, cu, vis, 1, 2048, bm=bm)
    for n_pool in (2048, 100):
        pool = torch.empty((2, n_pool), dtype=torch.int32, device="cuda")
        csa2.csa2_hier_candidate_pool(bm, torch.tensor(vis, dtype=torch.int32, device="cuda"),
                                      n_pool, pool, ws=_pool_ws(csa2, bm, n_pool))
        bmh = bm.cpu().numpy()
        ref_pool = oracle.hier_candidate_pool(bmh, vis, n_pool)  # same fp32 input: exact
        for n in range(2):
            assert np.array_equal(pool[n].cpu().numpy(), ref_pool[n])
    # Reindex with new queries over the GPU pool (2048 blocks)
    pool = torch.empty((2, 2048), dtype=torch.int32, device="cuda")
    csa2.csa2_hier_candidate_pool(bm, torch.tensor(vis, dtype=torch.int32, device="cuda"), 2048,
                                  pool, ws=_pool_ws(csa2, bm, 2048))
    g = torch.Generator().manual_seed(99)
    q2 = torch.randn(2, 8, 128, generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
    w2 = torch.rand(2, 8, generator=g)
    for topk in (2048, 512):
        got = _run_index(csa2, k, q2, w2, cu, vis, 1, topk, cand=pool)
        ref = oracle.index_score_topk(q2.numpy(), 1, w2.numpy(), kn, cu.numpy(), np.arange(2),
                                      np.array(vis), topk, cand_blocks=pool.cpu().numpy())
        for n in range(2):
            check_topk(got[n], ref[n], topk, f"reindex query {n}")


@pytest.mark.parametrize("lengths,topk,n_pool,with_bm", [
    ([30000, 16384 * 2 + 5], 2048, 2048, True),   # the pool is the Full block list
    ([30000, 16384 * 2 + 5], 512, 2048, False),   # pool larger than the block list
    ([30000, 20000], 2048, 100, True),            # pool smaller: its own selection
    ([700, 3], 64, 4096, True),                   # pool longer than the blocks: -1 padded
])
def test_index_with_pool_matches_separate_calls(csa2, lengths, topk, n_pool, with_bm):
    """csa2_index_score_topk_pool writes exactly what csa2_index_score_topk followed by
    csa2_hier_candidate_pool writes, and both equal the oracle."""
    k, q, w, cu, kn, qn = _index_case(lengths, 1, 8, sum(lengths) + n_pool, dup=0.05)
    vis = list(lengths)
    nq, max_vis = len(vis), max(vis)
    nb = (max_vis + 7) // 8
    qd, wd, kd, cud = q.cuda(), w.cuda(), k.cuda(), cu.cuda()
    seq = torch.arange(nq, dtype=torch.int32, device="cuda")
    vis_t = torch.tensor(vis, dtype=torch.int32, device="cuda")
    # separate calls
    bm1 = torch.empty((nq, nb), device="cuda")
    idx1 = torch.empty((nq, topk), dtype=torch.int32, device="cuda")
    ws = csa2.workspace(csa2.csa2_index_score_topk_workspace_size(nq, max_vis, 0, topk))
    csa2.csa2_index_score_topk(qd, 1, wd, kd, cud, seq, vis_t, max_vis, topk, idx1,
                               out_block_max=bm1, ws=ws)
    pool1 = torch.empty((nq, n_pool), dtype=torch.int32, device="cuda")
    csa2.csa2_hier_candidate_pool(bm1, vis_t, n_pool, pool1, ws=_pool_ws(csa2, bm1, n_pool))
    # fused call
    bm2 = torch.empty((nq, nb), device="cuda") if with_bm else None
    idx2 = torch.full((nq, topk), -7, dtype=torch.int32, device="cuda")
    pool2 = torch.full((nq, n_pool), -7, dtype=torch.int32, device="cuda")
    ws2 = csa2.workspace(csa2.csa2_index_score_topk_pool_workspace_size(nq, max_vis, topk, n_pool))
    csa2.csa2_index_score_topk_pool(qd, 1, wd, kd, cud, seq, vis_t, max_vis, topk, idx2, n_pool,
                                    pool2, out_block_max=bm2, ws=ws2)
    assert torch.equal(idx1, idx2)
    assert torch.equal(pool1, pool2)
    ref = oracle.index_score_topk(qn, 1, w.numpy(), kn, cu.numpy(), np.arange(nq), np.array(vis),
                                  topk)
    for n in range(nq):
        nbn = (vis[n] + 7) // 8
        if with_bm:
            assert torch.equal(bm1[n, :nbn], bm2[n, :nbn])
        check_topk(idx2[n].cpu().numpy(), ref[n], topk, f"query {n}")
        assert np.array_equal(pool2[n].cpu().numpy(),
                              oracle.candidate_pool(bm1[n, :nbn].cpu().numpy(), n_pool))


# ------------------------------------------------------------------------------------------------
# Sparse attention
# ------------------------------------------------------------------------------------------------
def _attn_case(B, H, n_rows, topk, seed, holes=True):
    g = torch.Generator().manual_seed(seed)
    x = _kv(B * n_rows, seed)
    q = torch.randn(B, H, 512, generator=g).to(torch.bfloat16)
    idx = torch.stack([torch.randperm(n_rows, generator=g)[:topk] for _ in range(B)]).to(torch.int32)
    if topk > n_rows:
        raise ValueError
    if holes:
        idx[:, ::7] = -1
    cu = torch.arange(0, (B + 1) * n_rows, n_rows, dtype=torch.int64)
    return x, q, idx, cu


@pytest.mark.parametrize("B,H,n_rows,topk", [(3, 64, 3000, 2048), (2, 64, 4000, 2048),
                                              (2, 16, 600, 512), (1, 64, 100, 33),
                                              (4, 64, 50, 1),
                                              (2, 128, 3000, 1024),   # H > 64: CUDA-core kernel
                                              (1, 80, 500, 300),
                                              (1, 64, 20000, 16384),  # largest topk
                                              (3, 16, 5000, 4096),    # 128-row tiles, 16 heads
                                              (5, 48, 3000, 2048),    # 128-row tiles, 48 heads
                                              (6, 64, 3000, 1000)])   # 128-row tiles, ragged
def test_decode_attention(csa2, B, H, n_rows, topk):
    """Batches of 1 to 5 sequences, 16 to 64 heads, Top-K 1 to 16,384 with empty slots (and one
    sequence with none).  Calls whose 32-row x 32-head tiles fit one wave take that kernel, the
    others (the first, the last four H <= 64 cases) the 128-row tiles with all heads per CTA;
    with 16 or 48 heads the 64 rows of a CTA's query and TMEM lanes are partly padding.  Two
    calls on one workspace must give the same result."""
    x, q, idx, cu = _attn_case(B, H, n_rows, topk, B * 1000 + topk)
    if topk == 1:
        idx[1] = -1  # a sequence with no valid slot
    codes = torch.empty((x.shape[0], 256), dtype=torch.uint8, device="cuda")
    sf = torch.empty((x.shape[0], 32), dtype=torch.uint8, device="cuda")
    csa2.csa2_kv_quant_fp4(x.cuda(), codes, sf)
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), device="cuda")
    ws = csa2.workspace(csa2.csa2_sparse_attn_decode_workspace_size(B, H, topk))
    scale = 1 / math.sqrt(512)
    csa2.csa2_sparse_attn_decode(q.cuda(), codes, sf, cu.cuda(), idx.cuda(), scale, out, lse, ws=ws)
    out2, lse2 = torch.empty_like(out), torch.empty_like(lse)
    csa2.csa2_sparse_attn_decode(q.cuda(), codes, sf, cu.cuda(), idx.cuda(), scale, out2, lse2,
                                 ws=ws)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    ref = oracle.sparse_attn_decode(_bits(q), codes.cpu().numpy(), sf.cpu().numpy(), cu.numpy(),
                                    idx.numpy(), scale)
    ob, lh = _bits(out), lse.cpu().numpy()
    for b in range(B):
        check_attn(ob[b], lh[b], ref[b][0], ref[b][1], oracle.double_to_bf16(ref[b][0]), f"seq {b}")


@pytest.mark.parametrize("T,H,topk", [(5, 64, 2048), (3, 16, 100), (2, 64, 40), (2, 64, 90),
                                      (3, 32, 200), (2, 64, 4000), (2, 128, 300)])
def test_prefill_attention(csa2, T, H, topk):
    """Tile counts from one to 32 (128 rows per tile, ragged last tiles), every 11th slot empty;
    more than 64 heads take the CUDA-core kernel."""
    n_rows = 4000
    x, _, _, _ = _attn_case(1, H, n_rows, topk, T)
    g = torch.Generator().manual_seed(T + 7)
    q = torch.randn(T, H, 512, generator=g).to(torch.bfloat16)
    idx = torch.stack([torch.randperm(n_rows, generator=g)[:topk] for _ in range(T)]).to(torch.int32)
    idx[:, 3::11] = -1
    cu = torch.tensor([0, n_rows], dtype=torch.int64)
    q_seq = torch.zeros(T, dtype=torch.int32)
    codes = torch.empty((n_rows, 256), dtype=torch.uint8, device="cuda")
    sf = torch.empty((n_rows, 32), dtype=torch.uint8, device="cuda")
    csa2.csa2_kv_quant_fp4(x.cuda(), codes, sf)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), device="cuda")
    ws = csa2.workspace(csa2.csa2_sparse_attn_prefill_workspace_size(T, H, topk))
    scale = 1 / math.sqrt(512)
    csa2.csa2_sparse_attn_prefill(q.cuda(), q_seq.cuda(), codes, sf, cu.cuda(), idx.cuda(), scale,
                                  out, lse, ws=ws)
    ref = oracle.sparse_attn_prefill(_bits(q), q_seq.numpy(), codes.cpu().numpy(),
                                     sf.cpu().numpy(), cu.numpy(), idx.numpy(), scale)
    ob, lh = _bits(out), lse.cpu().numpy()
    for i in range(T):
        check_attn(ob[i], lh[i], ref[i][0], ref[i][1], oracle.double_to_bf16(ref[i][0]), f"tok {i}")


@pytest.mark.parametrize("order,H", [("rising", 64), ("falling", 64), ("rising", 16)])
def test_prefill_attention_moving_maximum(csa2, order, H):
    """The prefill kernel's softmax keeps a per-head reference maximum that moves only when a
    score exceeds it by a wide margin.  Slots ordered by rising score (all heads share one
    direction, scores spanning hundreds of units) move it on every tile and rescale the running
    output; falling order never moves it after the first tile.  Token 1 starts with two empty
    tiles, token 2 has no valid slot at all."""
    n_rows, topk, T = 3000, 1000, 3
    x, _, _, _ = _attn_case(1, H, n_rows, topk, 77)
    g = torch.Generator().manual_seed(78)
    v = torch.randn(512, generator=g) * 40
    c = 1 + 2 * torch.rand(T, H, 1, generator=g)
    q = (c * v).to(torch.bfloat16)
    codes = torch.empty((n_rows, 256), dtype=torch.uint8, device="cuda")
    sf = torch.empty((n_rows, 32), dtype=torch.uint8, device="cuda")
    csa2.csa2_kv_quant_fp4(x.cuda(), codes, sf)
    kv = oracle.kv_dequant_fp4(codes.cpu().numpy(), sf.cpu().numpy())
    key = kv @ v.double().numpy()
    rows = np.argsort(key if order == "rising" else -key)
    idx = np.stack([rows[np.sort(np.random.default_rng(i).choice(n_rows, topk, replace=False))]
                    for i in range(T)]).astype(np.int32)
    idx[1, :256] = -1
    idx[2, :] = -1
    idx = torch.from_numpy(idx)
    cu = torch.tensor([0, n_rows], dtype=torch.int64)
    q_seq = torch.zeros(T, dtype=torch.int32)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), device="cuda")
    ws = csa2.workspace(csa2.csa2_sparse_attn_prefill_workspace_size(T, H, topk))
    scale = 1 / math.sqrt(512)
    csa2.csa2_sparse_attn_prefill(q.cuda(), q_seq.cuda(), codes, sf, cu.cuda(), idx.cuda(), scale,
                                  out, lse, ws=ws)
    ref = oracle.sparse_attn_prefill(_bits(q), q_seq.numpy(), codes.cpu().numpy(),
                                     sf.cpu().numpy(), cu.numpy(), idx.numpy(), scale)
    ob, lh = _bits(out), lse.cpu().numpy()
    for i in range(T):
        check_attn(ob[i], lh[i], ref[i][0], ref[i][1], oracle.double_to_bf16(ref[i][0]), f"tok {i}")
    assert not out[2].float().any() and torch.isneginf(lse[2]).all()


@pytest.mark.parametrize("dtype", [1, 0])
def test_index_exact_when_scores_are_exact(csa2, dtype):
    """Small-integer keys/queries and power-of-two head weights make every score exact in fp32,
    so the GPU's block maxima and selection must equal the oracle's exactly -- including the
    lower-position rule among the many exact ties this produces."""
    g = torch.Generator().manual_seed(7 + dtype)
    lengths = [5000, 12345]
    Di = 128 if dtype == 1 else 64
    kf = torch.randint(-3, 4, (sum(lengths), Di), generator=g).float()
    qf = torch.randint(-2, 3, (2, 8 if dtype == 1 else 4, Di), generator=g).float()
    w = torch.tensor([0.5, 0.25, 1.0, 2.0, 0.125, 4.0, 1.0, 0.5])[: qf.shape[1]].repeat(2, 1)
    if dtype == 1:
        k, q = kf.to(torch.float8_e4m3fn).view(torch.uint8), qf.to(torch.float8_e4m3fn).view(torch.uint8)
        kn, qn = k.numpy(), q.numpy()
    else:
        k, q = kf.to(torch.bfloat16), qf.to(torch.bfloat16)
        kn, qn = _bits(k), _bits(q)
    cu = torch.tensor([0, lengths[0], sum(lengths)], dtype=torch.int64)
    vis = lengths
    nb = (max(vis) + 7) // 8
    bm = torch.empty((2, nb), device="cuda")
    for topk in (1000, 37):
        got = _run_index(csa2, k, q, w, cu, vis, dtype, topk, bm=bm)
        ref = oracle.index_score_topk(qn, dtype, w.numpy(), kn, cu.numpy(), np.arange(2),
                                      np.array(vis), topk)
        for n in range(2):
            nbn = (vis[n] + 7) // 8
            assert np.array_equal(bm.cpu().numpy()[n, :nbn], ref[n]["bm"])
            assert np.array_equal(got[n], ref[n]["idx"])
    # Reindex over an explicit block list: exact too
    blocks = torch.tensor([[3, 10, 11, 200, 624, -1], [0, 5, 999, 1500, 1543, -1]], dtype=torch.int32)
    got = _run_index(csa2, k, q, w, cu, vis, dtype, 20, cand=blocks)
    ref = oracle.index_score_topk(qn, dtype, w.numpy(), kn, cu.numpy(), np.arange(2),
                                  np.array(vis), 20, cand_blocks=blocks.numpy())
    for n in range(2):
        assert np.array_equal(got[n], ref[n]["idx"])


@pytest.mark.parametrize("kind", ["random", "ties"])
def test_topk_over_many_blocks(csa2, kind):
    """Pool selection over more than 16,384 block maxima: random scores take the sampled
    shared-memory path; heavily tied integer scores overflow it and take the global path.
    Both must equal the oracle's selection on the same fp32 block maxima exactly."""
    L = 300_001
    if kind == "random":
        k, q, w, cu, kn, qn = _index_case([L], 1, 8, 21)
    else:
        g = torch.Generator().manual_seed(22)
        kf = torch.randint(-2, 3, (L, 128), generator=g).float()
        k = kf.to(torch.float8_e4m3fn).view(torch.uint8)
        q = torch.randint(-1, 2, (1, 8, 128), generator=g).float().to(torch.float8_e4m3fn).view(torch.uint8)
        w = torch.full((1, 8), 0.5)
        cu = torch.tensor([0, L], dtype=torch.int64)
    nb = (L + 7) // 8
    bm = torch.empty((1, nb), device="cuda")
    vis = torch.tensor([L], dtype=torch.int32, device="cuda")
    _run_index(csa2, k, q, w, cu, [L], 1, 2048, bm=bm)
    bmh = bm.cpu().numpy()
    for n_pool in (2048, 700, 4096):
        pool = torch.empty((1, n_pool), dtype=torch.int32, device="cuda")
        csa2.csa2_hier_candidate_pool(bm, vis, n_pool, pool, ws=_pool_ws(csa2, bm, n_pool))
        assert np.array_equal(pool[0].cpu().numpy(), oracle.candidate_pool(bmh[0], n_pool))


@pytest.mark.parametrize("nb,kind,vis_frac", [
    (131072, "normal", 1.0), (131069, "ties", 1.0), (131072, "ties", 0.37), (16384, "normal", 1.0),
    (16385, "ties", 1.0), (5, "normal", 1.0), (40000, "normal", 0.001),
    (16384, "strided", 1.0), (9001, "strided", 1.0), (16384, "ties", 1.0),
])
def test_pool_selection_cluster_sizes(csa2, nb, kind, vis_frac):
    """Candidate pool straight from given block maxima, at the element counts where one query's
    selection spans 1 to 8 cooperating CTAs (and ragged tails), with heavy ties and signed zeros.
    "strided": every 64th value is far above the rest, so regularly strided samples overstate
    the k-th value and a sampled threshold keeps fewer than k (the selection must recover).
    The selection must equal the oracle's on the same fp32 values exactly."""
    g = torch.Generator().manual_seed(nb + int(vis_frac * 100))
    B = 3
    if kind == "strided":
        bm = torch.randn(B, nb, generator=g)
        bm[:, ::64] += 100.0
    elif kind == "normal":
        bm = torch.randn(B, nb, generator=g) * 12 + 40
    else:
        bm = torch.randint(-3, 4, (B, nb), generator=g).float() * 0.5
        zeros = torch.rand(B, nb, generator=g) < 0.1
        bm[zeros] = torch.where(torch.rand(int(zeros.sum()), generator=g) < 0.5, 0.0, -0.0)
    vis = [max(1, int(nb * 8 * vis_frac)) - i for i in range(B)]
    vis = [max(1, v) for v in vis]
    vis_t = torch.tensor(vis, dtype=torch.int32, device="cuda")
    bmd = bm.cuda()
    for n_pool in (2048, 1, 4096):
        pool = torch.empty((B, n_pool), dtype=torch.int32, device="cuda")
        csa2.csa2_hier_candidate_pool(bmd, vis_t, n_pool, pool, ws=_pool_ws(csa2, bmd, n_pool))
        ref = oracle.hier_candidate_pool(bm.numpy(), vis, n_pool)
        got = pool.cpu().numpy()
        for n in range(B):
            assert np.array_equal(got[n], ref[n]), (n_pool, n)


@pytest.mark.parametrize("kind", ["two_values", "all_equal", "one_group"])
def test_pool_selection_many_queries_global_fallback(csa2, kind):
    """More than 64 queries over more than 16,384 block maxima each take the one-CTA-per-query
    selection; with heavy ties the keys at or above its sampled threshold overflow the staging
    room (or fall short of k), and it selects over global memory instead.  Exact against the
    oracle on the same fp32 values."""
    g = torch.Generator().manual_seed({"two_values": 1, "all_equal": 2, "one_group": 3}[kind])
    nq, nb = 80, 40000
    if kind == "two_values":     # ~20,000 keys equal the sampled threshold
        bm = torch.randint(0, 2, (nq, nb), generator=g).float()
    elif kind == "all_equal":    # every key ties; signed zeros mixed in
        bm = torch.where(torch.rand(nq, nb, generator=g) < 0.5, 0.0, -0.0)
    else:                        # a few large values, a plateau of ties below them
        bm = torch.full((nq, nb), 3.0)
        hot = torch.rand(nq, nb, generator=g) < 0.02
        bm[hot] = 5.0 + torch.rand(int(hot.sum()), generator=g)
    vis = [nb * 8 - 3 * i for i in range(nq)]
    vis_t = torch.tensor(vis, dtype=torch.int32, device="cuda")
    bmd = bm.cuda()
    for n_pool in (2048, 3000):
        pool = torch.empty((nq, n_pool), dtype=torch.int32, device="cuda")
        csa2.csa2_hier_candidate_pool(bmd, vis_t, n_pool, pool, ws=_pool_ws(csa2, bmd, n_pool))
        got = pool.cpu().numpy()
        for n in (0, 1, 37, nq - 1):
            assert np.array_equal(got[n], oracle.candidate_pool(bm[n].numpy()[:(vis[n] + 7) // 8],
                                                                n_pool)), (n_pool, n)


def test_prefill_indexer_many_queries(csa2):
    """More than 1,024 queries over one sequence takes the 32-queries-per-MMA scan: causal
    visibility per query (query i sees positions < P0 + i + 1), block maxima and Top-K."""
    P0, T, topk = 3000, 1100, 256
    L = P0 + T
    k, _, _, cu, kn, _ = _index_case([L], 1, 8, 31)
    g = torch.Generator().manual_seed(32)
    q = torch.randn(T, 8, 128, generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
    w = torch.rand(T, 8, generator=g)
    vis = np.arange(P0 + 1, P0 + 1 + T)
    nb = (L + 7) // 8
    bm = torch.full((T, nb), float("nan"), device="cuda")
    out = torch.empty((T, topk), dtype=torch.int32, device="cuda")
    ws = csa2.workspace(csa2.csa2_index_score_topk_workspace_size(T, L, 0, topk))
    csa2.csa2_index_score_topk(q.cuda(), 1, w.cuda(), k.cuda(), cu.cuda(),
                               torch.zeros(T, dtype=torch.int32, device="cuda"),
                               torch.tensor(vis, dtype=torch.int32, device="cuda"), L, topk, out,
                               out_block_max=bm, ws=ws)
    got, bmh = out.cpu().numpy(), bm.cpu().numpy()
    sample = [0, 1, 31, 32, 33, 500, 1023, 1024, 1057, T - 1]
    ref = oracle.index_score_topk(q.numpy(), 1, w.numpy(), kn, cu.numpy(), np.zeros(T, np.int32),
                                  vis, topk, queries=sample)
    for n in sample:
        check_topk(got[n], ref[n], topk, f"query {n}")
        nbn = (vis[n] + 7) // 8
        np.testing.assert_allclose(bmh[n, :nbn], ref[n]["bm"], rtol=2e-6, atol=1e-6)
