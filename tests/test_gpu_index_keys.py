"""GPU-vs-oracle parity of the index keys derived from main-KV rows (csa2_index_keys_from_kv),
and of a Full selection over those keys.

The projection accumulates in fp32 on the tensor cores, in an order the oracle does not follow,
so a key may differ from the oracle's by one adjacent E4M3 code (or by the sign of zero), and
only where the exact y_i / s lies within 1e-5 (relative) of the rounding boundary between the
two codes.  The per-row scale must agree to 1e-6 relative.  Everything else is exact.
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


def _cache(n, seed):
    g = torch.Generator().manual_seed(seed)
    sigma = 10.0 ** (torch.rand(512, generator=g) * 2 - 1)
    x = (torch.randn(n, 512, generator=g) * sigma).to(torch.bfloat16)
    x[3] = 0.0  # a zero row: zero keys, scale 1
    W = (torch.randn(128, 512, generator=g) / 16).to(torch.bfloat16)
    return x, W


def _check_keys(keys, ks, codes, sf, W):
    rk, rks = oracle.index_keys_from_kv(codes, sf, W.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_allclose(ks, rks, rtol=1e-6, atol=0)
    bad = np.nonzero(keys != rk)
    if bad[0].size == 0:
        return 0
    xd = oracle.kv_dequant_fp4(codes, sf)
    Wd = W.to(torch.float64).numpy()
    dec = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    g, r = dec(keys[bad]), dec(rk[bad])
    y = np.einsum("nc,nc->n", Wd[bad[1]], xd[bad[0]])
    q = y / rks[bad[0]].astype(np.float64)
    zero_sign = (g == 0) & (r == 0)
    mid = (g + r) / 2
    near = np.abs(q - mid) <= 1e-5 * np.abs(q)
    adjacent = np.abs(keys[bad].astype(int) - rk[bad].astype(int)) == 1
    ok = zero_sign | (near & adjacent)
    assert ok.all(), f"{int((~ok).sum())} keys differ away from a rounding boundary"
    return bad[0].size


@pytest.mark.parametrize("n", [1000, 100_003])
def test_index_keys_match_oracle(csa2, n):
    x, W = _cache(n, n)
    codes = torch.empty((n, 256), dtype=torch.uint8, device="cuda")
    sf = torch.empty((n, 32), dtype=torch.uint8, device="cuda")
    csa2.csa2_kv_quant_fp4(x.cuda(), codes, sf)
    keys = torch.empty((n, 128), dtype=torch.uint8, device="cuda")
    ks = torch.empty(n, dtype=torch.float32, device="cuda")
    csa2.csa2_index_keys_from_kv(codes, sf, W.cuda(), keys, ks)
    c, s = codes.cpu().numpy(), sf.cpu().numpy()
    sample = np.unique(np.concatenate([np.arange(min(n, 2000)),
                                       np.random.default_rng(0).integers(0, n, 2000)]))
    _check_keys(keys.cpu().numpy()[sample], ks.cpu().numpy()[sample], c[sample], s[sample], W)
    assert ks[3].item() == 1.0 and not (keys[3] & 0x7F).any()
    # listed rows (a decode step's new tokens) write only those rows
    rows = torch.tensor([5, 999, 17, 256], dtype=torch.int64)
    k2 = torch.full((n, 128), 0xAB, dtype=torch.uint8, device="cuda")
    s2 = torch.full((n,), -1.0, device="cuda")
    csa2.csa2_index_keys_from_kv(codes, sf, W.cuda(), k2, s2, rows=rows.cuda())
    assert torch.equal(k2[rows.cuda()], keys[rows.cuda()])
    assert torch.equal(s2[rows.cuda()], ks[rows.cuda()])
    others = torch.ones(n, dtype=torch.bool)
    others[rows] = False
    assert (k2[others.cuda()] == 0xAB).all() and (s2[others.cuda()] == -1.0).all()


def test_full_selection_over_derived_keys(csa2):
    """The Full layer's index keys derived from its main-KV rows, then scored with their per-row
    scales: the selection equals the oracle's on the same keys."""
    lengths = [20000, 7000]
    n = sum(lengths)
    x, W = _cache(n, 7)
    codes = torch.empty((n, 256), dtype=torch.uint8, device="cuda")
    sf = torch.empty((n, 32), dtype=torch.uint8, device="cuda")
    csa2.csa2_kv_quant_fp4(x.cuda(), codes, sf)
    keys = torch.empty((n, 128), dtype=torch.uint8, device="cuda")
    ks = torch.empty(n, dtype=torch.float32, device="cuda")
    csa2.csa2_index_keys_from_kv(codes, sf, W.cuda(), keys, ks)
    g = torch.Generator().manual_seed(8)
    q = torch.randn(2, 8, 128, generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
    w = torch.rand(2, 8, generator=g)
    cu = torch.tensor([0, lengths[0], n], dtype=torch.int64)
    vis = torch.tensor(lengths, dtype=torch.int32)
    topk = 512
    out = torch.empty((2, topk), dtype=torch.int32, device="cuda")
    ws = csa2.workspace(csa2.csa2_index_score_topk_workspace_size(2, max(lengths), 0, topk))
    csa2.csa2_index_score_topk(q.cuda(), 1, w.cuda(), keys, cu.cuda(),
                               torch.arange(2, dtype=torch.int32, device="cuda"), vis.cuda(),
                               max(lengths), topk, out, k_scale=ks, ws=ws)
    ref = oracle.index_score_topk(q.numpy(), 1, w.numpy(), keys.cpu().numpy(), cu.numpy(),
                                  np.arange(2), vis.numpy(), topk, k_scale=ks.cpu().numpy())
    got = out.cpu().numpy()
    for b in range(2):
        check_topk(got[b], ref[b], topk, f"query {b}")
