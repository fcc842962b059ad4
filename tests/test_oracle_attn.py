"""Pins of the oracle's sparse attention.

* Top-K = context length: sparse attention over every row equals dense softmax attention,
  computed here by torch's scaled_dot_product_attention and logsumexp in float64.
* Closed forms: a zero query gives the plain mean of the rows; one overwhelming score gives that
  row; empty slots (-1) are skipped; no valid slot gives 0 and lse = -inf.
* Prefill: a query that is exactly representable in FP4 quantises to itself, so prefill
  attention equals decode attention on it.
"""
import math

import numpy as np
import torch

import oracle


def _cache(n, seed):
    g = torch.Generator().manual_seed(seed)
    sigma = 10.0 ** (torch.rand(512, generator=g) * 2 - 1)
    x = (torch.randn(n, 512, generator=g) * sigma).to(torch.bfloat16)
    codes, sf = oracle.kv_quant_fp4(x.view(torch.int16).numpy().view(np.uint16))
    return codes, sf, oracle.kv_dequant_fp4(codes, sf)


def test_dense_equivalence_with_torch_sdpa():
    n, H = 300, 16
    codes, sf, kv = _cache(n, 0)
    g = torch.Generator().manual_seed(1)
    q = torch.randn(H, 512, generator=g, dtype=torch.float64)
    idx = np.random.default_rng(2).permutation(n).astype(np.int32)  # order must not matter
    out, lse = oracle.sparse_attn(q.numpy(), codes, sf, idx, 1 / math.sqrt(512))
    kvt = torch.from_numpy(kv)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q[None, None], kvt[None, None], kvt[None, None], scale=1 / math.sqrt(512))[0, 0]
    ref_lse = torch.logsumexp(q @ kvt.T / math.sqrt(512), dim=-1)
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, ref_lse.numpy(), rtol=1e-13, atol=1e-13)


def test_zero_query_gives_mean_and_dominant_score_gives_row():
    n = 64
    codes, sf, kv = _cache(n, 3)
    idx = np.arange(n, dtype=np.int32)
    out, lse = oracle.sparse_attn(np.zeros((1, 512)), codes, sf, idx, 0.1)
    assert np.allclose(out[0], kv.mean(0), rtol=1e-13, atol=1e-13)
    assert abs(lse[0] - math.log(n)) < 1e-13
    q = kv[17:18] * 1e3  # row 17 wins by an enormous margin
    out, _ = oracle.sparse_attn(q, codes, sf, idx, 1.0)
    assert np.array_equal(out[0], kv[17])


def test_empty_slots_skipped_and_all_empty():
    n = 50
    codes, sf, kv = _cache(n, 4)
    q = np.random.default_rng(5).standard_normal((4, 512))
    idx = np.arange(n, dtype=np.int32)
    holes = idx.copy()
    holes[::3] = -1
    a, la = oracle.sparse_attn(q, codes, sf, holes, 0.05)
    b, lb = oracle.sparse_attn(q, codes, sf, idx[holes >= 0], 0.05)
    assert np.array_equal(a, b) and np.array_equal(la, lb)
    out, lse = oracle.sparse_attn(q, codes, sf, np.full(8, -1, dtype=np.int32), 0.05)
    assert not out.any() and np.all(np.isneginf(lse))


def test_prefill_fp4_representable_query_equals_decode():
    n = 80
    codes, sf, _ = _cache(n, 6)
    rng = np.random.default_rng(7)
    e2m1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    q = rng.choice(e2m1, (4, 512)) * rng.choice([-1, 1], (4, 512))
    q[:, ::16] = 6.0  # amax 6 in every group -> scale 1, exact
    qb = torch.from_numpy(q).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    qhat = oracle.quantize_query_fp4(qb)
    assert np.array_equal(qhat, q)
    idx = np.arange(n, dtype=np.int32)[None, :]
    cu = np.array([0, n])
    pre = oracle.sparse_attn_prefill(qb[None], np.zeros(1, np.int32), codes, sf, cu, idx, 0.05)
    dec = oracle.sparse_attn_decode(qb[None], codes, sf, cu, idx, 0.05)
    assert np.array_equal(pre[0][0], dec[0][0]) and np.array_equal(pre[0][1], dec[0][1])
