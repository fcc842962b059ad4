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
import pytest
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


# ------------------------------------------------------------------------------------------------
# The prefill query is quantised to FP4 (16-channel E4M3 scales, E2M1 values) before the product.
# A query row built from the hand-worked groups of tests/golden/kv_quant_rows.txt (cases A-E: a
# tie to the even code, a scale that rounds up, a group that flushes to zero) is not
# FP4-representable; its quantised value comes from the worked codes, decoded with the OCP
# definitions (E2M1 magnitudes written out, E4M3 through torch's float8_e4m3fn).
# ------------------------------------------------------------------------------------------------
import os

_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _golden_query_row():
    path = os.path.join(os.path.dirname(__file__), "golden", "kv_quant_rows.txt")
    x = np.zeros(512)
    qhat = np.zeros(512)
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        _, g, xs, sf, by = line.split()
        g = int(g.split("=")[1])
        x[16 * g:16 * g + 16] = [float(v) for v in xs.split("=")[1].split(",")]
        s = float(torch.tensor([int(sf.split("=")[1], 16)], dtype=torch.uint8)
                  .view(torch.float8_e4m3fn).to(torch.float64))
        for j, b in enumerate(int(v, 16) for v in by.split("=")[1].split(",")):
            for c, code in ((2 * j, b & 15), (2 * j + 1, b >> 4)):
                qhat[16 * g + c] = (-1 if code & 8 else 1) * _E2M1[code & 7] * s
    return x, qhat


def _check_query_quant(fn):
    x, qhat = _golden_query_row()
    rows = np.stack([x, -x, 2.0 * x])  # three (token, head) rows: sign and scale change
    qb = torch.from_numpy(rows).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = fn(qb)
    assert np.array_equal(got[0], qhat) and np.array_equal(got[1], -qhat)
    assert np.array_equal(got[2], 2.0 * qhat)


def test_prefill_query_is_quantised_to_fp4():
    x, qhat = _golden_query_row()
    assert not np.array_equal(x, qhat)  # the row is not FP4-representable
    _check_query_quant(oracle.quantize_query_fp4)
    # prefill attention uses the quantised query: it equals decode attention on q-hat, and
    # differs from decode attention on the raw query
    n = 64
    codes, sf, _ = _cache(n, 8)
    idx = np.arange(n, dtype=np.int32)[None, :]
    cu = np.array([0, n])
    qb = torch.from_numpy(np.stack([x, 2 * x])).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    qh = torch.from_numpy(np.stack([qhat, 2 * qhat])).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    pre = oracle.sparse_attn_prefill(qb[None], np.zeros(1, np.int32), codes, sf, cu, idx, 0.5)
    dec_hat = oracle.sparse_attn_decode(qh[None], codes, sf, cu, idx, 0.5)
    dec_raw = oracle.sparse_attn_decode(qb[None], codes, sf, cu, idx, 0.5)
    assert np.array_equal(pre[0][0], dec_hat[0][0]) and np.array_equal(pre[0][1], dec_hat[0][1])
    assert not np.array_equal(pre[0][1], dec_raw[0][1])


def test_query_quant_pin_catches_a_skipped_quantisation():
    with pytest.raises(AssertionError):
        _check_query_quant(lambda qb: oracle.bf16_to_double(qb))
