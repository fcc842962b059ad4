"""Pins of the oracle's local sliding-window branch (FP8 local KV, one softmax over the selected
global rows and the window's local rows).

* FP8 encoding: torch's independent float32 -> float8_e4m3fn conversion (round to nearest even)
  on every bf16 value up to 464 in magnitude (above that torch gives NaN; the saturation to 448
  is pinned by the format's largest finite value).
* The union softmax: torch's scaled_dot_product_attention in float64 over the concatenated rows
  (dequantised FP4 rows, then decoded FP8 rows).
* Two closed forms: with no local rows the result is the sparse attention exactly; and the union
  equals the two branches' results merged through their log-sum-exp.
* The window and its ring-buffer rows, built independently here.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _bf16_bits(t):
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_fp8_encoding_matches_torch_on_every_bf16_value():
    bits = np.arange(1 << 16, dtype=np.uint16)
    f = (bits.astype(np.uint32) << 16).view(np.float32)
    ok = np.isfinite(f) & (np.abs(f) <= 464.0)
    bits, f = bits[ok], f[ok]
    ref = torch.from_numpy(f).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.fp8_quant(bits)
    # torch keeps the sign of zero and of values that round to zero, as the oracle does
    assert np.array_equal(got, ref)


def test_fp8_encoding_saturates():
    x = torch.tensor([465.0, 500.0, 1e5, 3e38, -465.0, -1e30])
    got = oracle.fp8_quant(_bf16_bits(x))
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert oracle.e4m3_value(0x7E) == 448.0


def _case(seed, n_rows=200, n_loc=50, H=8):
    g = torch.Generator().manual_seed(seed)
    sigma = 10.0 ** (torch.rand(512, generator=g) * 2 - 1)
    x = (torch.randn(n_rows, 512, generator=g) * sigma)
    codes, sf = oracle.kv_quant_fp4(_bf16_bits(x))
    loc = oracle.fp8_quant(_bf16_bits(torch.randn(n_loc, 512, generator=g) * sigma))
    q = torch.randn(H, 512, generator=g, dtype=torch.float64).numpy()
    idx = np.random.default_rng(seed).permutation(n_rows)[:120].astype(np.int32)
    idx[::9] = -1
    return codes, sf, loc, q, idx


def test_union_softmax_matches_torch_sdpa():
    codes, sf, loc, q, idx = _case(1)
    scale = 1 / math.sqrt(512)
    out, lse = oracle.sparse_swa_attn(q, codes, sf, idx, loc, scale)
    glob = oracle.kv_dequant_fp4(codes, sf)[idx[idx >= 0]]
    locd = torch.from_numpy(loc).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    rows = torch.from_numpy(np.concatenate([glob, locd]))
    qt = torch.from_numpy(q)
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt[None, None], rows[None, None], rows[None, None], scale=scale)[0, 0]
    ref_lse = torch.logsumexp(qt @ rows.T * scale, dim=-1)
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, ref_lse.numpy(), rtol=1e-13, atol=1e-13)


def test_no_local_rows_is_the_sparse_attention_and_union_is_the_lse_merge():
    codes, sf, loc, q, idx = _case(2)
    scale = 0.07
    a, la = oracle.sparse_attn(q, codes, sf, idx, scale)
    a2, la2 = oracle.sparse_swa_attn(q, codes, sf, idx, loc[:0], scale)
    assert np.array_equal(a, a2) and np.array_equal(la, la2)
    b, lb = oracle.sparse_swa_attn(q, codes, sf, np.full(4, -1, np.int32), loc, scale)
    u, lu = oracle.sparse_swa_attn(q, codes, sf, idx, loc, scale)
    m = np.maximum(la, lb)
    wa, wb = np.exp(la - m), np.exp(lb - m)
    merged = (wa[:, None] * a + wb[:, None] * b) / (wa + wb)[:, None]
    assert np.allclose(u, merged, rtol=1e-12, atol=1e-12)
    assert np.allclose(lu, m + np.log(wa + wb), rtol=1e-13, atol=1e-13)
    e, le = oracle.sparse_swa_attn(q, codes, sf, np.full(4, -1, np.int32), loc[:0], scale)
    assert not e.any() and np.all(np.isneginf(le))


@pytest.mark.parametrize("vis,n_win", [(100, 16), (10, 16), (16, 16), (0, 16), (5000, 1)])
def test_window_positions_and_ring_rows(vis, n_win):
    want = [t for t in range(vis) if t >= vis - n_win]
    assert oracle.window_positions(vis, n_win).tolist() == want
    # ring: position t of sequence b at local row b * ring + t % ring
    ring, B = 24, 3
    g = torch.Generator().manual_seed(vis + n_win)
    swa = oracle.fp8_quant(_bf16_bits(torch.randn(B * ring, 512, generator=g)))
    codes, sf, _, _, _ = _case(3, n_rows=max(vis, 1) * B + 1)
    qb = _bf16_bits(torch.randn(B, 4, 512, generator=g))
    cu = np.array([0, max(vis, 1), 2 * max(vis, 1), 3 * max(vis, 1)])
    idx = np.full((B, 8), -1, np.int32)
    if n_win <= ring:
        res = oracle.sparse_swa_attn_queries(qb, np.arange(B), np.full(B, vis), codes, sf, cu, idx,
                                             swa, ring, n_win, 0.05)
        for b in range(B):
            loc = np.stack([swa[b * ring + t % ring] for t in want]) if want else swa[:0]
            o, l = oracle.sparse_swa_attn(oracle.bf16_to_double(qb[b]), codes, sf, idx[b], loc,
                                          0.05)
            assert np.array_equal(res[b][0], o) and np.array_equal(res[b][1], l)
