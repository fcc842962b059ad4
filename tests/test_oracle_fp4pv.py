"""Pins of the oracle's full-FP4 PV variant of prefill attention (P and V re-quantised to
block-scaled FP4 along the slot axis, blocks of 16 consecutive slots).

* V's re-quantisation is the main-KV quantiser applied along the other axis: each (channel,
  16-slot block) column quantised by kv_quant_fp4 (pinned on its own) and dequantised.
* A zero query gives every valid slot the same numerator, so the output is the plain mean of the
  re-quantised rows and lse = log(n * Pt) with Pt = E2M1(1 / E4M3(1/6)) * E4M3(1/6) = 1.03125.
* A dominant set of identical rows takes all the weight: every other numerator underflows to 0,
  and the output is the mean of that set's re-quantised rows.
* Empty slots are zero rows that still occupy their place in the blocks.
"""
import math

import numpy as np
import torch

import oracle


def _rows(n, seed):
    g = torch.Generator().manual_seed(seed)
    sigma = 10.0 ** (torch.rand(512, generator=g) * 2 - 1)
    x = (torch.randn(n, 512, generator=g) * sigma).to(torch.bfloat16)
    codes, sf = oracle.kv_quant_fp4(x.view(torch.int16).numpy().view(np.uint16))
    return codes, sf, oracle.kv_dequant_fp4(codes, sf)


def _requant_columns(rows):
    """V re-quantised along slots with the (separately pinned) main-KV quantiser: each block of
    16 slots of one channel is a 16-value group."""
    K, d = rows.shape
    kp = (K + 15) // 16 * 16
    r = np.zeros((kp, d))
    r[:K] = rows
    groups = r.reshape(kp // 16, 16, d).transpose(0, 2, 1).reshape(-1, 16)  # [(b, c), 16]
    bits = torch.from_numpy(groups.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(bits.to(torch.float64), torch.from_numpy(groups))  # exact in bf16
    codes, sf = oracle.kv_quant_fp4(bits.view(torch.int16).numpy().view(np.uint16))
    deq = oracle.kv_dequant_fp4(codes, sf).reshape(kp // 16, d, 16).transpose(0, 2, 1)
    return deq.reshape(kp, d)[:K]


def test_zero_query_is_the_mean_of_requantised_rows():
    codes, sf, kv = _rows(300, 1)
    idx = np.random.default_rng(2).permutation(300)[:200].astype(np.int32)
    out, lse = oracle.attn_fp4pv(np.zeros((3, 512)), codes, sf, idx, 0.1)
    vt = _requant_columns(kv[idx])
    assert np.allclose(out, np.broadcast_to(vt.mean(0), out.shape), rtol=1e-13, atol=1e-13)
    assert np.allclose(lse, math.log(200 * 1.03125), rtol=0, atol=1e-13)


def test_empty_slots_keep_their_place_in_the_blocks():
    codes, sf, kv = _rows(300, 3)
    idx = np.random.default_rng(4).permutation(300)[:64].astype(np.int32)
    holes = idx.copy()
    holes[5::7] = -1
    out, lse = oracle.attn_fp4pv(np.zeros((2, 512)), codes, sf, holes, 0.1)
    rows = np.where((holes >= 0)[:, None], kv[np.maximum(holes, 0)], 0.0)
    vt = _requant_columns(rows)
    nv = int((holes >= 0).sum())
    assert np.allclose(out[0], vt[holes >= 0].sum(0) / nv, rtol=1e-13, atol=1e-13)
    assert np.allclose(lse, math.log(nv * 1.03125), atol=1e-13)
    e, le = oracle.attn_fp4pv(np.zeros((2, 512)), codes, sf, np.full(20, -1, np.int32), 0.1)
    assert not e.any() and np.all(np.isneginf(le))


def test_dominant_rows_take_all_the_weight():
    codes, sf, kv = _rows(400, 5)
    r = 17
    idx = np.random.default_rng(6).permutation(400)[:100].astype(np.int32)
    idx[[3, 40, 41, 99]] = r  # four slots of the same row, in three different blocks
    q = kv[r][None, :] * 50.0 / np.linalg.norm(kv[r]) ** 2 * 30  # scores of row r far ahead
    out, lse = oracle.attn_fp4pv(q, codes, sf, idx, 1.0)
    vt = _requant_columns(kv[idx])
    want = vt[[3, 40, 41, 99]].mean(0)
    assert np.allclose(out[0], want, rtol=1e-13, atol=1e-13)
