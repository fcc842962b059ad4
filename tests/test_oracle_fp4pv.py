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


# Worked example of P's re-quantisation.  The cache rows are one-hot: row j holds 1.0 in channel
# j, which quantises to E2M1 6 x E4M3(1/6) = 6 x 0.171875 = 1.03125, so the dequantised row is
# 1.03125 e_j.  Along the slots, channel j's 16-slot block then holds that single value, whose
# block scale is E4M3(1.03125 / 6) = 0.171875 again: V re-quantises to itself.  The query puts
# score ln(p_j) on slot j (maximum 0, so lse = ln sum Pt), and output channel j is
# Pt_j * 1.03125 / sum Pt.  Block 0's largest numerator is 1, scale E4M3(1/6) = 0.171875; block
# 1's is 0.5, scale E4M3(0.5/6 = 0.0833) = 0.0859375 (1.375 x 2^-4, nearer than 1.25 x 2^-4).
# Pt = E2M1(p / sc) * sc by hand, e.g. 0.75 / 0.171875 = 4.36 -> 4 -> 0.6875.  Exact ties,
# resolved to the even code: 0.04296875 / 0.171875 = 0.25 -> 0, 0.859375 / 0.171875 = 5 -> 4,
# 0.30078125 / 0.171875 = 1.75 -> 2, 0.064453125 / 0.0859375 = 0.75 -> 1,
# 0.21484375 / 0.0859375 = 2.5 -> 2.
P_BLOCK0 = [1.0, 0.75, 0.5, 0.3, 0.25, 0.2, 0.1, 0.05,
            0.04296875, 0.6, 0.4, 0.15, 0.12, 0.859375, 0.9, 0.30078125]
PT_BLOCK0 = [1.03125, 0.6875, 0.515625, 0.2578125, 0.2578125, 0.171875, 0.0859375, 0.0859375,
             0.0, 0.515625, 0.34375, 0.171875, 0.0859375, 0.6875, 1.03125, 0.34375]
P_BLOCK1 = [0.5, 0.45, 0.3, 0.2, 0.1, 0.07, 0.04, 0.02,
            0.064453125, 0.25, 0.15, 0.06, 0.03, 0.21484375, 0.38, 0.12]
PT_BLOCK1 = [0.515625, 0.515625, 0.2578125, 0.171875, 0.0859375, 0.0859375, 0.04296875, 0.0,
             0.0859375, 0.2578125, 0.12890625, 0.04296875, 0.04296875, 0.171875, 0.34375,
             0.12890625]


def test_numerators_requantised_per_block_worked_example():
    n = 32
    x = np.zeros((n, 512), dtype=np.float32)
    x[np.arange(n), np.arange(n)] = 1.0
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    codes, sf = oracle.kv_quant_fp4(bits)
    kv = oracle.kv_dequant_fp4(codes, sf)
    assert np.array_equal(kv, 1.03125 * np.eye(n, 512))
    p = np.array(P_BLOCK0 + P_BLOCK1)
    q = np.zeros((1, 512))
    q[0, :n] = np.log(p) / 1.03125
    out, lse = oracle.attn_fp4pv(q, codes, sf, np.arange(n, dtype=np.int32), 1.0)
    pt = np.array(PT_BLOCK0 + PT_BLOCK1)
    total = pt.sum()
    assert np.allclose(out[0, :n], pt * 1.03125 / total, rtol=1e-12, atol=0)
    assert not out[0, n:].any()
    assert abs(lse[0] - math.log(total)) < 1e-12
