"""Pins of the oracle's index keys derived from main-KV rows: key = E4M3(y / s) with
y = W x (x the dequantised FP4 row), s = max|y| / 448.

* A projection that picks channels (each row of W one-hot) reduces to quantising those channels:
  checked against torch's float32 division and float8_e4m3fn conversion.
* One non-zero weight: only that key is non-zero (the orientation of W).
* The largest |y| encodes to +-448 and every key times s stays within E4M3's rounding of the
  exact y (computed with Python fractions).
* Doubling W doubles s exactly and leaves the keys unchanged; a zero row gives zero keys.
"""
from fractions import Fraction

import numpy as np
import torch

import oracle


def _row(seed, n=3):
    g = torch.Generator().manual_seed(seed)
    sigma = 10.0 ** (torch.rand(512, generator=g) * 2 - 1)
    x = (torch.randn(n, 512, generator=g) * sigma).to(torch.bfloat16)
    codes, sf = oracle.kv_quant_fp4(x.view(torch.int16).numpy().view(np.uint16))
    return codes, sf, oracle.kv_dequant_fp4(codes, sf)


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_channel_picking_projection_is_plain_quantisation():
    codes, sf, x = _row(1)
    perm = np.random.default_rng(2).permutation(512)[:128]
    W = np.zeros((128, 512), np.float32)
    W[np.arange(128), perm] = 1.0
    keys, ks = oracle.index_keys_from_kv(codes, sf, _bf16(W))
    for r in range(x.shape[0]):
        # a sum of products starts from +0, so a channel holding -0 projects to +0
        y = torch.from_numpy(x[r, perm].astype(np.float32)) + 0.0
        s = (y.abs().max() / 448.0).to(torch.float32)
        ref = (y / s).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert ks[r] == s.item()
        assert np.array_equal(keys[r], ref)


def test_orientation_one_weight():
    codes, sf, x = _row(3, n=1)
    W = np.zeros((128, 512), np.float32)
    c0 = int(np.argmax(np.abs(x[0])))
    W[37, c0] = 1.5
    keys, ks = oracle.index_keys_from_kv(codes, sf, _bf16(W))
    nz = np.nonzero(keys[0] & 0x7F)[0]
    assert nz.tolist() == [37] and keys[0, 37] & 0x7F == 0x7E


def test_scale_and_rounding_against_exact_values():
    codes, sf, x = _row(4, n=4)
    g = torch.Generator().manual_seed(5)
    Wb = _bf16(torch.randn(128, 512, generator=g).numpy() / 16)
    Wf = (Wb.astype(np.uint32) << 16).view(np.float32)
    keys, ks = oracle.index_keys_from_kv(codes, sf, Wb)
    kv = torch.from_numpy(keys).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for r in range(x.shape[0]):
        y = [sum(Fraction(float(Wf[i, c])) * Fraction(float(x[r, c])) for c in range(512))
             for i in range(128)]
        amax = max(abs(v) for v in y)
        assert abs(Fraction(float(ks[r])) * 448 - amax) <= amax * Fraction(1, 1 << 22)
        assert np.abs(kv[r]).max() == 448.0
        for i in range(128):
            err = abs(Fraction(float(kv[r, i])) * Fraction(float(ks[r])) - y[i])
            assert err <= abs(y[i]) / 16 + Fraction(float(ks[r])) / 1024, (r, i)
    keys2, ks2 = oracle.index_keys_from_kv(codes, sf, _bf16(2.0 * Wf))
    assert np.array_equal(keys2, keys) and np.array_equal(ks2, 2.0 * ks)


def test_zero_row_gives_zero_keys():
    z = np.zeros((1, 512), np.uint16)
    codes, sf = oracle.kv_quant_fp4(z)
    W = _bf16(np.ones((128, 512), np.float32))
    keys, ks = oracle.index_keys_from_kv(codes, sf, W)
    assert not (keys & 0x7F).any() and ks[0] == 1.0
