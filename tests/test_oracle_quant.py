"""Pins of the oracle's FP4 main-KV quantisation (hand-worked rows, exact cases, invariants)."""
import os

import numpy as np
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _golden_rows():
    with open(os.path.join(GOLD, "kv_quant_rows.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, g, x, sf, by = line.split()
            yield (name, int(g.split("=")[1]), [float(v) for v in x.split("=")[1].split(",")],
                   int(sf.split("=")[1], 16), [int(b, 16) for b in by.split("=")[1].split(",")])


def test_hand_worked_groups():
    for name, g, x, sf, by in _golden_rows():
        row = np.zeros(512, dtype=np.float32)
        row[16 * g:16 * g + 16] = x
        codes, scales = oracle.kv_quant_fp4(_bf16(row)[None, :])
        assert scales[0, g] == sf, name
        assert list(codes[0, 8 * g:8 * g + 8]) == by, name
        # every other group is all-zero -> scale 0, codes 0
        other = [i for i in range(32) if i != g]
        assert not scales[0, other].any() and not np.delete(codes[0], range(8 * g, 8 * g + 8)).any()


def test_representable_rows_round_trip_exactly():
    """A group whose values are E2M1 values times a power of two with amax = 6 * 2^k has scale
    exactly 2^k, so dequantisation returns the input exactly."""
    rng = np.random.default_rng(0)
    e2m1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    rows = []
    for _ in range(64):
        row = []
        for g in range(32):
            k = int(rng.integers(-8, 7))
            v = rng.choice(e2m1, 16) * rng.choice([-1, 1], 16)
            v[rng.integers(16)] = 6.0 * rng.choice([-1, 1])
            row.append(v * 2.0 ** k)
        rows.append(np.concatenate(row))
    x = _bf16(np.array(rows))
    codes, sf = oracle.kv_quant_fp4(x)
    back = oracle.kv_dequant_fp4(codes, sf)
    assert np.array_equal(back, oracle.bf16_to_double(x))


def test_error_bound_and_group_locality():
    g = torch.Generator().manual_seed(3)
    sigma = 10.0 ** (torch.rand(512, generator=g) * 2 - 1)
    xt = (torch.randn(256, 512, generator=g) * sigma).to(torch.bfloat16)
    x = xt.view(torch.int16).numpy().view(np.uint16)
    codes, sf = oracle.kv_quant_fp4(x)
    xd = oracle.bf16_to_double(x)
    back = oracle.kv_dequant_fp4(codes, sf)
    s = np.array([[oracle.e4m3_value(c) for c in r] for r in sf])  # [256, 32]
    bound = np.repeat(s, 16, axis=1) + 6 * 2.0 ** -10
    # E2M1 grid spacing <= 2 (half-spacing 1) in units of the scale; saturation adds at most
    # 6 * (relative E4M3 rounding 2^-4) = 0.375 scales, or 6 * 2^-10 when the scale is subnormal.
    assert np.all(np.abs(back - xd) <= bound)
    # perturbing one channel changes only its own 16-channel group
    x2 = x.copy()
    x2[:, 100] = _bf16(np.full(256, 1234.0))
    c2, s2 = oracle.kv_quant_fp4(x2)
    grp = 100 // 16
    assert np.array_equal(np.delete(sf, grp, axis=1), np.delete(s2, grp, axis=1))
    assert np.array_equal(np.delete(codes, range(8 * grp, 8 * grp + 8), axis=1),
                          np.delete(c2, range(8 * grp, 8 * grp + 8), axis=1))
    assert np.all(s2[:, grp] == oracle.e4m3_encode(np.float32(1234.0) / np.float32(6.0)))


def test_scale_group_is_sixteen_channels():
    import json
    facts = json.load(open(os.path.join(GOLD, "pages_facts.json")))
    x = np.zeros((1, 512), dtype=np.float32)
    x[0, ::facts["scale_group"]] = 6.0
    codes, sf = oracle.kv_quant_fp4(_bf16(x))
    assert sf.shape[1] == 512 // facts["scale_group"]
    assert np.all(sf == 0x38)  # every group's amax is 6 -> scale 1.0
