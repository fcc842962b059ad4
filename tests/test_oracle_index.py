"""Pins of the oracle's indexer score, Top-K, block maxima and candidate pool.

Exact rational arithmetic (fractions) on tiny inputs, closed forms, brute-force selection with
Python's own sort, and the pages' fixed facts about the hierarchical pool (2,048 blocks of 8
positions, independent of context length; "DeepSeek V4.1-Flash", aiwiki.ai, section
"Compressed Sparse Attention 2").
"""
import json
import os
from fractions import Fraction

import numpy as np
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
FACTS = json.load(open(os.path.join(GOLD, "pages_facts.json")))


def _e4m3(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e4m3_frac(code):
    # exact rational value straight from the bit fields
    s, e, m = code >> 7, (code >> 3) & 15, code & 7
    v = Fraction(m, 512) if e == 0 else Fraction(8 + m, 8) * Fraction(2) ** (e - 7)
    return -v if s else v


def test_scores_exact_rational_e4m3():
    Hi, Di, n = 3, 128, 40
    q = _e4m3((Hi, Di), 1)
    k = _e4m3((n, Di), 2)
    w = np.array([0.25, 0.5, 0.75], dtype=np.float32)
    got = oracle.index_scores(q, oracle.E4M3, w, k, np.arange(n))
    for t in range(n):
        tot = Fraction(0)
        for h in range(Hi):
            dot = sum(_e4m3_frac(int(q[h, c])) * _e4m3_frac(int(k[t, c])) for c in range(Di))
            tot += Fraction(float(w[h])) * max(dot, Fraction(0))
        assert got[t] == np.float32(float(tot)), t  # float(Fraction) rounds correctly


def test_scores_bf16_one_hot_closed_form():
    Di, n = 64, 50
    g = torch.Generator().manual_seed(5)
    k = torch.randn(n, Di, generator=g).to(torch.bfloat16)
    q = torch.zeros(2, Di)
    q[0, 7] = 1.0
    q[1, 9] = -2.0
    w = np.array([0.5, 0.25], dtype=np.float32)
    kb = k.view(torch.int16).numpy().view(np.uint16)
    qb = q.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.index_scores(qb, oracle.BF16, w, kb, np.arange(n))
    kf = k.to(torch.float64).numpy()
    want = 0.5 * np.maximum(kf[:, 7], 0) + 0.25 * np.maximum(-2 * kf[:, 9], 0)
    assert np.array_equal(got, want.astype(np.float32))


def test_scores_k_scale_and_weights_linear():
    q = _e4m3((4, 128), 7)
    k = _e4m3((30, 128), 8)
    w = np.array([1, 2, 3, 4], dtype=np.float32) / 8
    base = oracle.index_scores(q, oracle.E4M3, w, k, np.arange(30))
    ks = np.full(30, 2.0, dtype=np.float32)
    assert np.array_equal(oracle.index_scores(q, oracle.E4M3, w, k, np.arange(30), ks), 2 * base)
    assert np.array_equal(oracle.index_scores(q, oracle.E4M3, 4 * w, k, np.arange(30)), 4 * base)
    # ReLU: a negated query makes every head's dot product change sign
    qn = q ^ 0x80  # flip sign bits
    neg = oracle.index_scores(qn, oracle.E4M3, w, k, np.arange(30))
    assert np.all(neg >= 0) and np.all(base >= 0)


def _brute_topk(scores, pos, K):
    order = sorted(range(len(scores)), key=lambda i: (-float(scores[i]), int(pos[i])))
    sel = sorted(int(pos[i]) for i in order[:K])
    return sel + [-1] * (K - len(sel))


def test_topk_brute_force_and_ties():
    rng = np.random.default_rng(0)
    for trial in range(200):
        n = int(rng.integers(0, 60))
        K = int(rng.integers(1, 70))
        # few distinct values -> many exact ties
        s = rng.choice(np.array([0.0, -0.0, 1.0, 2.5, -3.0, 7.25], dtype=np.float32), n)
        pos = rng.permutation(1000)[:n].astype(np.int64)
        assert list(oracle.topk(s, pos, K)) == _brute_topk(s, pos, K)


def test_topk_all_equal_takes_lowest_positions_and_signed_zero_equal():
    s = np.zeros(20, dtype=np.float32)
    s[::2] = -0.0
    assert list(oracle.topk(s, np.arange(20), 5)) == [0, 1, 2, 3, 4]


def test_block_max_brute_force():
    rng = np.random.default_rng(1)
    for n in (1, 7, 8, 9, 64, 100):
        s = rng.standard_normal(n).astype(np.float32)
        bm = oracle.block_max(s, 8)
        want = [max(s[8 * b:8 * b + 8]) for b in range((n + 7) // 8)]
        assert list(bm) == want


def _full_and_pool(L, K, seed, n_pool=FACTS["pool_blocks"]):
    q = _e4m3((8, 128), seed)
    k = _e4m3((L, 128), seed + 1)
    w = np.random.default_rng(seed).random(8).astype(np.float32)
    s = oracle.index_scores(q, oracle.E4M3, w, k, np.arange(L))
    full = oracle.topk(s, np.arange(L), K)
    pool = oracle.candidate_pool(oracle.block_max(s, FACTS["block_size"]), n_pool)
    return q, k, w, s, full, pool


def test_pool_size_independent_of_context_length():
    bs, nb = FACTS["block_size"], FACTS["pool_blocks"]
    assert bs * nb == FACTS["pool_positions"]
    for L in (100, 8 * nb - 3, 8 * nb, 8 * nb + 1, 40000):
        *_, pool = _full_and_pool(L, 64, L)
        n_valid = int((pool >= 0).sum())
        assert n_valid == min(nb, -(-L // bs))
        assert np.all(np.diff(pool[:n_valid]) > 0)


def test_full_topk_inside_pool_and_reindex_with_same_query_matches():
    for L, K in ((40000, 2048), (30001, 512), (20000, 1)):
        q, k, w, s, full, pool = _full_and_pool(L, K, 11 + K)
        pool_pos = oracle.candidate_positions(pool, L)
        assert set(full[full >= 0]).issubset(set(pool_pos))
        # Reindex over the pool with the Full layer's own query reproduces Full's selection
        s_pool = oracle.index_scores(q, oracle.E4M3, w, k, pool_pos)
        assert np.array_equal(oracle.topk(s_pool, pool_pos, K), full)


def test_pool_covers_everything_when_context_is_short():
    # ceil(L/8) <= 2048 -> the pool is every block, and Reindex equals Full scoring
    L = 5000
    q, k, w, s, full, pool = _full_and_pool(L, 512, 3)
    assert list(pool[pool >= 0]) == list(range(-(-L // 8)))
    pos = oracle.candidate_positions(pool, L)
    assert np.array_equal(pos, np.arange(L))
