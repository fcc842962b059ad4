"""The C-ABI library loads and exports every entry point include/csa2.h declares, and its
host-side validation rejects bad arguments before touching a GPU (runs without a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa2.h")


@pytest.fixture(scope="module")
def csa2():
    from fp4_kv_top_csa2_b300 import csa2 as _c  # noqa: F401  (fails loudly if not built)
    return _c


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_\w+)\s*\(", text)))


def test_header_declares_the_five_calls():
    names = _declared()
    for n in ("csa2_kv_quant_fp4", "csa2_index_score_topk", "csa2_hier_candidate_pool",
              "csa2_sparse_attn_decode", "csa2_sparse_attn_prefill"):
        assert n in names


def test_every_declared_symbol_is_exported(csa2):
    out = subprocess.run(["nm", "-D", "--defined-only", csa2.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (csa2_\w+)$", out, flags=re.M))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    for n in _declared():
        assert hasattr(csa2.lib, n)


def test_error_strings(csa2):
    for code in (0, -1, -2, -3, -4, -5, 7):
        assert csa2.lib.csa2_error_string(code)


def test_host_validation_rejects_bad_arguments(csa2):
    L = csa2.lib
    p = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    odd = ctypes.c_void_p(4097)
    # kv quant: bad d, negative rows, misaligned pointer
    assert L.csa2_kv_quant_fp4(p, 10, 500, None, p, p, None) == -1
    assert L.csa2_kv_quant_fp4(p, -1, 512, None, p, p, None) == -1
    assert L.csa2_kv_quant_fp4(odd, 10, 512, None, p, p, None) == -1
    assert L.csa2_kv_quant_fp4(None, 10, 512, None, p, p, None) == -1
    assert L.csa2_kv_quant_fp4(None, 0, 512, None, None, None, None) == 0  # nothing to do
    # index score: dtype mismatch, wrong Di, topk out of range, workspace too small
    args = lambda qdt, Di, kdt, topk, ws, wsb: L.csa2_index_score_topk(
        p, qdt, p, 1, 8, Di, p, kdt, 5000, None, p, 1, p, p, 1000, None, 0, topk, p, None, ws, wsb,
        None)
    assert args(1, 128, 0, 16, p, 1 << 30) == -1
    assert args(1, 64, 1, 16, p, 1 << 30) == -1
    assert args(0, 128, 0, 16, p, 1 << 30) == -1
    assert args(1, 128, 1, 0, p, 1 << 30) == -1
    assert args(1, 128, 1, 5000, p, 1 << 30) == -1
    assert args(1, 128, 1, 16, ctypes.c_void_p(4096 + 16), 1 << 30) == -1  # ws not 256-aligned
    assert args(1, 128, 1, 16, p, 0) == -4
    # index + pool: block size 8, pool size 1..4096, pool output required, workspace
    pargs = lambda bs, npool, outp, wsb: L.csa2_index_score_topk_pool(
        p, 1, p, 1, 8, 128, p, 1, 5000, None, p, 1, p, p, 1000, 16, p, None, bs, npool, outp, p,
        wsb, None, None)
    assert pargs(4, 2048, p, 1 << 30) == -1
    assert pargs(8, 0, p, 1 << 30) == -1
    assert pargs(8, 5000, p, 1 << 30) == -1
    assert pargs(8, 2048, None, 1 << 30) == -1
    assert pargs(8, 2048, odd, 1 << 30) == -1
    assert pargs(8, 2048, p, 0) == -4
    # pool: block size must be 8
    assert L.csa2_hier_candidate_pool(p, 1, p, 100, 4, 2048, p, None, 0, None) == -1
    assert L.csa2_hier_candidate_pool(p, 1, p, 100, 8, 0, p, None, 0, None) == -1
    # attention: scale must be > 0, H range
    assert L.csa2_sparse_attn_decode(p, 1, 64, p, p, p, p, 16, ctypes.c_float(0.0), p, None,
                                     None, 0, None) == -1
    assert L.csa2_sparse_attn_decode(p, 1, 0, p, p, p, p, 16, ctypes.c_float(0.1), p, None,
                                     None, 0, None) == -1
    assert L.csa2_sparse_attn_prefill(p, 4, 64, p, p, p, p, 1, p, 16, ctypes.c_float(0.1), p,
                                      None, p, 0, None) == -4


def test_workspace_sizes_are_host_only(csa2):
    L = csa2.lib
    assert L.csa2_index_score_topk_workspace_size(1, 1 << 20, 0, 2048) > 0
    assert L.csa2_index_score_topk_workspace_size(1, 1 << 20, 2048, 2048) >= 2048 * 8 * 4
    assert L.csa2_hier_candidate_pool_workspace_size(1, 16384, 2048) == 0  # one CTA, registers
    assert L.csa2_hier_candidate_pool_workspace_size(1, 131072, 2048) >= 131072 * 8  # chunked
    assert L.csa2_hier_candidate_pool_workspace_size(4096, 33280, 2048) == 0  # one CTA per query
    assert L.csa2_sparse_attn_prefill_workspace_size(16, 64, 2048) >= 16 * 64 * 288
    # index + pool: the pool is the block list, so no separate block list is carved
    full = L.csa2_index_score_topk_workspace_size(1, 1 << 20, 0, 2048)
    fused = L.csa2_index_score_topk_pool_workspace_size(1, 1 << 20, 2048, 2048)
    assert 0 < fused <= full
