"""CPU oracle of the CSA2 hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of ``bench.py``
may import this package.  It wraps ``csa2_oracle.c`` (plain single-threaded C, double
accumulation) through ctypes and shares nothing with the CUDA library in
``fp4_kv_top_csa2_b300``: no header, table, helper or generated constant.

Sources (prose only on the pages):
  * DeepSeek-V4.1-Flash model card, Introduction, paragraph "Compressed Sparse Attention 2 (CSA2)"
    -- Full / Reindex / Reuse modes, hierarchical indexer pool, FP4 main KV (E2M1 + one E4M3
    scale per 16 channels).
  * "DeepSeek V4.1-Flash" (aiwiki.ai), section "Compressed Sparse Attention 2" -- per-mode
    recomputation, block selection by maximum index score, pool of 2,048 blocks x 8 positions,
    Reindex selecting 512, every layer's own local sliding-window keys and values; section
    "KV-cache formats and bounded replay" -- FP4 main global KV, FP8 local sliding-window KV.

Every batch-level function below loops over queries in Python and calls the per-query C
routines; there is no blocking, fusion or reordering beyond the definitions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa2_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

BF16 = 0
E4M3 = 1
D = 512


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (no fast-math, no FP contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared",
               "-o", _LIB_PATH, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    i32 = ctypes.c_int
    lib.orc_e2m1_value.restype = ctypes.c_double
    lib.orc_e2m1_value.argtypes = [i32]
    lib.orc_e4m3_value.restype = ctypes.c_double
    lib.orc_e4m3_value.argtypes = [i32]
    lib.orc_e2m1_encode.restype = i32
    lib.orc_e2m1_encode.argtypes = [ctypes.c_float]
    lib.orc_e4m3_encode.restype = i32
    lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
    lib.orc_double_to_bf16.restype = ctypes.c_uint16
    lib.orc_double_to_bf16.argtypes = [ctypes.c_double]
    lib.orc_kv_quant_fp4.argtypes = [P, i64, i32, P, P]
    lib.orc_kv_dequant_fp4.argtypes = [P, P, i64, i32, P]
    lib.orc_index_scores.argtypes = [P, i32, P, i32, i32, P, P, P, i64, P]
    lib.orc_topk.restype = i32
    lib.orc_topk.argtypes = [P, P, i64, i32, P]
    lib.orc_block_max.argtypes = [P, i64, i32, P]
    lib.orc_candidate_pool.restype = i32
    lib.orc_candidate_pool.argtypes = [P, i64, i32, P]
    lib.orc_sparse_attn.argtypes = [P, i32, i32, P, P, P, i32, ctypes.c_double, P, P]
    lib.orc_fp8_quant.argtypes = [P, i64, P]
    lib.orc_sparse_swa_attn.argtypes = [P, i32, i32, P, P, P, i32, P, i32, ctypes.c_double, P, P]
    lib.orc_index_keys_from_kv.argtypes = [P, P, i64, i32, P, i32, P, P]
    lib.orc_attn_fp4pv.argtypes = [P, i32, i32, P, P, P, i32, ctypes.c_double, P, P]
    lib.orc_bf16_to_double.argtypes = [P, i64, P]
    lib.orc_double_to_bf16_array.argtypes = [P, i64, P]
    _lib = lib
    return lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


# ----------------------------------------------------------------------------------------------
# Number formats
# ----------------------------------------------------------------------------------------------
def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return _load().orc_e4m3_value(int(code))


def e2m1_encode(v: float) -> int:
    return _load().orc_e2m1_encode(float(v))


def e4m3_encode(v: float) -> int:
    return _load().orc_e4m3_encode(float(v))


def double_to_bf16(x: np.ndarray) -> np.ndarray:
    """float64 array -> bf16 bit patterns (uint16), round to nearest even in one step."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().orc_double_to_bf16_array(_p(x), x.size, _p(out))
    return out


def bf16_to_double(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint16)
    out = np.empty(x.shape, dtype=np.float64)
    _load().orc_bf16_to_double(_p(x), x.size, _p(out))
    return out


# ----------------------------------------------------------------------------------------------
# a1: FP4 main-KV quantisation
# ----------------------------------------------------------------------------------------------
def kv_quant_fp4(x_bf16: np.ndarray):
    """x: [n, d] uint16 (bf16 bits) -> (codes [n, d/2] uint8, sf [n, d/16] uint8)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    n, d = x.shape
    codes = np.zeros((n, d // 2), dtype=np.uint8)
    sf = np.zeros((n, d // 16), dtype=np.uint8)
    _load().orc_kv_quant_fp4(_p(x), n, d, _p(codes), _p(sf))
    return codes, sf


def kv_dequant_fp4(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    n = codes.shape[0]
    d = codes.shape[1] * 2
    out = np.empty((n, d), dtype=np.float64)
    _load().orc_kv_dequant_fp4(_p(codes), _p(sf), n, d, _p(out))
    return out


# ----------------------------------------------------------------------------------------------
# a2..a5: indexer scores, Top-K, block maxima, candidate pool
# ----------------------------------------------------------------------------------------------
def index_scores(q: np.ndarray, dtype: int, w: np.ndarray, k: np.ndarray, pos: np.ndarray,
                 k_scale: np.ndarray | None = None) -> np.ndarray:
    """Scores of one query q [Hi, Di] over key rows k[pos] (k = the sequence's rows)."""
    q = np.ascontiguousarray(q)
    w = np.ascontiguousarray(w, dtype=np.float32)
    k = np.ascontiguousarray(k)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    Hi, Di = q.shape
    out = np.empty(pos.shape[0], dtype=np.float32)
    ks = None if k_scale is None else np.ascontiguousarray(k_scale, dtype=np.float32)
    _load().orc_index_scores(_p(q), dtype, _p(w), Hi, Di, _p(k),
                             None if ks is None else _p(ks), _p(pos), pos.shape[0], _p(out))
    return out


def topk(scores: np.ndarray, pos: np.ndarray, K: int) -> np.ndarray:
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    out = np.empty(K, dtype=np.int32)
    _load().orc_topk(_p(scores), _p(pos), scores.shape[0], K, _p(out))
    return out


def block_max(scores: np.ndarray, bs: int = 8) -> np.ndarray:
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    n = scores.shape[0]
    out = np.empty((n + bs - 1) // bs, dtype=np.float32)
    if n:
        _load().orc_block_max(_p(scores), n, bs, _p(out))
    return out


def candidate_pool(bm: np.ndarray, n_pool: int) -> np.ndarray:
    bm = np.ascontiguousarray(bm, dtype=np.float32)
    out = np.empty(n_pool, dtype=np.int32)
    _load().orc_candidate_pool(_p(bm), bm.shape[0], n_pool, _p(out))
    return out


def candidate_positions(blocks: np.ndarray, vis: int, bs: int = 8) -> np.ndarray:
    """Positions of the given block ids (-1 ignored), clipped to [0, vis), in listed order."""
    b = np.asarray(blocks, dtype=np.int64)
    b = b[b >= 0]
    pos = (b[:, None] * bs + np.arange(bs, dtype=np.int64)[None, :]).reshape(-1)
    return pos[pos < vis]


def index_score_topk(q_idx, dtype, w, k_idx, cu_ctx, q_seq, q_vis, topk_k, cand_blocks=None,
                     k_scale=None, queries=None, block_size=8):
    """Batch form of csa2_index_score_topk for the queries listed in `queries` (default all).

    Returns a dict per query n: {"idx": [topk] int32, "pos": candidate positions,
    "scores": their fp32 scores, "bm": block maxima (Full mode only)}.
    """
    nq = q_idx.shape[0]
    queries = range(nq) if queries is None else queries
    res = {}
    for n in queries:
        b = int(q_seq[n])
        lo, hi = int(cu_ctx[b]), int(cu_ctx[b + 1])
        V = int(q_vis[n])
        k_seq = k_idx[lo:hi]
        ks = None if k_scale is None else k_scale[lo:hi]
        if cand_blocks is None:
            pos = np.arange(V, dtype=np.int64)
        else:
            pos = candidate_positions(cand_blocks[n], V, block_size)
        s = index_scores(q_idx[n], dtype, w[n], k_seq, pos, ks)
        r = {"pos": pos, "scores": s, "idx": topk(s, pos, topk_k)}
        if cand_blocks is None:
            r["bm"] = block_max(s, block_size)
        res[n] = r
    return res


def hier_candidate_pool(bm_rows, q_vis, n_pool_blocks, block_size=8, queries=None):
    """Batch form of csa2_hier_candidate_pool: bm_rows[n] holds the block maxima of query n."""
    out = {}
    queries = range(len(q_vis)) if queries is None else queries
    for n in queries:
        nb = (int(q_vis[n]) + block_size - 1) // block_size
        out[n] = candidate_pool(np.asarray(bm_rows[n][:nb]), n_pool_blocks)
    return out


# ----------------------------------------------------------------------------------------------
# a7 / a8: sparse attention
# ----------------------------------------------------------------------------------------------
def sparse_attn(q: np.ndarray, codes_seq: np.ndarray, sf_seq: np.ndarray, idx: np.ndarray,
                scale: float):
    """One query set q [H, d] float64 over the rows of one sequence; returns (out [H,d], lse [H])."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    H, d = q.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    codes_seq = np.ascontiguousarray(codes_seq, dtype=np.uint8)
    sf_seq = np.ascontiguousarray(sf_seq, dtype=np.uint8)
    out = np.empty((H, d), dtype=np.float64)
    lse = np.empty(H, dtype=np.float64)
    _load().orc_sparse_attn(_p(q), H, d, _p(codes_seq), _p(sf_seq), _p(idx), idx.shape[0],
                            float(scale), _p(out), _p(lse))
    return out, lse


def sparse_attn_decode(q_bf16, codes, sf, cu_ctx, idx, scale, seqs=None):
    """q_bf16 [B, H, d] uint16; idx [B, K].  Returns {b: (out float64 [H,d], lse [H])}."""
    res = {}
    seqs = range(q_bf16.shape[0]) if seqs is None else seqs
    for b in seqs:
        lo, hi = int(cu_ctx[b]), int(cu_ctx[b + 1])
        res[b] = sparse_attn(bf16_to_double(q_bf16[b]), codes[lo:hi], sf[lo:hi], idx[b], scale)
    return res


def quantize_query_fp4(q_bf16_rows: np.ndarray) -> np.ndarray:
    """Prefill query: each (token, head) row quantised with the main-KV FP4 rule, dequantised."""
    c, s = kv_quant_fp4(q_bf16_rows)
    return kv_dequant_fp4(c, s)


def sparse_attn_prefill(q_bf16, q_seq, codes, sf, cu_ctx, idx, scale, tokens=None):
    """q_bf16 [T, H, d] uint16; idx [T, K].  Returns {i: (out, lse)} for the listed tokens."""
    res = {}
    tokens = range(q_bf16.shape[0]) if tokens is None else tokens
    for i in tokens:
        b = int(q_seq[i])
        lo, hi = int(cu_ctx[b]), int(cu_ctx[b + 1])
        qhat = quantize_query_fp4(np.ascontiguousarray(q_bf16[i]))
        res[i] = sparse_attn(qhat, codes[lo:hi], sf[lo:hi], idx[i], scale)
    return res


# ----------------------------------------------------------------------------------------------
# f1: the local sliding-window branch (FP8 local KV, one softmax over both sets of rows)
# ----------------------------------------------------------------------------------------------
def fp8_quant(x_bf16: np.ndarray) -> np.ndarray:
    """bf16 bits -> E4M3 bytes (round to nearest even, saturating at +-448, no scale)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().orc_fp8_quant(_p(x), x.size, _p(out))
    return out


def window_positions(vis: int, n_win: int) -> np.ndarray:
    """The positions of a query's local window: the last n_win of the vis positions it sees."""
    return np.arange(max(0, vis - n_win), vis, dtype=np.int64)


def sparse_swa_attn(q: np.ndarray, codes_seq, sf_seq, idx, loc_rows, scale):
    """One query set q [H, d] float64 over the selected FP4 rows of one sequence and the local
    E4M3 rows loc_rows [n_loc, d]: (out [H, d], lse [H])."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    H, d = q.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    loc = np.ascontiguousarray(loc_rows, dtype=np.uint8).reshape(-1, d)
    codes_seq = np.ascontiguousarray(codes_seq, dtype=np.uint8)
    sf_seq = np.ascontiguousarray(sf_seq, dtype=np.uint8)
    out = np.empty((H, d), dtype=np.float64)
    lse = np.empty(H, dtype=np.float64)
    _load().orc_sparse_swa_attn(_p(q), H, d, _p(codes_seq), _p(sf_seq), _p(idx), idx.shape[0],
                                _p(loc), loc.shape[0], float(scale), _p(out), _p(lse))
    return out, lse


def sparse_swa_attn_queries(q_bf16, q_seq, q_vis, codes, sf, cu_ctx, idx, swa_kv, ring, n_win,
                            scale, queries=None, quantize_query=False):
    """Batch form of the sparse + local-window attention calls.  Query n (sequence b = q_seq[n],
    visible length q_vis[n]) attends to its selected rows idx[n] and to the local rows of the
    last n_win visible positions, position t of sequence b at local row b * ring + t % ring.
    quantize_query: the prefill rule (the query quantised to FP4 first)."""
    res = {}
    queries = range(q_bf16.shape[0]) if queries is None else queries
    for n in queries:
        b = int(q_seq[n])
        lo, hi = int(cu_ctx[b]), int(cu_ctx[b + 1])
        win = window_positions(int(q_vis[n]), n_win)
        loc = swa_kv[b * ring + win % ring]
        qn = np.ascontiguousarray(q_bf16[n])
        q = quantize_query_fp4(qn) if quantize_query else bf16_to_double(qn)
        res[n] = sparse_swa_attn(q, codes[lo:hi], sf[lo:hi], idx[n], loc, scale)
    return res


# ----------------------------------------------------------------------------------------------
# f3: index keys derived from main-KV entries
# ----------------------------------------------------------------------------------------------
def index_keys_from_kv(codes: np.ndarray, sf: np.ndarray, W_bf16: np.ndarray):
    """FP4 rows (codes [n, d/2], sf [n, d/16]) and a bf16 projection W [Di, d] (uint16 bits) ->
    (keys [n, Di] E4M3 bytes, k_scale [n] fp32)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    W = np.ascontiguousarray(W_bf16, dtype=np.uint16)
    n, d = codes.shape[0], codes.shape[1] * 2
    Di = W.shape[0]
    keys = np.empty((n, Di), dtype=np.uint8)
    ks = np.empty(n, dtype=np.float32)
    _load().orc_index_keys_from_kv(_p(codes), _p(sf), n, d, _p(W), Di, _p(keys), _p(ks))
    return keys, ks


# ----------------------------------------------------------------------------------------------
# f4: the full-FP4 PV variant of prefill attention
# ----------------------------------------------------------------------------------------------
def attn_fp4pv(q: np.ndarray, codes_seq, sf_seq, idx, scale):
    """One token's FP4-dequantised query q [H, d] over its selected slots idx [K] (blocks of 16
    consecutive slots): (out [H, d], lse [H])."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    H, d = q.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    codes_seq = np.ascontiguousarray(codes_seq, dtype=np.uint8)
    sf_seq = np.ascontiguousarray(sf_seq, dtype=np.uint8)
    out = np.empty((H, d), dtype=np.float64)
    lse = np.empty(H, dtype=np.float64)
    _load().orc_attn_fp4pv(_p(q), H, d, _p(codes_seq), _p(sf_seq), _p(idx), idx.shape[0],
                           float(scale), _p(out), _p(lse))
    return out, lse


def sparse_attn_prefill_fp4pv(q_bf16, q_seq, codes, sf, cu_ctx, idx, scale, tokens=None):
    """Batch form of the full-FP4 PV prefill call: {i: (out, lse)} for the listed tokens."""
    res = {}
    tokens = range(q_bf16.shape[0]) if tokens is None else tokens
    for i in tokens:
        b = int(q_seq[i])
        lo, hi = int(cu_ctx[b]), int(cu_ctx[b + 1])
        qhat = quantize_query_fp4(np.ascontiguousarray(q_bf16[i]))
        res[i] = attn_fp4pv(qhat, codes[lo:hi], sf[lo:hi], idx[i], scale)
    return res
