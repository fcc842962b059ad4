"""Thin Python binding of the CSA2 C ABI (include/csa2.h): argument marshalling only.

Every function takes torch CUDA tensors (device memory the caller owns), passes their pointers,
sizes and the current CUDA stream to the C entry point of the same name, and raises Csa2Error on
a non-zero status.  All arithmetic of the path runs in the CUDA kernels of libcsa2.so; there is
no CPU or PyTorch fallback: if the library is missing, importing this module fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

CSA2_BF16 = 0
CSA2_E4M3 = 1
D = 512


class Csa2Error(RuntimeError):
    def __init__(self, name: str, status: int, msg: str):
        super().__init__(f"{name} failed: {msg} (status {status})")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libcsa2.so not built ({LIB_PATH}); run python -m fp4_kv_top_csa2_b300.build")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, SZ, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    sig = {
        "csa2_error_string": (ctypes.c_char_p, [I]),
        "csa2_kv_quant_fp4": (I, [P, I64, I, P, P, P, P]),
        "csa2_index_score_topk_workspace_size": (SZ, [I, I64, I, I]),
        "csa2_index_score_topk": (I, [P, I, P, I, I, I, P, I, I64, P, P, I, P, P, I64, P, I, I, P,
                                      P, P, SZ, P]),
        "csa2_index_score_topk_reindex_noalloc": (I, [P, I, P, I, I, I, P, I, I64, P, P, I, P, P,
                                                      I64, P, I, I, P, P]),
        "csa2_index_block_max": (I, [P, I, P, I, I, I, P, I, I64, P, P, I, P, P, I64, P, P]),
        "csa2_index_score_topk_pool_workspace_size": (SZ, [I, I64, I, I]),
        "csa2_index_score_topk_pool": (I, [P, I, P, I, I, I, P, I, I64, P, P, I, P, P, I64, I, P,
                                           P, I, I, P, P, SZ, P, P]),
        "csa2_hier_candidate_pool_workspace_size": (SZ, [I, I64, I]),
        "csa2_hier_candidate_pool": (I, [P, I, P, I64, I, I, P, P, SZ, P]),
        "csa2_sparse_attn_decode_workspace_size": (SZ, [I, I, I]),
        "csa2_sparse_attn_decode": (I, [P, I, I, P, P, P, P, I, F, P, P, P, SZ, P]),
        "csa2_sparse_attn_prefill_workspace_size": (SZ, [I, I, I]),
        "csa2_sparse_attn_prefill": (I, [P, I, I, P, P, P, P, I, P, I, F, P, P, P, SZ, P]),
        "csa2_index_keys_from_kv": (I, [P, P, I64, P, P, I, P, P, P]),
        "csa2_sparse_attn_prefill_fp4pv": (I, [P, I, I, P, P, P, P, I, P, I, F, P, P, P]),
        "csa2_swa_kv_quant_fp8": (I, [P, I64, I, P, P, P]),
        "csa2_sparse_swa_attn_decode_workspace_size": (SZ, [I, I, I, I]),
        "csa2_sparse_swa_attn_decode": (I, [P, I, I, P, P, P, P, I, P, I, I, F, P, P, P, SZ, P]),
        "csa2_sparse_swa_attn_prefill_workspace_size": (SZ, [I, I, I, I]),
        "csa2_sparse_swa_attn_prefill": (I, [P, I, I, P, P, P, P, P, I, P, I, P, I, I, F, P, P,
                                             P, SZ, P]),
        "csa2_device_status": (I, [P, I, P]),
        "csa2_kernel_launches": (ctypes.c_uint64, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _event(ev):
    if ev is None:
        return None
    if not ev.cuda_event:
        raise ValueError("pool_event has no CUDA event yet: record it once before passing it")
    return ctypes.c_void_p(ev.cuda_event)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(name: str, status: int):
    if status != 0:
        raise Csa2Error(name, status, lib.csa2_error_string(status).decode())


def workspace(nbytes: int, device=None) -> torch.Tensor | None:
    """Caller-side workspace allocation (torch), 256-byte aligned by the caching allocator."""
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")


def _ws(ws):
    return (None, 0) if ws is None else (ctypes.c_void_p(ws.data_ptr()), ws.numel())


# --------------------------------------------------------------------------------------------
def csa2_kv_quant_fp4(x_bf16, codes, sf, out_rows=None, stream=None):
    n, d = x_bf16.shape
    _check("csa2_kv_quant_fp4", lib.csa2_kv_quant_fp4(_ptr(x_bf16), n, d, _ptr(out_rows),
                                                      _ptr(codes), _ptr(sf), _stream(stream)))


def csa2_index_score_topk_workspace_size(nq, max_vis, n_cand_blocks, topk):
    return lib.csa2_index_score_topk_workspace_size(nq, max_vis, n_cand_blocks, topk)


def csa2_index_score_topk(q_idx, q_dtype, w, k_idx, cu_ctx, q_seq, q_vis, max_vis, topk, out_idx,
                          k_scale=None, cand_blocks=None, out_block_max=None, ws=None,
                          stream=None):
    nq, Hi, Di = q_idx.shape
    B = cu_ctx.numel() - 1
    n_cand = 0 if cand_blocks is None else cand_blocks.shape[1]
    wp, wn = _ws(ws)
    _check("csa2_index_score_topk", lib.csa2_index_score_topk(
        _ptr(q_idx), q_dtype, _ptr(w), nq, Hi, Di, _ptr(k_idx), q_dtype, k_idx.shape[0],
        _ptr(k_scale),
        _ptr(cu_ctx), B, _ptr(q_seq), _ptr(q_vis), max_vis, _ptr(cand_blocks), n_cand, topk,
        _ptr(out_idx), _ptr(out_block_max), wp, wn, _stream(stream)))


def csa2_index_score_topk_reindex_noalloc(q_idx, q_dtype, w, k_idx, cu_ctx, q_seq, q_vis, max_vis,
                                          topk, out_idx, cand_blocks, k_scale=None, stream=None):
    """Reindex selection with the library's own fixed scratch (no workspace argument)."""
    nq, Hi, Di = q_idx.shape
    B = cu_ctx.numel() - 1
    _check("csa2_index_score_topk_reindex_noalloc", lib.csa2_index_score_topk_reindex_noalloc(
        _ptr(q_idx), q_dtype, _ptr(w), nq, Hi, Di, _ptr(k_idx), q_dtype, k_idx.shape[0],
        _ptr(k_scale), _ptr(cu_ctx), B, _ptr(q_seq), _ptr(q_vis), max_vis, _ptr(cand_blocks),
        cand_blocks.shape[1], topk, _ptr(out_idx), _stream(stream)))


def csa2_index_block_max(q_idx, q_dtype, w, k_idx, cu_ctx, q_seq, q_vis, max_vis, out_block_max,
                         k_scale=None, stream=None):
    """Full-mode block maxima only (the scan of csa2_index_score_topk without a selection)."""
    nq, Hi, Di = q_idx.shape
    B = cu_ctx.numel() - 1
    _check("csa2_index_block_max", lib.csa2_index_block_max(
        _ptr(q_idx), q_dtype, _ptr(w), nq, Hi, Di, _ptr(k_idx), q_dtype, k_idx.shape[0],
        _ptr(k_scale), _ptr(cu_ctx), B, _ptr(q_seq), _ptr(q_vis), max_vis, _ptr(out_block_max),
        _stream(stream)))


def csa2_index_score_topk_pool_workspace_size(nq, max_vis, topk, n_pool_blocks):
    return lib.csa2_index_score_topk_pool_workspace_size(nq, max_vis, topk, n_pool_blocks)


def csa2_index_score_topk_pool(q_idx, q_dtype, w, k_idx, cu_ctx, q_seq, q_vis, max_vis, topk,
                               out_idx, n_pool_blocks, out_pool_blocks, k_scale=None,
                               out_block_max=None, block_size=8, ws=None, stream=None,
                               pool_event=None):
    """Full-mode selection and the candidate pool of the same block maxima, in one call.
    `pool_event` (a torch.cuda.Event that has been recorded at least once, so that it exists) is
    recorded on the stream once the pool is complete."""
    nq, Hi, Di = q_idx.shape
    B = cu_ctx.numel() - 1
    wp, wn = _ws(ws)
    _check("csa2_index_score_topk_pool", lib.csa2_index_score_topk_pool(
        _ptr(q_idx), q_dtype, _ptr(w), nq, Hi, Di, _ptr(k_idx), q_dtype, k_idx.shape[0],
        _ptr(k_scale), _ptr(cu_ctx), B, _ptr(q_seq), _ptr(q_vis), max_vis, topk, _ptr(out_idx),
        _ptr(out_block_max), block_size, n_pool_blocks, _ptr(out_pool_blocks), wp, wn,
        _stream(stream), _event(pool_event)))


def csa2_hier_candidate_pool_workspace_size(nq, max_blocks, n_pool_blocks):
    return lib.csa2_hier_candidate_pool_workspace_size(nq, max_blocks, n_pool_blocks)


def csa2_hier_candidate_pool(block_max, q_vis, n_pool_blocks, out_pool_blocks, block_size=8,
                             ws=None, stream=None):
    nq, max_blocks = block_max.shape
    wp, wn = _ws(ws)
    _check("csa2_hier_candidate_pool", lib.csa2_hier_candidate_pool(
        _ptr(block_max), nq, _ptr(q_vis), max_blocks, block_size, n_pool_blocks,
        _ptr(out_pool_blocks), wp, wn, _stream(stream)))


def csa2_sparse_attn_decode_workspace_size(B, H, topk):
    return lib.csa2_sparse_attn_decode_workspace_size(B, H, topk)


def csa2_sparse_attn_decode(q_bf16, codes, sf, cu_ctx, idx, softmax_scale, out_bf16, lse=None,
                            ws=None, stream=None):
    B, H, _ = q_bf16.shape
    topk = idx.shape[1]
    wp, wn = _ws(ws)
    _check("csa2_sparse_attn_decode", lib.csa2_sparse_attn_decode(
        _ptr(q_bf16), B, H, _ptr(codes), _ptr(sf), _ptr(cu_ctx), _ptr(idx), topk,
        float(softmax_scale), _ptr(out_bf16), _ptr(lse), wp, wn, _stream(stream)))


def csa2_sparse_attn_prefill_workspace_size(T, H, topk):
    return lib.csa2_sparse_attn_prefill_workspace_size(T, H, topk)


def csa2_sparse_attn_prefill(q_bf16, q_seq, codes, sf, cu_ctx, idx, softmax_scale, out_bf16,
                             lse=None, ws=None, stream=None):
    T, H, _ = q_bf16.shape
    topk = idx.shape[1]
    B = cu_ctx.numel() - 1
    wp, wn = _ws(ws)
    _check("csa2_sparse_attn_prefill", lib.csa2_sparse_attn_prefill(
        _ptr(q_bf16), T, H, _ptr(q_seq), _ptr(codes), _ptr(sf), _ptr(cu_ctx), B, _ptr(idx), topk,
        float(softmax_scale), _ptr(out_bf16), _ptr(lse), wp, wn, _stream(stream)))


def csa2_sparse_attn_prefill_fp4pv(q_bf16, q_seq, codes, sf, cu_ctx, idx, softmax_scale,
                                   out_bf16, lse=None, stream=None):
    """Prefill attention with the probability-value product in block-scaled FP4 too."""
    T, H, _ = q_bf16.shape
    topk = idx.shape[1]
    B = cu_ctx.numel() - 1
    _check("csa2_sparse_attn_prefill_fp4pv", lib.csa2_sparse_attn_prefill_fp4pv(
        _ptr(q_bf16), T, H, _ptr(q_seq), _ptr(codes), _ptr(sf), _ptr(cu_ctx), B, _ptr(idx), topk,
        float(softmax_scale), _ptr(out_bf16), _ptr(lse), _stream(stream)))


def csa2_index_keys_from_kv(codes, sf, w_bf16, k_idx, k_scale, rows=None, n_rows=None,
                            stream=None):
    """Index keys (E4M3) and their per-row scales derived from the FP4 cache rows."""
    n = n_rows if n_rows is not None else (rows.numel() if rows is not None else codes.shape[0])
    _check("csa2_index_keys_from_kv", lib.csa2_index_keys_from_kv(
        _ptr(codes), _ptr(sf), n, _ptr(rows), _ptr(w_bf16), w_bf16.shape[0], _ptr(k_idx),
        _ptr(k_scale), _stream(stream)))


def csa2_swa_kv_quant_fp8(x_bf16, swa_kv, out_rows=None, stream=None):
    n, d = x_bf16.shape
    _check("csa2_swa_kv_quant_fp8", lib.csa2_swa_kv_quant_fp8(_ptr(x_bf16), n, d, _ptr(out_rows),
                                                              _ptr(swa_kv), _stream(stream)))


def csa2_sparse_swa_attn_decode_workspace_size(B, H, topk, n_win):
    return lib.csa2_sparse_swa_attn_decode_workspace_size(B, H, topk, n_win)


def csa2_sparse_swa_attn_decode(q_bf16, codes, sf, cu_ctx, idx, swa_kv, ring, n_win,
                                softmax_scale, out_bf16, lse=None, ws=None, stream=None):
    B, H, _ = q_bf16.shape
    topk = idx.shape[1]
    wp, wn = _ws(ws)
    _check("csa2_sparse_swa_attn_decode", lib.csa2_sparse_swa_attn_decode(
        _ptr(q_bf16), B, H, _ptr(codes), _ptr(sf), _ptr(cu_ctx), _ptr(idx), topk, _ptr(swa_kv),
        ring, n_win, float(softmax_scale), _ptr(out_bf16), _ptr(lse), wp, wn, _stream(stream)))


def csa2_sparse_swa_attn_prefill_workspace_size(T, H, topk, n_win):
    return lib.csa2_sparse_swa_attn_prefill_workspace_size(T, H, topk, n_win)


def csa2_sparse_swa_attn_prefill(q_bf16, q_seq, q_vis, codes, sf, cu_ctx, idx, swa_kv, ring,
                                 n_win, softmax_scale, out_bf16, lse=None, ws=None, stream=None):
    T, H, _ = q_bf16.shape
    topk = idx.shape[1]
    B = cu_ctx.numel() - 1
    wp, wn = _ws(ws)
    _check("csa2_sparse_swa_attn_prefill", lib.csa2_sparse_swa_attn_prefill(
        _ptr(q_bf16), T, H, _ptr(q_seq), _ptr(q_vis), _ptr(codes), _ptr(sf), _ptr(cu_ctx), B,
        _ptr(idx), topk, _ptr(swa_kv), ring, n_win, float(softmax_scale), _ptr(out_bf16),
        _ptr(lse), wp, wn, _stream(stream)))


def csa2_device_status(reset=True, stream=None) -> int:
    v = ctypes.c_int(0)
    _check("csa2_device_status", lib.csa2_device_status(ctypes.byref(v), int(reset),
                                                        _stream(stream)))
    return v.value


def kernel_launches() -> int:
    """Kernels enqueued by libcsa2.so in this process so far."""
    return int(lib.csa2_kernel_launches())
