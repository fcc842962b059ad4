"""Seeded synthetic inputs for the CSA2 hot path (shared by tests, smoke and bench).

This module only draws random numbers and lays them out; it contains none of the method's
arithmetic (no quantisation rule, no score, no selection, no attention).  Index keys/queries in
FP8 are produced with torch's own float32 -> float8_e4m3fn conversion, which is input
preparation, not part of the path under test.

Workloads (all seeded, torch CPU generator):
  * main-KV latent rows: N(0,1) * sigma_c per channel, sigma_c = 10**U(-1, 1) (log-uniform over
    [0.1, 10]), one sigma vector per workload, cast to bf16 (rows are then quantised to FP4 by
    the path itself);
  * index keys and index queries: N(0,1), as bf16 (dim 64) or FP8 E4M3 (dim 128);
  * indexer head weights: U(0,1) fp32;
  * attention queries: N(0,1) bf16, [heads, 512];
  * ragged decode: per-sequence context lengths U{lo..hi}; a fraction of index-key positions are
    near duplicates of a random earlier position of the same sequence (its float key plus
    N(0, 1e-3) noise before the FP8 cast), which yields exact FP8 ties and 1-ulp near ties;
  * local sliding-window rows (per layer): N(0,1) * sigma_c bf16, like the main-KV rows, for the
    ring buffer as it stands before the step and for the step's new tokens.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

BF16 = 0
E4M3 = 1
D = 512
BLOCK = 8


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "decode" | "hier" | "prefill"
    B: int = 1
    L: tuple = (4096,)  # context length per sequence (decode/hier); cached prefix P0 for prefill
    T: int = 0  # prefill: new query tokens appended after the cached prefix
    H: int = 64
    Hi: int = 8
    Di: int = 128
    idx_dtype: int = E4M3
    topk: int = 2048
    n_pool_blocks: int = 2048
    modes: tuple = ("full",)
    dup_frac: float = 0.0
    ragged: tuple | None = None  # (lo, hi) for ragged lengths drawn per sequence
    n_win: int = 0  # local sliding window per layer (0: none)
    seed: int = 0
    extra: dict = field(default_factory=dict)


# The five workloads of the hot path, by what they are.
WORKLOADS = {
    "decode_b1_l4096_bf16idx": Workload(
        "decode_b1_l4096_bf16idx", "decode", B=1, L=(4096,), H=16, Hi=4, Di=64, idx_dtype=BF16,
        topk=512),
    "decode_b8_l65536": Workload("decode_b8_l65536", "decode", B=8, L=(65536,) * 8, H=64),
    "decode_ragged_b32": Workload("decode_ragged_b32", "decode", B=32, ragged=(8192, 131072),
                                  dup_frac=0.1, H=64),
    "hier_decode_l1m": Workload(
        "hier_decode_l1m", "hier", B=1, L=(1 << 20,), H=64,
        modes=("full", "reindex", "reindex", "reindex", "reuse", "reuse")),
    "prefill_t4096_p262144": Workload("prefill_t4096_p262144", "prefill", B=1, L=(262144,),
                                      T=4096, H=64),
    # chunked prefill through the hierarchical indexer: the first Full layer builds a 2,048-block
    # candidate pool per query token, three Reindex layers rescore it, two Reuse layers reuse
    # the hierarchical decoder with every layer's local sliding window (128 FP8 local rows)
    "hier_decode_l1m_swa128": Workload(
        "hier_decode_l1m_swa128", "hier", B=1, L=(1 << 20,), H=64,
        modes=("full", "reindex", "reindex", "reindex", "reuse", "reuse"), n_win=128),
    "prefill_hier_t4096_p262144": Workload(
        "prefill_hier_t4096_p262144", "prefill", B=1, L=(262144,), T=4096, H=64,
        modes=("full", "reindex", "reindex", "reindex", "reuse", "reuse")),
}


def scaled(w: Workload, **kw) -> Workload:
    """A smaller (or otherwise changed) copy of a workload with the same structure."""
    return replace(w, **kw)


def _lengths(w: Workload, g: torch.Generator):
    if w.ragged is not None:
        lo, hi = w.ragged
        return [int(x) for x in torch.randint(lo, hi + 1, (w.B,), generator=g)]
    return [int(x) for x in w.L]


def _kv_rows(n: int, sigma: torch.Tensor, g: torch.Generator, chunk: int = 1 << 18):
    out = torch.empty((n, D), dtype=torch.bfloat16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = (torch.randn((e - s, D), generator=g) * sigma).to(torch.bfloat16)
    return out


def _index_vectors(shape, dtype: int, g: torch.Generator):
    x = torch.randn(shape, generator=g)
    if dtype == BF16:
        return x.to(torch.bfloat16)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def _index_keys(lengths, w: Workload, g: torch.Generator, chunk: int = 1 << 18):
    n = sum(lengths)
    kf = torch.empty((n, w.Di), dtype=torch.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        kf[s:e] = torch.randn((e - s, w.Di), generator=g)
    if w.dup_frac > 0:
        base = 0
        src_all, dst_all = [], []
        for L in lengths:
            n_dup = int(round(w.dup_frac * (L - 1)))
            dst = torch.randperm(L - 1, generator=g)[:n_dup] + 1  # positions 1..L-1
            # earlier source position, uniform in [0, dst)
            src = (torch.rand(n_dup, generator=g) * dst.to(torch.float64)).floor().to(torch.int64)
            src_all.append(src + base)
            dst_all.append(dst + base)
            base += L
        src = torch.cat(src_all)
        dst = torch.cat(dst_all)
        noise = torch.randn((dst.numel(), w.Di), generator=g) * 1e-3
        kf[dst] = kf[src] + noise
    if w.idx_dtype == BF16:
        return kf.to(torch.bfloat16)
    return kf.to(torch.float8_e4m3fn).view(torch.uint8)


def make_inputs(w: Workload, with_kv: bool = True) -> dict:
    """Draw every input of workload `w` (torch CPU tensors).

    Returns a dict with
      kv_bf16 [rows, 512] bf16, cu_ctx [B+1] int64, k_idx [rows, Di] (bf16 / uint8 E4M3 bits),
      lengths (list), and per layer a dict in "layers": q_idx [nq, Hi, Di], w [nq, Hi] fp32,
      q_attn [nq, H, 512] bf16, plus q_seq / q_vis int32 [nq] and max_vis.
    Decode: nq = B, q_vis = L_b (the cache already holds the current token).  Prefill: the
    cache holds P0 + T rows (the T new rows are part of the step's quantisation), query i sees
    positions [0, P0 + i].
    """
    g = torch.Generator().manual_seed(w.seed)
    lengths = _lengths(w, g)
    if w.kind == "prefill":
        lengths = [lengths[0] + w.T]
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    cu_ctx = torch.tensor(cu, dtype=torch.int64)
    sigma = 10.0 ** (torch.rand(D, generator=g) * 2.0 - 1.0)
    out = {"workload": w, "lengths": lengths, "cu_ctx": cu_ctx, "sigma": sigma}
    out["kv_bf16"] = _kv_rows(cu[-1], sigma, g) if with_kv else None
    out["k_idx"] = _index_keys(lengths, w, g)
    if w.kind == "prefill":
        nq = w.T
        P0 = lengths[0] - w.T
        q_seq = torch.zeros(nq, dtype=torch.int32)
        q_vis = torch.arange(P0 + 1, P0 + 1 + nq, dtype=torch.int32)
    else:
        nq = w.B
        q_seq = torch.arange(nq, dtype=torch.int32)
        q_vis = torch.tensor(lengths, dtype=torch.int32)
    out["q_seq"] = q_seq
    out["q_vis"] = q_vis
    out["max_vis"] = int(q_vis.max()) if nq else 0
    layers = []
    ring = swa_ring(w)
    for mode in w.modes:
        layer = {"mode": mode}
        if mode in ("full", "reindex"):
            layer["q_idx"] = _index_vectors((nq, w.Hi, w.Di), w.idx_dtype, g)
            layer["w"] = torch.rand((nq, w.Hi), generator=g)
        layer["q_attn"] = torch.randn((nq, w.H, D), generator=g).to(torch.bfloat16)
        if w.n_win:
            layer["swa_bf16"] = _kv_rows(len(lengths) * ring, sigma, g)  # the ring before
            layer["swa_new"] = _kv_rows(nq, sigma, g)                    # this step's tokens
        layers.append(layer)
    out["layers"] = layers
    out["swa_ring"] = ring
    return out


def swa_ring(w: Workload) -> int:
    """Local rows kept per sequence: the window, plus the chunk's own tokens for a prefill."""
    if not w.n_win:
        return 1
    return w.n_win + (w.T - 1 if w.kind == "prefill" else 0)


def swa_new_rows(inputs: dict) -> torch.Tensor:
    """Ring rows the step's new tokens' local rows go to (query token n: sequence q_seq[n] at
    position q_vis[n] - 1)."""
    ring = inputs["swa_ring"]
    pos = inputs["q_vis"].to(torch.int64) - 1
    return inputs["q_seq"].to(torch.int64) * ring + pos % ring


def new_token_rows(inputs: dict) -> torch.Tensor:
    """Cache rows written by one step: the last row of each sequence (decode), or the T new
    rows after the cached prefix (prefill)."""
    w = inputs["workload"]
    cu = inputs["cu_ctx"]
    if w.kind == "prefill":
        return torch.arange(int(cu[1]) - w.T, int(cu[1]), dtype=torch.int64)
    return cu[1:] - 1


def to_numpy_bits(t: torch.Tensor):
    """bf16 -> uint16 bit patterns; uint8 stays uint8; other dtypes as numpy."""
    import numpy as np
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    return t.contiguous().numpy()
