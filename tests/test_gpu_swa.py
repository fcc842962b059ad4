"""GPU-vs-oracle parity of the local sliding-window branch: the FP8 local-row encoding (every
finite bf16 value, bit-exact), and decode / prefill attention over the selected FP4 rows and the
window's FP8 local rows in one softmax (ring buffers, windows longer than the context, empty
selections, no window)."""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import check_attn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp4_kv_top_csa2_b300 import csa2 as c
    return c


def _bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def test_fp8_local_rows_bit_exact(csa2):
    bits = np.arange(1 << 16, dtype=np.uint16)
    f = (bits.astype(np.uint32) << 16).view(np.float32)
    bits = bits[np.isfinite(f)]
    n = bits.size // 512
    x = torch.from_numpy(bits[: n * 512].view(np.int16).reshape(n, 512).copy()).view(torch.bfloat16)
    out = torch.empty((n, 512), dtype=torch.uint8, device="cuda")
    csa2.csa2_swa_kv_quant_fp8(x.cuda(), out)
    assert np.array_equal(out.cpu().numpy(), oracle.fp8_quant(_bits(x)))
    # scattered destination rows
    rows = torch.randperm(200, generator=torch.Generator().manual_seed(1))[:n].to(torch.int64)
    dst = torch.zeros((200, 512), dtype=torch.uint8, device="cuda")
    csa2.csa2_swa_kv_quant_fp8(x.cuda(), dst, out_rows=rows.cuda())
    assert np.array_equal(dst.cpu().numpy()[rows.numpy()], oracle.fp8_quant(_bits(x)))


def _cache(lengths, seed):
    g = torch.Generator().manual_seed(seed)
    sigma = 10.0 ** (torch.rand(512, generator=g) * 2 - 1)
    x = (torch.randn(sum(lengths), 512, generator=g) * sigma).to(torch.bfloat16)
    return x, sigma, g


@pytest.mark.parametrize("lengths,H,topk,n_win,ring", [
    ([3000, 500, 40], 64, 2048, 128, 128),    # a sequence shorter than the window
    ([5000, 100], 16, 512, 33, 64),           # ring larger than the window
    ([4000], 64, 100, 1, 1),                  # the current token's local row only
    ([2000, 3000], 64, 2048, 200, 256),
    ([700], 64, 33, 0, 16),                   # no window: the plain sparse attention
    ([4000, 3500, 3000, 2500, 2100], 16, 2048, 100, 128),  # 128-row tiles, 16 heads
])
def test_swa_decode(csa2, lengths, H, topk, n_win, ring):
    x, sigma, g = _cache(lengths, sum(lengths) + n_win)
    B = len(lengths)
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int64)
    codes = torch.empty((x.shape[0], 256), dtype=torch.uint8, device="cuda")
    sf = torch.empty((x.shape[0], 32), dtype=torch.uint8, device="cuda")
    csa2.csa2_kv_quant_fp4(x.cuda(), codes, sf)
    q = torch.randn(B, H, 512, generator=g).to(torch.bfloat16)
    idx = torch.full((B, topk), -1, dtype=torch.int32)
    for b, L in enumerate(lengths):
        k = min(topk, L)
        idx[b, :k] = torch.randperm(L, generator=g)[:k].to(torch.int32)
    idx[:, 5::13] = -1
    loc = (torch.randn(B * ring, 512, generator=g) * sigma).to(torch.bfloat16)
    swa = torch.empty((B * ring, 512), dtype=torch.uint8, device="cuda")
    csa2.csa2_swa_kv_quant_fp8(loc.cuda(), swa)
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), device="cuda")
    scale = 1 / math.sqrt(512)
    ws = csa2.workspace(csa2.csa2_sparse_swa_attn_decode_workspace_size(B, H, topk, n_win))
    csa2.csa2_sparse_swa_attn_decode(q.cuda(), codes, sf, cu.cuda(), idx.cuda(), swa, ring, n_win,
                                     scale, out, lse, ws=ws)
    ref = oracle.sparse_swa_attn_queries(_bits(q), np.arange(B), np.array(lengths),
                                         codes.cpu().numpy(), sf.cpu().numpy(), cu.numpy(),
                                         idx.numpy(), swa.cpu().numpy(), ring, n_win, scale)
    ob, lh = _bits(out), lse.cpu().numpy()
    for b in range(B):
        check_attn(ob[b], lh[b], ref[b][0], ref[b][1], oracle.double_to_bf16(ref[b][0]), f"seq {b}")
    if n_win == 0:  # bit for bit the plain call
        out2, lse2 = torch.empty_like(out), torch.empty_like(lse)
        ws2 = csa2.workspace(csa2.csa2_sparse_attn_decode_workspace_size(B, H, topk))
        csa2.csa2_sparse_attn_decode(q.cuda(), codes, sf, cu.cuda(), idx.cuda(), scale, out2, lse2,
                                     ws=ws2)
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
        assert torch.equal(lse, lse2)


@pytest.mark.parametrize("P0,T,H,topk,n_win", [
    (3000, 5, 64, 300, 64),     # one window tile
    (3000, 4, 64, 2048, 130),   # three window tiles, 16 selected tiles
    (40, 6, 16, 40, 100),       # windows longer than what the first tokens see
    (500, 3, 64, 90, 1),
])
def test_swa_prefill(csa2, P0, T, H, topk, n_win):
    L = P0 + T
    x, sigma, g = _cache([L], P0 + T + n_win)
    cu = torch.tensor([0, L], dtype=torch.int64)
    codes = torch.empty((L, 256), dtype=torch.uint8, device="cuda")
    sf = torch.empty((L, 32), dtype=torch.uint8, device="cuda")
    csa2.csa2_kv_quant_fp4(x.cuda(), codes, sf)
    q = torch.randn(T, H, 512, generator=g).to(torch.bfloat16)
    vis = torch.arange(P0 + 1, P0 + 1 + T, dtype=torch.int32)
    idx = torch.stack([torch.randperm(int(v), generator=g)[:topk] if v >= topk else
                       torch.cat([torch.randperm(int(v), generator=g),
                                  torch.full((topk - int(v),), -1)])
                       for v in vis]).to(torch.int32)
    idx[:, 2::11] = -1
    ring = n_win + T - 1
    loc = (torch.randn(ring, 512, generator=g) * sigma).to(torch.bfloat16)
    swa = torch.empty((ring, 512), dtype=torch.uint8, device="cuda")
    csa2.csa2_swa_kv_quant_fp8(loc.cuda(), swa)
    q_seq = torch.zeros(T, dtype=torch.int32)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), device="cuda")
    scale = 1 / math.sqrt(512)
    csa2.csa2_sparse_swa_attn_prefill(q.cuda(), q_seq.cuda(), vis.cuda(), codes, sf, cu.cuda(),
                                      idx.cuda(), swa, ring, n_win, scale, out, lse)
    ref = oracle.sparse_swa_attn_queries(_bits(q), q_seq.numpy(), vis.numpy(), codes.cpu().numpy(),
                                         sf.cpu().numpy(), cu.numpy(), idx.numpy(),
                                         swa.cpu().numpy(), ring, n_win, scale,
                                         quantize_query=True)
    ob, lh = _bits(out), lse.cpu().numpy()
    for i in range(T):
        check_attn(ob[i], lh[i], ref[i][0], ref[i][1], oracle.double_to_bf16(ref[i][0]), f"tok {i}")


def test_swa_rejects_bad_windows(csa2):
    x = torch.zeros((1, 8, 512), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((10, 256), dtype=torch.uint8, device="cuda")
    s = torch.zeros((10, 32), dtype=torch.uint8, device="cuda")
    cu = torch.tensor([0, 10], dtype=torch.int64, device="cuda")
    idx = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    swa = torch.zeros((4, 512), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(x)
    for ring, n_win, status in ((4, 5, -1), (0, 0, -1), (4, -1, -1)):
        with pytest.raises(csa2.Csa2Error) as ei:
            csa2.csa2_sparse_swa_attn_decode(x, c, s, cu, idx, swa, ring, n_win, 0.1, out)
        assert ei.value.status == status
    xb = torch.zeros((1, 80, 512), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(csa2.Csa2Error) as ei:  # more than 64 heads: no window support
        csa2.csa2_sparse_swa_attn_decode(xb, c, s, cu, idx, swa, 4, 2, 0.1, torch.empty_like(xb))
    assert ei.value.status == -2
