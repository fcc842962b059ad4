"""GPU-vs-oracle parity of the full-FP4 PV variant of prefill attention
(csa2_sparse_attn_prefill_fp4pv): numerators and rows re-quantised to block-scaled FP4 along the
slots, blocks of 16 consecutive slots.

The re-quantised rows are exact on both sides.  A numerator code is decided from p / sc, where
the kernel's p comes from fp32 scores (tensor-core accumulation order) and the special-function
unit's 2^x, about 1e-6 relative from the oracle's exact value; where p / sc lies that close to an
E2M1 rounding boundary the two sides pick adjacent codes, which moves one slot's weight by one
E2M1 step for one head.  That happens for a few numerators in a hundred thousand.  So each token
must meet the attention tolerance of every other check (rel-L2 <= 1e-3 over the token, max-abs
<= max(2e-3, 1 bf16 ulp) per element, lse to 1e-4 relative) in all but at most two heads, and the
rel-L2 bound over the whole token always.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import ATTN_REL_L2, check_attn, bf16_bits_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa2():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp4_kv_top_csa2_b300 import csa2 as c
    return c


def _bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _check_token(ob, lh, ref_out, ref_lse, what, max_heads=2):
    rb = oracle.double_to_bf16(ref_out)
    g, r = bf16_bits_to_f64(ob), bf16_bits_to_f64(rb)
    nr = np.linalg.norm(r)
    rel = np.linalg.norm(g - r) / nr if nr > 0 else np.linalg.norm(g)
    assert rel <= ATTN_REL_L2, f"{what}: rel-L2 {rel:.3e}"
    bad = []
    for h in range(ob.shape[0]):
        try:
            check_attn(ob[h:h + 1], lh[h:h + 1], ref_out[h:h + 1], ref_lse[h:h + 1], rb[h:h + 1],
                       what)
        except AssertionError:
            bad.append(h)
    assert len(bad) <= max_heads, f"{what}: {len(bad)} heads outside the bounds: {bad[:8]}"
    return bad


@pytest.mark.parametrize("T,H,topk,n_rows", [(6, 64, 2048, 4000), (4, 16, 300, 3000),
                                              (5, 64, 130, 500), (3, 32, 17, 40),
                                              (2, 64, 4000, 5000)])
def test_fp4pv_prefill(csa2, T, H, topk, n_rows):
    g = torch.Generator().manual_seed(T * 1000 + topk)
    sigma = 10.0 ** (torch.rand(512, generator=g) * 2 - 1)
    x = (torch.randn(n_rows, 512, generator=g) * sigma).to(torch.bfloat16)
    q = torch.randn(T, H, 512, generator=g).to(torch.bfloat16)
    idx = torch.stack([torch.randperm(n_rows, generator=g)[:topk] for _ in range(T)]).to(torch.int32)
    idx[:, 3::11] = -1
    if T > 2:
        idx[2] = -1  # a token with no valid slot
    cu = torch.tensor([0, n_rows], dtype=torch.int64)
    q_seq = torch.zeros(T, dtype=torch.int32)
    codes = torch.empty((n_rows, 256), dtype=torch.uint8, device="cuda")
    sf = torch.empty((n_rows, 32), dtype=torch.uint8, device="cuda")
    csa2.csa2_kv_quant_fp4(x.cuda(), codes, sf)
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), device="cuda")
    scale = 1 / math.sqrt(512)
    csa2.csa2_sparse_attn_prefill_fp4pv(q.cuda(), q_seq.cuda(), codes, sf, cu.cuda(), idx.cuda(),
                                        scale, out, lse)
    ref = oracle.sparse_attn_prefill_fp4pv(_bits(q), q_seq.numpy(), codes.cpu().numpy(),
                                           sf.cpu().numpy(), cu.numpy(), idx.numpy(), scale)
    ob, lh = _bits(out), lse.cpu().numpy()
    for i in range(T):
        _check_token(ob[i], lh[i], ref[i][0], ref[i][1], f"tok {i}")


def test_fp4pv_full_size_prefill():
    """The full-FP4 PV variant on the chunked-prefill workload's own selection (4,096 tokens,
    2,048 rows each, 64 heads), 16 tokens checked."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp4_kv_top_csa2_b300 import csa2, synth
    from fp4_kv_top_csa2_b300.step import Step
    w = synth.WORKLOADS["prefill_t4096_p262144"]
    inp = synth.make_inputs(w)
    st = Step(inp)
    st.run()
    L = st.layers[0]
    out = torch.empty_like(L["out"])
    lse = torch.empty_like(L["lse"])
    csa2.csa2_sparse_attn_prefill_fp4pv(L["q_attn"], st.q_seq, st.codes, st.sf, st.cu_ctx,
                                        L["idx"], st.scale, out, lse)
    torch.cuda.synchronize()
    tokens = sorted(set(np.linspace(0, w.T - 1, 16).astype(int).tolist()))
    ref = oracle.sparse_attn_prefill_fp4pv(_bits(inp["layers"][0]["q_attn"]),
                                           inp["q_seq"].numpy(), st.codes.cpu().numpy(),
                                           st.sf.cpu().numpy(), inp["cu_ctx"].numpy(),
                                           L["idx"].cpu().numpy(), st.scale, tokens=tokens)
    ob, lh = _bits(out), lse.cpu().numpy()
    for i in tokens:
        _check_token(ob[i], lh[i], ref[i][0], ref[i][1], f"tok {i}")
