"""Full-size parity: the seven workloads at their stated sizes, run through the same Step (and so
the same launch configuration) that bench.py times, checked against the oracle.

Each check uses the GPU's own upstream result as the oracle's input where a step depends on an
earlier one (the pool is rebuilt by the oracle from the GPU's block maxima, attention is
recomputed by the oracle on the GPU's indices), so every call is judged on its own; the
upstream results are themselves checked against the oracle.  Chunked prefill is checked on 64
query tokens spread evenly over the chunk (first and last included): the oracle scores all 262,144+
visible positions for each of them.  The hierarchical prefill (a candidate pool per query token,
three Reindex and two Reuse layers) checks every layer's selection on the same 64 tokens and its
six attentions on 16 of them.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_attn, check_topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from fp4_kv_top_csa2_b300 import step, synth
    return step, synth


def _bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _np(t):
    if t.dtype == torch.bfloat16:
        return _bits(t)
    return t.cpu().contiguous().numpy()


def _check_cache(st, inp, rng):
    rows = inp["kv_bf16"].shape[0]
    sample = np.unique(np.concatenate([rng.integers(0, rows, 4000),
                                       st.new_rows.cpu().numpy()]))
    rc, rs = oracle.kv_quant_fp4(_bits(inp["kv_bf16"][torch.from_numpy(sample)]))
    assert np.array_equal(st.codes[torch.from_numpy(sample).cuda()].cpu().numpy(), rc)
    assert np.array_equal(st.sf[torch.from_numpy(sample).cuda()].cpu().numpy(), rs)


def _check_pool(gpu_pool, gpu_bm, ref_bm, vis, n_pool):
    """The pool built from the GPU's block maxima is exact; against the oracle's own block maxima
    it may differ only at blocks whose oracle maximum is within 1e-5 of the n_pool-th one."""
    nb = (vis + 7) // 8
    exact = oracle.candidate_pool(gpu_bm[:nb], n_pool)
    assert np.array_equal(gpu_pool, exact)
    ref = {"idx": oracle.candidate_pool(ref_bm, n_pool), "pos": np.arange(nb), "scores": ref_bm}
    check_topk(gpu_pool, ref, n_pool, "pool")


@pytest.mark.parametrize("name", ["decode_b1_l4096_bf16idx", "decode_b8_l65536",
                                  "decode_ragged_b32", "hier_decode_l1m",
                                  "hier_decode_l1m_swa128", "prefill_t4096_p262144",
                                  "prefill_hier_t4096_p262144"])
def test_workload_full_size(mods, name):
    step, synth = mods
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w)
    st = step.Step(inp)
    st.run()
    torch.cuda.synchronize()
    assert st.layers[0]["out"].isfinite().all()
    rng = np.random.default_rng(0)
    _check_cache(st, inp, rng)

    k_idx = _np(inp["k_idx"])
    cu = inp["cu_ctx"].numpy()
    q_seq = inp["q_seq"].numpy()
    q_vis = inp["q_vis"].numpy()
    codes, sf = st.codes.cpu().numpy(), st.sf.cpu().numpy()
    if w.kind == "prefill":
        nq = w.T
        queries = sorted(set(np.linspace(0, nq - 1, 62).astype(int).tolist() + [1, nq - 2]))
    else:
        queries = list(range(w.B))
    # attention: every sampled query of a one-layer step; with six layers every fourth one
    attn_queries = queries if len(st.layers) == 1 or w.kind != "prefill" else queries[::4]

    last_idx = None
    for li, L in enumerate(st.layers):
        mode = L["mode"]
        if mode in ("full", "reindex"):
            gpu_idx = L["idx"].cpu().numpy()
            cand = None if mode == "full" else st.pool.cpu().numpy()
            ref = oracle.index_score_topk(_np(inp["layers"][li]["q_idx"]), w.idx_dtype,
                                          inp["layers"][li]["w"].numpy(), k_idx, cu, q_seq, q_vis,
                                          w.topk, cand_blocks=cand, queries=queries)
            for n in queries:
                check_topk(gpu_idx[n], ref[n], w.topk, f"{name} layer {li} ({mode}) query {n}")
            if mode == "full" and st.pool is not None and li == 0:  # the pool per query
                gbm = st.bm.cpu().numpy()
                gpool = st.pool.cpu().numpy()
                for n in queries:
                    nbn = (int(q_vis[n]) + 7) // 8
                    np.testing.assert_allclose(gbm[n, :nbn], ref[n]["bm"], rtol=1e-5, atol=1e-5)
                    _check_pool(gpool[n], gbm[n], ref[n]["bm"], int(q_vis[n]), w.n_pool_blocks)
            last_idx = gpu_idx
        # attention on the GPU's own indices
        q_attn = _np(inp["layers"][li]["q_attn"])
        out_b, lse = _bits(L["out"]), L["lse"].cpu().numpy()
        if w.n_win:  # the layer's local window: its new FP8 rows, then one softmax over both
            swa = L["swa_kv"].cpu().numpy()
            new_rows = st.swa_rows.cpu().numpy()
            assert np.array_equal(swa[new_rows],
                                  oracle.fp8_quant(_np(inp["layers"][li]["swa_new"])))
            ref_a = oracle.sparse_swa_attn_queries(
                q_attn, q_seq, q_vis, codes, sf, cu, last_idx, swa, st.swa_ring, w.n_win,
                st.scale, queries=attn_queries, quantize_query=w.kind == "prefill")
        elif w.kind == "prefill":
            ref_a = oracle.sparse_attn_prefill(q_attn, q_seq, codes, sf, cu, last_idx,
                                               st.scale, tokens=attn_queries)
        else:
            ref_a = oracle.sparse_attn_decode(q_attn, codes, sf, cu, last_idx, st.scale,
                                              seqs=attn_queries)
        for n in attn_queries:
            o, l = ref_a[n]
            check_attn(out_b[n], lse[n], o, l, oracle.double_to_bf16(o),
                       f"{name} layer {li} ({mode}) attention {n}")


@pytest.mark.parametrize("B,L", [(1, 65536), (3, 40000)])
def test_overlapped_layers_match_model_order(mods, B, L):
    """The hierarchical decoder's layers on their own streams (ordered by events along the
    pool and index dependencies), run directly and as a replayed CUDA graph, give bit for bit
    what the model-order step gives."""
    step, synth = mods
    w = synth.scaled(synth.WORKLOADS["hier_decode_l1m"], B=B, L=(L,) * B)
    inp = synth.make_inputs(w)
    ser = step.Step(inp)
    con = step.Step(inp, overlap_layers=True)
    assert not ser.side and len(con.side) == len(w.modes) - 1
    ser.run()
    torch.cuda.synchronize()
    want = [(M["out"].clone(), M["lse"].clone(), M.get("idx")) for M in ser.layers]
    want_idx = [None if i is None else i.clone() for _, _, i in want]

    def same():
        torch.cuda.synchronize()
        for li, (M, (o, l, _), ix) in enumerate(zip(con.layers, want, want_idx)):
            assert torch.equal(M["out"].view(torch.int16), o.view(torch.int16)), li
            assert torch.equal(M["lse"], l), li
            if ix is not None:
                assert torch.equal(M["idx"], ix), li
        assert torch.equal(con.pool, ser.pool)

    for _ in range(3):
        for M in con.layers:
            M["out"].zero_()
        con.run()
        same()
    con.capture()
    for _ in range(3):
        for M in con.layers:
            M["out"].zero_()
        con.replay()
        same()


@pytest.mark.parametrize("name,B,L", [("hier_decode_l1m", 1, 65536),
                                      ("hier_decode_l1m_swa128", 2, 30000)])
def test_step_with_host_copies_matches_device_step(mods, name, B, L):
    """The step with its inputs copied in and its outputs copied out layer by layer, overlapped
    with the computation (Step.run(io=...), as bench.py's end-to-end timing runs it), directly
    and as a replayed graph: the host output buffer holds exactly the device step's outputs,
    and a changed host input reaches the device (the copies are not skipped)."""
    step, synth = mods
    w = synth.scaled(synth.WORKLOADS[name], B=B, L=(L,) * B)
    st = step.Step(synth.make_inputs(w))
    st.run()
    torch.cuda.synchronize()
    want = st.out_arena.buf.clone().cpu()
    host_in = st.in_arena.buf.cpu().pin_memory()
    host_out = torch.zeros(st.out_arena.size, dtype=torch.uint8).pin_memory()
    st.run(io=(host_in, host_out))
    torch.cuda.synchronize()
    assert torch.equal(host_out, want)
    g = st.capture(io=(host_in, host_out))
    for _ in range(2):
        host_out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(host_out, want)
    # a different last-layer attention query on the host changes only the last layer's output
    qa = st.in_arena.offsets[f"q_attn{len(st.layers) - 1}"]
    host_in[qa:qa + 64] = 0
    g.replay()
    torch.cuda.synchronize()
    oa, ob = st.out_ranges[-1]
    assert torch.equal(host_out[:oa], want[:oa])
    assert not torch.equal(host_out[oa:ob], want[oa:ob])
