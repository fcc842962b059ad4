"""The CSA2 decode and prefill steps as sequences of C-ABI calls.

Decode (one token per sequence; every layer of the workload's mode list, in order):
  * the new token's latent row is quantised into the FP4 cache;
  * Full layer: indexer scan + Top-K (and, in the hierarchical decoder, the block maxima that
    build the candidate pool: 2,048 blocks of 8 positions, "DeepSeek V4.1-Flash", aiwiki.ai,
    section "Compressed Sparse Attention 2"), then sparse attention;
  * Reindex layer: its own index query/weights over the pool, Top-K, sparse attention;
  * Reuse layer: sparse attention with the most recent layer's indices.
Prefill: the T new rows are quantised into the cache, the indexer selects Top-K per query token
(query i sees positions [0, P0 + i]), then sparse prefill attention.  With Reindex layers in the
mode list the first Full layer also builds a candidate pool per query token, which the Reindex
layers search, exactly as in the hierarchical decoder.

All device buffers (cache, queries, outputs, workspaces) are allocated once here with torch
(caller-side allocation); `run()` only enqueues C-ABI calls.

Order of the calls.  In a decoder, layer i+1's index and attention queries are computed from
layer i's output, so `run()` issues the layers one after another, in the model's order, on the
caller's stream.  The one overlap it uses is the quantisation of the new rows, which runs on a
second stream beside layer 0's selection (the indexer does not read the main-KV cache) and is
waited for before the first attention.

`overlap_layers=True` is for callers whose layer inputs are all known before the step (as in
this synthetic step, or layers of independent requests): the layers' calls then depend on one
another only through indices -- a Reindex layer needs the candidate pool of the first Full layer
(complete before that layer's own position selection, which csa2_index_score_topk_pool marks
with an event), a Reuse layer the indices of the layer it reuses -- and each layer runs on its
own stream, ordered by events along exactly those dependencies, with its own workspaces.
"""
from __future__ import annotations

import math

import torch

from . import csa2
from .synth import BLOCK, D, new_token_rows, swa_new_rows


class _Arena:
    """One contiguous device buffer holding several tensors as 256-byte aligned views, so a
    step's per-token inputs (or outputs) cross between host and device in one copy."""

    def __init__(self, specs, device):
        placed, off = [], 0
        for name, shape, dtype in specs:
            nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
            placed.append((name, off, shape, dtype, nbytes))
            off += (nbytes + 255) // 256 * 256
        self.buf = torch.empty(max(off, 256), dtype=torch.uint8, device=device)
        self.views = {name: self.buf[o:o + nb].view(dtype).view(shape)
                      for name, o, shape, dtype, nb in placed}
        self.offsets = {name: o for name, o, _, _, _ in placed}  # byte offset of each view
        self.size = self.buf.numel()


class Step:
    def __init__(self, inputs: dict, device="cuda", build_cache=True, overlap_layers=False):
        self.inp = inputs
        self.w = w = inputs["workload"]
        self.dev = device
        dev = device
        self.scale = 1.0 / math.sqrt(D)
        self.kv_bf16 = inputs["kv_bf16"].to(dev)
        rows = self.kv_bf16.shape[0]
        self.codes = torch.empty((rows, D // 2), dtype=torch.uint8, device=dev)
        self.sf = torch.empty((rows, D // 16), dtype=torch.uint8, device=dev)
        self.k_idx = inputs["k_idx"].to(dev)
        self.cu_ctx = inputs["cu_ctx"].to(dev)
        self.q_seq = inputs["q_seq"].to(dev)
        self.q_vis = inputs["q_vis"].to(dev)
        self.max_vis = inputs["max_vis"]
        self.nq = inputs["q_seq"].numel()
        self.new_rows = new_token_rows(inputs).to(dev)
        # per-step inputs (new rows, each layer's queries and weights) and outputs live in two
        # arenas, one host<->device copy each
        in_specs = [("new_x", (self.new_rows.numel(), D), torch.bfloat16)]
        out_specs = []
        for i, L in enumerate(inputs["layers"]):
            in_specs.append((f"q_attn{i}", tuple(L["q_attn"].shape), L["q_attn"].dtype))
            if "q_idx" in L:
                in_specs.append((f"q_idx{i}", tuple(L["q_idx"].shape), L["q_idx"].dtype))
                in_specs.append((f"w{i}", tuple(L["w"].shape), L["w"].dtype))
            if w.n_win:
                in_specs.append((f"swa_new{i}", (self.nq, D), torch.bfloat16))
            out_specs.append((f"out{i}", (self.nq, w.H, D), torch.bfloat16))
        self.in_arena = _Arena(in_specs, dev)
        self.out_arena = _Arena(out_specs, dev)
        self.new_x = self.in_arena.views["new_x"]
        self.new_x.copy_(self.kv_bf16[self.new_rows])
        if build_cache:  # the cache as it stands before the step (all rows), quantised on the GPU
            csa2.csa2_kv_quant_fp4(self.kv_bf16, self.codes, self.sf)
        self.layers = []
        self.swa_ring = inputs.get("swa_ring", 1)
        self.swa_rows = swa_new_rows(inputs).to(dev) if w.n_win else None
        nb = (self.max_vis + BLOCK - 1) // BLOCK
        # the hierarchical indexer: a candidate pool built by the first Full layer, searched by
        # the Reindex layers (decode and chunked prefill alike)
        hier = any(m == "reindex" for m in w.modes)
        for i, L in enumerate(inputs["layers"]):
            d = {"mode": L["mode"], "q_attn": self.in_arena.views[f"q_attn{i}"]}
            d["q_attn"].copy_(L["q_attn"])
            if "q_idx" in L:
                d["q_idx"] = self.in_arena.views[f"q_idx{i}"]
                d["q_idx"].copy_(L["q_idx"])
                d["w"] = self.in_arena.views[f"w{i}"]
                d["w"].copy_(L["w"])
                d["idx"] = torch.empty((self.nq, w.topk), dtype=torch.int32, device=dev)
            if w.n_win:  # the layer's local FP8 ring, as it stands before the step
                d["swa_kv"] = torch.empty((L["swa_bf16"].shape[0], D), dtype=torch.uint8,
                                          device=dev)
                csa2.csa2_swa_kv_quant_fp8(L["swa_bf16"].to(dev), d["swa_kv"])
                d["swa_new"] = self.in_arena.views[f"swa_new{i}"]
                d["swa_new"].copy_(L["swa_new"])
            d["out"] = self.out_arena.views[f"out{i}"]
            d["lse"] = torch.empty((self.nq, w.H), dtype=torch.float32, device=dev)
            self.layers.append(d)
        # byte ranges of each layer's inputs (layer 0's also holds the new rows) and output in
        # the arenas, for copies that overlap the step (run(io=...))
        n_l = len(self.layers)
        starts = [0] + [self.in_arena.offsets[f"q_attn{i}"] for i in range(1, n_l)]
        self.in_ranges = [(starts[i], starts[i + 1] if i + 1 < n_l else self.in_arena.size)
                          for i in range(n_l)]
        self.out_ranges = [(self.out_arena.offsets[f"out{i}"],
                            self.out_arena.offsets[f"out{i}"] + self.layers[i]["out"].numel() * 2)
                           for i in range(n_l)]
        self.bm = torch.empty((self.nq, nb), dtype=torch.float32, device=dev) if hier else None
        self.pool = (torch.empty((self.nq, w.n_pool_blocks), dtype=torch.int32, device=dev)
                     if hier else None)
        ws = csa2.csa2_index_score_topk_workspace_size(self.nq, self.max_vis, 0, w.topk)
        if hier:
            ws = max(ws, csa2.csa2_index_score_topk_workspace_size(self.nq, self.max_vis,
                                                                   w.n_pool_blocks, w.topk),
                     csa2.csa2_index_score_topk_pool_workspace_size(self.nq, self.max_vis,
                                                                    w.topk, w.n_pool_blocks))
        self.ws_index = csa2.workspace(ws, dev)
        # the layer each layer takes its indices from
        self.src, last = [], None
        for i, L in enumerate(self.layers):
            if L["mode"] in ("full", "reindex"):
                last = i
            self.src.append(last)
        self.overlap_layers = overlap_layers and len(self.layers) > 1
        self.qstream = torch.cuda.Stream(device=dev)
        self.ev_start = torch.cuda.Event()
        self.ev_ready = torch.cuda.Event()
        self.h2d_stream = torch.cuda.Stream(device=dev)
        self.d2h_stream = torch.cuda.Stream(device=dev)
        self.ev_in = [torch.cuda.Event() for _ in self.layers]
        self.ev_out = [torch.cuda.Event() for _ in self.layers]
        self.side = []
        if self.overlap_layers:
            self.side = [torch.cuda.Stream(device=dev) for _ in self.layers[1:]]
            self.ev_pool = torch.cuda.Event()
            # creates the event on the step's device, where the C ABI records into it
            self.ev_pool.record(torch.cuda.current_stream(dev))
            self.ev_idx = [torch.cuda.Event() for _ in self.layers]
            self.ev_done = [torch.cuda.Event() for _ in self.layers]
        for i, L in enumerate(self.layers):
            if "idx" in L:
                L["ws_index"] = (csa2.workspace(ws, dev) if self.overlap_layers and i > 0
                                 else self.ws_index)
        self.ws_pool = (csa2.workspace(csa2.csa2_hier_candidate_pool_workspace_size(
            self.nq, nb, w.n_pool_blocks), dev) if hier else None)
        if w.kind == "prefill":
            ws_a = (csa2.csa2_sparse_swa_attn_prefill_workspace_size(self.nq, w.H, w.topk, w.n_win)
                    if w.n_win else
                    csa2.csa2_sparse_attn_prefill_workspace_size(self.nq, w.H, w.topk))
        else:
            ws_a = (csa2.csa2_sparse_swa_attn_decode_workspace_size(self.nq, w.H, w.topk, w.n_win)
                    if w.n_win else
                    csa2.csa2_sparse_attn_decode_workspace_size(self.nq, w.H, w.topk))
        self.ws_attn = csa2.workspace(ws_a, dev)
        for i, L in enumerate(self.layers):
            L["ws_attn"] = (csa2.workspace(ws_a, dev) if self.overlap_layers and i > 0
                            else self.ws_attn)

    def drop_source_rows(self):
        """Free the bf16 rows the cache was quantised from (the step only reads the new rows)."""
        self.kv_bf16 = None
        torch.cuda.empty_cache()

    # ------------------------------------------------------------------------------------------
    def quantize_new_rows(self, stream=None):
        csa2.csa2_kv_quant_fp4(self.new_x, self.codes, self.sf, out_rows=self.new_rows,
                               stream=stream)

    def index(self, layer, cand=None, block_max=None, stream=None):
        csa2.csa2_index_score_topk(
            layer["q_idx"], self.w.idx_dtype, layer["w"], self.k_idx, self.cu_ctx, self.q_seq,
            self.q_vis, self.max_vis, self.w.topk, layer["idx"], cand_blocks=cand,
            out_block_max=block_max, ws=layer["ws_index"], stream=stream)

    def attend(self, layer, idx, stream=None):
        if self.w.n_win:  # the layer's local window joins the same softmax
            # this step's tokens' local rows go into the ring first
            csa2.csa2_swa_kv_quant_fp8(layer["swa_new"], layer["swa_kv"], out_rows=self.swa_rows,
                                       stream=stream)
            if self.w.kind == "prefill":
                csa2.csa2_sparse_swa_attn_prefill(
                    layer["q_attn"], self.q_seq, self.q_vis, self.codes, self.sf, self.cu_ctx,
                    idx, layer["swa_kv"], self.swa_ring, self.w.n_win, self.scale, layer["out"],
                    layer["lse"], ws=layer["ws_attn"], stream=stream)
            else:
                csa2.csa2_sparse_swa_attn_decode(
                    layer["q_attn"], self.codes, self.sf, self.cu_ctx, idx, layer["swa_kv"],
                    self.swa_ring, self.w.n_win, self.scale, layer["out"], layer["lse"],
                    ws=layer["ws_attn"], stream=stream)
            return
        if self.w.kind == "prefill":
            csa2.csa2_sparse_attn_prefill(layer["q_attn"], self.q_seq, self.codes, self.sf,
                                          self.cu_ctx, idx, self.scale, layer["out"],
                                          layer["lse"], ws=layer["ws_attn"], stream=stream)
        else:
            csa2.csa2_sparse_attn_decode(layer["q_attn"], self.codes, self.sf, self.cu_ctx, idx,
                                         self.scale, layer["out"], layer["lse"],
                                         ws=layer["ws_attn"], stream=stream)

    def block_max(self, layer, out, stream=None):
        """The Full layer's scan alone: block maxima of every visible position into `out`
        (csa2_index_block_max)."""
        csa2.csa2_index_block_max(layer["q_idx"], self.w.idx_dtype, layer["w"], self.k_idx,
                                  self.cu_ctx, self.q_seq, self.q_vis, self.max_vis, out,
                                  stream=stream)

    def index_with_pool(self, layer, stream=None, pool_event=None):
        """The first Full layer of the hierarchical decoder: its selection and the candidate
        pool in one call (csa2_index_score_topk_pool)."""
        csa2.csa2_index_score_topk_pool(
            layer["q_idx"], self.w.idx_dtype, layer["w"], self.k_idx, self.cu_ctx, self.q_seq,
            self.q_vis, self.max_vis, self.w.topk, layer["idx"], self.w.n_pool_blocks, self.pool,
            out_block_max=self.bm, ws=layer["ws_index"], stream=stream, pool_event=pool_event)

    def _select(self, i, L, stream, pool_event=None):
        """Layer i's own selection (Full or Reindex)."""
        if L["mode"] == "full":
            if self.pool is not None and all(M["mode"] != "full" for M in self.layers[:i]):
                self.index_with_pool(L, stream=stream, pool_event=pool_event)
            else:
                self.index(L, stream=stream)
        elif L["mode"] == "reindex":
            self.index(L, cand=self.pool, stream=stream)

    def run(self, stream=None, io=None):
        """One step: quantise the new rows, then every layer (see the module docstring for the
        order of the calls).  io = (host_in, host_out), pinned host buffers laid out like the
        input and output arenas: the step's inputs are copied in and its outputs out as part of
        the step, overlapped with the computation.  Layer 0's inputs (with the new rows) cross
        first on the step's stream; the other layers' inputs follow on a copy stream while
        layer 0 computes, and layer 1 waits for them.  The outputs of all layers but the last
        leave on a copy stream while the last layer computes, and the last one on the step's
        stream, which then waits for both copies."""
        main = stream if stream is not None else torch.cuda.current_stream()
        n_l = len(self.layers)
        if io is not None:
            assert not self.overlap_layers, "the host copies follow the model order"
            host_in, host_out = io
            h2d, d2h = self.h2d_stream, self.d2h_stream
            _, b0 = self.in_ranges[0]
            self.in_arena.buf[:b0].copy_(host_in[:b0], non_blocking=True)
            if n_l > 1:
                h2d.wait_stream(main)  # the previous step has finished with the arena
                with torch.cuda.stream(h2d):
                    self.in_arena.buf[b0:].copy_(host_in[b0:], non_blocking=True)
                self.ev_in[1].record(h2d)
        # the new rows go into the cache beside layer 0's selection (which does not read it)
        self.ev_start.record(main)
        self.qstream.wait_event(self.ev_start)
        self.quantize_new_rows(self.qstream)
        self.ev_ready.record(self.qstream)
        if not self.overlap_layers:
            for i, L in enumerate(self.layers):
                if io is not None and i == 1:
                    main.wait_event(self.ev_in[1])
                self._select(i, L, main)
                if i == 0:
                    main.wait_event(self.ev_ready)
                self.attend(L, self.layers[self.src[i]]["idx"], stream=main)
                if io is not None and i == n_l - 2:  # every output but the last one's
                    self.ev_out[i].record(main)
                    d2h.wait_event(self.ev_out[i])
                    e = self.out_ranges[i][1]
                    with torch.cuda.stream(d2h):
                        host_out[:e].copy_(self.out_arena.buf[:e], non_blocking=True)
            if io is not None:
                a = self.out_ranges[n_l - 2][1] if n_l > 1 else 0
                host_out[a:].copy_(self.out_arena.buf[a:], non_blocking=True)
                if n_l > 1:
                    main.wait_stream(d2h)
            return
        streams = [main] + self.side
        for i, L in enumerate(self.layers):
            s = streams[i]
            if i > 0:
                s.wait_event(self.ev_start)
            if L["mode"] == "reindex" and self.pool is not None:
                s.wait_event(self.ev_pool)
            elif L["mode"] not in ("full", "reindex"):
                s.wait_event(self.ev_idx[self.src[i]])
            self._select(i, L, s, pool_event=self.ev_pool)
            if L["mode"] in ("full", "reindex"):
                self.ev_idx[i].record(s)
            s.wait_event(self.ev_ready)
            self.attend(L, self.layers[self.src[i]]["idx"], stream=s)
            if i > 0:
                self.ev_done[i].record(s)
        for i in range(1, len(self.layers)):
            main.wait_event(self.ev_done[i])

    # ------------------------------------------------------------------------------------------
    def capture(self, io=None):
        """Record one step (the same C-ABI calls as run(), with the host copies when io is
        given) into a CUDA graph; replay() then re-issues the whole step with one launch.
        Without io, inputs and outputs stay in the buffers above, so a caller refreshes inputs
        in place between replays; with io, the graph copies from and to those host buffers."""
        self.run(io=io)  # first calls on this device: one-time set-up outside the capture
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
                self.run(stream=side, io=io)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        if io is None:
            self.graph = graph
        return graph

    def replay(self):
        self.graph.replay()

    # ------------------------------------------------------------------------------------------
    def algorithmic_bytes(self) -> dict:
        """Bytes the step must move at least once (HBM), by part."""
        w = self.w
        key_row = 128
        vis_total = int(self.inp["q_vis"].to(torch.int64).sum())
        n_full = sum(1 for L in self.layers if L["mode"] == "full")
        n_re = sum(1 for L in self.layers if L["mode"] == "reindex")
        n_att = len(self.layers)
        row = D // 2 + D // 16
        by = {
            "new_rows": self.new_x.numel() * 2 + self.new_rows.numel() * row,
            "index_keys_full": n_full * vis_total * key_row if w.kind != "prefill"
            else int(self.inp["cu_ctx"][-1]) * key_row,
            "index_keys_reindex": n_re * self.nq * w.n_pool_blocks * BLOCK * key_row,
            "gathered_rows": n_att * self.nq * w.topk * row,
            "q_out": n_att * self.nq * w.H * D * 2 * 2,
            "local_window_rows": n_att * self.nq * min(w.n_win, self.max_vis) * D if w.n_win else 0,
        }
        by["total"] = sum(by.values())
        return by
