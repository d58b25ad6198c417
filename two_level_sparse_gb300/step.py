"""One indexer step through the C ABI: the source layer's dense keys and
published blocks, then every layer's top-k positions.

Call sequence (sglang PR #40352, Design: the source computes its dense scores,
publishes its candidate blocks and runs its own top-512; each consumer selects
within the published blocks):

  ci_score_dense_amax8(source)                   keys, rows with > min(K, P+1) blocks
  ci_publish_blocks2(keys, K, P + 1)             the consumers' and the source's candidates
                                                 (ci_publish_blocks when P + 1 == K)
  ci_select_sparse(source, P + 1 blocks)         the source's top-P
  ci_select_sparse(consumer j, K blocks)         each consumer's top-P
  (with fewer rows than SMs, one ci_select_sparse_layers launch for all)

Every position of the dense top-P lies in the top P + 1 blocks by key (the
newest block's key is +inf and every other block that outranks a position's
block holds a distinct higher-scoring position), so the source's top-P over
its top-(P+1) blocks is its dense top-P, and the source gathers only those.

The layers' selects are independent of one another and share the page
table.  With fewer rows than SMs one persistent launch works through all
(layer, row) pairs, so a small batch fills every SM and a CTA's units
overlap one another; with more, each layer has its own launch (a fixed
layer reads its pointers as constant operands, a little faster per tile) on
its own stream, forked from and joined back into the caller's stream, so
that each launch's last rows overlap the next one's first.

This module only allocates the output buffers (torch device memory) and
marshals arguments; all computation runs in libci.so.
"""
from __future__ import annotations

import torch

from . import ci


class IndexerStep:
    def __init__(self, wl, with_scores: bool = False):
        dev = wl.seq_len.device
        self.wl = wl
        self.rows = wl.rows
        self.max_len = wl.max_len
        self.K = wl.topk_blocks
        self.P = wl.topk
        self.Kp = self.P + 1  # the source's own candidate blocks
        self.skip = min(self.K, self.Kp)  # rows with at most this many blocks need no keys
        nb_max = (self.max_len + 7) // 8
        stride = max(8, (nb_max + 7) // 8 * 8)
        i32 = torch.int32
        self.keys = torch.empty(self.rows, stride, dtype=torch.float32, device=dev)
        self.blocks = torch.empty(self.rows, self.K, dtype=i32, device=dev)
        self.nvalid = torch.empty(self.rows, dtype=i32, device=dev)
        if self.Kp == self.K:
            self.blocks_src, self.nvalid_src = self.blocks, self.nvalid
        else:
            self.blocks_src = torch.empty(self.rows, self.Kp, dtype=i32, device=dev)
            self.nvalid_src = torch.empty(self.rows, dtype=i32, device=dev)
        nl = len(wl.layers)
        self.pos = torch.empty(nl, self.rows, self.P, dtype=i32, device=dev)
        self.score = torch.empty(nl, self.rows, self.P, dtype=torch.float32, device=dev) if with_scores else None
        self.dev_err = torch.zeros(1, dtype=i32, device=dev)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count if dev.type == "cuda" else 1
        self.fused = self.rows < sms  # one select launch for every layer
        self.side = [] if self.fused or dev.type != "cuda" else [torch.cuda.Stream(device=dev) for _ in range(nl - 1)]

    def launches(self) -> int:
        """Kernels one run() enqueues: dense, publish, and one select for all
        layers or one per layer."""
        return 3 if self.fused else 2 + len(self.wl.layers)

    def run(self, stream=None, skip_dense=False, mark=None, layer_done=None):
        """Enqueue the step on `stream` (default: torch's current stream).
        ``skip_dense`` leaves out the first call, for callers that enqueue it
        themselves.  ``mark(name)``, if given, is called after each launch is
        enqueued (the benchmark records a CUDA event there);
        ``layer_done(j, s)`` after layer j's select is enqueued on stream s."""
        mark = mark or (lambda name: None)
        layer_done = layer_done or (lambda j, s: None)
        wl = self.wl
        src = wl.layers[0]
        common = dict(page_table=wl.page_table, layout=wl.layout, seq_len=wl.seq_len, max_len=self.max_len,
                      dev_err=self.dev_err, stream=stream, req_start=wl.req_start)
        if not skip_dense:
            ci.ci_score_dense_amax8(src.q_fp4, src.q_sf, src.w, src.k_pool, skip_le_blocks=self.skip, keys=self.keys,
                                    **common)
            mark("dense")
        if self.Kp != self.K:
            ci.ci_publish_blocks2(wl.seq_len, self.max_len, self.keys, self.K, self.blocks, self.nvalid, self.Kp,
                                  self.blocks_src, self.nvalid_src, dev_err=self.dev_err, stream=stream)
        else:
            ci.ci_publish_blocks(wl.seq_len, self.max_len, self.keys, self.K, self.blocks, self.nvalid,
                                 dev_err=self.dev_err, stream=stream)
        mark("publish")
        layers = []
        for j, layer in enumerate(wl.layers):
            blocks, nvalid, mb = (self.blocks_src, self.nvalid_src, self.Kp) if j == 0 else (self.blocks,
                                                                                            self.nvalid, self.K)
            layers.append(dict(q_fp4=layer.q_fp4, q_sf=layer.q_sf, w=layer.w, k_pool=layer.k_pool, blocks=blocks,
                               nvalid=nvalid, max_blocks=mb, out_pos=self.pos[j],
                               out_score=None if self.score is None else self.score[j]))
        main = stream if stream is not None else torch.cuda.current_stream(self.dev_err.device)
        if self.fused:
            ci.ci_select_sparse_layers(layers, wl.page_table, wl.layout, wl.seq_len, self.max_len, self.P,
                                       dev_err=self.dev_err, stream=stream, req_start=wl.req_start)
            for j in range(len(layers)):
                layer_done(j, main)
        else:
            fork = torch.cuda.Event()
            fork.record(main)
            for j, ly in enumerate(layers):
                on = main
                if j > 0:
                    on = self.side[j - 1]
                    on.wait_event(fork)
                ci.ci_select_sparse(ly["q_fp4"], ly["q_sf"], ly["w"], ly["k_pool"], blocks=ly["blocks"],
                                    nvalid=ly["nvalid"], max_blocks=ly["max_blocks"], topk=self.P,
                                    out_pos=ly["out_pos"], out_score=ly["out_score"], **dict(common, stream=on))
                layer_done(j, on)
            for side in self.side:
                joined = torch.cuda.Event()
                joined.record(side)
                main.wait_event(joined)
        mark("select")

    def capture(self, stream):
        """The step captured as a CUDA graph on ``stream`` (same buffers):
        replaying it enqueues every launch (side streams' fork and join
        included) without per-launch host work -- what small decode batches,
        bound by launch latency, need.  Run the step once before capturing
        (the first launches set kernel attributes)."""
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            self.run(stream)
        return graph

    def device_inputs(self):
        """The step's input tensors, shared ones first, then layer by layer."""
        wl = self.wl
        shared = [wl.seq_len, wl.page_table] + ([] if wl.req_start is None else [wl.req_start])
        return shared, [[l.q_fp4, l.q_sf, l.w, l.k_pool] for l in wl.layers]

    def run_host(self, host_shared, host_layers, host_out, stream=None):
        """The step from pinned host inputs to pinned host outputs.

        ``host_shared`` / ``host_layers`` mirror ``device_inputs()``;
        ``host_out`` receives (blocks, nvalid, pos[layer] ...).  The shared
        and source-layer inputs are copied first; the consumers' inputs copy on
        a second stream while the source is scored; the published blocks copy
        back while the layers' selects run, and each layer's positions as soon
        as its select is done.  All copies finish before ``stream`` does."""
        main = stream if stream is not None else torch.cuda.current_stream(self.dev_err.device)
        if not hasattr(self, "_copy"):
            self._copy = torch.cuda.Stream(device=self.dev_err.device)
        cp = self._copy
        shared, layers = self.device_inputs()
        start = torch.cuda.Event()
        start.record(main)  # the previous step on `main` is done with these buffers once this passes
        with torch.cuda.stream(main):
            for d, h in zip(shared + layers[0], host_shared + host_layers[0]):
                d.copy_(h, non_blocking=True)
        cp.wait_event(start)
        ready = []
        with torch.cuda.stream(cp):
            for dl, hl in zip(layers[1:], host_layers[1:]):
                for d, h in zip(dl, hl):
                    d.copy_(h, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cp)
                ready.append(ev)
        outs = [self.blocks, self.nvalid] + [self.pos[j] for j in range(len(layers))]

        def mark(name):
            if name == "publish":
                # consumers need their inputs; copy the published table back
                for ev in ready:
                    main.wait_event(ev)
                done = torch.cuda.Event()
                done.record(main)
                cp.wait_event(done)
                with torch.cuda.stream(cp):
                    host_out[0].copy_(outs[0], non_blocking=True)
                    host_out[1].copy_(outs[1], non_blocking=True)

        def layer_done(j, s):
            done = torch.cuda.Event()
            done.record(s)
            cp.wait_event(done)
            with torch.cuda.stream(cp):
                host_out[2 + j].copy_(outs[2 + j], non_blocking=True)

        self.run(main, mark=mark, layer_done=layer_done)
        end = torch.cuda.Event()
        end.record(cp)
        main.wait_event(end)

    def outputs_numpy(self):
        out = dict(keys=self.keys.cpu().numpy(), blocks=self.blocks.cpu().numpy(), nvalid=self.nvalid.cpu().numpy(),
                   blocks_src=self.blocks_src.cpu().numpy(), nvalid_src=self.nvalid_src.cpu().numpy(),
                   pos=self.pos.cpu().numpy())
        if self.score is not None:
            out["score"] = self.score.cpu().numpy()
        return out
