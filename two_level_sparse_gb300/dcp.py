"""A context-sharded indexer step, emulated on one device.

W shards, interleave 1: global position s lives on shard s % W at local
position s // W, so a shard's local block b (8 / W positions) is its part of
global block b (vLLM sparse_attn_indexer.py, two-level candidate filtering
under DCP, and _merge_dcp_topk_global).  Per step:

  ci_score_dense_amax8(shard r, block_positions = 8 / W)   local block maxima
  ci_dcp_merge_keys                                       global keys, newest pinned
  ci_publish_blocks2(global keys, K, P + 1)               as unsharded
  ci_select_sparse(shard r, layer j, block_positions = 8 / W)  local top-P
  ci_dcp_merge_topk                                       global top-P

The results equal the unsharded step's exactly: a global block's key is the
maximum of its shards' maxima, and a position of the global top-P is in its
own shard's local top-P.  On W devices the two merges are the collectives
(a MAX-reduce of the keys, an all-gather of the candidates); here every
shard's buffers live on the one device and the merges read them all.

Allocation and argument marshalling only; the computation runs in libci.so.
"""
from __future__ import annotations

import torch

from . import ci, synth


class DcpStep:
    def __init__(self, wl, world: int, with_scores: bool = True):
        assert world in (2, 4, 8)
        dev = wl.seq_len.device
        self.wl, self.world = wl, world
        self.shards = synth.shard_workload(wl, world)
        self.bs = 8 // world
        self.rows, self.max_len = wl.rows, wl.max_len
        self.K, self.P = wl.topk_blocks, wl.topk
        self.Kp = self.P + 1
        self.skip = min(self.K, self.Kp)
        nb = (self.max_len + 7) // 8
        max_local = max(s.max_len for s in self.shards)
        lstride = max(8, (max(nb, (max_local + self.bs - 1) // self.bs) + 7) // 8 * 8)
        gstride = max(8, (nb + 7) // 8 * 8)
        i32, f32 = torch.int32, torch.float32
        self.keys_local = torch.empty(world, self.rows, lstride, dtype=f32, device=dev)
        self.keys = torch.empty(self.rows, gstride, dtype=f32, device=dev)
        self.blocks = torch.empty(self.rows, self.K, dtype=i32, device=dev)
        self.nvalid = torch.empty(self.rows, dtype=i32, device=dev)
        if self.Kp == self.K:
            self.blocks_src, self.nvalid_src = self.blocks, self.nvalid
        else:
            self.blocks_src = torch.empty(self.rows, self.Kp, dtype=i32, device=dev)
            self.nvalid_src = torch.empty(self.rows, dtype=i32, device=dev)
        nl = len(wl.layers)
        self.pos_local = torch.empty(world, self.rows, self.P, dtype=i32, device=dev)
        self.score_local = torch.empty(world, self.rows, self.P, dtype=f32, device=dev)
        self.pos = torch.empty(nl, self.rows, self.P, dtype=i32, device=dev)
        self.score = torch.empty(nl, self.rows, self.P, dtype=f32, device=dev) if with_scores else None
        self.dev_err = torch.zeros(1, dtype=i32, device=dev)

    def run(self, stream=None):
        wl = self.wl
        for r, sh in enumerate(self.shards):
            src = sh.layers[0]
            ci.ci_score_dense_amax8(src.q_fp4, src.q_sf, src.w, src.k_pool, sh.page_table, sh.layout, sh.seq_len,
                                    max(sh.max_len, 1), 0, self.keys_local[r], dev_err=self.dev_err, stream=stream,
                                    req_start=sh.req_start, block_positions=self.bs)
        ci.ci_dcp_merge_keys(self.keys_local, wl.seq_len, self.max_len, self.skip, self.keys, dev_err=self.dev_err,
                             stream=stream)
        if self.Kp != self.K:
            ci.ci_publish_blocks2(wl.seq_len, self.max_len, self.keys, self.K, self.blocks, self.nvalid, self.Kp,
                                  self.blocks_src, self.nvalid_src, dev_err=self.dev_err, stream=stream)
        else:
            ci.ci_publish_blocks(wl.seq_len, self.max_len, self.keys, self.K, self.blocks, self.nvalid,
                                 dev_err=self.dev_err, stream=stream)
        for j in range(len(wl.layers)):
            blocks, nvalid, mb = (self.blocks_src, self.nvalid_src, self.Kp) if j == 0 else (self.blocks,
                                                                                            self.nvalid, self.K)
            for r, sh in enumerate(self.shards):
                layer = sh.layers[j]
                ci.ci_select_sparse(layer.q_fp4, layer.q_sf, layer.w, layer.k_pool, sh.page_table, sh.layout,
                                    sh.seq_len, max(sh.max_len, 1), blocks, nvalid, mb, self.P, self.pos_local[r],
                                    out_score=self.score_local[r], dev_err=self.dev_err, stream=stream,
                                    req_start=sh.req_start, block_positions=self.bs)
            ci.ci_dcp_merge_topk(self.pos_local, self.score_local, self.pos[j],
                                 out_score=None if self.score is None else self.score[j], stream=stream)

    def outputs_numpy(self):
        out = dict(keys=self.keys.cpu().numpy(), blocks=self.blocks.cpu().numpy(), nvalid=self.nvalid.cpu().numpy(),
                   blocks_src=self.blocks_src.cpu().numpy(), nvalid_src=self.nvalid_src.cpu().numpy(),
                   pos=self.pos.cpu().numpy())
        if self.score is not None:
            out["score"] = self.score.cpu().numpy()
        return out
