"""A decoder layer's decode step driven through the library's calls.

The step is the path's sequence of launches on one stream, per command of at
most eight rows:

    dl_gemv_q8(Wqkv)  ->  dl_rope_kv_store  ->  dl_decode_attn  ->  dl_attn_merge
    ->  dl_gemv_q8(Wo)  ->  dl_gemv_q8(Wgate|up)  ->  dl_gemv_q8(Wdown)

or, with `fused_rope`, dl_decode_attn_rope in place of the rope/store and the
attention (one launch fewer, the same stored halves and results); with
`l2_prefetch`, two launches ask L2 for part of a later kernel's weights while
they run (dl_l2_prefetch_next; results unchanged): the merge for the first
half of the gate/up tiles, the O projection for the first quarter of the down
tiles (the schedule that measured best at eight rows; it is off by default,
since at one row it measured slower); with
`cluster_merge`, dl_decode_attn_cluster in place of the attention and the merge
(the pieces of a KV head merge inside their thread-block cluster); with
`tail_merge`, dl_decode_attn_merged in place of them for commands whose work
items serve at most eight queries (the last piece of a KV head merges); with
`gemv_chain`, the O, gate/up and down projections as the phases of one
dl_gemv_q8_chain launch; with `one_launch`, the whole step of a command as one
dl_layer_step launch (the f16 mirror; its plan sized for about one attention
work item per SM).  A step of several commands (sessions past eight rows) may
run them on streams of their own (`concurrent`), since they share nothing but
the weights; not with `one_launch` or `gemv_chain`, whose launches hold every
SM while their CTAs wait on one another, so that two side by side could wait on
each other.

Norms, SwiGLU and residual adds are not part of the path: the gate/up and down
projections read their own activation buffers (filled by the caller).  More
than eight rows run as the fewest balanced commands, the weights read once per
command.  Nothing here computes: it owns buffers and issues the calls.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import torch

from . import (KVCache, PackedQ8, Rope, device_sm_count, dl_attn_merge, dl_attn_plan_build,
               dl_attn_plan_build_cluster, dl_decode_attn, dl_decode_attn_cluster, dl_decode_attn_merged,
               dl_decode_attn_rope, dl_gemv_q8, dl_gemv_q8_chain, dl_l2_prefetch_next, dl_layer_step,
               dl_layer_step_workspace_size, dl_plan_groups, dl_rope_kv_store, layer_weights_c, workspace_for)



def _prefetch_head(w: Optional[PackedQ8], frac: float) -> None:
    """Hand the first `frac` of w's weight tiles (whole 16-byte units) to the next launch."""
    if w is None:
        dl_l2_prefetch_next([])
        return
    dl_l2_prefetch_next([(w.qs.data_ptr(), int(w.qs.numel() * frac) // 16 * 16)])


@dataclasses.dataclass
class LayerWeights:
    """Packed Q8_0 projections of one layer (gate and up concatenated; FFN optional)."""
    wqkv: PackedQ8
    wo: PackedQ8
    wgu: Optional[PackedQ8] = None
    wdown: Optional[PackedQ8] = None

    def q8_bytes(self) -> int:
        return sum(w.nbytes_q8_0 for w in (self.wqkv, self.wo, self.wgu, self.wdown) if w is not None)

    def c(self):
        """The weights as the C struct of dl_layer_step (built once)."""
        if getattr(self, "_c", None) is None:
            self._c = layer_weights_c(self.wqkv, self.wo, self.wgu, self.wdown)
        return self._c


class Command:
    """Buffers and plan of one command (1..8 rows) of a layer step."""

    def __init__(self, rows: Sequence[int], positions: Sequence[int], regions: Sequence[int],
                 n_q: int, n_kv: int, head_dim: int, hidden: int, ffn: int, device, sm_count: int = 0,
                 force_chunk: int = 0, gemv_path: int = 0, attn_path: int = 0, fused_rope: bool = False,
                 cluster_merge: bool = False, gemv_chain: bool = False, l2_prefetch: bool = False,
                 tail_merge: bool = False, one_launch: bool = False, chain_ffn: bool = False):
        """one_launch: the whole step as one dl_layer_step launch.  chain_ffn: the gate/up
        projection reads the O output and the down projection the first `ffn` columns of the
        gate/up output (instead of buffers of their own), the order a decoder layer imposes."""
        n = len(rows)
        assert 1 <= n <= 8
        self.one_launch = bool(one_launch)
        if self.one_launch and (cluster_merge or gemv_chain or l2_prefetch or tail_merge):
            raise ValueError("one_launch runs the whole step in one launch: no other step form applies")
        self.chain_ffn = bool(chain_ffn) and ffn > 0
        self.l2_prefetch = bool(l2_prefetch)
        self.gemv_path, self.attn_path = gemv_path, attn_path
        self.fused_rope = bool(fused_rope)
        self.cluster_merge = bool(cluster_merge)
        self.gemv_chain = bool(gemv_chain) and ffn > 0
        self.rows = list(rows)
        self.n = n
        D = head_dim
        self.n_q, self.n_kv, self.D = n_q, n_kv, D
        self.positions = [int(p) for p in positions]
        self.regions = [int(r) for r in regions]
        self.seqlen_host = [p + 1 for p in self.positions]
        # the last piece merges when a work item serves at most 8 queries (sessions of few rows)
        sess_rows = max(self.regions.count(r) for r in set(self.regions))
        self.tail_merge = bool(tail_merge) and not cluster_merge and sess_rows * (n_q // n_kv) <= 8
        if self.cluster_merge:
            self.plan = dl_attn_plan_build_cluster(self.seqlen_host, n_q, n_kv, D, regions=self.regions,
                                                   sm_count=sm_count)
        elif self.one_launch:
            # about one work item per SM: the launch holds one CTA per SM
            sms = sm_count if sm_count > 0 else device_sm_count(device)
            self.plan = dl_attn_plan_build(self.seqlen_host, n_q, n_kv, D, regions=self.regions,
                                           sm_count=max(1, sms // 2), force_chunk=force_chunk)
        else:
            self.plan = dl_attn_plan_build(self.seqlen_host, n_q, n_kv, D, regions=self.regions,
                                           sm_count=sm_count, force_chunk=force_chunk)
        dev = device
        f32 = dict(dtype=torch.float32, device=dev)
        self.x = torch.zeros(n, hidden, **f32)
        self.qkv = torch.zeros(n, (n_q + 2 * n_kv) * D, **f32)
        self.attn = torch.zeros(n, n_q * D, **f32)
        self.lse = torch.zeros(n, n_q, **f32)
        self.y_o = torch.zeros(n, hidden, **f32)
        self.x_ffn = torch.zeros(n, hidden, **f32) if ffn else None
        self.gu = torch.zeros(n, 2 * ffn, **f32) if ffn else None
        self.h = torch.zeros(n, ffn, **f32) if ffn else None
        self.y_down = torch.zeros(n, hidden, **f32) if ffn else None
        i32 = dict(dtype=torch.int32, device=dev)
        self.pos = torch.tensor(self.positions, **i32)
        self.seqlen = torch.tensor(self.seqlen_host, **i32)
        self.region = torch.tensor(self.regions, **i32)
        self.status = torch.zeros(1, **i32)
        self.workspace = workspace_for(self.plan, dev)
        self.sync = torch.zeros(4, **i32)                    # the chain launch's barrier words
        self.step_ws = None                                  # dl_layer_step's workspace (sized at first run)
        qd, kd = n_q * D, n_kv * D
        self.q = self.qkv[:, :qd]
        self.k = self.qkv[:, qd:qd + kd]
        self.v = self.qkv[:, qd + kd:]

    def ffn_inputs(self):
        """The gate/up and down inputs: buffers of their own, or (chain_ffn) the O output and the
        gate half of the gate/up output."""
        if self.x_ffn is None:
            return None, None
        if self.chain_ffn:
            return self.y_o, self.gu[:, :self.h.shape[1]]
        return self.x_ffn, self.h

    def run(self, W: LayerWeights, rope: Rope, kv: KVCache, stream=None):
        # the separate GEMV's CUDA-core form serves 1 or 2 rows; the one launch's serves up to 8
        gp = self.gemv_path if (self.gemv_path != 1 or self.n <= 2 or self.one_launch) else 0
        if self.one_launch:
            Wc = W.c()
            if self.step_ws is None:
                self.step_ws = torch.zeros(dl_layer_step_workspace_size(Wc, self.plan), dtype=torch.uint8,
                                           device=self.x.device)
            xf, xd = self.ffn_inputs() if W.wgu is not None else (None, None)
            dl_layer_step(Wc, self.x, self.qkv, self.attn, self.lse, self.y_o, xf,
                          self.gu if W.wgu is not None else None, xd,
                          self.y_down if W.wgu is not None else None, self.pos, rope, kv, self.seqlen,
                          self.plan, self.step_ws, status=self.status, stream=stream, path=gp)
            return
        pf = self.l2_prefetch and not self.gemv_chain
        dl_gemv_q8(W.wqkv, self.x, self.qkv, stream=stream, path=gp)
        if self.cluster_merge:
            if self.fused_rope:
                dl_decode_attn_cluster(self.q, kv, self.seqlen, self.plan, self.attn, self.lse, k=self.k, v=self.v,
                                       pos=self.pos, rope=rope, status=self.status, stream=stream,
                                       path=self.attn_path)
            else:
                dl_rope_kv_store(self.q, self.k, self.v, self.pos, rope, kv, self.n_q, row_region=self.region,
                                 status=self.status, stream=stream)
                dl_decode_attn_cluster(self.q, kv, self.seqlen, self.plan, self.attn, self.lse, status=self.status,
                                       stream=stream, path=self.attn_path)
        elif self.tail_merge:
            rin = dict(k=self.k, v=self.v, pos=self.pos, rope=rope) if self.fused_rope else {}
            if not self.fused_rope:
                dl_rope_kv_store(self.q, self.k, self.v, self.pos, rope, kv, self.n_q, row_region=self.region,
                                 status=self.status, stream=stream)
            dl_decode_attn_merged(self.q, kv, self.seqlen, self.plan, self.workspace, self.attn, self.lse,
                                  status=self.status, stream=stream, path=self.attn_path, **rin)
        elif self.fused_rope:
            dl_decode_attn_rope(self.q, self.k, self.v, self.pos, rope, kv, self.seqlen, self.plan,
                                self.workspace, status=self.status, stream=stream, path=self.attn_path)
        else:
            dl_rope_kv_store(self.q, self.k, self.v, self.pos, rope, kv, self.n_q, row_region=self.region,
                             status=self.status, stream=stream)
            dl_decode_attn(self.q, kv, self.seqlen, self.plan, self.workspace, status=self.status, stream=stream,
                           path=self.attn_path)
        if not self.cluster_merge and not self.tail_merge:
            if pf:
                _prefetch_head(W.wgu, 0.5)
            dl_attn_merge(self.workspace, self.plan, self.seqlen, self.attn, self.lse, stream=stream)
        if self.gemv_chain and W.wgu is not None:
            dl_gemv_q8_chain([W.wo, W.wgu, W.wdown], [self.attn, self.x_ffn, self.h], [self.y_o, self.gu, self.y_down],
                             self.sync, status=self.status, stream=stream, path=gp)
            return
        if pf:
            _prefetch_head(W.wdown, 0.25)
        dl_gemv_q8(W.wo, self.attn, self.y_o, stream=stream, path=gp)
        if W.wgu is not None:
            xf, xd = self.ffn_inputs()
            dl_gemv_q8(W.wgu, xf, self.gu, stream=stream, path=gp)
            dl_gemv_q8(W.wdown, xd, self.y_down, stream=stream, path=gp)

    @property
    def launches(self) -> int:
        if self.one_launch:
            return 1
        return (7 - int(self.fused_rope) - int(self.cluster_merge or self.tail_merge) -
                2 * int(self.gemv_chain))


class LayerStep:
    """All commands of one layer step: rows grouped into commands of at most eight."""

    def __init__(self, positions: Sequence[int], regions: Sequence[int], n_q: int, n_kv: int, head_dim: int,
                 hidden: int, ffn: int, device, sm_count: int = 0, force_chunk: int = 0, gemv_path: int = 0,
                 attn_path: int = 0, fused_rope: bool = False, cluster_merge: bool = False,
                 gemv_chain: bool = False, l2_prefetch: bool = False, concurrent: bool = False,
                 tail_merge: bool = False, one_launch: bool = False, chain_ffn: bool = False):
        """concurrent: the commands (independent sessions) run on streams of their own, forked
        from the caller's stream and joined back into it, so that one command's launch latencies
        overlap another's work.  Refused with one_launch and gemv_chain: those launches hold every
        SM and their CTAs wait on one another, so two of them at once could each hold SMs the
        other waits for."""
        if concurrent and (one_launch or gemv_chain):
            raise ValueError("concurrent commands cannot run as one_launch or gemv_chain launches")
        n = len(positions)
        sizes = dl_plan_groups(n)
        self.commands: List[Command] = []
        r0 = 0
        for s in sizes:
            idx = list(range(r0, r0 + s))
            self.commands.append(Command(idx, [positions[i] for i in idx], [regions[i] for i in idx],
                                         n_q, n_kv, head_dim, hidden, ffn, device, sm_count, force_chunk,
                                         gemv_path, attn_path, fused_rope, cluster_merge, gemv_chain,
                                         l2_prefetch, tail_merge, one_launch, chain_ffn))
            r0 += s
        self.group_sizes = sizes
        self.concurrent = bool(concurrent) and len(self.commands) > 1
        self.side_streams = ([torch.cuda.Stream(device=device) for _ in self.commands] if self.concurrent
                             else [])

    def run(self, W: LayerWeights, rope: Rope, kv: KVCache, stream=None):
        if not self.concurrent:
            for c in self.commands:
                c.run(W, rope, kv, stream)
            return
        main = stream if stream is not None else torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(main)
        for c, s in zip(self.commands, self.side_streams):
            s.wait_event(fork)
            c.run(W, rope, kv, s)
        for s in self.side_streams:
            main.wait_stream(s)

    @property
    def launches(self) -> int:
        return sum(c.launches for c in self.commands)
