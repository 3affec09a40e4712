"""Ulysses attention across real processes: one rank per process (one GPU
each in a deployment), the exchanges as all-to-all collectives between them.

This is the attention wrapper of huggingface/accelerate PR #4209 as a rank
runs it, where ``UlyssesAttention`` emulates all P ranks inside one GPU:

1. position_ids are all-gathered once per forward (the comment that moves the
   gather into the model's pre-hook) and the document boundaries are rebuilt
   from the gathered positions, never from the collator's per-shard ones (the
   comment on stale ``cu_seq_lens_q/k``);
2. q, k and v go through the seq->head all-to-all ("gather sequence, scatter
   heads", the comment on the four ``_SeqAllToAll.apply`` call sites): the
   rank packs one chunk per destination rank (``usp_a2a_pack_seq_to_head``),
   the collective delivers, and the received chunks are the whole sequence of
   the rank's heads;
3. varlen attention runs on that gathered sequence with the rank's slice of
   the sink logits (the gpt-oss finding: one sink per head, sliced to the
   rank's heads);
4. O goes back through the head->seq all-to-all; the backward runs the same
   exchanges swapped, and dK/dV of replicated key/value heads (fewer of them
   than ranks) are summed over the replicas on the way back.

The collectives are ``torch.distributed`` calls on the given process group.
With NCCL they run on the device buffers; with gloo (CPU transport) the
buffers are staged through host memory.  Every local step runs in the
library's kernels (``LibraryOps``); the ``ops`` argument exists so that the
orchestration above can be exercised with a stand-in on machines without a
GPU.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch
import torch.distributed as dist

from . import binding as B_


@dataclass
class RankShape:
    """Global sizes of one attention layer, P = the number of ranks."""
    B: int
    S: int
    Hq: int
    Hkv: int
    D: int
    P: int
    causal: bool = True
    window_left: int = -1
    softmax_scale: float = 0.0

    def __post_init__(self):
        if self.S % self.P != 0:
            raise ValueError(f"sp size {self.P} does not divide sequence length {self.S}")
        if self.Hq % self.P != 0:
            raise ValueError(f"sp size {self.P} does not divide {self.Hq} query heads")
        if (self.Hkv % self.P if self.Hkv >= self.P else self.P % self.Hkv) != 0:
            raise ValueError(f"sp size {self.P} and {self.Hkv} key/value heads: neither divides the other")
        if self.Hq % self.Hkv != 0:
            raise ValueError("key/value heads must divide query heads")

    @property
    def Sl(self) -> int:
        return self.S // self.P

    @property
    def hq(self) -> int:
        return self.Hq // self.P

    @property
    def hk(self) -> int:
        """Key/value heads per rank (1 replicated head when Hkv < P)."""
        return self.Hkv // self.P if self.Hkv >= self.P else 1

    def heads_per_rank(self, H: int) -> int:
        return H // self.P if H >= self.P else 1


class LibraryOps:
    """A rank's local steps, as the library's CUDA kernels."""

    def __init__(self, shape: RankShape, device):
        self.s = shape
        self.device = torch.device(device)
        s = shape
        self.cu_seqlens = torch.empty((s.B * s.S + 1,), dtype=torch.int32, device=self.device)
        self.n_docs = torch.zeros((1,), dtype=torch.int32, device=self.device)
        self.max_len = torch.zeros((1,), dtype=torch.int32, device=self.device)
        self.status = torch.zeros((1,), dtype=torch.int32, device=self.device)
        self.scan_ws = torch.empty((B_.usp_cu_seqlens_workspace_bytes(s.B, s.S),), dtype=torch.uint8,
                                   device=self.device)
        self._bwd_ws = None

    # -- exchanges: the rank's chunks for the collective and back
    def pack_seq_to_head(self, x_local, H):
        s = self.s
        send = torch.empty((s.P, s.B, s.Sl, s.heads_per_rank(H), s.D), dtype=x_local.dtype, device=self.device)
        B_.usp_a2a_pack_seq_to_head(x_local, send, s.B, s.Sl, H, s.D, s.P)
        return send

    def unpack_seq_to_head(self, recv, H):
        s = self.s
        hpr = s.heads_per_rank(H)
        if s.B == 1:   # the received chunks already are the gathered sequence
            return recv.view(1, s.S, hpr, s.D)
        x_head = torch.empty((s.B, s.S, hpr, s.D), dtype=recv.dtype, device=self.device)
        B_.usp_a2a_unpack_seq_to_head(recv, x_head, s.B, s.Sl, H, s.D, s.P)
        return x_head

    def pack_head_to_seq(self, x_head, H):
        s = self.s
        hpr = s.heads_per_rank(H)
        if s.B == 1:   # positions are already grouped by destination rank
            return x_head.view(s.P, 1, s.Sl, hpr, s.D)
        send = torch.empty((s.P, s.B, s.Sl, hpr, s.D), dtype=x_head.dtype, device=self.device)
        B_.usp_a2a_pack_head_to_seq(x_head, send, s.B, s.Sl, H, s.D, s.P)
        return send

    def unpack_head_to_seq(self, recv, H):
        s = self.s
        x_local = torch.empty((s.B, s.Sl, H, s.D), dtype=recv.dtype, device=self.device)
        B_.usp_a2a_unpack_head_to_seq(recv, x_local, s.B, s.Sl, H, s.D, s.P)
        return x_local

    # -- document boundaries from the gathered positions [P][B][Sl]
    def boundaries(self, pos_all):
        s = self.s
        B_.usp_cu_seqlens_from_position_ids(pos_all, s.B, s.S, s.P, self.cu_seqlens, self.n_docs, self.max_len,
                                            self.scan_ws, self.status)

    # -- attention over the gathered sequence of the rank's heads (P = 1 to the kernels)
    def _params(self, sinks_r):
        s = self.s
        return B_.attn_params(s.B, s.S, s.hq, s.hk, s.D, 1, self.cu_seqlens, self.n_docs, s.causal, s.window_left,
                              s.softmax_scale, sinks_r, B_.USP_IO_HEAD)

    def attention_fwd(self, q_h, k_h, v_h, sinks_r):
        s = self.s
        o_h = torch.empty_like(q_h)
        lse = torch.empty((1, s.B, s.hq, s.S), dtype=torch.float32, device=self.device)
        B_.usp_attn_fwd(self._params(sinks_r), q_h, k_h, v_h, o_h, lse, self.status)
        return o_h, lse

    def attention_bwd(self, q_h, k_h, v_h, o_h, lse, do_h, sinks_r):
        from .pipeline import backward_workspace
        prm = self._params(sinks_r)
        if self._bwd_ws is None:
            self._bwd_ws, _, _ = backward_workspace(prm, self.device)
        dq, dk, dv = torch.empty_like(q_h), torch.empty_like(k_h), torch.empty_like(v_h)
        dz = None if sinks_r is None else torch.zeros((self.s.hq,), dtype=torch.float32, device=self.device)
        B_.usp_attn_bwd(prm, q_h, k_h, v_h, o_h, lse, do_h, dq, dk, dv, dz, self._bwd_ws, self.status)
        return dq, dk, dv, dz

    def read_status(self) -> int:
        return int(self.status.item())


def _staged(t: torch.Tensor, group) -> bool:
    """gloo moves host memory: device tensors go through the host."""
    return t.is_cuda and dist.get_backend(group) == "gloo"


def all_to_all(send: torch.Tensor, group=None) -> torch.Tensor:
    """The exchange: chunk p of ``send`` (dim 0) goes to rank p; chunk p of
    the result came from rank p."""
    staged = _staged(send, group)
    src = send.cpu() if staged else send.contiguous()
    recv = torch.empty_like(src)
    dist.all_to_all_single(recv, src, group=group)
    return recv.to(send.device) if staged else recv


def all_gather(x: torch.Tensor, group=None) -> torch.Tensor:
    """[P][...]: every rank's x, in rank order."""
    staged = _staged(x, group)
    src = x.cpu() if staged else x.contiguous()
    parts = [torch.empty_like(src) for _ in range(dist.get_world_size(group))]
    dist.all_gather(parts, src, group=group)
    out = torch.stack(parts)
    return out.to(x.device) if staged else out


class UlyssesRankAttention:
    """One rank's attention layer: its sequence chunk in, its sequence chunk out."""

    def __init__(self, shape: RankShape, group=None, device=None, ops=None):
        self.s = shape
        self.group = group
        self.rank = dist.get_rank(group)
        if dist.get_world_size(group) != shape.P:
            raise ValueError(f"shape.P = {shape.P} but the group has {dist.get_world_size(group)} ranks")
        if ops is None:
            dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
            ops = LibraryOps(shape, dev)
        self.ops = ops
        self._saved = None

    def _to_head(self, x_local, H):
        return self.ops.unpack_seq_to_head(all_to_all(self.ops.pack_seq_to_head(x_local, H), self.group), H)

    def _to_seq(self, x_head, H):
        return self.ops.unpack_head_to_seq(all_to_all(self.ops.pack_head_to_seq(x_head, H), self.group), H)

    def _sinks_slice(self, sinks):
        if sinks is None:
            return None
        hq = self.s.hq
        return sinks[self.rank * hq:(self.rank + 1) * hq].contiguous()

    def forward(self, q_local, k_local, v_local, pos_local, sinks=None):
        """q/k/v ``[B][S/P][H][D]`` and position_ids ``[B][S/P]`` of this rank's
        chunk (sinks: the global ``[Hq]`` logits) -> O ``[B][S/P][Hq][D]``."""
        s = self.s
        self.ops.boundaries(all_gather(pos_local, self.group))
        q_h = self._to_head(q_local, s.Hq)
        k_h = self._to_head(k_local, s.Hkv)
        v_h = self._to_head(v_local, s.Hkv)
        o_h, lse = self.ops.attention_fwd(q_h, k_h, v_h, self._sinks_slice(sinks))
        self._saved = (q_h, k_h, v_h, o_h, lse)
        self.lse = lse
        return self._to_seq(o_h, s.Hq)

    def backward(self, do_local, sinks=None):
        """dO of this rank's chunk -> (dQ, dK, dV) of this rank's chunk and the
        gradient of the global sink logits (every rank gets all of it)."""
        s = self.s
        q_h, k_h, v_h, o_h, lse = self._saved
        do_h = self._to_head(do_local, s.Hq)
        dq_h, dk_h, dv_h, dz = self.ops.attention_bwd(q_h, k_h, v_h, o_h, lse, do_h, self._sinks_slice(sinks))
        dq = self._to_seq(dq_h, s.Hq)
        dk = self._to_seq(dk_h, s.Hkv)
        dv = self._to_seq(dv_h, s.Hkv)
        dsinks = None if dz is None else all_gather(dz, self.group).reshape(-1)
        return dq, dk, dv, dsinks
