"""One attention layer of emulated Ulysses, composed from the C entry points.

``UlyssesAttention`` owns the device buffers of one problem shape and calls
the library in the order of the attention wrapper of huggingface/accelerate
PR #4209: the q/k/v exchange (gather sequence, scatter heads), document
boundaries from the gathered position_ids, attention over the gathered
sequence, and the output exchange back; the backward swaps the exchanges.
torch only allocates the buffers and supplies the stream; every step runs in
the library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import binding as B_


@dataclass
class Shape:
    B: int
    S: int
    Hq: int
    Hkv: int
    D: int
    P: int
    causal: bool = True
    window_left: int = -1
    softmax_scale: float = 0.0

    @property
    def hq(self):
        return self.Hq // self.P

    @property
    def hk(self):
        return self.Hkv // self.P


class UlyssesAttention:
    """Buffers and calls for one shape on one device."""

    def __init__(self, shape: Shape, device="cuda", with_backward: bool = True):
        s = self.shape = shape
        dev = torch.device(device)
        bf = torch.bfloat16
        P, Bb, S, D = s.P, s.B, s.S, s.D
        self.q_head = torch.empty((P, Bb, S, s.hq, D), dtype=bf, device=dev)
        self.k_head = torch.empty((P, Bb, S, s.hk, D), dtype=bf, device=dev)
        self.v_head = torch.empty((P, Bb, S, s.hk, D), dtype=bf, device=dev)
        self.o_head = torch.empty((P, Bb, S, s.hq, D), dtype=bf, device=dev)
        self.lse = torch.empty((P, Bb, s.hq, S), dtype=torch.float32, device=dev)
        self.o_seq = torch.empty((P, Bb, S // P, s.Hq, D), dtype=bf, device=dev)
        self.cu_seqlens = torch.empty((Bb * S + 1,), dtype=torch.int32, device=dev)
        self.n_docs = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.max_len = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)
        ws = B_.usp_cu_seqlens_workspace_bytes(Bb, S)
        self.scan_ws = torch.empty((ws,), dtype=torch.uint8, device=dev)
        self.with_backward = with_backward
        if with_backward:
            self.do_head = torch.empty_like(self.o_head)
            self.dq_head = torch.empty_like(self.q_head)
            self.dk_head = torch.empty_like(self.k_head)
            self.dv_head = torch.empty_like(self.v_head)
            self.dq_seq = torch.empty((P, Bb, S // P, s.Hq, D), dtype=bf, device=dev)
            self.dk_seq = torch.empty((P, Bb, S // P, s.Hkv, D), dtype=bf, device=dev)
            self.dv_seq = torch.empty((P, Bb, S // P, s.Hkv, D), dtype=bf, device=dev)
            self.dsinks = torch.zeros((s.Hq,), dtype=torch.float32, device=dev)
        self._bwd_ws = None

    def params(self, sinks: Optional[torch.Tensor]) -> B_.AttnParams:
        s = self.shape
        return B_.attn_params(s.B, s.S, s.Hq, s.Hkv, s.D, s.P, self.cu_seqlens, self.n_docs, s.causal,
                              s.window_left, s.softmax_scale, sinks)

    # -- steps ---------------------------------------------------------------
    def exchange_qkv(self, q_seq, k_seq, v_seq, stream=None):
        s = self.shape
        B_.usp_relayout_fwd_qkv(q_seq, k_seq, v_seq, self.q_head, self.k_head, self.v_head,
                                s.B, s.S, s.Hq, s.Hkv, s.D, s.P, stream)

    def boundaries(self, pos_shards, stream=None):
        s = self.shape
        B_.usp_cu_seqlens_from_position_ids(pos_shards, s.B, s.S, s.P, self.cu_seqlens, self.n_docs,
                                            self.max_len, self.scan_ws, self.status, stream)

    def attention(self, sinks=None, stream=None):
        B_.usp_attn_fwd(self.params(sinks), self.q_head, self.k_head, self.v_head, self.o_head, self.lse,
                        self.status, stream)

    def exchange_out(self, stream=None):
        s = self.shape
        B_.usp_relayout_bwd(self.o_head, self.o_seq, s.B, s.S, s.Hq, s.D, s.P, stream)

    def forward(self, q_seq, k_seq, v_seq, pos_shards, sinks=None, stream=None):
        """Sequence shards in, sequence shards out (``self.o_seq``)."""
        self.exchange_qkv(q_seq, k_seq, v_seq, stream)
        self.boundaries(pos_shards, stream)
        self.attention(sinks, stream)
        self.exchange_out(stream)
        return self.o_seq

    def backward(self, do_seq, sinks=None, stream=None):
        """dO shards in; dQ/dK/dV shards out (``self.dq_seq`` ...), dsinks."""
        s = self.shape
        prm = self.params(sinks)
        if self._bwd_ws is None:
            n = B_.usp_attn_bwd_workspace_bytes(prm)
            self._bwd_ws = torch.empty((max(n, 256),), dtype=torch.uint8, device=self.o_head.device)
        B_.usp_relayout_fwd(do_seq, self.do_head, s.B, s.S, s.Hq, s.D, s.P, stream)
        B_.usp_attn_bwd(prm, self.q_head, self.k_head, self.v_head, self.o_head, self.lse, self.do_head,
                        self.dq_head, self.dk_head, self.dv_head, self.dsinks if sinks is not None else None,
                        self._bwd_ws, self.status, stream)
        B_.usp_relayout_bwd(self.dq_head, self.dq_seq, s.B, s.S, s.Hq, s.D, s.P, stream)
        B_.usp_relayout_bwd(self.dk_head, self.dk_seq, s.B, s.S, s.Hkv, s.D, s.P, stream)
        B_.usp_relayout_bwd(self.dv_head, self.dv_seq, s.B, s.S, s.Hkv, s.D, s.P, stream)
        return self.dq_seq, self.dk_seq, self.dv_seq

    def read_status(self) -> int:
        return int(self.status.item())
