"""One attention layer of emulated Ulysses, composed from the C entry points.

``UlyssesAttention`` owns the device buffers of one problem shape and calls
the library in the order of the attention wrapper of huggingface/accelerate
PR #4209: the q/k/v exchange (gather sequence, scatter heads), document
boundaries from the gathered position_ids, attention over the gathered
sequence, and the output exchange back; the backward swaps the exchanges.

Two ways to run the exchanges:

* fused (default when S/P is a multiple of 128): the attention kernels read
  q/dO (and, in the backward, k/v) straight from the sequence shards and
  write O/dQ/dK/dV straight back (``io_layout = USP_IO_SEQ``); the
  permutation happens in their TMA loads and stores.  Only k and v are
  exchanged explicitly for the forward (``USP_IO_SEQ_KV_HEAD``), which
  re-reads every k/v tile many times and runs faster from head-layout rows;
* explicit: ``usp_relayout_*`` kernels move the tensors between the shard
  layout and the head layout around head-layout attention.

With fewer key/value heads than ranks (P a multiple of Hkv) every key/value
head is replicated on P/Hkv ranks; the exchange back of dK/dV sums the
replicas (explicit mode), or the dK/dV kernel sums the whole query group
directly (fused mode).

The backward stores dS for the dQ pass when the workspace fits in half the
free memory; for long sequences whose whole dS does not, the dK/dV and dQ
passes run one group of key/value heads at a time over one workspace
(``plan_backward``).

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
        """Key/value heads per rank; with fewer of them than ranks each rank
        holds one replicated head."""
        return self.Hkv // self.P if self.Hkv >= self.P else 1

    @property
    def can_fuse(self) -> bool:
        return (self.S // self.P) % 128 == 0


def plan_backward(prm: B_.AttnParams, free_bytes: int, stored_ds: Optional[bool] = None, Hkv: int = 0,
                  groups_ok: bool = False, group_size: Optional[int] = None):
    """(workspace bytes, stored dS?, key/value head groups) of the backward
    calls for ``free_bytes`` of free device memory (host arithmetic only).

    With stored dS the dK/dV pass writes dS blocks and the dQ pass reads them
    instead of recomputing S and dP.  None picks it when its workspace takes
    at most half of the free memory, for all heads at once or, when
    ``groups_ok`` (fused layout), for the largest group of key/value heads
    that fits (the passes then run group by group over the same workspace);
    True insists on it (ValueError if the shape has none).  ``group_size``
    forces groups of that many key/value heads.  A group is (first key/value
    head, count); [(0, 0)] means all heads in one pass."""
    def with_group(c):
        prm_c = B_.AttnParams(*[getattr(prm, f) for f, _ in prm._fields_])
        prm_c.head_first, prm_c.head_count = 0, c
        return B_.usp_attn_bwd_fast_workspace_bytes(prm_c)

    fast = B_.usp_attn_bwd_fast_workspace_bytes(prm)
    groups = [(0, 0)]
    if group_size is not None:
        if not groups_ok or stored_ds is False:
            raise ValueError("head groups need the fused layout and the stored-dS backward")
        if not 0 < group_size <= Hkv:
            raise ValueError(f"group_size must be in [1, {Hkv}]")
        fast, stored_ds = with_group(group_size), True
        groups = [(h, min(group_size, Hkv - h)) for h in range(0, Hkv, group_size)]
    elif stored_ds is None:
        stored_ds = 0 < fast <= free_bytes // 2
        if not stored_ds and fast > 0 and groups_ok:
            for c in range(Hkv - 1, 0, -1):
                need = with_group(c)
                if 0 < need <= free_bytes // 2:
                    fast, stored_ds = need, True
                    groups = [(h, min(c, Hkv - h)) for h in range(0, Hkv, c)]
                    break
    if stored_ds and fast == 0:
        raise ValueError("this shape has no stored-dS backward (it needs a causal mask and S % 128 == 0)")
    n = fast if stored_ds else B_.usp_attn_bwd_workspace_bytes(prm)
    return n, bool(stored_ds), groups


def backward_workspace(prm: B_.AttnParams, device, stored_ds: Optional[bool] = None, Hkv: int = 0,
                       groups_ok: bool = False, group_size: Optional[int] = None):
    """The workspace tensor of the backward calls on ``device``, with the
    choices of ``plan_backward`` for the device's free memory."""
    free = torch.cuda.mem_get_info(device)[0] if stored_ds is None and group_size is None else 0
    n, stored_ds, groups = plan_backward(prm, free, stored_ds, Hkv, groups_ok, group_size)
    return torch.empty((max(n, 256),), dtype=torch.uint8, device=device), stored_ds, groups


class UlyssesAttention:
    """Buffers and calls for one shape on one device."""

    def __init__(self, shape: Shape, device="cuda", with_backward: bool = True, fused: Optional[bool] = None,
                 stored_ds: Optional[bool] = None, ds_group_size: Optional[int] = None):
        s = self.shape = shape
        self.stored_ds = stored_ds
        self.ds_group_size = ds_group_size
        self.fused = shape.can_fuse if fused is None else bool(fused)
        if self.fused and not shape.can_fuse:
            raise ValueError("fused exchanges need S/P to be a multiple of 128")
        dev = torch.device(device)
        bf = torch.bfloat16
        P, Bb, S, D = s.P, s.B, s.S, s.D
        seq_q = (P, Bb, S // P, s.Hq, D)
        seq_kv = (P, Bb, S // P, s.Hkv, D)
        self.k_head = torch.empty((P, Bb, S, s.hk, D), dtype=bf, device=dev)
        self.v_head = torch.empty((P, Bb, S, s.hk, D), dtype=bf, device=dev)
        if not self.fused:
            self.q_head = torch.empty((P, Bb, S, s.hq, D), dtype=bf, device=dev)
            self.o_head = torch.empty((P, Bb, S, s.hq, D), dtype=bf, device=dev)
        self.lse = torch.empty((P, Bb, s.hq, S), dtype=torch.float32, device=dev)
        self.o_seq = torch.empty(seq_q, dtype=bf, device=dev)
        self.cu_seqlens = torch.empty((Bb * S + 1,), dtype=torch.int32, device=dev)
        self.n_docs = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.max_len = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)
        ws = B_.usp_cu_seqlens_workspace_bytes(Bb, S)
        self.scan_ws = torch.empty((ws,), dtype=torch.uint8, device=dev)
        self.with_backward = with_backward
        if with_backward:
            if not self.fused:
                self.do_head = torch.empty((P, Bb, S, s.hq, D), dtype=bf, device=dev)
                self.dq_head = torch.empty((P, Bb, S, s.hq, D), dtype=bf, device=dev)
                self.dk_head = torch.empty((P, Bb, S, s.hk, D), dtype=bf, device=dev)
                self.dv_head = torch.empty((P, Bb, S, s.hk, D), dtype=bf, device=dev)
            self.dq_seq = torch.empty(seq_q, dtype=bf, device=dev)
            self.dk_seq = torch.empty(seq_kv, dtype=bf, device=dev)
            self.dv_seq = torch.empty(seq_kv, dtype=bf, device=dev)
            self.dsinks = torch.zeros((s.Hq,), dtype=torch.float32, device=dev)
        self._bwd_ws = None
        self.ds_groups = [(0, 0)]
        self._inputs = None  # the forward's q/k/v as the attention kernels read them

    def params(self, sinks: Optional[torch.Tensor], io: Optional[int] = None, group=(0, 0)) -> B_.AttnParams:
        s = self.shape
        if io is None:
            io = B_.USP_IO_SEQ if self.fused else B_.USP_IO_HEAD
        return B_.attn_params(s.B, s.S, s.Hq, s.Hkv, s.D, s.P, self.cu_seqlens, self.n_docs, s.causal,
                              s.window_left, s.softmax_scale, sinks, io, head_first=group[0], head_count=group[1])

    def _ws(self, prm):
        if self._bwd_ws is None:
            self._bwd_ws, self.stored_ds, self.ds_groups = backward_workspace(
                prm, self.lse.device, self.stored_ds, self.shape.Hkv, groups_ok=self.fused,
                group_size=self.ds_group_size)
        return self._bwd_ws

    # -- steps ---------------------------------------------------------------
    def exchange_qkv(self, q_seq, k_seq, v_seq, stream=None):
        s = self.shape
        if self.fused:
            # q stays in its shards; k and v go to head layout for the forward
            B_.usp_relayout_fwd(k_seq, self.k_head, s.B, s.S, s.Hkv, s.D, s.P, stream)
            B_.usp_relayout_fwd(v_seq, self.v_head, s.B, s.S, s.Hkv, s.D, s.P, stream)
            self._inputs = (q_seq, k_seq, v_seq)
            return
        B_.usp_relayout_fwd_qkv(q_seq, k_seq, v_seq, self.q_head, self.k_head, self.v_head,
                                s.B, s.S, s.Hq, s.Hkv, s.D, s.P, stream)
        self._inputs = (self.q_head, self.k_head, self.v_head)

    def boundaries(self, pos_shards, stream=None):
        s = self.shape
        B_.usp_cu_seqlens_from_position_ids(pos_shards, s.B, s.S, s.P, self.cu_seqlens, self.n_docs,
                                            self.max_len, self.scan_ws, self.status, stream)

    def attention(self, sinks=None, stream=None):
        q, k, v = self._inputs
        if self.fused:
            B_.usp_attn_fwd(self.params(sinks, B_.USP_IO_SEQ_KV_HEAD), q, self.k_head, self.v_head, self.o_seq,
                            self.lse, self.status, stream)
        else:
            B_.usp_attn_fwd(self.params(sinks), q, k, v, self.o_head, self.lse, self.status, stream)

    def exchange_out(self, stream=None):
        s = self.shape
        if not self.fused:
            B_.usp_relayout_bwd(self.o_head, self.o_seq, s.B, s.S, s.Hq, s.D, s.P, stream)

    def forward(self, q_seq, k_seq, v_seq, pos_shards, sinks=None, stream=None):
        """Sequence shards in, sequence shards out (``self.o_seq``)."""
        self.exchange_qkv(q_seq, k_seq, v_seq, stream)
        self.boundaries(pos_shards, stream)
        self.attention(sinks, stream)
        self.exchange_out(stream)
        return self.o_seq

    def backward_phases(self, do_seq, sinks=None, stream=None, marks=None, group_marks=None):
        """The backward as its separate library calls; `marks(i)` is called
        between them (for timing): 0 before, 1 after the dO exchange, 2 after
        the preprocess, 3 after dK/dV, 4 after dQ, 5 after the output exchanges.
        When the passes run in key/value head groups, marks 3 and 4 both come
        after the last group and `group_marks(g, 0)` / `group_marks(g, 1)`
        after group g's dK/dV and dQ passes."""
        s = self.shape
        prm = self.params(sinks)
        ws = self._ws(prm)
        mark = marks or (lambda i: None)
        q, k, v = self._inputs
        mark(0)
        if self.fused:
            do, o, dq, dk, dv = do_seq, self.o_seq, self.dq_seq, self.dk_seq, self.dv_seq
        else:
            B_.usp_relayout_fwd(do_seq, self.do_head, s.B, s.S, s.Hq, s.D, s.P, stream)
            do, o, dq, dk, dv = self.do_head, self.o_head, self.dq_head, self.dk_head, self.dv_head
        mark(1)
        B_.usp_attn_bwd_preprocess(prm, o, self.lse, do, self.dsinks if sinks is not None else None, ws,
                                   self.status, stream)
        mark(2)
        if len(self.ds_groups) == 1:
            B_.usp_attn_bwd_dkdv(prm, q, k, v, self.lse, do, dk, dv, ws, self.status, stream)
            mark(3)
            B_.usp_attn_bwd_dq(prm, q, k, v, self.lse, do, dq, ws, self.status, stream)
        else:  # stored dS a key/value head group at a time (both passes per group)
            gmark = group_marks or (lambda g, i: None)
            for gi, grp in enumerate(self.ds_groups):
                prm_g = self.params(None, group=grp)
                B_.usp_attn_bwd_dkdv(prm_g, q, k, v, self.lse, do, dk, dv, ws, self.status, stream)
                gmark(gi, 0)
                B_.usp_attn_bwd_dq(prm_g, q, k, v, self.lse, do, dq, ws, self.status, stream)
                gmark(gi, 1)
            mark(3)
        mark(4)
        if not self.fused:
            B_.usp_relayout_bwd(self.dq_head, self.dq_seq, s.B, s.S, s.Hq, s.D, s.P, stream)
            B_.usp_relayout_bwd(self.dk_head, self.dk_seq, s.B, s.S, s.Hkv, s.D, s.P, stream)
            B_.usp_relayout_bwd(self.dv_head, self.dv_seq, s.B, s.S, s.Hkv, s.D, s.P, stream)
        mark(5)
        return self.dq_seq, self.dk_seq, self.dv_seq

    def backward(self, do_seq, sinks=None, stream=None):
        """dO shards in; dQ/dK/dV shards out (``self.dq_seq`` ...), dsinks.
        In explicit mode this is the single ``usp_attn_bwd`` call."""
        if self.fused:
            return self.backward_phases(do_seq, sinks, stream)
        s = self.shape
        prm = self.params(sinks)
        ws = self._ws(prm)
        q, k, v = self._inputs
        B_.usp_relayout_fwd(do_seq, self.do_head, s.B, s.S, s.Hq, s.D, s.P, stream)
        B_.usp_attn_bwd(prm, q, k, v, self.o_head, self.lse, self.do_head, self.dq_head, self.dk_head,
                        self.dv_head, self.dsinks if sinks is not None else None, ws, self.status, stream)
        B_.usp_relayout_bwd(self.dq_head, self.dq_seq, s.B, s.S, s.Hq, s.D, s.P, stream)
        B_.usp_relayout_bwd(self.dk_head, self.dk_seq, s.B, s.S, s.Hkv, s.D, s.P, stream)
        B_.usp_relayout_bwd(self.dv_head, self.dv_seq, s.B, s.S, s.Hkv, s.D, s.P, stream)
        return self.dq_seq, self.dk_seq, self.dv_seq

    def read_status(self) -> int:
        return int(self.status.item())


class HybridAttention:
    """Ring x Ulysses (USP) over P = ring * ulysses emulated ranks.

    The Ulysses exchange runs inside each ring group; then ``ring`` steps
    each run the attention kernels restricted to the key/value super-chunk a
    ring rank holds at that step (``params.ring``/``ring_step``).  The forward
    merges each step's (O, LSE) into the running result
    (``usp_ring_fwd_merge``, sink folded in at the last step); the backward
    sums each step's bf16 block gradients in fp32
    (``usp_ring_grad_accumulate``) with the final LSE and D statistics
    computed once.

    Fused (default when each sequence shard is a multiple of 128 tokens): the
    kernels read and write the sequence shards directly and every
    intermediate is in that layout, so no exchange kernel runs.  Explicit:
    ``usp_hybrid_relayout_*`` move tensors to and from the hybrid head layout
    [U][B][S][H/U][D].
    """

    def __init__(self, shape: Shape, ring: int, device="cuda", with_backward: bool = True,
                 stored_ds: Optional[bool] = None, fused: Optional[bool] = None, ds_group_size: Optional[int] = None):
        s = self.shape = shape
        self.stored_ds = stored_ds
        self.ds_group_size = ds_group_size
        if ring < 1 or s.P % ring != 0:
            raise ValueError("the ring degree must divide the ranks")
        self.ring = R = ring
        self.U = U = s.P // ring
        can_fuse = (s.S // s.P) % 128 == 0
        self.fused = can_fuse if fused is None else bool(fused)
        if self.fused and not can_fuse:
            raise ValueError("fused exchanges need each sequence shard to be a multiple of 128 tokens")
        dev = torch.device(device)
        bf, f32 = torch.bfloat16, torch.float32
        Bb, S, D = s.B, s.S, s.D
        self.hq = hq = s.Hq // U
        self.hk = hk = s.Hkv // U if s.Hkv >= U else 1
        seq_q, seq_kv = (s.P, Bb, S // s.P, s.Hq, D), (s.P, Bb, S // s.P, s.Hkv, D)
        head_q, head_kv = (U, Bb, S, hq, D), (U, Bb, S, hk, D)
        lay_q, lay_kv = (seq_q, seq_kv) if self.fused else (head_q, head_kv)
        stat = (U, Bb, hq, S)
        self.k_head = torch.empty(head_kv, dtype=bf, device=dev)
        self.v_head = torch.empty(head_kv, dtype=bf, device=dev)
        if not self.fused:
            self.q_head = torch.empty(head_q, dtype=bf, device=dev)
            self.o_head = torch.empty(head_q, dtype=bf, device=dev)
        self.o_step = torch.empty(lay_q, dtype=bf, device=dev)
        self.lse_step = torch.empty(stat, dtype=f32, device=dev)
        self.o_acc = torch.empty(lay_q, dtype=f32, device=dev) if R > 1 else None
        self.lse_acc = torch.empty(stat, dtype=f32, device=dev) if R > 1 else None
        self.lse = torch.empty(stat, dtype=f32, device=dev)
        self.o_seq = torch.empty(seq_q, dtype=bf, device=dev)
        self.cu_seqlens = torch.empty((Bb * S + 1,), dtype=torch.int32, device=dev)
        self.n_docs = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.max_len = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.scan_ws = torch.empty((B_.usp_cu_seqlens_workspace_bytes(Bb, S),), dtype=torch.uint8, device=dev)
        self.with_backward = with_backward
        if with_backward:
            if not self.fused:
                self.do_head = torch.empty(head_q, dtype=bf, device=dev)
                self.dq_head = torch.empty(head_q, dtype=bf, device=dev)
                self.dk_head = torch.empty(head_kv, dtype=bf, device=dev)
                self.dv_head = torch.empty(head_kv, dtype=bf, device=dev)
            self.dq_step = torch.empty(lay_q, dtype=bf, device=dev)
            self.dk_step = torch.empty(lay_kv, dtype=bf, device=dev)
            self.dv_step = torch.empty(lay_kv, dtype=bf, device=dev)
            self.dq_acc = torch.empty(lay_q, dtype=f32, device=dev) if R > 1 else None
            self.dk_acc = torch.empty(lay_kv, dtype=f32, device=dev) if R > 1 else None
            self.dv_acc = torch.empty(lay_kv, dtype=f32, device=dev) if R > 1 else None
            self.dq_seq = torch.empty(seq_q, dtype=bf, device=dev)
            self.dk_seq = torch.empty(seq_kv, dtype=bf, device=dev)
            self.dv_seq = torch.empty(seq_kv, dtype=bf, device=dev)
            self.dsinks = torch.zeros((s.Hq,), dtype=torch.float32, device=dev)
        self._bwd_ws = None
        self.ds_groups = [(0, 0)]
        self._inputs = None

    def params(self, sinks=None, step: int = 0, io: Optional[int] = None, group=(0, 0)) -> B_.AttnParams:
        s = self.shape
        if io is None:
            io = B_.USP_IO_SEQ if self.fused else B_.USP_IO_HEAD
        return B_.attn_params(s.B, s.S, s.Hq, s.Hkv, s.D, self.U, self.cu_seqlens, self.n_docs, s.causal,
                              s.window_left, s.softmax_scale, sinks, io, self.ring, step, group[0], group[1])

    def _flags(self, step: int) -> int:
        return (B_.USP_RING_FIRST if step == 0 else 0) | (B_.USP_RING_LAST if step == self.ring - 1 else 0)

    def forward_phases(self, q_seq, k_seq, v_seq, pos_shards, sinks=None, stream=None, marks=None):
        """marks(i): 0 before, 1 after the q/k/v exchange, 2 after the document
        boundaries, 3 after the ring steps and merges, 4 after the O exchange."""
        s = self.shape
        mark = marks or (lambda i: None)
        mark(0)
        if self.fused:
            # q stays in its shards; k and v go to the hybrid head layout for the forward
            B_.usp_hybrid_relayout_fwd(k_seq, self.k_head, s.B, s.S, s.Hkv, s.D, self.ring, self.U, stream)
            B_.usp_hybrid_relayout_fwd(v_seq, self.v_head, s.B, s.S, s.Hkv, s.D, self.ring, self.U, stream)
            self._inputs = (q_seq, k_seq, v_seq)
            o_out = self.o_seq
        else:
            B_.usp_hybrid_relayout_fwd_qkv(q_seq, k_seq, v_seq, self.q_head, self.k_head, self.v_head,
                                           s.B, s.S, s.Hq, s.Hkv, s.D, self.ring, self.U, stream)
            self._inputs = (self.q_head, self.k_head, self.v_head)
            o_out = self.o_head
        mark(1)
        B_.usp_cu_seqlens_from_position_ids(pos_shards, s.B, s.S, s.P, self.cu_seqlens, self.n_docs,
                                            self.max_len, self.scan_ws, self.status, stream)
        mark(2)
        q, k, v = self._inputs
        io_fwd = B_.USP_IO_SEQ_KV_HEAD if self.fused else B_.USP_IO_HEAD
        for st in range(self.ring):
            B_.usp_attn_fwd(self.params(None, st, io_fwd), q, self.k_head, self.v_head, self.o_step, self.lse_step,
                            self.status, stream)
            B_.usp_ring_fwd_merge(self.params(sinks, st), self.o_step, self.lse_step, self.o_acc, self.lse_acc,
                                  o_out, self.lse, self._flags(st), stream)
        mark(3)
        if not self.fused:
            B_.usp_hybrid_relayout_bwd(self.o_head, self.o_seq, s.B, s.S, s.Hq, s.D, self.ring, self.U, stream)
        mark(4)
        return self.o_seq

    def forward(self, q_seq, k_seq, v_seq, pos_shards, sinks=None, stream=None):
        return self.forward_phases(q_seq, k_seq, v_seq, pos_shards, sinks, stream)

    def backward_phases(self, do_seq, sinks=None, stream=None, marks=None):
        """marks(i): 0 before, 1 after the dO exchange, 2 after the
        statistics, 3 after the dK/dV ring steps, 4 after the dQ ring steps,
        5 after the dQ/dK/dV exchanges."""
        s = self.shape
        mark = marks or (lambda i: None)
        prm = self.params(sinks, 0)
        if self._bwd_ws is None:
            self._bwd_ws, self.stored_ds, self.ds_groups = backward_workspace(
                prm, self.lse.device, self.stored_ds, s.Hkv, groups_ok=self.fused, group_size=self.ds_group_size)
        ws = self._bwd_ws
        q, k, v = self._inputs
        mark(0)
        if self.fused:
            do, o = do_seq, self.o_seq
            dq_out, dk_out, dv_out = self.dq_seq, self.dk_seq, self.dv_seq
        else:
            B_.usp_hybrid_relayout_fwd(do_seq, self.do_head, s.B, s.S, s.Hq, s.D, self.ring, self.U, stream)
            do, o = self.do_head, self.o_head
            dq_out, dk_out, dv_out = self.dq_head, self.dk_head, self.dv_head
        mark(1)
        B_.usp_attn_bwd_preprocess(prm, o, self.lse, do, self.dsinks if sinks is not None else None, ws,
                                   self.status, stream)
        mark(2)
        if len(self.ds_groups) == 1:
            for st in range(self.ring):
                B_.usp_attn_bwd_dkdv(self.params(None, st), q, k, v, self.lse, do, self.dk_step, self.dv_step, ws,
                                     self.status, stream)
                B_.usp_ring_grad_accumulate(self.dk_step, self.dk_acc, dk_out, self._flags(st), stream)
                B_.usp_ring_grad_accumulate(self.dv_step, self.dv_acc, dv_out, self._flags(st), stream)
            mark(3)
            for st in range(self.ring):
                B_.usp_attn_bwd_dq(self.params(None, st), q, k, v, self.lse, do, self.dq_step, ws, self.status,
                                   stream)
                B_.usp_ring_grad_accumulate(self.dq_step, self.dq_acc, dq_out, self._flags(st), stream)
        else:  # stored dS a key/value head group at a time (both passes per group)
            for st in range(self.ring):
                for grp in self.ds_groups:
                    prm_g = self.params(None, st, group=grp)
                    B_.usp_attn_bwd_dkdv(prm_g, q, k, v, self.lse, do, self.dk_step, self.dv_step, ws, self.status,
                                         stream)
                    B_.usp_attn_bwd_dq(prm_g, q, k, v, self.lse, do, self.dq_step, ws, self.status, stream)
                B_.usp_ring_grad_accumulate(self.dk_step, self.dk_acc, dk_out, self._flags(st), stream)
                B_.usp_ring_grad_accumulate(self.dv_step, self.dv_acc, dv_out, self._flags(st), stream)
                B_.usp_ring_grad_accumulate(self.dq_step, self.dq_acc, dq_out, self._flags(st), stream)
            mark(3)
        mark(4)
        if not self.fused:
            B_.usp_hybrid_relayout_bwd(self.dq_head, self.dq_seq, s.B, s.S, s.Hq, s.D, self.ring, self.U, stream)
            B_.usp_hybrid_relayout_bwd(self.dk_head, self.dk_seq, s.B, s.S, s.Hkv, s.D, self.ring, self.U, stream)
            B_.usp_hybrid_relayout_bwd(self.dv_head, self.dv_seq, s.B, s.S, s.Hkv, s.D, self.ring, self.U, stream)
        mark(5)
        return self.dq_seq, self.dk_seq, self.dv_seq

    def backward(self, do_seq, sinks=None, stream=None):
        return self.backward_phases(do_seq, sinks, stream)

    def read_status(self) -> int:
        return int(self.status.item())
