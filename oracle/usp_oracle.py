"""fp64 CPU oracle for the Ulysses sequence-parallel attention hot path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` (``cpu_baseline`` and ``--impl reference``) use it.  It
shares no code, header, table or helper with the CUDA library; its inputs come
from the seeded generators in ``usp_workloads`` (which hold no arithmetic of
the method) or from the tests themselves.

Everything here is the plain definition, written out in float64 with numpy:

* ``relayout_fwd`` / ``relayout_bwd``: the two all-to-all exchanges of the
  attention wrapper, ``_gather_seq_scatter_heads`` (queries, keys and values go
  from "my sequence chunk, all heads" to "whole sequence, my heads") and
  ``_gather_heads_scatter_seq`` (the output goes back).  The backward of each
  is the other one ("swap scatter and gather").  huggingface/accelerate PR
  #4209, the comment on the four ``_SeqAllToAll.apply`` call sites.
* ``cu_seqlens_from_position_ids``: document boundaries of the *gathered*
  sequence, recomputed from the gathered position_ids instead of the
  collator's per-shard ``cu_seq_lens_q/k``/``max_length_q/k`` (PR #4209, the
  comment on stale kwargs: 41.8% of logits mismatched when the per-shard ones
  were used; and the comment moving the position_ids gather into the forward
  pre-hook, one gather per forward shared by every layer).
* ``attention_fwd`` / ``attention_bwd``: varlen softmax attention over the
  gathered sequence of one rank's heads: documents never see each other,
  causal, optional sliding window, GQA (ArcticTraining PR #45, "gqa works"),
  and one sink logit per head sliced to the rank's heads (PR #4209, the
  gpt-oss finding about ``s_aux``).  The gradients are the textbook ones of
  that function.
* ``hybrid_fwd`` / ``hybrid_bwd``: yunchang's ring x Ulysses hybrid (USP):
  the ranks form a (ring, ulysses) mesh with the Ulysses dimension innermost
  and contiguous ("basic") sequence chunks; the Ulysses exchange runs inside
  each ring group, then the ring passes key/value super-chunks around and
  merges the partial outputs through their log-sum-exp
  (feifeibear/long-context-attention issue #135, the device-mesh script).
* ``ulysses_fwd`` / ``ulysses_bwd``: the whole emulated P-rank path, and
  ``unsharded_fwd`` / ``unsharded_bwd``: the same attention run on the
  unsharded tensors, the pages' correctness reference (PR #4209 checks the
  sharded forward and backward against an unsharded run; the yunchang script compares against
  ``flash_attn_func`` on the full tensors).

With fewer key/value heads than ranks (P a multiple of Hkv), each key/value
head is replicated on P/Hkv ranks and the exchange back of dK/dV sums the
replicas (kv-head replication, a follow-up listed in PR #4209).

Readings where the pages are silent (each is listed in the design notes):
the softmax scale defaults to 1/sqrt(D) (``flash_attn_func`` is called with no
scale in the yunchang script); a sink is an extra logit with no value, not
multiplied by the scale, and the log-sum-exp includes it; window_left=w lets
query i see keys j with i-j <= w (w=127 for "sliding window 128"); a document
starts at every row start and wherever position_ids is 0; LSE is the natural
log; heads go to ranks in contiguous blocks; sequence chunks are contiguous in
rank order.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, library special cases, finite differences, semantic
encodings); none is "parity unpinned".
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np

__all__ = [
    "OracleError",
    "relayout_fwd", "relayout_bwd",
    "cu_seqlens_from_position_ids", "gather_position_ids",
    "attention_fwd", "attention_fwd_rows", "attention_bwd", "attention_bwd_rows",
    "attention_bwd_keys",
    "ulysses_fwd", "ulysses_bwd", "unsharded_fwd", "unsharded_bwd",
    "visible_pairs",
    "hybrid_relayout_fwd", "hybrid_relayout_bwd", "ring_block_fwd", "ring_merge",
    "hybrid_fwd", "hybrid_bwd",
    "a2a_pack_seq_to_head", "a2a_unpack_seq_to_head", "a2a_pack_head_to_seq", "a2a_unpack_head_to_seq",
    "all_to_all",
]


class OracleError(ValueError):
    """Raised for inputs the method refuses (indivisible heads, bad positions)."""


# ---------------------------------------------------------------------------
# all-to-all exchanges (accelerate PR #4209, _gather_seq_scatter_heads /
# _gather_heads_scatter_seq)
# ---------------------------------------------------------------------------

def _check_divisible(S: int, H: int, P: int, replicate: bool = False) -> None:
    # The torch backend refuses an sp size that does not divide the heads
    # (accelerate PR #4209, "What does this PR do?", the list under "How").
    # Key/value heads fewer than the ranks are replicated instead when the
    # ranks are a multiple of them (the kv-head replication the same PR lists
    # as a follow-up).
    if P <= 0:
        raise OracleError("sp size must be positive")
    if H % P != 0 and not (replicate and H < P and P % H == 0):
        raise OracleError(f"sp size {P} does not divide {H} heads")
    if S % P != 0:
        raise OracleError(f"sp size {P} does not divide sequence length {S}")


def relayout_fwd(x_seq: np.ndarray, P: int, replicate: bool = False) -> np.ndarray:
    """Gather the sequence, scatter the heads.

    ``x_seq`` is ``[P][B][S/P][H][D]``: rank r' holds positions
    ``[r'*S/P, (r'+1)*S/P)`` of every row, all heads.  The result is
    ``[P][B][S][H/P][D]``: rank r holds every position, heads
    ``[r*H/P, (r+1)*H/P)``.  Element for element::

        out[r][b][r'*S/P + s'][j][d] = x_seq[r'][b][s'][r*H/P + j][d]

    Written as a reshape that names the two rank axes and a transpose that
    swaps them, which is that formula.

    With ``replicate`` and fewer heads than ranks (H < P, P a multiple of H),
    each head goes to the P/H ranks r with r // (P/H) equal to it, and every
    rank holds one head::

        out[r][b][r'*S/P + s'][0][d] = x_seq[r'][b][s'][r // (P/H)][d]
    """
    Px, B, Sl, H, D = x_seq.shape
    if Px != P:
        raise OracleError("leading axis must be the rank axis")
    _check_divisible(Sl * P, H, P, replicate)
    if H < P:
        owner = np.arange(P) // (P // H)        # the head rank r receives
        y = x_seq[:, :, :, owner, :]            # [r'][b][s'][r][d]
        y = y.transpose(3, 1, 0, 2, 4)          # [r][b][r'][s'][d]
        return np.ascontiguousarray(y).reshape(P, B, P * Sl, 1, D)
    Hp = H // P
    y = x_seq.reshape(P, B, Sl, P, Hp, D)       # [r'][b][s'][r][j][d]
    y = y.transpose(3, 1, 0, 2, 4, 5)           # [r][b][r'][s'][j][d]
    return np.ascontiguousarray(y).reshape(P, B, P * Sl, Hp, D)


def relayout_bwd(x_head: np.ndarray, P: int, heads: Optional[int] = None) -> np.ndarray:
    """Gather the heads, scatter the sequence: the inverse exchange.

    ``x_head`` is ``[P][B][S][H/P][D]``; the result is ``[P][B][S/P][H][D]``::

        out[r'][b][s'][r*H/P + j][d] = x_head[r][b][r'*S/P + s'][j][d]

    With ``heads`` = H < P (replicated heads, one per rank) the exchange back
    of a gradient is the adjoint of the replication: the replicas are summed::

        out[r'][b][s'][h][d] = sum over r with r // (P/H) == h of x_head[r][b][r'*S/P + s'][0][d]
    """
    Px, B, S, Hp, D = x_head.shape
    if Px != P:
        raise OracleError("leading axis must be the rank axis")
    H = Hp * P if heads is None else heads
    _check_divisible(S, H, P, replicate=True)
    Sl = S // P
    if H < P:
        if Hp != 1:
            raise OracleError("replicated heads hold one head per rank")
        y = x_head.reshape(H, P // H, B, P, Sl, D).sum(axis=1)   # [h][b][r'][s'][d]
        y = y.transpose(2, 1, 3, 0, 4)                           # [r'][b][s'][h][d]
        return np.ascontiguousarray(y)
    if H != Hp * P:
        raise OracleError("head count does not match the head-layout tensor")
    y = x_head.reshape(P, B, P, Sl, Hp, D)      # [r][b][r'][s'][j][d]
    y = y.transpose(2, 1, 3, 0, 4, 5)           # [r'][b][s'][r][j][d]
    return np.ascontiguousarray(y).reshape(P, B, Sl, P * Hp, D)


# ---------------------------------------------------------------------------
# one real rank's side of the same exchanges: what it sends to every other
# rank and how it lays out what it receives (the all-to-all of the comment on
# the four _SeqAllToAll.apply call sites, seen from rank r)
# ---------------------------------------------------------------------------

def a2a_pack_seq_to_head(x_local: np.ndarray, P: int, replicate: bool = False) -> np.ndarray:
    """Rank r's send buffer of the seq->head exchange: chunk p holds rank p's
    heads of r's sequence chunk.  ``x_local`` is ``[B][Sl][H][D]``; the result
    is ``[P][B][Sl][H/P][D]`` with ``send[p][b][s][j][d] = x_local[b][s][p*H/P + j][d]``,
    or, with ``replicate`` and H < P, ``send[p][b][s][0][d] = x_local[b][s][p // (P/H)][d]``."""
    B, Sl, H, D = x_local.shape
    _check_divisible(Sl * P, H, P, replicate)
    if H < P:
        owner = np.arange(P) // (P // H)
        y = x_local[:, :, owner, :]                  # [b][s][p][d]
        return np.ascontiguousarray(y.transpose(2, 0, 1, 3)).reshape(P, B, Sl, 1, D)
    y = x_local.reshape(B, Sl, P, H // P, D)         # [b][s][p][j][d]
    return np.ascontiguousarray(y.transpose(2, 0, 1, 3, 4))


def a2a_unpack_seq_to_head(recv: np.ndarray) -> np.ndarray:
    """The received chunks ``[P][B][Sl][hpr][D]`` (chunk p = rank p's positions)
    as the whole sequence of the rank's heads, ``[B][P*Sl][hpr][D]``:
    ``x_head[b][p*Sl + s] = recv[p][b][s]``."""
    P, B, Sl, hpr, D = recv.shape
    return np.ascontiguousarray(recv.transpose(1, 0, 2, 3, 4)).reshape(B, P * Sl, hpr, D)


def a2a_pack_head_to_seq(x_head: np.ndarray, P: int) -> np.ndarray:
    """Rank r's send buffer of the head->seq exchange: chunk p holds rank p's
    positions of r's heads, ``send[p][b][s] = x_head[b][p*Sl + s]``."""
    B, S, hpr, D = x_head.shape
    if S % P != 0:
        raise OracleError(f"sp size {P} does not divide sequence length {S}")
    y = x_head.reshape(B, P, S // P, hpr, D)
    return np.ascontiguousarray(y.transpose(1, 0, 2, 3, 4))


def a2a_unpack_head_to_seq(recv: np.ndarray, heads: Optional[int] = None) -> np.ndarray:
    """The received chunks ``[P][B][Sl][hpr][D]`` (chunk p = rank p's heads) as
    the rank's sequence chunk with all heads ``[B][Sl][H][D]``:
    ``x_local[b][s][p*hpr + j] = recv[p][b][s][j]``.  With ``heads`` = H < P
    (replicated heads) the replicas' values are summed, the adjoint of the
    replication: ``x_local[b][s][h] = sum over p with p // (P/H) == h of recv[p][b][s][0]``."""
    P, B, Sl, hpr, D = recv.shape
    H = hpr * P if heads is None else heads
    if H < P:
        if hpr != 1 or P % H != 0:
            raise OracleError("replicated heads hold one head per rank")
        y = recv.reshape(H, P // H, B, Sl, D).sum(axis=1)     # [h][b][s][d]
        return np.ascontiguousarray(y.transpose(1, 2, 0, 3))
    if H != hpr * P:
        raise OracleError("head count does not match the received chunks")
    return np.ascontiguousarray(recv.transpose(1, 2, 0, 3, 4)).reshape(B, Sl, H, D)


def all_to_all(sends):
    """The collective itself for P ranks at once: rank r receives chunk r of
    every rank's send buffer, in source-rank order (``recv_r[p] = send_p[r]``)."""
    P = len(sends)
    return [np.stack([sends[p][r] for p in range(P)]) for r in range(P)]


# ---------------------------------------------------------------------------
# position_ids gather and document boundaries (accelerate PR #4209)
# ---------------------------------------------------------------------------

def gather_position_ids(pos_shards: np.ndarray) -> np.ndarray:
    """[P][B][S/P] shards -> [B][S]: the all-gather done once per forward."""
    P, B, Sl = pos_shards.shape
    out = np.empty((B, P * Sl), dtype=np.int64)
    for r in range(P):
        out[:, r * Sl:(r + 1) * Sl] = pos_shards[r]
    return out


def cu_seqlens_from_position_ids(pos_shards: np.ndarray) -> Tuple[np.ndarray, int, int]:
    """Document boundaries of the gathered sequence, one sequential pass.

    A document starts at every row start and wherever the gathered position is
    0 (position_ids count 0, 1, 2, ... inside each packed document).  Returns
    ``(cu_seqlens, n_docs, max_len)`` with ``cu_seqlens`` int32 of length
    ``n_docs + 1``, ``cu_seqlens[0] = 0``, ``cu_seqlens[n_docs] = B*S`` and
    ``max_len`` the longest document.  Negative positions are refused.
    """
    pos = gather_position_ids(np.asarray(pos_shards))
    B, S = pos.shape
    flat = pos.reshape(-1)
    starts = []
    for i in range(flat.shape[0]):
        p = int(flat[i])
        if p < 0:
            raise OracleError(f"negative position id {p} at gathered index {i}")
        if i % S == 0 or p == 0:
            starts.append(i)
    cu = starts + [B * S]
    max_len = 0
    for a, b in zip(cu[:-1], cu[1:]):
        max_len = max(max_len, b - a)
    return np.asarray(cu, dtype=np.int32), len(starts), max_len


# ---------------------------------------------------------------------------
# varlen attention over one rank's heads
# ---------------------------------------------------------------------------

def _visible(i0: int, i1: int, ka: int, kb: int, causal: bool, window_left: int,
             a: Optional[int] = None, b: Optional[int] = None) -> np.ndarray:
    """Boolean [i1-i0][kb-ka]: may query i (global index) see key j in [ka, kb)?

    Queries and keys belong to the document [a, b) (default: [ka, kb))."""
    a = ka if a is None else a
    b = kb if b is None else b
    i = np.arange(i0, i1)[:, None]
    j = np.arange(ka, kb)[None, :]
    vis = (j >= a) & (j < b) & np.ones((i1 - i0, kb - ka), dtype=bool)
    if causal:
        vis &= j <= i
    if window_left >= 0:
        vis &= (i - j) <= window_left
        if not causal:
            vis &= (j - i) <= window_left
    return vis


def _block_key_span(i0: int, i1: int, a: int, b: int, causal: bool, window_left: int):
    """Keys of document [a, b) that at least one query in [i0, i1) may see."""
    ka, kb = a, b
    if causal:
        kb = i1
    if window_left >= 0:
        ka = max(a, i0 - window_left)
        if not causal:
            kb = min(b, i1 + window_left)
    return ka, kb


def _doc_row_blocks(a: int, b: int, block: int):
    for i0 in range(a, b, block):
        yield i0, min(b, i0 + block)


def attention_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, cu_seqlens: np.ndarray,
                  causal: bool = True, window_left: int = -1, scale: Optional[float] = None,
                  sinks: Optional[np.ndarray] = None, row_block: int = 512,
                  heads: Optional[list] = None):
    """Softmax attention of one rank over its gathered sequence.

    ``q`` [T][hq][D], ``k``/``v`` [T][hk][D] (T = B*S tokens, every document a
    contiguous range ``[cu[n], cu[n+1])``), ``sinks`` [hq] or None.  Query
    head h reads key/value head ``h // (hq/hk)``.  For query i of document
    [a, b) the visible keys are j in [a, b) with j <= i (causal) and
    i - j <= window_left (window).  With s_ij = scale * q_i . k_j and t the
    head's sink logit (if any)::

        LSE_i = log( sum_j exp(s_ij) + exp(t) )
        O_i   = sum_j exp(s_ij - LSE_i) v_j

    Returns ``O`` [T][hq][D] and ``LSE`` [hq][T] in float64.  ``heads``
    restricts the work to those query heads (other outputs stay NaN).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, hq, D = q.shape
    hk = k.shape[1]
    if hq % hk != 0:
        raise OracleError("query heads must be a multiple of key/value heads")
    G = hq // hk
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    cu = [int(x) for x in cu_seqlens]
    O = np.full((T, hq, D), np.nan)
    LSE = np.full((hq, T), np.nan)
    for h in (range(hq) if heads is None else heads):
        kh = h // G
        t = None if sinks is None else float(sinks[h])
        for a, b in zip(cu[:-1], cu[1:]):
            for i0, i1 in _doc_row_blocks(a, b, row_block):
                # keys outside [ka, kb) are hidden from every row of the block
                ka, kb = _block_key_span(i0, i1, a, b, causal, window_left)
                K = k[ka:kb, kh]
                V = v[ka:kb, kh]
                s = scale * (q[i0:i1, h] @ K.T)
                s = np.where(_visible(i0, i1, ka, kb, causal, window_left, a, b), s, -np.inf)
                m = s.max(axis=1)
                if t is not None:
                    m = np.maximum(m, t)
                e = np.exp(s - m[:, None])
                z = e.sum(axis=1)
                if t is not None:
                    z = z + np.exp(t - m)
                LSE[h, i0:i1] = m + np.log(z)
                O[i0:i1, h] = (e / z[:, None]) @ V
    return O, LSE


def attention_fwd_rows(q, k, v, cu_seqlens, rows, head: int, causal: bool = True,
                       window_left: int = -1, scale: Optional[float] = None,
                       sink: Optional[float] = None):
    """``attention_fwd`` for the listed query rows of one query head only.

    Same definition, evaluated row by row, so that single rows of a very long
    document can be checked without computing the whole head.  Returns
    ``O`` [len(rows)][D] and ``LSE`` [len(rows)].
    """
    T, hq, D = q.shape
    G = hq // k.shape[1]
    kh = head // G
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    O = np.empty((len(rows), D))
    LSE = np.empty(len(rows))
    for n, i in enumerate(rows):
        d = int(np.searchsorted(cu, i, side="right")) - 1
        a, b = int(cu[d]), int(cu[d + 1])
        ka, kb = _block_key_span(i, i + 1, a, b, causal, window_left)
        s = scale * (np.asarray(k[ka:kb, kh], np.float64) @ np.asarray(q[i, head], np.float64))
        s = np.where(_visible(i, i + 1, ka, kb, causal, window_left, a, b)[0], s, -np.inf)
        m = s.max() if sink is None else max(s.max(), sink)
        e = np.exp(s - m)
        z = e.sum() + (0.0 if sink is None else np.exp(sink - m))
        LSE[n] = m + np.log(z)
        O[n] = (e / z) @ np.asarray(v[ka:kb, kh], np.float64)
    return O, LSE


def attention_bwd(q, k, v, o, lse, do, cu_seqlens, causal: bool = True, window_left: int = -1,
                  scale: Optional[float] = None, sinks: Optional[np.ndarray] = None,
                  row_block: int = 512, heads: Optional[list] = None):
    """Gradients of ``attention_fwd`` for the loss sum(O * dO).

    With P_ij = exp(s_ij - LSE_i) (zero where key j is hidden from i) and
    D_i = sum_d dO_id O_id::

        dV_j  = sum_i P_ij dO_i
        dP_ij = dO_i . v_j
        dS_ij = P_ij (dP_ij - D_i)
        dQ_i  = scale sum_j dS_ij k_j
        dK_j  = scale sum_i dS_ij q_i
        dt    = -sum_i exp(t - LSE_i) D_i          (sink logit of the head)

    Key/value gradients of a GQA group sum over its query heads.  Returns
    ``dq, dk, dv, dsinks`` (dsinks None without sinks), float64.  ``heads``
    restricts the sums to those query heads (a whole GQA group gives that
    key/value head's complete gradients).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    T, hq, D = q.shape
    hk = k.shape[1]
    G = hq // hk
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    cu = [int(x) for x in cu_seqlens]
    Dvec = np.sum(do * o, axis=2)                  # [T][hq]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dsinks = None if sinks is None else np.zeros(hq)
    for h in (range(hq) if heads is None else heads):
        kh = h // G
        for a, b in zip(cu[:-1], cu[1:]):
            for i0, i1 in _doc_row_blocks(a, b, row_block):
                ka, kb = _block_key_span(i0, i1, a, b, causal, window_left)
                K = k[ka:kb, kh]
                V = v[ka:kb, kh]
                s = scale * (q[i0:i1, h] @ K.T)
                vis = _visible(i0, i1, ka, kb, causal, window_left, a, b)
                Pm = np.where(vis, np.exp(s - lse[h, i0:i1][:, None]), 0.0)
                dv[ka:kb, kh] += Pm.T @ do[i0:i1, h]
                dP = do[i0:i1, h] @ V.T
                dS = Pm * (dP - Dvec[i0:i1, h][:, None])
                dq[i0:i1, h] += scale * (dS @ K)
                dk[ka:kb, kh] += scale * (dS.T @ q[i0:i1, h])
                if dsinks is not None:
                    dsinks[h] += -np.sum(np.exp(float(sinks[h]) - lse[h, i0:i1]) * Dvec[i0:i1, h])
    return dq, dk, dv, dsinks


def attention_bwd_rows(q, k, v, do, cu_seqlens, rows, head: int, causal: bool = True,
                       window_left: int = -1, scale: Optional[float] = None,
                       sink: Optional[float] = None, key_window: Optional[Tuple[int, int]] = None):
    """dQ of the listed query rows of one head, each row from its own forward.

    Row t needs only its own O_t, LSE_t and D_t = dO_t . O_t, so a single row
    of a very long document is checked without the whole head.  With
    ``key_window = (k0, k1)`` only the keys in [k0, k1) contribute to the sum
    (one ring step's share of dQ); O, LSE and D stay those of the whole row.
    """
    T, hq, D = q.shape
    kh = head // (hq // k.shape[1])
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    O, L = attention_fwd_rows(q, k, v, cu_seqlens, rows, head, causal, window_left, scale, sink)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    dq = np.empty((len(rows), D))
    for n, t in enumerate(rows):
        d = int(np.searchsorted(cu, t, side="right")) - 1
        a, b = int(cu[d]), int(cu[d + 1])
        ka, kb = _block_key_span(t, t + 1, a, b, causal, window_left)
        K = np.asarray(k[ka:kb, kh], np.float64)
        V = np.asarray(v[ka:kb, kh], np.float64)
        dot = np.asarray(do[t, head], np.float64)
        s = scale * (K @ np.asarray(q[t, head], np.float64))
        vis = _visible(t, t + 1, ka, kb, causal, window_left, a, b)[0]
        if key_window is not None:
            kk = np.arange(ka, kb)
            vis = vis & (kk >= key_window[0]) & (kk < key_window[1])
        Pm = np.where(vis, np.exp(s - L[n]), 0.0)
        dS = Pm * (V @ dot - dot @ O[n])
        dq[n] = scale * (dS @ K)
    return dq


def attention_bwd_keys(q, k, v, do, cu_seqlens, keys, kv_head: int, causal: bool = True,
                       window_left: int = -1, scale: Optional[float] = None,
                       sinks: Optional[np.ndarray] = None, row_window: Optional[Tuple[int, int]] = None):
    """dK and dV of the listed keys of one key/value head.

    Every query row that sees one of the keys, in every query head of the
    group, gets its O, LSE and D from its own forward (``attention_fwd_rows``);
    then dV_u = sum P_tu dO_t and dK_u = scale sum dS_tu q_t over those rows.
    Cheap when the keys sit near the end of their document.  With
    ``row_window = (q0, q1)`` only the rows in [q0, q1) contribute (one ring
    step's share of dK/dV).
    """
    T, hq, D = q.shape
    G = hq // k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    dk = np.zeros((len(keys), D))
    dv = np.zeros((len(keys), D))
    for h in range(kv_head * G, (kv_head + 1) * G):
        sink = None if sinks is None else float(sinks[h])
        for n, u in enumerate(keys):
            d = int(np.searchsorted(cu, u, side="right")) - 1
            a, b = int(cu[d]), int(cu[d + 1])
            rows = [t for t in range(a, b) if _visible(t, t + 1, u, u + 1, causal, window_left, a, b)[0, 0]
                    and (row_window is None or row_window[0] <= t < row_window[1])]
            if not rows:
                continue
            O, L = attention_fwd_rows(q, k, v, cu, rows, h, causal, window_left, scale, sink)
            Qr = np.asarray(q[rows, h], np.float64)
            dOr = np.asarray(do[rows, h], np.float64)
            s = scale * (Qr @ np.asarray(k[u, kv_head], np.float64))
            Pm = np.exp(s - L)
            dS = Pm * (dOr @ np.asarray(v[u, kv_head], np.float64) - np.sum(dOr * O, axis=1))
            dv[n] += Pm @ dOr
            dk[n] += scale * (dS @ Qr)
    return dk, dv


def visible_pairs(cu_seqlens, causal: bool = True, window_left: int = -1) -> int:
    """Number of (query, key) pairs the mask keeps, summed over documents."""
    total = 0
    cu = [int(x) for x in cu_seqlens]
    for a, b in zip(cu[:-1], cu[1:]):
        L = b - a
        for i in range(L):
            lo = 0
            hi = i if causal else L - 1
            if window_left >= 0:
                lo = max(0, i - window_left)
                if not causal:
                    hi = min(L - 1, i + window_left)
            total += hi - lo + 1
    return total


# ---------------------------------------------------------------------------
# the emulated P-rank path and the unsharded reference
# ---------------------------------------------------------------------------

def _rank_sinks(sinks, r, hq):
    # Each head has a single sink logit; after the exchange rank r holds heads
    # [r*hq, (r+1)*hq), so it uses that slice (accelerate PR #4209, gpt-oss).
    return None if sinks is None else np.asarray(sinks, dtype=np.float64)[r * hq:(r + 1) * hq]


def ulysses_fwd(q_seq, k_seq, v_seq, pos_shards, causal=True, window_left=-1, scale=None,
                sinks=None):
    """Whole forward of P emulated ranks.

    Inputs are in sequence-shard layout ``[P][B][S/P][H][D]`` (float64 or
    anything numpy can widen).  Returns a dict with the head-layout tensors,
    ``cu_seqlens``, per-rank ``o_head``/``lse`` and the output back in
    sequence-shard layout ``o_seq``.
    """
    P, B, Sl, Hq, D = q_seq.shape
    S = P * Sl
    qh = relayout_fwd(np.asarray(q_seq, np.float64), P)
    # key/value heads fewer than the ranks are replicated (one per rank)
    kh = relayout_fwd(np.asarray(k_seq, np.float64), P, replicate=True)
    vh = relayout_fwd(np.asarray(v_seq, np.float64), P, replicate=True)
    cu, n, max_len = cu_seqlens_from_position_ids(pos_shards)
    hq, hk = Hq // P, kh.shape[3]
    o_head = np.empty((P, B, S, hq, D))
    lse = np.empty((P, B, hq, S))
    for r in range(P):
        O, L = attention_fwd(qh[r].reshape(B * S, hq, D), kh[r].reshape(B * S, hk, D),
                             vh[r].reshape(B * S, hk, D), cu, causal, window_left, scale,
                             _rank_sinks(sinks, r, hq))
        o_head[r] = O.reshape(B, S, hq, D)
        lse[r] = L.reshape(hq, B, S).transpose(1, 0, 2)
    return dict(q_head=qh, k_head=kh, v_head=vh, cu_seqlens=cu, n_docs=n, max_len=max_len,
                o_head=o_head, lse=lse, o_seq=relayout_bwd(o_head, P), Hkv=k_seq.shape[3])


def ulysses_bwd(fwd: dict, do_seq, causal=True, window_left=-1, scale=None, sinks=None):
    """Whole backward of P emulated ranks: dO goes seq->head, the attention
    gradients run per rank, and dQ/dK/dV go head->seq (the exchanges swapped)."""
    P = do_seq.shape[0]
    doh = relayout_fwd(np.asarray(do_seq, np.float64), P)
    _, B, S, hq, D = doh.shape
    hk = fwd["k_head"].shape[3]
    dqh = np.empty_like(fwd["q_head"])
    dkh = np.empty_like(fwd["k_head"])
    dvh = np.empty_like(fwd["v_head"])
    dsinks = None if sinks is None else np.zeros(hq * P)
    for r in range(P):
        lse_r = fwd["lse"][r].transpose(1, 0, 2).reshape(hq, B * S)
        dq, dk, dv, ds = attention_bwd(
            fwd["q_head"][r].reshape(B * S, hq, D), fwd["k_head"][r].reshape(B * S, hk, D),
            fwd["v_head"][r].reshape(B * S, hk, D), fwd["o_head"][r].reshape(B * S, hq, D),
            lse_r, doh[r].reshape(B * S, hq, D), fwd["cu_seqlens"], causal, window_left,
            scale, _rank_sinks(sinks, r, hq))
        dqh[r] = dq.reshape(B, S, hq, D)
        dkh[r] = dk.reshape(B, S, hk, D)
        dvh[r] = dv.reshape(B, S, hk, D)
        if ds is not None:
            dsinks[r * hq:(r + 1) * hq] = ds
    Hkv = fwd.get("Hkv", hk * P)
    # replicated key/value heads: the exchange back sums the replicas' gradients
    return dict(do_head=doh, dq_head=dqh, dk_head=dkh, dv_head=dvh, dsinks=dsinks,
                dq_seq=relayout_bwd(dqh, P), dk_seq=relayout_bwd(dkh, P, Hkv),
                dv_seq=relayout_bwd(dvh, P, Hkv))


def _unshard(x_seq):
    P, B, Sl = x_seq.shape[:3]
    return np.moveaxis(np.asarray(x_seq, np.float64), 0, 1).reshape((B, P * Sl) + x_seq.shape[3:])


def unsharded_fwd(q_seq, k_seq, v_seq, pos_shards, causal=True, window_left=-1, scale=None,
                  sinks=None):
    """Attention on the unsharded [B*S][H][D] tensors with all heads at once."""
    q = _unshard(q_seq)
    B, S, Hq, D = q.shape
    k = _unshard(k_seq)
    v = _unshard(v_seq)
    cu, _, _ = cu_seqlens_from_position_ids(pos_shards)
    O, L = attention_fwd(q.reshape(B * S, Hq, D), k.reshape(B * S, -1, D), v.reshape(B * S, -1, D),
                         cu, causal, window_left, scale, sinks)
    return O.reshape(B, S, Hq, D), L


def unsharded_bwd(q_seq, k_seq, v_seq, do_seq, pos_shards, causal=True, window_left=-1,
                  scale=None, sinks=None):
    q = _unshard(q_seq)
    B, S, Hq, D = q.shape
    k = _unshard(k_seq).reshape(B * S, -1, D)
    v = _unshard(v_seq).reshape(B * S, -1, D)
    do = _unshard(do_seq).reshape(B * S, Hq, D)
    q = q.reshape(B * S, Hq, D)
    cu, _, _ = cu_seqlens_from_position_ids(pos_shards)
    O, L = attention_fwd(q, k, v, cu, causal, window_left, scale, sinks)
    dq, dk, dv, ds = attention_bwd(q, k, v, O, L, do, cu, causal, window_left, scale, sinks)
    return (dq.reshape(B, S, Hq, D), dk.reshape(B, S, -1, D), dv.reshape(B, S, -1, D), ds)


# ---------------------------------------------------------------------------
# ring x Ulysses (USP hybrid): feifeibear/long-context-attention issue #135,
# the device-mesh script (mesh (ring, ulysses) with the Ulysses dimension
# innermost, "basic" contiguous chunks, the result compared with a
# non-distributed flash attention over the full tensors)
# ---------------------------------------------------------------------------

def hybrid_relayout_fwd(x_seq: np.ndarray, ring: int, ulysses: int, replicate: bool = False) -> np.ndarray:
    """The Ulysses exchange inside each ring group.

    ``x_seq`` is ``[P][B][S/P][H][D]`` with P = ring * ulysses; rank
    p = rho * ulysses + u holds positions ``[p*S/P, (p+1)*S/P)``.  The ranks of
    ring group rho (p = rho*U .. rho*U + U - 1) exchange among themselves, so
    that rank (rho, w) holds the super-chunk ``[rho*C, (rho+1)*C)``
    (C = S/ring) for heads ``[w*H/U, (w+1)*H/U)``.  The result is laid out
    ``[U][B][S][H/U][D]``: for each Ulysses index w the ring ranks'
    super-chunks end to end::

        out[w][b][rho*C + u*S/P + s'][j][d] = x_seq[rho*U + u][b][s'][w*H/U + j][d]

    With ``replicate`` and fewer heads than ``ulysses`` (U a multiple of H),
    rank (rho, w) receives head w // (U/H) as its one head.  ring = 1 is
    ``relayout_fwd``.
    """
    P, B, Sp, H, D = x_seq.shape
    U = ulysses
    if ring <= 0 or U <= 0 or P != ring * U:
        raise OracleError("the rank axis must hold ring * ulysses shards")
    _check_divisible(Sp * U, H, U, replicate)
    if H < U:
        owner = np.arange(U) // (U // H)
        y = x_seq[:, :, :, owner, :]                          # [p][b][s'][w][d]
        y = y.reshape(ring, U, B, Sp, U, D).transpose(4, 2, 0, 1, 3, 5)   # [w][b][rho][u][s'][d]
        return np.ascontiguousarray(y).reshape(U, B, P * Sp, 1, D)
    Hp = H // U
    y = x_seq.reshape(ring, U, B, Sp, U, Hp, D)               # [rho][u][b][s'][w][j][d]
    y = y.transpose(4, 2, 0, 1, 3, 5, 6)                      # [w][b][rho][u][s'][j][d]
    return np.ascontiguousarray(y).reshape(U, B, P * Sp, Hp, D)


def hybrid_relayout_bwd(x_head: np.ndarray, ring: int, ulysses: int, heads: Optional[int] = None) -> np.ndarray:
    """The inverse exchange inside each ring group::

        out[rho*U + u][b][s'][w*H/U + j][d] = x_head[w][b][rho*C + u*S/P + s'][j][d]

    With ``heads`` = H < U (replicated heads) the replicas' values are summed
    (the adjoint of the replication), as in ``relayout_bwd``.
    """
    U, B, S, Hp, D = x_head.shape
    if U != ulysses or ring <= 0 or S % (ring * U) != 0:
        raise OracleError("head-layout tensor does not match ring * ulysses")
    P = ring * U
    Sp = S // P
    H = Hp * U if heads is None else heads
    _check_divisible(S, H, U, replicate=True)
    if H < U:
        if Hp != 1:
            raise OracleError("replicated heads hold one head per rank")
        y = x_head.reshape(H, U // H, B, ring, U, Sp, D).sum(axis=1)     # [h][b][rho][u][s'][d]
        y = y.transpose(2, 3, 1, 4, 0, 5)                                # [rho][u][b][s'][h][d]
        return np.ascontiguousarray(y).reshape(P, B, Sp, H, D)
    y = x_head.reshape(U, B, ring, U, Sp, Hp, D)              # [w][b][rho][u][s'][j][d]
    y = y.transpose(2, 3, 1, 4, 0, 5, 6)                      # [rho][u][b][s'][w][j][d]
    return np.ascontiguousarray(y).reshape(P, B, Sp, U * Hp, D)


def _block_mask(i0, i1, k0, k1, cu, causal, window_left):
    """Boolean [i1-i0][k1-k0]: query i may see key j (same document, causal,
    window), for the query rows [i0, i1) and the keys [k0, k1)."""
    cu = np.asarray(cu, dtype=np.int64)
    i = np.arange(i0, i1)
    j = np.arange(k0, k1)
    di = np.searchsorted(cu, i, side="right") - 1
    dj = np.searchsorted(cu, j, side="right") - 1
    vis = di[:, None] == dj[None, :]
    if causal:
        vis &= j[None, :] <= i[:, None]
    if window_left >= 0:
        vis &= (i[:, None] - j[None, :]) <= window_left
        if not causal:
            vis &= (j[None, :] - i[:, None]) <= window_left
    return vis


def ring_block_fwd(q, k, v, cu_seqlens, rows, keys, causal: bool = True, window_left: int = -1,
                   scale: Optional[float] = None):
    """One ring step's attention: the query rows ``rows = (i0, i1)`` over the
    keys ``keys = (k0, k1)`` only (the key/value super-chunk the rank holds at
    that step), with the document, causal and window masks of
    ``attention_fwd`` and no sink.  ``q`` [T][hq][D], ``k``/``v`` [T][hk][D].
    Returns ``O`` [i1-i0][hq][D] and ``LSE`` [hq][i1-i0]; a row that sees no
    key of the block has O = 0 and LSE = -inf."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    T, hq, D = q.shape
    G = hq // k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    i0, i1 = rows
    k0, k1 = keys
    vis = _block_mask(i0, i1, k0, k1, cu_seqlens, causal, window_left)
    O = np.zeros((i1 - i0, hq, D))
    L = np.full((hq, i1 - i0), -np.inf)
    seen = vis.any(axis=1)
    for h in range(hq):
        s = np.where(vis, scale * (q[i0:i1, h] @ k[k0:k1, h // G].T), -np.inf)
        m = np.where(seen, s.max(axis=1), 0.0)
        e = np.where(vis, np.exp(s - m[:, None]), 0.0)
        z = e.sum(axis=1)
        L[h, seen] = m[seen] + np.log(z[seen])
        O[seen, h] = (e[seen] / z[seen, None]) @ v[k0:k1, h // G]
    return O, L


def ring_merge(O1, L1, O2, L2):
    """Combine two softmax-normalised partial outputs over disjoint key sets
    into the one over their union: LSE = log(e^L1 + e^L2) and
    O = e^(L1-LSE) O1 + e^(L2-LSE) O2 (a part with LSE = -inf adds nothing).
    ``O`` [..., hq, D] with ``L`` [hq, ...] matching its leading row axis."""
    L = np.logaddexp(L1, L2)
    fin = np.isfinite(L)
    w1 = np.where(fin, np.exp(np.where(fin, L1 - L, 0.0)), 0.0)
    w2 = np.where(fin, np.exp(np.where(fin, L2 - L, 0.0)), 0.0)
    # L is [hq][rows]; O is [rows][hq][D]
    return O1 * w1.T[:, :, None] + O2 * w2.T[:, :, None], L


def hybrid_fwd(q_seq, k_seq, v_seq, pos_shards, ring: int, causal=True, window_left=-1, scale=None,
               sinks=None):
    """Forward of the ring x Ulysses hybrid over P = ring * ulysses emulated ranks.

    1. Ulysses exchange inside each ring group (``hybrid_relayout_fwd``).
    2. For each Ulysses index w, ``ring`` steps: at step s ring rank rho
       attends its query super-chunk rho to the key/value super-chunk
       (rho - s) mod ring (``ring_block_fwd``) and merges the result into its
       running (O, LSE) (``ring_merge``).
    3. The sink logit of each head, if any, joins the softmax once, as a
       final part with LSE = sink and no value.
    4. The inverse exchange brings O back to the sequence shards.

    Document boundaries come from the gathered position_ids as in
    ``ulysses_fwd``.  Returns the head-layout tensors, ``o_head``
    [U][B][S][hq][D], ``lse`` [U][B][hq][S] and ``o_seq``.
    """
    P, B, Sp, Hq, D = q_seq.shape
    if P % ring != 0:
        raise OracleError("ring degree must divide the ranks")
    U = P // ring
    S = P * Sp
    if Hq % U != 0:
        raise OracleError(f"ulysses degree {U} does not divide {Hq} heads")
    C = S // ring
    qh = hybrid_relayout_fwd(np.asarray(q_seq, np.float64), ring, U)
    kh = hybrid_relayout_fwd(np.asarray(k_seq, np.float64), ring, U, replicate=True)
    vh = hybrid_relayout_fwd(np.asarray(v_seq, np.float64), ring, U, replicate=True)
    cu, n, max_len = cu_seqlens_from_position_ids(pos_shards)
    hq, T = Hq // U, B * S
    o_head = np.empty((U, B, S, hq, D))
    lse = np.empty((U, B, hq, S))
    for w in range(U):
        Q = qh[w].reshape(T, hq, D)
        K = kh[w].reshape(T, -1, D)
        V = vh[w].reshape(T, -1, D)
        O = np.zeros((T, hq, D))
        L = np.full((hq, T), -np.inf)
        for step in range(ring):
            for rho in range(ring):
                kc = (rho - step) % ring
                for b in range(B):
                    rows = (b * S + rho * C, b * S + (rho + 1) * C)
                    keys = (b * S + kc * C, b * S + (kc + 1) * C)
                    Ob, Lb = ring_block_fwd(Q, K, V, cu, rows, keys, causal, window_left, scale)
                    sl = slice(*rows)
                    O[sl], L[:, sl] = ring_merge(O[sl], L[:, sl], Ob, Lb)
        if sinks is not None:
            z = np.asarray(sinks, np.float64)[w * hq:(w + 1) * hq]
            O, L = ring_merge(O, L, np.zeros_like(O), np.repeat(z[:, None], T, axis=1))
        o_head[w] = O.reshape(B, S, hq, D)
        lse[w] = L.reshape(hq, B, S).transpose(1, 0, 2)
    return dict(q_head=qh, k_head=kh, v_head=vh, cu_seqlens=cu, n_docs=n, max_len=max_len,
                o_head=o_head, lse=lse, o_seq=hybrid_relayout_bwd(o_head, ring, U), Hkv=k_seq.shape[3],
                ring=ring)


def hybrid_bwd(fwd: dict, do_seq, causal=True, window_left=-1, scale=None, sinks=None, return_steps=False):
    """Backward of the ring x Ulysses hybrid: dO goes through the Ulysses
    exchange; every ring step recomputes its block's probabilities from the
    final LSE and adds its share to dQ (kept by the query's rank) and to dK/dV
    (carried with the key/value super-chunk back to its owner); the inverse
    exchange returns dQ/dK/dV (replicas summed).  ``return_steps`` also
    returns each step's block gradients (head layout) under ``steps``."""
    ring = fwd["ring"]
    P = do_seq.shape[0]
    U = P // ring
    doh = hybrid_relayout_fwd(np.asarray(do_seq, np.float64), ring, U)
    _, B, S, hq, D = doh.shape
    T, C = B * S, S // ring
    hk = fwd["k_head"].shape[3]
    G = hq // hk
    sc = 1.0 / np.sqrt(D) if scale is None else scale
    cu = fwd["cu_seqlens"]
    dqh = np.zeros_like(fwd["q_head"])
    dkh = np.zeros_like(fwd["k_head"])
    dvh = np.zeros_like(fwd["v_head"])
    dsinks = None if sinks is None else np.zeros(hq * U)
    steps = [dict(dq_head=np.zeros_like(dqh), dk_head=np.zeros_like(dkh), dv_head=np.zeros_like(dvh))
             for _ in range(ring)] if return_steps else None
    for w in range(U):
        Q = fwd["q_head"][w].reshape(T, hq, D)
        K = fwd["k_head"][w].reshape(T, hk, D)
        V = fwd["v_head"][w].reshape(T, hk, D)
        O = fwd["o_head"][w].reshape(T, hq, D)
        dO = doh[w].reshape(T, hq, D)
        L = fwd["lse"][w].transpose(1, 0, 2).reshape(hq, T)
        Dvec = np.sum(dO * O, axis=2)                     # [T][hq]
        dq = np.zeros((T, hq, D))
        dk = np.zeros((T, hk, D))
        dv = np.zeros((T, hk, D))
        for step in range(ring):
            for rho in range(ring):
                kc = (rho - step) % ring
                for b in range(B):
                    i0, i1 = b * S + rho * C, b * S + (rho + 1) * C
                    k0, k1 = b * S + kc * C, b * S + (kc + 1) * C
                    vis = _block_mask(i0, i1, k0, k1, cu, causal, window_left)
                    for h in range(hq):
                        kv = h // G
                        s = sc * (Q[i0:i1, h] @ K[k0:k1, kv].T)
                        Pm = np.where(vis, np.exp(np.where(vis, s, 0.0) - L[h, i0:i1][:, None]), 0.0)
                        bv = Pm.T @ dO[i0:i1, h]
                        dS = Pm * (dO[i0:i1, h] @ V[k0:k1, kv].T - Dvec[i0:i1, h][:, None])
                        bq = sc * (dS @ K[k0:k1, kv])
                        bk = sc * (dS.T @ Q[i0:i1, h])
                        dv[k0:k1, kv] += bv
                        dq[i0:i1, h] += bq
                        dk[k0:k1, kv] += bk
                        if steps is not None:
                            st = steps[step]
                            st["dv_head"][w].reshape(T, hk, D)[k0:k1, kv] += bv
                            st["dq_head"][w].reshape(T, hq, D)[i0:i1, h] += bq
                            st["dk_head"][w].reshape(T, hk, D)[k0:k1, kv] += bk
        if dsinks is not None:
            z = np.asarray(sinks, np.float64)[w * hq:(w + 1) * hq]
            dsinks[w * hq:(w + 1) * hq] = -np.sum(np.exp(z[:, None] - L) * Dvec.T, axis=1)
        dqh[w] = dq.reshape(B, S, hq, D)
        dkh[w] = dk.reshape(B, S, hk, D)
        dvh[w] = dv.reshape(B, S, hk, D)
    Hkv = fwd["Hkv"]
    return dict(do_head=doh, dq_head=dqh, dk_head=dkh, dv_head=dvh, dsinks=dsinks,
                dq_seq=hybrid_relayout_bwd(dqh, ring, U), dk_seq=hybrid_relayout_bwd(dkh, ring, U, Hkv),
                dv_seq=hybrid_relayout_bwd(dvh, ring, U, Hkv), steps=steps)
