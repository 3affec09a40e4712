"""Pins for the fp64 oracle: it is checked against things other than itself.

Every check here is either a closed form, a special case that reduces to a
library routine (torch's fp64 scaled_dot_product_attention and autograd),
a semantic encoding of coordinates, a finite difference, or a value fixed by
the workload's own definition (tests/golden).  A plausible slip in the oracle
(a dropped mask term, a swapped operand, a wrong sign, a head assigned to the
wrong rank) fails at least one of them.
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import usp_workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------------------
# relayout
# ---------------------------------------------------------------------------

def _encoded_seq_tensor(P, B, S, H, D):
    """x[r'][b][s'][h][d] = code(b, global position, head, d): values say where they came from."""
    Sl = S // P
    x = np.empty((P, B, Sl, H, D), dtype=np.int64)
    for r in range(P):
        for b in range(B):
            for s in range(Sl):
                for h in range(H):
                    for d in range(D):
                        x[r, b, s, h, d] = (((b * S + r * Sl + s) * H + h) * D + d)
    return x


def _decode(code, S, H, D):
    d = code % D
    h = (code // D) % H
    pos = (code // (D * H)) % S
    b = code // (D * H * S)
    return b, pos, h, d


@pytest.mark.parametrize("P,B,S,H,D", [(2, 1, 8, 4, 3), (4, 2, 8, 8, 2), (1, 1, 4, 3, 2), (3, 1, 6, 6, 1)])
def test_relayout_fwd_rank_holds_whole_sequence_for_its_heads(P, B, S, H, D):
    x = _encoded_seq_tensor(P, B, S, H, D)
    y = oracle.relayout_fwd(x, P)
    Hp = H // P
    assert y.shape == (P, B, S, Hp, D)
    for r in range(P):
        for b in range(B):
            for pos in range(S):
                for j in range(Hp):
                    for d in range(D):
                        bb, pp, hh, dd = _decode(int(y[r, b, pos, j, d]), S, H, D)
                        # rank r sees every position of row b, heads [r*Hp, (r+1)*Hp)
                        assert (bb, pp, hh, dd) == (b, pos, r * Hp + j, d)


@pytest.mark.parametrize("P,B,S,H,D", [(2, 1, 8, 4, 3), (4, 2, 8, 8, 2), (8, 1, 16, 8, 1)])
def test_relayout_is_a_permutation_and_bwd_inverts_fwd(P, B, S, H, D):
    x = _encoded_seq_tensor(P, B, S, H, D)
    y = oracle.relayout_fwd(x, P)
    assert sorted(y.reshape(-1).tolist()) == sorted(x.reshape(-1).tolist())
    assert len(set(y.reshape(-1).tolist())) == x.size
    assert np.array_equal(oracle.relayout_bwd(y, P), x)
    # and the other way round, starting from head layout
    z = _rng(1).standard_normal((P, B, S, H // P, D))
    assert np.array_equal(oracle.relayout_fwd(oracle.relayout_bwd(z, P), P), z)


def test_relayout_p1_is_a_copy():
    x = _rng(2).standard_normal((1, 2, 5, 3, 4))
    assert np.array_equal(oracle.relayout_fwd(x, 1), x)
    assert np.array_equal(oracle.relayout_bwd(x, 1), x)


def test_relayout_refuses_indivisible_heads():
    # "sp_size not dividing the heads" is refused (accelerate PR #4209)
    with pytest.raises(oracle.OracleError):
        oracle.relayout_fwd(np.zeros((4, 1, 2, 6, 2)), 4)
    # fewer heads than ranks are replicated only when asked and when P is a multiple of H
    with pytest.raises(oracle.OracleError):
        oracle.relayout_fwd(np.zeros((4, 1, 2, 2, 2)), 4)
    with pytest.raises(oracle.OracleError):
        oracle.relayout_fwd(np.zeros((4, 1, 2, 3, 2)), 4, replicate=True)


@pytest.mark.parametrize("P,B,S,H,D", [(4, 1, 8, 2, 3), (4, 2, 8, 1, 2), (8, 1, 16, 2, 1)])
def test_relayout_replicated_rank_holds_a_copy_of_its_head(P, B, S, H, D):
    x = _encoded_seq_tensor(P, B, S, H, D)
    y = oracle.relayout_fwd(x, P, replicate=True)
    assert y.shape == (P, B, S, 1, D)
    rep = P // H
    for r in range(P):
        for b in range(B):
            for pos in range(S):
                for d in range(D):
                    # rank r sees every position of row b, and head r // (P/H)
                    assert _decode(int(y[r, b, pos, 0, d]), S, H, D) == (b, pos, r // rep, d)


@pytest.mark.parametrize("P,H", [(4, 2), (4, 1), (8, 2)])
def test_relayout_replicated_bwd_is_the_adjoint_of_fwd(P, H):
    # The exchange back of a gradient must be the adjoint (transpose) of the
    # forward exchange: <fwd(x), y> = <x, bwd(y)> for all x, y.  For a copy to
    # P/H ranks that is the sum over the replicas.
    B, S, D = 2, 8, 3
    x = _rng(21).standard_normal((P, B, S // P, H, D))
    y = _rng(22).standard_normal((P, B, S, 1, D))
    lhs = float(np.sum(oracle.relayout_fwd(x, P, replicate=True) * y))
    rhs = float(np.sum(x * oracle.relayout_bwd(y, P, H)))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))
    # a gradient that is the same on every replica comes back P/H times
    xi = _rng(23).integers(-100, 100, size=(P, B, S // P, H, D)).astype(np.float64)
    assert np.array_equal(oracle.relayout_bwd(oracle.relayout_fwd(xi, P, replicate=True), P, H), (P // H) * xi)


# ---------------------------------------------------------------------------
# one real rank's side of the exchanges (send buffers, received chunks)
# ---------------------------------------------------------------------------

def _ranks_seq_to_head(x, P, replicate=False):
    """Every rank packs its shard, the collective delivers, every rank unpacks."""
    sends = [oracle.a2a_pack_seq_to_head(x[r], P, replicate) for r in range(P)]
    return [oracle.a2a_unpack_seq_to_head(rv) for rv in oracle.all_to_all(sends)]


@pytest.mark.parametrize("P,B,S,H,D", [(2, 1, 8, 4, 3), (4, 2, 8, 8, 2), (1, 1, 4, 3, 2), (3, 2, 6, 6, 1)])
def test_rank_exchange_seq_to_head_gives_whole_sequence_of_own_heads(P, B, S, H, D):
    x = _encoded_seq_tensor(P, B, S, H, D)
    Sl, Hp = S // P, H // P
    for r in range(P):
        send = oracle.a2a_pack_seq_to_head(x[r], P)
        assert send.shape == (P, B, Sl, Hp, D)
        # chunk p of rank r's send buffer: rank p's heads of r's positions
        for p in range(P):
            for b in range(B):
                for s in range(Sl):
                    for j in range(Hp):
                        assert _decode(int(send[p, b, s, j, 0]), S, H, D) == (b, r * Sl + s, p * Hp + j, 0)
    heads = _ranks_seq_to_head(x, P)
    for r in range(P):
        assert heads[r].shape == (B, S, Hp, D)
        for b in range(B):
            for pos in range(S):
                for j in range(Hp):
                    for d in range(D):
                        assert _decode(int(heads[r][b, pos, j, d]), S, H, D) == (b, pos, r * Hp + j, d)
        # the same as the emulated exchange's rank r
        assert np.array_equal(heads[r], oracle.relayout_fwd(x, P)[r])


@pytest.mark.parametrize("P,B,S,H,D", [(4, 1, 8, 2, 3), (4, 2, 8, 1, 2), (8, 1, 16, 2, 1)])
def test_rank_exchange_replicated_heads(P, B, S, H, D):
    x = _encoded_seq_tensor(P, B, S, H, D)
    heads = _ranks_seq_to_head(x, P, replicate=True)
    rep = P // H
    for r in range(P):
        for b in range(B):
            for pos in range(S):
                assert _decode(int(heads[r][b, pos, 0, 1 % D]), S, H, D) == (b, pos, r // rep, 1 % D)
        assert np.array_equal(heads[r], oracle.relayout_fwd(x, P, replicate=True)[r])
    # the way back sums the replicas: the adjoint of the replicating exchange
    y = _rng(24).standard_normal((P, B, S, 1, D))
    sends = [oracle.a2a_pack_head_to_seq(y[r], P) for r in range(P)]
    back = [oracle.a2a_unpack_head_to_seq(rv, H) for rv in oracle.all_to_all(sends)]
    xs = _rng(25).standard_normal((P, B, S // P, H, D))
    lhs = float(np.sum(oracle.relayout_fwd(xs, P, replicate=True) * y))
    rhs = float(sum(np.sum(xs[r] * back[r]) for r in range(P)))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


@pytest.mark.parametrize("P,B,S,H,D", [(2, 1, 8, 4, 3), (4, 2, 8, 8, 2), (3, 1, 6, 6, 2)])
def test_rank_exchange_head_to_seq_inverts_seq_to_head(P, B, S, H, D):
    x = _encoded_seq_tensor(P, B, S, H, D)
    heads = _ranks_seq_to_head(x, P)
    sends = [oracle.a2a_pack_head_to_seq(heads[r], P) for r in range(P)]
    for r in range(P):
        # chunk p of rank r's send buffer: rank p's positions of r's heads
        for p in range(P):
            assert _decode(int(sends[r][p, 0, 0, 0, 0]), S, H, D) == (0, p * (S // P), r * (H // P), 0)
    back = [oracle.a2a_unpack_head_to_seq(rv) for rv in oracle.all_to_all(sends)]
    for r in range(P):
        assert np.array_equal(back[r], x[r])


# ---------------------------------------------------------------------------
# cu_seqlens
# ---------------------------------------------------------------------------

def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [int(x) for x in rest]
    return vals


def test_cu_seqlens_tiny_golden():
    g = _read_golden("tiny_packed_cu_seqlens.txt")
    cu, n, mx = oracle.cu_seqlens_from_position_ids(W.position_ids_shards(W.TINY))
    assert cu.tolist() == g["cu_seqlens"]
    assert n == g["n_docs"][0] and mx == g["max_len"][0]
    # rank 0's shard alone gives the stale per-shard boundaries
    shard0 = W.position_ids_shards(W.TINY)[:1]
    cu0, _, _ = oracle.cu_seqlens_from_position_ids(shard0)
    assert cu0.tolist() == g["stale_rank0_cu_seqlens"]


@pytest.mark.parametrize("w", [W.MHA4K, W.LLAMA32K, W.GPTOSS_WIN, W.LONG128K], ids=lambda w: w.name)
def test_cu_seqlens_equals_cumsum_of_document_lengths(w):
    lens = W.document_lengths(w)[0]
    cu, n, mx = oracle.cu_seqlens_from_position_ids(W.position_ids_shards(w))
    assert cu.tolist() == [0] + np.cumsum(lens).tolist()
    assert n == len(lens) and mx == max(lens)


def test_cu_seqlens_special_case_flatnonzero():
    rng = _rng(3)
    lens = rng.integers(1, 40, size=30)
    pos = np.concatenate([np.arange(n) for n in lens]).astype(np.int32)
    S = pos.size - pos.size % 4
    pos = pos[:S]
    shards = pos.reshape(1, 4, S // 4).transpose(1, 0, 2)
    cu, n, mx = oracle.cu_seqlens_from_position_ids(shards)
    ref = np.append(np.flatnonzero(pos == 0), S)
    assert cu.tolist() == ref.tolist()
    assert mx == int(np.max(np.diff(ref)))


def test_cu_seqlens_row_starts_are_boundaries():
    # B=2: the second row starts a document even though its first position is 5
    pos = np.array([[0, 1, 2, 0, 1, 2, 3, 4], [5, 6, 7, 8, 0, 1, 2, 3]], dtype=np.int32)
    shards = W.shard_sequence(pos, 2)
    cu, n, mx = oracle.cu_seqlens_from_position_ids(shards)
    assert cu.tolist() == [0, 3, 8, 12, 16] and n == 4 and mx == 5


def test_cu_seqlens_refuses_negative_positions():
    pos = np.array([[0, 1, -1, 3]], dtype=np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.cu_seqlens_from_position_ids(W.shard_sequence(pos, 2))


# ---------------------------------------------------------------------------
# attention forward
# ---------------------------------------------------------------------------

def _rand_qkv(T, hq, hk, D, seed=0):
    r = _rng(seed)
    return (r.standard_normal((T, hq, D)), r.standard_normal((T, hk, D)),
            r.standard_normal((T, hk, D)))


def _sdpa(q, k, v, causal, mask=None):
    """torch fp64 SDPA on one document; q [L][h][D], k/v [L][h][D] (already GQA-expanded)."""
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2)[None]
    o = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, is_causal=causal)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("causal", [True, False])
def test_fwd_single_document_is_textbook_sdpa(causal):
    q, k, v = _rand_qkv(37, 3, 3, 16, seed=4)
    O, _ = oracle.attention_fwd(q, k, v, [0, 37], causal=causal)
    np.testing.assert_allclose(O, _sdpa(q, k, v, causal), rtol=0, atol=1e-12)


def test_fwd_packed_equals_each_document_alone():
    q, k, v = _rand_qkv(50, 2, 2, 8, seed=5)
    cu = [0, 13, 14, 41, 50]
    O, _ = oracle.attention_fwd(q, k, v, cu, causal=True)
    for a, b in zip(cu[:-1], cu[1:]):
        np.testing.assert_allclose(O[a:b], _sdpa(q[a:b], k[a:b], v[a:b], True), rtol=0, atol=1e-12)


def test_fwd_gqa_equals_mha_with_repeated_kv():
    q, k, v = _rand_qkv(24, 6, 2, 8, seed=6)
    O, _ = oracle.attention_fwd(q, k, v, [0, 10, 24])
    kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    for a, b in [(0, 10), (10, 24)]:
        np.testing.assert_allclose(O[a:b], _sdpa(q[a:b], kr[a:b], vr[a:b], True), rtol=0, atol=1e-12)


def test_fwd_window_zero_sees_only_itself():
    q, k, v = _rand_qkv(20, 2, 1, 8, seed=7)
    O, L = oracle.attention_fwd(q, k, v, [0, 20], window_left=0)
    np.testing.assert_allclose(O, np.repeat(v, 2, axis=1), rtol=0, atol=1e-14)
    s_ii = np.einsum("thd,thd->ht", q, np.repeat(k, 2, axis=1)) / np.sqrt(8)
    np.testing.assert_allclose(L, s_ii, rtol=0, atol=1e-13)


def test_fwd_window_one_two_key_closed_form():
    q, k, v = _rand_qkv(9, 1, 1, 4, seed=8)
    O, _ = oracle.attention_fwd(q, k, v, [0, 9], window_left=1)
    sc = 0.5
    for i in range(1, 9):
        a = sc * q[i, 0] @ k[i, 0]
        b = sc * q[i, 0] @ k[i - 1, 0]
        ref = (np.exp(a) * v[i, 0] + np.exp(b) * v[i - 1, 0]) / (np.exp(a) + np.exp(b))
        np.testing.assert_allclose(O[i, 0], ref, rtol=1e-13, atol=1e-14)


def test_fwd_wide_window_is_plain_causal():
    q, k, v = _rand_qkv(30, 2, 2, 8, seed=9)
    O1, L1 = oracle.attention_fwd(q, k, v, [0, 12, 30], window_left=29)
    O2, L2 = oracle.attention_fwd(q, k, v, [0, 12, 30])
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_fwd_window_matches_sdpa_with_band_mask():
    q, k, v = _rand_qkv(40, 2, 2, 8, seed=10)
    O, _ = oracle.attention_fwd(q, k, v, [0, 40], window_left=5)
    band = torch.ones(40, 40, dtype=torch.bool).tril().triu(-5)
    np.testing.assert_allclose(O, _sdpa(q, k, v, False, mask=band), rtol=0, atol=1e-12)


def test_sink_minus_infinity_is_no_sink_and_large_sink_silences():
    q, k, v = _rand_qkv(16, 2, 1, 8, seed=11)
    O0, L0 = oracle.attention_fwd(q, k, v, [0, 7, 16])
    O1, L1 = oracle.attention_fwd(q, k, v, [0, 7, 16], sinks=np.array([-np.inf, -np.inf]))
    np.testing.assert_allclose(O1, O0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(L1, L0, rtol=0, atol=1e-14)
    O2, L2 = oracle.attention_fwd(q, k, v, [0, 7, 16], sinks=np.array([60.0, 60.0]))
    assert np.abs(O2).max() < 1e-15
    np.testing.assert_allclose(L2, 60.0, rtol=0, atol=1e-12)


def test_sink_one_key_closed_form_and_lse_relation():
    q, k, v = _rand_qkv(12, 2, 2, 8, seed=12)
    t = np.array([0.7, -1.3])
    O, L = oracle.attention_fwd(q, k, v, [0, 5, 12], sinks=t)
    O0, L0 = oracle.attention_fwd(q, k, v, [0, 5, 12])
    sc = 1 / np.sqrt(8)
    for a in (0, 5):                         # first row of each document sees one key
        for h in range(2):
            s = sc * q[a, h] @ k[a, h]
            np.testing.assert_allclose(O[a, h], v[a, h] * np.exp(s) / (np.exp(s) + np.exp(t[h])),
                                       rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(L[a, h] if False else L[h, a], np.log(np.exp(s) + np.exp(t[h])),
                                       rtol=1e-13)
    # a sink adds exp(t) to the partition function: LSE_sink = logaddexp(LSE, t)
    np.testing.assert_allclose(L, np.logaddexp(L0, t[:, None]), rtol=1e-13)
    # and shrinks the output by the probability mass the sink takes
    w = np.exp(L0 - L)                       # [h][T]
    np.testing.assert_allclose(O, O0 * w.T[:, :, None], rtol=1e-12, atol=1e-14)


def test_softmax_rows_with_sink_sum_to_one():
    q, k, v = _rand_qkv(25, 2, 1, 8, seed=13)
    t = np.array([0.3, 1.1])
    cu = [0, 9, 25]
    _, L = oracle.attention_fwd(q, k, v, cu, sinks=t, window_left=4)
    sc = 1 / np.sqrt(8)
    for h in range(2):
        for a, b in zip(cu[:-1], cu[1:]):
            for i in range(a, b):
                js = [j for j in range(a, i + 1) if i - j <= 4]
                tot = sum(np.exp(sc * q[i, h] @ k[j, 0] - L[h, i]) for j in js)
                tot += np.exp(t[h] - L[h, i])
                assert abs(tot - 1.0) < 1e-12


# ---------------------------------------------------------------------------
# attention backward
# ---------------------------------------------------------------------------

def _torch_grads(q, k, v, do, causal):
    tq = torch.from_numpy(q).permute(1, 0, 2)[None].requires_grad_()
    tk = torch.from_numpy(k).permute(1, 0, 2)[None].requires_grad_()
    tv = torch.from_numpy(v).permute(1, 0, 2)[None].requires_grad_()
    o = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)
    o.backward(torch.from_numpy(do).permute(1, 0, 2)[None])
    return [t.grad[0].permute(1, 0, 2).numpy() for t in (tq, tk, tv)]


@pytest.mark.parametrize("causal", [True, False])
def test_bwd_single_document_matches_torch_autograd(causal):
    q, k, v = _rand_qkv(33, 2, 2, 16, seed=14)
    do = _rng(15).standard_normal(q.shape)
    O, L = oracle.attention_fwd(q, k, v, [0, 33], causal=causal)
    dq, dk, dv, ds = oracle.attention_bwd(q, k, v, O, L, do, [0, 33], causal=causal)
    rq, rk, rv = _torch_grads(q, k, v, do, causal)
    for a, b in ((dq, rq), (dk, rk), (dv, rv)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)
    assert ds is None


def test_bwd_packed_gqa_matches_torch_autograd_per_document():
    q, k, v = _rand_qkv(40, 4, 2, 8, seed=16)
    do = _rng(17).standard_normal(q.shape)
    cu = [0, 17, 18, 40]
    O, L = oracle.attention_fwd(q, k, v, cu)
    dq, dk, dv, _ = oracle.attention_bwd(q, k, v, O, L, do, cu)
    for a, b in zip(cu[:-1], cu[1:]):
        kr, vr = np.repeat(k[a:b], 2, axis=1), np.repeat(v[a:b], 2, axis=1)
        rq, rk, rv = _torch_grads(q[a:b], kr, vr, do[a:b], True)
        np.testing.assert_allclose(dq[a:b], rq, rtol=0, atol=1e-11)
        # GQA: a key/value head's gradient sums the gradients of its query heads
        np.testing.assert_allclose(dk[a:b], rk.reshape(b - a, 2, 2, 8).sum(2), rtol=0, atol=1e-11)
        np.testing.assert_allclose(dv[a:b], rv.reshape(b - a, 2, 2, 8).sum(2), rtol=0, atol=1e-11)


def _loss(q, k, v, do, cu, window_left, sinks):
    O, _ = oracle.attention_fwd(q, k, v, cu, window_left=window_left, sinks=sinks)
    return float(np.sum(O * do))


@pytest.mark.parametrize("window_left,use_sink", [(-1, False), (-1, True), (3, True), (0, True)])
def test_bwd_finite_differences(window_left, use_sink):
    T, hq, hk, D = 16, 2, 1, 4
    q, k, v = _rand_qkv(T, hq, hk, D, seed=18)
    do = _rng(19).standard_normal(q.shape)
    cu = [0, 6, 16]
    t = np.array([0.4, -0.8]) if use_sink else None
    O, L = oracle.attention_fwd(q, k, v, cu, window_left=window_left, sinks=t)
    dq, dk, dv, ds = oracle.attention_bwd(q, k, v, O, L, do, cu, window_left=window_left, sinks=t)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            lp = _loss(q, k, v, do, cu, window_left, t)
            x[idx] = old - eps
            lm = _loss(q, k, v, do, cu, window_left, t)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * eps)
        err = np.abs(num - g).max() / max(1e-12, np.abs(num).max())
        assert err < 1e-6, (name, err)
    if use_sink:
        for h in range(hq):
            tp, tm = t.copy(), t.copy()
            tp[h] += eps
            tm[h] -= eps
            num = (_loss(q, k, v, do, cu, window_left, tp) - _loss(q, k, v, do, cu, window_left, tm)) / (2 * eps)
            assert abs(num - ds[h]) < 1e-6 * max(1.0, abs(num)), (h, num, ds[h])


# ---------------------------------------------------------------------------
# emulated P-rank path == unsharded
# ---------------------------------------------------------------------------

def _small_workload_tensors(w):
    t = W.qkv_do_shards(w)
    return {n: W.bf16_to_f64(x) for n, x in t.items()}


@pytest.mark.parametrize("w", [
    W.TINY,
    W.Workload("gqa_p4", B=1, S=64, Hq=8, Hkv=4, D=16, P=4, doc_mode="explicit", doc_lens=(5, 40, 19)),
    W.Workload("sink_win_p2", B=2, S=32, Hq=4, Hkv=2, D=8, P=2, window_left=6, sinks=True,
               doc_mode="explicit", doc_lens=(20, 12)),
    # kv-head replication: fewer key/value heads than ranks
    W.Workload("kv_rep_p4", B=1, S=64, Hq=8, Hkv=2, D=8, P=4, doc_mode="explicit", doc_lens=(30, 34)),
    W.Workload("mqa_rep_sink_win_p4", B=1, S=48, Hq=4, Hkv=1, D=8, P=4, window_left=9, sinks=True,
               doc_mode="explicit", doc_lens=(7, 41)),
], ids=lambda w: w.name)
def test_ulysses_equals_unsharded(w):
    x = _small_workload_tensors(w)
    pos = W.position_ids_shards(w)
    snk = None if W.sinks(w) is None else W.sinks(w).double().numpy()
    f = oracle.ulysses_fwd(x["q"], x["k"], x["v"], pos, window_left=w.window_left, sinks=snk)
    O, L = oracle.unsharded_fwd(x["q"], x["k"], x["v"], pos, window_left=w.window_left, sinks=snk)
    np.testing.assert_allclose(f["o_seq"], W.shard_sequence(O, w.P), rtol=0, atol=1e-13)
    # per-rank LSE holds that rank's heads of the unsharded LSE
    hq = w.Hq // w.P
    for r in range(w.P):
        np.testing.assert_allclose(f["lse"][r].transpose(1, 0, 2).reshape(hq, -1),
                                   L[r * hq:(r + 1) * hq], rtol=0, atol=1e-13)
    g = oracle.ulysses_bwd(f, x["do"], window_left=w.window_left, sinks=snk)
    dq, dk, dv, ds = oracle.unsharded_bwd(x["q"], x["k"], x["v"], x["do"], pos,
                                          window_left=w.window_left, sinks=snk)
    np.testing.assert_allclose(g["dq_seq"], W.shard_sequence(dq, w.P), rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["dk_seq"], W.shard_sequence(dk, w.P), rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["dv_seq"], W.shard_sequence(dv, w.P), rtol=0, atol=1e-12)
    if snk is not None:
        np.testing.assert_allclose(g["dsinks"], ds, rtol=0, atol=1e-12)


def test_visible_pairs_closed_forms():
    assert oracle.visible_pairs([0, 4096]) == 4096 * 4097 // 2
    assert oracle.visible_pairs([0, 100, 190, 256]) == 100 * 101 // 2 + 90 * 91 // 2 + 66 * 67 // 2
    L, w = 1000, 127
    assert oracle.visible_pairs([0, L], window_left=w) == sum(min(i + 1, w + 1) for i in range(L))


def test_fwd_rows_agree_with_sdpa_rows():
    q, k, v = _rand_qkv(45, 4, 2, 8, seed=20)
    cu = [0, 20, 45]
    rows = [0, 5, 19, 20, 33, 44]
    t = np.array([0.2, -0.5, 1.0, 0.0])
    for h in range(4):
        O, L = oracle.attention_fwd_rows(q, k, v, cu, rows, h, window_left=6, sink=t[h])
        # reference: the logits of the row written out with torch, hidden keys
        # at -inf and the sink appended as one more logit (value row zero)
        for n, i in enumerate(rows):
            a, b = (0, 20) if i < 20 else (20, 45)
            jj = np.arange(a, b)
            seen = (jj <= i) & (i - jj <= 6)
            logits = torch.from_numpy(k[a:b, h // 2] @ q[i, h] / np.sqrt(8))
            logits = torch.where(torch.from_numpy(seen), logits, torch.tensor(-np.inf, dtype=torch.float64))
            lg = torch.cat([logits, torch.tensor([t[h]], dtype=torch.float64)])
            ref_o = torch.softmax(lg, 0)[:-1] @ torch.from_numpy(v[a:b, h // 2])
            np.testing.assert_allclose(O[n], ref_o.numpy(), rtol=0, atol=1e-12)
            np.testing.assert_allclose(L[n], torch.logsumexp(lg, 0).item(), rtol=1e-13)


@pytest.mark.parametrize("causal,window_left,use_sink", [(True, -1, False), (True, 5, True), (False, 4, False)])
def test_bwd_rows_and_keys_agree_with_full_backward(causal, window_left, use_sink):
    # the sampled forms are pinned to attention_bwd, itself pinned to torch
    # autograd and finite differences above
    q, k, v = _rand_qkv(40, 4, 2, 8, seed=21)
    do = _rng(22).standard_normal(q.shape)
    cu = [0, 11, 12, 40]
    t = np.array([0.5, -0.2, 0.9, 0.1]) if use_sink else None
    O, L = oracle.attention_fwd(q, k, v, cu, causal, window_left, sinks=t)
    dq, dk, dv, _ = oracle.attention_bwd(q, k, v, O, L, do, cu, causal, window_left, sinks=t)
    rows = [0, 10, 11, 12, 25, 39]
    for h in range(4):
        got = oracle.attention_bwd_rows(q, k, v, do, cu, rows, h, causal, window_left,
                                        sink=None if t is None else t[h])
        np.testing.assert_allclose(got, dq[rows, h], rtol=0, atol=1e-11)
    keys = [0, 5, 11, 12, 30, 39]
    for kh in range(2):
        gk, gv = oracle.attention_bwd_keys(q, k, v, do, cu, keys, kh, causal, window_left, sinks=t)
        np.testing.assert_allclose(gk, dk[keys, kh], rtol=0, atol=1e-11)
        np.testing.assert_allclose(gv, dv[keys, kh], rtol=0, atol=1e-11)
    # restricting to one GQA group gives that key/value head's full gradient
    dq2, dk2, dv2, _ = oracle.attention_bwd(q, k, v, O, L, do, cu, causal, window_left, sinks=t, heads=[2, 3])
    np.testing.assert_allclose(dk2[:, 1], dk[:, 1], rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv2[:, 1], dv[:, 1], rtol=0, atol=1e-12)
    assert np.all(dk2[:, 0] == 0) and np.all(dq2[:, :2] == 0)


# ---------------------------------------------------------------------------
# ring x Ulysses hybrid (USP)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("ring,U,B,S,H,D", [(2, 2, 1, 16, 4, 2), (3, 2, 2, 24, 2, 1), (4, 1, 1, 8, 3, 2),
                                            (1, 4, 2, 8, 4, 1)])
def test_hybrid_relayout_rank_holds_its_super_chunk_for_its_heads(ring, U, B, S, H, D):
    P = ring * U
    x = _encoded_seq_tensor(P, B, S, H, D)
    y = oracle.hybrid_relayout_fwd(x, ring, U)
    Hp = H // U
    assert y.shape == (U, B, S, Hp, D)
    for w in range(U):
        for b in range(B):
            for pos in range(S):
                for j in range(Hp):
                    for d in range(D):
                        # Ulysses rank w of every ring group: global position pos, heads block w
                        assert _decode(int(y[w, b, pos, j, d]), S, H, D) == (b, pos, w * Hp + j, d)
    assert np.array_equal(oracle.hybrid_relayout_bwd(y, ring, U), x)
    if ring == 1:
        assert np.array_equal(y, oracle.relayout_fwd(x, U))


def test_hybrid_relayout_replicated_is_adjoint():
    ring, U, H = 2, 4, 2
    x = _rng(31).standard_normal((ring * U, 2, 3, H, 4))
    y = _rng(32).standard_normal((U, 2, ring * U * 3, 1, 4))
    lhs = float(np.sum(oracle.hybrid_relayout_fwd(x, ring, U, replicate=True) * y))
    rhs = float(np.sum(x * oracle.hybrid_relayout_bwd(y, ring, U, H)))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


def test_ring_merge_of_two_key_blocks_is_the_union():
    # softmax over a key set = log-sum-exp merge of the softmaxes over a split of it
    q, k, v = _rand_qkv(40, 2, 1, 8, seed=33)
    cu = [0, 13, 40]
    for causal in (True, False):
        Oa, La = oracle.ring_block_fwd(q, k, v, cu, (20, 40), (0, 20), causal)
        Ob, Lb = oracle.ring_block_fwd(q, k, v, cu, (20, 40), (20, 40), causal)
        Ou, Lu = oracle.ring_block_fwd(q, k, v, cu, (20, 40), (0, 40), causal)
        Om, Lm = oracle.ring_merge(Oa, La, Ob, Lb)
        np.testing.assert_allclose(Om, Ou, rtol=0, atol=1e-13)
        np.testing.assert_allclose(Lm, Lu, rtol=0, atol=1e-13)
        # and the whole-range block is plain attention over those rows
        O, L = oracle.attention_fwd(q, k, v, cu, causal)
        np.testing.assert_allclose(Ou, O[20:40], rtol=0, atol=1e-13)
    # rows with no key in the block: O = 0, LSE = -inf
    O0, L0 = oracle.ring_block_fwd(q, k, v, cu, (0, 10), (20, 40), True)
    assert np.all(O0 == 0) and np.all(L0 == -np.inf)


HYBRID = [
    (W.Workload("usp_r2u2", B=1, S=64, Hq=4, Hkv=2, D=8, P=4, ring=2, doc_mode="explicit", doc_lens=(23, 41)), ),
    (W.Workload("usp_r4u1_noncausal", B=1, S=32, Hq=2, Hkv=1, D=4, P=4, ring=4, causal=False,
                doc_mode="explicit", doc_lens=(32,)), ),
    (W.Workload("usp_r2u2_win_sink_b2", B=2, S=48, Hq=4, Hkv=2, D=8, P=4, ring=2, window_left=9, sinks=True,
                doc_mode="explicit", doc_lens=(30, 18)), ),
    (W.Workload("usp_r2u4_kv_rep", B=1, S=64, Hq=8, Hkv=2, D=4, P=8, ring=2, doc_mode="explicit",
                doc_lens=(5, 50, 9)), ),
    (W.Workload("usp_r1u2", B=1, S=32, Hq=4, Hkv=2, D=4, P=2, ring=1, doc_mode="explicit", doc_lens=(20, 12)), ),
]


@pytest.mark.parametrize("w", [c[0] for c in HYBRID], ids=lambda w: w.name)
def test_hybrid_equals_unsharded(w):
    """The pages validate the hybrid against a non-distributed attention over
    the full tensors; the oracle's hybrid must agree with the unsharded
    definition in the forward and the backward."""
    x = _small_workload_tensors(w)
    pos = W.position_ids_shards(w)
    snk = None if W.sinks(w) is None else W.sinks(w).double().numpy()
    kw = dict(causal=w.causal, window_left=w.window_left, sinks=snk)
    f = oracle.hybrid_fwd(x["q"], x["k"], x["v"], pos, w.ring, **kw)
    O, L = oracle.unsharded_fwd(x["q"], x["k"], x["v"], pos, **kw)
    np.testing.assert_allclose(f["o_seq"], W.shard_sequence(O, w.P), rtol=0, atol=1e-12)
    U, hq = w.P // w.ring, w.Hq // (w.P // w.ring)
    for u in range(U):
        np.testing.assert_allclose(f["lse"][u].transpose(1, 0, 2).reshape(hq, -1), L[u * hq:(u + 1) * hq],
                                   rtol=0, atol=1e-12)
    g = oracle.hybrid_bwd(f, x["do"], **kw)
    dq, dk, dv, ds = oracle.unsharded_bwd(x["q"], x["k"], x["v"], x["do"], pos, **kw)
    np.testing.assert_allclose(g["dq_seq"], W.shard_sequence(dq, w.P), rtol=0, atol=1e-11)
    np.testing.assert_allclose(g["dk_seq"], W.shard_sequence(dk, w.P), rtol=0, atol=1e-11)
    np.testing.assert_allclose(g["dv_seq"], W.shard_sequence(dv, w.P), rtol=0, atol=1e-11)
    if snk is not None:
        np.testing.assert_allclose(g["dsinks"], ds, rtol=0, atol=1e-11)
    if w.ring == 1:
        u = oracle.ulysses_fwd(x["q"], x["k"], x["v"], pos, **kw)
        np.testing.assert_allclose(f["o_seq"], u["o_seq"], rtol=0, atol=1e-13)
    # the per-step block gradients add up to the result
    gs = oracle.hybrid_bwd(f, x["do"], return_steps=True, **kw)
    for n in ("dq_head", "dk_head", "dv_head"):
        np.testing.assert_allclose(sum(st[n] for st in gs["steps"]), g[n], rtol=0, atol=1e-12)


def test_bwd_rows_and_keys_split_over_windows_add_up():
    # one ring step's share of dQ (keys of a window) and of dK/dV (rows of a
    # window): the shares over a partition of the sequence add up to the whole
    q, k, v = _rand_qkv(48, 2, 1, 8, seed=34)
    do = _rng(35).standard_normal(q.shape)
    cu = [0, 20, 48]
    rows = [5, 19, 20, 33, 47]
    whole = oracle.attention_bwd_rows(q, k, v, do, cu, rows, 1)
    parts = [oracle.attention_bwd_rows(q, k, v, do, cu, rows, 1, key_window=wd) for wd in ((0, 24), (24, 48))]
    np.testing.assert_allclose(parts[0] + parts[1], whole, rtol=0, atol=1e-12)
    keys = [0, 10, 21, 30, 47]
    dk, dv = oracle.attention_bwd_keys(q, k, v, do, cu, keys, 0)
    p0 = oracle.attention_bwd_keys(q, k, v, do, cu, keys, 0, row_window=(0, 24))
    p1 = oracle.attention_bwd_keys(q, k, v, do, cu, keys, 0, row_window=(24, 48))
    np.testing.assert_allclose(p0[0] + p1[0], dk, rtol=0, atol=1e-12)
    np.testing.assert_allclose(p0[1] + p1[1], dv, rtol=0, atol=1e-12)
    # and a key window that excludes every key of a row gives it no gradient
    assert np.all(oracle.attention_bwd_rows(q, k, v, do, cu, [5], 0, key_window=(24, 48)) == 0)
