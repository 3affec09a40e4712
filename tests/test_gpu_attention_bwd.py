"""GPU parity of the backward path through the C ABI: dO exchanged seq->head,
tcgen05 dK/dV and dQ kernels, dQ/dK/dV exchanged head->seq, dsinks; compared
with the fp64 oracle (max-abs <= 2e-2, relative L2 <= 5e-3)."""
import numpy as np
import pytest
import torch

import oracle
import usp_workloads as W
from gpu_util import (assert_close, built_lib, device_inputs, dsink_bound, half_ulp_bf16, head_values, modes,
                      seq_head_values, shape_of)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built_lib()


def _fwd_bwd(w, fused=False, stored_ds=None, ds_group_size=None):
    from ulysses_sequence_long_gb300.pipeline import UlyssesAttention
    dev, host = device_inputs(w)
    ua = UlyssesAttention(shape_of(w), with_backward=True, fused=fused, stored_ds=stored_ds,
                          ds_group_size=ds_group_size)
    ua.forward(dev["q"], dev["k"], dev["v"], dev["pos"], dev["sinks"])
    ua.backward(dev["do"], dev["sinks"])
    torch.cuda.synchronize()
    assert ua.read_status() == 0
    return ua, dev, host


SMALL = [
    W.TINY,
    W.MHA4K,
    W.Workload("gqa_win_sink_d128", B=1, S=1024, Hq=8, Hkv=2, D=128, P=2, window_left=200, sinks=True,
               doc_mode="explicit", doc_lens=(300, 1, 423, 300)),
    W.Workload("gqa_win_sink_d64", B=1, S=1536, Hq=8, Hkv=4, D=64, P=4, window_left=127, sinks=True,
               doc_mode="geometric", doc_mean=400, seed=3),
    W.Workload("two_rows_ragged", B=2, S=640, Hq=4, Hkv=2, D=128, P=2, doc_mode="geometric", doc_mean=150,
               seed=5),
    W.Workload("noncausal_d64", B=1, S=512, Hq=2, Hkv=1, D=64, P=1, causal=False, doc_mode="explicit",
               doc_lens=(100, 250, 162)),
    # kv-head replication: more ranks than key/value heads
    W.Workload("kv_rep_d64", B=1, S=512, Hq=8, Hkv=2, D=64, P=4, doc_mode="explicit", doc_lens=(200, 180, 132)),
    W.Workload("mqa_rep_win_sink_d128", B=1, S=1024, Hq=8, Hkv=1, D=128, P=8, window_left=150, sinks=True,
               doc_mode="explicit", doc_lens=(300, 1, 400, 323)),
]


# both dQ passes: from the stored dS blocks (causal shapes) and by recomputing S and dP
CASES = [(w, f, d) for w in SMALL for f in modes(w) for d in ([True, False] if w.causal else [False])]


@pytest.mark.parametrize("w,fused,stored_ds", CASES,
                         ids=[f"{w.name}-{'fused' if f else 'explicit'}-{'stored_ds' if d else 'recompute'}"
                              for w, f, d in CASES])
def test_backward_full_parity_small(w, fused, stored_ds):
    ua, dev, host = _fwd_bwd(w, fused, stored_ds)
    assert ua.stored_ds == stored_ds
    snk = host["sinks"]
    f = oracle.ulysses_fwd(host["q"], host["k"], host["v"], host["pos"], w.causal, w.window_left, None, snk)
    g = oracle.ulysses_bwd(f, host["do"], w.causal, w.window_left, None, snk)
    assert_close("dq", ua.dq_seq.float().cpu().numpy(), g["dq_seq"])
    sk = sv = None
    if not fused and w.Hkv < w.P:
        # replicated key/value heads, explicit exchange: each rank's partial
        # dK/dV is stored in bf16 before the exchange back sums the replicas
        sk = oracle.relayout_bwd(half_ulp_bf16(g["dk_head"]), w.P, w.Hkv)
        sv = oracle.relayout_bwd(half_ulp_bf16(g["dv_head"]), w.P, w.Hkv)
    assert_close("dk", ua.dk_seq.float().cpu().numpy(), g["dk_seq"], slack=sk)
    assert_close("dv", ua.dv_seq.float().cpu().numpy(), g["dv_seq"], slack=sv)
    if snk is not None:
        got = ua.dsinks.cpu().numpy().astype(np.float64)
        bound = dsink_bound(f["lse"], snk, f["o_head"], g["do_head"], w.Hq // w.P)
        print(f"[parity] dsinks: max err {np.max(np.abs(got - g['dsinks'])):.3e}, min bound {bound.min():.3e}")
        assert np.all(np.abs(got - g["dsinks"]) <= bound)


def _rank_views(w, host, r):
    hq = w.Hq // w.P
    T = w.B * w.S
    qh = oracle.relayout_fwd(host["q"], w.P)[r].reshape(T, hq, w.D)
    kh = oracle.relayout_fwd(host["k"], w.P, replicate=True)[r].reshape(T, -1, w.D)
    vh = oracle.relayout_fwd(host["v"], w.P, replicate=True)[r].reshape(T, -1, w.D)
    doh = oracle.relayout_fwd(host["do"], w.P)[r].reshape(T, hq, w.D)
    cu, _, _ = oracle.cu_seqlens_from_position_ids(host["pos"])
    snk = None if host["sinks"] is None else host["sinks"][r * hq:(r + 1) * hq]
    return qh, kh, vh, doh, cu, snk


def _gpu_head(ua, name, w, r, heads):
    """[T][heads][D] float64 of all local heads of rank r for output `name`."""
    return np.stack([head_values(ua, name, r, j, heads) for j in range(heads)], axis=1)


@pytest.mark.parametrize("w,groups,fused,stored_ds", [
    (W.GPTOSS_WIN, [(0, 0), (5, 0)], True, True),
    (W.LLAMA32K, [(2, 0), (7, 0)], True, True),
    (W.LLAMA32K, [(4, 0)], False, False),
], ids=["gptoss_win-fused-stored_ds", "llama32k-fused-stored_ds", "llama32k-explicit-recompute"])
def test_backward_full_size_whole_groups(w, groups, fused, stored_ds):
    """Every query head of a GQA group on a rank: dQ of those heads and the
    complete dK/dV of their key/value head, compared element by element."""
    ua, dev, host = _fwd_bwd(w, fused, stored_ds)
    G = w.Hq // w.Hkv
    for r, kvh in groups:
        qh, kh, vh, doh, cu, snk = _rank_views(w, host, r)
        heads = list(range(kvh * G, (kvh + 1) * G))
        O, L = oracle.attention_fwd(qh, kh, vh, cu, w.causal, w.window_left, None, snk, heads=heads)
        dq, dk, dv, ds = oracle.attention_bwd(qh, kh, vh, O, L, doh, cu, w.causal, w.window_left, None, snk,
                                              heads=heads)
        gq = _gpu_head(ua, "dq", w, r, w.Hq // w.P)
        gk = _gpu_head(ua, "dk", w, r, w.Hkv // w.P)
        gv = _gpu_head(ua, "dv", w, r, w.Hkv // w.P)
        assert_close(f"dq r{r}", gq[:, heads], dq[:, heads])
        assert_close(f"dk r{r} kv{kvh}", gk[:, kvh], dk[:, kvh])
        assert_close(f"dv r{r} kv{kvh}", gv[:, kvh], dv[:, kvh])
        if ds is not None:
            hq = w.Hq // w.P
            got = ua.dsinks.cpu().numpy().astype(np.float64)[r * hq:(r + 1) * hq][heads]
            lse_r = L.reshape(hq, w.B, w.S).transpose(1, 0, 2)[None]
            o_r = O.reshape(1, w.B, w.S, hq, w.D)
            do_r = doh.reshape(1, w.B, w.S, hq, w.D)
            bound = dsink_bound(lse_r, snk, o_r, do_r, hq)[heads]
            assert np.all(np.abs(got - ds[heads]) <= bound), (np.abs(got - ds[heads]), bound)


@pytest.mark.parametrize("w,group", [(SMALL[2], 1), (SMALL[3], 3), (SMALL[6], 1), (W.MHA4K, 5)],
                         ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_backward_stored_ds_in_head_groups(w, group):
    """The stored-dS passes run a group of key/value heads at a time over one
    workspace (how a long sequence fits): same gradients as the oracle."""
    ua, dev, host = _fwd_bwd(w, True, None, group)
    assert ua.stored_ds and len(ua.ds_groups) == -(-w.Hkv // group)
    snk = host["sinks"]
    f = oracle.ulysses_fwd(host["q"], host["k"], host["v"], host["pos"], w.causal, w.window_left, None, snk)
    g = oracle.ulysses_bwd(f, host["do"], w.causal, w.window_left, None, snk)
    assert_close("dq", ua.dq_seq.float().cpu().numpy(), g["dq_seq"])
    assert_close("dk", ua.dk_seq.float().cpu().numpy(), g["dk_seq"])
    assert_close("dv", ua.dv_seq.float().cpu().numpy(), g["dv_seq"])


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "explicit"])
def test_backward_full_size_replicated_kv_head(fused):
    """Sp size 16 over 8 key/value heads: one key/value head, held by two
    ranks.  dQ of both ranks' query heads element by element; dK/dV of the
    head equal the sum of the two ranks' partial gradients (each rank's
    partial checked too in explicit mode, where it is a separate buffer)."""
    w = W.LLAMA32K_P16
    ua, dev, host = _fwd_bwd(w, fused)
    rep, hq, h = w.P // w.Hkv, w.Hq // w.P, 5
    dk_sum, dv_sum = 0.0, 0.0
    sk, sv = 0.0, 0.0      # explicit exchange: the partials are rounded to bf16 before the sum
    for r in range(h * rep, (h + 1) * rep):
        qh, kh, vh, doh, cu, snk = _rank_views(w, host, r)
        O, L = oracle.attention_fwd(qh, kh, vh, cu, w.causal, w.window_left, None, snk)
        dq, dk, dv, _ = oracle.attention_bwd(qh, kh, vh, O, L, doh, cu, w.causal, w.window_left, None, snk)
        assert_close(f"dq r{r}", _gpu_head(ua, "dq", w, r, hq), dq)
        if not fused:
            assert_close(f"dk partial r{r}", ua.dk_head[r].reshape(-1, w.D).double().cpu().numpy(), dk[:, 0])
            assert_close(f"dv partial r{r}", ua.dv_head[r].reshape(-1, w.D).double().cpu().numpy(), dv[:, 0])
        dk_sum = dk_sum + dk[:, 0]
        dv_sum = dv_sum + dv[:, 0]
        sk = sk + half_ulp_bf16(dk[:, 0])
        sv = sv + half_ulp_bf16(dv[:, 0])
    assert_close(f"dk head {h}", seq_head_values(ua.dk_seq, h), dk_sum, slack=None if fused else sk)
    assert_close(f"dv head {h}", seq_head_values(ua.dv_seq, h), dv_sum, slack=None if fused else sv)


@pytest.mark.parametrize("w", [W.GPTOSS_FULL, W.LONG128K], ids=lambda w: w.name)
def test_backward_full_size_sampled(w):
    """Long single documents: dQ at seeded rows, dK/dV at seeded keys near the
    end of the document (few rows see them), all query heads of the group."""
    ua, dev, host = _fwd_bwd(w, fused=True)
    rng = np.random.Generator(np.random.PCG64(17))
    G = w.Hq // w.Hkv
    r, kvh = w.P - 1, 0
    qh, kh, vh, doh, cu, snk = _rank_views(w, host, r)
    # a uniform sample of rows stands for the tensor in both measures; the
    # document's first and last rows are checked against the max-abs bound
    # (the first row sees one key, so dP - D cancels and the bf16 rounding of
    # O, which D is computed from, is amplified there)
    rows = np.sort(rng.choice(w.S, 16, replace=False))
    edge = np.array([0, 1, w.S - 1])
    gq = _gpu_head(ua, "dq", w, r, w.Hq // w.P)
    for h in (kvh * G, kvh * G + G - 1):
        sink = None if snk is None else snk[h]
        dq = oracle.attention_bwd_rows(qh, kh, vh, doh, cu, rows, h, w.causal, w.window_left, sink=sink)
        assert_close(f"dq rows h{h}", gq[rows, h], dq)
        dq = oracle.attention_bwd_rows(qh, kh, vh, doh, cu, edge, h, w.causal, w.window_left, sink=sink)
        assert_close(f"dq edge rows h{h}", gq[edge, h], dq, rel_l2=np.inf)
    keys = np.sort(np.concatenate([w.S - 1 - rng.choice(384, 6, replace=False), [w.S - 1]]))
    dk, dv = oracle.attention_bwd_keys(qh, kh, vh, doh, cu, keys, kvh, w.causal, w.window_left, sinks=snk)
    gk = _gpu_head(ua, "dk", w, r, w.Hkv // w.P)
    gv = _gpu_head(ua, "dv", w, r, w.Hkv // w.P)
    assert_close("dk keys", gk[keys, kvh], dk)
    assert_close("dv keys", gv[keys, kvh], dv)


def test_backward_conservation_at_full_size():
    """Properties that hold at any size, checked over every key of a 128K
    document: without a sink each softmax row of dS sums to zero, so
    sum_u dK_u = 0; and each row of P sums to one, so sum_u dV_u equals the sum
    of dO over the group's query heads and rows."""
    w = W.LONG128K
    ua, dev, host = _fwd_bwd(w, fused=False)
    G = w.Hq // w.Hkv
    for r in range(w.P):
        gk = ua.dk_head[r].reshape(w.S, -1, w.D).double().sum(0).cpu().numpy()
        ak = ua.dk_head[r].reshape(w.S, -1, w.D).double().abs().sum(0).cpu().numpy()
        assert np.all(np.abs(gk) <= 5e-3 * ak + 1e-2), float(np.max(np.abs(gk) / ak))
        gv = ua.dv_head[r].reshape(w.S, -1, w.D).double().sum(0).cpu().numpy()
        av = ua.dv_head[r].reshape(w.S, -1, w.D).double().abs().sum(0).cpu().numpy()
        hq = w.Hq // w.P
        doh = oracle.relayout_fwd(host["do"], w.P)[r, 0]
        want = doh.reshape(w.S, hq // G, G, w.D).sum(axis=(0, 2))
        assert np.all(np.abs(gv - want) <= 5e-3 * (av + np.abs(want)) + 1e-2), float(np.max(np.abs(gv - want)))
