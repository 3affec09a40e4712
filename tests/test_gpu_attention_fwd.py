"""GPU parity of the forward path through the C ABI: exchange q/k/v, rebuild
document boundaries, tcgen05 attention, exchange O back; compared with the
fp64 oracle on the same seeded bf16 inputs (max-abs <= 2e-2 and relative L2
<= 5e-3 on O and LSE)."""
import numpy as np
import pytest
import torch

import oracle
import usp_workloads as W
from gpu_util import assert_close, built_lib, device_inputs, head_values, modes, shape_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built_lib()


def _forward(w, fused=False):
    from ulysses_sequence_long_gb300.pipeline import UlyssesAttention
    dev, host = device_inputs(w)
    ua = UlyssesAttention(shape_of(w), with_backward=False, fused=fused)
    ua.forward(dev["q"], dev["k"], dev["v"], dev["pos"], dev["sinks"])
    torch.cuda.synchronize()
    assert ua.read_status() == 0
    return ua, dev, host


def _oracle_rank_head(w, host, ua, r, j):
    """fp64 O [T][D] and LSE [T] of rank r, local head j, from the oracle alone."""
    hq = w.Hq // w.P
    qh = oracle.relayout_fwd(host["q"], w.P)[r].reshape(w.B * w.S, hq, w.D)
    kh = oracle.relayout_fwd(host["k"], w.P, replicate=True)[r].reshape(w.B * w.S, -1, w.D)
    vh = oracle.relayout_fwd(host["v"], w.P, replicate=True)[r].reshape(w.B * w.S, -1, w.D)
    cu, _, _ = oracle.cu_seqlens_from_position_ids(host["pos"])
    snk = None if host["sinks"] is None else host["sinks"][r * hq:(r + 1) * hq]
    O, L = oracle.attention_fwd(qh, kh, vh, cu, w.causal, w.window_left, None, snk, heads=[j])
    return O[:, j], L[j]


def _gpu_rank_head(w, ua, r, j):
    o = head_values(ua, "o", r, j, w.Hq // w.P)
    lse = ua.lse[r][:, j].reshape(-1).cpu().numpy()
    return o, lse


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
    # short causal windows at D=64 (the persistent schedule over a group's heads):
    # an odd group size, a replicated key/value head at window 128, window 0 with
    # a ragged batch of rows that are not a multiple of 128 tokens
    W.Workload("win_d64_odd_group", B=1, S=1024, Hq=12, Hkv=4, D=64, P=4, window_left=100, sinks=True,
               doc_mode="geometric", doc_mean=300, seed=7),
    W.Workload("win_d64_rep_w128", B=2, S=512, Hq=8, Hkv=2, D=64, P=4, window_left=128,
               doc_mode="geometric", doc_mean=150, seed=9),
    W.Workload("win_d64_w0_ragged", B=3, S=200, Hq=4, Hkv=2, D=64, P=2, window_left=0, sinks=True,
               doc_mode="geometric", doc_mean=60, seed=13),
    # ... and a group of one query head (MHA): the second softmax group has no head
    W.Workload("win_d64_mha", B=1, S=512, Hq=4, Hkv=4, D=64, P=2, window_left=64,
               doc_mode="explicit", doc_lens=(130, 382)),
    # a wider window at D=64 (one Q tile per CTA, two K/V stages)
    W.Workload("win_d64_wide", B=1, S=1024, Hq=8, Hkv=2, D=64, P=2, window_left=300, sinks=True,
               doc_mode="explicit", doc_lens=(700, 324)),
]


CASES = [(w, f) for w in SMALL for f in modes(w)]


@pytest.mark.parametrize("w,fused", CASES, ids=[f"{w.name}-{'fused' if f else 'explicit'}" for w, f in CASES])
def test_forward_full_parity_small(w, fused):
    ua, dev, host = _forward(w, fused)
    snk = host["sinks"]
    ref = oracle.ulysses_fwd(host["q"], host["k"], host["v"], host["pos"], w.causal, w.window_left, None, snk)
    assert_close("o_seq", ua.o_seq.float().cpu().numpy(), ref["o_seq"])
    assert_close("lse", ua.lse.cpu().numpy(), ref["lse"], bf16_out=False)
    cu = ua.cu_seqlens[: ua.n_docs.item() + 1].cpu().numpy()
    assert np.array_equal(cu, ref["cu_seqlens"])


@pytest.mark.parametrize("w,pairs,fused", [
    (W.GPTOSS_WIN, [(0, 0), (3, 5), (7, 7)], True),
    (W.GPTOSS_FULL, [(2, 1), (6, 6)], False),
    (W.LLAMA32K, [(0, 0), (5, 3), (7, 2)], True),
    (W.LLAMA32K, [(1, 1)], False),
    (W.LLAMA32K_P16, [(0, 0), (9, 1), (15, 1)], True),
    (W.LLAMA32K_P16, [(6, 1)], False),
], ids=["gptoss_win-fused", "gptoss_full-explicit", "llama32k-fused", "llama32k-explicit", "llama32k_p16-fused",
        "llama32k_p16-explicit"])
def test_forward_full_size_sampled_heads(w, pairs, fused):
    ua, dev, host = _forward(w, fused)
    for r, j in pairs:
        O, L = _oracle_rank_head(w, host, ua, r, j)
        o, lse = _gpu_rank_head(w, ua, r, j)
        assert_close(f"O r{r} h{j}", o, O)
        assert_close(f"LSE r{r} h{j}", lse, L, bf16_out=False)


def test_forward_long_context_sampled_rows():
    w = W.LONG128K
    ua, dev, host = _forward(w, fused=True)
    rng = np.random.Generator(np.random.PCG64(11))
    hq, hk = w.Hq // w.P, w.Hkv // w.P
    for r, j in [(0, 0), (3, 6)]:
        rows = np.sort(np.concatenate([rng.choice(w.S, 24, replace=False), [0, 1, 127, 128, w.S - 1]]))
        qh = oracle.relayout_fwd(host["q"], w.P)[r, 0]
        kh = oracle.relayout_fwd(host["k"], w.P)[r, 0]
        vh = oracle.relayout_fwd(host["v"], w.P)[r, 0]
        O, L = oracle.attention_fwd_rows(qh, kh, vh, [0, w.S], rows, j)
        o, lse = _gpu_rank_head(w, ua, r, j)
        assert_close(f"O r{r} h{j}", o[rows], O)
        assert_close(f"LSE r{r} h{j}", lse[rows], L, bf16_out=False)


def test_stale_per_shard_cu_seqlens_are_flagged():
    """The per-shard boundaries a collator computes describe S/P tokens; the
    kernel runs on the gathered S (accelerate PR #4209: 41.8% of logits
    were wrong, silently).  Here the device check reports it."""
    from ulysses_sequence_long_gb300 import binding as B
    w = W.TINY
    ua, dev, host = _forward(w)
    stale = oracle.cu_seqlens_from_position_ids(host["pos"][:1])[0]       # rank 0's view: [0,100,128]
    ua.cu_seqlens[: stale.size].copy_(torch.from_numpy(stale))
    ua.n_docs.fill_(stale.size - 1)
    ua.status.zero_()
    ua.attention(dev["sinks"])
    torch.cuda.synchronize()
    assert ua.read_status() == B.USP_ERR_BAD_SEQLENS


def test_attention_refuses_indivisible_heads():
    from ulysses_sequence_long_gb300 import binding as B
    from ulysses_sequence_long_gb300.pipeline import Shape, UlyssesAttention
    ua = UlyssesAttention(Shape(B=1, S=256, Hq=4, Hkv=2, D=64, P=2), with_backward=False, fused=False)
    prm = B.attn_params(1, 256, 4, 2, 64, 8, ua.cu_seqlens, ua.n_docs)   # P=8 does not divide Hq=4
    with pytest.raises(B.UspError) as e:
        B.usp_attn_fwd(prm, ua.q_head, ua.k_head, ua.v_head, ua.o_head, ua.lse)
    assert e.value.code == B.USP_ERR_INDIVISIBLE
    prm = B.attn_params(1, 256, 12, 3, 64, 4, ua.cu_seqlens, ua.n_docs)  # 3 kv heads cannot replicate over 4 ranks
    with pytest.raises(B.UspError) as e:
        B.usp_attn_fwd(prm, ua.q_head, ua.k_head, ua.v_head, ua.o_head, ua.lse)
    assert e.value.code == B.USP_ERR_INDIVISIBLE
    prm = B.attn_params(1, 256, 4, 2, 96, 2, ua.cu_seqlens, ua.n_docs)   # head dim 96
    with pytest.raises(B.UspError) as e:
        B.usp_attn_fwd(prm, ua.q_head, ua.k_head, ua.v_head, ua.o_head, ua.lse)
    assert e.value.code == B.USP_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_fused_exchanges_need_shards_of_128_rows():
    """Sequence-shard I/O tiles each shard in 128-row blocks: a shape whose
    S/P is not a multiple of 128 is refused by the pipeline and by the C ABI."""
    from ulysses_sequence_long_gb300 import binding as B
    from ulysses_sequence_long_gb300.pipeline import Shape, UlyssesAttention
    sh = Shape(B=1, S=320, Hq=4, Hkv=2, D=64, P=2)
    with pytest.raises(ValueError):
        UlyssesAttention(sh, with_backward=False, fused=True)
    ua = UlyssesAttention(sh, with_backward=False)
    assert not ua.fused
    q = torch.zeros((2, 1, 160, 4, 64), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((2, 1, 160, 2, 64), dtype=torch.bfloat16, device="cuda")
    prm = B.attn_params(1, 320, 4, 2, 64, 2, ua.cu_seqlens, ua.n_docs, io_layout=B.USP_IO_SEQ)
    with pytest.raises(B.UspError) as e:
        B.usp_attn_fwd(prm, q, kv, kv, q, ua.lse)
    assert e.value.code == B.USP_ERR_UNSUPPORTED
