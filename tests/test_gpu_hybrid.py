"""GPU parity of the ring x Ulysses hybrid (USP) through the C ABI: the
hybrid exchange (bit-exact), one attention launch per ring step restricted to
the key/value super-chunk held at that step, the log-sum-exp merge with the
sink folded in once, and the ring backward (block gradients summed in fp32);
compared with the fp64 oracle's hybrid and, at full size, with the attention
definition on sampled rows and keys."""
import numpy as np
import pytest
import torch

import oracle
import usp_workloads as W
from gpu_util import assert_close, built_lib, device_inputs, dsink_bound, half_ulp_bf16, seq_head_values, shape_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built_lib()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


def _run(w, backward=True, stored_ds=None, fused=None, ds_group_size=None):
    from ulysses_sequence_long_gb300.pipeline import HybridAttention
    dev, host = device_inputs(w)
    ha = HybridAttention(shape_of(w), w.ring, with_backward=backward, stored_ds=stored_ds, fused=fused,
                         ds_group_size=ds_group_size)
    ha.forward(dev["q"], dev["k"], dev["v"], dev["pos"], dev["sinks"])
    if backward:
        ha.backward(dev["do"], dev["sinks"])
    torch.cuda.synchronize()
    assert ha.read_status() == 0
    return ha, dev, host


@pytest.mark.parametrize("ring,U,S,H,D", [(2, 2, 1024, 4, 64), (4, 2, 2048, 2, 128), (2, 4, 32768, 8, 128),
                                          (4, 4, 1024, 2, 64)])
def test_hybrid_relayout_bit_exact(ring, U, S, H, D):
    from ulysses_sequence_long_gb300 import binding as B
    P = ring * U
    g = torch.Generator(device="cpu").manual_seed(S + H)
    x = torch.randn((P, 1, S // P, H, D), generator=g).to(torch.bfloat16)
    hpr = H // U if H >= U else 1
    y = torch.empty((U, 1, S, hpr, D), dtype=torch.bfloat16, device="cuda")
    B.usp_hybrid_relayout_fwd(x.cuda(), y, 1, S, H, D, ring, U)
    gy = torch.randn((U, 1, S, hpr, D), generator=g).to(torch.bfloat16)
    z = torch.empty((P, 1, S // P, H, D), dtype=torch.bfloat16, device="cuda")
    B.usp_hybrid_relayout_bwd(gy.cuda(), z, 1, S, H, D, ring, U)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y), oracle.hybrid_relayout_fwd(_bits(x), ring, U, replicate=True))
    if H >= U:   # a pure permutation: bit-exact both ways
        assert np.array_equal(_bits(z), oracle.hybrid_relayout_bwd(_bits(gy), ring, U))
    else:        # replicas summed in fp32, one rounding
        want = oracle.hybrid_relayout_bwd(W.bf16_to_f64(gy), ring, U, H)
        got = z.double().cpu().numpy()
        assert np.all(np.abs(got - want) <= half_ulp_bf16(want) * (1 + 2.0 ** -6))


SMALL = [
    W.Workload("usp_r2u2_packed_d64", B=1, S=1024, Hq=8, Hkv=2, D=64, P=4, ring=2, doc_mode="explicit",
               doc_lens=(300, 400, 324)),
    W.Workload("usp_r4u2_win_sink_d128", B=1, S=2048, Hq=4, Hkv=2, D=128, P=8, ring=4, window_left=200,
               sinks=True, doc_mode="explicit", doc_lens=(700, 1, 900, 447)),
    W.Workload("usp_r2u1_noncausal_d128", B=1, S=512, Hq=2, Hkv=1, D=128, P=2, ring=2, causal=False,
               doc_mode="explicit", doc_lens=(512,)),
    W.Workload("usp_r2u4_kv_rep_d64", B=1, S=1024, Hq=8, Hkv=2, D=64, P=8, ring=2, doc_mode="explicit",
               doc_lens=(600, 424)),
    W.Workload("usp_r2u2_two_rows_d128", B=2, S=512, Hq=4, Hkv=2, D=128, P=4, ring=2, doc_mode="geometric",
               doc_mean=150, seed=7),
    # a short causal window at D=64 (the persistent window forward): ring steps
    # whose units see no key at all
    W.Workload("usp_r2u2_win_sink_d64", B=1, S=1024, Hq=8, Hkv=2, D=64, P=4, ring=2, window_left=100,
               sinks=True, doc_mode="explicit", doc_lens=(400, 1, 623)),
]


def _can_fuse(w):
    return (w.S // w.P) % 128 == 0


# exchanges fused into the kernels' I/O or explicit; dQ from stored dS or recomputed
CASES = [(w, f, d) for w in SMALL for f in ([True, False] if _can_fuse(w) else [False])
         for d in ([True, False] if w.causal else [False])]


@pytest.mark.parametrize("w,fused,stored_ds", CASES,
                         ids=[f"{w.name}-{'fused' if f else 'explicit'}-{'stored_ds' if d else 'recompute'}"
                              for w, f, d in CASES])
def test_hybrid_full_parity_small(w, fused, stored_ds):
    ha, dev, host = _run(w, stored_ds=stored_ds, fused=fused)
    assert ha.stored_ds == stored_ds and ha.fused == fused
    _check_parity(ha, w, host)


@pytest.mark.parametrize("w", [SMALL[0], SMALL[3]], ids=lambda w: w.name)
def test_hybrid_stored_ds_in_head_groups(w):
    """Every ring step's dK/dV and dQ passes run one key/value head at a
    time over one stored-dS workspace: same gradients as the oracle."""
    ha, dev, host = _run(w, fused=True, ds_group_size=1)
    assert ha.stored_ds and len(ha.ds_groups) == w.Hkv
    _check_parity(ha, w, host)


def _check_parity(ha, w, host):
    snk = host["sinks"]
    kw = dict(causal=w.causal, window_left=w.window_left, sinks=snk)
    f = oracle.hybrid_fwd(host["q"], host["k"], host["v"], host["pos"], w.ring, **kw)
    assert_close("o_seq", ha.o_seq.float().cpu().numpy(), f["o_seq"])
    assert_close("lse", ha.lse.cpu().numpy(), f["lse"], bf16_out=False)
    g = oracle.hybrid_bwd(f, host["do"], return_steps=True, **kw)
    # Each ring step's block gradient is stored in bf16 before the fp32 sum,
    # and with replicated key/value heads each replica's sum is stored in bf16
    # before the exchange adds the replicas: the tolerance leaves out half a
    # bf16 ulp of each of those intermediate values (from the oracle's own).
    U = w.P // w.ring
    slack = {}
    for n, H in (("dq", w.Hq), ("dk", w.Hkv), ("dv", w.Hkv)):
        sl = 0.0
        if w.ring > 1:
            sl = sum(half_ulp_bf16(st[n + "_head"]) for st in g["steps"])
        if n != "dq" and w.Hkv < U:
            sl = sl + half_ulp_bf16(g[n + "_head"])
        slack[n] = None if np.isscalar(sl) else oracle.hybrid_relayout_bwd(sl, w.ring, U, H if H < U else None)
    assert_close("dq", ha.dq_seq.float().cpu().numpy(), g["dq_seq"], slack=slack["dq"])
    assert_close("dk", ha.dk_seq.float().cpu().numpy(), g["dk_seq"], slack=slack["dk"])
    assert_close("dv", ha.dv_seq.float().cpu().numpy(), g["dv_seq"], slack=slack["dv"])
    if snk is not None:
        got = ha.dsinks.cpu().numpy().astype(np.float64)
        bound = dsink_bound(f["lse"], snk, f["o_head"], g["do_head"], w.Hq // U)
        assert np.all(np.abs(got - g["dsinks"]) <= bound), (np.abs(got - g["dsinks"]), bound)


def test_hybrid_ring_step_without_keys_gives_empty_block():
    """A causal ring step whose key/value super-chunk lies after the rows:
    the step's output is O = 0 and LSE = -inf (nothing to merge)."""
    from ulysses_sequence_long_gb300 import binding as B
    w = SMALL[0]
    ha, dev, host = _run(w, backward=False, fused=False)
    # step 1: super-chunk 0 holds keys of super-chunk 1 (after its rows)
    B.usp_attn_fwd(ha.params(None, 1), ha.q_head, ha.k_head, ha.v_head, ha.o_step, ha.lse_step, ha.status)
    torch.cuda.synchronize()
    C = w.S // w.ring
    assert torch.all(ha.o_step[:, :, :C] == 0)
    assert torch.all(torch.isinf(ha.lse_step[:, :, :, :C])) and torch.all(ha.lse_step[:, :, :, :C] < 0)
    assert ha.read_status() == 0


def test_hybrid_refusals():
    from ulysses_sequence_long_gb300 import binding as B
    w = SMALL[0]
    ha, dev, host = _run(w, backward=False, fused=False)
    bad = [
        (B.attn_params(1, 1024, 8, 2, 64, 2, ha.cu_seqlens, ha.n_docs, ring=2, ring_step=2), B.USP_ERR_INVALID_ARG),
        (B.attn_params(1, 1024, 8, 2, 64, 2, ha.cu_seqlens, ha.n_docs, ring=8, ring_step=0), B.USP_ERR_UNSUPPORTED),
        # sequence shards of 1024 / (4 * 4) = 64 tokens are too short for fused I/O
        (B.attn_params(1, 1024, 8, 2, 64, 4, ha.cu_seqlens, ha.n_docs, ring=4, ring_step=0,
                       io_layout=B.USP_IO_SEQ), B.USP_ERR_UNSUPPORTED),
        (B.attn_params(1, 1024, 8, 2, 64, 2, ha.cu_seqlens, ha.n_docs, ring=1, ring_step=1), B.USP_ERR_INVALID_ARG),
        (B.attn_params(1, 1024, 8, 2, 64, 2, ha.cu_seqlens, ha.n_docs, sinks=torch.zeros(8, device="cuda"), ring=2,
                       ring_step=0), B.USP_ERR_INVALID_ARG),     # the sink joins in the merge, not per step
    ]
    for prm, code in bad:
        with pytest.raises(B.UspError) as e:
            B.usp_attn_fwd(prm, ha.q_head, ha.k_head, ha.v_head, ha.o_step, ha.lse_step)
        assert e.value.code == code


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "explicit"])
def test_hybrid_full_size_sampled(fused):
    """Llama-shaped 32K packed workload as ring 2 x ulysses 4: sampled rows
    of O/LSE/dQ and keys of dK/dV against the attention definition."""
    w = W.LLAMA32K_RING2
    ha, dev, host = _run(w, fused=fused)
    U = w.P // w.ring
    hq, hk = w.Hq // U, w.Hkv // U
    G = hq // hk
    qh = oracle.hybrid_relayout_fwd(host["q"], w.ring, U)
    kh = oracle.hybrid_relayout_fwd(host["k"], w.ring, U, replicate=True)
    vh = oracle.hybrid_relayout_fwd(host["v"], w.ring, U, replicate=True)
    doh = oracle.hybrid_relayout_fwd(host["do"], w.ring, U)
    cu, _, _ = oracle.cu_seqlens_from_position_ids(host["pos"])
    rng = np.random.Generator(np.random.PCG64(23))
    C = w.S // w.ring

    def vals(name, u, h, H_per_u):
        """float64 [S][D] of local head h of Ulysses rank u for output `name`."""
        if not fused:
            return getattr(ha, name + "_head")[u, 0, :, h].double().cpu().numpy()
        return seq_head_values(getattr(ha, name + "_seq"), u * H_per_u + h)
    for u, j in [(0, 0), (3, 7)]:
        Q, K, V, dO = qh[u, 0], kh[u, 0], vh[u, 0], doh[u, 0]
        # rows on both sides of the super-chunk boundary and at document starts
        rows = np.sort(np.unique(np.concatenate([rng.choice(w.S, 12, replace=False), [0, C - 1, C, C + 1, w.S - 1],
                                                 cu[1:-1], cu[1:-1] + 1])))
        rows = rows[rows < w.S]
        O, L = oracle.attention_fwd_rows(Q, K, V, cu, rows, j)
        assert_close(f"O u{u} h{j}", vals("o", u, j, hq)[rows], O)
        assert_close(f"LSE u{u} h{j}", ha.lse[u, 0, j, rows].double().cpu().numpy(), L, bf16_out=False)
        inner = rows[~np.isin(rows, np.concatenate([cu[:-1], cu[:-1] + 1]))]
        dq = oracle.attention_bwd_rows(Q, K, V, dO, cu, inner, j)
        dq_steps = [oracle.attention_bwd_rows(Q, K, V, dO, cu, inner, j, key_window=(c * C, (c + 1) * C))
                    for c in range(w.ring)]
        assert_close(f"dQ u{u} h{j}", vals("dq", u, j, hq)[inner], dq,
                     slack=sum(half_ulp_bf16(x) for x in dq_steps))
        # keys near the end of the last document (few rows see them) and just
        # before the super-chunk boundary (rows of both super-chunks see them)
        kvh = j // G
        keys = np.sort(np.concatenate([w.S - 1 - rng.choice(256, 4, replace=False), [C - 2, C - 1]]))
        dk, dv = oracle.attention_bwd_keys(Q, K, V, dO, cu, keys, kvh)
        parts = [oracle.attention_bwd_keys(Q, K, V, dO, cu, keys, kvh, row_window=(c * C, (c + 1) * C))
                 for c in range(w.ring)]
        assert_close(f"dK u{u} kv{kvh}", vals("dk", u, kvh, hk)[keys], dk,
                     slack=sum(half_ulp_bf16(x[0]) for x in parts))
        assert_close(f"dV u{u} kv{kvh}", vals("dv", u, kvh, hk)[keys], dv,
                     slack=sum(half_ulp_bf16(x[1]) for x in parts))
