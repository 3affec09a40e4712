"""The multi-process Ulysses path on the GPU: 2 or 4 ranks, each its own
process on cuda:0, the exchanges as gloo all-to-all collectives staged
through host memory (no kernel waits for another rank), every local step in
the library's kernels (pack/unpack of the exchange, document boundaries,
attention forward and backward).  Compared with the fp64 oracle of the
emulated P-rank path: the head layouts after the exchange bit for bit, the
attention outputs within the parity bar."""
import numpy as np
import pytest

import oracle
import usp_workloads as W
from dist_launch import run_ranks
from gpu_util import assert_close, dsink_bound, half_ulp_bf16, need_gpu

pytestmark = pytest.mark.gpu

CASES = [
    W.Workload("gpu_dist_gqa_win_sink_p2", B=1, S=1024, Hq=8, Hkv=2, D=128, P=2, window_left=200, sinks=True,
               doc_mode="explicit", doc_lens=(300, 1, 423, 300)),
    W.Workload("gpu_dist_kv_replicated_p4", B=1, S=512, Hq=8, Hkv=2, D=64, P=4, doc_mode="explicit",
               doc_lens=(200, 180, 132)),
    W.Workload("gpu_dist_two_rows_p2", B=2, S=640, Hq=4, Hkv=2, D=128, P=2, doc_mode="geometric", doc_mean=150,
               seed=5),
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_gpu_ranks_over_gloo_match_the_oracle(w, tmp_path):
    need_gpu()
    from ulysses_sequence_long_gb300 import _build
    _build.build()
    ranks = run_ranks(w, "library", tmp_path)
    t = W.qkv_do_shards(w)
    host = {n: W.bf16_to_f64(x) for n, x in t.items()}
    pos = W.position_ids_shards(w)
    sk = W.sinks(w)
    snk = None if sk is None else sk.double().numpy()
    f = oracle.ulysses_fwd(host["q"], host["k"], host["v"], pos, w.causal, w.window_left, None, snk)
    g = oracle.ulysses_bwd(f, host["do"], w.causal, w.window_left, None, snk)
    for r, got in enumerate(ranks):
        assert int(got["status"][0]) == 0
        assert np.array_equal(got["q_h"], f["q_head"][r])
        assert np.array_equal(got["k_h"], f["k_head"][r])
        assert np.array_equal(got["v_h"], f["v_head"][r])
        assert_close(f"{w.name} O rank {r}", got["o"], f["o_seq"][r])
        assert_close(f"{w.name} LSE rank {r}", got["lse"][0], f["lse"][r], bf16_out=False)
        assert_close(f"{w.name} dQ rank {r}", got["dq"], g["dq_seq"][r])
        # replicated key/value heads: each replica's partial gradient is bf16
        # before the exchange back sums them (half a bf16 ulp of each part)
        sk = sv = None
        if w.Hkv < w.P:
            sk = oracle.relayout_bwd(half_ulp_bf16(g["dk_head"]), w.P, w.Hkv)[r]
            sv = oracle.relayout_bwd(half_ulp_bf16(g["dv_head"]), w.P, w.Hkv)[r]
        assert_close(f"{w.name} dK rank {r}", got["dk"], g["dk_seq"][r], slack=sk)
        assert_close(f"{w.name} dV rank {r}", got["dv"], g["dv_seq"][r], slack=sv)
        if w.sinks:
            hq = w.Hq // w.P
            bound = dsink_bound(f["lse"], snk, f["o_head"], g["do_head"], hq)
            assert np.all(np.abs(got["dsinks"] - g["dsinks"]) <= bound)
