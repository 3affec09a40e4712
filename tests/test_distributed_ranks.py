"""The multi-process Ulysses path with real ranks over gloo, on the CPU.

Each rank is its own process; the exchanges are real all-to-all collectives
between them.  The local steps are the fp64 oracle's per-rank functions (a
stand-in for the CUDA kernels, which need a GPU), so what is checked here is
the orchestration: the position_ids gather, which chunks go to which rank,
the sink slices, the replica sums of dK/dV and the dsinks gather.  Every
rank's results must equal the emulated P-rank oracle's rank r: the head
layout after the exchange bit for bit, the attention outputs to fp64
rounding.
"""
import numpy as np
import pytest

import oracle
import usp_workloads as W
from dist_launch import run_ranks

CASES = [
    W.Workload("dist_gqa_packed_p2", B=1, S=256, Hq=4, Hkv=2, D=16, P=2, doc_mode="explicit", doc_lens=(100, 90, 66)),
    W.Workload("dist_win_sink_p4", B=1, S=256, Hq=8, Hkv=4, D=8, P=4, window_left=20, sinks=True,
               doc_mode="explicit", doc_lens=(60, 1, 130, 65)),
    W.Workload("dist_kv_replicated_p4", B=1, S=128, Hq=8, Hkv=2, D=8, P=4, doc_mode="explicit", doc_lens=(70, 58)),
    W.Workload("dist_two_rows_p2", B=2, S=96, Hq=4, Hkv=2, D=8, P=2, doc_mode="geometric", doc_mean=30, seed=4),
]


def _reference(w):
    t = W.qkv_do_shards(w)
    host = {n: W.bf16_to_f64(x) for n, x in t.items()}
    pos = W.position_ids_shards(w)
    sk = W.sinks(w)
    snk = None if sk is None else sk.double().numpy()
    f = oracle.ulysses_fwd(host["q"], host["k"], host["v"], pos, w.causal, w.window_left, None, snk)
    g = oracle.ulysses_bwd(f, host["do"], w.causal, w.window_left, None, snk)
    return f, g


def _close(got, want, name):
    scale = max(1.0, float(np.max(np.abs(want))))
    err = float(np.max(np.abs(got - want)))
    assert err <= 1e-12 * scale, f"{name}: {err:.3e}"


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_ranks_over_gloo_equal_the_emulated_ranks(w, tmp_path):
    ranks = run_ranks(w, "oracle", tmp_path)
    f, g = _reference(w)
    for r, got in enumerate(ranks):
        # the exchange itself: rank r holds the whole sequence of its heads
        assert np.array_equal(got["q_h"], f["q_head"][r])
        assert np.array_equal(got["k_h"], f["k_head"][r])
        assert np.array_equal(got["v_h"], f["v_head"][r])
        _close(got["o"], f["o_seq"][r], f"O rank {r}")
        _close(got["lse"][0], f["lse"][r], f"LSE rank {r}")
        _close(got["dq"], g["dq_seq"][r], f"dQ rank {r}")
        _close(got["dk"], g["dk_seq"][r], f"dK rank {r}")
        _close(got["dv"], g["dv_seq"][r], f"dV rank {r}")
        if w.sinks:
            _close(got["dsinks"], g["dsinks"], f"dsinks rank {r}")
