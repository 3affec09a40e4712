"""The workspace-free document-boundary call, for callers that cannot
allocate device memory (their memory is reserved by another allocator, or
they only receive input and output pointers).

It must give exactly what the workspace form gives, on consecutive calls
that share its fixed internal scratch array.  This file is collected last so
that a run stopping at the first failure has run every other test already.
"""
import numpy as np
import pytest
import torch

import oracle
import usp_workloads as W

pytestmark = pytest.mark.gpu


def _outputs(n_tokens):
    return (torch.full((n_tokens + 1,), -1, dtype=torch.int32, device="cuda"),
            torch.zeros(1, dtype=torch.int32, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda"),
            torch.zeros(1, dtype=torch.int32, device="cuda"))


def _with_workspace(pos, B, S, P):
    from ulysses_sequence_long_gb300 import binding as Bd
    cu, n, mx, st = _outputs(B * S)
    ws = torch.empty((Bd.usp_cu_seqlens_workspace_bytes(B, S),), dtype=torch.uint8, device="cuda")
    Bd.usp_cu_seqlens_from_position_ids(pos, B, S, P, cu, n, mx, ws, st)
    return cu, n, mx, st


def _without_workspace(pos, B, S, P):
    from ulysses_sequence_long_gb300 import binding as Bd
    cu, n, mx, st = _outputs(B * S)
    Bd.usp_cu_seqlens_from_position_ids_noalloc(pos, B, S, P, cu, n, mx, st)
    return cu, n, mx, st


def test_noalloc_matches_workspace_form_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from ulysses_sequence_long_gb300 import _build
    _build.build()
    cases = [
        W.Workload("many_docs", B=1, S=1 << 20, Hq=8, Hkv=8, D=64, P=8, doc_mode="geometric", doc_mean=37, seed=9),
        W.Workload("two_rows", B=2, S=12288, Hq=4, Hkv=4, D=64, P=4, doc_mode="geometric", doc_mean=900, seed=2),
        # the largest size the fixed array takes: B*S = 2^24 positions
        W.Workload("at_the_limit", B=1, S=1 << 24, Hq=8, Hkv=8, D=64, P=8, doc_mode="geometric", doc_mean=5000,
                   seed=4),
    ]
    for w in cases:   # calls in a row, each over different data
        pos_np = W.position_ids_shards(w)
        pos = torch.from_numpy(pos_np).cuda()
        a = _with_workspace(pos, w.B, w.S, w.P)
        b = _without_workspace(pos, w.B, w.S, w.P)
        torch.cuda.synchronize()
        n = int(a[1].item())
        assert int(b[1].item()) == n and int(b[2].item()) == int(a[2].item())
        assert int(a[3].item()) == 0 and int(b[3].item()) == 0
        assert np.array_equal(a[0][: n + 1].cpu().numpy(), b[0][: n + 1].cpu().numpy())
        # and straight against the oracle's sequential scan
        rcu, rn, rmx = oracle.cu_seqlens_from_position_ids(pos_np)
        assert int(b[1].item()) == rn and int(b[2].item()) == rmx
        assert np.array_equal(b[0][: rn + 1].cpu().numpy(), rcu)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from ulysses_sequence_long_gb300 import binding as Bd
    pos = torch.zeros((1,), dtype=torch.int32, device="cuda")
    cu, n, mx, st = _outputs(1)
    with pytest.raises(Bd.UspError) as e:
        Bd.usp_cu_seqlens_from_position_ids_noalloc(pos, 1, (1 << 24) + 2, 2, cu, n, mx, st)
    assert e.value.code == Bd.USP_ERR_UNSUPPORTED
