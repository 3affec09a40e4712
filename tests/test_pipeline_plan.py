"""Host logic of the backward plan (no GPU): when the dK/dV pass stores dS
for the dQ pass, and in which key/value head groups the two passes run."""
import ctypes

import pytest

from ulysses_sequence_long_gb300 import binding as B
from ulysses_sequence_long_gb300.pipeline import plan_backward

GB = 1 << 30


@pytest.fixture(scope="module")
def lib():
    from ulysses_sequence_long_gb300 import _build
    _build.build()
    return B.load()


def params(S=131072, Hq=28, Hkv=4, P=4, causal=1, io=B.USP_IO_SEQ):
    # device pointers are never touched by the size queries
    return B.AttnParams(1, S, Hq, Hkv, 128, P, causal, -1, 0.0, 16, 16, None, io)


def blocks_per_head(S):
    """dS blocks of one query head for a causal mask without window: key tile
    kt meets the 64-query slices [2kt, S/64)."""
    return sum(S // 64 - 2 * kt for kt in range(S // 128))


def test_plan_for_a_long_single_document(lib):
    prm = params()
    stats = lib.usp_attn_bwd_workspace_bytes(ctypes.byref(prm))
    per_head = blocks_per_head(131072) * 128 * 64 * 2
    # everything fits: one pass over all heads
    n, stored, groups = plan_backward(prm, 4096 * GB, None, 4, groups_ok=True)
    assert (n, stored, groups) == (stats + 28 * per_head, True, [(0, 0)])
    # half of 500 GB holds two key/value heads (14 query heads) at a time
    n, stored, groups = plan_backward(prm, 500 * GB, None, 4, groups_ok=True)
    assert (n, stored, groups) == (stats + 14 * per_head, True, [(0, 2), (2, 2)])
    # half of a GB300 holds one key/value head at a time
    n, stored, groups = plan_backward(prm, 280 * GB, None, 4, groups_ok=True)
    assert (n, stored, groups) == (stats + 7 * per_head, True, [(0, 1), (1, 1), (2, 1), (3, 1)])
    # not even one group fits: the dQ pass recomputes S and dP
    n, stored, groups = plan_backward(prm, 100 * GB, None, 4, groups_ok=True)
    assert (n, stored, groups) == (stats, False, [(0, 0)])
    # head-layout I/O runs no groups
    prm_h = params(io=B.USP_IO_HEAD)
    n, stored, groups = plan_backward(prm_h, 280 * GB, None, 4, groups_ok=False)
    assert (stored, groups) == (False, [(0, 0)])


def test_forced_groups_and_refusals(lib):
    prm = params()
    stats = lib.usp_attn_bwd_workspace_bytes(ctypes.byref(prm))
    per_head = blocks_per_head(131072) * 128 * 64 * 2
    n, stored, groups = plan_backward(prm, 0, None, 4, groups_ok=True, group_size=3)
    assert (n, stored, groups) == (stats + 21 * per_head, True, [(0, 3), (3, 1)])
    with pytest.raises(ValueError):
        plan_backward(prm, 0, None, 4, groups_ok=False, group_size=1)
    with pytest.raises(ValueError):
        plan_backward(prm, 0, False, 4, groups_ok=True, group_size=1)
    with pytest.raises(ValueError):
        plan_backward(prm, 0, None, 4, groups_ok=True, group_size=5)
    # a non-causal shape has no stored-dS backward
    with pytest.raises(ValueError):
        plan_backward(params(S=4096, causal=0), 4096 * GB, True, 4)
    n, stored, _ = plan_backward(params(S=4096, causal=0), 4096 * GB, None, 4, groups_ok=True)
    assert not stored
