"""The C library builds, loads and exports every entry point include/usp.h
declares; the host-side checks that need no GPU behave."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "usp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(usp_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from ulysses_sequence_long_gb300 import _build, binding
    _build.build()
    return binding.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "usp_attn_fwd" in names and "usp_relayout_fwd" in names
    for n in names:
        assert hasattr(lib, n), n
    from ulysses_sequence_long_gb300 import binding
    assert sorted(binding.EXPORTED) == names


def test_status_strings(lib):
    from ulysses_sequence_long_gb300 import binding
    for code in range(10):
        s = binding.status_string(code)
        assert s.startswith("USP_")
    assert binding.status_string(999) == "USP_ERR_UNKNOWN"
    assert lib.usp_version() >= 100


def test_host_checks_without_gpu(lib):
    from ulysses_sequence_long_gb300 import binding as B
    # argument checks return before touching the device
    assert lib.usp_relayout_fwd(None, None, 1, 8, 4, 8, 2, 2, None) == B.USP_ERR_INVALID_ARG
    p = ctypes.c_void_p(16)
    assert lib.usp_relayout_fwd(p, ctypes.c_void_p(1 << 20), 1, 8, 6, 8, 4, 2, None) == B.USP_ERR_INDIVISIBLE
    assert lib.usp_relayout_fwd(p, ctypes.c_void_p(1 << 20), 1, 8, 2, 3, 2, 2, None) == B.USP_ERR_ALIGNMENT
    assert lib.usp_relayout_fwd(p, ctypes.c_void_p(32), 1, 8, 2, 8, 2, 2, None) == B.USP_ERR_INVALID_ARG  # overlap
    assert lib.usp_cu_seqlens_workspace_bytes(1, 4096) >= 16
    # one real rank's exchange buffers: the same refusals as the emulated exchange
    q = ctypes.c_void_p(1 << 20)
    assert lib.usp_a2a_pack_seq_to_head(None, q, 1, 8, 4, 8, 2, 2, None) == B.USP_ERR_INVALID_ARG
    assert lib.usp_a2a_pack_seq_to_head(p, q, 1, 8, 6, 8, 4, 2, None) == B.USP_ERR_INDIVISIBLE
    assert lib.usp_a2a_unpack_seq_to_head(p, q, 1, 8, 6, 8, 4, 2, None) == B.USP_ERR_INDIVISIBLE
    assert lib.usp_a2a_pack_head_to_seq(p, q, 1, 8, 3, 8, 2, 2, None) == B.USP_ERR_INDIVISIBLE
    assert lib.usp_a2a_unpack_head_to_seq(p, q, 1, 8, 2, 3, 2, 2, None) == B.USP_ERR_ALIGNMENT
    assert lib.usp_a2a_unpack_head_to_seq(p, q, 1, 8, 2, 8, 4, 4, None) == B.USP_ERR_UNSUPPORTED  # fp32 replica sum
    prm = B.AttnParams(1, 256, 4, 2, 96, 2, 1, -1, 0.0, 16, 16, None)
    assert lib.usp_attn_fwd(ctypes.byref(prm), p, p, p, p, p, None, None) == B.USP_ERR_UNSUPPORTED
    prm = B.AttnParams(1, 256, 4, 2, 64, 8, 1, -1, 0.0, 16, 16, None)   # 8 ranks, 4 query heads
    assert lib.usp_attn_fwd(ctypes.byref(prm), p, p, p, p, p, None, None) == B.USP_ERR_INDIVISIBLE
    prm = B.AttnParams(1, 258, 6, 2, 64, 3, 1, -1, 0.0, 16, 16, None)   # 2 kv heads cannot replicate over 3 ranks
    assert lib.usp_attn_fwd(ctypes.byref(prm), p, p, p, p, p, None, None) == B.USP_ERR_INDIVISIBLE
    prm = B.AttnParams(1, 256, 4, 2, 64, 2, 1, -5, 0.0, 16, 16, None)
    assert lib.usp_attn_fwd(ctypes.byref(prm), p, p, p, p, p, None, None) == B.USP_ERR_UNSUPPORTED
    prm = B.AttnParams(1, 256, 4, 2, 64, 2, 1, -1, -1.0, 16, 16, None)
    assert lib.usp_attn_fwd(ctypes.byref(prm), p, p, p, p, p, None, None) == B.USP_ERR_INVALID_ARG
    prm = B.AttnParams(1, 256, 4, 2, 64, 2, 1, -1, 0.0, 16, 16, None)
    assert lib.usp_attn_fwd(ctypes.byref(prm), ctypes.c_void_p(18), p, p, p, p, None, None) == B.USP_ERR_ALIGNMENT
    # sequence-shard I/O: unknown layouts are rejected; S/P must be a multiple of 128
    prm = B.AttnParams(1, 256, 4, 2, 64, 2, 1, -1, 0.0, 16, 16, None, 7)
    assert lib.usp_attn_fwd(ctypes.byref(prm), p, p, p, p, p, None, None) == B.USP_ERR_INVALID_ARG
    prm = B.AttnParams(1, 320, 4, 2, 64, 2, 1, -1, 0.0, 16, 16, None, B.USP_IO_SEQ)
    assert lib.usp_attn_fwd(ctypes.byref(prm), p, p, p, p, p, None, None) == B.USP_ERR_UNSUPPORTED
    ws = ctypes.c_void_p(1 << 20)
    assert lib.usp_attn_bwd_dkdv(ctypes.byref(prm), p, p, p, p, p, p, p, ws, 1 << 20, None, None) == \
        B.USP_ERR_UNSUPPORTED
    assert lib.usp_attn_bwd_dq(ctypes.byref(prm), p, p, p, p, p, p, ws, 1 << 20, None, None) == B.USP_ERR_UNSUPPORTED
    # q/o in shards with k/v in head layout is a forward-only layout
    prm = B.AttnParams(1, 256, 4, 2, 64, 2, 1, -1, 0.0, 16, 16, None, B.USP_IO_SEQ_KV_HEAD)
    assert lib.usp_attn_bwd_dkdv(ctypes.byref(prm), p, p, p, p, p, p, p, ws, 1 << 20, None, None) == \
        B.USP_ERR_UNSUPPORTED
    # head groups: sequence-shard I/O only, inside [0, Hkv), backward passes only
    def grp(io, h0, hc, S=256, Hq=4, Hkv=2, P=2, w=-1):
        return B.AttnParams(1, S, Hq, Hkv, 64, P, 1, w, 0.0, 16, 16, None, io, 1, 0, h0, hc)
    dkdv = lambda prm: lib.usp_attn_bwd_dkdv(ctypes.byref(prm), p, p, p, p, p, p, p, ws, 1 << 20, None, None)
    assert dkdv(grp(B.USP_IO_HEAD, 0, 1)) == B.USP_ERR_UNSUPPORTED
    seq = B.USP_IO_SEQ
    assert dkdv(grp(seq, 1, 2)) == \
        B.USP_ERR_INVALID_ARG
    assert dkdv(grp(seq, 1, 0)) == \
        B.USP_ERR_INVALID_ARG
    assert dkdv(grp(seq, -1, 1)) == \
        B.USP_ERR_INVALID_ARG
    prm = grp(seq, 1, 1)
    assert lib.usp_attn_fwd(ctypes.byref(prm), p, p, p, p, p, None, None) == B.USP_ERR_INVALID_ARG
    assert lib.usp_attn_bwd_preprocess(ctypes.byref(prm), p, p, p, None, ws, 1 << 20, None, None) == B.USP_ERR_INVALID_ARG


def test_fast_workspace_is_stats_plus_stored_ds_blocks(lib):
    """The stored-dS workspace = the statistics + one 16 KiB block per
    (query head, batch row, key tile kt, 64-query slice) a causal mask can
    reach: slices [2kt, 2kt + min(S/64 - 2kt, 2 (1 + ceil(w/128)))).  Counted
    here by brute force over the slices each key tile meets."""
    from ulysses_sequence_long_gb300 import binding as B

    def brute(Bb, S, Hq, w):
        n = 0
        for kt in range(S // 128):
            u_last = kt * 128 + 127
            hi = S if w < 0 else min(S, u_last + w + 1)
            hi = -(-hi // 128) * 128                      # whole 128-row query tiles
            n += len(range(2 * kt, min(hi // 64, S // 64)))
        return n * Hq * Bb * 128 * 64 * 2

    for Bb, S, Hq, Hkv, P, w in [(1, 256, 4, 2, 2, -1), (1, 32768, 32, 8, 8, -1), (1, 16384, 64, 8, 8, 127),
                                 (2, 640, 4, 2, 2, -1), (1, 1024, 8, 2, 2, 200), (1, 4096, 12, 12, 4, 0)]:
        prm = B.AttnParams(Bb, S, Hq, Hkv, 64, P, 1, w, 0.0, 16, 16, None)
        stats = lib.usp_attn_bwd_workspace_bytes(ctypes.byref(prm))
        assert lib.usp_attn_bwd_fast_workspace_bytes(ctypes.byref(prm)) == stats + brute(Bb, S, Hq, w)
    # a head group stores the blocks of its own query heads only; the statistics stay whole
    for Bb, S, Hq, Hkv, P, w, h0, hc in [(1, 32768, 32, 8, 8, -1, 2, 3), (1, 16384, 64, 8, 8, 127, 7, 1),
                                         (1, 4096, 12, 12, 4, -1, 0, 5)]:
        prm = B.AttnParams(Bb, S, Hq, Hkv, 64, P, 1, w, 0.0, 16, 16, None, B.USP_IO_SEQ, 1, 0, h0, hc)
        whole = B.AttnParams(Bb, S, Hq, Hkv, 64, P, 1, w, 0.0, 16, 16, None, B.USP_IO_SEQ)
        stats = lib.usp_attn_bwd_workspace_bytes(ctypes.byref(whole))
        assert lib.usp_attn_bwd_workspace_bytes(ctypes.byref(prm)) == stats
        assert lib.usp_attn_bwd_fast_workspace_bytes(ctypes.byref(prm)) == stats + brute(Bb, S, hc * Hq // Hkv, w)
    # no stored-dS path without a causal mask, or with rows not a multiple of 128
    for Bb, S, causal in [(1, 512, 0), (1, 320, 1)]:
        prm = B.AttnParams(Bb, S, 4, 2, 64, 2, causal, -1, 0.0, 16, 16, None)
        assert lib.usp_attn_bwd_fast_workspace_bytes(ctypes.byref(prm)) == 0
