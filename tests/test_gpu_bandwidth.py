"""GPU parity of the bandwidth kernels through the C ABI: relayout (both
directions, and the fused q/k/v launch) and the document-boundary scan.  Both
must be bit-exact against the oracle, whole, at every workload's full size."""
import numpy as np
import pytest
import torch

import oracle
import usp_workloads as W
from gpu_util import built_lib, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    built_lib()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


RELAYOUT_CASES = [W.TINY, W.MHA4K, W.LLAMA32K, W.GPTOSS_WIN, W.LONG128K]


@pytest.mark.parametrize("w", RELAYOUT_CASES, ids=lambda w: w.name)
def test_relayout_fwd_bwd_bit_exact(w):
    from ulysses_sequence_long_gb300 import binding as B
    for H in sorted({w.Hq, w.Hkv}):
        g = torch.Generator(device="cpu").manual_seed(H)
        x = torch.randn((w.P, w.B, w.S // w.P, H, w.D), generator=g).to(torch.bfloat16)
        xd = x.cuda()
        y = torch.empty((w.P, w.B, w.S, H // w.P, w.D), dtype=torch.bfloat16, device="cuda")
        B.usp_relayout_fwd(xd, y, w.B, w.S, H, w.D, w.P)
        z = torch.empty_like(xd)
        B.usp_relayout_bwd(y, z, w.B, w.S, H, w.D, w.P)
        torch.cuda.synchronize()
        ref = oracle.relayout_fwd(_bits(x), w.P)
        assert np.array_equal(_bits(y), ref)
        assert np.array_equal(_bits(z), _bits(x))
        del xd, y, z


def test_relayout_qkv_fused_equals_separate():
    from ulysses_sequence_long_gb300 import binding as B
    w = W.LLAMA32K
    t = W.qkv_do_shards(w, names=("q", "k", "v"))
    d = {n: x.cuda() for n, x in t.items()}
    heads = {n: torch.empty((w.P, w.B, w.S, (w.Hq if n == "q" else w.Hkv) // w.P, w.D), dtype=torch.bfloat16,
                            device="cuda") for n in d}
    B.usp_relayout_fwd_qkv(d["q"], d["k"], d["v"], heads["q"], heads["k"], heads["v"],
                           w.B, w.S, w.Hq, w.Hkv, w.D, w.P)
    torch.cuda.synchronize()
    for n in ("q", "k", "v"):
        assert np.array_equal(_bits(heads[n]), oracle.relayout_fwd(_bits(t[n]), w.P)), n


@pytest.mark.parametrize("P,B,S,H,D", [(2, 2, 64, 4, 8), (4, 1, 96, 12, 16), (3, 1, 30, 3, 8), (1, 3, 40, 2, 64)])
def test_relayout_ragged_shapes(P, B, S, H, D):
    from ulysses_sequence_long_gb300 import binding as Bd
    g = torch.Generator(device="cpu").manual_seed(P * 100 + S)
    x = torch.randn((P, B, S // P, H, D), generator=g).to(torch.bfloat16)
    y = torch.empty((P, B, S, H // P, D), dtype=torch.bfloat16, device="cuda")
    Bd.usp_relayout_fwd(x.cuda(), y, B, S, H, D, P)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y), oracle.relayout_fwd(_bits(x), P))


@pytest.mark.parametrize("P,S,H,D", [(4, 512, 2, 64), (8, 1024, 1, 128), (16, 32768, 8, 128)])
def test_relayout_replicated_heads(P, S, H, D):
    """Fewer heads than ranks: the exchange copies head r // (P/H) to rank r
    (bit-exact), and the exchange back sums the replicas in fp32, rounded
    once to bf16."""
    from ulysses_sequence_long_gb300 import binding as B
    g = torch.Generator(device="cpu").manual_seed(P * 7 + H)
    x = torch.randn((P, 1, S // P, H, D), generator=g).to(torch.bfloat16)
    y = torch.empty((P, 1, S, 1, D), dtype=torch.bfloat16, device="cuda")
    B.usp_relayout_fwd(x.cuda(), y, 1, S, H, D, P)
    gy = torch.randn((P, 1, S, 1, D), generator=g).to(torch.bfloat16)
    z = torch.empty((P, 1, S // P, H, D), dtype=torch.bfloat16, device="cuda")
    B.usp_relayout_bwd(gy.cuda(), z, 1, S, H, D, P)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y), oracle.relayout_fwd(_bits(x), P, replicate=True))
    want = oracle.relayout_bwd(W.bf16_to_f64(gy), P, H)
    got = z.double().cpu().numpy()
    # fp32 sum of P/H bf16 values, one rounding to bf16: within half an ulp
    # of bf16 at the exact sum (plus the fp32 rounding of the sum)
    a = np.maximum(np.abs(want), 2.0 ** -126)
    half_ulp = np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 8)
    assert np.all(np.abs(got - want) <= half_ulp * (1 + 2.0 ** -6)), float(np.max(np.abs(got - want) / half_ulp))


def test_relayout_qkv_replicated_kv():
    from ulysses_sequence_long_gb300 import binding as B
    w = W.LLAMA32K_P16
    t = W.qkv_do_shards(w, names=("q", "k", "v"))
    d = {n: x.cuda() for n, x in t.items()}
    heads = {n: torch.empty((w.P, w.B, w.S, w.Hq // w.P if n == "q" else 1, w.D), dtype=torch.bfloat16,
                            device="cuda") for n in d}
    B.usp_relayout_fwd_qkv(d["q"], d["k"], d["v"], heads["q"], heads["k"], heads["v"],
                           w.B, w.S, w.Hq, w.Hkv, w.D, w.P)
    torch.cuda.synchronize()
    for n in ("q", "k", "v"):
        assert np.array_equal(_bits(heads[n]), oracle.relayout_fwd(_bits(t[n]), w.P, replicate=(n != "q"))), n


def test_relayout_refusals():
    from ulysses_sequence_long_gb300 import binding as B
    x = torch.zeros((4, 1, 4, 6, 8), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((4, 1, 16, 2, 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.UspError) as e:
        B.usp_relayout_fwd(x, y, 1, 16, 6, 8, 4)       # 4 ranks do not divide 6 heads
    assert e.value.code == B.USP_ERR_INDIVISIBLE
    x2 = torch.zeros((2, 1, 4, 2, 3), dtype=torch.bfloat16, device="cuda")
    y2 = torch.zeros((2, 1, 8, 1, 3), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.UspError) as e:
        B.usp_relayout_fwd(x2, y2, 1, 8, 2, 3, 2)      # 6-byte runs cannot move as 16-byte vectors
    assert e.value.code == B.USP_ERR_ALIGNMENT
    with pytest.raises(TypeError):
        B.usp_relayout_fwd(x.cpu(), y, 1, 16, 6, 8, 4)  # no CPU path
    x3 = torch.zeros((4, 1, 4, 3, 8), dtype=torch.bfloat16, device="cuda")
    y3 = torch.zeros((4, 1, 16, 1, 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.UspError) as e:
        B.usp_relayout_fwd(x3, y3, 1, 16, 3, 8, 4)      # 3 heads cannot be replicated over 4 ranks
    assert e.value.code == B.USP_ERR_INDIVISIBLE
    x4 = torch.zeros((4, 1, 4, 2, 8), dtype=torch.float32, device="cuda")
    y4 = torch.zeros((4, 1, 16, 1, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(B.UspError) as e:
        B.usp_relayout_bwd(y4, x4, 1, 16, 2, 8, 4)      # summing replicas is defined for bf16 only
    assert e.value.code == B.USP_ERR_UNSUPPORTED


# ------------------------------------------------------------------ cu_seqlens

def _run_scan(pos_shards, B, S, P, offset=0, ws=None):
    """The scan on the device; `offset` int32 elements of padding in front of
    the positions (offset 1: a buffer that is not 16-byte aligned)."""
    from ulysses_sequence_long_gb300 import binding as Bd
    flat = torch.from_numpy(np.ascontiguousarray(pos_shards, dtype=np.int32).reshape(-1))
    buf = torch.zeros((offset + flat.numel(),), dtype=torch.int32, device="cuda")
    buf[offset:] = flat.cuda()
    pos = buf[offset:]
    cu = torch.full((B * S + 1,), -7, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    mx = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if ws is None:
        ws = torch.empty((Bd.usp_cu_seqlens_workspace_bytes(B, S),), dtype=torch.uint8, device="cuda")
    Bd.usp_cu_seqlens_from_position_ids(pos, B, S, P, cu, n, mx, ws, st)
    torch.cuda.synchronize()
    nn = int(n.item())
    return cu[: nn + 1].cpu().numpy(), nn, int(mx.item()), int(st.item())


@pytest.mark.parametrize("w", W.ALL, ids=lambda w: w.name)
def test_cu_seqlens_bit_exact(w):
    pos = W.position_ids_shards(w)
    cu, n, mx, st = _run_scan(pos, w.B, w.S, w.P)
    rcu, rn, rmx = oracle.cu_seqlens_from_position_ids(pos)
    assert st == 0
    assert n == rn and mx == rmx
    assert np.array_equal(cu, rcu)


@pytest.mark.parametrize("B,S,P,mean", [(2, 4096, 4, 300), (1, 1 << 20, 8, 37), (3, 12288, 3, 5000),
                                        (1, 4096 * 3 + 64, 2, 1), (2, 256, 1, 100000), (2, 4104, 3, 200),
                                        (3, 1000, 5, 7), (1, 4096 * 40 + 24, 4, 4096 * 9)])
def test_cu_seqlens_many_blocks_and_rows(B, S, P, mean):
    w = W.Workload("scan", B=B, S=S, Hq=P, Hkv=P, D=64, P=P, doc_mode="geometric", doc_mean=mean, seed=B + S)
    pos = W.position_ids_shards(w)
    cu, n, mx, st = _run_scan(pos, B, S, P)
    rcu, rn, rmx = oracle.cu_seqlens_from_position_ids(pos)
    assert st == 0 and n == rn and mx == rmx and np.array_equal(cu, rcu)


@pytest.mark.parametrize("B,S,P,mean", [(1, 1 << 16, 4, 300), (2, 8192, 2, 50)])
def test_cu_seqlens_unaligned_positions(B, S, P, mean):
    # positions that do not start on a 16-byte boundary take the scalar loads
    w = W.Workload("scan_unaligned", B=B, S=S, Hq=P, Hkv=P, D=64, P=P, doc_mode="geometric", doc_mean=mean, seed=3)
    pos = W.position_ids_shards(w)
    rcu, rn, rmx = oracle.cu_seqlens_from_position_ids(pos)
    for offset in (1, 2, 3):
        cu, n, mx, st = _run_scan(pos, B, S, P, offset=offset)
        assert st == 0 and n == rn and mx == rmx and np.array_equal(cu, rcu)


def test_cu_seqlens_workspace_reused_across_calls():
    # the block states left by one call must never leak into the next
    from ulysses_sequence_long_gb300 import binding as Bd
    ws = torch.empty((Bd.usp_cu_seqlens_workspace_bytes(1, 1 << 20),), dtype=torch.uint8, device="cuda")
    for seed, mean in ((1, 500), (2, 20000), (3, 3), (4, 1 << 21)):
        w = W.Workload("scan_reuse", B=1, S=1 << 20, Hq=8, Hkv=8, D=64, P=8, doc_mode="geometric", doc_mean=mean,
                       seed=seed)
        pos = W.position_ids_shards(w)
        cu, n, mx, st = _run_scan(pos, 1, 1 << 20, 8, ws=ws)
        rcu, rn, rmx = oracle.cu_seqlens_from_position_ids(pos)
        assert st == 0 and n == rn and mx == rmx and np.array_equal(cu, rcu)


def test_cu_seqlens_flags_negative_positions():
    from ulysses_sequence_long_gb300 import binding as Bd
    pos = W.position_ids_shards(W.TINY).copy()
    pos[1, 0, 5] = -3
    _, _, _, st = _run_scan(pos, 1, 256, 2)
    assert st == Bd.USP_ERR_BAD_POSITIONS
