"""Shared helpers of the GPU parity tests: seeded inputs on the device, the
error measures of the parity bar, and the library build."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import usp_workloads as W

# Parity bar for attention outputs (bf16 inputs, fp32 accumulation) against the
# fp64 oracle: max-abs error and relative L2 error.
MAX_ABS = 2e-2
REL_L2 = 5e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def built_lib():
    need_gpu()
    from ulysses_sequence_long_gb300 import _build, binding
    _build.build()
    return binding.load()


def half_ulp_bf16(x):
    """Half the bf16 spacing at |x|: the rounding error of storing x in bf16."""
    a = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 8)


def errors(got, ref, bf16_out=True, slack=None):
    """(max-abs error, relative L2 error) of got against the fp64 reference.

    For bf16 outputs the max-abs error leaves out the output format's own
    rounding (half a bf16 ulp at the reference value): above |x| = 8 that
    alone exceeds 2e-2, so no bf16-output implementation could meet the bound
    otherwise.  `slack` (per element) leaves out further roundings that the
    method itself takes, e.g. the bf16 partial gradients of replicated
    key/value heads before the exchange sums them.  The relative L2 error is
    taken as is.
    """
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in the GPU output"
    d = np.abs(got - ref)
    if bf16_out:
        d = np.maximum(d - half_ulp_bf16(ref), 0.0)
    if slack is not None:
        d = np.maximum(d - np.asarray(slack, dtype=np.float64), 0.0)
    max_abs = float(np.max(d)) if d.size else 0.0
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    return max_abs, rel


def assert_close(name, got, ref, max_abs=MAX_ABS, rel_l2=REL_L2, bf16_out=True, slack=None):
    ma, rl = errors(got, ref, bf16_out, slack)
    raw = float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))))
    print(f"[parity] {name}: max_abs={ma:.3e} (raw {raw:.3e}) rel_l2={rl:.3e} "
          f"|ref|max={float(np.max(np.abs(ref))):.3e}")
    assert ma <= max_abs and rl <= rel_l2, f"{name}: max_abs={ma:.3e} (<= {max_abs}) rel_l2={rl:.3e} (<= {rel_l2})"
    return ma, rl


def dsink_bound(lse, sinks, o, do, hq):
    """Error bound of dsinks, from the arithmetic (fp32 output, no stated tolerance).

    dz_h = -sum_t exp(z_h - LSE_t) D_t with D_t = dO_t . O_t computed from the
    bf16-rounded O the forward returns: each O element carries a relative
    rounding error up to 2^-9, so |error| <= 2^-9 sum_t exp(z - LSE_t)
    sum_d |dO_td O_td| to first order; twice that plus 1e-4 is allowed.
    Arguments are the oracle's fp64 values in head layout: lse [P][B][hq][S],
    sinks [Hq], o/do [P][B][S][hq][D].
    """
    P = lse.shape[0]
    out = np.zeros(P * hq)
    for r in range(P):
        z = np.asarray(sinks[r * hq:(r + 1) * hq], np.float64)          # [hq]
        w = np.exp(z[None, :, None] - lse[r])                           # [B][hq][S]
        mag = np.abs(do[r] * o[r]).sum(-1).transpose(0, 2, 1)          # [B][hq][S]
        out[r * hq:(r + 1) * hq] = (w * mag).sum(axis=(0, 2))
    return 2.0 * 2.0 ** -9 * out + 1e-4


def device_inputs(w: W.Workload, device="cuda"):
    """Seeded shards on the device plus the same values as float64 for the oracle."""
    t = W.qkv_do_shards(w)
    pos = W.position_ids_shards(w)
    sk = W.sinks(w)
    dev = {n: x.to(device) for n, x in t.items()}
    dev["pos"] = torch.from_numpy(pos).to(device)
    dev["sinks"] = None if sk is None else sk.to(device)
    host = {n: W.bf16_to_f64(x) for n, x in t.items()}
    host["pos"] = pos
    host["sinks"] = None if sk is None else sk.double().numpy()
    return dev, host


def head_values(ua, name, r, j, heads_per_rank):
    """float64 [B*S][D] of local head j of rank r for output `name` ("o", "dq",
    "dk", "dv"), read from the head-layout buffer (explicit exchanges) or from
    the seq-layout output (fused exchanges)."""
    if not ua.fused:
        t = getattr(ua, name + "_head")                      # [P][B][S][hpr][D]
        return t[r].reshape(-1, heads_per_rank, t.shape[-1])[:, j].double().cpu().numpy()
    return seq_head_values(getattr(ua, name + "_seq"), r * heads_per_rank + j)


def seq_head_values(t, h):
    """float64 [B*S][D] of global head h of a seq-layout tensor [P][B][S/P][H][D]."""
    P, Bb, Sl, H, D = t.shape
    x = t.permute(1, 0, 2, 3, 4).reshape(Bb * P * Sl, H, D)  # token b*S + r'*Sl + s'
    return x[:, h].double().cpu().numpy()


def modes(w: W.Workload):
    """Exchange modes a workload can run: explicit always, fused when S/P % 128 == 0."""
    return [False] + ([True] if (w.S // w.P) % 128 == 0 else [])


def shape_of(w: W.Workload):
    from ulysses_sequence_long_gb300.pipeline import Shape
    return Shape(B=w.B, S=w.S, Hq=w.Hq, Hkv=w.Hkv, D=w.D, P=w.P, causal=w.causal, window_left=w.window_left)
