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


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in the GPU output"
    d = got - ref
    max_abs = float(np.max(np.abs(d))) if d.size else 0.0
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30))
    return max_abs, rel


def assert_close(name, got, ref, max_abs=MAX_ABS, rel_l2=REL_L2):
    ma, rl = errors(got, ref)
    print(f"[parity] {name}: max_abs={ma:.3e} rel_l2={rl:.3e} |ref|max={float(np.max(np.abs(ref))):.3e}")
    assert ma <= max_abs and rl <= rel_l2, f"{name}: max_abs={ma:.3e} (<= {max_abs}) rel_l2={rl:.3e} (<= {rel_l2})"
    return ma, rl


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


def shape_of(w: W.Workload):
    from ulysses_sequence_long_gb300.pipeline import Shape
    return Shape(B=w.B, S=w.S, Hq=w.Hq, Hkv=w.Hkv, D=w.D, P=w.P, causal=w.causal, window_left=w.window_left)
