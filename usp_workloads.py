"""Seeded synthetic workloads for the Ulysses attention hot path.

This module only *makes inputs*: shapes, seeded N(0,1) tensors rounded once to
bf16, position_ids with a document-length mix, and per-head sink logits.  It
holds none of the method's arithmetic (no relayout, no document-boundary scan,
no attention), so both the fp64 oracle and the CUDA path can take their inputs
from it without sharing any computation.

Shapes follow the workloads named on the pages:

* the yunchang USP test tensor ``[batch=1, seq=4096, heads=12, head_dim=128]``
  in bf16 (feifeibear/long-context-attention issue #135, the test script);
* packed documents marked by position_ids that restart at 0 for each document
  ("padding-free collator", huggingface/accelerate PR #4209, the comment on
  stale ``cu_seq_lens_q/k``);
* GQA (ArcticTraining PR #45, "gqa works"), sliding windows and one sink logit
  per head (accelerate PR #4209, the gpt-oss and Cohere2/Gemma3 findings).

Layouts produced here are the *sequence-sharded* ones a rank holds before the
all-to-all: ``[P][B][S/P][H][D]`` for q/k/v/dO and ``[P][B][S/P]`` int32 for
position_ids, rank r holding the contiguous chunk ``[r*S/P, (r+1)*S/P)`` of
every row (the "basic" extraction in the yunchang test script).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    Hq: int
    Hkv: int
    D: int
    P: int
    causal: bool = True
    window_left: int = -1          # -1: no window; else query i sees keys j with i-j <= window_left
    sinks: bool = False            # one fp32 logit per (global) query head
    doc_lens: Optional[tuple] = None  # explicit document lengths for each row (None: see doc_mode)
    doc_mode: str = "single"       # "single" | "explicit" | "geometric"
    doc_mean: int = 4096           # mean length for doc_mode == "geometric"
    seed: int = 0
    ring: int = 1                  # ring degree of the ring x Ulysses hybrid (P = ring * ulysses)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def T(self) -> int:
        return self.B * self.S

    def describe(self) -> dict:
        d = dataclasses.asdict(self)
        d.pop("doc_lens")
        return d


# The five workloads: tiny packed, yunchang-shaped MHA, Llama-3-8B-shaped packed
# GQA, gpt-oss-shaped (window layer and full layer), and a 128K single document.
TINY = Workload("tiny_packed_s256", B=1, S=256, Hq=4, Hkv=2, D=64, P=2,
                doc_mode="explicit", doc_lens=(100, 90, 66))
MHA4K = Workload("mha_causal_s4096_h12_d128", B=1, S=4096, Hq=12, Hkv=12, D=128, P=4)
LLAMA32K = Workload("llama3_8b_gqa_packed_s32768", B=1, S=32768, Hq=32, Hkv=8, D=128, P=8,
                    doc_mode="geometric", doc_mean=4096)
GPTOSS_WIN = Workload("gpt_oss_window128_s16384", B=1, S=16384, Hq=64, Hkv=8, D=64, P=8,
                      window_left=127, sinks=True)
GPTOSS_FULL = Workload("gpt_oss_full_s16384", B=1, S=16384, Hq=64, Hkv=8, D=64, P=8,
                       window_left=-1, sinks=True)
LONG128K = Workload("long_context_s131072", B=1, S=131072, Hq=28, Hkv=4, D=128, P=4)

ALL = [TINY, MHA4K, LLAMA32K, GPTOSS_WIN, GPTOSS_FULL, LONG128K]
# A quarter-length Llama-shaped case for profiler captures: the same kernels and
# tile mix, inputs still larger than L2 (168 MB of q/k/v/dO), far fewer launches.
LLAMA8K_PROFILE = Workload("llama3_8b_gqa_packed_s8192", B=1, S=8192, Hq=32, Hkv=8, D=128, P=8,
                           doc_mode="geometric", doc_mean=4096, seed=1)
# kv-head replication (more ranks than key/value heads): the Llama-shaped
# packed case at sp size 16, each of the 8 key/value heads on 2 ranks.
LLAMA32K_P16 = Workload("llama3_8b_gqa_packed_s32768_p16", B=1, S=32768, Hq=32, Hkv=8, D=128, P=16,
                        doc_mode="geometric", doc_mean=4096)
# ring x Ulysses hybrid: the same Llama-shaped workload over 8 ranks as ring 2
# x ulysses 4 (the yunchang test's mesh shape with the degrees swapped).
LLAMA32K_RING2 = Workload("llama3_8b_gqa_packed_s32768_ring2x4", B=1, S=32768, Hq=32, Hkv=8, D=128, P=8,
                          ring=2, doc_mode="geometric", doc_mean=4096)
BY_NAME = {w.name: w for w in ALL + [LLAMA8K_PROFILE, LLAMA32K_P16, LLAMA32K_RING2]}


def document_lengths(w: Workload) -> List[List[int]]:
    """Per row of the batch, the lengths of the packed documents (summing to S)."""
    rows = []
    rng = np.random.Generator(np.random.PCG64(w.seed + 7919))
    for _ in range(w.B):
        if w.doc_mode == "single":
            lens = [w.S]
        elif w.doc_mode == "explicit":
            lens = list(w.doc_lens)
            assert sum(lens) == w.S, (lens, w.S)
        elif w.doc_mode == "geometric":
            # geometric on {1, 2, ...} with mean doc_mean; draw until the row is
            # full, then cut the last document at the row end.
            lens, tot = [], 0
            while tot < w.S:
                n = int(rng.geometric(1.0 / w.doc_mean))
                n = min(n, w.S - tot)
                lens.append(n)
                tot += n
        else:
            raise ValueError(w.doc_mode)
        rows.append(lens)
    return rows


def position_ids_gathered(w: Workload) -> np.ndarray:
    """int32 [B][S]: positions count 0,1,2,... inside each document."""
    out = np.empty((w.B, w.S), dtype=np.int32)
    for b, lens in enumerate(document_lengths(w)):
        out[b] = np.concatenate([np.arange(n, dtype=np.int32) for n in lens])
    return out


def shard_sequence(x: np.ndarray, P: int) -> np.ndarray:
    """[B][S][...] -> [P][B][S/P][...]: rank r keeps the r-th contiguous chunk."""
    B, S = x.shape[:2]
    assert S % P == 0
    xs = x.reshape((B, P, S // P) + x.shape[2:])
    return np.ascontiguousarray(np.moveaxis(xs, 1, 0))


def position_ids_shards(w: Workload) -> np.ndarray:
    """int32 [P][B][S/P]: each rank's shard of position_ids."""
    return shard_sequence(position_ids_gathered(w), w.P)


def _normal_bf16(shape, seed: int) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


_TENSOR_SEED = {"q": 11, "k": 23, "v": 37, "do": 41, "sinks": 53}


def qkv_do_shards(w: Workload, names=("q", "k", "v", "do")) -> dict:
    """bf16 tensors in sequence-shard layout [P][B][S/P][H][D], N(0,1) from the seed.

    The full [B][S][H][D] tensor is drawn first and then cut into contiguous
    sequence chunks, so the same bytes stand for the unsharded input too.
    """
    out = {}
    for n in names:
        H = w.Hq if n in ("q", "do") else w.Hkv
        full = _normal_bf16((w.B, w.S, H, w.D), w.seed * 1000 + _TENSOR_SEED[n])
        out[n] = full.view(w.B, w.P, w.S // w.P, H, w.D).transpose(0, 1).contiguous()
    return out


def sinks(w: Workload) -> Optional[torch.Tensor]:
    """fp32 [Hq] sink logits ~ N(0,1), or None when the workload has none."""
    if not w.sinks:
        return None
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed * 1000 + _TENSOR_SEED["sinks"])
    return torch.randn((w.Hq,), generator=g, dtype=torch.float32)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a bf16 tensor to a float64 numpy array."""
    return t.to(torch.float64).numpy()
