"""One rank of the multi-process Ulysses tests, run as a child process.

Every rank takes its sequence chunk of a seeded workload, runs the layer
forward and backward through ``UlyssesRankAttention`` over a gloo process
group (rendezvous from MASTER_ADDR/MASTER_PORT/RANK/WORLD_SIZE), and saves
what it computed to ``<out>.rank<r>.npz`` for the parent test to compare
with the oracle.

``--ops library``: the library's CUDA kernels on cuda:0 (several ranks may
share the one GPU: the collectives go through the host, so no kernel ever
waits for another rank).  ``--ops oracle``: a stand-in made of the fp64
oracle's per-rank functions on the CPU, which exercises the orchestration
(position gather, exchanges, sink slices, replica sums, dsinks gather) on
machines without a GPU.
"""
import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import usp_workloads as W  # noqa: E402
from ulysses_sequence_long_gb300.distributed import RankShape, UlyssesRankAttention  # noqa: E402


class OracleOps:
    """The local steps of a rank from the oracle (float64 CPU tensors)."""

    def __init__(self, shape: RankShape):
        import oracle
        self.o = oracle
        self.s = shape

    def pack_seq_to_head(self, x_local, H):
        return torch.from_numpy(self.o.a2a_pack_seq_to_head(x_local.numpy(), self.s.P, replicate=H < self.s.P))

    def unpack_seq_to_head(self, recv, H):
        return torch.from_numpy(self.o.a2a_unpack_seq_to_head(recv.numpy()))

    def pack_head_to_seq(self, x_head, H):
        return torch.from_numpy(self.o.a2a_pack_head_to_seq(x_head.numpy(), self.s.P))

    def unpack_head_to_seq(self, recv, H):
        return torch.from_numpy(self.o.a2a_unpack_head_to_seq(recv.numpy(), H))

    def boundaries(self, pos_all):
        self.cu, self.n, _ = self.o.cu_seqlens_from_position_ids(pos_all.numpy())

    def attention_fwd(self, q_h, k_h, v_h, sinks_r):
        s = self.s
        T = s.B * s.S
        O, L = self.o.attention_fwd(q_h.numpy().reshape(T, s.hq, s.D), k_h.numpy().reshape(T, s.hk, s.D),
                                    v_h.numpy().reshape(T, s.hk, s.D), self.cu, s.causal, s.window_left, None,
                                    None if sinks_r is None else sinks_r.numpy())
        return (torch.from_numpy(O.reshape(s.B, s.S, s.hq, s.D)),
                torch.from_numpy(L.reshape(s.hq, s.B, s.S).transpose(1, 0, 2).copy()).unsqueeze(0))

    def attention_bwd(self, q_h, k_h, v_h, o_h, lse, do_h, sinks_r):
        s = self.s
        T = s.B * s.S
        lse_r = lse[0].numpy().transpose(1, 0, 2).reshape(s.hq, T)
        dq, dk, dv, dz = self.o.attention_bwd(
            q_h.numpy().reshape(T, s.hq, s.D), k_h.numpy().reshape(T, s.hk, s.D), v_h.numpy().reshape(T, s.hk, s.D),
            o_h.numpy().reshape(T, s.hq, s.D), lse_r, do_h.numpy().reshape(T, s.hq, s.D), self.cu, s.causal,
            s.window_left, None, None if sinks_r is None else sinks_r.numpy())
        return (torch.from_numpy(dq.reshape(s.B, s.S, s.hq, s.D)), torch.from_numpy(dk.reshape(s.B, s.S, s.hk, s.D)),
                torch.from_numpy(dv.reshape(s.B, s.S, s.hk, s.D)), None if dz is None else torch.from_numpy(dz))

    def read_status(self) -> int:
        return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--ops", choices=["library", "oracle"], required=True)
    ap.add_argument("--workload", required=True, help="JSON of a usp_workloads.Workload")
    ap.add_argument("--out", required=True)
    args = ap.parse_args()
    rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
    wd = json.loads(args.workload)
    if wd.get("doc_lens") is not None:
        wd["doc_lens"] = tuple(wd["doc_lens"])
    w = W.Workload(**wd)
    assert w.P == world
    dist.init_process_group("gloo", rank=rank, world_size=world)
    shape = RankShape(w.B, w.S, w.Hq, w.Hkv, w.D, w.P, w.causal, w.window_left)
    t = W.qkv_do_shards(w)
    pos = torch.from_numpy(np.ascontiguousarray(W.position_ids_shards(w)[rank]))
    sk = W.sinks(w)
    if args.ops == "oracle":
        ua = UlyssesRankAttention(shape, ops=OracleOps(shape))
        x = {n: torch.from_numpy(W.bf16_to_f64(t[n][rank])) for n in t}
        sinks = None if sk is None else sk.double()
    else:
        torch.cuda.set_device(0)
        ua = UlyssesRankAttention(shape, device="cuda:0")
        x = {n: t[n][rank].contiguous().cuda() for n in t}
        pos = pos.cuda()
        sinks = None if sk is None else sk.cuda()
    o = ua.forward(x["q"], x["k"], x["v"], pos, sinks)
    dq, dk, dv, dz = ua.backward(x["do"], sinks)
    if args.ops == "library":
        torch.cuda.synchronize()
    q_h, k_h, v_h, o_h, lse = ua._saved

    def f64(a):
        return None if a is None else a.detach().double().cpu().numpy()

    out = dict(o=f64(o), dq=f64(dq), dk=f64(dk), dv=f64(dv), lse=f64(lse), q_h=f64(q_h), k_h=f64(k_h),
               v_h=f64(v_h), status=np.array([ua.ops.read_status()]))
    if dz is not None:
        out["dsinks"] = f64(dz)
    np.savez(f"{args.out}.rank{rank}.npz", **out)
    dist.barrier()
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
