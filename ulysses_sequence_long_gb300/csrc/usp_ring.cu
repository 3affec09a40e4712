// usp_ring.cu — the combination steps of the ring x Ulysses hybrid
// (feifeibear/long-context-attention issue #135: a (ring, ulysses) device mesh
// whose ring dimension passes key/value super-chunks from rank to rank):
//   * forward: after each ring step the rank's running output and log-sum-exp
//     absorb the step's block result, O = e^(L1-L) O1 + e^(L2-L) O2 with
//     L = log(e^L1 + e^L2); after the last step the head's sink logit joins
//     once, and O is rounded to bf16;
//   * backward: each step's bf16 dQ/dK/dV block gradients are summed in fp32
//     (dQ stays with its rank, dK/dV travel with their super-chunk; on one
//     device both are a sum at the element's own address), rounded once.
// Both are HBM-bound elementwise passes: one thread handles 8 consecutive
// elements (16 bytes of bf16, 32 of fp32).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "usp_internal.h"
#include "usp_ptx.cuh"

namespace usp {
namespace ring {

constexpr int kThreads = 256;

__device__ __forceinline__ float logaddexp(float a, float b) {
  const float m = fmaxf(a, b);
  if (m == -INFINITY) return -INFINITY;
  return m + log1pf(expf(-fabsf(a - b)));
}

__device__ __forceinline__ void unpack8(const uint4 x, float f[8]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = bf16lo(w[e]);
    f[2 * e + 1] = bf16hi(w[e]);
  }
}

__device__ __forceinline__ uint4 pack8(const float f[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

struct MergeGeom {
  int BS, S, B, hq, vpr;  // vpr: 8-element vectors per row (D/8)
  uint32_t n_vec;         // vectors in the whole tensor
  int seq, Sl, Hq;        // seq-layout [Ps][B][Sl][Hq][D] (shard length Sl) instead of head layout
};

// Row (rank r, token t, local head j) of the head layout, or (shard, row b,
// position, global head r*hq + j) of the sequence shards; its LSE sits at
// [r][b][j][s] of the [P][B][hq][S] statistics.  The lanes of one row are in
// one warp (vpr divides 32), so the __syncwarp orders every lane's read of
// the running LSE before the row's first lane overwrites it.
__global__ void __launch_bounds__(kThreads) fwd_merge_kernel(const uint4* __restrict__ o_step,
                                                             const float* __restrict__ lse_step, float* o_acc,
                                                             float* lse_acc, uint4* __restrict__ o_out,
                                                             float* __restrict__ lse_out,
                                                             const float* __restrict__ sinks, MergeGeom g,
                                                             int flags) {
  const uint32_t stride = gridDim.x * blockDim.x;
  const uint32_t n_pad = (g.n_vec + 31u) & ~31u;
  for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < n_pad; v += stride) {
    const bool act = v < g.n_vec;
    const uint32_t row = v / g.vpr, e8 = v - row * g.vpr;
    uint32_t r, j, b, s;
    if (!g.seq) {  // head layout: row = (r, t, j)
      j = row % g.hq;
      const uint32_t rt = row / g.hq;
      r = rt / g.BS;
      const uint32_t t = rt - r * g.BS;
      b = t / g.S;
      s = t - b * g.S;
    } else {       // seq layout: row = (shard, b, position in shard, global head)
      const uint32_t h = row % g.Hq, tok = row / g.Hq;
      const uint32_t bl = static_cast<uint32_t>(g.B) * g.Sl, rp = tok / bl, rem = tok - rp * bl;
      b = rem / g.Sl;
      s = rp * g.Sl + (rem - b * g.Sl);
      r = h / g.hq;
      j = h - r * g.hq;
    }
    const size_t li = ((static_cast<size_t>(r) * g.B + b) * g.hq + j) * g.S + s;
    float la = -INFINITY, ls = -INFINITY, oa[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, os[8];
    if (act) {
      ls = __ldg(lse_step + li);
      unpack8(__ldg(o_step + v), os);
      if (!(flags & USP_RING_FIRST)) {
        la = lse_acc[li];
        const float4 a0 = reinterpret_cast<const float4*>(o_acc)[2 * static_cast<size_t>(v)];
        const float4 a1 = reinterpret_cast<const float4*>(o_acc)[2 * static_cast<size_t>(v) + 1];
        oa[0] = a0.x; oa[1] = a0.y; oa[2] = a0.z; oa[3] = a0.w;
        oa[4] = a1.x; oa[5] = a1.y; oa[6] = a1.z; oa[7] = a1.w;
      }
    }
    __syncwarp();
    if (!act) continue;
    float L = logaddexp(la, ls);
    const float wa = L == -INFINITY ? 0.f : expf(la - L);
    const float ws = L == -INFINITY ? 0.f : expf(ls - L);
    float o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = wa * oa[e] + ws * os[e];
    if (flags & USP_RING_LAST) {
      if (sinks != nullptr) {  // the sink logit joins the softmax once, with no value
        const float z = __ldg(sinks + r * g.hq + j);
        const float L2 = logaddexp(L, z);
        const float w = L == -INFINITY ? 0.f : expf(L - L2);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] *= w;
        L = L2;
      }
      o_out[v] = pack8(o);
      if (e8 == 0) lse_out[li] = L;
    } else {
      reinterpret_cast<float4*>(o_acc)[2 * static_cast<size_t>(v)] = make_float4(o[0], o[1], o[2], o[3]);
      reinterpret_cast<float4*>(o_acc)[2 * static_cast<size_t>(v) + 1] = make_float4(o[4], o[5], o[6], o[7]);
      if (e8 == 0) lse_acc[li] = L;
    }
  }
}

__global__ void __launch_bounds__(kThreads) grad_accumulate_kernel(const uint4* __restrict__ g_step,
                                                                   float4* __restrict__ g_acc,
                                                                   uint4* __restrict__ g_out, uint32_t n_vec,
                                                                   int flags) {
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < n_vec; v += stride) {
    float f[8];
    unpack8(__ldg(g_step + v), f);
    if (!(flags & USP_RING_FIRST)) {
      const float4 a0 = g_acc[2 * static_cast<size_t>(v)], a1 = g_acc[2 * static_cast<size_t>(v) + 1];
      f[0] += a0.x; f[1] += a0.y; f[2] += a0.z; f[3] += a0.w;
      f[4] += a1.x; f[5] += a1.y; f[6] += a1.z; f[7] += a1.w;
    }
    if (flags & USP_RING_LAST) {
      __stcs(g_out + v, pack8(f));
    } else {
      g_acc[2 * static_cast<size_t>(v)] = make_float4(f[0], f[1], f[2], f[3]);
      g_acc[2 * static_cast<size_t>(v) + 1] = make_float4(f[4], f[5], f[6], f[7]);
    }
  }
}

static int grid_for(uint64_t n_vec) {
  uint64_t want = (n_vec + kThreads - 1) / kThreads;
  const uint64_t cap = static_cast<uint64_t>(device_sm_count()) * (2048 / kThreads) * 2;
  if (want > cap) want = cap;
  return static_cast<int>(want < 1 ? 1 : want);
}

}  // namespace ring

int launch_ring_fwd_merge(const usp_attn_params& p, const void* o_step, const float* lse_step, float* o_acc,
                          float* lse_acc, void* o, float* lse, int flags, cudaStream_t st) {
  ring::MergeGeom g;
  g.BS = p.B * p.S;
  g.S = p.S;
  g.B = p.B;
  g.hq = p.Hq / p.P;
  g.vpr = p.D / 8;
  g.n_vec = static_cast<uint32_t>(static_cast<uint64_t>(p.P) * g.BS * g.hq * g.vpr);
  const int ring = p.ring > 1 ? p.ring : 1;
  g.seq = p.io_layout == USP_IO_SEQ ? 1 : 0;
  g.Sl = p.S / (p.P * ring);
  g.Hq = p.Hq;
  if (g.n_vec == 0) return USP_OK;
  ring::fwd_merge_kernel<<<ring::grid_for(g.n_vec), ring::kThreads, 0, st>>>(
      static_cast<const uint4*>(o_step), lse_step, o_acc, lse_acc, static_cast<uint4*>(o), lse, p.sinks, g, flags);
  return check_launch();
}

int launch_ring_grad_accumulate(const void* g_step, float* g_acc, void* g_out, size_t n, int flags,
                                cudaStream_t st) {
  const uint32_t n_vec = static_cast<uint32_t>(n / 8);
  if (n_vec == 0) return USP_OK;
  ring::grad_accumulate_kernel<<<ring::grid_for(n_vec), ring::kThreads, 0, st>>>(
      static_cast<const uint4*>(g_step), reinterpret_cast<float4*>(g_acc), static_cast<uint4*>(g_out), n_vec, flags);
  return check_launch();
}

}  // namespace usp
