// usp_attn_common.cuh — pieces shared by the forward and backward attention
// kernels: kernel parameters, document lookup in cu_seqlens, the visibility
// rule, the validity check of cu_seqlens and the tensor-map encoder.
//
// Visibility (the varlen mask over the gathered sequence): token t of document
// [a, b) sees key u when a <= u < b, u <= t if causal, and t - u <= window_left
// (also u - t <= window_left when not causal) if window_left >= 0.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/usp.h"
#include "usp_ptx.cuh"

namespace usp {

constexpr int kBM = 128;  // query rows per tile (TMEM lanes)
constexpr int kBN = 128;  // keys per tile

struct AttnArgs {
  int BS;           // tokens per rank: B*S
  int S;            // row length
  int B, P, hq, hk, G;  // hk: key/value heads per rank (1 when Hkv < P: replicated); G = hq / hk
  int Hq, Hkv;          // global head counts
  int causal, window_left;
  float scale;       // softmax scale
  float scale_log2;  // softmax scale * log2(e)
  const int32_t* cu;
  const int32_t* n_docs;
  const float* sinks;  // global [Hq] or null
  int32_t* status;
  int seq_io;     // 1: inputs and outputs in seq-layout [Ps][B][S/Ps][H][D] (exchanges fused)
  int kv_seq_io;  // k and v in seq-layout too (0 with USP_IO_SEQ_KV_HEAD: k, v in head layout)
  int Sl;      // shard length S/Ps; Ps = P sequence shards, P*ring for the ring x Ulysses hybrid
  int ring, ring_step, C;  // ring x Ulysses: ring degree (1: none), step, super-chunk length S/ring
  // backward head group: key/value heads [kvh0, kvh0 + n_kvh) and their query
  // heads [hq0, hq0 + n_qh) (all heads unless a group was asked for)
  int kvh0, n_kvh, hq0, n_qh;
};

// Ring x Ulysses: at ring step `ring_step` the rows of super-chunk a (of
// C = S/ring positions) see only the keys of super-chunk (a - ring_step) mod
// ring, the key/value block their ring rank holds at that step.  Key window
// [k0, k1) of rank-local token t, and the query window [q0, q1) of key u.
__device__ __forceinline__ void ring_key_window(const AttnArgs& p, int t, int& k0, int& k1) {
  const int b = t / p.S, s = t - b * p.S;
  const int kc = (s / p.C + p.ring - p.ring_step) % p.ring;
  k0 = b * p.S + kc * p.C;
  k1 = k0 + p.C;
}

__device__ __forceinline__ void ring_query_window(const AttnArgs& p, int u, int& q0, int& q1) {
  const int b = u / p.S, s = u - b * p.S;
  const int qc = (s / p.C + p.ring_step) % p.ring;
  q0 = b * p.S + qc * p.C;
  q1 = q0 + p.C;
}

// A head as the kernels address it: rank r and local index j in the
// head-layout [P][B][S][hpr][D], global index g in the seq-layout
// [P][B][S/P][H][D].
struct HeadRef {
  int r, j, g;
};

__device__ __forceinline__ HeadRef q_head_ref(const AttnArgs& p, int r, int j) { return {r, j, r * p.hq + j}; }
// Local key/value head kl of rank r: global head r*Hkv/P + kl (with Hkv < P the
// P/Hkv ranks r*Hkv/P == h all hold a replica of head h).
__device__ __forceinline__ HeadRef kv_head_ref(const AttnArgs& p, int r, int kl) {
  return {r, kl, (r * p.Hkv) / p.P + kl};
}

// Element offset of the D-vector of head h at rank-local token t = b*S + s in
// either layout (hpr heads per rank in head-layout, H heads in seq-layout):
//   head-layout  ((r*B*S + t)*hpr + j)*D
//   seq-layout   (((r'*B + b)*Sl + s')*H + g)*D,   s = r'*Sl + s'
__device__ __forceinline__ size_t row_offset(const AttnArgs& p, HeadRef h, int hpr, int H, int t, int D) {
  if (!p.seq_io) return ((static_cast<size_t>(h.r) * p.BS + t) * hpr + h.j) * D;
  const int b = t / p.S, s = t - b * p.S;
  const int rp = s / p.Sl, sp = s - rp * p.Sl;
  return ((static_cast<size_t>(rp * p.B + b) * p.Sl + sp) * H + h.g) * D;
}

// TMA load of `rows` tokens starting at rank-local token t (64 columns of the
// D-vectors starting at column c64*64) of head h, from either layout's tensor
// map.  In seq-layout the rows must lie in one shard of one row of the batch
// (the kernels align tiles to make sure).
__device__ __forceinline__ void tma_load_rows(void* dst, const CUtensorMap* m, uint64_t* bar, const AttnArgs& p,
                                              int c64, HeadRef h, int t, bool seq) {
  if (!seq) {
    tma_load_4d(dst, m, bar, c64 * 64, h.j, t, h.r);
  } else {
    const int b = t / p.S, s = t - b * p.S;
    const int rp = s / p.Sl, sp = s - rp * p.Sl;
    tma_load_5d(dst, m, bar, c64 * 64, h.g, sp, b, rp);
  }
}

__device__ __forceinline__ void tma_load_rows(void* dst, const CUtensorMap* m, uint64_t* bar, const AttnArgs& p,
                                              int c64, HeadRef h, int t) {
  tma_load_rows(dst, m, bar, p, c64, h, t, p.seq_io != 0);
}

// TMA store of a tile staged in shared memory (fenced by the caller) to the
// rows starting at rank-local token t of head h, same addressing as the loads;
// rows past the tensor's end are dropped by the copy.
__device__ __forceinline__ void tma_store_rows(const CUtensorMap* m, const void* src, const AttnArgs& p, int c64,
                                               HeadRef h, int t) {
  if (!p.seq_io) {
    tma_store_4d(m, src, c64 * 64, h.j, t, h.r);
  } else {
    const int b = t / p.S, s = t - b * p.S;
    const int rp = s / p.Sl, sp = s - rp * p.Sl;
    tma_store_5d(m, src, c64 * 64, h.g, sp, b, rp);
  }
}

// Document index d with cu[d] <= t < cu[d+1] (cu assumed valid, n >= 1).
__device__ __forceinline__ int find_doc(const int32_t* __restrict__ cu, int n, int t) {
  int lo = 0, hi = n;  // invariant: cu[lo] <= t < cu[hi]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid;
  }
  return lo;
}

// [start, end) of the document holding token t, clamped so that a malformed
// cu_seqlens (already reported) can never send an index out of [0, BS).
__device__ __forceinline__ void doc_bounds(const int32_t* __restrict__ cu, int n, int BS, int t, int& a, int& b) {
  int d = find_doc(cu, n, t);
  a = __ldg(cu + d);
  b = __ldg(cu + d + 1);
  a = max(0, min(a, t));
  b = min(BS, max(b, t + 1));
}

__device__ __forceinline__ bool visible(int t, int u, int a, int b, int causal, int wl) {
  bool v = (u >= a) && (u < b);
  if (causal) v = v && (u <= t);
  if (wl >= 0) v = v && (t - u <= wl) && (causal || u - t <= wl);
  return v;
}

// The same rule seen from the key: query t sees key u of document [a, b) when
// t lies in that document and the causal/window conditions hold.
__device__ __forceinline__ bool visible_from_key(int t, int u, int a, int b, int causal, int wl) {
  bool v = (t >= a) && (t < b);
  if (causal) v = v && (u <= t);
  if (wl >= 0) v = v && (t - u <= wl) && (causal || u - t <= wl);
  return v;
}

// The visibility rule as one interval: the keys row t of document [a, b)
// sees are exactly [vlo, vhi] (empty when vlo > vhi), so a mask costs two
// compares per element.
__device__ __forceinline__ void visible_keys(int t, int a, int b, int causal, int wl, bool ok, int& vlo, int& vhi) {
  vlo = a;
  vhi = b - 1;
  if (causal) vhi = min(vhi, t);
  if (wl >= 0) {
    vlo = max(vlo, t - wl);
    if (!causal) vhi = min(vhi, t + wl);
  }
  if (!ok) {
    vlo = 1;
    vhi = 0;
  }
}

// The rows [vlo, vhi] that see key u, when [a, b) is the key's document.
__device__ __forceinline__ void visible_rows(int u, int a, int b, int causal, int wl, bool ok, int& vlo, int& vhi) {
  vlo = a;
  vhi = b - 1;
  if (causal) vlo = max(vlo, u);
  if (wl >= 0) {
    vhi = min(vhi, u + wl);
    if (!causal) vlo = max(vlo, u - wl);
  }
  if (!ok) {
    vlo = 1;
    vhi = 0;
  }
}

// First and one-past-last key any of the rows [t_first, t_last] may see.
__device__ __forceinline__ void key_range(const AttnArgs& p, int n, int t_first, int t_last, int& lo, int& hi) {
  int a0, b0, a1, b1;
  doc_bounds(p.cu, n, p.BS, t_first, a0, b0);
  doc_bounds(p.cu, n, p.BS, t_last, a1, b1);
  lo = a0;
  hi = p.causal ? t_last + 1 : b1;
  if (p.window_left >= 0) {
    lo = max(lo, t_first - p.window_left);
    if (!p.causal) hi = min(hi, t_last + p.window_left + 1);
  }
}

// First and one-past-last query row that may see any of the keys [u_first, u_last].
__device__ __forceinline__ void query_range(const AttnArgs& p, int n, int u_first, int u_last, int& lo, int& hi) {
  int a0, b0, a1, b1;
  doc_bounds(p.cu, n, p.BS, u_first, a0, b0);
  doc_bounds(p.cu, n, p.BS, u_last, a1, b1);
  lo = p.causal ? u_first : a0;
  hi = b1;
  if (p.window_left >= 0) {
    hi = min(hi, u_last + p.window_left + 1);
    if (!p.causal) lo = max(lo, u_first - p.window_left);
  }
}

// Cheap per-CTA check of cu_seqlens: returns n_docs, or 0 (after recording
// USP_ERR_BAD_SEQLENS) when it cannot describe the gathered sequence.  Block 0
// also checks that every document is non-empty.
__device__ __forceinline__ int checked_docs(const AttnArgs& p) {
  int n = __ldg(p.n_docs);
  bool ok = n >= 1 && n <= p.BS;
  if (ok) ok = __ldg(p.cu) == 0 && __ldg(p.cu + n) == p.BS;
  if (!ok) {
    if (threadIdx.x == 0) set_status(p.status, USP_ERR_BAD_SEQLENS);
    return 0;
  }
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    for (int d = threadIdx.x; d < n; d += blockDim.x)
      if (__ldg(p.cu + d + 1) <= __ldg(p.cu + d)) set_status(p.status, USP_ERR_BAD_SEQLENS);
  }
  return n;
}

}  // namespace usp

// ------------------------------------------------------------------ host side
namespace usp {

// Tensor map of a head-layout bf16 tensor [P][BS][H][D]: dims {D, H, BS, P},
// box {64, 1, rows, 1}, 128-byte swizzle (one 128-byte row per token).
int make_head_tmap(CUtensorMap* m, const void* base, int P, int BS, int H, int D, int box_rows);
int make_seq_tmap(CUtensorMap* m, const void* base, int P, int B, int Sl, int H, int D, int box_rows);

// The map for either layout: head-layout (hpr heads per rank) or seq-layout (H heads).
inline int make_rows_tmap(CUtensorMap* m, const void* base, const AttnArgs& a, int hpr, int H, int D, int box_rows,
                          bool seq) {
  // seq-layout: P*ring shards of Sl tokens (the hybrid's ring groups hold P shards each)
  return seq ? make_seq_tmap(m, base, a.P * a.ring, a.B, a.Sl, H, D, box_rows)
             : make_head_tmap(m, base, a.P, a.BS, hpr, D, box_rows);
}
inline int make_rows_tmap(CUtensorMap* m, const void* base, const AttnArgs& a, int hpr, int H, int D, int box_rows) {
  return make_rows_tmap(m, base, a, hpr, H, D, box_rows, a.seq_io != 0);
}

// Forward for short causal windows at D = 64 (usp_attn_fwd_window.cu): whether
// the shape qualifies, and the launch with the general forward's tensor maps.
bool fwd_window_fits(const AttnArgs& a, int D);
int run_fwd_window(const AttnArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, void* o,
                   float* lse, cudaStream_t st);

int make_ds_tmap(CUtensorMap* m, const void* base, long long n_blocks);
int make_ds_store_tmap(CUtensorMap* m, void* base, long long n_blocks);

// Tensor map of the backward's planar statistics, fp32 [P*hq][2][pitch]: dims
// {BS, 2, P*hq}, box {box_rows, 2, 1} (box_rows tokens of both planes of one
// head); the token coordinate of a load must be a multiple of 4.
int make_stats_tmap(CUtensorMap* m, const void* base, int BS, int pitch, int rows, int box_rows);

}  // namespace usp
