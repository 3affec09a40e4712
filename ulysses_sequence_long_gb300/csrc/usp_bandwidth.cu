// usp_bandwidth.cu — the HBM-bound kernels of the path:
//   * the emulated all-to-all (relayout between sequence shards and head
//     shards; huggingface/accelerate PR #4209, _gather_seq_scatter_heads and
//     _gather_heads_scatter_seq), one 16-byte vector per thread-iteration,
//     writes fully coalesced, reads in contiguous runs of (H/P)*D elements;
//   * the document-boundary scan over the gathered position_ids (same PR: the
//     per-shard cu_seq_lens_q/k are dropped and rebuilt from the gathered
//     positions), as count -> block scan -> scatter.
#include <cuda_runtime.h>
#include <stdint.h>

#include "usp_internal.h"
#include "usp_ptx.cuh"

namespace usp {

// ============================================================== relayout
//
// Sizes are counted in 16-byte vectors.  A "run" is the hpr*D elements one
// rank's block of heads occupies at one position: contiguous in both layouts
// (hpr = H/P heads per rank; when H < P each head is replicated on P/H ranks,
// hpr = 1, and rank r holds head r/(P/H)).
//   head-layout run index  hr = (r*B + b)*S + s              (rank r, row b, position s)
//   seq-layout  run index  sr = ((r'*B + b)*Sl + s')*R + r/rep  (s = r'*Sl + s', R = H/hpr runs per token)
struct RelayoutGeom {
  uint32_t n_vec;      // vectors in the destination tensor
  FastDiv run_vec;     // vectors per run
  FastDiv S, B, Sl, R, rep;
  uint32_t Sl_u, B_u, S_u, R_u, rep_u;
};

__device__ __forceinline__ uint32_t head_run_to_seq_run(const RelayoutGeom& g, uint32_t hr) {
  uint32_t rb = g.S.div(hr);
  uint32_t s = hr - rb * g.S_u;
  uint32_t r = g.B.div(rb);
  uint32_t b = rb - r * g.B_u;
  uint32_t rp = g.Sl.div(s);
  uint32_t sp = s - rp * g.Sl_u;
  return ((rp * g.B_u + b) * g.Sl_u + sp) * g.R_u + g.rep.div(r);
}

// Head-layout run of replica `rr` (0 <= rr < rep) of seq-layout run sr.
__device__ __forceinline__ uint32_t seq_run_to_head_run(const RelayoutGeom& g, uint32_t sr, uint32_t rr) {
  uint32_t t = g.R.div(sr);
  uint32_t r = (sr - t * g.R_u) * g.rep_u + rr;
  uint32_t t2 = g.Sl.div(t);
  uint32_t sp = t - t2 * g.Sl_u;
  uint32_t rp = g.B.div(t2);
  uint32_t b = t2 - rp * g.B_u;
  return (r * g.B_u + b) * g.S_u + rp * g.Sl_u + sp;
}

constexpr int kRelayoutThreads = 256;
constexpr int kRelayoutUnroll = 4;

// Destination-ordered: every thread-iteration writes consecutive vectors of
// the destination, so stores are fully coalesced; loads come from runs of at
// least 128 bytes in every configuration this path is used with.  Towards the
// head layout a replicated head is simply read by each of its replicas.
template <bool kToHead>
__device__ __forceinline__ void relayout_body(const int4* __restrict__ src, int4* __restrict__ dst,
                                              const RelayoutGeom& g, uint32_t first, uint32_t stride) {
  for (uint32_t base = first; base < g.n_vec; base += stride * kRelayoutUnroll) {
    int4 val[kRelayoutUnroll];
    uint32_t idx[kRelayoutUnroll];
#pragma unroll
    for (int u = 0; u < kRelayoutUnroll; ++u) {
      uint32_t v = base + u * stride;
      idx[u] = v;
      if (v < g.n_vec) {
        uint32_t run = g.run_vec.div(v);
        uint32_t k = v - run * g.run_vec.d;
        uint32_t srun = kToHead ? head_run_to_seq_run(g, run) : seq_run_to_head_run(g, run, 0);
        val[u] = __ldg(src + static_cast<size_t>(srun) * g.run_vec.d + k);
      }
    }
#pragma unroll
    for (int u = 0; u < kRelayoutUnroll; ++u)
      if (idx[u] < g.n_vec) __stcs(dst + idx[u], val[u]);
  }
}

template <bool kToHead>
__global__ void __launch_bounds__(kRelayoutThreads) relayout_kernel(const int4* __restrict__ src,
                                                                    int4* __restrict__ dst, RelayoutGeom g) {
  relayout_body<kToHead>(src, dst, g, blockIdx.x * blockDim.x + threadIdx.x, gridDim.x * blockDim.x);
}

// Head layout -> seq layout when heads are replicated (bf16 only): the
// exchange back sums the rep replicas of every head (the adjoint of the
// replication), in fp32 in replica order, rounded once to bf16.
__global__ void __launch_bounds__(kRelayoutThreads) relayout_reduce_kernel(const int4* __restrict__ src,
                                                                           int4* __restrict__ dst, RelayoutGeom g) {
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < g.n_vec; v += stride) {
    const uint32_t run = g.run_vec.div(v);
    const uint32_t k = v - run * g.run_vec.d;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (uint32_t rr = 0; rr < g.rep_u; ++rr) {
      const int4 x = __ldg(src + static_cast<size_t>(seq_run_to_head_run(g, run, rr)) * g.run_vec.d + k);
      const uint32_t w[4] = {static_cast<uint32_t>(x.x), static_cast<uint32_t>(x.y), static_cast<uint32_t>(x.z),
                             static_cast<uint32_t>(x.w)};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[2 * e] += bf16lo(w[e]);
        acc[2 * e + 1] += bf16hi(w[e]);
      }
    }
    int4 out;
    out.x = static_cast<int>(pack_bf16x2(acc[0], acc[1]));
    out.y = static_cast<int>(pack_bf16x2(acc[2], acc[3]));
    out.z = static_cast<int>(pack_bf16x2(acc[4], acc[5]));
    out.w = static_cast<int>(pack_bf16x2(acc[6], acc[7]));
    __stcs(dst + v, out);
  }
}

// q, k and v in one launch: the grid is split in proportion to their sizes.
struct Relayout3 {
  const int4* src[3];
  int4* dst[3];
  RelayoutGeom g[3];
  uint32_t block_end[3];  // exclusive prefix of blocks per tensor
};

__global__ void __launch_bounds__(kRelayoutThreads) relayout_qkv_kernel(Relayout3 a) {
  int t = blockIdx.x < a.block_end[0] ? 0 : (blockIdx.x < a.block_end[1] ? 1 : 2);
  uint32_t b0 = t == 0 ? 0 : a.block_end[t - 1];
  uint32_t nb = a.block_end[t] - b0;
  relayout_body<true>(a.src[t], a.dst[t], a.g[t], (blockIdx.x - b0) * blockDim.x + threadIdx.x,
                      nb * blockDim.x);
}

// Ps sequence shards, Ph head blocks: Ps = Ph = P for the Ulysses exchange;
// for the ring x Ulysses hybrid Ps = ring*ulysses shards and Ph = ulysses
// blocks, each block holding the whole sequence (the ring ranks' super-chunks
// end to end).  The shard of a position is s / (S/Ps) in both cases.
static RelayoutGeom make_geom(int B, int S, int H, int D, int Ps, int Ph, int eb, bool to_head) {
  RelayoutGeom g;
  const int P = Ph;
  const int hpr = H >= P ? H / P : 1, rep = H >= P ? 1 : P / H;
  uint64_t run_bytes = static_cast<uint64_t>(hpr) * D * eb;
  uint64_t seq_vec = static_cast<uint64_t>(B) * S * H * D * eb / 16;
  g.n_vec = static_cast<uint32_t>(to_head ? seq_vec * rep : seq_vec);
  g.run_vec = FastDiv(static_cast<uint32_t>(run_bytes / 16));
  g.S = FastDiv(S);
  g.B = FastDiv(B);
  g.Sl = FastDiv(S / Ps);
  g.R = FastDiv(H / hpr);
  g.rep = FastDiv(rep);
  g.Sl_u = S / Ps;
  g.B_u = B;
  g.S_u = S;
  g.R_u = H / hpr;
  g.rep_u = rep;
  return g;
}

static int relayout_grid(uint64_t n_vec) {
  uint64_t want = (n_vec + static_cast<uint64_t>(kRelayoutThreads) * kRelayoutUnroll - 1) /
                  (static_cast<uint64_t>(kRelayoutThreads) * kRelayoutUnroll);
  uint64_t cap = static_cast<uint64_t>(device_sm_count()) * (2048 / kRelayoutThreads) * 2;
  if (want > cap) want = cap;
  return static_cast<int>(want < 1 ? 1 : want);
}

int launch_relayout(const void* src, void* dst, int B, int S, int H, int D, int Ps, int Ph, int eb, bool to_head,
                    cudaStream_t st) {
  RelayoutGeom g = make_geom(B, S, H, D, Ps, Ph, eb, to_head);
  if (g.n_vec == 0) return USP_OK;
  int grid = relayout_grid(g.n_vec);
  if (!to_head && g.rep_u > 1)
    relayout_reduce_kernel<<<grid, kRelayoutThreads, 0, st>>>(static_cast<const int4*>(src), static_cast<int4*>(dst), g);
  else if (to_head)
    relayout_kernel<true><<<grid, kRelayoutThreads, 0, st>>>(static_cast<const int4*>(src), static_cast<int4*>(dst), g);
  else
    relayout_kernel<false><<<grid, kRelayoutThreads, 0, st>>>(static_cast<const int4*>(src), static_cast<int4*>(dst), g);
  return check_launch();
}

int launch_relayout_qkv(const void* const src[3], void* const dst[3], const int H[3], int B, int S, int D, int Ps,
                        int Ph, int eb, cudaStream_t st) {
  Relayout3 a;
  uint64_t total = 0, nv[3];
  for (int t = 0; t < 3; ++t) {
    a.src[t] = static_cast<const int4*>(src[t]);
    a.dst[t] = static_cast<int4*>(dst[t]);
    a.g[t] = make_geom(B, S, H[t], D, Ps, Ph, eb, true);
    nv[t] = a.g[t].n_vec;
    total += nv[t];
  }
  if (total == 0) return USP_OK;
  int grid = relayout_grid(total);
  uint32_t acc = 0;
  for (int t = 0; t < 3; ++t) {
    uint32_t nb = static_cast<uint32_t>((nv[t] * grid + total - 1) / total);
    if (nb < 1) nb = 1;
    acc += nb;
    a.block_end[t] = acc;
  }
  relayout_qkv_kernel<<<acc, kRelayoutThreads, 0, st>>>(a);
  return check_launch();
}

// ============================================================== cu_seqlens
//
// Gathered index g = b*S + s (s = r*Sl + s') reads pos[r][b][s'].  A document
// starts at g when s == 0 or the position there is 0.
constexpr int kScanThreads = 256;
constexpr int kScanItems = 16;                      // consecutive items per thread
constexpr int kScanChunk = kScanThreads * kScanItems;  // items per block
constexpr int kBig = 0x7FFFFFFF;

struct ScanGeom {
  int B, S, P, Sl, total;
};

__device__ __forceinline__ int load_pos(const int32_t* __restrict__ pos, const ScanGeom& g, int gi) {
  if (g.P == 1 || g.B == 1) return __ldg(pos + gi);  // the shards already sit in gathered order
  int b = gi / g.S, s = gi - b * g.S;
  int r = s / g.Sl, sp = s - r * g.Sl;
  return __ldg(pos + (static_cast<size_t>(r) * g.B + b) * g.Sl + sp);
}

// Flags of this thread's kScanItems consecutive items (bit i), and whether any position was negative.
__device__ __forceinline__ uint32_t thread_flags(const int32_t* __restrict__ pos, const ScanGeom& g, int first,
                                                 bool& negative) {
  uint32_t f = 0;
  negative = false;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    int gi = first + i;
    if (gi < g.total) {
      int p = load_pos(pos, g, gi);
      negative |= p < 0;
      int s = gi % g.S;
      if (p == 0 || s == 0) f |= 1u << i;
    }
  }
  return f;
}

// Block-wide exclusive sum (returned) and total (in *total) of one int per thread.
__device__ __forceinline__ int block_excl_sum(int x, int* total, int* sh) {
  int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh[w] = incl;
  __syncthreads();
  if (w == 0) {
    int v = lane < kScanThreads / 32 ? sh[lane] : 0;
    int vi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, vi, o);
      if (lane >= o) vi += y;
    }
    if (lane < kScanThreads / 32) sh[32 + lane] = vi - v;
    if (lane == kScanThreads / 32 - 1) sh[64] = vi;
  }
  __syncthreads();
  int r = sh[32 + w] + incl - x;
  *total = sh[64];
  __syncthreads();
  return r;
}

// Pass 1: per block, the number of document starts and the first start index.
__global__ void __launch_bounds__(kScanThreads) scan_count_kernel(const int32_t* __restrict__ pos, ScanGeom g,
                                                                  int32_t* __restrict__ counts,
                                                                  int32_t* __restrict__ firsts, int32_t* status) {
  __shared__ int sh[72];
  __shared__ int first_sh;
  int first = blockIdx.x * kScanChunk + threadIdx.x * kScanItems;
  bool neg;
  uint32_t f = thread_flags(pos, g, first, neg);
  if (neg) set_status(status, USP_ERR_BAD_POSITIONS);
  if (threadIdx.x == 0) first_sh = kBig;
  __syncthreads();
  if (f) atomicMin(&first_sh, first + __ffs(f) - 1);
  int total;
  block_excl_sum(__popc(f), &total, sh);
  if (threadIdx.x == 0) {
    counts[blockIdx.x] = total;
    firsts[blockIdx.x] = first_sh;
  }
}

// Pass 2 (one block): exclusive offsets of the blocks, the first start after
// each block, n_docs, cu[n_docs] = B*S, and max_len reset.
__global__ void __launch_bounds__(1024) scan_blocks_kernel(int nblk, const int32_t* __restrict__ counts,
                                                           const int32_t* __restrict__ firsts,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ next_after, int total_items,
                                                           int32_t* cu, int32_t* n_docs, int32_t* max_len) {
  __shared__ int sh_sum[1024];
  __shared__ int sh_min[1024];
  int per = (nblk + blockDim.x - 1) / blockDim.x;
  int b0 = threadIdx.x * per, b1 = min(nblk, b0 + per);
  int s = 0, mn = kBig;
  for (int b = b0; b < b1; ++b) s += counts[b];
  for (int b = b0; b < b1; ++b) mn = min(mn, firsts[b]);
  sh_sum[threadIdx.x] = s;
  sh_min[threadIdx.x] = mn;
  __syncthreads();
  // Hillis-Steele scans over 1024 thread partials: prefix sums, suffix minima.
  for (int o = 1; o < 1024; o <<= 1) {
    int a = threadIdx.x >= o ? sh_sum[threadIdx.x - o] : 0;
    int m = threadIdx.x + o < 1024 ? sh_min[threadIdx.x + o] : kBig;
    __syncthreads();
    sh_sum[threadIdx.x] += a;
    sh_min[threadIdx.x] = min(sh_min[threadIdx.x], m);
    __syncthreads();
  }
  int run = sh_sum[threadIdx.x] - s;                                  // exclusive
  int after = threadIdx.x + 1 < 1024 ? sh_min[threadIdx.x + 1] : kBig;  // first start beyond my blocks
  for (int b = b0; b < b1; ++b) {
    offsets[b] = run;
    run += counts[b];
  }
  for (int b = b1 - 1; b >= b0; --b) {
    next_after[b] = after == kBig ? total_items : after;
    after = min(after, firsts[b]);
  }
  if (threadIdx.x == 1023) {
    int n = sh_sum[1023];
    *n_docs = n;
    cu[n] = total_items;
    *max_len = 0;
  }
}

// Pass 3: scatter every document start to its slot; max document length.
__global__ void __launch_bounds__(kScanThreads) scan_scatter_kernel(const int32_t* __restrict__ pos, ScanGeom g,
                                                                    const int32_t* __restrict__ offsets,
                                                                    const int32_t* __restrict__ next_after,
                                                                    int32_t* __restrict__ cu, int32_t* max_len) {
  __shared__ int sh[72];
  __shared__ int nxt[kScanThreads];
  __shared__ int bmax;
  int first = blockIdx.x * kScanChunk + threadIdx.x * kScanItems;
  bool neg;
  uint32_t f = thread_flags(pos, g, first, neg);
  int total;
  int off = block_excl_sum(__popc(f), &total, sh) + offsets[blockIdx.x];
  // first start owned by each thread, then the first start after each thread
  nxt[threadIdx.x] = f ? first + __ffs(f) - 1 : kBig;
  if (threadIdx.x == 0) bmax = 0;
  __syncthreads();
  for (int o = 1; o < kScanThreads; o <<= 1) {
    int m = threadIdx.x + o < kScanThreads ? nxt[threadIdx.x + o] : kBig;
    __syncthreads();
    nxt[threadIdx.x] = min(nxt[threadIdx.x], m);
    __syncthreads();
  }
  int after = threadIdx.x + 1 < kScanThreads ? nxt[threadIdx.x + 1] : kBig;
  if (after == kBig) after = next_after[blockIdx.x];
  int local_max = 0;
  int prev = -1;
  for (int i = 0; i < kScanItems; ++i) {
    if (f & (1u << i)) {
      int gi = first + i;
      cu[off++] = gi;
      if (prev >= 0) local_max = max(local_max, gi - prev);
      prev = gi;
    }
  }
  if (prev >= 0) local_max = max(local_max, after - prev);
  if (local_max) atomicMax(&bmax, local_max);
  __syncthreads();
  if (threadIdx.x == 0 && bmax) atomicMax(max_len, bmax);
}

size_t cu_seqlens_ws_bytes(int B, int S) {
  size_t total = static_cast<size_t>(B) * S;
  size_t nblk = (total + kScanChunk - 1) / kScanChunk;
  if (nblk < 1) nblk = 1;
  return ((4 * nblk * sizeof(int32_t)) + 255) / 256 * 256;
}

int launch_cu_seqlens(const int32_t* pos, int B, int S, int P, int32_t* cu, int32_t* n_docs, int32_t* max_len,
                      int32_t* ws, int32_t* status, cudaStream_t st) {
  ScanGeom g{B, S, P, S / P, B * S};
  int nblk = (g.total + kScanChunk - 1) / kScanChunk;
  int32_t* counts = ws;
  int32_t* firsts = ws + nblk;
  int32_t* offsets = ws + 2 * nblk;
  int32_t* next_after = ws + 3 * nblk;
  scan_count_kernel<<<nblk, kScanThreads, 0, st>>>(pos, g, counts, firsts, status);
  scan_blocks_kernel<<<1, 1024, 0, st>>>(nblk, counts, firsts, offsets, next_after, g.total, cu, n_docs, max_len);
  scan_scatter_kernel<<<nblk, kScanThreads, 0, st>>>(pos, g, offsets, next_after, cu, max_len);
  return check_launch();
}

}  // namespace usp
