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

#include <algorithm>

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
//
// One pass over the positions.  The grid is persistent-sized (at most one
// 1024-thread block per SM); block k, in the order blocks start (a ticket,
// so that every block a block waits for is already running), owns the k-th
// contiguous range of the gathered sequence:
//   1. it streams its range (1024 consecutive positions per warp and step,
//      coalesced 16-byte loads), keeps the start flags as bits in shared
//      memory, and publishes its aggregate: number of starts and latest start;
//   2. it sums the aggregates of all blocks before it (32 at a time, one
//      warp) for its prefix: starts before it and the latest start before it.
//      Every aggregate is published after one pass over one range, so no
//      block waits on a chain of other blocks' prefixes;
//   3. every thread takes a contiguous run of the flag words, a block-wide
//      scan gives each its first output slot and the start before its run,
//      and it writes its starts into cu_seqlens.  A document's length is
//      taken where it ends (the next start, or B*S after the last start).
// Flags beyond the shared-memory budget (ranges longer than kScanSmemWords *
// 32 positions) are recomputed from the positions in step 3.  With several
// blocks a small kernel before it resets the block states; a sequence of at
// most one block's range (every workload here) takes the one launch alone.
constexpr int kScanThreads = 1024;
constexpr int kScanItems = 32;                                 // positions per thread and step: one flag word
constexpr int kScanStep = kScanThreads * kScanItems;           // positions per block and step
constexpr int kScanSmemWords = 56 * 1024;                      // 224 KB of flag words
static_assert(kScanChunk % kScanStep == 0, "ranges are whole steps");

struct ScanGeom {
  int B, S, P, Sl, total;
  int nblk;   // blocks in the grid (1: no ticket, no block states, no reset kernel)
  int range;  // positions per block (a multiple of kScanStep)
  int vec;    // 1: each thread's 32 positions are one aligned, contiguous run
};

// Per-block state, one 64-bit word: flag (2 bits: 0 nothing yet, 1 the
// block's aggregate), starts counted (31 bits) and latest start + 1 (31 bits,
// 0 = none).  B*S < 2^31 - 1 keeps both in range.
__device__ __forceinline__ uint64_t scan_state(uint32_t flag, uint32_t count, int last) {
  return (static_cast<uint64_t>(flag) << 62) | (static_cast<uint64_t>(count & 0x7FFFFFFFu) << 31) |
         static_cast<uint64_t>(static_cast<uint32_t>(last + 1) & 0x7FFFFFFFu);
}
__device__ __forceinline__ uint32_t state_flag(uint64_t s) { return static_cast<uint32_t>(s >> 62); }
__device__ __forceinline__ uint32_t state_count(uint64_t s) { return static_cast<uint32_t>(s >> 31) & 0x7FFFFFFFu; }
__device__ __forceinline__ int state_last(uint64_t s) { return static_cast<int>(s & 0x7FFFFFFFu) - 1; }

// A state word carries everything a reader needs (no other data is published
// with it), so relaxed gpu-scope accesses suffice.
__device__ __forceinline__ void st_state(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_state(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Workspace: [0] ticket counter, then (from byte 256) one state per block.
struct ScanWs {
  uint32_t* ticket;
  uint64_t* state;
};

__device__ __forceinline__ int load_pos(const int32_t* __restrict__ pos, const ScanGeom& g, int gi) {
  if (g.P == 1 || g.B == 1) return __ldg(pos + gi);  // the shards already sit in gathered order
  int b = gi / g.S, s = gi - b * g.S;
  int r = s / g.Sl, sp = s - r * g.Sl;
  return __ldg(pos + (static_cast<size_t>(r) * g.B + b) * g.Sl + sp);
}

// This thread's kScanItems positions starting at gathered index `first`:
// start flags (bit i) and whether any position was negative.
__device__ __forceinline__ uint32_t thread_flags(const int32_t* __restrict__ pos, const ScanGeom& g, int first,
                                                 bool& negative) {
  int v[kScanItems];
  if (g.vec && first + kScanItems <= g.total) {
    // 32 consecutive positions of one shard row: eight 16-byte loads
    size_t at = static_cast<size_t>(first);
    if (g.P != 1 && g.B != 1) {
      const int b = first / g.S, s = first - b * g.S, r = s / g.Sl;
      at = (static_cast<size_t>(r) * g.B + b) * g.Sl + (s - r * g.Sl);
    }
    const int4* p4 = reinterpret_cast<const int4*>(pos + at);
#pragma unroll
    for (int k = 0; k < kScanItems / 4; ++k) {
      const int4 x = __ldg(p4 + k);
      v[4 * k] = x.x;
      v[4 * k + 1] = x.y;
      v[4 * k + 2] = x.z;
      v[4 * k + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) v[i] = first + i < g.total ? load_pos(pos, g, first + i) : 1;
  }
  // row starts inside [first, first + kScanItems): one division per thread
  const int rem = first % g.S;
  long long next_row = rem == 0 ? first : static_cast<long long>(first) + (g.S - rem);
  uint32_t f = 0;
  negative = false;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    const int gi = first + i;
    const bool in = gi < g.total;
    negative |= in && v[i] < 0;
    const bool row = gi == next_row;
    if (row) next_row += g.S;
    if (in && (v[i] == 0 || row)) f |= 1u << i;
  }
  return f;
}

// Flags of the 1024 positions [base, base + 1024) for one warp, loaded
// coalesced: at step k every lane reads the four positions base + 128k + 4L
// (one 16-byte vector per lane when `vec`, else four scalar loads).  The
// 32-position flag word w = 4k + L/8 is assembled from eight lanes' nibbles
// by a segmented OR over shuffles; lane L ends up holding word (L % 8) * 4 +
// L / 8 (returned, with that word's index in *wi).
__device__ __forceinline__ uint32_t warp_flags(const int32_t* __restrict__ pos, const ScanGeom& g, int base,
                                               bool vec, int& wi, bool& negative) {
  const int lane = threadIdx.x & 31;
  int v[8][4];
  if (vec) {
    size_t at = static_cast<size_t>(base);
    if (g.P != 1 && g.B != 1) {
      const int b = base / g.S, s = base - b * g.S, r = s / g.Sl;
      at = (static_cast<size_t>(r) * g.B + b) * g.Sl + (s - r * g.Sl);
    }
    const int4* p4 = reinterpret_cast<const int4*>(pos + at) + lane;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int4 x = __ldg(p4 + 32 * k);
      v[k][0] = x.x;
      v[k][1] = x.y;
      v[k][2] = x.z;
      v[k][3] = x.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int gi = base + 128 * k + 4 * lane + e;
        v[k][e] = gi < g.total ? load_pos(pos, g, gi) : 1;
      }
  }
  uint32_t mine = 0;
  negative = false;
  int rem = (base + 4 * lane) % g.S;  // g0 mod S, carried from step to step when S > 128
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int g0 = base + 128 * k + 4 * lane;
    if (k > 0) {
      if (g.S > 128) {
        rem += 128;
        if (rem >= g.S) rem -= g.S;
      } else {
        rem = g0 % g.S;
      }
    }
    // the next row start at or after g0 is g0 + (S - rem) % S; with rows of
    // 4 or more positions it is the only one among these four
    const int to_row = rem == 0 ? 0 : g.S - rem;
    const bool long_rows = g.S >= 4;
    uint32_t nib = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool in = g0 + e < g.total;
      negative |= in && v[k][e] < 0;
      const bool row = long_rows ? e == to_row : (e >= to_row) && ((e - to_row) % g.S == 0);
      if (in && (v[k][e] == 0 || row)) nib |= 1u << e;
    }
    uint32_t w = nib << (4 * (lane & 7));
    w |= __shfl_xor_sync(0xffffffffu, w, 1);
    w |= __shfl_xor_sync(0xffffffffu, w, 2);
    w |= __shfl_xor_sync(0xffffffffu, w, 4);
    if ((lane & 7) == k) mine = w;
  }
  wi = (lane & 7) * 4 + (lane >> 3);
  return mine;
}

__global__ void scan_init_kernel(ScanWs ws, int nblk, int32_t* max_len) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nblk; i += gridDim.x * blockDim.x) ws.state[i] = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *ws.ticket = 0;
    *max_len = 0;
  }
}

// Block-wide exclusive sum and max (-1 for none) of one value per thread;
// `tot_*` receive the block's totals.  sh: 2 * 32 ints.
__device__ __forceinline__ void block_scan2(int c, int l, int& ex_c, int& ex_l, int& tot_c, int& tot_l, int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ic = c, il = l;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int yc = __shfl_up_sync(0xffffffffu, ic, o);
    const int yl = __shfl_up_sync(0xffffffffu, il, o);
    if (lane >= o) {
      ic += yc;
      il = max(il, yl);
    }
  }
  if (lane == 31) {
    sh[warp] = ic;
    sh[32 + warp] = il;
  }
  __syncthreads();
  if (warp == 0) {
    const int wc = sh[lane], wl = sh[32 + lane];
    int jc = wc, jl = wl;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yc = __shfl_up_sync(0xffffffffu, jc, o);
      const int yl = __shfl_up_sync(0xffffffffu, jl, o);
      if (lane >= o) {
        jc += yc;
        jl = max(jl, yl);
      }
    }
    sh[lane] = jc - wc;                                             // exclusive over warps
    sh[32 + lane] = __shfl_up_sync(0xffffffffu, jl, 1) * (lane > 0) + (lane == 0 ? -1 : 0);
    if (lane == 31) {
      sh[64] = jc;
      sh[65] = jl;
    }
  }
  __syncthreads();
  const int up_l = __shfl_up_sync(0xffffffffu, il, 1);
  ex_c = sh[warp] + ic - c;
  ex_l = max(sh[32 + warp], lane > 0 ? up_l : -1);
  tot_c = sh[64];
  tot_l = sh[65];
  __syncthreads();
}

__global__ void __launch_bounds__(kScanThreads, 1) scan_kernel(const int32_t* __restrict__ pos, ScanGeom g, ScanWs ws,
                                                               int32_t* __restrict__ cu, int32_t* n_docs,
                                                               int32_t* max_len, int32_t* status) {
  extern __shared__ uint32_t flag_words[];  // min(range/32, kScanSmemWords)
  __shared__ int sh[72];
  __shared__ int sh_bid, sh_pre_cnt, sh_pre_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool single = g.nblk == 1;
  if (tid == 0) {
    sh_bid = single ? 0 : static_cast<int>(atomicAdd(ws.ticket, 1u));
    if (single) *max_len = 0;  // (the reset kernel does this when there are several blocks)
  }
  __syncthreads();
  const int bid = sh_bid;
  const int lo = bid * g.range;                                  // first position of this block's range
  const int hi = min(g.total, lo + g.range);
  const int n_steps = hi > lo ? (hi - lo + kScanStep - 1) / kScanStep : 0;
  const int n_words = n_steps * kScanThreads;

  // 1. flags of the range (kept as bits), count and latest start: each warp
  // takes 1024 consecutive positions per step
  int cnt = 0, last = -1;
  bool neg = false;
  for (int k = 0; k < n_steps; ++k) {
    const int base = lo + k * kScanStep + warp * (32 * kScanItems);
    if (base >= hi) {  // past the end of the sequence: these words hold no start
      const int w = k * kScanThreads + warp * 32 + lane;
      if (w < kScanSmemWords) flag_words[w] = 0u;
      continue;
    }
    int wl;
    bool n_ = false;
    // whole 1024-position chunks of one shard row take 16-byte loads
    const bool vec = g.vec && base + 32 * kScanItems <= hi;
    const uint32_t b = warp_flags(pos, g, base, vec, wl, n_);
    neg |= n_;
    const int w = k * kScanThreads + warp * 32 + wl;  // word index in the range
    if (w < kScanSmemWords) flag_words[w] = b;
    cnt += __popc(b);
    if (b) last = max(last, lo + w * kScanItems + 31 - __clz(b));
  }
  if (neg) set_status(status, USP_ERR_BAD_POSITIONS);
  int ex_c, ex_l, b_cnt, b_last;
  block_scan2(cnt, last, ex_c, ex_l, b_cnt, b_last, sh);
  if (tid == 0 && !single) st_state(ws.state + bid, scan_state(1, b_cnt, b_last));

  // 2. prefix: the aggregates of every block before this one
  if (warp == 0 && single) {
    if (lane == 0) {
      sh_pre_cnt = 0;
      sh_pre_last = -1;
    }
  } else if (warp == 0) {
    int pre_cnt = 0, pre_last = -1;
    const uint64_t t0 = global_ns();
    for (int j0 = 0; j0 < bid; j0 += 32) {
      const int j = j0 + lane;
      uint64_t s = j < bid ? ld_state(ws.state + j) : scan_state(1, 0, -1);
      while (state_flag(s) == 0) {  // that block is still on its range (it has started: it took a ticket first)
        if (global_ns() - t0 > 2000000000ull) {
          set_status(status, USP_ERR_TIMEOUT);
          s = scan_state(1, 0, -1);
          break;
        }
        __nanosleep(128);
        s = ld_state(ws.state + j);
      }
      pre_cnt += static_cast<int>(state_count(s));
      pre_last = max(pre_last, state_last(s));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      pre_cnt += __shfl_xor_sync(0xffffffffu, pre_cnt, o);
      pre_last = max(pre_last, __shfl_xor_sync(0xffffffffu, pre_last, o));
    }
    if (lane == 0) {
      sh_pre_cnt = pre_cnt;
      sh_pre_last = pre_last;
    }
  }
  __syncthreads();

  // 3. every thread a contiguous run of flag words: slots and the start before it
  const int per = (n_words + kScanThreads - 1) / kScanThreads;
  const int wa = min(n_words, tid * per), wb = min(n_words, wa + per);
  auto word = [&](int wi) -> uint32_t {
    if (wi < kScanSmemWords) return flag_words[wi];
    const int f = lo + wi * kScanItems;  // beyond the shared-memory budget: recompute
    bool n_ = false;
    return f < hi ? thread_flags(pos, g, f, n_) : 0u;
  };
  int rc = 0, rl = -1;
  for (int wi = wa; wi < wb; ++wi) {
    const uint32_t w = word(wi);
    rc += __popc(w);
    if (w) rl = max(rl, lo + wi * kScanItems + 31 - __clz(w));
  }
  int off, prev, tc, tl;
  block_scan2(rc, rl, off, prev, tc, tl, sh);
  off += sh_pre_cnt;
  prev = max(prev, sh_pre_last);
  int local_max = 0;
  for (int wi = wa; wi < wb; ++wi) {
    uint32_t w = word(wi);
    while (w) {
      const int gi = lo + wi * kScanItems + __ffs(w) - 1;
      w &= w - 1;
      cu[off++] = gi;
      if (prev >= 0) local_max = max(local_max, gi - prev);
      prev = gi;
    }
  }
  if (bid == g.nblk - 1 && tid == 0) {
    // the last document ends at B*S
    const int n = sh_pre_cnt + b_cnt;
    *n_docs = n;
    cu[n] = g.total;
    local_max = max(local_max, g.total - max(sh_pre_last, b_last));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) local_max = max(local_max, __shfl_xor_sync(0xffffffffu, local_max, o));
  if (lane == 0 && local_max) atomicMax(max_len, local_max);
}

size_t cu_seqlens_ws_bytes(int B, int S) {
  return cu_seqlens_ws_bytes_for(static_cast<long long>(B) * S);
}

int launch_cu_seqlens(const int32_t* pos, int B, int S, int P, int32_t* cu, int32_t* n_docs, int32_t* max_len,
                      int32_t* ws, int32_t* status, cudaStream_t st) {
  ScanGeom g{B, S, P, S / P, B * S, 0, 0, 0};
  // as many blocks as SMs (at most one per kScanChunk positions, the
  // workspace's state count); each block's range a whole number of steps
  const long long chunks = (static_cast<long long>(g.total) + kScanChunk - 1) / kScanChunk;
  const int want = static_cast<int>(std::min<long long>(std::max<long long>(chunks, 1), device_sm_count()));
  const long long steps = (static_cast<long long>(g.total) + kScanStep - 1) / kScanStep;
  g.range = static_cast<int>((steps + want - 1) / want) * kScanStep;
  g.nblk = static_cast<int>((static_cast<long long>(g.total) + g.range - 1) / g.range);
  if (g.nblk < 1) g.nblk = 1;
  // 16-byte loads: an aligned buffer whose 32-position runs (one thread, when
  // recomputing) and 1024-position runs (one warp) never cross a shard row
  g.vec = (reinterpret_cast<uintptr_t>(pos) & 15u) == 0 &&
          (P == 1 || B == 1 || (g.Sl % (32 * kScanItems) == 0 && S % (32 * kScanItems) == 0));
  ScanWs w{reinterpret_cast<uint32_t*>(ws),
           reinterpret_cast<uint64_t*>(reinterpret_cast<char*>(ws) + kScanHeaderBytes)};
  const size_t smem = sizeof(uint32_t) * std::min<size_t>(g.range / kScanItems, kScanSmemWords);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
    return USP_ERR_CUDA;
  // (one block needs no ticket and no block states: no reset kernel)
  if (g.nblk > 1) scan_init_kernel<<<1, 256, 0, st>>>(w, g.nblk, max_len);
  scan_kernel<<<g.nblk, kScanThreads, smem, st>>>(pos, g, w, cu, n_docs, max_len, status);
  return check_launch();
}

}  // namespace usp
