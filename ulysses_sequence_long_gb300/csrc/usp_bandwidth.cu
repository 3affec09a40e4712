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
// One pass over the positions (single-pass scan with decoupled look-back,
// Merrill & Garland, "Single-pass Parallel Prefix Scan with Decoupled
// Look-back", NVIDIA tech report NVR-2016-002): every block takes kScanChunk
// positions in the order blocks start (a ticket, so that every block a block
// looks back at is already running), counts its document starts and notes
// its last one, publishes that aggregate, then looks back over its
// predecessors' published states for the exclusive prefix (number of starts
// before it, latest start before it), publishes its inclusive state and
// scatters its starts into cu_seqlens.  A document's length is taken where it
// ends: at the next start (in the same block or, for a block's first start,
// after the latest start before the block), and after the last start by the
// last block.  A small kernel before it resets the block states.
constexpr int kScanThreads = 256;
constexpr int kScanItems = kScanChunk / kScanThreads;  // 16 consecutive positions per thread
static_assert(kScanItems == 16, "a thread's positions are four 16-byte vectors");

struct ScanGeom {
  int B, S, P, Sl, total, nblk;
  int vec;  // 1: each thread's 16 positions are one aligned, contiguous run
};

// Per-block state, one 64-bit word: flag (2 bits: 0 nothing yet, 1 the
// block's own aggregate, 2 its inclusive prefix), starts counted (31 bits)
// and latest start + 1 (31 bits, 0 = none).  B*S < 2^31 - 1 keeps both in range.
__device__ __forceinline__ uint64_t scan_state(uint32_t flag, uint32_t count, int last) {
  return (static_cast<uint64_t>(flag) << 62) | (static_cast<uint64_t>(count & 0x7FFFFFFFu) << 31) |
         static_cast<uint64_t>(static_cast<uint32_t>(last + 1) & 0x7FFFFFFFu);
}
__device__ __forceinline__ uint32_t state_flag(uint64_t s) { return static_cast<uint32_t>(s >> 62); }
__device__ __forceinline__ uint32_t state_count(uint64_t s) { return static_cast<uint32_t>(s >> 31) & 0x7FFFFFFFu; }
__device__ __forceinline__ int state_last(uint64_t s) { return static_cast<int>(s & 0x7FFFFFFFu) - 1; }

__device__ __forceinline__ void st_release(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_acquire(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
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
    // sixteen consecutive positions of one shard row: four 16-byte loads
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

__global__ void scan_init_kernel(ScanWs ws, int nblk, int32_t* max_len) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nblk; i += gridDim.x * blockDim.x) ws.state[i] = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *ws.ticket = 0;
    *max_len = 0;
  }
}

__global__ void __launch_bounds__(kScanThreads) scan_kernel(const int32_t* __restrict__ pos, ScanGeom g, ScanWs ws,
                                                            int32_t* __restrict__ cu, int32_t* n_docs,
                                                            int32_t* max_len, int32_t* status) {
  __shared__ int sh_cnt[kScanThreads / 32], sh_last[kScanThreads / 32];
  __shared__ int sh_bid, sh_pre_cnt, sh_pre_last, sh_max;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    sh_bid = static_cast<int>(atomicAdd(ws.ticket, 1u));
    sh_max = 0;
  }
  __syncthreads();
  const int bid = sh_bid;
  const int first = bid * kScanChunk + tid * kScanItems;
  bool neg;
  const uint32_t f = thread_flags(pos, g, first, neg);
  if (neg) set_status(status, USP_ERR_BAD_POSITIONS);

  // block scan of (starts, latest start) over the threads: warp shuffles,
  // then the warps' totals
  const int cnt = __popc(f);
  const int last = f ? first + 31 - __clz(f) : -1;
  int inc_cnt = cnt, inc_last = last;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int c = __shfl_up_sync(0xffffffffu, inc_cnt, o);
    const int l = __shfl_up_sync(0xffffffffu, inc_last, o);
    if (lane >= o) {
      inc_cnt += c;
      inc_last = max(inc_last, l);
    }
  }
  if (lane == 31) {
    sh_cnt[warp] = inc_cnt;
    sh_last[warp] = inc_last;
  }
  __syncthreads();
  int w_cnt = 0, w_last = -1, b_cnt = 0, b_last = -1;  // before this warp; the whole block
#pragma unroll
  for (int w = 0; w < kScanThreads / 32; ++w) {
    if (w < warp) {
      w_cnt += sh_cnt[w];
      w_last = max(w_last, sh_last[w]);
    }
    b_cnt += sh_cnt[w];
    b_last = max(b_last, sh_last[w]);
  }
  const int ex_cnt = w_cnt + inc_cnt - cnt;                                         // starts before this thread
  const int up_last = __shfl_up_sync(0xffffffffu, inc_last, 1);
  const int ex_last = max(w_last, lane > 0 ? up_last : -1);                          // latest start before it

  // look back over the predecessors (warp 0)
  if (warp == 0) {
    int pre_cnt = 0, pre_last = -1;
    if (bid == 0) {
      if (lane == 0) st_release(ws.state, scan_state(2, b_cnt, b_last));
    } else {
      if (lane == 0) st_release(ws.state + bid, scan_state(1, b_cnt, b_last));
      int base = bid - 1;
      const uint64_t t0 = global_ns();
      while (true) {
        const int j = base - lane;
        const uint64_t s = j >= 0 ? ld_acquire(ws.state + j) : scan_state(2, 0, -1);
        const uint32_t fl = state_flag(s);
        const uint32_t incl = __ballot_sync(0xffffffffu, fl == 2);
        const uint32_t none = __ballot_sync(0xffffffffu, fl == 0);
        // lanes up to the nearest inclusive state (all 32 if there is none here)
        const uint32_t upto = incl ? ((incl & (0u - incl)) << 1) - 1u : 0xffffffffu;
        if ((none & upto) == 0) {
          int c = (upto >> lane) & 1u ? static_cast<int>(state_count(s)) : 0;
          int l = (upto >> lane) & 1u ? state_last(s) : -1;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            c += __shfl_xor_sync(0xffffffffu, c, o);
            l = max(l, __shfl_xor_sync(0xffffffffu, l, o));
          }
          pre_cnt += c;
          pre_last = max(pre_last, l);
          if (incl) break;
          base -= 32;
        } else if (global_ns() - t0 > 2000000000ull) {  // every block looked at is running: never expected
          if (lane == 0) set_status(status, USP_ERR_TIMEOUT);
          break;
        }
      }
      if (lane == 0) st_release(ws.state + bid, scan_state(2, pre_cnt + b_cnt, max(pre_last, b_last)));
    }
    if (lane == 0) {
      sh_pre_cnt = pre_cnt;
      sh_pre_last = pre_last;
    }
  }
  __syncthreads();

  // scatter the starts; each document's length where it ends
  int off = sh_pre_cnt + ex_cnt;
  int prev = max(sh_pre_last, ex_last);
  int local_max = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    if (f & (1u << i)) {
      const int gi = first + i;
      cu[off++] = gi;
      if (prev >= 0) local_max = max(local_max, gi - prev);
      prev = gi;
    }
  }
  if (bid == g.nblk - 1 && tid == kScanThreads - 1) {
    // the last document ends at B*S
    const int n = sh_pre_cnt + b_cnt;
    *n_docs = n;
    cu[n] = g.total;
    local_max = max(local_max, g.total - max(sh_pre_last, b_last));
  }
  if (local_max) atomicMax(&sh_max, local_max);
  __syncthreads();
  if (tid == 0 && sh_max) atomicMax(max_len, sh_max);
}

size_t cu_seqlens_ws_bytes(int B, int S) {
  return cu_seqlens_ws_bytes_for(static_cast<long long>(B) * S);
}

int launch_cu_seqlens(const int32_t* pos, int B, int S, int P, int32_t* cu, int32_t* n_docs, int32_t* max_len,
                      int32_t* ws, int32_t* status, cudaStream_t st) {
  ScanGeom g{B, S, P, S / P, B * S, 0, 0};
  g.nblk = (g.total + kScanChunk - 1) / kScanChunk;
  g.vec = (reinterpret_cast<uintptr_t>(pos) & 15u) == 0 &&
          (P == 1 || B == 1 || (g.Sl % kScanItems == 0 && S % kScanItems == 0));
  ScanWs w{reinterpret_cast<uint32_t*>(ws),
           reinterpret_cast<uint64_t*>(reinterpret_cast<char*>(ws) + kScanHeaderBytes)};
  const int init_grid = std::min(std::max(1, (g.nblk + 255) / 256), 4 * device_sm_count());
  scan_init_kernel<<<init_grid, 256, 0, st>>>(w, g.nblk, max_len);
  scan_kernel<<<g.nblk, kScanThreads, 0, st>>>(pos, g, w, cu, n_docs, max_len, status);
  return check_launch();
}

}  // namespace usp
