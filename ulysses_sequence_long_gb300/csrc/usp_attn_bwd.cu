// usp_attn_bwd.cu — attention backward on the tcgen05 tensor core, all P
// emulated ranks per launch, deterministic (no floating-point atomics).
//
// Gradients of O_t = sum_u exp(s_tu - LSE_t) v_u, s_tu = scale q_t.k_u, for the
// loss sum(O * dO), with P_tu = exp(s_tu - LSE_t) and D_t = dO_t . O_t:
//   dV_u = sum_t P_tu dO_t          dK_u = scale sum_t dS_tu q_t
//   dQ_t = scale sum_u dS_tu k_u    dS_tu = P_tu (dO_t . v_u - D_t)
//   dz   = -sum_t exp(z - LSE_t) D_t   (sink logit of the head)
// Key/value gradients sum over the query heads of their GQA group; on each
// rank those are its own heads (contiguous head blocks keep groups local).
//
// Launches (each phase has its own entry point):
//   preprocess  D_t and -LSE_t*log2(e) for every (rank, query head, token), in a
//               planar fp32 workspace [P*hq][2][B*S padded to 4]; then the sink
//               gradients (one block per head, fixed-order tree reduction).
//   dK/dV       CTA = (rank, kv head, 128 keys).  K and V stay resident for
//               the whole CTA (TMEM at D=64, shared memory at D=128) as the A
//               operands of S^T = K Q^T and dP^T = V dO^T; 128-query slices of
//               Q, dO and their statistics stream through shared memory; P^T
//               and dS^T (bf16) are written over S^T / dP^T and feed
//               dV += P^T dO, dK += dS^T Q.
//   dQ          CTA = (rank, query head, 128 rows).  Q and dO live in TMEM as
//               the A operands of S = Q K^T and dP = dO V^T; 128-key tiles of
//               K and V stream through shared memory; dS (bf16 over S) feeds
//               dQ += dS K.
// The products with P^T and dS^T take their A operand from TMEM.  The dK/dV
// scores read K (or V) from TMEM at D=64 and from shared memory at D=128,
// where TMEM holds only the four accumulators: with N = 128 such an SS MMA
// reads 8 KB per 128x128x16 step, about the shared-memory bandwidth of the SM
// over the step's duration (at N = 64 the step would take as long for half the
// work).
// Warp roles (320 threads): warps 0-7 compute (warp w owns TMEM lanes
// 32*(w%4)..+31), warp 8 feeds shared memory (TMA), warp 9 issues the MMAs
// from one thread.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "usp_attn_common.cuh"
#include "usp_internal.h"

namespace usp {

namespace bwd {

constexpr int kThreads = 320;
constexpr int kSL = 64;                      // queries of a stored dS block
constexpr int kAtomBytes = kBN * 128;        // 128-row, 128-byte-wide swizzle column
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxDynSmem = 227 * 1024;      // opt-in dynamic shared memory per CTA

// index of (rank r, local head j, rank-local token t) in a [P][B][hq][S] array
__device__ __forceinline__ size_t stat_index(const AttnArgs& p, int r, int j, int t) {
  const int b = t / p.S, s = t - b * p.S;
  return (static_cast<size_t>(r * p.B + b) * p.hq + j) * p.S + s;
}

// Planar statistics: plane 0 = -LSE*log2(e) (negated, so that the packed FMA
// adds it), plane 1 = D, rows of `bsp` (B*S rounded up to a multiple of 4, so
// every plane starts 16-byte aligned).
__device__ __forceinline__ size_t plane_index(int bsp, int hq, int r, int j, int plane, int t) {
  return ((static_cast<size_t>(r) * hq + j) * 2 + plane) * bsp + t;
}

// --------------------------------------------------------------- preprocess
// A block takes a chunk of `tok` consecutive tokens (32; 16 or 8 when a short
// sequence would leave SMs without a chunk) with every head stored next to
// them (seq-layout: all H heads of the shard; head-layout: the hq heads of one
// rank), so its O/dO reads are one contiguous run.  Row sums go to shared
// memory, then each head's `tok` statistics are written (and its LSE read) as
// one contiguous run.
constexpr int kPreTok = 32;  // the most tokens of a chunk

template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dO,
                                                         const float* __restrict__ lse, float* __restrict__ stats,
                                                         AttnArgs p, int bsp, int n_chunks, int tok) {
  constexpr int LPR = D / 8;           // 16-byte lanes per row
  // passes whose loads are issued before any of them is reduced, so that
  // enough bytes are in flight (D = 64 rows are short; D = 128 keeps one)
  constexpr int kPreUnroll = D == 64 ? 4 : 1;
  constexpr int RPP = 256 / LPR;       // rows per pass of the block
  extern __shared__ float dsum[];      // [Hb][tok]
  const int Hb = p.seq_io ? p.P * p.hq : p.hq;
  const int tid = threadIdx.x, lane_row = tid % LPR;
  const int nct = (p.BS + tok - 1) / tok;  // head-layout chunks per rank
  for (int c = blockIdx.x; c < n_chunks; c += gridDim.x) {
    // chunk -> first token t0 (rank-local, b*S + s), its rank (head-layout) and
    // the element offset of its first row
    int r0 = 0, t0, ntok;
    size_t base;
    if (p.seq_io) {
      const int g0 = c * tok;                        // token index in memory order (shard, row, position)
      const int rp = g0 / (p.B * p.Sl), rem = g0 - rp * p.B * p.Sl;
      const int b = rem / p.Sl, sp = rem - b * p.Sl;
      t0 = b * p.S + rp * p.Sl + sp;
      ntok = tok;                                    // S/P is a multiple of 128
      base = static_cast<size_t>(g0) * Hb * D;
    } else {
      r0 = c / nct;
      t0 = (c - r0 * nct) * tok;
      ntok = min(tok, p.BS - t0);
      base = (static_cast<size_t>(r0) * p.BS + t0) * Hb * D;
    }
    const int nrows = ntok * Hb;
    for (int i0 = 0; i0 < nrows; i0 += kPreUnroll * RPP) {
      uint4 a[kPreUnroll], bq[kPreUnroll];
#pragma unroll
      for (int u = 0; u < kPreUnroll; ++u) {
        const int i = i0 + u * RPP + tid / LPR;
        a[u] = bq[u] = make_uint4(0, 0, 0, 0);
        if (i < nrows) {
          const size_t e = (base + static_cast<size_t>(i) * D) / 8 + lane_row;
          a[u] = __ldg(o + e);
          bq[u] = __ldg(dO + e);
        }
      }
#pragma unroll
      for (int u = 0; u < kPreUnroll; ++u) {
        const int i = i0 + u * RPP + tid / LPR;
        const uint32_t av[4] = {a[u].x, a[u].y, a[u].z, a[u].w}, bv[4] = {bq[u].x, bq[u].y, bq[u].z, bq[u].w};
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) acc += bf16lo(av[k]) * bf16lo(bv[k]) + bf16hi(av[k]) * bf16hi(bv[k]);
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (i < nrows && lane_row == 0) dsum[(i % Hb) * tok + i / Hb] = acc;
      }
    }
    __syncthreads();
    for (int idx = tid; idx < Hb * tok; idx += 256) {
      const int h = idx / tok, k = idx - h * tok;
      if (k < ntok) {
        const int r = p.seq_io ? h / p.hq : r0, j = p.seq_io ? h - r * p.hq : h, t = t0 + k;
        stats[plane_index(bsp, p.hq, r, j, 0, t)] = __ldg(lse + stat_index(p, r, j, t)) * -kLog2e;
        stats[plane_index(bsp, p.hq, r, j, 1, t)] = dsum[idx];
      }
    }
    __syncthreads();
  }
}

// --------------------------------------------------------------- dsink
__global__ void __launch_bounds__(256) dsink_kernel(const float* __restrict__ stats, float* __restrict__ dsinks,
                                                    AttnArgs p, int bsp) {
  __shared__ float red[256];
  const int r = blockIdx.x / p.hq, j = blockIdx.x % p.hq;
  const float z2 = __ldg(p.sinks + r * p.hq + j) * kLog2e;
  const float* l2 = stats + plane_index(bsp, p.hq, r, j, 0, 0);
  const float* dd = stats + plane_index(bsp, p.hq, r, j, 1, 0);
  float acc = 0.f;
  for (int t = threadIdx.x; t < p.BS; t += blockDim.x) acc -= ex2(z2 + __ldg(l2 + t)) * __ldg(dd + t);
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) dsinks[r * p.hq + j] = red[0];
}

// --------------------------------------------------------------- helpers
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&x)[N]) {
  static_assert(N % 32 == 0, "");
#pragma unroll
  for (int c = 0; c < N / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(taddr + c * 32, v);
#pragma unroll
    for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(v[e]);
  }
  tmem_wait_ld();
}

// x[0..2M) as M packed bf16 pairs into TMEM columns [taddr, taddr + M).
template <int M>
__device__ __forceinline__ void tmem_st_packed(uint32_t taddr, const float* x) {
  uint32_t pk[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) pk[e] = e < M ? pack_bf16x2(x[2 * e], x[2 * e + 1]) : 0u;
  if constexpr (M == 32) {
    tmem_st32(taddr, pk);
  } else {
    static_assert(M == 16, "");
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]), "r"(pk[6]), "r"(pk[7]), "r"(pk[8]),
        "r"(pk[9]), "r"(pk[10]), "r"(pk[11]), "r"(pk[12]), "r"(pk[13]), "r"(pk[14]), "r"(pk[15])
        : "memory");
  }
  tmem_wait_st();
}

// 16 packed columns into TMEM columns [taddr, taddr + 16) (this warp's lanes).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&pk)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]), "r"(pk[6]), "r"(pk[7]), "r"(pk[8]),
      "r"(pk[9]), "r"(pk[10]), "r"(pk[11]), "r"(pk[12]), "r"(pk[13]), "r"(pk[14]), "r"(pk[15])
      : "memory");
  tmem_wait_st();
}

// One bf16 row of D elements (global, 16-byte aligned) into TMEM as D/2 packed
// columns: the A-operand layout (lane = row, column = pair of K elements).
template <int D>
__device__ __forceinline__ void row_to_tmem(uint32_t taddr, const __nv_bfloat16* src, bool ok) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t v[32];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      uint4 w = ok ? __ldg(reinterpret_cast<const uint4*>(src + c * 64) + e) : make_uint4(0, 0, 0, 0);
      v[4 * e] = w.x;
      v[4 * e + 1] = w.y;
      v[4 * e + 2] = w.z;
      v[4 * e + 3] = w.w;
    }
    tmem_st32(taddr + c * 32, v);
  }
  tmem_wait_st();
}

// Write one TMEM row (NCOL fp32 columns at `taddr`) times `mul` as bf16 to `dst` (if `ok`).
template <int NCOL>
__device__ __forceinline__ void store_row(uint32_t taddr, __nv_bfloat16* dst, float mul, bool ok) {
#pragma unroll 1
  for (int c = 0; c < NCOL / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(taddr + c * 32, v);
    tmem_wait_ld();
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
    if (ok) {
      uint4* d = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
      for (int e = 0; e < 4; ++e) d[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
    }
  }
}

// K-major B operand (rows x D, 128-byte swizzle, `atom_bytes` per 64-column
// atom), MMA step kk over D: one descriptor per tile, moved per step.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int atom_bytes, int kk) {
  return sdesc_add(sdesc_sw128(base, 16, 1024), (kk >> 2) * atom_bytes + (kk & 3) * 32);
}
// MN-major B operand (rows = the MMA's K dimension, 128-byte rows of D), step kk over rows.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int atom_bytes, int kk) {
  return sdesc_add(sdesc_sw128(base, atom_bytes, 1024), kk * 16 * 128);
}

template <int D>
struct Cfg {
  static constexpr int NCH = D / 64;
  // dK/dV: 128-query slices.  At D=128 TMEM holds only the four 128-column
  // accumulators S^T, dP^T, dV, dK, so K and V sit in shared memory as the A
  // operands of S^T and dP^T; at D=64 they fit into TMEM beside them.
  static constexpr bool KV_SMEM = D == 128;
  static constexpr int SL = 128;
  static constexpr int SLB = SL * 128;            // one 64-column swizzle atom of a slice
  static constexpr int SLICE = NCH * SLB;         // SL-row bf16 tile
  static constexpr int STAT = 2 * SL * 4;         // [2][SL] fp32: -LSE*log2e, D
  static constexpr int NST = KV_SMEM ? 2 : 5;     // stages of the streamed slices
  static constexpr int STG = 32 * (SL / 2) * 2;   // a compute warp's [32 keys][64 queries] dS part
  // dK/dV: K and V tiles (KV_SMEM), rings of Q and dO slices and statistics,
  // one dS staging buffer per compute warp
  static constexpr int A_KV = 0;
  static constexpr int A_Q = KV_SMEM ? 2 * NCH * kBN * 128 : 0;
  static constexpr int A_DO = A_Q + NST * SLICE;
  static constexpr int A_STAT = A_DO + NST * SLICE;
  static constexpr int A_DS = (A_STAT + NST * STAT + 1023) / 1024 * 1024;
  static constexpr int A_BAR = A_DS + 8 * STG;
  static constexpr int A_NEED = A_BAR + 256;      // bytes used past the 1024-aligned base
  static constexpr int A_SMEM = A_NEED + 1024 < kMaxDynSmem ? A_NEED + 1024 : kMaxDynSmem;
  // dQ: ring of (K, V) 128-key tiles
  static constexpr int TILE = NCH * kBN * 128;       // 128-row bf16 tile
  static constexpr int KST = (D == 128) ? 3 : 6;
  static constexpr int B_K = 0;
  static constexpr int B_V = B_K + KST * TILE;
  static constexpr int B_BAR = B_V + KST * TILE;
  static constexpr int B_SMEM = B_BAR + 1024 + 1024;
};

struct BarsA {
  uint64_t kv_ready;  // K, V in place (TMEM rows from the compute warps, or the TMA tiles)
  uint64_t q_full[5], q_empty[5], do_full[5];  // q_empty: the slice pair (Q and dO) is free
  uint64_t st_full, dpt_full, p_full, ds_full;
  uint64_t fin, mma_done;
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(BarsA) <= 256, "dK/dV barrier block");
static_assert(Cfg<128>::A_NEED <= kMaxDynSmem && Cfg<64>::A_NEED + 1024 <= kMaxDynSmem, "dK/dV shared memory");

struct BarsB {
  uint64_t qd_ready;  // Q, dO rows stored into TMEM by the compute warps
  uint64_t k_full[8], v_full[8], kv_empty[8];
  uint64_t s_full, dp_full, ds_full;
  uint64_t fin, mma_done;
  uint32_t tmem;
  int abort;
};

// Stored dS blocks (the dK/dV pass writes them, the dQ pass reads them): one
// block = [128 keys][64 queries] bf16 of one (query head, batch row, key tile
// kt, 64-query slice qs), dS^T rows of 128 bytes.  Causal masks only: key tile
// kt meets the slices qs in [2kt, 2kt + n(kt)), n(kt) = min(N - 2kt, Wc), with
// N = S/64 slices per row and Wc = 2 (1 + ceil(window_left/128)) (N without a
// window).  Blocks of one (head, row) are numbered by key tile, then slice:
//   off(kt) = sum_{k < kt} n(k),  block(kt, qs) = off(kt) + qs - 2kt.
struct DsGeom {
  int N;              // 64-query slices per row
  int Wc;             // slices a key tile may meet (N without a window)
  int kc;             // key tiles [0, kc) meet Wc slices, later ones N - 2k
  long long per_row;  // blocks per (query head, batch row)
};

__host__ __device__ __forceinline__ int ds_count(const DsGeom& g, int kt) {
  const int n = g.N - 2 * kt;
  return n < g.Wc ? n : g.Wc;
}

__host__ __device__ __forceinline__ long long ds_off(const DsGeom& g, int kt) {
  if (kt <= g.kc) return static_cast<long long>(kt) * g.Wc;
  const long long k = kt, c = g.kc;
  return c * g.Wc + (k - c) * g.N - (k * (k - 1) - c * (c - 1));
}

struct Grads {
  const __nv_bfloat16* q;  // head layout, read row by row into TMEM
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const __nv_bfloat16* dO;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const float* stats;  // planar [P*hq][2][bsp]
  int bsp;
  int n_tiles;         // 128-token tiles per rank
  __nv_bfloat16* ds;   // stored dS blocks, or null (the dQ pass recomputes S and dP)
  DsGeom dsg;
};

// --------------------------------------------------------------- dK / dV
// TMEM: S^T [0,128)  dP^T [128,256)  dV [256,256+D)  dK [256+D,256+2D), and at
//       D=64 K [384,416)  V [416,448) as packed A operands (D=128: K and V are
//       128-key tiles in shared memory, the A operands of SS MMAs).
// Compute warps w: TMEM lanes 32*(w%4).. = key rows; group g = w/4 takes query
// columns [64g, 64g+64) of every slice (one stored 64-query dS block) and
// writes its 32 packed columns of P^T / dS^T at column 64g (columns it has
// read itself).
// Q and dO slices (with the statistics) stream through a ring whose slot is
// freed by one commit after dK_i (dV_i, which read dO_i, is done by then); the
// MMA thread waits for the next Q slice itself.  The MMA thread issues, per
// slice i:  [P^T_i] dV_i, S^T_{i+1}  [dS^T_i] dK_i, dP^T_{i+1}  (brackets: the
// compute warps' hand-offs), so the tensor core works on the next slice's
// scores while the compute warps turn the current one into P^T and dS^T.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                const __grid_constant__ CUtensorMap tst, const __grid_constant__ CUtensorMap tds_st,
                const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, AttnArgs p,
                Grads g) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (static_cast<int>(smem - smem_raw) > C::A_SMEM - C::A_NEED) {  // the launch's bytes cannot hold the layout
    if (tid == 0) set_status(p.status, USP_ERR_CUDA);
    return;
  }
  BarsA* bars = reinterpret_cast<BarsA*>(smem + C::A_BAR);

  // key tiles in order (early keys of a causal document see the most queries).
  // A CTA owns one key/value head: in head-layout the local head kl of rank r
  // (its gradient sums that rank's G query heads; replicas of a head are
  // summed by the exchange back), in seq-layout the global head, whose
  // gradient sums the whole group of Hq/Hkv query heads over the ranks.
  const int per = p.seq_io ? p.n_kvh : p.P * p.hk;
  const int kt = static_cast<int>(blockIdx.x) / per;
  const int unit = static_cast<int>(blockIdx.x) % per;
  const HeadRef kvh = p.seq_io ? HeadRef{0, 0, p.kvh0 + unit} : kv_head_ref(p, unit / p.hk, unit % p.hk);
  const int n_heads = p.seq_io ? p.Hq / p.Hkv : p.G;
  const int hg0 = p.seq_io ? (p.kvh0 + unit) * n_heads : kvh.r * p.hq + kvh.j * p.G;  // first query head (global)
  const int u0 = kt * kBN;

  const int n_docs = checked_docs(p);
  if (n_docs == 0) return;
  int qlo, qhi;
  query_range(p, n_docs, u0, min(u0 + kBN, p.BS) - 1, qlo, qhi);
  // ring x Ulysses step: only the queries of the super-chunk that holds this
  // key/value block at this step
  int rq0 = 0, rq1 = 0x7FFFFFFF;
  if (p.ring > 1) {
    ring_query_window(p, u0, rq0, rq1);
    qlo = max(qlo, rq0);
    qhi = min(qhi, rq1);
  }
  // statistics slices are fetched by TMA from 16-byte aligned tokens; with the
  // exchanges fused, slices must also stay inside one rank's shard.  When dS
  // is stored, whole 128-row query tiles are covered (their extra rows are
  // masked, so their blocks hold zeros): the dQ pass then finds a block for
  // every (key tile, query tile) pair it meets.
  const bool store_ds = g.ds != nullptr;
  if (store_ds) {
    qlo &= ~(kBM - 1);
    qhi = (qhi + kBM - 1) & ~(kBM - 1);
  } else {
    qlo &= p.seq_io ? ~(C::SL - 1) : ~3;
  }
  const int n_q = qhi > qlo ? (qhi - qlo + C::SL - 1) / C::SL : 0;
  const int n_it = n_heads * n_q;
  // stored dS: this key tile's place in the block numbering of its row
  const int ds_rowb = u0 / p.S, ds_row0 = ds_rowb * p.S, ds_kt = (u0 - ds_row0) / kBN;
  const int ds_cnt = store_ds ? ds_count(g.dsg, ds_kt) : 0;
  const long long ds_off0 = store_ds ? ds_off(g.dsg, ds_kt) : 0;

  if (tid == 0) {
    mbar_init(&bars->kv_ready, C::KV_SMEM ? 1 : 8);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
      mbar_init(&bars->do_full[s], 1);
    }
    mbar_init(&bars->st_full, 1);
    mbar_init(&bars->dpt_full, 1);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->ds_full, 8);
    mbar_init(&bars->fin, 1);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem, 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  volatile int* abort = &bars->abort;
  const uint32_t sbase = smem_u32(smem);
  constexpr uint32_t T_S = 0, T_DP = C::SL, T_DV = 2 * C::SL, T_DK = T_DV + D, T_K = T_DK + D, T_V = T_K + D / 2;
  static_assert(C::KV_SMEM ? T_K <= 512 : T_V + D / 2 <= 512, "TMEM columns");

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tdo);
      prefetch_tmap(&tst);
      if (C::KV_SMEM && n_it > 0) {
        mbar_arrive_expect_tx(&bars->kv_ready, 2 * C::NCH * kAtomBytes);
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_rows(smem + C::A_KV + c * kAtomBytes, &tk, &bars->kv_ready, p, c, kvh, u0);
          tma_load_rows(smem + C::A_KV + (C::NCH + c) * kAtomBytes, &tv, &bars->kv_ready, p, c, kvh, u0);
        }
      }
      int issued = 0;
      for (int i = 0; i < n_it; ++i) {
        const int s = i % C::NST;
        // dK_i done means dV_i is done too (in order): both slices are free
        if (i >= C::NST && !mbar_wait(&bars->q_empty[s], ((i / C::NST) - 1) & 1, abort, p.status)) break;
        const int hg = hg0 + i / n_q;
        const HeadRef qh{hg / p.hq, hg % p.hq, hg};
        const int q0 = qlo + (i % n_q) * C::SL;
        mbar_arrive_expect_tx(&bars->q_full[s], C::SLICE + C::STAT);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_rows(smem + C::A_Q + s * C::SLICE + c * C::SLB, &tq, &bars->q_full[s], p, c, qh, q0);
        tma_load_3d(smem + C::A_STAT + s * C::STAT, &tst, &bars->q_full[s], q0, 0, hg);
        mbar_arrive_expect_tx(&bars->do_full[s], C::SLICE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_rows(smem + C::A_DO + s * C::SLICE + c * C::SLB, &tdo, &bars->do_full[s], p, c, qh, q0);
        issued = i + 1;
      }
      // never leave the CTA with copies still landing in its shared memory
      if (C::KV_SMEM && n_it > 0) mbar_wait(&bars->kv_ready, 0, abort, p.status);
      for (int i = max(0, issued - C::NST); i < issued; ++i) {
        mbar_wait(&bars->q_full[i % C::NST], (i / C::NST) & 1, abort, p.status);
        mbar_wait(&bars->do_full[i % C::NST], (i / C::NST) & 1, abort, p.status);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(kBN, C::SL, false, false);  // [128 keys x SL queries], K = D
      constexpr uint32_t id_g = idesc_bf16(kBN, D, false, true);       // [128 keys x D], K = SL queries
      // S^T_i = K Q_i^T and dP^T_i = V dO_i^T (their slices have landed)
      auto issue_scores = [&](uint32_t t_out, uint32_t kv_t, uint32_t kv_s, uint32_t slice, uint64_t* done) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          if constexpr (C::KV_SMEM)
            mma_ss(tmem + t_out, kmajor_desc(kv_s, kAtomBytes, kk), kmajor_desc(slice, C::SLB, kk), id_s, kk > 0);
          else
            mma_ts(tmem + t_out, tmem + kv_t + kk * 8, kmajor_desc(slice, C::SLB, kk), id_s, kk > 0);
        }
        mma_commit(done);
      };
      const uint32_t k_s = sbase + C::A_KV, v_s = k_s + C::NCH * kAtomBytes;
      auto q_slot = [&](int i) { return sbase + C::A_Q + (i % C::NST) * C::SLICE; };
      auto do_slot = [&](int i) { return sbase + C::A_DO + (i % C::NST) * C::SLICE; };
      // A operand columns of a packed slice: compute group g packs its SL/2
      // queries into the SL/4 columns at g*SL/2 (K step kk: 16 queries, 8 columns)
      auto acol = [](int kk) -> uint32_t {
        constexpr int per = C::SL / 32;  // K steps per group
        return static_cast<uint32_t>((kk / per) * (C::SL / 2) + (kk % per) * 8);
      };
      bool ok = n_it == 0 || mbar_wait(&bars->kv_ready, 0, abort, p.status);
      if (ok && n_it > 0 && (ok = mbar_wait(&bars->q_full[0], 0, abort, p.status))) {
        tc_fence_after();
        issue_scores(T_S, T_K, k_s, q_slot(0), &bars->st_full);
        if ((ok = mbar_wait(&bars->do_full[0], 0, abort, p.status))) {
          tc_fence_after();
          issue_scores(T_DP, T_V, v_s, do_slot(0), &bars->dpt_full);
        }
      }
      for (int i = 0; i < n_it && ok; ++i) {
        const int s = i % C::NST;
        const uint32_t ph = i & 1, pn = ((i + 1) / C::NST) & 1;
        const bool more = i + 1 < n_it;
        // dV += P^T_i dO_i
        if (!(ok = mbar_wait(&bars->p_full, ph, abort, p.status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C::SL / 16; ++kk)
          mma_ts(tmem + T_DV, tmem + T_S + acol(kk), mnmajor_desc(do_slot(i), C::SLB, kk), id_g,
                 (i > 0 || kk > 0) ? 1u : 0u);
        // S^T_{i+1}: the S^T columns are free once dV_i has read P^T_i (in order)
        if (more) {
          if (!(ok = mbar_wait(&bars->q_full[(i + 1) % C::NST], pn, abort, p.status))) break;
          tc_fence_after();
          issue_scores(T_S, T_K, k_s, q_slot(i + 1), &bars->st_full);
        }
        // dK += dS^T_i Q_i; then the slices of iteration i (Q, dO, statistics) are free
        if (!(ok = mbar_wait(&bars->ds_full, ph, abort, p.status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C::SL / 16; ++kk)
          mma_ts(tmem + T_DK, tmem + T_DP + acol(kk), mnmajor_desc(q_slot(i), C::SLB, kk), id_g,
                 (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->q_empty[s]);
        if (more) {
          if (!(ok = mbar_wait(&bars->do_full[(i + 1) % C::NST], pn, abort, p.status))) break;
          tc_fence_after();
          issue_scores(T_DP, T_V, v_s, do_slot(i + 1), &bars->dpt_full);
        } else {
          mma_commit(&bars->fin);
        }
      }
      mma_commit(&bars->mma_done);
      mbar_wait(&bars->mma_done, 0, abort, p.status);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int grp = warp >> 2;                      // query columns [grp*SL/2, (grp+1)*SL/2) of each slice
    const int krow = (warp & 3) * 32 + lane;        // TMEM lane = key row
    const int u = u0 + krow;
    const bool key_ok = u < p.BS;
    int a = 0, b = 0;
    if (key_ok) doc_bounds(p.cu, n_docs, p.BS, u, a, b);
    a = max(a, rq0);  // a ring step: queries of one super-chunk only
    b = min(b, rq1);
    int vlo, vhi;     // the rows that see this key
    visible_rows(u, a, b, p.causal, p.window_left, key_ok, vlo, vhi);
    const uint32_t lb = tmem + ((static_cast<uint32_t>(warp & 3) * 32) << 16);
    if constexpr (!C::KV_SMEM) {
      // K (group 0) or V (group 1) row of this key into TMEM
      const size_t off = row_offset(p, kvh, p.hk, p.Hkv, key_ok ? u : 0, D);
      row_to_tmem<D>(lb + (grp == 0 ? T_K : T_V), (grp == 0 ? g.k : g.v) + off, key_ok);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->kv_ready);
    }
    // The group's SL/2 query columns of a slice, in 32-column chunks.  Packed
    // P^T (dS^T) of chunk c goes to the group's columns gc + 16c, over fp32
    // columns the group has already read.
    constexpr int NCK = C::SL / 64;
    const int gc = grp * (C::SL / 2);
    uint8_t* stg = smem + C::A_DS + warp * C::STG;  // this warp's dS staging buffer
    bool ok = true, staged = false;
    for (int i = 0; i < n_it && ok; ++i) {
      const int s = i % C::NST;
      const uint32_t ph = i & 1;
      const int q0 = qlo + (i % n_q) * C::SL + gc;  // first query column of this group
      // the statistics came with Q_i: observing its barrier makes them visible
      if (!(ok = mbar_wait(&bars->q_full[s], (i / C::NST) & 1, abort, p.status))) break;
      const float* st = reinterpret_cast<const float*>(smem + C::A_STAT + s * C::STAT) + gc;
      if (!(ok = mbar_wait(&bars->st_full, ph, abort, p.status))) break;
      tc_fence_after();
      const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
      // bit c: some key row of this warp sees a query of chunk c; the other
      // chunks have P = dS = 0 and skip their loads and exponentials
      uint32_t vis = 0;
#pragma unroll
      for (int c = 0; c < NCK; ++c) {
        const int c_lo = vlo - (q0 + 32 * c), c_hi = vhi - (q0 + 32 * c);
        vis |= (__any_sync(0xffffffffu, c_lo <= c_hi && c_hi >= 0 && c_lo <= 31) ? 1u : 0u) << c;
      }
      float pr[NCK][32];
#pragma unroll
      for (int c = 0; c < NCK; ++c) {
        if (!(vis >> c & 1u)) {
#pragma unroll
          for (int e = 0; e < 32; ++e) pr[c][e] = 0.f;
          tmem_st_packed<16>(lb + T_S + gc + 16 * c, pr[c]);
          continue;
        }
        float x[32];
        tmem_ld_cols<32>(lb + T_S + gc + 32 * c, x);
        // only chunks that straddle a document, diagonal or window edge pay
        // for the per-element mask (hidden scores become -inf, so exp2 gives 0)
        const int c_lo = vlo - (q0 + 32 * c), c_hi = vhi - (q0 + 32 * c);
        if (!(c_lo <= 0 && c_hi >= 31)) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e < c_lo || e > c_hi) x[e] = -INFINITY;
        }
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 l4 = *reinterpret_cast<const float4*>(st + 32 * c + 4 * c4);  // -LSE*log2(e)
          const float2 e0 = f2_unpack(f2_fma(f2_pack(x[4 * c4], x[4 * c4 + 1]), sc2, f2_pack(l4.x, l4.y)));
          const float2 e1 = f2_unpack(f2_fma(f2_pack(x[4 * c4 + 2], x[4 * c4 + 3]), sc2, f2_pack(l4.z, l4.w)));
          pr[c][4 * c4] = ex2(e0.x);
          pr[c][4 * c4 + 1] = ex2(e0.y);
          pr[c][4 * c4 + 2] = ex2(e1.x);
          pr[c][4 * c4 + 3] = ex2(e1.y);
        }
        tmem_st_packed<16>(lb + T_S + gc + 16 * c, pr[c]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);
      if (!(ok = mbar_wait(&bars->dpt_full, ph, abort, p.status))) break;
      tc_fence_after();
      // dS^T packed once: into TMEM for the dK MMA (first: the MMA thread
      // waits on it), then, if dS is stored, into the staging buffer
      uint32_t pk[NCK][16];
#pragma unroll
      for (int c = 0; c < NCK; ++c) {
        if (!(vis >> c & 1u)) {
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[c][e] = 0u;
          tmem_st16(lb + T_DP + gc + 16 * c, pk[c]);
          continue;
        }
        float x[32];
        tmem_ld_cols<32>(lb + T_DP + gc + 32 * c, x);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 d4 = *reinterpret_cast<const float4*>(st + C::SL + 32 * c + 4 * c4);
          const float2 g0 = f2_unpack(f2_mul(f2_pack(pr[c][4 * c4], pr[c][4 * c4 + 1]),
                                             f2_sub(f2_pack(x[4 * c4], x[4 * c4 + 1]), f2_pack(d4.x, d4.y))));
          const float2 g1 = f2_unpack(f2_mul(f2_pack(pr[c][4 * c4 + 2], pr[c][4 * c4 + 3]),
                                             f2_sub(f2_pack(x[4 * c4 + 2], x[4 * c4 + 3]), f2_pack(d4.z, d4.w))));
          x[4 * c4] = g0.x;
          x[4 * c4 + 1] = g0.y;
          x[4 * c4 + 2] = g1.x;
          x[4 * c4 + 3] = g1.y;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[c][e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
        tmem_st16(lb + T_DP + gc + 16 * c, pk[c]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ds_full);
      if (store_ds) {
        // The warp's [32 key rows][64 query columns] part of the dS^T block
        // (head, row, kt, qs): staged in shared memory in the 128-byte swizzle
        // (16-byte chunk e of row r at r*128 + (e ^ r%8)*16: every store
        // instruction is conflict-free) and written by one TMA store.
        const int hg = hg0 + i / n_q;
        const int qs = (qlo - ds_row0) / kSL + (i % n_q) * (C::SL / kSL) + grp;
        const int rel = qs - 2 * ds_kt;
        if (rel >= 0 && rel < ds_cnt) {
          const long long blk = (static_cast<long long>(hg - p.hq0) * p.B + ds_rowb) * g.dsg.per_row + ds_off0 + rel;
          if (staged && lane == 0) bulk_wait_group_read<0>();  // the previous store has read the buffer
          __syncwarp();
#pragma unroll
          for (int e = 0; e < 8; ++e)
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((e ^ (lane & 7)) << 4)) =
                make_uint4(pk[e / 4][4 * (e % 4)], pk[e / 4][4 * (e % 4) + 1], pk[e / 4][4 * (e % 4) + 2],
                           pk[e / 4][4 * (e % 4) + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tds_st, stg, 0, (warp & 3) * 32, static_cast<int>(blk));
            bulk_commit_group();
          }
          staged = true;
        }
      }
    }
    if (ok && n_it > 0 && (ok = mbar_wait(&bars->fin, 0, abort, p.status))) {
      tc_fence_after();
      const size_t off = row_offset(p, kvh, p.hk, p.Hkv, key_ok ? u : 0, D);
      if (grp == 0)
        store_row<D>(lb + T_DV, g.dv + off, 1.f, key_ok);
      else
        store_row<D>(lb + T_DK, g.dk + off, p.scale, key_ok);
    } else if (ok && n_it == 0 && key_ok) {
      __nv_bfloat16* dst = (grp == 0 ? g.dv : g.dk) + row_offset(p, kvh, p.hk, p.Hkv, u, D);
      for (int e = 0; e < D; e += 8) *reinterpret_cast<uint4*>(dst + e) = make_uint4(0, 0, 0, 0);
    }
    if (staged && lane == 0) bulk_wait_group_all();  // the dS stores are complete before the CTA ends
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// --------------------------------------------------------------- dQ
// TMEM: S [0,128)  dP [128,256)  dQ [256,256+D)  Q [256+D, 256+D+D/2)
//       dO [256+D+D/2, 256+2D)                                  (D=128: 512 columns)
// Iteration n covers a 128-key tile.  Compute group g = warp/4 takes key
// columns [64g, 64g+64) of S and dP and writes its 32 packed bf16 columns of dS
// at column 64g of S (columns it has read itself).  The MMA thread issues
// dQ(n), S(n+1), dP(n+1) as soon as dS(n) is complete: S is free once dQ(n)
// has read dS(n) (in-order), dP once the compute warps have read it.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, AttnArgs p, Grads g) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BarsB* bars = reinterpret_cast<BarsB*>(smem + C::B_BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // late query tiles first (they see the most keys)
  const int per = p.n_qh;  // the query heads of this pass's head group
  const int qt = g.n_tiles - 1 - static_cast<int>(blockIdx.x) / per;
  const int hg = p.hq0 + static_cast<int>(blockIdx.x) % per;
  const int r = hg / p.hq, j = hg % p.hq;
  const HeadRef qh = q_head_ref(p, r, j), kvh = kv_head_ref(p, r, j / p.G);
  const int t0 = qt * kBM;

  const int n_docs = checked_docs(p);
  if (n_docs == 0) return;
  int lo, hi;
  key_range(p, n_docs, t0, min(t0 + kBM, p.BS) - 1, lo, hi);
  int rk0 = 0, rk1 = 0x7FFFFFFF;  // ring x Ulysses step: one key/value super-chunk
  if (p.ring > 1) {
    ring_key_window(p, t0, rk0, rk1);
    lo = max(lo, rk0);
    hi = min(hi, rk1);
  }
  if (p.seq_io) lo &= ~(kBN - 1);  // key tiles inside one rank's shard
  const int n_kv = hi > lo ? (hi - lo + kBN - 1) / kBN : 0;

  if (tid == 0) {
    mbar_init(&bars->qd_ready, 8);
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->ds_full, 8);
    mbar_init(&bars->fin, 1);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem, 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  volatile int* abort = &bars->abort;
  const uint32_t sbase = smem_u32(smem);
  constexpr uint32_t T_S = 0, T_DP = 128, T_DQ = 256, T_Q = 256 + D, T_DO = T_Q + D / 2;

  if (warp == 8) {
    if (lane == 0) {
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      int issued = 0;
      for (int n = 0; n < n_kv; ++n) {
        const int s = n % C::KST;
        if (n >= C::KST && !mbar_wait(&bars->kv_empty[s], ((n / C::KST) - 1) & 1, abort, p.status)) break;
        const int kv0 = lo + n * kBN;
        mbar_arrive_expect_tx(&bars->k_full[s], C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_rows(smem + C::B_K + s * C::TILE + c * kAtomBytes, &tk, &bars->k_full[s], p, c, kvh, kv0);
        mbar_arrive_expect_tx(&bars->v_full[s], C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_rows(smem + C::B_V + s * C::TILE + c * kAtomBytes, &tv, &bars->v_full[s], p, c, kvh, kv0);
        issued = n + 1;
      }
      for (int n = max(0, issued - C::KST); n < issued; ++n) {
        mbar_wait(&bars->k_full[n % C::KST], (n / C::KST) & 1, abort, p.status);
        mbar_wait(&bars->v_full[n % C::KST], (n / C::KST) & 1, abort, p.status);
      }
    }
  } else if (warp == 9) {
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(kBM, kBN, false, false);  // [128 rows x 128 keys], K = D
      constexpr uint32_t id_q = idesc_bf16(kBM, D, false, true);      // [128 rows x D], K = 128 keys
      // A operand columns of the packed dS tile: the two 64-key halves sit at +0 and +64
      auto acol = [](int kk) -> uint32_t { return kk < 4 ? kk * 8 : 64 + (kk - 4) * 8; };
      auto issue_s = [&](int n) -> bool {
        const int s = n % C::KST;
        if (!mbar_wait(&bars->k_full[s], (n / C::KST) & 1, abort, p.status)) return false;
        tc_fence_after();
        const uint32_t ka = sbase + C::B_K + s * C::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ts(tmem + T_S, tmem + T_Q + kk * 8, kmajor_desc(ka, kAtomBytes, kk), id_s, kk > 0);
        mma_commit(&bars->s_full);
        return true;
      };
      auto issue_dp = [&](int n) -> bool {
        const int s = n % C::KST;
        if (!mbar_wait(&bars->v_full[s], (n / C::KST) & 1, abort, p.status)) return false;
        tc_fence_after();
        const uint32_t va = sbase + C::B_V + s * C::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ts(tmem + T_DP, tmem + T_DO + kk * 8, kmajor_desc(va, kAtomBytes, kk), id_s, kk > 0);
        mma_commit(&bars->dp_full);
        return true;
      };
      bool ok = mbar_wait(&bars->qd_ready, 0, abort, p.status);
      if (ok && n_kv > 0) ok = issue_s(0) && issue_dp(0);
      for (int n = 0; n < n_kv && ok; ++n) {
        const int s = n % C::KST;
        if (!(ok = mbar_wait(&bars->ds_full, n & 1, abort, p.status))) break;
        tc_fence_after();
        const uint32_t ka = sbase + C::B_K + s * C::TILE;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(tmem + T_DQ, tmem + T_S + acol(kk), mnmajor_desc(ka, kAtomBytes, kk), id_q,
                 (n > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->kv_empty[s]);
        if (n + 1 < n_kv)
          ok = issue_s(n + 1) && issue_dp(n + 1);
        else
          mma_commit(&bars->fin);
      }
      mma_commit(&bars->mma_done);
      mbar_wait(&bars->mma_done, 0, abort, p.status);
    }
  } else {
    const int grp = warp >> 2;             // key columns [64*grp, 64*grp + 64) of every tile
    const int row = (warp & 3) * 32 + lane;
    const int t = t0 + row;
    const bool row_ok = t < p.BS;
    const uint32_t lb = tmem + ((static_cast<uint32_t>(warp & 3) * 32) << 16);
    // Q (group 0) or dO (group 1) row into TMEM
    {
      const size_t off = row_offset(p, qh, p.hq, p.Hq, row_ok ? t : 0, D);
      row_to_tmem<D>(lb + (grp == 0 ? T_Q : T_DO), (grp == 0 ? g.q : g.dO) + off, row_ok);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->qd_ready);
    }
    int a = 0, b = 0;
    float nlse2 = -INFINITY, dvt = 0.f;  // -LSE*log2(e) of the row
    if (row_ok) {
      doc_bounds(p.cu, n_docs, p.BS, t, a, b);
      nlse2 = __ldg(g.stats + plane_index(g.bsp, p.hq, r, j, 0, t));
      dvt = __ldg(g.stats + plane_index(g.bsp, p.hq, r, j, 1, t));
    }
    a = max(a, rk0);  // a ring step: one key/value super-chunk only
    b = min(b, rk1);
    int vlo, vhi;     // the row's visible keys
    visible_keys(t, a, b, p.causal, p.window_left, row_ok, vlo, vhi);
    const uint32_t s_col = T_S + grp * 64, dp_col = T_DP + grp * 64;
    bool ok = true;
    for (int n = 0; n < n_kv && ok; ++n) {
      const uint32_t ph = n & 1;
      const int k0 = lo + n * kBN + grp * 64;  // first key of this group's columns
      if (!(ok = mbar_wait(&bars->s_full, ph, abort, p.status))) break;
      tc_fence_after();
      float x[64];
      tmem_ld_cols<64>(lb + s_col, x);
      const int c_lo = vlo - k0, c_hi = vhi - k0;
      if (!(c_lo <= 0 && c_hi >= 63)) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < c_lo || c > c_hi) x[c] = -INFINITY;
      }
      float pr[64];
      {
        const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nl2 = f2_pack(nlse2, nlse2);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 e = f2_unpack(f2_fma(f2_pack(x[c], x[c + 1]), sc2, nl2));
          pr[c] = ex2(e.x);
          pr[c + 1] = ex2(e.y);
        }
      }
      if (!(ok = mbar_wait(&bars->dp_full, ph, abort, p.status))) break;
      tc_fence_after();
      tmem_ld_cols<64>(lb + dp_col, x);
      {
        const uint64_t d2 = f2_pack(dvt, dvt);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 g2 = f2_unpack(f2_mul(f2_pack(pr[c], pr[c + 1]), f2_sub(f2_pack(x[c], x[c + 1]), d2)));
          x[c] = g2.x;
          x[c + 1] = g2.y;
        }
      }
      tmem_st_packed<32>(lb + s_col, x);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ds_full);
    }
    if (ok && n_kv > 0 && (ok = mbar_wait(&bars->fin, 0, abort, p.status))) {
      tc_fence_after();
      __nv_bfloat16* dst = g.dq + row_offset(p, qh, p.hq, p.Hq, row_ok ? t : 0, D) + grp * (D / 2);
      store_row<D / 2>(lb + T_DQ + grp * (D / 2), dst, p.scale, row_ok);
    } else if (ok && n_kv == 0 && row_ok) {  // no key at this ring step: dQ = 0
      __nv_bfloat16* dst = g.dq + row_offset(p, qh, p.hq, p.Hq, t, D) + grp * (D / 2);
      for (int e = 0; e < D / 2; e += 8) *reinterpret_cast<uint4*>(dst + e) = make_uint4(0, 0, 0, 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// --------------------------------------------------------------- dQ from stored dS
// dQ_t = scale sum_u dS_tu k_u with dS read back from the blocks the dK/dV
// pass stored: no recomputation of S and dP, one GEMM per key tile.  A unit
// of work = (rank, query head, 128 rows); the kernel is persistent: each CTA
// walks units blockIdx.x, +gridDim.x, ... (late query tiles first), so the
// next unit's tiles stream in while the current one finishes.  Per 128-key
// tile the two 64-query dS blocks (A operand, MN-major: queries contiguous)
// and the K tile (B operand, MN-major: D contiguous) pass through a
// shared-memory ring; dQ accumulates in one of two TMEM buffers (128 lanes x
// D columns each) while the epilogue drains the other.  dS holds the masks
// already, so no mask is evaluated here.  Warps 0-3: epilogue, warp 4: TMA
// producer, warp 5: MMA.
constexpr int kDsThreads = 192;

template <int D>
struct CfgDs {
  static constexpr int NCH = D / 64;
  static constexpr int DSB = 2 * kBN * 128;     // two [128 keys][64 queries] bf16 blocks
  static constexpr int KT = NCH * kBN * 128;    // K tile [128 keys][D]
  static constexpr int STAGE = DSB + KT;
  static constexpr int NST = (D == 128) ? 3 : 4;
  static constexpr int STG = NCH * kBM * 128;   // the unit's dQ tile, staged for its TMA store
  static constexpr int OFF_STG = NST * STAGE;
  static constexpr int BAR = OFF_STG + STG;
  static constexpr int SMEM = BAR + 1024 + 1024;
};
static_assert(CfgDs<128>::SMEM <= 227 * 1024 && CfgDs<64>::SMEM <= 227 * 1024, "dQ shared memory");

struct BarsDs {
  uint64_t full[4], empty[4];
  uint64_t fin[2], tfree[2];  // dQ buffer b: accumulated / read out by the epilogue
  uint64_t stg_full;          // the 4 epilogue warps have staged the unit's dQ tile
  uint64_t stg_free;          // its TMA store has read the staging tile
  uint64_t mma_done;
  uint32_t tmem;
  int abort;
};

// One unit's geometry, computed identically by every role.
struct DsUnit {
  int t0, r, j, row0, kt0, qs0, n_kv;
  long long head_base;
};

__device__ __forceinline__ DsUnit ds_unit(const AttnArgs& p, const Grads& g, int n_docs, int u) {
  DsUnit w;
  const int per = p.n_qh;  // the query heads of this pass's head group
  const int qt = g.n_tiles - 1 - u / per;
  const int rem = u % per, hg = p.hq0 + rem;
  w.r = hg / p.hq;
  w.j = hg % p.hq;
  w.t0 = qt * kBM;
  int lo, hi;
  key_range(p, n_docs, w.t0, min(w.t0 + kBM, p.BS) - 1, lo, hi);
  if (p.ring > 1) {  // ring x Ulysses step: one key/value super-chunk
    int rk0, rk1;
    ring_key_window(p, w.t0, rk0, rk1);
    lo = max(lo, rk0);
    hi = min(hi, rk1);
  }
  const int rowb = w.t0 / p.S;
  w.row0 = rowb * p.S;
  lo = w.row0 + ((lo - w.row0) & ~(kBN - 1));  // blocks belong to aligned key tiles
  w.n_kv = hi > lo ? (hi - lo + kBN - 1) / kBN : 0;
  w.kt0 = (lo - w.row0) / kBN;
  w.qs0 = (w.t0 - w.row0) / kSL;  // the tile's first 64-query slice
  w.head_base = (static_cast<long long>(rem) * p.B + rowb) * g.dsg.per_row;
  return w;
}

template <int D>
__global__ void __launch_bounds__(kDsThreads, 1)
    dq_ds_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tds,
                 const __grid_constant__ CUtensorMap tdq, AttnArgs p, Grads g, int n_units) {
  using C = CfgDs<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BarsDs* bars = reinterpret_cast<BarsDs*>(smem + C::BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int n_docs = checked_docs(p);
  if (n_docs == 0) return;

  if (tid == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->fin[b], 1);
      mbar_init(&bars->tfree[b], 4);
    }
    mbar_init(&bars->stg_full, 4);
    mbar_init(&bars->stg_free, 1);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem, 2 * D);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  volatile int* abort = &bars->abort;
  const uint32_t sbase = smem_u32(smem);

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tk);
      prefetch_tmap(&tds);
      int gn = 0;  // tiles issued by this CTA over all its units (ring position)
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const DsUnit w = ds_unit(p, g, n_docs, u);
        const HeadRef kvh = kv_head_ref(p, w.r, w.j / p.G);
        for (int n = 0; n < w.n_kv; ++n, ++gn) {
          const int s = gn % C::NST;
          if (gn >= C::NST && !(ok = mbar_wait(&bars->empty[s], ((gn / C::NST) - 1) & 1, abort, p.status)))
            break;
          const int kt = w.kt0 + n, rel = w.qs0 - 2 * kt;
          // the dK/dV pass covered whole query tiles, so both blocks exist for
          // every key tile this query tile meets; anything else is a broken
          // invariant, recorded instead of read
          if (rel < 0 || rel + 1 >= ds_count(g.dsg, kt)) {
            set_status(p.status, USP_ERR_BAD_SEQLENS);
            *abort = 1;
            ok = false;
            break;
          }
          uint8_t* st = smem + s * C::STAGE;
          mbar_arrive_expect_tx(&bars->full[s], C::STAGE);
          tma_load_3d(st, &tds, &bars->full[s], 0, 0, static_cast<int>(w.head_base + ds_off(g.dsg, kt) + rel));
          for (int c = 0; c < C::NCH; ++c)
            tma_load_rows(st + C::DSB + c * kAtomBytes, &tk, &bars->full[s], p, c, kvh, w.row0 + kt * kBN);
        }
      }
      // never leave the CTA with copies still landing in its shared memory
      for (int n = max(0, gn - C::NST); n < gn; ++n)
        mbar_wait(&bars->full[n % C::NST], (n / C::NST) & 1, abort, p.status);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kBM, D, true, true);  // [128 queries x D], K = 128 keys
      bool ok = true;
      int gn = 0, ub = 0;  // tiles consumed; units accumulated (buffer ub & 1)
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const DsUnit w = ds_unit(p, g, n_docs, u);
        if (w.n_kv == 0) continue;
        const int b = ub & 1;
        // the epilogue has read this buffer's previous unit out
        if (ub >= 2 && !(ok = mbar_wait(&bars->tfree[b], ((ub >> 1) - 1) & 1, abort, p.status))) break;
        tc_fence_after();
        for (int n = 0; n < w.n_kv && ok; ++n, ++gn) {
          const int s = gn % C::NST;
          if (!(ok = mbar_wait(&bars->full[s], (gn / C::NST) & 1, abort, p.status))) break;
          tc_fence_after();
          const uint32_t a = sbase + s * C::STAGE, bb = a + C::DSB;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ss(tmem + b * D, mnmajor_desc(a, kBN * 128, kk), mnmajor_desc(bb, kAtomBytes, kk), idesc,
                   (n > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars->empty[s]);
        }
        if (ok) mma_commit(&bars->fin[b]);
        ++ub;
      }
      mma_commit(&bars->mma_done);
      mbar_wait(&bars->mma_done, 0, abort, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // dQ rows leave through a staging tile in the 128-byte swizzle of the
    // tensor map (16-byte chunk e of row r of a 64-column atom at
    // r*128 + (e ^ r%8)*16, conflict-free) and one TMA store per atom, issued
    // by thread 0 once the four warps have staged the tile: per-thread row
    // stores would touch 32 lines per store instruction.
    bool ok = true, stored = false;
    int ub = 0;
    uint8_t* stg = smem + C::OFF_STG;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const DsUnit w = ds_unit(p, g, n_docs, u);
      const HeadRef qh = q_head_ref(p, w.r, w.j);
      const int t = w.t0 + warp * 32 + lane;
      const bool row_ok = t < p.BS;
      if (w.n_kv == 0) {  // no key at this ring step: dQ = 0
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(g.dq + row_offset(p, qh, p.hq, p.Hq, t, D));
          for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int b = ub & 1;
      if (!(ok = mbar_wait(&bars->fin[b], (ub >> 1) & 1, abort, p.status))) break;
      tc_fence_after();
      const uint32_t lb = tmem + b * D + ((static_cast<uint32_t>(warp) * 32) << 16);
      // the previous unit's store has read the staging tile
      if (ub > 0 && !(ok = mbar_wait(&bars->stg_free, (ub - 1) & 1, abort, p.status))) break;
      const int row = warp * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(lb + c * 32, v);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * p.scale, __uint_as_float(v[2 * e + 1]) * p.scale);
        uint8_t* atom = stg + (c >> 1) * (kBM * 128);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          *reinterpret_cast<uint4*>(atom + row * 128 + ((((c & 1) * 4 + k4) ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * k4], pk[4 * k4 + 1], pk[4 * k4 + 2], pk[4 * k4 + 3]);
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->tfree[b]);
        mbar_arrive(&bars->stg_full);
      }
      if (warp == 0 && lane == 0 && mbar_wait(&bars->stg_full, ub & 1, abort, p.status)) {
        for (int c = 0; c < C::NCH; ++c) tma_store_rows(&tdq, stg + c * (kBM * 128), p, c, qh, w.t0);
        bulk_commit_group();
        stored = true;
        bulk_wait_group_read<0>();
        mbar_arrive(&bars->stg_free);
      }
      __syncwarp();
      if (*abort) {  // a wait gave up (the whole warp leaves together)
        ok = false;
        break;
      }
      ++ub;
    }
    if (stored) bulk_wait_group_all();  // the dQ stores are complete before the CTA ends
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * D);
  }
}

}  // namespace bwd

static int stats_row_pitch(int BS) { return (BS + 3) & ~3; }

size_t attn_bwd_ws_bytes(const usp_attn_params& p) {
  // planar {-LSE*log2e, D} per (rank, query head), rows padded to 4 tokens
  size_t n = static_cast<size_t>(p.Hq) * 2 * stats_row_pitch(p.B * p.S);
  return (n * sizeof(float) + 255) / 256 * 256;
}

// Block numbering of the stored dS (see DsGeom); false when the shape has no
// stored-dS path (non-causal masks, rows not a multiple of 128 tokens, or more
// blocks than a tensor-map coordinate holds).
static bool ds_geom(const usp_attn_params& p, bwd::DsGeom& g, long long& n_blocks) {
  if (!p.causal || p.S % kBN != 0) return false;
  g.N = p.S / bwd::kSL;
  g.Wc = g.N;
  if (p.window_left >= 0) {
    const long long wc = 2ll * (1 + (p.window_left + kBN - 1) / kBN);
    if (wc < g.N) g.Wc = static_cast<int>(wc);
  }
  g.kc = (g.N - g.Wc) / 2 + 1;
  g.per_row = bwd::ds_off(g, p.S / kBN);
  const long long heads = p.head_count > 0 ? static_cast<long long>(p.head_count) * (p.Hq / p.Hkv) : p.Hq;
  n_blocks = heads * p.B * g.per_row;
  return n_blocks > 0 && n_blocks < (1ll << 31);
}

size_t attn_bwd_ds_bytes(const usp_attn_params& p) {
  bwd::DsGeom g;
  long long n_blocks;
  if (!ds_geom(p, g, n_blocks)) return 0;
  return static_cast<size_t>(n_blocks) * kBN * bwd::kSL * 2;
}

static AttnArgs make_args(const usp_attn_params& prm, int32_t* status) {
  AttnArgs a;
  a.B = prm.B;
  a.S = prm.S;
  a.BS = prm.B * prm.S;
  a.P = prm.P;
  a.hq = prm.Hq / prm.P;
  a.hk = prm.Hkv >= prm.P ? prm.Hkv / prm.P : 1;
  a.G = a.hq / a.hk;
  a.Hq = prm.Hq;
  a.Hkv = prm.Hkv;
  a.causal = prm.causal ? 1 : 0;
  a.window_left = prm.window_left;
  a.scale = prm.softmax_scale > 0.f ? prm.softmax_scale : 1.0f / sqrtf(static_cast<float>(prm.D));
  a.scale_log2 = a.scale * 1.4426950408889634f;
  a.cu = prm.cu_seqlens;
  a.n_docs = prm.n_docs;
  a.sinks = prm.sinks;
  a.status = status;
  a.seq_io = prm.io_layout == USP_IO_SEQ ? 1 : 0;
  a.kv_seq_io = a.seq_io;
  a.ring = prm.ring > 1 ? prm.ring : 1;
  a.ring_step = a.ring > 1 ? prm.ring_step : 0;
  a.C = prm.S / a.ring;
  a.Sl = prm.S / (prm.P * a.ring);  // sequence shard: P Ulysses ranks in each of `ring` groups
  const int gf = prm.Hq / prm.Hkv;
  a.kvh0 = prm.head_count > 0 ? prm.head_first : 0;
  a.n_kvh = prm.head_count > 0 ? prm.head_count : prm.Hkv;
  a.hq0 = a.kvh0 * gf;
  a.n_qh = a.n_kvh * gf;
  return a;
}

// 1. D = rowsum(dO * O) and -LSE*log2e into the workspace, then the sink gradients.
int launch_attn_bwd_preprocess(const usp_attn_params& prm, const void* o, const float* lse, const void* dO,
                               float* dsinks, void* ws, int32_t* status, cudaStream_t st) {
  const AttnArgs a = make_args(prm, status);
  float* stats = static_cast<float*>(ws);
  const int bsp = stats_row_pitch(a.BS);
  const int Hb = a.seq_io ? a.P * a.hq : a.hq;
  // tokens per chunk: halved (down to 8) while there are fewer than two chunks per SM
  auto chunks_of = [&](int tok) { return a.seq_io ? a.BS / tok : a.P * ((a.BS + tok - 1) / tok); };
  int tok = bwd::kPreTok;
  while (tok > 8 && chunks_of(tok) < device_sm_count() * 2) tok /= 2;
  const int n_chunks = chunks_of(tok);
  const int smem = Hb * tok * static_cast<int>(sizeof(float));
  int grid = n_chunks < device_sm_count() * 8 ? n_chunks : device_sm_count() * 8;
  auto kern = prm.D == 128 ? bwd::preprocess_kernel<128> : bwd::preprocess_kernel<64>;
  if (smem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return USP_ERR_CUDA;
  kern<<<grid, 256, smem, st>>>(static_cast<const uint4*>(o), static_cast<const uint4*>(dO), lse, stats, a, bsp,
                                n_chunks, tok);
  if (check_launch() != USP_OK) return USP_ERR_CUDA;
  if (dsinks != nullptr && a.sinks != nullptr) {
    bwd::dsink_kernel<<<a.P * a.hq, 256, 0, st>>>(stats, dsinks, a, bsp);
    if (check_launch() != USP_OK) return USP_ERR_CUDA;
  }
  return USP_OK;
}

template <int D>
static int run_grad_pass(bool dq_pass, const AttnArgs& a, const void* q, const void* k, const void* v,
                         const void* dO, void* dq, void* dk, void* dv, const float* stats, void* ds,
                         const bwd::DsGeom& dsg, long long ds_blocks, cudaStream_t st) {
  using C = bwd::Cfg<D>;
  bwd::Grads g{static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
               static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(dO),
               static_cast<__nv_bfloat16*>(dq), static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv),
               stats, stats_row_pitch(a.BS), (a.BS + kBM - 1) / kBM, static_cast<__nv_bfloat16*>(ds), dsg};
  int rc;
  if (dq_pass && ds != nullptr) {
    // dQ = dS K from the blocks the dK/dV pass stored
    using CD = bwd::CfgDs<D>;
    CUtensorMap tk, tds, tdq;
    if ((rc = make_rows_tmap(&tk, k, a, a.hk, a.Hkv, D, kBN)) != USP_OK) return rc;
    if ((rc = make_ds_tmap(&tds, ds, ds_blocks)) != USP_OK) return rc;
    if ((rc = make_rows_tmap(&tdq, dq, a, a.hq, a.Hq, D, kBM)) != USP_OK) return rc;
    if (cudaFuncSetAttribute(bwd::dq_ds_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, CD::SMEM) !=
        cudaSuccess)
      return USP_ERR_CUDA;
    const int n_units = g.n_tiles * a.n_qh;
    const int grid = n_units < device_sm_count() ? n_units : device_sm_count();  // persistent: one CTA per SM
    bwd::dq_ds_kernel<D><<<grid, bwd::kDsThreads, CD::SMEM, st>>>(tk, tds, tdq, a, g, n_units);
    return check_launch();
  }
  if (!dq_pass) {
    // query slices of Q, dO and their statistics stream past TMEM-resident K, V
    CUtensorMap tq, tdo, tst;
    if ((rc = make_rows_tmap(&tq, q, a, a.hq, a.Hq, D, C::SL)) != USP_OK) return rc;
    if ((rc = make_rows_tmap(&tdo, dO, a, a.hq, a.Hq, D, C::SL)) != USP_OK) return rc;
    if ((rc = make_stats_tmap(&tst, stats, a.BS, g.bsp, a.P * a.hq, C::SL)) != USP_OK) return rc;
    CUtensorMap tds_st, tk, tv;
    memset(&tds_st, 0, sizeof(tds_st));  // unused unless dS is stored
    memset(&tk, 0, sizeof(tk));          // unused unless K, V are shared-memory tiles
    memset(&tv, 0, sizeof(tv));
    if (ds != nullptr && (rc = make_ds_store_tmap(&tds_st, ds, ds_blocks)) != USP_OK) return rc;
    if (C::KV_SMEM) {
      if ((rc = make_rows_tmap(&tk, k, a, a.hk, a.Hkv, D, kBN)) != USP_OK) return rc;
      if ((rc = make_rows_tmap(&tv, v, a, a.hk, a.Hkv, D, kBN)) != USP_OK) return rc;
    }
    if (cudaFuncSetAttribute(bwd::dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::A_SMEM) !=
        cudaSuccess)
      return USP_ERR_CUDA;
    const unsigned grid = static_cast<unsigned>(g.n_tiles) * (a.seq_io ? a.n_kvh : a.P * a.hk);
    bwd::dkdv_kernel<D><<<grid, bwd::kThreads, C::A_SMEM, st>>>(tq, tdo, tst, tds_st, tk, tv, a, g);
  } else {
    // 128-key tiles of K and V stream past TMEM-resident Q, dO
    CUtensorMap tk, tv;
    if ((rc = make_rows_tmap(&tk, k, a, a.hk, a.Hkv, D, kBN)) != USP_OK) return rc;
    if ((rc = make_rows_tmap(&tv, v, a, a.hk, a.Hkv, D, kBN)) != USP_OK) return rc;
    if (cudaFuncSetAttribute(bwd::dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::B_SMEM) != cudaSuccess)
      return USP_ERR_CUDA;
    bwd::dq_kernel<D><<<static_cast<unsigned>(g.n_tiles) * a.n_qh, bwd::kThreads, C::B_SMEM, st>>>(tk, tv, a, g);
  }
  return check_launch();
}

// The stored-dS region of the workspace (after the statistics), or null when
// the workspace is too small for it or the shape has no such path.
static void* ds_region(const usp_attn_params& prm, const void* ws, size_t ws_bytes, bwd::DsGeom& g,
                       long long& n_blocks) {
  const size_t need = attn_bwd_ds_bytes(prm);
  if (need == 0 || ws_bytes < attn_bwd_ws_bytes(prm) + need || !ds_geom(prm, g, n_blocks)) return nullptr;
  return static_cast<uint8_t*>(const_cast<void*>(ws)) + attn_bwd_ws_bytes(prm);
}

// 2. dK, dV (and the dS blocks, when the workspace holds them)
int launch_attn_bwd_dkdv(const usp_attn_params& prm, const void* q, const void* k, const void* v, const float* lse,
                         const void* dO, void* dk, void* dv, const void* ws, size_t ws_bytes, int32_t* status,
                         cudaStream_t st) {
  const AttnArgs a = make_args(prm, status);
  const float* stats = static_cast<const float*>(ws);
  (void)lse;  // read through the preprocess's statistics
  bwd::DsGeom g{};
  long long nb = 0;
  void* ds = ds_region(prm, ws, ws_bytes, g, nb);
  if (prm.D == 128) return run_grad_pass<128>(false, a, q, k, v, dO, nullptr, dk, dv, stats, ds, g, nb, st);
  return run_grad_pass<64>(false, a, q, k, v, dO, nullptr, dk, dv, stats, ds, g, nb, st);
}

// 3. dQ (from the stored dS blocks when the workspace holds them, else by
// recomputing S and dP)
int launch_attn_bwd_dq(const usp_attn_params& prm, const void* q, const void* k, const void* v, const float* lse,
                       const void* dO, void* dq, const void* ws, size_t ws_bytes, int32_t* status, cudaStream_t st) {
  const AttnArgs a = make_args(prm, status);
  const float* stats = static_cast<const float*>(ws);
  (void)lse;
  bwd::DsGeom g{};
  long long nb = 0;
  void* ds = ds_region(prm, ws, ws_bytes, g, nb);
  if (prm.D == 128) return run_grad_pass<128>(true, a, q, k, v, dO, dq, nullptr, nullptr, stats, ds, g, nb, st);
  return run_grad_pass<64>(true, a, q, k, v, dO, dq, nullptr, nullptr, stats, ds, g, nb, st);
}

int launch_attn_bwd(const usp_attn_params& prm, const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dO, void* dq, void* dk, void* dv, float* dsinks, void* ws,
                    size_t ws_bytes, int32_t* status, cudaStream_t st) {
  int rc;
  if ((rc = launch_attn_bwd_preprocess(prm, o, lse, dO, dsinks, ws, status, st)) != USP_OK) return rc;
  if ((rc = launch_attn_bwd_dkdv(prm, q, k, v, lse, dO, dk, dv, ws, ws_bytes, status, st)) != USP_OK) return rc;
  return launch_attn_bwd_dq(prm, q, k, v, lse, dO, dq, ws, ws_bytes, status, st);
}

}  // namespace usp
