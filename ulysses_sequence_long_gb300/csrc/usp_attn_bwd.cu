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
// Four launches:
//   1. preprocess   D_t for every (rank, query head, token): fp32 workspace
//   2. dK/dV        CTA = (rank, kv head, 128 keys); loops over the group's
//                   query heads and the 128-row query tiles that see the keys:
//                     S^T = K Q^T, dP^T = V dO^T            (TMEM, fp32)
//                     P^T, dS^T -> bf16 in TMEM over S^T / dP^T
//                     dV += P^T dO, dK += dS^T Q           (A operand from TMEM)
//   3. dQ           CTA = (rank, query head, 128 rows); loops over key tiles:
//                     S = Q K^T, dP = dO V^T, dS -> bf16 in TMEM, dQ += dS K
//   4. dsink        one block per (rank, head): a fixed-order tree reduction
// (1 and 4 form the preprocess phase; each phase has its own entry point.)
// Warp roles in 2 and 3 (320 threads): warps 0-7 compute (warp w owns TMEM lanes
// 32*(w%4).. and column half w/4 of every 128-column tile), warp 8 feeds
// shared memory (TMA), warp 9 issues the MMAs from one thread.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "usp_attn_common.cuh"
#include "usp_internal.h"

namespace usp {

namespace bwd {

constexpr int kThreads = 320;
constexpr int kAtomBytes = kBM * 128;
constexpr float kLog2e = 1.4426950408889634f;

// index of (rank r, local head j, rank-local token t) in a [P][B][hq][S] array
__device__ __forceinline__ size_t stat_index(const AttnArgs& p, int r, int j, int t) {
  const int b = t / p.S, s = t - b * p.S;
  return (static_cast<size_t>(r * p.B + b) * p.hq + j) * p.S + s;
}

// --------------------------------------------------------------- preprocess
// One row = D bf16 = D/8 lanes of 16 bytes.  Rows are (rank, token, head) in
// head-layout order, so reads are contiguous.  Output: one 16-byte record per
// (rank, head, token), {LSE*log2(e), D, 0, 0}, laid out [P][hq][B*S] so that a
// 128-token tile of one head is one contiguous 2 KB box for TMA.
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dO,
                                                         const float* __restrict__ lse, float4* __restrict__ stats,
                                                         AttnArgs p, uint32_t n_rows) {
  constexpr int LPR = D / 8;  // lanes per row
  const uint32_t lane_row = threadIdx.x % LPR;
  for (uint32_t row = (blockIdx.x * blockDim.x + threadIdx.x) / LPR; row < n_rows + (32 / LPR);
       row += gridDim.x * blockDim.x / LPR) {
    const bool ok = row < n_rows;
    float acc = 0.f;
    if (ok) {
      const uint4 a = __ldg(o + static_cast<size_t>(row) * LPR + lane_row);
      const uint4 b = __ldg(dO + static_cast<size_t>(row) * LPR + lane_row);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) acc += bf16lo(av[e]) * bf16lo(bv[e]) + bf16hi(av[e]) * bf16hi(bv[e]);
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (ok && lane_row == 0) {
      const uint32_t j = row % p.hq;
      const uint32_t rt = row / p.hq;
      const uint32_t r = rt / p.BS, t = rt - r * p.BS;
      const float l2 = __ldg(lse + stat_index(p, r, j, t)) * kLog2e;
      stats[(static_cast<size_t>(r) * p.hq + j) * p.BS + t] = make_float4(l2, acc, 0.f, 0.f);
    }
  }
}

// --------------------------------------------------------------- dsink
__global__ void __launch_bounds__(256) dsink_kernel(const float4* __restrict__ stats, float* __restrict__ dsinks,
                                                    AttnArgs p) {
  __shared__ float red[256];
  const int r = blockIdx.x / p.hq, j = blockIdx.x % p.hq;
  const float z2 = __ldg(p.sinks + r * p.hq + j) * kLog2e;
  const float4* row = stats + (static_cast<size_t>(r) * p.hq + j) * p.BS;
  float acc = 0.f;
  for (int t = threadIdx.x; t < p.BS; t += blockDim.x) {
    const float4 st = __ldg(row + t);
    acc -= ex2(z2 - st.x) * st.y;
  }
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) dsinks[r * p.hq + j] = red[0];
}

// --------------------------------------------------------------- helpers
__device__ __forceinline__ void ld64(uint32_t taddr, float (&x)[64]) {
  uint32_t a[32], b[32];
  tmem_ld32(taddr, a);
  tmem_ld32(taddr + 32, b);
  tmem_wait_ld();
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    x[e] = __uint_as_float(a[e]);
    x[32 + e] = __uint_as_float(b[e]);
  }
}

__device__ __forceinline__ void st_packed64(uint32_t taddr, const float (&x)[64]) {
  uint32_t pk[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) pk[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
  tmem_st32(taddr, pk);
  tmem_wait_st();
}

// Write one TMEM row (D fp32 columns at `taddr`) times `mul` as bf16 to `dst` (if `ok`).
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

// Both gradient kernels work on 64-wide slices of the 128-lane tiles and keep
// two slices in TMEM at once (buffers 0 and 1): while compute group g forms
// P and dS for its slice, the tensor core computes the other group's next
// slice and the gradient products of the previous one.
constexpr int kSL = 64;                        // slice width (queries in dK/dV, keys in dQ)
constexpr int kSliceBytes = kSL * 128;          // one 64-row, 128-byte-wide swizzle column

template <int D>
struct Cfg {
  static constexpr int NCH = D / 64;
  static constexpr int TILE = NCH * kAtomBytes;   // 128-row bf16 tile
  static constexpr int SLICE = NCH * kSliceBytes;  // 64-row bf16 tile
  static constexpr int STAT = kSL * 16;           // 64 records {LSE*log2e, D, 0, 0}
  // dK/dV: K, V (128 keys) once; ring of (Q, dO, stats) 64-query slices
  static constexpr int QST = (D == 128) ? 4 : 8;
  static constexpr int A_K = 0;
  static constexpr int A_V = A_K + TILE;
  static constexpr int A_Q = A_V + TILE;
  static constexpr int A_DO = A_Q + QST * SLICE;
  static constexpr int A_STAT = A_DO + QST * SLICE;
  static constexpr int A_BAR = A_STAT + QST * STAT;
  static constexpr int A_SMEM = A_BAR + 1024 + 1024;
  // dQ: Q, dO (128 rows) once; ring of (K, V) 64-key slices
  static constexpr int KST = (D == 128) ? 4 : 8;
  static constexpr int B_Q = 0;
  static constexpr int B_DO = B_Q + TILE;
  static constexpr int B_K = B_DO + TILE;
  static constexpr int B_V = B_K + KST * SLICE;
  static constexpr int B_BAR = B_V + KST * SLICE;
  static constexpr int B_SMEM = B_BAR + 1024 + 1024;
};

struct BarsA {
  uint64_t kv_full;
  uint64_t qdo_full[8];
  uint64_t qdo_empty[8];
  uint64_t st_full[2], dpt_full[2], p_full[2], ds_full[2];
  uint64_t fin, mma_done;
  uint32_t tmem;
  int abort;
};

struct BarsB {
  uint64_t q_full;
  uint64_t k_full[8], v_full[8], kv_empty[8];
  uint64_t s_full[2], dp_full[2], ds_full[2];
  uint64_t fin, mma_done;
  uint32_t tmem;
  int abort;
};

struct Grads {
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const float4* stats;  // [P][hq][B*S] {LSE*log2e, D, 0, 0}
  int n_tiles;          // 128-token tiles per rank
};

// K-major operand (rows x D, 128-byte swizzle) of `rows_bytes` per 64-column
// atom, MMA step kk over D.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int atom_bytes, int kk) {
  return sdesc_sw128(base + (kk >> 2) * atom_bytes + (kk & 3) * 32, 16, 1024);
}
// MN-major operand (rows = K dimension, 128-byte rows of D), MMA step kk over rows.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int atom_bytes, int kk) {
  return sdesc_sw128(base + kk * 16 * 128, atom_bytes, 1024);
}

// --------------------------------------------------------------- dK / dV
// CTA = (rank, kv head, 128 keys).  Iteration i covers 64 query rows of one
// query head of the group; buffer b = i & 1 holds S^T_i (TMEM cols 64b..) and
// dP^T_i (128 + 64b..); compute group g = b handles it.  dV at 256, dK at 256+D.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                const __grid_constant__ CUtensorMap tst, AttnArgs p, Grads g) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BarsA* bars = reinterpret_cast<BarsA*>(smem + C::A_BAR);
  const float4* stat = reinterpret_cast<const float4*>(smem + C::A_STAT);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // key tiles in order (early keys of a causal document see the most queries)
  const int per = p.P * p.hk;
  const int kt = static_cast<int>(blockIdx.x) / per;
  const int rem = static_cast<int>(blockIdx.x) % per;
  const int r = rem / p.hk, kh = rem % p.hk;
  const int u0 = kt * kBN;

  const int n_docs = checked_docs(p);
  if (n_docs == 0) return;
  int qlo, qhi;
  query_range(p, n_docs, u0, min(u0 + kBN, p.BS) - 1, qlo, qhi);
  const int n_q = (qhi - qlo + kSL - 1) / kSL;
  const int n_it = p.G * n_q;

  if (tid == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < C::QST; ++s) {
      mbar_init(&bars->qdo_full[s], 1);
      mbar_init(&bars->qdo_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->st_full[b], 1);
      mbar_init(&bars->dpt_full[b], 1);
      mbar_init(&bars->p_full[b], 4);
      mbar_init(&bars->ds_full[b], 4);
    }
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
  constexpr uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + D;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tdo);
      prefetch_tmap(&tst);
      mbar_arrive_expect_tx(&bars->kv_full, 2 * C::TILE);
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_4d(smem + C::A_K + c * kAtomBytes, &tk, &bars->kv_full, c * 64, kh, u0, r);
        tma_load_4d(smem + C::A_V + c * kAtomBytes, &tv, &bars->kv_full, c * 64, kh, u0, r);
      }
      int issued = 0;
      for (int i = 0; i < n_it; ++i) {
        const int s = i % C::QST;
        if (i >= C::QST && !mbar_wait(&bars->qdo_empty[s], ((i / C::QST) - 1) & 1, abort, p.status)) break;
        const int jq = kh * p.G + i / n_q;
        const int q0 = qlo + (i % n_q) * kSL;
        mbar_arrive_expect_tx(&bars->qdo_full[s], 2 * C::SLICE + C::STAT);
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_4d(smem + C::A_Q + s * C::SLICE + c * kSliceBytes, &tq, &bars->qdo_full[s], c * 64, jq, q0, r);
          tma_load_4d(smem + C::A_DO + s * C::SLICE + c * kSliceBytes, &tdo, &bars->qdo_full[s], c * 64, jq, q0, r);
        }
        tma_load_3d(smem + C::A_STAT + s * C::STAT, &tst, &bars->qdo_full[s], 0, q0, r * p.hq + jq);
        issued = i + 1;
      }
      mbar_wait(&bars->kv_full, 0, abort, p.status);
      for (int i = max(0, issued - C::QST); i < issued; ++i)
        mbar_wait(&bars->qdo_full[i % C::QST], (i / C::QST) & 1, abort, p.status);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(kBN, kSL, false, false);  // [128 keys x 64 queries], K = D
      constexpr uint32_t id_g = idesc_bf16(kBN, D, false, true);      // [128 keys x D], K = 64 queries
      // S^T_i = K Q_i^T and dP^T_i = V dO_i^T into buffer i&1
      auto issue_front = [&](int i) -> bool {
        const int s = i % C::QST, b = i & 1;
        if (!mbar_wait(&bars->qdo_full[s], (i / C::QST) & 1, abort, p.status)) return false;
        tc_fence_after();
        const uint32_t qa = sbase + C::A_Q + s * C::SLICE, da = sbase + C::A_DO + s * C::SLICE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + T_S + b * kSL, kmajor_desc(sbase + C::A_K, kAtomBytes, kk), kmajor_desc(qa, kSliceBytes, kk),
                 id_s, kk > 0);
        mma_commit(&bars->st_full[b]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + T_DP + b * kSL, kmajor_desc(sbase + C::A_V, kAtomBytes, kk), kmajor_desc(da, kSliceBytes, kk),
                 id_s, kk > 0);
        mma_commit(&bars->dpt_full[b]);
        return true;
      };
      bool ok = mbar_wait(&bars->kv_full, 0, abort, p.status);
      for (int i = 0; i < 2 && i < n_it && ok; ++i) ok = issue_front(i);
      for (int i = 0; i < n_it && ok; ++i) {
        const int s = i % C::QST, b = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        // dV += P^T_i dO_i  (A: packed bf16 P^T in TMEM cols 64b..64b+32)
        if (!(ok = mbar_wait(&bars->p_full[b], ph, abort, p.status))) break;
        tc_fence_after();
        const uint32_t da = sbase + C::A_DO + s * C::SLICE, qa = sbase + C::A_Q + s * C::SLICE;
#pragma unroll
        for (int kk = 0; kk < kSL / 16; ++kk)
          mma_ts(tmem + T_DV, tmem + T_S + b * kSL + kk * 8, mnmajor_desc(da, kSliceBytes, kk), id_g,
                 (i > 0 || kk > 0) ? 1u : 0u);
        // dK += dS^T_i Q_i
        if (!(ok = mbar_wait(&bars->ds_full[b], ph, abort, p.status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kSL / 16; ++kk)
          mma_ts(tmem + T_DK, tmem + T_DP + b * kSL + kk * 8, mnmajor_desc(qa, kSliceBytes, kk), id_g,
                 (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->qdo_empty[s]);
        if (i + 2 < n_it)
          ok = issue_front(i + 2);
        if (i == n_it - 1) mma_commit(&bars->fin);
      }
      mma_commit(&bars->mma_done);
      mbar_wait(&bars->mma_done, 0, abort, p.status);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int grp = warp >> 2;                      // handles iterations i with i & 1 == grp
    const int krow = (warp & 3) * 32 + lane;        // TMEM lane = key row
    const int u = u0 + krow;
    const bool key_ok = u < p.BS;
    int a = 0, b = 0;
    if (key_ok) doc_bounds(p.cu, n_docs, p.BS, u, a, b);
    const uint32_t lb = tmem + ((static_cast<uint32_t>(warp & 3) * 32) << 16);
    const uint32_t s_col = T_S + grp * kSL, dp_col = T_DP + grp * kSL;
    bool ok = true;
    for (int i = grp; i < n_it && ok; i += 2) {
      const int s = i % C::QST;
      const uint32_t ph = (i >> 1) & 1;
      const int q0 = qlo + (i % n_q) * kSL;  // first query of the slice
      if (!(ok = mbar_wait(&bars->qdo_full[s], (i / C::QST) & 1, abort, p.status))) break;
      const float4* st4 = stat + s * kSL;
      if (!(ok = mbar_wait(&bars->st_full[grp], ph, abort, p.status))) break;
      tc_fence_after();
      float x[64];
      ld64(lb + s_col, x);
      bool full = key_ok && q0 >= a && q0 + kSL <= b && (!p.causal || q0 >= u);
      if (p.window_left >= 0) full = full && (q0 + kSL - 1 - u <= p.window_left) && (p.causal || u - q0 <= p.window_left);
      float pr[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const bool vis = full || (key_ok && visible_from_key(q0 + c, u, a, b, p.causal, p.window_left));
        pr[c] = vis ? ex2(fmaf(x[c], p.scale_log2, -st4[c].x)) : 0.f;
      }
      st_packed64(lb + s_col, pr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[grp]);
      if (!(ok = mbar_wait(&bars->dpt_full[grp], ph, abort, p.status))) break;
      tc_fence_after();
      ld64(lb + dp_col, x);
#pragma unroll
      for (int c = 0; c < 64; ++c) x[c] = pr[c] * (x[c] - st4[c].y);
      st_packed64(lb + dp_col, x);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ds_full[grp]);
    }
    if (ok && n_it > 0 && (ok = mbar_wait(&bars->fin, 0, abort, p.status))) {
      tc_fence_after();
      const size_t row = (static_cast<size_t>(r) * p.BS + (key_ok ? u : 0)) * p.hk + kh;
      if (grp == 0)
        store_row<D>(lb + T_DV, g.dv + row * D, 1.f, key_ok);
      else
        store_row<D>(lb + T_DK, g.dk + row * D, p.scale, key_ok);
    } else if (ok && n_it == 0 && key_ok) {
      const size_t row = (static_cast<size_t>(r) * p.BS + u) * p.hk + kh;
      __nv_bfloat16* dst = (grp == 0 ? g.dv : g.dk) + row * D;
      for (int e = 0; e < D; e += 8) *reinterpret_cast<uint4*>(dst + e) = make_uint4(0, 0, 0, 0);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// --------------------------------------------------------------- dQ
// CTA = (rank, query head, 128 rows).  Iteration n covers 64 keys; buffer
// b = n & 1 holds S_n (TMEM cols 64b..) and dP_n (128 + 64b..); compute group
// g = b handles it.  dQ accumulates at 256.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo, AttnArgs p, Grads g) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BarsB* bars = reinterpret_cast<BarsB*>(smem + C::B_BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // late query tiles first (they see the most keys)
  const int per = p.P * p.hq;
  const int qt = g.n_tiles - 1 - static_cast<int>(blockIdx.x) / per;
  const int rem = static_cast<int>(blockIdx.x) % per;
  const int r = rem / p.hq, j = rem % p.hq, kvh = j / p.G;
  const int t0 = qt * kBM;

  const int n_docs = checked_docs(p);
  if (n_docs == 0) return;
  int lo, hi;
  key_range(p, n_docs, t0, min(t0 + kBM, p.BS) - 1, lo, hi);
  const int n_kv = (hi - lo + kSL - 1) / kSL;

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->dp_full[b], 1);
      mbar_init(&bars->ds_full[b], 4);
    }
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
  constexpr uint32_t T_S = 0, T_DP = 128, T_DQ = 256;

  if (warp == 8) {
    if (lane == 0) {
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      mbar_arrive_expect_tx(&bars->q_full, 2 * C::TILE);
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_4d(smem + C::B_Q + c * kAtomBytes, &tq, &bars->q_full, c * 64, j, t0, r);
        tma_load_4d(smem + C::B_DO + c * kAtomBytes, &tdo, &bars->q_full, c * 64, j, t0, r);
      }
      int issued = 0;
      for (int n = 0; n < n_kv; ++n) {
        const int s = n % C::KST;
        if (n >= C::KST && !mbar_wait(&bars->kv_empty[s], ((n / C::KST) - 1) & 1, abort, p.status)) break;
        const int kv0 = lo + n * kSL;
        mbar_arrive_expect_tx(&bars->k_full[s], C::SLICE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(smem + C::B_K + s * C::SLICE + c * kSliceBytes, &tk, &bars->k_full[s], c * 64, kvh, kv0, r);
        mbar_arrive_expect_tx(&bars->v_full[s], C::SLICE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(smem + C::B_V + s * C::SLICE + c * kSliceBytes, &tv, &bars->v_full[s], c * 64, kvh, kv0, r);
        issued = n + 1;
      }
      mbar_wait(&bars->q_full, 0, abort, p.status);
      for (int n = max(0, issued - C::KST); n < issued; ++n) {
        mbar_wait(&bars->k_full[n % C::KST], (n / C::KST) & 1, abort, p.status);
        mbar_wait(&bars->v_full[n % C::KST], (n / C::KST) & 1, abort, p.status);
      }
    }
  } else if (warp == 9) {
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(kBM, kSL, false, false);  // [128 rows x 64 keys], K = D
      constexpr uint32_t id_q = idesc_bf16(kBM, D, false, true);      // [128 rows x D], K = 64 keys
      auto issue_front = [&](int n) -> bool {
        const int s = n % C::KST, b = n & 1;
        const uint32_t ph = (n / C::KST) & 1;
        if (!mbar_wait(&bars->k_full[s], ph, abort, p.status)) return false;
        tc_fence_after();
        const uint32_t ka = sbase + C::B_K + s * C::SLICE, va = sbase + C::B_V + s * C::SLICE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + T_S + b * kSL, kmajor_desc(sbase + C::B_Q, kAtomBytes, kk), kmajor_desc(ka, kSliceBytes, kk),
                 id_s, kk > 0);
        mma_commit(&bars->s_full[b]);
        if (!mbar_wait(&bars->v_full[s], ph, abort, p.status)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + T_DP + b * kSL, kmajor_desc(sbase + C::B_DO, kAtomBytes, kk), kmajor_desc(va, kSliceBytes, kk),
                 id_s, kk > 0);
        mma_commit(&bars->dp_full[b]);
        return true;
      };
      bool ok = mbar_wait(&bars->q_full, 0, abort, p.status);
      for (int n = 0; n < 2 && n < n_kv && ok; ++n) ok = issue_front(n);
      for (int n = 0; n < n_kv && ok; ++n) {
        const int s = n % C::KST, b = n & 1;
        if (!(ok = mbar_wait(&bars->ds_full[b], (n >> 1) & 1, abort, p.status))) break;
        tc_fence_after();
        const uint32_t ka = sbase + C::B_K + s * C::SLICE;
#pragma unroll
        for (int kk = 0; kk < kSL / 16; ++kk)
          mma_ts(tmem + T_DQ, tmem + T_S + b * kSL + kk * 8, mnmajor_desc(ka, kSliceBytes, kk), id_q,
                 (n > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->kv_empty[s]);
        if (n + 2 < n_kv) ok = issue_front(n + 2);
        if (n == n_kv - 1) mma_commit(&bars->fin);
      }
      mma_commit(&bars->mma_done);
      mbar_wait(&bars->mma_done, 0, abort, p.status);
    }
  } else {
    const int grp = warp >> 2;             // handles iterations n with n & 1 == grp
    const int row = (warp & 3) * 32 + lane;
    const int t = t0 + row;
    const bool row_ok = t < p.BS;
    int a = 0, b = 0;
    float lse2 = INFINITY, dvt = 0.f;
    if (row_ok) {
      doc_bounds(p.cu, n_docs, p.BS, t, a, b);
      const float4 st = __ldg(g.stats + (static_cast<size_t>(r) * p.hq + j) * p.BS + t);
      lse2 = st.x;
      dvt = st.y;
    }
    const uint32_t lb = tmem + ((static_cast<uint32_t>(warp & 3) * 32) << 16);
    const uint32_t s_col = T_S + grp * kSL, dp_col = T_DP + grp * kSL;
    bool ok = true;
    for (int n = grp; n < n_kv && ok; n += 2) {
      const uint32_t ph = (n >> 1) & 1;
      const int k0 = lo + n * kSL;
      if (!(ok = mbar_wait(&bars->s_full[grp], ph, abort, p.status))) break;
      tc_fence_after();
      float x[64];
      ld64(lb + s_col, x);
      bool full = row_ok && k0 >= a && k0 + kSL <= b && (!p.causal || k0 + kSL - 1 <= t);
      if (p.window_left >= 0) full = full && (t - k0 <= p.window_left) && (p.causal || k0 + kSL - 1 - t <= p.window_left);
      float pr[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const bool vis = full || (row_ok && visible(t, k0 + c, a, b, p.causal, p.window_left));
        pr[c] = vis ? ex2(fmaf(x[c], p.scale_log2, -lse2)) : 0.f;
      }
      if (!(ok = mbar_wait(&bars->dp_full[grp], ph, abort, p.status))) break;
      tc_fence_after();
      ld64(lb + dp_col, x);
#pragma unroll
      for (int c = 0; c < 64; ++c) x[c] = pr[c] * (x[c] - dvt);
      st_packed64(lb + s_col, x);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ds_full[grp]);
    }
    if (ok && n_kv > 0 && (ok = mbar_wait(&bars->fin, 0, abort, p.status))) {
      tc_fence_after();
      __nv_bfloat16* dst = g.dq + ((static_cast<size_t>(r) * p.BS + (row_ok ? t : 0)) * p.hq + j) * D + grp * (D / 2);
      store_row<D / 2>(lb + T_DQ + grp * (D / 2), dst, p.scale, row_ok);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace bwd

size_t attn_bwd_ws_bytes(const usp_attn_params& p) {
  size_t rows = static_cast<size_t>(p.B) * p.S * p.Hq;  // one {LSE*log2e, D, 0, 0} record per row and head
  return (rows * 16 + 255) / 256 * 256;
}

static AttnArgs make_args(const usp_attn_params& prm, int32_t* status) {
  AttnArgs a;
  a.B = prm.B;
  a.S = prm.S;
  a.BS = prm.B * prm.S;
  a.P = prm.P;
  a.hq = prm.Hq / prm.P;
  a.hk = prm.Hkv / prm.P;
  a.G = prm.Hq / prm.Hkv;
  a.causal = prm.causal ? 1 : 0;
  a.window_left = prm.window_left;
  a.scale = prm.softmax_scale > 0.f ? prm.softmax_scale : 1.0f / sqrtf(static_cast<float>(prm.D));
  a.scale_log2 = a.scale * 1.4426950408889634f;
  a.cu = prm.cu_seqlens;
  a.n_docs = prm.n_docs;
  a.sinks = prm.sinks;
  a.status = status;
  return a;
}

// 1. D = rowsum(dO * O) into the workspace, then the sink gradients.
int launch_attn_bwd_preprocess(const usp_attn_params& prm, const void* o, const float* lse, const void* dO,
                               float* dsinks, void* ws, int32_t* status, cudaStream_t st) {
  const AttnArgs a = make_args(prm, status);
  float4* stats = static_cast<float4*>(ws);
  const uint32_t n_rows = static_cast<uint32_t>(static_cast<uint64_t>(a.P) * a.BS * a.hq);
  const int per_block = 256 / (prm.D / 8);
  int grid = static_cast<int>((n_rows + per_block - 1) / per_block);
  grid = grid < device_sm_count() * 8 ? grid : device_sm_count() * 8;
  if (prm.D == 128)
    bwd::preprocess_kernel<128><<<grid, 256, 0, st>>>(static_cast<const uint4*>(o), static_cast<const uint4*>(dO),
                                                      lse, stats, a, n_rows);
  else
    bwd::preprocess_kernel<64><<<grid, 256, 0, st>>>(static_cast<const uint4*>(o), static_cast<const uint4*>(dO),
                                                     lse, stats, a, n_rows);
  if (check_launch() != USP_OK) return USP_ERR_CUDA;
  if (dsinks != nullptr && a.sinks != nullptr) {
    bwd::dsink_kernel<<<a.P * a.hq, 256, 0, st>>>(stats, dsinks, a);
    if (check_launch() != USP_OK) return USP_ERR_CUDA;
  }
  return USP_OK;
}

template <int D>
static int run_grad_pass(bool dq_pass, const AttnArgs& a, const void* q, const void* k, const void* v,
                         const void* dO, void* dq, void* dk, void* dv, const float4* stats, cudaStream_t st) {
  using C = bwd::Cfg<D>;
  CUtensorMap tq, tk, tv, tdo, tst;
  int rc;
  // dK/dV streams 64-row Q/dO/stats slices past 128-key K/V tiles; dQ streams
  // 64-key K/V slices past 128-row Q/dO tiles.
  const int q_rows = dq_pass ? kBM : bwd::kSL, kv_rows = dq_pass ? bwd::kSL : kBN;
  if ((rc = make_stats_tmap(&tst, stats, a.BS, a.P * a.hq, bwd::kSL)) != USP_OK) return rc;
  if ((rc = make_head_tmap(&tq, q, a.P, a.BS, a.hq, D, q_rows)) != USP_OK) return rc;
  if ((rc = make_head_tmap(&tdo, dO, a.P, a.BS, a.hq, D, q_rows)) != USP_OK) return rc;
  if ((rc = make_head_tmap(&tk, k, a.P, a.BS, a.hk, D, kv_rows)) != USP_OK) return rc;
  if ((rc = make_head_tmap(&tv, v, a.P, a.BS, a.hk, D, kv_rows)) != USP_OK) return rc;
  bwd::Grads g{static_cast<__nv_bfloat16*>(dq), static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), stats,
               (a.BS + kBM - 1) / kBM};
  if (!dq_pass) {
    if (cudaFuncSetAttribute(bwd::dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::A_SMEM) !=
        cudaSuccess)
      return USP_ERR_CUDA;
    bwd::dkdv_kernel<D><<<static_cast<unsigned>(g.n_tiles) * a.P * a.hk, bwd::kThreads, C::A_SMEM, st>>>(
        tq, tk, tv, tdo, tst, a, g);
  } else {
    if (cudaFuncSetAttribute(bwd::dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::B_SMEM) != cudaSuccess)
      return USP_ERR_CUDA;
    bwd::dq_kernel<D><<<static_cast<unsigned>(g.n_tiles) * a.P * a.hq, bwd::kThreads, C::B_SMEM, st>>>(tq, tk, tv,
                                                                                                       tdo, a, g);
  }
  return check_launch();
}

// 2. dK, dV
int launch_attn_bwd_dkdv(const usp_attn_params& prm, const void* q, const void* k, const void* v, const float* lse,
                         const void* dO, void* dk, void* dv, const void* ws, int32_t* status, cudaStream_t st) {
  const AttnArgs a = make_args(prm, status);
  const float4* stats = static_cast<const float4*>(ws);
  (void)lse;  // read through the preprocess's records
  if (prm.D == 128) return run_grad_pass<128>(false, a, q, k, v, dO, nullptr, dk, dv, stats, st);
  return run_grad_pass<64>(false, a, q, k, v, dO, nullptr, dk, dv, stats, st);
}

// 3. dQ
int launch_attn_bwd_dq(const usp_attn_params& prm, const void* q, const void* k, const void* v, const float* lse,
                       const void* dO, void* dq, const void* ws, int32_t* status, cudaStream_t st) {
  const AttnArgs a = make_args(prm, status);
  const float4* stats = static_cast<const float4*>(ws);
  (void)lse;
  if (prm.D == 128) return run_grad_pass<128>(true, a, q, k, v, dO, dq, nullptr, nullptr, stats, st);
  return run_grad_pass<64>(true, a, q, k, v, dO, dq, nullptr, nullptr, stats, st);
}

int launch_attn_bwd(const usp_attn_params& prm, const void* q, const void* k, const void* v, const void* o,
                    const float* lse, const void* dO, void* dq, void* dk, void* dv, float* dsinks, void* ws,
                    int32_t* status, cudaStream_t st) {
  int rc;
  if ((rc = launch_attn_bwd_preprocess(prm, o, lse, dO, dsinks, ws, status, st)) != USP_OK) return rc;
  if ((rc = launch_attn_bwd_dkdv(prm, q, k, v, lse, dO, dk, dv, ws, status, st)) != USP_OK) return rc;
  return launch_attn_bwd_dq(prm, q, k, v, lse, dO, dq, ws, status, st);
}

}  // namespace usp
