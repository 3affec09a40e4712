// usp_attn_fwd.cu — varlen causal GQA attention forward on the 5th-generation
// tensor core (tcgen05), one launch for all P emulated ranks.
//
// What it computes (huggingface/accelerate PR #4209: attention runs on the
// gathered sequence of the rank's heads; each head has a single sink logit,
// taken from the slice of the rank's heads; sliding windows and packing keep
// working): for every
// rank r, local query head j, token t,
//     LSE_t = ln( sum_{u visible} exp(scale q_t.k_u) + exp(z_{r*hq+j}) )
//     O_t   = sum_{u visible} exp(scale q_t.k_u - LSE_t) v_u
//
// CTA = one (rank, query head, block of 128*NQT query rows) = NQT 128-row Q
// tiles that share every K/V tile.  Warp roles (NQT = 2: 320 threads):
//   warps 0-3   softmax for Q tile 0 (thread = query row = TMEM lane)
//   warps 4-7   softmax for Q tile 1 (NQT = 2)
//   warp  4NQT  TMA producer: Q tiles once, then a ring of K/V stages
//   warp  4NQT+1 MMA issuer (one thread): S_q = Q_q K^T into TMEM, then
//               O_q += P_q V with P_q read from TMEM (bf16, written over S_q)
// TMEM: S_q [128q, 128q+128), O_q [128NQT + qD, 128NQT + (q+1)D) (512 columns
// for NQT = 2).  With two tiles the MMA thread alternates them (PV_0, S_0
// next, PV_1, S_1 next), so the tensor core works on one tile while the other
// tile's softmax runs; with one tile (short windows at D = 64) two CTAs share
// an SM and overlap instead.
//
// Online softmax in the log2 domain with a lazy rescale: the running max only
// moves when a row's new max exceeds it by more than 8 (a factor 256), and the
// O row in TMEM is rescaled then.  Because S_q[n] is committed after
// PV_q[n-1], waiting for S_q[n] also guarantees PV_q[n-1] has finished, so the
// softmax threads may rescale O without another barrier.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "usp_attn_common.cuh"
#include "usp_internal.h"

namespace usp {

namespace fwd {

constexpr int kAtomBytes = kBM * 128;  // one 64-column (128-byte) swizzle column of a 128-row tile
// Stage-release barriers in flight: more than the K/V stages, so that the
// producer's waits (at most ST - 1 releases behind the MMA thread) never see
// a barrier two phases ahead.
constexpr int kRel = 8;

// NQT Q tiles per CTA: 2 (two softmax warpgroups that alternate on the tensor
// core, 512 TMEM columns, one CTA per SM) or 1 (one softmax warpgroup; at
// D = 64 its 192 TMEM columns and 82 KB of shared memory let two CTAs share
// an SM, which then overlap each other's latencies).
template <int D, int NQT>
struct Cfg {
  static constexpr int THREADS = 128 * NQT + 64;      // softmax warpgroups, producer warp, MMA warp
  static constexpr int WP = 4 * NQT;                  // producer warp (the MMA warp is WP + 1)
  static constexpr int CTAS = (NQT == 1 && D == 64) ? 2 : 1;  // CTAs per SM
  static constexpr uint32_t TCOLS = NQT == 2 ? 512 : 256;     // TMEM columns allocated
  static constexpr int NCH = D / 64;                  // 64-wide column atoms per row
  static constexpr int ST = (D == 128 || NQT == 1) ? 2 : 4;  // K/V pipeline stages
  static constexpr bool KV_ONE = ST >= 4;             // one barrier for a stage's K and V
  static constexpr int TILE = NCH * kAtomBytes;       // bytes of one 128-row tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQT * TILE;
  static constexpr int OFF_V = OFF_K + ST * TILE;
  static constexpr int OFF_BAR = OFF_V + ST * TILE;
  static constexpr int SMEM = OFF_BAR + 1024 + 1024;  // barriers + alignment slack
  static constexpr uint32_t T_O = 128 * NQT;          // first O column (S_q at 128q)
};

struct Bars {
  uint64_t q_full[2];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_final[2];
  uint64_t mma_done;
  // Four stages (KV_ONE): kv_full[s] = K and V of the tile in stage s
  // landed (V has time to land before S, so PV needs no wait of its own).
  // Two stages: K_0 signals k_first, and kv_full[m % 2] = V_m and K_{m+1}
  // landed (both are loaded once release m-1 completes, and one wait before
  // PV_m covers them).
  uint64_t kv_full[4], k_first;
  // rel[j % kRel] completes once the MMAs issued up to S_j are done: K_j's
  // stage and V_{j-1}'s (its PV was issued before S_j) are free
  uint64_t rel[8];
  uint32_t tmem;
  int abort;
};

struct Out {
  __nv_bfloat16* o;
  float* lse;
  int nqb;  // query blocks (NQT tiles of 128 rows) per (rank, head)
};

template <int D, int NQT>
__global__ void __launch_bounds__(Cfg<D, NQT>::THREADS, Cfg<D, NQT>::CTAS)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, AttnArgs p, Out out) {
  using C = Cfg<D, NQT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- work unit: late query blocks first (they see the most keys); the
  // query heads of one key/value head are adjacent, so they share K/V in L2.
  const int per_blk = p.P * p.hq;
  const int qb = out.nqb - 1 - static_cast<int>(blockIdx.x) / per_blk;
  const int rem = static_cast<int>(blockIdx.x) % per_blk;
  const int r = rem / p.hq, j = rem % p.hq;
  const HeadRef qh = q_head_ref(p, r, j), kvh = kv_head_ref(p, r, j / p.G);
  const int t0 = qb * NQT * kBM;

  const int n_docs = checked_docs(p);
  if (n_docs == 0) return;

  bool tile_ok[NQT];
  int lo = 0x7FFFFFFF, hi = 0;
  for (int q = 0; q < NQT; ++q) {
    int first = t0 + q * kBM;
    tile_ok[q] = first < p.BS;
    if (tile_ok[q]) {
      int last = min(first + kBM, p.BS) - 1, l0, h0;
      key_range(p, n_docs, first, last, l0, h0);
      lo = min(lo, l0);
      hi = max(hi, h0);
    }
  }
  // Ring x Ulysses step: only the key/value super-chunk held at this step (the
  // CTA's rows lie in one super-chunk).
  int rk0 = 0, rk1 = 0x7FFFFFFF;
  if (p.ring > 1) {
    ring_key_window(p, t0, rk0, rk1);
    lo = max(lo, rk0);
    hi = min(hi, rk1);
  }
  // With k/v read from the sequence shards, key tiles are aligned to 128
  // tokens so that a tile never straddles a shard (keys before the document
  // are masked).
  if (p.kv_seq_io) lo &= ~(kBN - 1);
  const int n_kv = hi > lo ? (hi - lo + kBN - 1) / kBN : 0;
  if (n_kv == 0) {
    // no key to see (a ring step whose block lies after these rows): O = 0 and
    // LSE = the sink logit alone, or -inf
    if (warp < C::WP) {
      const int q = warp >> 2, t = t0 + q * kBM + (tid & 127);
      if (tile_ok[q] && t < p.BS) {
        uint4* dst = reinterpret_cast<uint4*>(out.o + row_offset(p, qh, p.hq, p.Hq, t, D));
        for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
        const int bb = t / p.S, ss = t - bb * p.S;
        out.lse[(static_cast<size_t>(r * p.B + bb) * p.hq + j) * p.S + ss] =
            p.sinks != nullptr ? __ldg(p.sinks + r * p.hq + j) : -INFINITY;
      }
    }
    return;
  }

  if (tid == 0) {
    for (int q = 0; q < NQT; ++q) {
      mbar_init(&bars->q_full[q], 1);
      mbar_init(&bars->s_full[q], 1);
      mbar_init(&bars->p_full[q], 4);
      mbar_init(&bars->o_final[q], 1);
    }
    mbar_init(&bars->mma_done, 1);
    for (int j = 0; j < kRel; ++j) mbar_init(&bars->rel[j], 1);
    mbar_init(&bars->k_first, 1);
    for (int s = 0; s < C::ST; ++s) {
      mbar_init(&bars->kv_full[s], 1);

    }
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem, C::TCOLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  volatile int* abort = &bars->abort;
  const uint32_t sbase = smem_u32(smem);

  if (warp == C::WP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      for (int q = 0; q < NQT; ++q) {
        if (!tile_ok[q]) continue;
        mbar_arrive_expect_tx(&bars->q_full[q], C::TILE);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_rows(smem + C::OFF_Q + q * C::TILE + c * kAtomBytes, &tq, &bars->q_full[q], p, c, qh, t0 + q * kBM);
      }
      auto load = [&](int kv, int n, uint64_t* full) {  // K (kv 0) or V tile n into its stage
        uint8_t* dst = smem + (kv == 0 ? C::OFF_K : C::OFF_V) + (n % C::ST) * C::TILE;
        for (int c = 0; c < C::NCH; ++c)
          tma_load_rows(dst + c * kAtomBytes, kv == 0 ? &tk : &tv, full, p, c, kvh, lo + n * kBN, p.kv_seq_io != 0);
      };
      int issued = 0;  // KV_ONE: tiles whose K and V loads were issued; else V_m (with K_{m+1}) groups
      if constexpr (C::KV_ONE) {
        // K_n and V_n once their stage is free: K_n replaces K_{n-ST} (free
        // after release n-ST), V_n replaces V_{n-ST} (release n-ST+1)
        for (int n = 0; n < n_kv; ++n) {
          const int st = n % C::ST;
          bool ok_n = true;
          for (int kv = 0; kv < 2 && ok_n; ++kv) {
            const int j = n - C::ST + kv;  // the release this load waits for
            if (n >= C::ST && !(ok_n = mbar_wait(&bars->rel[j % kRel], (j / kRel) & 1, abort, p.status))) break;
            if (kv == 0) mbar_arrive_expect_tx(&bars->kv_full[st], 2 * C::TILE);
            load(kv, n, &bars->kv_full[st]);
          }
          if (!ok_n) break;
          issued = n + 1;
        }
        for (int n = max(0, issued - C::ST); n < issued; ++n)
          mbar_wait(&bars->kv_full[n % C::ST], (n / C::ST) & 1, abort, p.status);
      } else {
        // K_0 alone; then V_m with K_{m+1}: V_m replaces V_{m-2} (free after
        // PV_{m-2}), K_{m+1} replaces K_{m-1} (free after S_{m-1}), both by
        // release m-1
        mbar_arrive_expect_tx(&bars->k_first, C::TILE);
        load(0, 0, &bars->k_first);
        for (int m = 0; m < n_kv; ++m) {
          if (m >= 1 && !mbar_wait(&bars->rel[(m - 1) % kRel], ((m - 1) / kRel) & 1, abort, p.status)) break;
          const bool k_next = m + 1 < n_kv;
          uint64_t* full = &bars->kv_full[m & 1];
          mbar_arrive_expect_tx(full, (k_next ? 2 : 1) * C::TILE);
          load(1, m, full);
          if (k_next) load(0, m + 1, full);
          issued = m + 1;
        }
        mbar_wait(&bars->k_first, 0, abort, p.status);
        for (int m = max(0, issued - 2); m < issued; ++m)
          mbar_wait(&bars->kv_full[m & 1], (m >> 1) & 1, abort, p.status);
      }
      // Never leave the CTA with copies still landing in its shared memory (above).
      for (int q = 0; q < NQT; ++q)
        if (tile_ok[q]) mbar_wait(&bars->q_full[q], 0, abort, p.status);
    }
  } else if (warp == C::WP + 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(kBM, D, false, true);
      bool ok = true;
      for (int q = 0; q < NQT && ok; ++q)
        if (tile_ok[q]) ok = mbar_wait(&bars->q_full[q], 0, abort, p.status);
      // descriptors are built once per tile and moved by a constant per MMA step
      auto issue_s = [&](int q, int st) {
        const uint64_t qd = sdesc_sw128(sbase + C::OFF_Q + q * C::TILE, 16, 1024);
        const uint64_t kd = sdesc_sw128(sbase + C::OFF_K + st * C::TILE, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
          mma_ss(tmem + q * kBN, sdesc_add(qd, off), sdesc_add(kd, off), idesc_s, kk > 0);
        }
      };
      // Release j (after S_j): one commit frees K_j and V_{j-1}; only the
      // releases a later load waits for are committed (j - 1 + ST < n_kv).
      auto release = [&](int j) {
        if (j - 1 + C::ST < n_kv) mma_commit(&bars->rel[j % kRel]);
      };
      auto issue_pv = [&](int q, int st, bool acc) {
        const uint64_t vd = sdesc_sw128(sbase + C::OFF_V + st * C::TILE, kAtomBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(tmem + C::T_O + q * D, tmem + q * kBN + kk * 8, sdesc_add(vd, kk * 16 * 128), idesc_o,
                 (acc || kk > 0) ? 1u : 0u);
      };
      if (ok) ok = C::KV_ONE ? mbar_wait(&bars->kv_full[0], 0, abort, p.status)
                             : mbar_wait(&bars->k_first, 0, abort, p.status);
      if (ok) {
        tc_fence_after();
        for (int q = 0; q < NQT; ++q)
          if (tile_ok[q]) {
            issue_s(q, 0);
            mma_commit(&bars->s_full[q]);
          }
        release(0);
      }
      for (int n = 0; n < n_kv && ok; ++n) {
        const int st = n % C::ST;
        // two stages: V_n and K_{n+1} in one wait; KV_ONE: V_n landed with K_n
        if (!C::KV_ONE && !(ok = mbar_wait(&bars->kv_full[n & 1], (n >> 1) & 1, abort, p.status))) break;
        bool next_k_ready = !C::KV_ONE;
        for (int q = 0; q < NQT && ok; ++q) {
          if (!tile_ok[q]) continue;
          if (!(ok = mbar_wait(&bars->p_full[q], n & 1, abort, p.status))) break;
          tc_fence_after();
          issue_pv(q, st, n > 0);
          if (n + 1 < n_kv) {
            if (!next_k_ready) {
              const int st1 = (n + 1) % C::ST;
              if (!(ok = mbar_wait(&bars->kv_full[st1], ((n + 1) / C::ST) & 1, abort, p.status))) break;
              tc_fence_after();
              next_k_ready = true;
            }
            issue_s(q, (n + 1) % C::ST);
            mma_commit(&bars->s_full[q]);
          } else {
            mma_commit(&bars->o_final[q]);
          }
        }
        if (ok && n + 1 < n_kv) release(n + 1);
      }
      // Every MMA issued above has finished before TMEM can be released.
      mma_commit(&bars->mma_done);
      mbar_wait(&bars->mma_done, 0, abort, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int q = warp >> 2;            // which Q tile
    const int row = tid & 127;          // TMEM lane = row of the tile
    const int t = t0 + q * kBM + row;   // rank-local token
    const bool row_ok = t < p.BS;
    const uint32_t lane_base = tmem + ((static_cast<uint32_t>(warp & 3) * 32) << 16);
    const uint32_t s_tm = lane_base + q * kBN;
    const uint32_t o_tm = lane_base + C::T_O + q * D;
    int a = 0, b = 0;
    if (row_ok) doc_bounds(p.cu, n_docs, p.BS, t, a, b);
    a = max(a, rk0);  // a ring step sees one key/value super-chunk
    b = min(b, rk1);
    const int gh = r * p.hq + j;  // global query head: the sink slice of this rank
    float m = -INFINITY, l = 0.f;
    if (p.sinks != nullptr) {
      m = __ldg(p.sinks + gh) * 1.4426950408889634f;
      l = 1.f;
    }
    bool ok = tile_ok[q];
    for (int n = 0; n < n_kv && ok; ++n) {
      if (!(ok = mbar_wait(&bars->s_full[q], n & 1, abort, p.status))) break;
      tc_fence_after();
      uint32_t sr[kBN / 32][32];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) tmem_ld32(s_tm + c * 32, sr[c]);
      tmem_wait_ld();
      float s[kBN];
#pragma unroll
      for (int c = 0; c < kBN; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
      const int kv0 = lo + n * kBN;
      // rows whose keys in this tile are all visible skip the per-element mask
      bool full = row_ok && kv0 >= a && kv0 + kBN <= b && (!p.causal || kv0 + kBN - 1 <= t);
      if (p.window_left >= 0) full = full && (t - kv0 <= p.window_left) && (p.causal || kv0 + kBN - 1 - t <= p.window_left);
      if (!full) {
        int vlo, vhi;  // the row's visible keys, as one interval: two compares per element
        visible_keys(t, a, b, p.causal, p.window_left, row_ok, vlo, vhi);
        const int c_lo = vlo - kv0, c_hi = vhi - kv0;
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (c < c_lo || c > c_hi) s[c] = -INFINITY;
      }
      // row max as 8 independent chains
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = s[e];
#pragma unroll
      for (int c = 8; c < kBN; c += 8)
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(mx8[e], s[c + e]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_tile = mx * p.scale_log2;  // -inf stays -inf
      const float m_new = fmaxf(m, m_tile);
      const bool need = m_new > m + 8.f;
      const bool rescale = __any_sync(0xffffffffu, need);
      const float alpha = need ? ex2(m - m_new) : 1.f;
      if (need) {
        l *= alpha;
        m = m_new;
      }
      const float m_use = (m == -INFINITY) ? 0.f : m;
      uint64_t rs2[4] = {0, 0, 0, 0};  // 8 independent partial sums, two per register
      const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nm2 = f2_pack(-m_use, -m_use);
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // each 64-column half is packed and stored as soon as it is done
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 e = f2_unpack(f2_fma(f2_pack(s[64 * h + 2 * c], s[64 * h + 2 * c + 1]), sc2, nm2));
          const float p0 = ex2(e.x), p1 = ex2(e.y);
          rs2[c & 3] = f2_add(rs2[c & 3], f2_pack(p0, p1));
          pk[c] = pack_bf16x2(p0, p1);
        }
        tmem_st32(s_tm + 32 * h, pk);
      }
      const float2 r01 = f2_unpack(f2_add(rs2[0], rs2[1])), r23 = f2_unpack(f2_add(rs2[2], rs2[3]));
      l += (r01.x + r01.y) + (r23.x + r23.y);
      // The running max moved for some row of this warp: rescale the O rows.
      // PV of the previous tile has finished (S of this tile was committed
      // after it), and PV of this tile waits for this warp's arrival below.
      if (rescale && n > 0) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(o_tm + c * 32, ov);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32(o_tm + c * 32, ov);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[q]);
    }
    // ---- epilogue: O /= l, bf16 out; LSE = ln(sum) including the sink
    if (ok && (ok = mbar_wait(&bars->o_final[q], 0, abort, p.status))) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = out.o + row_offset(p, qh, p.hq, p.Hq, row_ok ? t : 0, D);
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(o_tm + c * 32, ov);
        tmem_wait_ld();
        uint32_t pkd[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pkd[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv_l, __uint_as_float(ov[2 * e + 1]) * inv_l);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pkd[4 * e], pkd[4 * e + 1], pkd[4 * e + 2], pkd[4 * e + 3]);
        }
      }
      if (row_ok) {
        const int bb = t / p.S, ss = t - bb * p.S;
        out.lse[(static_cast<size_t>(r * p.B + bb) * p.hq + j) * p.S + ss] =
            l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TCOLS);
  }
}

}  // namespace fwd

template <int D, int NQT>
static int run_fwd(const AttnArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, void* o,
                   float* lse, cudaStream_t st) {
  using C = fwd::Cfg<D, NQT>;
  fwd::Out out{static_cast<__nv_bfloat16*>(o), lse, (a.BS + NQT * kBM - 1) / (NQT * kBM)};
  if (cudaFuncSetAttribute(fwd::attn_fwd_kernel<D, NQT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
      cudaSuccess)
    return USP_ERR_CUDA;
  const unsigned grid = static_cast<unsigned>(out.nqb) * a.P * a.hq;
  fwd::attn_fwd_kernel<D, NQT><<<grid, C::THREADS, C::SMEM, st>>>(tq, tk, tv, a, out);
  return check_launch();
}

template <int D>
static int run_fwd(const AttnArgs& a, const void* q, const void* k, const void* v, void* o, float* lse,
                   cudaStream_t st) {
  CUtensorMap tq, tk, tv;
  int rc;
  if ((rc = make_rows_tmap(&tq, q, a, a.hq, a.Hq, D, kBM)) != USP_OK) return rc;
  if ((rc = make_rows_tmap(&tk, k, a, a.hk, a.Hkv, D, kBN, a.kv_seq_io != 0)) != USP_OK) return rc;
  if ((rc = make_rows_tmap(&tv, v, a, a.hk, a.Hkv, D, kBN, a.kv_seq_io != 0)) != USP_OK) return rc;
  // Short causal windows at D = 64: the persistent schedule over the heads of
  // a key/value group.  Other short windows at D = 64: one Q tile per CTA (the
  // two tiles of a CTA would share little, and two small CTAs per SM overlap
  // each other's set-up and latencies instead).
  if (fwd_window_fits(a, D)) return run_fwd_window(a, tq, tk, tv, o, lse, st);
  const bool one = D == 64 && a.window_left >= 0 && a.window_left < 4 * kBN;
  return one ? run_fwd<D, 1>(a, tq, tk, tv, o, lse, st) : run_fwd<D, 2>(a, tq, tk, tv, o, lse, st);
}

int launch_attn_fwd(const usp_attn_params& prm, const void* q, const void* k, const void* v, void* o, float* lse,
                    int32_t* status, cudaStream_t st) {
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
  a.seq_io = prm.io_layout != USP_IO_HEAD ? 1 : 0;
  a.kv_seq_io = prm.io_layout == USP_IO_SEQ ? 1 : 0;
  a.ring = prm.ring > 1 ? prm.ring : 1;
  a.ring_step = a.ring > 1 ? prm.ring_step : 0;
  a.C = prm.S / a.ring;
  a.Sl = prm.S / (prm.P * a.ring);  // sequence shard: P Ulysses ranks in each of `ring` groups
  a.kvh0 = 0;
  a.n_kvh = prm.Hkv;
  a.hq0 = 0;
  a.n_qh = prm.Hq;
  if (prm.D == 128) return run_fwd<128>(a, q, k, v, o, lse, st);
  return run_fwd<64>(a, q, k, v, o, lse, st);
}

}  // namespace usp
