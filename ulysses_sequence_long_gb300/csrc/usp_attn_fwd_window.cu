// usp_attn_fwd_window.cu — attention forward for short causal sliding windows
// (window_left <= 128) at D = 64: the gpt-oss sliding-window layers of
// huggingface/accelerate PR #4209 ("sliding windows keep working").
//
// Same arithmetic as the general forward (usp_attn_fwd.cu): for rank r, query
// head j, token t,
//     LSE_t = ln( sum_{u visible} exp(scale q_t.k_u) + exp(z_{r*hq+j}) )
//     O_t   = sum_{u visible} exp(scale q_t.k_u - LSE_t) v_u
// but scheduled for key ranges of at most two 128-key tiles per 128-row tile,
// where the general kernel spends most of a CTA's life in set-up, first loads
// and epilogue:
//   * persistent: one CTA per SM walks units (rank, key/value head, 128-row
//     query tile); TMEM, barriers and tensor maps are set up once;
//   * a unit's K/V tiles (at most two) are loaded once and serve all G query
//     heads of the key/value head; K/V stages are double-buffered across units
//     so the next unit's tiles land while the current one computes;
//   * two softmax warpgroups take the query heads in pairs (head 2i to group 0,
//     2i+1 to group 1) and share the tensor core;
//   * 32-column chunks that every row of a warp has masked skip the
//     exponentials (about half of the two tiles' columns at window 127), and
//     only chunks a row cuts pay for the per-element mask;
//   * O leaves through the head's Q tile (its S MMAs are done) with one TMA
//     store instead of per-thread row stores.
// Warp roles (320 threads): warps 0-3 softmax group 0, 4-7 group 1 (thread =
// query row = TMEM lane), warp 8 TMA producer, warp 9 MMA issuer (one thread).
// TMEM: S_q [128q, 128q+128), O_q [256 + 64q, 256 + 64q + 64).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "usp_attn_common.cuh"
#include "usp_internal.h"

namespace usp {

namespace fwdw {

constexpr int D = 64;
constexpr int kThreads = 320;
constexpr int kTile = kBM * 128;   // one 128-row tile of 64 bf16 columns (one swizzle atom)
constexpr int kKV = 4;             // K/V stages: two units' worth of (at most) two key tiles
constexpr int kMaxKV = kKV / 2;    // key tiles per unit
constexpr int OFF_Q = 0;           // [2 sets][2 heads] Q tiles
constexpr int OFF_K = OFF_Q + 4 * kTile;
constexpr int OFF_V = OFF_K + kKV * kTile;
constexpr int OFF_BAR = OFF_V + kKV * kTile;
constexpr int SMEM = OFF_BAR + 1024 + 1024;  // barriers + alignment slack
constexpr uint32_t T_O = 256;

struct Bars {
  // per Q set (one head pair); a group's Q tile is reused to stage its O tile
  // for the TMA store, so the set is free once both O tiles have been read
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kKV], v_full[kKV], kv_empty[kKV];
  uint64_t s_full[2], p_full[2], o_final[2];  // per softmax group
  uint64_t o_staged[2];                       // per softmax group: its 4 warps have staged an O tile
  uint64_t mma_done;
  uint32_t tmem;
  int abort;
};

// One unit's geometry, computed identically by every role.
struct Unit {
  int r, kl, t0;  // rank, local key/value head, first query row
  int lo, n_kv;   // first key, key tiles (0: no key to see)
  int rk0, rk1;   // ring step key window
};

__device__ __forceinline__ Unit unit_at(const AttnArgs& p, int n_docs, int u) {
  Unit w;
  const int per = p.P * p.hk;
  const int qt = u / per, rem = u - qt * per;
  w.r = rem / p.hk;
  w.kl = rem - w.r * p.hk;
  w.t0 = qt * kBM;
  int lo, hi;
  key_range(p, n_docs, w.t0, min(w.t0 + kBM, p.BS) - 1, lo, hi);
  w.rk0 = 0;
  w.rk1 = 0x7FFFFFFF;
  if (p.ring > 1) {
    ring_key_window(p, w.t0, w.rk0, w.rk1);
    lo = max(lo, w.rk0);
    hi = min(hi, w.rk1);
  }
  if (p.kv_seq_io) lo &= ~(kBN - 1);  // tiles never straddle a sequence shard
  w.lo = lo;
  w.n_kv = hi > lo ? (hi - lo + kBN - 1) / kBN : 0;
  return w;
}

// 16 packed columns into TMEM (this warp's lanes).
__device__ __forceinline__ void tmem_st16_cols(uint32_t taddr, const uint32_t (&pk)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]), "r"(pk[6]), "r"(pk[7]), "r"(pk[8]),
      "r"(pk[9]), "r"(pk[10]), "r"(pk[11]), "r"(pk[12]), "r"(pk[13]), "r"(pk[14]), "r"(pk[15])
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_window_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                           const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                           AttnArgs p, __nv_bfloat16* o_out, float* lse_out, int n_units) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + OFF_BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_docs = checked_docs(p);
  if (n_docs == 0) return;
  const int G = p.G, n_pairs = (G + 1) / 2;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 2);  // one arrival per softmax group (its O tile has left)
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 4);
      mbar_init(&bars->o_final[s], 1);
      mbar_init(&bars->o_staged[s], 4);
    }
    for (int s = 0; s < kKV; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
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

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      int gk = 0, it = 0;  // key tiles and head pairs issued (ring positions)
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const Unit w = unit_at(p, n_docs, u);
        if (w.n_kv == 0 || w.n_kv > kMaxKV) continue;
        const HeadRef kvh = kv_head_ref(p, w.r, w.kl);
        for (int n = 0; n < w.n_kv; ++n, ++gk) {
          const int st = gk % kKV;
          if (gk >= kKV && !(ok = mbar_wait(&bars->kv_empty[st], ((gk / kKV) - 1) & 1, abort, p.status))) break;
          const int kv0 = w.lo + n * kBN;
          mbar_arrive_expect_tx(&bars->k_full[st], kTile);
          tma_load_rows(smem + OFF_K + st * kTile, &tk, &bars->k_full[st], p, 0, kvh, kv0, p.kv_seq_io != 0);
          mbar_arrive_expect_tx(&bars->v_full[st], kTile);
          tma_load_rows(smem + OFF_V + st * kTile, &tv, &bars->v_full[st], p, 0, kvh, kv0, p.kv_seq_io != 0);
        }
        for (int pr = 0; pr < n_pairs && ok; ++pr, ++it) {
          const int s = it & 1;
          if (it >= 2 && !(ok = mbar_wait(&bars->q_empty[s], ((it >> 1) - 1) & 1, abort, p.status))) break;
          const int nq = min(2, G - 2 * pr);
          mbar_arrive_expect_tx(&bars->q_full[s], nq * kTile);
          for (int q = 0; q < nq; ++q)
            tma_load_rows(smem + OFF_Q + (2 * s + q) * kTile, &tq, &bars->q_full[s], p, 0,
                          q_head_ref(p, w.r, w.kl * G + 2 * pr + q), w.t0);
        }
      }
      // never leave the CTA with copies still landing in its shared memory
      for (int n = max(0, gk - kKV); n < gk; ++n) {
        mbar_wait(&bars->k_full[n % kKV], (n / kKV) & 1, abort, p.status);
        mbar_wait(&bars->v_full[n % kKV], (n / kKV) & 1, abort, p.status);
      }
      for (int i = max(0, it - 2); i < it; ++i) mbar_wait(&bars->q_full[i & 1], (i >> 1) & 1, abort, p.status);
    }
  }
 else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(kBM, D, false, true);
      auto issue_s = [&](int q, int set, int st) {  // S_q = Q_q K^T
        const uint64_t qd = sdesc_sw128(sbase + OFF_Q + (2 * set + q) * kTile, 16, 1024);
        const uint64_t kd = sdesc_sw128(sbase + OFF_K + st * kTile, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + q * kBN, sdesc_add(qd, kk * 32), sdesc_add(kd, kk * 32), idesc_s, kk > 0);
        mma_commit(&bars->s_full[q]);
      };
      auto issue_pv = [&](int q, int st, bool acc) {  // O_q += P_q V (P_q bf16 in TMEM over S_q)
        const uint64_t vd = sdesc_sw128(sbase + OFF_V + st * kTile, kTile, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(tmem + T_O + q * D, tmem + q * kBN + kk * 8, sdesc_add(vd, kk * 16 * 128), idesc_o,
                 (acc || kk > 0) ? 1u : 0u);
      };
      int gk = 0, it = 0, pc[2] = {0, 0};  // key tiles, head pairs, p_full phases per group
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const Unit w = unit_at(p, n_docs, u);
        if (w.n_kv == 0) continue;
        if (w.n_kv > kMaxKV) {  // outside what this schedule holds: the host never sends such a shape
          set_status(p.status, USP_ERR_UNSUPPORTED);
          continue;
        }
        for (int pr = 0; pr < n_pairs && ok; ++pr, ++it) {
          const int set = it & 1, nq = min(2, G - 2 * pr);
          if (!(ok = mbar_wait(&bars->q_full[set], (it >> 1) & 1, abort, p.status))) break;
          if (!(ok = mbar_wait(&bars->k_full[gk % kKV], (gk / kKV) & 1, abort, p.status))) break;
          tc_fence_after();
          for (int q = 0; q < nq; ++q) issue_s(q, set, gk % kKV);
          for (int n = 0; n < w.n_kv && ok; ++n) {
            const int g = gk + n, st = g % kKV;
            if (!(ok = mbar_wait(&bars->v_full[st], (g / kKV) & 1, abort, p.status))) break;
            if (n + 1 < w.n_kv && !(ok = mbar_wait(&bars->k_full[(g + 1) % kKV], ((g + 1) / kKV) & 1, abort,
                                                    p.status)))
              break;
            for (int q = 0; q < nq && ok; ++q) {
              if (!(ok = mbar_wait(&bars->p_full[q], pc[q] & 1, abort, p.status))) break;
              ++pc[q];
              tc_fence_after();
              issue_pv(q, st, n > 0);
              if (n + 1 < w.n_kv)
                issue_s(q, set, (g + 1) % kKV);  // S_q is free once PV_q has read P_q (in order)
              else
                mma_commit(&bars->o_final[q]);
            }
          }
        }
        if (!ok) break;
        for (int n = 0; n < w.n_kv; ++n) mma_commit(&bars->kv_empty[(gk + n) % kKV]);
        gk += w.n_kv;
      }
      // Every MMA issued above has finished before TMEM can be released.
      mma_commit(&bars->mma_done);
      mbar_wait(&bars->mma_done, 0, abort, p.status);
    }
  }
 else {
    // ------------------------------------------------------------ softmax
    const int q = warp >> 2;    // softmax group: heads 2i + q of the unit
    const int row = tid & 127;  // TMEM lane = query row of the tile
    const uint32_t lane_base = tmem + ((static_cast<uint32_t>(warp & 3) * 32) << 16);
    const uint32_t s_tm = lane_base + q * kBN;
    const uint32_t o_tm = lane_base + T_O + q * D;
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
    int sc = 0, oc = 0;  // s_full and o_final phases of this group
    int it = 0;          // head pairs of this CTA (the Q set of pair it is it & 1)
    bool stored = false; // this thread has issued O stores
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const Unit w = unit_at(p, n_docs, u);
      if (w.n_kv > kMaxKV) continue;
      const int t = w.t0 + row;
      const bool row_ok = t < p.BS;
      if (w.n_kv == 0) {
        // no key to see (a ring step whose block lies after these rows): O = 0
        // and LSE = the sink logit alone, or -inf
        for (int g = q; g < G && row_ok; g += 2) {
          const int j = w.kl * G + g;
          const int bb = t / p.S, ss = t - bb * p.S;
          uint4* dst = reinterpret_cast<uint4*>(o_out + row_offset(p, q_head_ref(p, w.r, j), p.hq, p.Hq, t, D));
          for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
          lse_out[(static_cast<size_t>(w.r * p.B + bb) * p.hq + j) * p.S + ss] =
              p.sinks != nullptr ? __ldg(p.sinks + w.r * p.hq + j) : -INFINITY;
        }
        continue;
      }
      int a = 0, b = 0;
      if (row_ok) doc_bounds(p.cu, n_docs, p.BS, t, a, b);
      a = max(a, w.rk0);  // a ring step sees one key/value super-chunk
      b = min(b, w.rk1);
      int vlo, vhi;  // the row's visible keys, as one interval
      visible_keys(t, a, b, p.causal, p.window_left, row_ok, vlo, vhi);
      for (int pr = 0; pr < n_pairs && ok; ++pr, ++it) {
        const int set = it & 1;
        if (2 * pr + q >= G) {  // odd group size: the last pair has one head
          if (row == 0) mbar_arrive(&bars->q_empty[set]);
          continue;
        }
        const int j = w.kl * G + 2 * pr + q;
        const int gh = w.r * p.hq + j;  // global query head: the sink slice of this rank
        float m = -INFINITY, l = 0.f;
        if (p.sinks != nullptr) {
          m = __ldg(p.sinks + gh) * 1.4426950408889634f;
          l = 1.f;
        }
        for (int n = 0; n < w.n_kv && ok; ++n) {
          if (!(ok = mbar_wait(&bars->s_full[q], sc & 1, abort, p.status))) break;
          ++sc;
          tc_fence_after();
          const int kv0 = w.lo + n * kBN;
          const int c_lo = vlo - kv0, c_hi = vhi - kv0;  // visible columns of this tile: [c_lo, c_hi]
          // 32-column chunk c: bit c of vis = some row of this warp sees it
          // (else P is 0 there: no exponentials), bit c of cut = some row
          // does not see all of it (only then a per-element mask).  In a
          // window each row cuts one chunk per tile, so most chunks are clean.
          uint32_t vis = 0, cut = 0;
#pragma unroll
          for (int c = 0; c < kBN / 32; ++c) {
            const int lo_c = c_lo - 32 * c, hi_c = c_hi - 32 * c;
            vis |= (__any_sync(0xffffffffu, lo_c <= hi_c && hi_c >= 0 && lo_c <= 31) ? 1u : 0u) << c;
            cut |= (__any_sync(0xffffffffu, !(lo_c <= 0 && hi_c >= 31)) ? 1u : 0u) << c;
          }
          uint32_t sr[kBN / 32][32];
#pragma unroll
          for (int c = 0; c < kBN / 32; ++c) tmem_ld32(s_tm + c * 32, sr[c]);
          tmem_wait_ld();
          float s[kBN];
          float mx8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
#pragma unroll
          for (int c = 0; c < kBN / 32; ++c) {
#pragma unroll
            for (int e = 0; e < 32; ++e) s[32 * c + e] = __uint_as_float(sr[c][e]);
            if (vis >> c & 1u) {
              if (cut >> c & 1u) {
                const int lo_c = c_lo - 32 * c, hi_c = c_hi - 32 * c;
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (e < lo_c || e > hi_c) s[32 * c + e] = -INFINITY;
              }
#pragma unroll
              for (int e = 0; e < 32; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], s[32 * c + e]);
            }
          }
          const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                 fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
          const float m_tile = mx * p.scale_log2;  // -inf stays -inf
          const float m_new = fmaxf(m, m_tile);
          const bool need = m_new > m + 8.f;  // lazy rescale: only when the max grows by more than 2^8
          const bool rescale = __any_sync(0xffffffffu, need);
          const float alpha = need ? ex2(m - m_new) : 1.f;
          if (need) {
            l *= alpha;
            m = m_new;
          }
          const float m_use = (m == -INFINITY) ? 0.f : m;
          const uint64_t nm2 = f2_pack(-m_use, -m_use);
          uint64_t rs2[2] = {0, 0};
#pragma unroll
          // P of chunk c, packed, to the 16 columns at 16c (S is all in registers)
#pragma unroll
          for (int c = 0; c < kBN / 32; ++c) {
            uint32_t pk[16];
            if (vis >> c & 1u) {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int col = 32 * c + 2 * e;
                const float2 x = f2_unpack(f2_fma(f2_pack(s[col], s[col + 1]), sc2, nm2));
                const float p0 = ex2(x.x), p1 = ex2(x.y);
                rs2[e & 1] = f2_add(rs2[e & 1], f2_pack(p0, p1));
                pk[e] = pack_bf16x2(p0, p1);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) pk[e] = 0u;
            }
            tmem_st16_cols(s_tm + 16 * c, pk);
          }
          const float2 r01 = f2_unpack(f2_add(rs2[0], rs2[1]));
          l += r01.x + r01.y;
          // The running max moved for some row of this warp: rescale the O
          // rows.  PV of the previous tile has finished (S of this tile was
          // issued after it), and PV of this tile waits for this warp below.
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
        // ---- epilogue of this head: O /= l, bf16 out; LSE = ln(sum) with the sink
        if (!ok || !(ok = mbar_wait(&bars->o_final[q], oc & 1, abort, p.status))) break;
        ++oc;
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        // O goes through this head's Q tile (its MMAs are done) in the
        // 128-byte swizzle of the tensor map: 16-byte chunk e of row r at
        // r*128 + (e ^ r%8)*16, conflict-free; one TMA store writes the tile.
        // (The next head's first PV overwrites these O columns only after this
        // warp hands in that head's P, which follows these loads.)
        uint8_t* stg = smem + OFF_Q + (2 * set + q) * kTile;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(o_tm + c * 32, ov);
          tmem_wait_ld();
          uint32_t pkd[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pkd[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv_l, __uint_as_float(ov[2 * e + 1]) * inv_l);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            *reinterpret_cast<uint4*>(stg + row * 128 + (((4 * c + k4) ^ (row & 7)) << 4)) =
                make_uint4(pkd[4 * k4], pkd[4 * k4 + 1], pkd[4 * k4 + 2], pkd[4 * k4 + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->o_staged[q]);
        if (row == 0 && mbar_wait(&bars->o_staged[q], (oc - 1) & 1, abort, p.status)) {
          tma_store_rows(&to, stg, p, 0, q_head_ref(p, w.r, j), w.t0);
          bulk_commit_group();
          bulk_wait_group_read<0>();  // the tile has been read: the Q set may be reloaded
          mbar_arrive(&bars->q_empty[set]);
          stored = true;
        }
        __syncwarp();
        if (*abort) {  // a wait gave up: the whole warp leaves (the others see it at their next wait)
          ok = false;
          break;
        }
        if (row_ok) {
          const int bb = t / p.S, ss = t - bb * p.S;
          lse_out[(static_cast<size_t>(w.r * p.B + bb) * p.hq + j) * p.S + ss] =
              l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
      }
    }
    if (stored) bulk_wait_group_all();  // the O stores are complete before the CTA ends
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fwdw

bool fwd_window_fits(const AttnArgs& a, int D) {
  // causal, window_left <= 128: a 128-row tile meets at most two key tiles
  return D == fwdw::D && a.causal && a.window_left >= 0 && a.window_left <= kBN;
}

int run_fwd_window(const AttnArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, void* o,
                   float* lse, cudaStream_t st) {
  const int n_tiles = (a.BS + kBM - 1) / kBM;
  const int n_units = n_tiles * a.P * a.hk;
  CUtensorMap to;  // O: same geometry as q
  int rc;
  if ((rc = make_rows_tmap(&to, o, a, a.hq, a.Hq, fwdw::D, kBM)) != USP_OK) return rc;
  if (cudaFuncSetAttribute(fwdw::attn_fwd_window_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, fwdw::SMEM) !=
      cudaSuccess)
    return USP_ERR_CUDA;
  const int sms = device_sm_count();
  const int grid = n_units < sms ? n_units : sms;  // persistent: one CTA per SM
  fwdw::attn_fwd_window_kernel<<<grid, fwdw::kThreads, fwdw::SMEM, st>>>(
      tq, tk, tv, to, a, static_cast<__nv_bfloat16*>(o), lse, n_units);
  return check_launch();
}

}  // namespace usp
