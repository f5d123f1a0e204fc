// attn_tc.cu — block attention forward on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA) for sm_103a, bf16 q/k/v, fp32 (out, lse).
//
// What one CTA computes: two 128-row query tiles of one (batch, head) from one
// simulated rank's shard, against the K/V blocks of that rank's ring lap (or
// of one ring step), with the online-softmax state (row max m, row sum l,
// unnormalised output O) carried across K/V tiles and across blocks. Carrying
// the state across a block boundary is exactly the fp32 LSE merge of the two
// blocks' (out, lse) partials: with out_a = O_a / l_a and lse_a = m_a + ln l_a,
//   e^{lse_a - lse} out_a + e^{lse_b - lse} out_b
//     = (e^{m_a} O_a + e^{m_b} O_b) / (e^{m_a} l_a + e^{m_b} l_b),
// which is what rescaling O and l to a common maximum computes.
// (diffusers "Paralelismo de contexto" page, section "Atenção em Anel": each
// GPU attends to the K/V block it holds, then passes it on; the "Paralelismo"
// API page, ContextParallelConfig.convert_to_fp32: fp32 output and LSE.)
//
// Warp roles (320 threads):
//   warp 0        TMA producer (the whole warp runs the loop, an elected lane
//                 issues): Q tile 0, K(0), Q tile 1, then K and V tiles
//                 through a two-stage ring each, 128B-swizzled.
//   warp 1        TMEM allocator and MMA issuer (the whole warp runs the
//                 loop, an elected lane issues and commits):
//                 S_i = Q_i K^T (SS MMA, M=128 N=128 K=16 steps) and
//                 O_i += P_i V (TS MMA, P read from TMEM), ping-ponging the
//                 two query tiles so that one tile's softmax overlaps the
//                 other tile's MMAs.
//   warps 2-5     softmax of query tile 0, warps 6-9 of tile 1 (a warp reads
//                 the TMEM lane quadrant warp id mod 4): one thread
//                 per query row (TMEM lane), row max and sum in registers,
//                 P = 2^(s*scale*log2e - m) rounded to bf16 into TMEM over S
//                 (l sums the rounded P, so out and lse are exact attention of
//                 logits perturbed by at most one bf16 rounding of P). After
//                 the first tile P is computed with the running maximum and
//                 the row sum checks it afterwards; O and l are rescaled only
//                 when the row max grows by more than 2^8 (the stale maximum
//                 is exact: it cancels in O / l).
//                 Epilogue: O / l staged through shared memory and stored
//                 coalesced; lse = (m + log2 l) * ln 2.
// kMasked: the instance that also applies a key-padding mask, packed per K/V
// tile by ballots of the tile's mask bytes.
// Work items: two query tiles each; a shard's leftover odd tile pairs with
// another shard's over a full lap (the decode below).
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+D),
// O_1 [256+D, 256+2D); P_i overwrites the first 64 columns of S_i as packed
// bf16 pairs.
// Every wait is bounded (see cp_ptx.cuh); on expiry the CTA drains its
// in-flight TMA loads and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "cp_internal.h"
#include "cp_ptx.cuh"

namespace cp {

__device__ uint32_t g_dev_error;  // the device error word (see cp_check_device_status)

namespace {

constexpr int kThreads = 320;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale only when the max grows by > 2^8
constexpr uint32_t kTmemCols = 512;

template <int D>
struct Smem {
  static constexpr int kQTile = kTileM * D * 2;   // bytes of one bf16 Q tile
  static constexpr int kKVTile = kTileN * D * 2;  // bytes of one bf16 K or V tile
  static constexpr int kHalf = kTileM * 128;      // one 64-column (128-byte) box of a 128-row tile
  static constexpr int kStages = 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQTile;
  static constexpr int kOffV = kOffK + kStages * kKVTile;
  static constexpr int kOffBar = kOffV + kStages * kKVTile;
  static constexpr int kNumBars = 17;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 64;
  // slack to align the base to 1024 bytes; at least 116 KB so that two CTAs
  // never share an SM (each allocates all 512 TMEM columns)
  static constexpr int kAlloc = (kBytes + 1024) > 116 * 1024 ? (kBytes + 1024) : 116 * 1024;
};

// barrier indices
enum : int {
  kBarQFull = 0,
  kBarKFull = 1,   // +stage
  kBarKEmpty = 3,  // +stage
  kBarVFull = 5,   // +stage
  kBarVEmpty = 7,  // +stage
  kBarSFull = 9,   // +tile
  kBarPFull = 11,  // +tile
  kBarOFull = 13,  // +tile
  kBarDrain = 15,
  kBarQFull1 = 16,  // Q tile 1 (Q tile 0 completes kBarQFull)
};

__device__ __forceinline__ int ring_block(const RingGeom& g, int r, int t) {
  const int s = g.step >= 0 ? g.step : t;
  int j = (r - s) % g.n_kv;
  return j < 0 ? j + g.n_kv : j;
}

// Walks the K/V tiles of rank r's lap in ring order, skipping empty blocks.
struct KvCursor {
  int t, nblk, tile, ntile, off, len;
  __device__ __forceinline__ void init(const RingGeom& g, int r) {
    nblk = g.step >= 0 ? 1 : g.n_kv;
    t = -1;
    next_block(g, r);
  }
  __device__ __forceinline__ void next_block(const RingGeom& g, int r) {
    tile = 0;
    while (true) {
      ++t;
      if (t >= nblk) return;
      const int j = ring_block(g, r, t);
      off = g.kv_off[j];
      len = g.kv_len[j];
      ntile = (len + kTileN - 1) / kTileN;
      if (ntile > 0) return;
    }
  }
  __device__ __forceinline__ int kv0() const { return off + tile * kTileN; }
  __device__ __forceinline__ int nvalid() const { return min(kTileN, len - tile * kTileN); }
  __device__ __forceinline__ void advance(const RingGeom& g, int r) {
    if (++tile >= ntile) next_block(g, r);
  }
};

__device__ __forceinline__ int total_tiles(const RingGeom& g, int r) {
  const int nblk = g.step >= 0 ? 1 : g.n_kv;
  int n = 0;
  for (int t = 0; t < nblk; ++t) n += (g.kv_len[ring_block(g, r, t)] + kTileN - 1) / kTileN;
  return n;
}

// Bounded wait that ignores the abort flag (used while draining).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1; !mbar_try_wait(bar, parity); ++n) {
    if ((n & 255u) == 0 && global_timer_ns() - t0 > timeout_ns) return;
  }
}

template <int D, bool kMasked>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, const __grid_constant__ AttnArgs a) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_addr(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);  // [0] TMEM base, [1] abort flag
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) -> uint32_t { return sb + L::kOffBar + 8 * i; };
  int blk_h, blk_b;

  // ---- work item: all two-tile items of all (head, batch) first, then all
  // one-tile items; items vary fastest, then heads. A shard with an odd tile
  // count leaves its last tile over. Over a whole ring lap every shard visits
  // every K/V block, so two such leftover tiles of different shards share one
  // item (and one K/V stream, in the first shard's ring order); only an odd
  // one out, or any leftover of a single-step launch, runs alone. ----
  const int n_pairs = a.g.pair_prefix[a.g.n_q];
  const int n_single = a.g.single_prefix[a.g.n_q];
  const int n_cross = a.g.step < 0 ? n_single / 2 : 0;
  const int n_two = n_pairs + n_cross;
  const int n_one = n_single - 2 * n_cross;
  // shard holding leftover tile k, and the first row of that tile
  auto leftover = [&](int k, int& shard, int& row0) {
    int rr = 0;
    while (rr + 1 < a.g.n_q && a.g.single_prefix[rr + 1] <= k) ++rr;
    shard = rr;
    row0 = a.g.q_off[rr] + (a.g.pair_prefix[rr + 1] - a.g.pair_prefix[rr]) * 2 * kTileM;
  };
  int id = blockIdx.x;
  int r = 0, nq, qrow[2], rows[2];
  {
    const int64_t two_ctas = static_cast<int64_t>(n_two) * a.H * a.B;
    int item, h_, b_;
    if (id < two_ctas) {
      item = id % n_two;
      h_ = (id / n_two) % a.H;
      b_ = id / (n_two * a.H);
      nq = 2;
      if (item < n_pairs) {
        while (r + 1 < a.g.n_q && a.g.pair_prefix[r + 1] <= item) ++r;
        qrow[0] = a.g.q_off[r] + (item - a.g.pair_prefix[r]) * 2 * kTileM;
        qrow[1] = qrow[0] + kTileM;
        const int rem = a.g.q_off[r] + a.g.q_len[r] - qrow[0];
        rows[0] = min(kTileM, rem);
        rows[1] = min(kTileM, rem - kTileM);
      } else {
        const int k = 2 * (item - n_pairs);
        int r1;
        leftover(k, r, qrow[0]);
        leftover(k + 1, r1, qrow[1]);
        rows[0] = a.g.q_off[r] + a.g.q_len[r] - qrow[0];
        rows[1] = a.g.q_off[r1] + a.g.q_len[r1] - qrow[1];
      }
    } else {
      id -= static_cast<int>(two_ctas);
      item = id % n_one;
      h_ = (id / n_one) % a.H;
      b_ = id / (n_one * a.H);
      nq = 1;
      leftover(2 * n_cross + item, r, qrow[0]);
      qrow[1] = qrow[0];
      rows[0] = a.g.q_off[r] + a.g.q_len[r] - qrow[0];
      rows[1] = 0;
    }
    blk_h = h_;
    blk_b = b_;
  }
  const int h = blk_h, b = blk_b;
  if (attn_head_is_padding(a, h, b)) return;  // uniform per CTA, before any barrier or TMEM
  const int NT = total_tiles(a.g, r);

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNumBars; ++i) mbar_init(bar(i), (i == kBarPFull || i == kBarPFull + 1) ? 4 : 1);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(misc), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const uint64_t tmo = a.timeout_ns;

  if (warp == 0) {
    // ===================== TMA producer =====================
    // The whole warp runs the loop; one elected lane issues the copies.
    const bool leader = elect_one();
    if (NT > 0) {
      if (leader) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
      }
      int k_issued[2] = {0, 0}, v_issued[2] = {0, 0};
      // Q tile 0 and K(0) first, so that S_0(0) can start while Q tile 1
      // is still on its way (each Q tile completes its own barrier)
      auto load_q = [&](int i) {
        if (!leader) return;
        const uint32_t qb = bar(i == 0 ? kBarQFull : kBarQFull1);
        mbar_arrive_expect_tx(qb, L::kQTile);
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d(sb + L::kOffQ + i * L::kQTile + c * L::kHalf, &tq, qb, c * 64, h, qrow[i], b);
      };
      load_q(0);
      KvCursor cur;
      cur.init(a.g, r);
      for (int it = 0; it < NT; ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait_bounded(bar(kBarKEmpty + s), ph ^ 1, abort_flag, a.err, tmo)) break;
        if (leader) {
          mbar_arrive_expect_tx(bar(kBarKFull + s), L::kKVTile);
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(sb + L::kOffK + s * L::kKVTile + c * L::kHalf, &tk, bar(kBarKFull + s), c * 64, h,
                        cur.kv0(), b);
        }
        ++k_issued[s];
        if (it == 0 && nq == 2) load_q(1);
        if (!mbar_wait_bounded(bar(kBarVEmpty + s), ph ^ 1, abort_flag, a.err, tmo)) break;
        if (leader) {
          mbar_arrive_expect_tx(bar(kBarVFull + s), L::kKVTile);
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(sb + L::kOffV + s * L::kKVTile + c * L::kHalf, &tv, bar(kBarVFull + s), c * 64, h,
                        cur.kv0(), b);
        }
        ++v_issued[s];
        cur.advance(a.g, r);
      }
      if (*abort_flag) {
        // let every issued copy land before the CTA's shared memory goes away
        drain_wait(bar(kBarQFull), 0, tmo);
        if (nq == 2 && k_issued[0] > 0) drain_wait(bar(kBarQFull1), 0, tmo);
        for (int s = 0; s < 2; ++s) {
          if (k_issued[s]) drain_wait(bar(kBarKFull + s), (k_issued[s] - 1) & 1, tmo);
          if (v_issued[s]) drain_wait(bar(kBarVFull + s), (v_issued[s] - 1) & 1, tmo);
        }
      }
    }
  } else if (warp == 1) {
    // ===================== MMA issuer =====================
    // The whole warp runs the loop (every operand is warp-uniform); one
    // elected lane issues the MMAs and commits.
    const bool leader = elect_one();
    if (NT > 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kTileM, kTileN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kTileM, D, false, true);
      // Descriptor halves of every operand buffer, built once (see
      // mma_ss_lohi: nothing but an add may sit between two MMAs).
      const uint64_t dq = smem_desc_sw128(sb + L::kOffQ, 16, 1024);
      const uint64_t dk = smem_desc_sw128(sb + L::kOffK, 16, 1024);
      const uint64_t dv = smem_desc_sw128(sb + L::kOffV, L::kHalf, 1024);
      const uint32_t qk_hi = static_cast<uint32_t>(dq >> 32);  // same for Q and K (SBO 1024, 128B swizzle)
      const uint32_t v_hi = static_cast<uint32_t>(dv >> 32);
      const uint32_t q_lo = static_cast<uint32_t>(dq), k_lo = static_cast<uint32_t>(dk);
      const uint32_t v_lo = static_cast<uint32_t>(dv);
      auto commit = [&](uint32_t bar_addr) {
        if (leader) mma_commit(bar_addr);
      };
      auto issue_s = [&](int i, int stage) {
        const uint32_t a0 = q_lo + ((i * L::kQTile) >> 4);
        const uint32_t b0 = k_lo + ((stage * L::kKVTile) >> 4);
        const uint32_t d_tmem = tmem + i * kTileN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::kHalf + (kk & 3) * 32) >> 4;
          if (leader) mma_ss_lohi(d_tmem, a0 + off, qk_hi, b0 + off, qk_hi, idesc_s, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int i, int stage, bool acc) {
        const uint32_t b0 = v_lo + ((stage * L::kKVTile) >> 4);
        const uint32_t d_tmem = tmem + 256 + i * D;
        const uint32_t a_tmem = tmem + i * kTileN;
        const uint32_t acc0 = acc ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk)
          if (leader) mma_ts_lohi(d_tmem, a_tmem + kk * 8, b0 + ((kk * 2048) >> 4), v_hi, idesc_o, kk > 0 ? 1u : acc0);
      };
      bool ok = mbar_wait_bounded(bar(kBarQFull), 0, abort_flag, a.err, tmo) &&
                mbar_wait_bounded(bar(kBarKFull), 0, abort_flag, a.err, tmo);
      if (ok) {
        for (int i = 0; i < nq && ok; ++i) {
          if (i == 1 && !mbar_wait_bounded(bar(kBarQFull1), 0, abort_flag, a.err, tmo)) {
            ok = false;
            break;
          }
          issue_s(i, 0);
          commit(bar(kBarSFull + i));
        }
        if (ok) commit(bar(kBarKEmpty));
      }
      // The tensor pipe queues about one MMA: whatever this thread does
      // between two MMA groups leaves the pipe idle. Each step therefore
      // waits at two points only: V(it), K(it+1) and P_0(it) before
      // PV_0(it) + S_0(it+1); P_1(it) before PV_1(it) + S_1(it+1). The step
      // is instantiated per tile count and ring stage so that every MMA
      // operand is a compile-time offset from one base: a run-time tile or
      // stage index in the issue sequence measurably stalls the pipe.
      auto step = [&](auto nq_c, auto stage_c, int it) -> bool {
        constexpr int kNq = decltype(nq_c)::value;
        constexpr int s = decltype(stage_c)::value;
        constexpr int s2 = s ^ 1;
        const uint32_t ph = (it >> 1) & 1;
        const bool more = it + 1 < NT;
        if (!mbar_wait_bounded(bar(kBarVFull + s), ph, abort_flag, a.err, tmo) ||
            (more && !mbar_wait_bounded(bar(kBarKFull + s2), ((it + 1) >> 1) & 1, abort_flag, a.err, tmo)))
          return false;
#pragma unroll
        for (int i = 0; i < kNq; ++i) {
          if (!mbar_wait_bounded(bar(kBarPFull + i), it & 1, abort_flag, a.err, tmo)) return false;
          tc_fence_after();
          issue_pv(i, s, it > 0);
          if (more) {
            issue_s(i, s2);
            commit(bar(kBarSFull + i));
          } else {
            commit(bar(kBarOFull + i));
          }
          if (i == kNq - 1) {
            commit(bar(kBarVEmpty + s));
            if (more) commit(bar(kBarKEmpty + s2));
          }
        }
        return true;
      };
      auto run_steps = [&](auto nq_c) {
        for (int it = 0; ok && it < NT; it += 2) {
          ok = step(nq_c, std::integral_constant<int, 0>{}, it);
          if (ok && it + 1 < NT) ok = step(nq_c, std::integral_constant<int, 1>{}, it + 1);
        }
      };
      if (nq == 2)
        run_steps(std::integral_constant<int, 2>{});
      else
        run_steps(std::integral_constant<int, 1>{});
      if (!ok) {
        commit(bar(kBarDrain));
        drain_wait(bar(kBarDrain), 0, tmo);
      }
    }
  } else if (warp >= 2) {
    // ===================== softmax + epilogue =====================
    const int i = (warp - 2) >> 2;  // query tile of this warpgroup
    const int wq = warp & 3;        // TMEM lane quadrant of this warp (warp id mod 4)
    const int row = wq * 32 + lane;
    if (i < nq) {
      const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
      const uint32_t t_s = tmem + lane_off + i * kTileN;
      const uint32_t t_o = tmem + lane_off + 256 + i * D;
      const float sl2 = a.scale_log2;
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      KvCursor cur;
      cur.init(a.g, r);
      const uint8_t* km = kMasked ? a.kmask + (b % a.km_bmod) * a.km_bstride : nullptr;
      for (int it = 0; it < NT; ++it) {
        // key mask of this tile as four 32-bit words: bit l of word j is key
        // kv0 + 4l + j (read before the wait, so its latency overlaps it)
        uint32_t kmw[4] = {~0u, ~0u, ~0u, ~0u};
        if constexpr (kMasked) {
          const int kv0 = cur.kv0(), nvk = cur.nvalid();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c = 4 * lane + j;
            kmw[j] = __ballot_sync(0xffffffffu, c < nvk && km[kv0 + c] != 0);
          }
        }
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarSFull + i), it & 1, abort_flag, a.err, tmo));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[kTileN];
#pragma unroll
        for (int c = 0; c < kTileN / 32; ++c) tmem_ld32(t_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
        tmem_wait_ld();
        const int nv = cur.nvalid();
        if (nv < kTileN) {
#pragma unroll
          for (int c = 0; c < kTileN; ++c)
            if (c >= nv) sr[c] = __float_as_uint(-INFINITY);
        }
        const bool tile_masked = kMasked && (kmw[0] & kmw[1] & kmw[2] & kmw[3]) != ~0u;  // uniform in the warp
        if (tile_masked) {
#pragma unroll
          for (int c = 0; c < kTileN; ++c)
            if (!((kmw[c & 3] >> (c >> 2)) & 1u)) sr[c] = __float_as_uint(-INFINITY);
        }
        // P = 2^(s*scale*log2e - m_used) rounded to bf16, packed in pairs into
        // pk; returns the row sum of the rounded P (the values the PV product
        // consumes, so that O / l is a convex combination of V rows). S stays
        // intact in TMEM until P is stored over its first 64 columns.
        uint32_t pk[kTileN / 2];
        auto exp_pass = [&](float nm) -> float {
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int e = 0; e < kTileN / 2; ++e) {
            float x0, x1;
            fma_f32x2(x0, x1, __uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]), sl2, nm);
            pk[e] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
            add_bf16x2_to_f32(ls[(2 * e) & 3], ls[(2 * e + 1) & 3], pk[e]);
          }
          return (ls[0] + ls[1]) + (ls[2] + ls[3]);
        };
        auto row_max = [&]() -> float {  // of the raw scores, times scale*log2e
          float mx[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) mx[c] = fmaxf(__uint_as_float(sr[c]), __uint_as_float(sr[8 + c]));
#pragma unroll
          for (int c = 16; c < kTileN; c += 16) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
              mx[u] = fmax3(mx[u], __uint_as_float(sr[c + u]), __uint_as_float(sr[c + 8 + u]));
          }
          return fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * sl2;
        };
        auto reload_s = [&]() {
#pragma unroll
          for (int c = 0; c < kTileN / 32; ++c)
            tmem_ld32(t_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
          tmem_wait_ld();
          if (nv < kTileN) {
#pragma unroll
            for (int c = 0; c < kTileN; ++c)
              if (c >= nv) sr[c] = __float_as_uint(-INFINITY);
          }
          if (tile_masked) {
#pragma unroll
            for (int c = 0; c < kTileN; ++c)
              if (!((kmw[c & 3] >> (c >> 2)) & 1u)) sr[c] = __float_as_uint(-INFINITY);
          }
        };
        float f = 1.f, lsum;
        if (it == 0 || (kMasked && m_used == -INFINITY)) {
          // no running maximum yet (first tile, or every key so far masked,
          // which holds for every row alike): the row maximum first; a row
          // with every key of the tile masked keeps -inf and P = 0
          m_used = row_max();
          lsum = exp_pass(m_used == -INFINITY ? 0.f : -m_used);
        } else {
          // speculatively with the running maximum. Every P is at most the
          // row sum, so a row sum within 2^8 proves that the row maximum is
          // within 2^8 of the running maximum (the bound the rescaling keeps;
          // an overflow to inf fails the test too). Otherwise reload S, take
          // the row maximum, move to it if it grew by more than 2^8, and redo
          // the tile; O and l are rescaled by the same factor (O is idle
          // here: PV of the previous tile completed before S of this tile was
          // committed, and PV of this tile waits for P).
          lsum = exp_pass(-m_used);
          if (__any_sync(0xffffffffu, !(lsum <= 256.f))) {
            reload_s();
            const float mxs = row_max();
            const bool need = mxs > m_used + kRescaleThreshold;
            if (need) {
              f = ex2_approx(m_used - mxs);
              m_used = mxs;
            }
            lsum = exp_pass(-m_used);
            if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
              for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(t_o + c * 32, o);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                tmem_st32(t_o + c * 32, o);
              }
            }
          }
        }
        tmem_st32(t_s, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        tmem_st32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        l = l * f + lsum;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull + i));
        cur.advance(a.g, r);
      }
      if (ok && NT > 0) ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarOFull + i), 0, abort_flag, a.err, tmo));
      if (ok) {
        tc_fence_after();
        const int rows_valid = rows[i];
        const int tok0 = qrow[i];  // first token of this tile
        // l = 0: no key (an empty lap, or every key masked) -> out 0, lse -inf
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const float lse_v = l > 0.f ? (m_used + log2f(l)) * 0.69314718055994531f : -INFINITY;
        if (row < rows_valid) a.lse[b * a.l_bstride + h * a.l_hstride + tok0 + row] = lse_v;
        // all of O's row from TMEM at once, then per 32-column chunk: stage 32
        // rows x 32 fp32 per warp in this tile's (now idle) Q buffer, 128B-
        // swizzled (double-buffered where the buffer has room), and store 4
        // rows x 128 contiguous bytes per warp instruction
        uint32_t o[D];
        if (NT > 0) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) tmem_ld32(t_o + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[c * 32]));
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < D; ++e) o[e] = 0u;
        }
        float* out_b = a.out + b * a.o_bstride + static_cast<int64_t>(h) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          // 8 KB per warp (two 4 KB buffers) when the Q tile has 32 KB, else one buffer
          constexpr int kWarpStage = L::kQTile / 4 >= 8192 ? 8192 : 4096;
          float* stage = reinterpret_cast<float*>(smem + L::kOffQ + i * L::kQTile + wq * kWarpStage +
                                                  (kWarpStage == 8192 ? (c & 1) * 4096 : 0));
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const uint32_t* oc = &o[c * 32 + 4 * q4];
            float4 val = make_float4(__uint_as_float(oc[0]) * inv_l, __uint_as_float(oc[1]) * inv_l,
                                     __uint_as_float(oc[2]) * inv_l, __uint_as_float(oc[3]) * inv_l);
            *reinterpret_cast<float4*>(stage + lane * 32 + ((q4 ^ (lane & 7)) * 4)) = val;
          }
          __syncwarp();
#pragma unroll
          for (int pass = 0; pass < 8; ++pass) {
            const int rr = pass * 4 + (lane >> 3);
            const int q4 = lane & 7;
            const float4 val = *reinterpret_cast<const float4*>(stage + rr * 32 + ((q4 ^ (rr & 7)) * 4));
            const int grow = wq * 32 + rr;
            if (grow < rows_valid)
              *reinterpret_cast<float4*>(out_b + static_cast<int64_t>(tok0 + grow) * a.o_sstride + c * 32 + q4 * 4) = val;
          }
          __syncwarp();  // the buffer is read before it is staged again
        }
      }
    }
  }

  // ---- teardown: every thread of the CTA arrives here, aborted or not ----
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// A kernel that exercises the bounded wait on a barrier that nothing
// completes: every thread times out, the first raises the error word.
__global__ void wait_probe_kernel(uint32_t* err, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar_storage;
  __shared__ uint32_t abort_word;
  const uint32_t bar = smem_addr(&bar_storage);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    abort_word = 0;
    fence_mbar_init();
  }
  __syncthreads();
  (void)mbar_wait_bounded(bar, 0, &abort_word, err, timeout_ns);
  __syncthreads();
}

template <int D>
cudaError_t launch_tc_d(const AttnArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        cudaStream_t s) {
  using L = Smem<D>;
  static_assert(L::kAlloc <= 227 * 1024, "shared memory budget");
  // the key-mask code is compiled only into the masked instance
  auto kernel = a.kmask ? attn_fwd_tc_kernel<D, true> : attn_fwd_tc_kernel<D, false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  // two-tile items (pairs, plus leftover tiles paired across shards over a
  // whole lap) and one-tile items; see the work-item decode in the kernel
  const int n_single = a.g.single_prefix[a.g.n_q];
  const int n_cross = a.g.step < 0 ? n_single / 2 : 0;
  const int64_t items = static_cast<int64_t>(a.g.pair_prefix[a.g.n_q] + n_single - n_cross) * a.H * a.B;
  if (items == 0) return cudaSuccess;
  if (items > 0x7fffffff) return cudaErrorInvalidValue;
  kernel<<<dim3(static_cast<unsigned>(items)), kThreads, L::kAlloc, s>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

uint32_t* device_error_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_dev_error) != cudaSuccess) return nullptr;
  return static_cast<uint32_t*>(p);
}

cudaError_t launch_attn_tc(const AttnArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           cudaStream_t s) {
  if (a.D == 64) return launch_tc_d<64>(a, tq, tk, tv, s);
  if (a.D == 128) return launch_tc_d<128>(a, tq, tk, tv, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_wait_probe(uint32_t* err, uint64_t timeout_ns, cudaStream_t s) {
  wait_probe_kernel<<<1, 64, 0, s>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace cp
