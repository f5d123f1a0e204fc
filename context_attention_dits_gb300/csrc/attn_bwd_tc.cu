// attn_bwd_tc.cu — backward of block / ring attention on the 5th-generation
// tensor cores (tcgen05, bf16 operands, fp32 accumulators in tensor memory).
//
// The gradients are those of the CUDA-core backward (same formulas, same
// ring walk; context parallelism page, Ring Attention section):
//   p_ij = exp(scale q_i.k_j - lse_i),  ds_ij = p_ij (dout_i.v_j - delta_i),
//   dv_j = sum_i p_ij dout_i,  dk_j = scale sum_i ds_ij q_i,  dq_i = scale sum_j ds_ij k_j.
//
// Two kinds of CTA, in one launch (attn_bwd_tc_kernel: the dk/dv CTAs first,
// then the dq CTAs, which fill the SMs the last wave of dk/dv CTAs leaves
// idle), neither with atomics, each walking its lap in 64-row sub-steps whose
// S / dP pair alternates between two TMEM slots, so that the row pass of one
// sub-step runs while the tensor cores work on the other's:
//
// dk / dv: one CTA owns a tile of 128 keys of one (batch entry, head) and
// walks every 64-row query sub-tile of the lap, rank by rank in the order its
// K/V block visits them ((j + t) mod n). Per sub-tile, four MMAs (M = 128):
//   1. S^T  = K Q^T      (A = K tile, B = Q sub-tile; both K-major; N = 64)
//   2. dP^T = V dO^T     (A = V tile, B = dO sub-tile)
//   3. dV  += P^T dO     (A = P^T in TMEM, B = dO MN-major; K = 64 rows)
//   4. dK  += dS^T Q     (A = dS^T in TMEM, B = Q MN-major)
// S^T and dP^T of sub-step j sit in TMEM slot j mod 2 (columns [0, 64) and
// [64, 128) of the slot); dV and dK in [256, 256 + D) and [256 + D, 256 + 2D).
// Between 2 and 3 the row warps (one thread per key row and column half)
// turn S^T and dP^T into P^T and dS^T (bf16: the 32 query columns of a half
// over the first 16 TMEM columns of that half, so that the two halves never
// write where the other reads). The MMAs
// 1 and 2 of sub-step j + 2 are issued right after 3 and 4 of sub-step j, so
// they run while the row pass works on sub-step j + 1. Q, dO, lse and delta
// stream through four 64-row slots. After the last sub-tile it writes dk, dv.
//
// dq: one CTA owns 128 query rows, whose Q and dO rows the row warps place
// in TMEM once, and walks the 64-key K/V sub-tiles of its rank's lap in ring
// order ((r - t) mod n): S = Q K^T and dP = dO V^T (N = 64, A read from
// TMEM) into TMEM slot j mod 2, then dQ += dS K with dS (a thread per query
// row and column half, over the first 16 columns of each 32-column half of
// S); dq is stored once. It recomputes S and dP, 1.4x the MMA work of a single
// fused kernel, in exchange for no reduction of dq tiles across key-tile
// CTAs. K and V stream through six 64-row slots.
//
// Warp roles (320 threads): 0 = TMA producer, 1 = MMA issuer, 2-9 = row warps:
// a warp reaches TMEM lanes 32 (warp mod 4) and up, so two warps share each
// lane quarter, warps 2-5 taking the first 32 columns of a sub-step and warps
// 6-9 the other 32.
// Every wait is bounded; on expiry the CTA records a timeout, lets its copies
// land, frees its tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "cp_internal.h"
#include "cp_ptx.cuh"

namespace cp {
namespace {

constexpr int kRowWarps = 8;  // two per TMEM lane quarter, one per 32-column half of a sub-step
constexpr int kThreadsB = 64 + 32 * kRowWarps;
constexpr uint32_t kTmemColsB = 512;
constexpr int kT = kBwdTcTile;  // keys per dk/dv CTA, query rows per dq CTA
constexpr int kSub = 64;        // rows of a streamed sub-tile: query rows (dk/dv) or keys (dq) per sub-step
constexpr int kSlots = 4;       // streamed sub-tile slots in shared memory
constexpr float kLog2eB = 1.4426950408889634f;

// K-major operand of 128 rows: 16-element K steps within a 64-column box,
// then the next box (boxes of 128 rows x 128 bytes)
__device__ __forceinline__ uint32_t kstep128(int kk) {
  return static_cast<uint32_t>(((kk >> 2) * (kT * 128) + (kk & 3) * 32) >> 4);
}
// the same for a 64-row sub-tile (boxes of 64 rows x 128 bytes)
__device__ __forceinline__ uint32_t kstep64(int kk) {
  return static_cast<uint32_t>(((kk >> 2) * (kSub * 128) + (kk & 3) * 32) >> 4);
}

template <int D>
struct BSmem {
  static constexpr int kTile = kT * D * 2;    // one bf16 128-row tile (K or V)
  static constexpr int kSubT = kSub * D * 2;  // one bf16 64-row sub-tile (Q or dO)
  static constexpr int kHalfS = kSub * 128;   // one 64-column box of a sub-tile
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTile;
  static constexpr int kOffQ = kOffV + kTile;            // kSlots sub-tiles
  static constexpr int kOffO = kOffQ + kSlots * kSubT;   // dO, kSlots sub-tiles
  static constexpr int kOffLse = kOffO + kSlots * kSubT;     // kSlots x 64 floats: lse * log2 e
  static constexpr int kOffDlt = kOffLse + kSlots * kSub * 4; // kSlots x 64 floats: delta
  static constexpr int kOffBar = kOffDlt + kSlots * kSub * 4;
  static constexpr int kNumBars = 15;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  // + room to align the base to 1024 bytes, as much as the 227 KB budget leaves
  static constexpr int kMax = 227 * 1024;
  static constexpr int kAlloc = kBytes + 1024 <= kMax ? kBytes + 1024 : kMax;
};

enum : int {
  kBarKV = 0,      // K and V tiles landed
  kBarQFull = 1,   // +slot (4): Q, dO, lse, delta of a sub-tile landed (TMA bytes)
  kBarQEmpty = 5,  // +slot (4): MMAs done with the slot
  kBarSFull = 9,   // +TMEM slot (2): S^T and dP^T of the sub-step in TMEM
  kBarPFull = 11,  // +TMEM slot (2): P^T, dS^T written (every row warp arrives)
  kBarDone = 13,   // every MMA of the CTA done: dK, dV final
  kBarDrain = 14,
};

// 64-row query sub-tiles of the lap of K/V block jb, in the order the block
// visits the ranks.
struct QCursor {
  int t, r, tile, ntile, off, len;
  __device__ __forceinline__ void init(const BwdArgs& a, int jb) {
    t = -1;
    next_block(a, jb);
  }
  __device__ __forceinline__ void next_block(const BwdArgs& a, int jb) {
    tile = 0;
    while (true) {
      ++t;
      if (t >= a.n) return;
      r = (jb + t) % a.n;
      off = a.off[r];
      len = a.len[r];
      ntile = (len + kSub - 1) / kSub;
      if (ntile > 0) return;
    }
  }
  __device__ __forceinline__ int q0() const { return off + tile * kSub; }
  __device__ __forceinline__ void advance(const BwdArgs& a, int jb) {
    if (++tile >= ntile) next_block(a, jb);
  }
};

__device__ __forceinline__ void drain_wait_b(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1; !mbar_try_wait(bar, parity); ++n)
    if ((n & 255u) == 0 && global_timer_ns() - t0 > timeout_ns) return;
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// TMEM column (within S's or dP's 64) of the bf16 A operand for K step kk of
// a sub-step: rows [32 h, 32 h + 32) of the sub-step (written by the row warps
// of column half h) sit in columns [32 h, 32 h + 16), 8 columns per K step
__device__ __forceinline__ uint32_t pcol(int kk) { return static_cast<uint32_t>((kk >> 1) * 32 + (kk & 1) * 8); }

// tq64, to64: Q and dO with 64-row boxes; tk, tv: K and V with 128-row boxes
// One dk/dv CTA: key tile bx of the lap's key tiles (kv_prefix) of head h,
// batch entry b; smem_raw holds alloc bytes of dynamic shared memory.
template <int D>
__device__ __forceinline__ void bwd_dkdv_cta(const CUtensorMap& tq64, const CUtensorMap& tk, const CUtensorMap& tv,
                                             const CUtensorMap& to64, const BwdArgs& a, uint8_t* smem_raw, int alloc,
                                             int bx, int h, int b) {
  using L = BSmem<D>;
  // the swizzled tiles need a 1024-byte aligned base; a base that would need
  // more padding than the allocation holds is reported (uniformly, before any
  // barrier or TMEM use) instead of used
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  if (pad > static_cast<uint32_t>(alloc - L::kBytes)) {
    if (threadIdx.x == 0) atomicOr(a.err, kDevErrLayout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = smem_addr(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);  // [0] TMEM base, [1] abort flag
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) -> uint32_t { return sb + L::kOffBar + 8 * i; };
  float* s_lse = reinterpret_cast<float*>(smem + L::kOffLse);
  float* s_dlt = reinterpret_cast<float*>(smem + L::kOffDlt);

  if (bwd_head_is_padding(a, h, b)) return;  // uniform per CTA, before any barrier or TMEM
  int jb = 0;
  while (jb + 1 < a.n && a.kv_prefix[jb + 1] <= bx) ++jb;
  const int key0 = a.off[jb] + (bx - a.kv_prefix[jb]) * kT;
  const int nk = min(kT, a.off[jb] + a.len[jb] - key0);
  int NJ = 0;  // 64-row query sub-steps of the lap
  for (int t = 0; t < a.n; ++t) NJ += (a.len[(jb + t) % a.n] + kSub - 1) / kSub;

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNumBars; ++i) {
      const bool four = i == kBarPFull || i == kBarPFull + 1;
      mbar_init(bar(i), four ? kRowWarps : 1);
    }
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(misc), kTmemColsB);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const uint64_t tmo = a.timeout_ns;

  if (warp == 0) {
    // ===================== TMA producer =====================
    const bool leader = elect_one();
    if (leader) {
      tma_prefetch_desc(&tq64);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&to64);
      mbar_arrive_expect_tx(bar(kBarKV), 2 * L::kTile);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_4d(sb + L::kOffK + c * (kT * 128), &tk, bar(kBarKV), c * 64, h, key0, b);
        tma_load_4d(sb + L::kOffV + c * (kT * 128), &tv, bar(kBarKV), c * 64, h, key0, b);
      }
    }
    int issued[kSlots] = {0, 0, 0, 0};
    QCursor cur;
    cur.init(a, jb);
    for (int j = 0; j < NJ; ++j) {
      const int s = j & (kSlots - 1);
      const uint32_t ph = (j >> 2) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarQEmpty + s), ph ^ 1, abort_flag, a.err, tmo))) break;
      const int q0 = cur.q0();
      if (leader) {
        mbar_arrive_expect_tx(bar(kBarQFull + s), 2 * L::kSubT + 2 * kSub * 4);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(sb + L::kOffQ + s * L::kSubT + c * L::kHalfS, &tq64, bar(kBarQFull + s), c * 64, h, q0, b);
          tma_load_4d(sb + L::kOffO + s * L::kSubT + c * L::kHalfS, &to64, bar(kBarQFull + s), c * 64, h, q0, b);
        }
        // the rows' lse (times log2 e) and delta from the padded per-shard
        // copies: rows past the shard, and rows that saw no key, hold lse =
        // +inf, so that p = 0
        const int64_t pr = ((static_cast<int64_t>(b) * a.H + h) * a.n + cur.r) * a.lpad + cur.tile * kSub;
        bulk_g2s(smem_addr(s_lse + s * kSub), a.lse2p + pr, kSub * 4, bar(kBarQFull + s));
        bulk_g2s(smem_addr(s_dlt + s * kSub), a.dltp + pr, kSub * 4, bar(kBarQFull + s));
      }
      __syncwarp();
      ++issued[s];
      cur.advance(a, jb);
    }
    if (*abort_flag) {
      // let every issued copy land before the CTA's shared memory goes away
      drain_wait_b(bar(kBarKV), 0, tmo);
      for (int s = 0; s < kSlots; ++s)
        if (issued[s]) drain_wait_b(bar(kBarQFull + s), (issued[s] - 1) & 1, tmo);
    }
  } else if (warp == 1) {
    // ===================== MMA issuer =====================
    const bool leader = elect_one();
    constexpr uint32_t idesc_s = idesc_bf16_f32(kT, kSub, false, false);  // S^T, dP^T: M = keys, N = 64 queries
    constexpr uint32_t idesc_g = idesc_bf16_f32(kT, D, false, true);      // dV, dK: A in TMEM, B MN-major
    const uint64_t k_km = smem_desc_sw128(sb + L::kOffK, 16, 1024);
    const uint64_t v_km = smem_desc_sw128(sb + L::kOffV, 16, 1024);
    const uint64_t q_km = smem_desc_sw128(sb + L::kOffQ, 16, 1024);
    const uint64_t o_km = smem_desc_sw128(sb + L::kOffO, 16, 1024);
    const uint64_t q_mn = smem_desc_sw128(sb + L::kOffQ, L::kHalfS, 1024);
    const uint64_t o_mn = smem_desc_sw128(sb + L::kOffO, L::kHalfS, 1024);
    const uint32_t km_hi = static_cast<uint32_t>(k_km >> 32), mn_hi = static_cast<uint32_t>(q_mn >> 32);
    const uint32_t k_km_lo = static_cast<uint32_t>(k_km), v_km_lo = static_cast<uint32_t>(v_km);
    const uint32_t q_km_lo = static_cast<uint32_t>(q_km), o_km_lo = static_cast<uint32_t>(o_km);
    const uint32_t q_mn_lo = static_cast<uint32_t>(q_mn), o_mn_lo = static_cast<uint32_t>(o_mn);
    auto commit = [&](uint32_t bar_addr) {
      if (leader) mma_commit(bar_addr);
    };
    // S^T and dP^T of the sub-tile in smem slot q, into TMEM slot ts
    auto issue_sdp = [&](int q, int ts) {
      const uint32_t slot = static_cast<uint32_t>((q * L::kSubT) >> 4);
      const uint32_t d = tmem + ts * 128;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        if (leader) mma_ss_lohi(d, k_km_lo + kstep128(kk), km_hi, q_km_lo + slot + kstep64(kk), km_hi, idesc_s, kk > 0);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        if (leader)
          mma_ss_lohi(d + kSub, v_km_lo + kstep128(kk), km_hi, o_km_lo + slot + kstep64(kk), km_hi, idesc_s, kk > 0);
    };
    // dV += P^T dO and dK += dS^T Q over the sub-tile's 64 query rows (K = rows:
    // 16 rows = 2048 bytes of an MN-major sub-tile; the bf16 P^T / dS^T of
    // rows [32 h, 32 h + 32) sit in TMEM columns [32 h, 32 h + 16) of theirs)
    auto issue_g = [&](int q, int ts, bool acc) {
      const uint32_t slot = static_cast<uint32_t>((q * L::kSubT) >> 4);
      const uint32_t pa = tmem + ts * 128;
#pragma unroll
      for (int kk = 0; kk < kSub / 16; ++kk)
        if (leader) mma_ts_lohi(tmem + 256, pa + pcol(kk), o_mn_lo + slot + ((kk * 2048) >> 4), mn_hi, idesc_g,
                                (acc || kk > 0) ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < kSub / 16; ++kk)
        if (leader) mma_ts_lohi(tmem + 256 + D, pa + kSub + pcol(kk), q_mn_lo + slot + ((kk * 2048) >> 4), mn_hi,
                                idesc_g, (acc || kk > 0) ? 1u : 0u);
    };
    auto wait_q = [&](int j) -> bool {
      return mbar_wait_bounded(bar(kBarQFull + (j & (kSlots - 1))), (j >> 2) & 1, abort_flag, a.err, tmo);
    };
    bool ok = mbar_wait_bounded(bar(kBarKV), 0, abort_flag, a.err, tmo);
    // prologue: S^T, dP^T of the first two sub-steps
    for (int j = 0; ok && j < 2 && j < NJ; ++j) {
      if (!wait_q(j)) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_sdp(j, j);
      commit(bar(kBarSFull + j));
    }
    // sub-step j: once P^T, dS^T are in TMEM slot j mod 2, dV and dK consume
    // them and S^T, dP^T of sub-step j + 2 go into the same slot; the step is
    // instantiated per smem slot so every operand offset is a constant
    auto step = [&](auto q_c, int j) -> bool {
      constexpr int q = decltype(q_c)::value;
      constexpr int ts = q & 1;
      if (!mbar_wait_bounded(bar(kBarPFull + ts), (j >> 1) & 1, abort_flag, a.err, tmo)) return false;
      tc_fence_after();
      issue_g(q, ts, j > 0);
      commit(bar(kBarQEmpty + q));
      if (j + 2 < NJ) {
        if (!wait_q(j + 2)) return false;
        tc_fence_after();
        issue_sdp((q + 2) & (kSlots - 1), ts);
        commit(bar(kBarSFull + ts));
      }
      return true;
    };
    for (int j = 0; ok && j < NJ; j += kSlots) {
      ok = step(std::integral_constant<int, 0>{}, j);
      if (ok && j + 1 < NJ) ok = step(std::integral_constant<int, 1>{}, j + 1);
      if (ok && j + 2 < NJ) ok = step(std::integral_constant<int, 2>{}, j + 2);
      if (ok && j + 3 < NJ) ok = step(std::integral_constant<int, 3>{}, j + 3);
    }
    if (ok) {
      commit(bar(kBarDone));
    } else {
      commit(bar(kBarDrain));
      drain_wait_b(bar(kBarDrain), 0, tmo);
    }
  } else {
    // ===================== row pass: one thread per key row and column half =====================
    const int wq = warp & 3;
    const int hc = (warp - 2) >> 2;  // this warp's 32 query columns of each sub-step
    const int key = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const bool kvalid = key < nk;
    const float c2 = a.scale * kLog2eB;
    bool ok = true;
    for (int j = 0; j < NJ; ++j) {
      const int q = j & (kSlots - 1), ts = j & 1;
      ok = __all_sync(0xffffffffu,
                      mbar_wait_bounded(bar(kBarQFull + q), (j >> 2) & 1, abort_flag, a.err, tmo) &&
                          mbar_wait_bounded(bar(kBarSFull + ts), (j >> 1) & 1, abort_flag, a.err, tmo));
      if (!ok) break;
      tc_fence_after();
      const uint32_t t_s = tmem + lane_off + ts * 128, t_dp = t_s + kSub;
      const float* lse2 = s_lse + q * kSub;
      const float* dlt = s_dlt + q * kSub;
      {
        const int c = hc;
        uint32_t sr[32], dr[32];
        tmem_ld32(t_s + c * 32, sr);
        tmem_ld32(t_dp + c * 32, dr);
        tmem_wait_ld();
        uint32_t pp[16], dd[16];
        if (kvalid) {
          // p = 2^(s c2 - lse2) (lse2 = +inf past the sub-tile: p = 0), ds = p (dp - delta); pairs of
          // columns in packed fp32x2 FMAs, lse and delta read as 16-byte vectors
          const float4* l4 = reinterpret_cast<const float4*>(lse2 + c * 32);
          const float4* d4 = reinterpret_cast<const float4*>(dlt + c * 32);
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            const float4 lv = l4[x], dv4 = d4[x];
            const float nl[4] = {-lv.x, -lv.y, -lv.z, -lv.w}, nd[4] = {-dv4.x, -dv4.y, -dv4.z, -dv4.w};
#pragma unroll
            for (int y = 0; y < 4; y += 2) {
              const int e = 4 * x + y;
              float t0, t1, g0, g1, d0, d1;
              fma2(t0, t1, u2f(sr[e]), u2f(sr[e + 1]), c2, c2, nl[y], nl[y + 1]);
              fma2(g0, g1, u2f(dr[e]), u2f(dr[e + 1]), 1.f, 1.f, nd[y], nd[y + 1]);
              const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
              fma2(d0, d1, p0, p1, g0, g1, 0.f, 0.f);
              pp[e >> 1] = pack_bf16x2(p0, p1);
              dd[e >> 1] = pack_bf16x2(d0, d1);
            }
          }
        } else {
#pragma unroll
          for (int x = 0; x < 16; ++x) pp[x] = dd[x] = 0u;  // a key past the tile: p = ds = 0
        }
        // P^T over the first half of this warp's S^T columns, dS^T over those of dP^T
        tmem_st16(t_s + c * 32, pp);
        tmem_st16(t_dp + c * 32, dd);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull + ts));
    }
    // ---- dk, dv of this CTA's keys ----
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kBarDone), 0, abort_flag, a.err, tmo));
    if (ok) {
      tc_fence_after();
      const int64_t o = b * a.bstride + static_cast<int64_t>(key0 + key) * a.sstride + h * D;
      {
        const int g = hc;  // column half 0 writes dv, half 1 dk
        float* dst = g == 0 ? a.dv : a.dk;
        const float mul = g == 0 ? 1.f : a.scale;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + 256 + g * D + c * 32, r);
          tmem_wait_ld();
          if (kvalid) {
#pragma unroll
            for (int x = 0; x < 32; x += 4)
              *reinterpret_cast<float4*>(dst + o + c * 32 + x) =
                  make_float4(u2f(r[x]) * mul, u2f(r[x + 1]) * mul, u2f(r[x + 2]) * mul, u2f(r[x + 3]) * mul);
          }
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
    tmem_dealloc(tmem, kTmemColsB);
  }
}

// ----------------------------------------------------------------------------
// dq: one CTA per 128 query rows of one (batch entry, head). The row warps
// load the CTA's Q and dO rows once into TMEM (bf16 pairs, the A-operand
// layout: columns [384, 384 + D/2) and [384 + D/2, 384 + D)); 64-key K and V
// sub-tiles of the rank's lap stream in ring order ((r - t) mod n) through
// kDqSlots shared-memory slots. Per sub-tile three MMAs (M = 128 rows):
//   S  = Q K^T    (TS: Q in TMEM, K K-major; N = 64) -> TMEM slot j mod 2, [0, 64)
//   dP = dO V^T   (TS)                               -> the same slot, [64, 128)
//   dQ += dS K    (TS: dS over S's first 32 columns, K read MN-major)
//                                                    -> TMEM [256, 256 + D)
// Only K and V come from shared memory. S and dP of sub-step j + 2 are issued
// right after dQ of sub-step j, so they run while the row warps (one thread
// per query row and column half, lse and delta in registers) form
// dS = p (dp - delta) of sub-step j + 1. dq is stored once, without atomics.
// ----------------------------------------------------------------------------
constexpr int kDqSlots = 6;  // K/V sub-tile slots of the dq kernel

template <int D>
struct DqSmem {
  static constexpr int kSubT = kSub * D * 2;  // a K or V sub-tile: 64 keys
  static constexpr int kHalfS = kSub * 128;
  static constexpr int kOffK = 0;                          // kDqSlots sub-tiles
  static constexpr int kOffV = kOffK + kDqSlots * kSubT;   // kDqSlots sub-tiles
  static constexpr int kOffBar = kOffV + kDqSlots * kSubT;
  static constexpr int kNumBars = 1 + 2 * kDqSlots + 6;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kMax = 227 * 1024;
  static constexpr int kAlloc = kBytes + 1024 <= kMax ? kBytes + 1024 : kMax;
};

enum : int {
  kDqBarQ = 0,                             // Q and dO in TMEM (every row warp arrives)
  kDqBarKVFull = 1,                        // +slot: K and V sub-tiles landed
  kDqBarKVEmpty = 1 + kDqSlots,            // +slot: MMAs done with the slot
  kDqBarSFull = 1 + 2 * kDqSlots,          // +TMEM slot (2): S and dP in TMEM
  kDqBarPFull = kDqBarSFull + 2,           // +TMEM slot (2): dS written (every row warp arrives)
  kDqBarDone = kDqBarPFull + 2,            // every MMA done: dQ final
  kDqBarDrain = kDqBarDone + 1,
};

// 64-key K/V sub-tiles of rank r's lap, blocks in ring order (r - t) mod n.
struct KvWalk {
  int t, tile, ntile, off, len;
  __device__ __forceinline__ void init(const BwdArgs& a, int r) {
    t = -1;
    next_block(a, r);
  }
  __device__ __forceinline__ void next_block(const BwdArgs& a, int r) {
    tile = 0;
    while (true) {
      ++t;
      if (t >= a.n) return;
      int j = (r - t) % a.n;
      if (j < 0) j += a.n;
      off = a.off[j];
      len = a.len[j];
      ntile = (len + kSub - 1) / kSub;
      if (ntile > 0) return;
    }
  }
  __device__ __forceinline__ int k0() const { return off + tile * kSub; }
  __device__ __forceinline__ int nvalid() const { return min(kSub, len - tile * kSub); }
  __device__ __forceinline__ void advance(const BwdArgs& a, int r) {
    if (++tile >= ntile) next_block(a, r);
  }
};

// One dq CTA: query tile bx of the lap's query tiles (q_prefix) of head h,
// batch entry b. tk64, tv64: K and V with 64-row boxes.
template <int D>
__device__ __forceinline__ void bwd_dq_cta(const CUtensorMap& tk64, const CUtensorMap& tv64, const BwdArgs& a,
                                           uint8_t* smem_raw, int alloc, int bx, int h, int b) {
  using L = DqSmem<D>;
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  if (pad > static_cast<uint32_t>(alloc - L::kBytes)) {
    if (threadIdx.x == 0) atomicOr(a.err, kDevErrLayout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = smem_addr(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);  // [0] TMEM base, [1] abort flag
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) -> uint32_t { return sb + L::kOffBar + 8 * i; };

  if (bwd_head_is_padding(a, h, b)) return;  // uniform per CTA, before any barrier or TMEM
  int r = 0;
  while (r + 1 < a.n && a.q_prefix[r + 1] <= bx) ++r;
  const int q0 = a.off[r] + (bx - a.q_prefix[r]) * kT;
  const int nq = min(kT, a.off[r] + a.len[r] - q0);
  int NJ = 0;  // 64-key sub-steps of the lap
  for (int t = 0; t < a.n; ++t) {
    int j = (r - t) % a.n;
    if (j < 0) j += a.n;
    NJ += (a.len[j] + kSub - 1) / kSub;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kNumBars; ++i)
      mbar_init(bar(i), (i == kDqBarQ || i == kDqBarPFull || i == kDqBarPFull + 1) ? kRowWarps : 1);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(misc), kTmemColsB);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const uint64_t tmo = a.timeout_ns;

  if (warp == 0) {
    // ===================== TMA producer =====================
    const bool leader = elect_one();
    if (leader) {
      tma_prefetch_desc(&tk64);
      tma_prefetch_desc(&tv64);
    }
    int issued[kDqSlots] = {};
    KvWalk cur;
    cur.init(a, r);
    for (int j = 0; j < NJ; ++j) {
      const int s = j % kDqSlots;
      const uint32_t ph = (j / kDqSlots) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar(kDqBarKVEmpty + s), ph ^ 1, abort_flag, a.err, tmo)))
        break;
      if (leader) {
        mbar_arrive_expect_tx(bar(kDqBarKVFull + s), 2 * L::kSubT);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(sb + L::kOffK + s * L::kSubT + c * L::kHalfS, &tk64, bar(kDqBarKVFull + s), c * 64, h,
                      cur.k0(), b);
          tma_load_4d(sb + L::kOffV + s * L::kSubT + c * L::kHalfS, &tv64, bar(kDqBarKVFull + s), c * 64, h,
                      cur.k0(), b);
        }
      }
      ++issued[s];
      cur.advance(a, r);
    }
    if (*abort_flag) {
      // let every issued copy land before the CTA's shared memory goes away
      for (int s = 0; s < kDqSlots; ++s)
        if (issued[s]) drain_wait_b(bar(kDqBarKVFull + s), (issued[s] - 1) & 1, tmo);
    }
  } else if (warp == 1) {
    // ===================== MMA issuer =====================
    const bool leader = elect_one();
    constexpr uint32_t idesc_s = idesc_bf16_f32(kT, kSub, false, false);  // S, dP: M = query rows, N = 64 keys
    constexpr uint32_t idesc_q = idesc_bf16_f32(kT, D, false, true);      // dQ: A (dS) in TMEM, B (K) MN-major
    const uint64_t k_km = smem_desc_sw128(sb + L::kOffK, 16, 1024);
    const uint64_t v_km = smem_desc_sw128(sb + L::kOffV, 16, 1024);
    const uint64_t k_mn = smem_desc_sw128(sb + L::kOffK, L::kHalfS, 1024);
    const uint32_t km_hi = static_cast<uint32_t>(k_km >> 32), mn_hi = static_cast<uint32_t>(k_mn >> 32);
    const uint32_t k_lo = static_cast<uint32_t>(k_km), v_lo = static_cast<uint32_t>(v_km);
    const uint32_t k_mn_lo = static_cast<uint32_t>(k_mn);
    const uint32_t t_q = tmem + 384, t_o = tmem + 384 + D / 2;  // Q and dO rows in TMEM (8 columns per K step)
    auto commit = [&](uint32_t bar_addr) {
      if (leader) mma_commit(bar_addr);
    };
    // S and dP of the K/V sub-tile in smem slot q, into TMEM slot ts
    auto issue_sdp = [&](int q, int ts) {
      const uint32_t slot = static_cast<uint32_t>((q * L::kSubT) >> 4);
      const uint32_t d = tmem + ts * 128;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        if (leader) mma_ts_lohi(d, t_q + kk * 8, k_lo + slot + kstep64(kk), km_hi, idesc_s, kk > 0 ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        if (leader) mma_ts_lohi(d + kSub, t_o + kk * 8, v_lo + slot + kstep64(kk), km_hi, idesc_s, kk > 0 ? 1u : 0u);
    };
    auto wait_kv = [&](int j) -> bool {
      return mbar_wait_bounded(bar(kDqBarKVFull + (j % kDqSlots)), (j / kDqSlots) & 1, abort_flag, a.err, tmo);
    };
    bool ok = mbar_wait_bounded(bar(kDqBarQ), 0, abort_flag, a.err, tmo);
    for (int j = 0; ok && j < 2 && j < NJ; ++j) {
      if (!wait_kv(j)) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_sdp(j, j);
      commit(bar(kDqBarSFull + j));
    }
    // sub-step j: dQ += dS K once dS is in TMEM slot j mod 2 (K = keys: 16 key
    // rows = 2048 bytes of the MN-major sub-tile), then S, dP of sub-step j + 2
    // into the same slot; instantiated per smem slot (kDqSlots is even, so the
    // TMEM slot is the smem slot's parity)
    static_assert(kDqSlots % 2 == 0, "TMEM slot = smem slot parity");
    auto step = [&](auto q_c, int j) -> bool {
      constexpr int q = decltype(q_c)::value;
      constexpr int ts = q & 1;
      if (!mbar_wait_bounded(bar(kDqBarPFull + ts), (j >> 1) & 1, abort_flag, a.err, tmo)) return false;
      tc_fence_after();
      const uint32_t slot = static_cast<uint32_t>((q * L::kSubT) >> 4);
#pragma unroll
      for (int kk = 0; kk < kSub / 16; ++kk)
        if (leader) mma_ts_lohi(tmem + 256, tmem + ts * 128 + pcol(kk), k_mn_lo + slot + ((kk * 2048) >> 4), mn_hi,
                                idesc_q, (j > 0 || kk > 0) ? 1u : 0u);
      commit(bar(kDqBarKVEmpty + q));
      if (j + 2 < NJ) {
        if (!wait_kv(j + 2)) return false;
        tc_fence_after();
        issue_sdp((q + 2) % kDqSlots, ts);
        commit(bar(kDqBarSFull + ts));
      }
      return true;
    };
    for (int j = 0; ok && j < NJ; j += kDqSlots) {
      ok = step(std::integral_constant<int, 0>{}, j);
      if (ok && j + 1 < NJ) ok = step(std::integral_constant<int, 1>{}, j + 1);
      if (ok && j + 2 < NJ) ok = step(std::integral_constant<int, 2>{}, j + 2);
      if (ok && j + 3 < NJ) ok = step(std::integral_constant<int, 3>{}, j + 3);
      if (ok && j + 4 < NJ) ok = step(std::integral_constant<int, 4>{}, j + 4);
      if (ok && j + 5 < NJ) ok = step(std::integral_constant<int, 5>{}, j + 5);
    }
    if (ok) {
      commit(bar(kDqBarDone));
    } else {
      commit(bar(kDqBarDrain));
      drain_wait_b(bar(kDqBarDrain), 0, tmo);
    }
  } else {
    // ===================== dS: one thread per query row and column half =====================
    const int wq = warp & 3;
    const int hc = (warp - 2) >> 2;  // this warp's 32 key columns of each sub-step
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float c2 = a.scale * kLog2eB;
    // the row's lse (times log2 e) and delta; a row past the shard, or one that
    // saw no key, gets lse = +inf so that p = 0
    float nl2 = -INFINITY, ndl = 0.f;
    if (row < nq) {
      const int64_t o = b * a.l_bstride + static_cast<int64_t>(h) * a.S + q0 + row;
      const float l = a.lse[o];
      nl2 = l == -INFINITY ? -INFINITY : -l * kLog2eB;
      ndl = -a.delta[o];
    }
    // this row's Q (column half 0) or dO (half 1) into TMEM as the A operand
    // of S and dP: column c holds elements 2c and 2c + 1 of the row, which is
    // the row's memory read as 32-bit words; rows past the shard are zero
    // (they take no part)
    {
      const int64_t ro = b * a.bstride + static_cast<int64_t>(q0 + row) * a.sstride + static_cast<int64_t>(h) * D;
      {
        const int g = hc;
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(g == 0 ? a.q : a.dout) + ro);
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          uint32_t w[32];
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            const uint4 u = row < nq ? src[c * 8 + x] : make_uint4(0u, 0u, 0u, 0u);
            w[4 * x] = u.x;
            w[4 * x + 1] = u.y;
            w[4 * x + 2] = u.z;
            w[4 * x + 3] = u.w;
          }
          tmem_st32(tmem + lane_off + 384 + g * (D / 2) + c * 32, w);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kDqBarQ));
    }
    bool ok = true;
    KvWalk cur;
    cur.init(a, r);
    for (int j = 0; j < NJ; ++j) {
      const int ts = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kDqBarSFull + ts), (j >> 1) & 1, abort_flag, a.err, tmo));
      if (!ok) break;
      tc_fence_after();
      const uint32_t t_s = tmem + lane_off + ts * 128, t_dp = t_s + kSub;  // this sub-step's slot
      const int nvk = cur.nvalid();
      {
        const int c = hc;
        uint32_t sr[32], dr[32];
        tmem_ld32(t_s + c * 32, sr);
        tmem_ld32(t_dp + c * 32, dr);
        tmem_wait_ld();
        uint32_t dd[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float t0, t1, g0, g1, d0, d1;
          fma_f32x2(t0, t1, u2f(sr[e]), u2f(sr[e + 1]), c2, nl2);
          fma_f32x2(g0, g1, u2f(dr[e]), u2f(dr[e + 1]), 1.f, ndl);
          const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
          fma2(d0, d1, p0, p1, g0, g1, 0.f, 0.f);
          // keys past the sub-tile (the next block's rows, or zero fill) take no part
          d0 = c * 32 + e < nvk ? d0 : 0.f;
          d1 = c * 32 + e + 1 < nvk ? d1 : 0.f;
          dd[e >> 1] = pack_bf16x2(d0, d1);
        }
        // dS over the first half of this warp's S columns
        tmem_st16(t_s + c * 32, dd);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kDqBarPFull + ts));
      cur.advance(a, r);
    }
    // ---- dq of this CTA's rows ----
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kDqBarDone), 0, abort_flag, a.err, tmo));
    if (ok) {
      tc_fence_after();
      float* dst = a.dq + b * a.bstride + static_cast<int64_t>(q0 + row) * a.sstride + h * D;
#pragma unroll 1
      for (int c = hc * (D / 64); c < (hc + 1) * (D / 64); ++c) {  // this half's D / 2 columns
        uint32_t rr[32];
        tmem_ld32(tmem + lane_off + 256 + c * 32, rr);
        tmem_wait_ld();
        if (row < nq) {
#pragma unroll
          for (int x = 0; x < 32; x += 4)
            *reinterpret_cast<float4*>(dst + c * 32 + x) =
                make_float4(u2f(rr[x]) * a.scale, u2f(rr[x + 1]) * a.scale, u2f(rr[x + 2]) * a.scale,
                            u2f(rr[x + 3]) * a.scale);
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
    tmem_dealloc(tmem, kTmemColsB);
  }
}

template <int D>
__host__ __device__ constexpr int bwd_tc_alloc() {
  return BSmem<D>::kAlloc > DqSmem<D>::kAlloc ? BSmem<D>::kAlloc : DqSmem<D>::kAlloc;
}

// Both kinds of CTA in one launch, the dk/dv CTAs (the longer ones) first:
// the dq CTAs then fill the SMs that the last wave of dk/dv CTAs leaves idle,
// and neither kind waits for the other's tail. The two kinds are independent
// (they read the same inputs and write dk, dv or dq).
template <int D>
__global__ void __launch_bounds__(kThreadsB, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tq64, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to64,
                       const __grid_constant__ CUtensorMap tk64, const __grid_constant__ CUtensorMap tv64,
                       const __grid_constant__ BwdArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int nkv = a.kv_prefix[a.n], nq = a.q_prefix[a.n];
  const int kv_ctas = nkv * a.H * a.B;
  const int id = static_cast<int>(blockIdx.x);
  if (id < kv_ctas) {
    bwd_dkdv_cta<D>(tq64, tk, tv, to64, a, smem_raw, bwd_tc_alloc<D>(), id % nkv, (id / nkv) % a.H, id / (nkv * a.H));
  } else {
    const int i = id - kv_ctas;
    bwd_dq_cta<D>(tk64, tv64, a, smem_raw, bwd_tc_alloc<D>(), i % nq, (i / nq) % a.H, i / (nq * a.H));
  }
}

template <int D>
cudaError_t launch_bwd_tc_d(const BwdArgs& a, const BwdTensorMaps& m, cudaStream_t s) {
  constexpr int kAlloc = bwd_tc_alloc<D>();
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
  if (e != cudaSuccess) return e;
  const int64_t ctas = (static_cast<int64_t>(a.kv_prefix[a.n]) + a.q_prefix[a.n]) * a.H * a.B;
  if (ctas == 0) return cudaSuccess;
  if (ctas > 0x7fffffff) return cudaErrorInvalidValue;
  attn_bwd_tc_kernel<D><<<static_cast<unsigned>(ctas), kThreadsB, kAlloc, s>>>(m.q64, m.k, m.v, m.o64, m.k64, m.v64, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd_tc(const BwdArgs& a, int D, const BwdTensorMaps& m, cudaStream_t s) {
  if (D == 128) return launch_bwd_tc_d<128>(a, m, s);
  if (D == 64) return launch_bwd_tc_d<64>(a, m, s);
  return cudaErrorInvalidValue;
}

}  // namespace cp
