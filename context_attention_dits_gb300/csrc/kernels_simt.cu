// kernels_simt.cu — the CUDA-core kernels of libcpattn.so:
//   * block attention for fp32 q/k/v (one warp per query row, lanes split D,
//     dot products and the online max/sum reduced with warp shuffles);
//   * the fp32 LSE merge of a block partial into the accumulator
//     (bandwidth-bound, 128-bit loads and stores);
//   * the segment copy behind the Ulysses seq<->head regroups (bandwidth-bound):
//     bulk TMA copies through a shared-memory ring when segments are 16-byte
//     multiples of a few hundred bytes or more (up to 24 independent copies
//     per launch), else warps of 128-bit vectors.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "cp_internal.h"
#include "cp_ptx.cuh"

namespace cp {
namespace {

// ----------------------------------------------------------------------------
// fp32 block attention. Same ring walk as the tensor-core kernel: rank r's
// rows visit blocks (r - t) mod n_kv, t = 0.. (or the single step g.step),
// and the online-softmax state carried across blocks is their LSE merge.
// ----------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(32 * kF32RowsPerCta) attn_fwd_f32_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int NPL = D / 32;  // elements of a row per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (attn_head_is_padding(a, h, b)) return;
  int r = 0;
  while (r + 1 < a.g.n_q && a.g.cta_prefix[r + 1] <= item) ++r;
  const int row = (item - a.g.cta_prefix[r]) * kF32RowsPerCta + warp;
  if (row >= a.g.q_len[r]) return;
  const int tok = a.g.q_off[r] + row;

  const float* qrow = a.qf + b * a.q_bstride + tok * a.q_sstride + h * D;
  float qv[NPL], acc[NPL];
#pragma unroll
  for (int c = 0; c < NPL; ++c) {
    qv[c] = qrow[lane + 32 * c] * a.scale;
    acc[c] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int nblk = a.g.step >= 0 ? 1 : a.g.n_kv;
  for (int t = 0; t < nblk; ++t) {
    const int s = a.g.step >= 0 ? a.g.step : t;
    int j = (r - s) % a.g.n_kv;
    if (j < 0) j += a.g.n_kv;
    const int off = a.g.kv_off[j], len = a.g.kv_len[j];
    const uint8_t* km = a.kmask ? a.kmask + (b % a.km_bmod) * a.km_bstride : nullptr;
    for (int key = off; key < off + len; ++key) {
      if (km && km[key] == 0) continue;  // masked key: no part in the softmax
      const float* krow = a.kf + b * a.kv_bstride + key * a.kv_sstride + h * D;
      const float* vrow = a.vf + b * a.kv_bstride + key * a.kv_sstride + h * D;
      float part = 0.f;
#pragma unroll
      for (int c = 0; c < NPL; ++c) part = fmaf(qv[c], krow[lane + 32 * c], part);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      const float m_new = fmaxf(m, part);
      const float f = expf(m - m_new);  // 0 for the first key (m = -inf)
      const float p = expf(part - m_new);
      l = l * f + p;
#pragma unroll
      for (int c = 0; c < NPL; ++c) acc[c] = fmaf(acc[c], f, p * vrow[lane + 32 * c]);
      m = m_new;
    }
  }
  float* orow = a.out + b * a.o_bstride + tok * a.o_sstride + h * D;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int c = 0; c < NPL; ++c) orow[lane + 32 * c] = acc[c] * inv;
  if (lane == 0) a.lse[b * a.l_bstride + h * a.l_hstride + tok] = l > 0.f ? m + logf(l) : -INFINITY;
}

// ----------------------------------------------------------------------------
// LSE merge. Grid: x over token chunks, y over (batch, head) pairs, so a
// CTA's rows share b and h and no index needs a division. A group of g lanes
// owns one (b, token, h) row of D/4 float4 (g = D/4 when that divides 32,
// else 32 lanes looping over the row); a warp takes 32/g rows per slot and
// kMergeRows slots per pass. The rows' out loads are issued first, then their
// LSE loads, so a pass waits for one memory round trip. Each lane computes
// its row's weights itself, and the first lane of the row writes the merged
// LSE once every lane of the row has read the old one.
// ----------------------------------------------------------------------------
constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMergeRows = 4;

struct MergeW {
  float wa, wb, lse;
};

__device__ __forceinline__ MergeW merge_weights(float la, float lb) {
  const float m = fmaxf(la, lb);
  if (m == -INFINITY) return {0.f, 0.f, -INFINITY};  // both partials empty
  const float xa = __expf(la - m), xb = __expf(lb - m);  // one of them is exactly 1
  const float sum = xa + xb;
  const float inv = __fdividef(1.f, sum);
  return {xa * inv, xb * inv, m + __logf(sum)};
}

__device__ __forceinline__ float4 merge4(const MergeW& w, const float4& p, const float4& q) {
  return make_float4(w.wa * p.x + w.wb * q.x, w.wa * p.y + w.wb * q.y, w.wa * p.z + w.wb * q.z,
                     w.wa * p.w + w.wb * q.w);
}

// Idx: the index type, int when every float4 and LSE index fits (the host
// checks). kOneVec: D/4 divides 32, so each lane holds one float4 of a row.
template <typename Idx, bool kOneVec>
__global__ void __launch_bounds__(kMergeThreads, 4) lse_merge_kernel(float* __restrict__ out_acc,
                                                                     float* __restrict__ lse_acc,
                                                                     const float* __restrict__ out_blk,
                                                                     const float* __restrict__ lse_blk, int B, int H,
                                                                     int S, int dv) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = (dv <= 32 && 32 % dv == 0) ? dv : 32;  // lanes per row
  const int rpw = 32 / g;                               // rows per warp slot
  const int sub = lane / g, j0 = lane - sub * g;
  const int per_cta = kMergeWarps * kMergeRows * rpw;  // tokens per CTA and (b, h)
  const int s0 = blockIdx.x * per_cta;
  float4* oa = reinterpret_cast<float4*>(out_acc);
  const float4* ob = reinterpret_cast<const float4*>(out_blk);
  for (int bh = blockIdx.y; bh < B * H; bh += gridDim.y) {
    const int b = bh / H, h = bh - b * H;
    const Idx lse0 = static_cast<Idx>(bh) * S;
    // float4 index of element (b, t, h, 0)
    auto vbase = [&](int t) { return ((static_cast<Idx>(b) * S + t) * H + h) * dv; };
    int tok[kMergeRows];
#pragma unroll
    for (int u = 0; u < kMergeRows; ++u) tok[u] = s0 + (u * kMergeWarps + warp) * rpw + sub;
    if (kOneVec) {
      float4 p[kMergeRows], q[kMergeRows];
#pragma unroll
      for (int u = 0; u < kMergeRows; ++u)
        if (tok[u] < S) {
          p[u] = oa[vbase(tok[u]) + j0];
          q[u] = ob[vbase(tok[u]) + j0];
        }
      float la[kMergeRows], lb[kMergeRows];
#pragma unroll
      for (int u = 0; u < kMergeRows; ++u) {
        la[u] = tok[u] < S ? lse_acc[lse0 + tok[u]] : -INFINITY;
        lb[u] = tok[u] < S ? lse_blk[lse0 + tok[u]] : -INFINITY;
      }
      __syncwarp();  // every lane of a row has read its old LSE
#pragma unroll
      for (int u = 0; u < kMergeRows; ++u)
        if (tok[u] < S) {
          const MergeW w = merge_weights(la[u], lb[u]);
          oa[vbase(tok[u]) + j0] = merge4(w, p[u], q[u]);
          if (j0 == 0) lse_acc[lse0 + tok[u]] = w.lse;
        }
    } else {
      MergeW w[kMergeRows];
#pragma unroll
      for (int u = 0; u < kMergeRows; ++u)
        w[u] = merge_weights(tok[u] < S ? lse_acc[lse0 + tok[u]] : -INFINITY,
                             tok[u] < S ? lse_blk[lse0 + tok[u]] : -INFINITY);
#pragma unroll
      for (int u = 0; u < kMergeRows; ++u)
        if (tok[u] < S)
          for (int j = j0; j < dv; j += g) oa[vbase(tok[u]) + j] = merge4(w[u], oa[vbase(tok[u]) + j],
                                                                          ob[vbase(tok[u]) + j]);
      __syncwarp();  // every lane of a row has read its old LSE
      if (j0 == 0) {
#pragma unroll
        for (int u = 0; u < kMergeRows; ++u)
          if (tok[u] < S) lse_acc[lse0 + tok[u]] = w[u].lse;
      }
    }
  }
}

// ----------------------------------------------------------------------------
// Segment copy: warp w copies a contiguous range of output segments, two at a
// time, advancing the strided input offset with carries (one index
// decomposition per warp); every lane issues up to kCopySegs x kCopyVec loads
// before its stores. VEC-byte vectors.
// ----------------------------------------------------------------------------
constexpr int kCopySegs = 2;
constexpr int kCopyVec = 4;

template <typename V>
__global__ void __launch_bounds__(256) segment_copy_kernel(const SegCopy c, int64_t per_warp) {
  const int lane = threadIdx.x & 31;
  const int64_t nseg = c.n0 * c.n1 * c.n2 * c.n3;
  const int64_t seg_bytes = c.seg_elems * c.elem_bytes;
  const int64_t nv = seg_bytes / static_cast<int64_t>(sizeof(V));
  const char* in = static_cast<const char*>(c.in);
  char* out = static_cast<char*>(c.out);
  int64_t sg = (static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * per_warp;
  const int64_t end = sg + per_warp < nseg ? sg + per_warp : nseg;
  if (sg >= end) return;
  const bool out_contig = (c.ost0 | c.ost1 | c.ost2 | c.ost3) == 0;
  int64_t rest = sg;
  int64_t i3 = rest % c.n3;
  rest /= c.n3;
  int64_t i2 = rest % c.n2;
  rest /= c.n2;
  int64_t i1 = rest % c.n1;
  int64_t src_el = (rest / c.n1) * c.st0 + i1 * c.st1 + i2 * c.st2 + i3 * c.st3;
  int64_t dst_el = (rest / c.n1) * c.ost0 + i1 * c.ost1 + i2 * c.ost2 + i3 * c.ost3;
  auto advance = [&]() {  // to the next segment in (i0, i1, i2, i3) order
    src_el += c.st3;
    dst_el += c.ost3;
    if (++i3 == c.n3) {
      i3 = 0;
      src_el += c.st2 - c.n3 * c.st3;
      dst_el += c.ost2 - c.n3 * c.ost3;
      if (++i2 == c.n2) {
        i2 = 0;
        src_el += c.st1 - c.n2 * c.st2;
        dst_el += c.ost1 - c.n2 * c.ost2;
        if (++i1 == c.n1) {
          i1 = 0;
          src_el += c.st0 - c.n1 * c.st1;
          dst_el += c.ost0 - c.n1 * c.ost1;
        }
      }
    }
  };
  for (; sg < end; sg += kCopySegs) {
    const V* src[kCopySegs];
    V* dst[kCopySegs];
    bool ok[kCopySegs];
#pragma unroll
    for (int k = 0; k < kCopySegs; ++k) {
      ok[k] = sg + k < end;
      src[k] = reinterpret_cast<const V*>(in + src_el * c.elem_bytes);
      dst[k] = reinterpret_cast<V*>(out + (out_contig ? (sg + k) * seg_bytes : dst_el * c.elem_bytes));
      if (ok[k]) advance();
    }
    for (int64_t base = 0; base < nv; base += 32 * kCopyVec) {
      V x[kCopySegs][kCopyVec];
#pragma unroll
      for (int k = 0; k < kCopySegs; ++k)
#pragma unroll
        for (int j = 0; j < kCopyVec; ++j) {
          const int64_t v = base + lane + 32 * j;
          if (ok[k] && v < nv) x[k][j] = src[k][v];
        }
#pragma unroll
      for (int k = 0; k < kCopySegs; ++k)
#pragma unroll
        for (int j = 0; j < kCopyVec; ++j) {
          const int64_t v = base + lane + 32 * j;
          if (ok[k] && v < nv) dst[k][v] = x[k][j];
        }
    }
  }
}

// The same copy for few, long segments: each segment is cut into `parts`
// ranges of chunk_v vectors, and each warp copies one (segment, range) unit,
// so that the copy spreads over the GPU instead of a few warps walking whole
// segments.
template <typename V>
__global__ void __launch_bounds__(256) segment_copy_parts_kernel(const SegCopy c, int64_t parts, int64_t chunk_v) {
  const int lane = threadIdx.x & 31;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nseg = c.n0 * c.n1 * c.n2 * c.n3;
  if (unit >= nseg * parts) return;
  const int64_t seg = unit / parts, part = unit - seg * parts;
  const int64_t nv = c.seg_elems * c.elem_bytes / static_cast<int64_t>(sizeof(V));
  const int64_t v0 = part * chunk_v, v1 = v0 + chunk_v < nv ? v0 + chunk_v : nv;
  int64_t rest = seg;
  const int64_t i3 = rest % c.n3;
  rest /= c.n3;
  const int64_t i2 = rest % c.n2;
  rest /= c.n2;
  const int64_t i1 = rest % c.n1, i0 = rest / c.n1;
  const bool out_contig = (c.ost0 | c.ost1 | c.ost2 | c.ost3) == 0;
  const int64_t src_el = i0 * c.st0 + i1 * c.st1 + i2 * c.st2 + i3 * c.st3;
  const int64_t dst_b = out_contig ? seg * c.seg_elems * c.elem_bytes
                                   : (i0 * c.ost0 + i1 * c.ost1 + i2 * c.ost2 + i3 * c.ost3) * c.elem_bytes;
  const V* src = reinterpret_cast<const V*>(static_cast<const char*>(c.in) + src_el * c.elem_bytes);
  V* dst = reinterpret_cast<V*>(static_cast<char*>(c.out) + dst_b);
  for (int64_t base = v0; base < v1; base += 32 * kCopyVec) {
    V x[kCopyVec];
#pragma unroll
    for (int j = 0; j < kCopyVec; ++j) {
      const int64_t v = base + lane + 32 * j;
      if (v < v1) x[j] = src[v];
    }
#pragma unroll
    for (int j = 0; j < kCopyVec; ++j) {
      const int64_t v = base + lane + 32 * j;
      if (v < v1) dst[v] = x[j];
    }
  }
}

// ----------------------------------------------------------------------------
// Segment copy with bulk TMA copies. One thread per CTA walks a contiguous
// range of output segments in chunks of K consecutive segments (K * segment
// bytes <= one ring slot): K bulk loads gather a chunk's segments from their
// strided sources into a shared-memory slot (completing on the slot's
// mbarrier), and one bulk store writes the slot to the chunk's contiguous
// output range. Loads run kBulkSlots - 1 chunks ahead of stores; a slot is
// refilled only after the store that last read it has finished reading.
// Every wait is bounded; on expiry the thread records the timeout, waits
// (bounded) for its in-flight loads and all its stores, and returns.
// ----------------------------------------------------------------------------
constexpr int kBulkSlots = 4;
constexpr uint64_t kCopyWaitTimeoutNs = 1000000000ull;  // 1 s per device-side wait
constexpr int kBulkSlotBytes = 24 * 1024;
constexpr int kBulkSmem = kBulkSlots * kBulkSlotBytes;

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Bounded wait for phase `parity` of an mbarrier; false on expiry.
__device__ __forceinline__ bool bulk_bar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1; !mbar_try_wait(bar, parity); ++n)
    if ((n & 255u) == 0 && global_timer_ns() - t0 > timeout_ns) return false;
  return true;
}

// One copy of a batch: its descriptor (all output strides 0 when the output
// is contiguous in segment order), segments per CTA and segments per ring slot.
struct BulkCopy {
  SegCopy c;
  int64_t per_cta;
  int K;
};
constexpr int kMaxBulkBatch = 24;
struct BulkBatch {
  BulkCopy d[kMaxBulkBatch];
};

// Position of one segment in (i0, i1, i2, i3) order and its element offset
// under strides (s0, s1, s2, s3).
struct SegIter {
  int64_t i1, i2, i3, el;
  __device__ __forceinline__ void init(const SegCopy& c, int64_t sg, int64_t s0, int64_t s1, int64_t s2, int64_t s3) {
    i3 = sg % c.n3;
    sg /= c.n3;
    i2 = sg % c.n2;
    sg /= c.n2;
    i1 = sg % c.n1;
    el = (sg / c.n1) * s0 + i1 * s1 + i2 * s2 + i3 * s3;
  }
  __device__ __forceinline__ void next(const SegCopy& c, int64_t s0, int64_t s1, int64_t s2, int64_t s3) {
    el += s3;
    if (++i3 == c.n3) {
      i3 = 0;
      el += s2 - c.n3 * s3;
      if (++i2 == c.n2) {
        i2 = 0;
        el += s1 - c.n2 * s2;
        if (++i1 == c.n1) {
          i1 = 0;
          el += s0 - c.n1 * s1;
        }
      }
    }
  }
};

// blockIdx.y picks the copy of the batch, blockIdx.x its range of segments.
__global__ void __launch_bounds__(32) segment_copy_bulk_kernel(const __grid_constant__ BulkBatch batch,
                                                               uint32_t* err, uint64_t timeout_ns) {
  const BulkCopy& d = batch.d[blockIdx.y];
  const SegCopy& c = d.c;
  const int64_t per_cta = d.per_cta;
  const int K = d.K;
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t bars[kBulkSlots];
  if (threadIdx.x != 0) return;
  const int64_t nseg = c.n0 * c.n1 * c.n2 * c.n3;
  const int64_t seg_bytes = c.seg_elems * c.elem_bytes;
  const int64_t sg0 = static_cast<int64_t>(blockIdx.x) * per_cta;
  const int64_t end = sg0 + per_cta < nseg ? sg0 + per_cta : nseg;
  if (sg0 >= end) return;
  for (int i = 0; i < kBulkSlots; ++i) mbar_init(smem_addr(&bars[i]), 1);
  fence_mbar_init();
  const char* in = static_cast<const char*>(c.in);
  char* out = static_cast<char*>(c.out);
  const bool strided_out = (c.ost0 | c.ost1 | c.ost2 | c.ost3) != 0;
  SegIter src, dst;  // next segment to load, next segment to store (strided output)
  src.init(c, sg0, c.st0, c.st1, c.st2, c.st3);
  dst.init(c, sg0, c.ost0, c.ost1, c.ost2, c.ost3);
  const int64_t nchunks = (end - sg0 + K - 1) / K;
  const uint32_t ring0 = smem_addr(ring);
  int64_t loaded = 0;  // chunks whose loads were issued
  bool ok = true;
  for (int64_t ci = 0; ci < nchunks + (kBulkSlots - 1) && ok; ++ci) {
    if (ci < nchunks) {
      const int slot = static_cast<int>(ci % kBulkSlots);
      if (ci >= kBulkSlots) bulk_wait_read_all();  // the store that last read this slot
      const int64_t first = sg0 + ci * K;
      const int n = static_cast<int>(end - first < K ? end - first : K);
      const uint32_t bar = smem_addr(&bars[slot]);
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n * seg_bytes));
      for (int k = 0; k < n; ++k) {
        bulk_load(ring0 + slot * kBulkSlotBytes + static_cast<uint32_t>(k * seg_bytes), in + src.el * c.elem_bytes,
                  static_cast<uint32_t>(seg_bytes), bar);
        src.next(c, c.st0, c.st1, c.st2, c.st3);
      }
      ++loaded;
    }
    const int64_t cj = ci - (kBulkSlots - 1);
    if (cj >= 0 && cj < nchunks) {
      const int slot = static_cast<int>(cj % kBulkSlots);
      if (!bulk_bar_wait(smem_addr(&bars[slot]), static_cast<uint32_t>((cj / kBulkSlots) & 1), timeout_ns)) {
        atomicOr(err, kDevErrTimeout);
        ok = false;
        break;
      }
      const int64_t first = sg0 + cj * K;
      const int64_t n = end - first < K ? end - first : K;
      if (!strided_out) {
        bulk_store(out + first * seg_bytes, ring0 + slot * kBulkSlotBytes, static_cast<uint32_t>(n * seg_bytes));
      } else {
        for (int64_t k = 0; k < n; ++k) {
          bulk_store(out + dst.el * c.elem_bytes, ring0 + slot * kBulkSlotBytes + static_cast<uint32_t>(k * seg_bytes),
                     static_cast<uint32_t>(seg_bytes));
          dst.next(c, c.ost0, c.ost1, c.ost2, c.ost3);
        }
      }
    }
  }
  if (!ok) {
    // let every issued load land before the CTA's shared memory goes away
    for (int64_t cj = loaded - kBulkSlots < 0 ? 0 : loaded - kBulkSlots; cj < loaded; ++cj)
      (void)bulk_bar_wait(smem_addr(&bars[cj % kBulkSlots]), static_cast<uint32_t>((cj / kBulkSlots) & 1),
                          timeout_ns);
  }
  bulk_wait_all();
}

template <int D>
cudaError_t launch_f32_d(const AttnArgs& a, cudaStream_t s) {
  dim3 grid(a.g.cta_prefix[a.g.n_q], a.H, a.B);
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  attn_fwd_f32_kernel<D><<<grid, 32 * kF32RowsPerCta, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_f32(const AttnArgs& a, cudaStream_t s) {
  if (a.D == 64) return launch_f32_d<64>(a, s);
  if (a.D == 128) return launch_f32_d<128>(a, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_lse_merge(float* out_acc, float* lse_acc, const float* out_blk, const float* lse_blk, int B, int H,
                             int S, int D, cudaStream_t s) {
  if (B == 0 || S == 0 || H == 0) return cudaSuccess;
  const int dv = D / 4;
  const int g = (dv <= 32 && 32 % dv == 0) ? dv : 32;
  const int per_cta = kMergeWarps * kMergeRows * (32 / g);
  const int64_t bh = static_cast<int64_t>(B) * H;
  dim3 grid((S + per_cta - 1) / per_cta, static_cast<unsigned>(bh < 65535 ? bh : 65535));
  const bool small = bh * S * dv < (1LL << 31);
  if (g == dv && small)
    lse_merge_kernel<int, true><<<grid, kMergeThreads, 0, s>>>(out_acc, lse_acc, out_blk, lse_blk, B, H, S, dv);
  else if (g == dv)
    lse_merge_kernel<int64_t, true><<<grid, kMergeThreads, 0, s>>>(out_acc, lse_acc, out_blk, lse_blk, B, H, S, dv);
  else
    lse_merge_kernel<int64_t, false><<<grid, kMergeThreads, 0, s>>>(out_acc, lse_acc, out_blk, lse_blk, B, H, S, dv);
  return cudaGetLastError();
}

static int sm_count() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

// Whether copy c can take the bulk path: 16-byte aligned addresses and
// strides, and segments of 256 B to one ring slot.
static bool bulk_eligible(const SegCopy& c) {
  const int64_t seg_bytes = c.seg_elems * c.elem_bytes;
  uint64_t align = static_cast<uint64_t>(seg_bytes) | reinterpret_cast<uintptr_t>(c.in) |
                   reinterpret_cast<uintptr_t>(c.out);
  for (int64_t st : {c.st0, c.st1, c.st2, c.st3, c.ost0, c.ost1, c.ost2, c.ost3})
    align |= static_cast<uint64_t>(st * c.elem_bytes);
  return align % 16 == 0 && seg_bytes >= 256 && seg_bytes <= kBulkSlotBytes;
}

// c with all output strides 0 when they describe the contiguous layout (a
// stride of a dimension of extent 1 never matters), so that the kernel
// stores whole chunks.
static SegCopy normalise_out(SegCopy c) {
  const int64_t nat3 = c.seg_elems, nat2 = c.n3 * nat3, nat1 = c.n2 * nat2, nat0 = c.n1 * nat1;
  if ((c.n3 == 1 || c.ost3 == nat3) && (c.n2 == 1 || c.ost2 == nat2) && (c.n1 == 1 || c.ost1 == nat1) &&
      (c.n0 == 1 || c.ost0 == nat0))
    c.ost0 = c.ost1 = c.ost2 = c.ost3 = 0;
  return c;
}

static int64_t seg_count(const SegCopy& c) { return c.n0 * c.n1 * c.n2 * c.n3; }

// One bulk launch for n (1..kMaxBulkBatch) eligible, non-empty copies. Two
// CTAs per SM (two rings fit in shared memory), split among the copies in
// proportion to their chunks, at least one each.
static cudaError_t launch_bulk(const SegCopy* const* cs, int n, cudaStream_t s) {
  uint32_t* err = device_error_word();
  if (err == nullptr) return cudaErrorUnknown;
  static_assert(kBulkSmem <= 227 * 1024, "shared memory budget");
  static_assert(sizeof(BulkBatch) <= 4096, "kernel parameter space");
  cudaError_t e = cudaFuncSetAttribute(segment_copy_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kBulkSmem);
  if (e != cudaSuccess) return e;
  const int64_t budget = 2LL * sm_count();
  int64_t chunks[kMaxBulkBatch], total = 0;
  for (int i = 0; i < n; ++i) {
    const int64_t K = kBulkSlotBytes / (cs[i]->seg_elems * cs[i]->elem_bytes);
    chunks[i] = (seg_count(*cs[i]) + K - 1) / K;
    total += chunks[i];
  }
  BulkBatch batch;
  int64_t grid = 1;
  for (int i = 0; i < kMaxBulkBatch; ++i) {
    BulkCopy& d = batch.d[i];
    d.c = normalise_out(*cs[i < n ? i : 0]);
    d.K = static_cast<int>(kBulkSlotBytes / (d.c.seg_elems * d.c.elem_bytes));
    if (i >= n) {  // unused entries: never read (gridDim.y == n)
      d.per_cta = 1;
      continue;
    }
    int64_t ctas = budget * chunks[i] / total;
    ctas = ctas < 1 ? 1 : (ctas > chunks[i] ? chunks[i] : ctas);
    d.per_cta = (chunks[i] + ctas - 1) / ctas * d.K;
    const int64_t g = (seg_count(d.c) + d.per_cta - 1) / d.per_cta;
    grid = g > grid ? g : grid;
  }
  segment_copy_bulk_kernel<<<dim3(static_cast<unsigned>(grid), static_cast<unsigned>(n)), 32, kBulkSmem, s>>>(
      batch, err, kCopyWaitTimeoutNs);
  return cudaGetLastError();
}

// One launch of the vector kernel for copy c.
static cudaError_t launch_vector(const SegCopy& c, cudaStream_t s) {
  const int64_t nseg = seg_count(c);
  const int64_t seg_bytes = c.seg_elems * c.elem_bytes;
  const int sms = sm_count();
  uint64_t align = static_cast<uint64_t>(seg_bytes) | reinterpret_cast<uintptr_t>(c.in) |
                   reinterpret_cast<uintptr_t>(c.out);
  for (int64_t st : {c.st0, c.st1, c.st2, c.st3, c.ost0, c.ost1, c.ost2, c.ost3})
    align |= static_cast<uint64_t>(st * c.elem_bytes);
  // few, long segments (fewer than one per resident warp, each many
  // vector rounds): a warp per part of a segment instead
  auto launch_parts = [&](auto kernel, int64_t vec_bytes) -> bool {
    const int64_t nv = seg_bytes / vec_bytes;
    const int64_t warps_cap = static_cast<int64_t>(sms) * 2 * 8;
    const int64_t round = 32 * kCopyVec;  // vectors a warp moves per round
    if (nseg * 4 > warps_cap || nv < 8 * round) return false;
    int64_t parts = warps_cap / nseg;
    if (parts > nv / (4 * round)) parts = nv / (4 * round);  // at least 4 rounds per part
    if (parts < 2) return false;
    const int64_t chunk_v = (nv + parts - 1) / parts;
    parts = (nv + chunk_v - 1) / chunk_v;
    const int64_t blocks = (nseg * parts + 7) / 8;
    kernel<<<static_cast<int>(blocks), 256, 0, s>>>(c, parts, chunk_v);
    return true;
  };
  auto launch = [&](auto kernel) {
    int per_sm = 1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0);
    // one resident wave of 8-warp CTAs, each warp a contiguous range of segments
    const int64_t warps_cap = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1) * 8;
    const int64_t warps_want = (nseg + kCopySegs - 1) / kCopySegs;
    const int64_t warps = warps_want < warps_cap ? warps_want : warps_cap;
    const int64_t per_warp = (nseg + warps - 1) / warps;
    const int64_t blocks = ((nseg + per_warp - 1) / per_warp + 7) / 8;
    kernel<<<static_cast<int>(blocks), 256, 0, s>>>(c, per_warp);
    return cudaGetLastError();
  };
  if (align % 16 == 0)
    return launch_parts(segment_copy_parts_kernel<uint4>, 16) ? cudaGetLastError() : launch(segment_copy_kernel<uint4>);
  if (align % 8 == 0)
    return launch_parts(segment_copy_parts_kernel<uint2>, 8) ? cudaGetLastError() : launch(segment_copy_kernel<uint2>);
  if (align % 4 == 0)
    return launch_parts(segment_copy_parts_kernel<uint32_t>, 4) ? cudaGetLastError()
                                                                : launch(segment_copy_kernel<uint32_t>);
  return launch_parts(segment_copy_parts_kernel<uint8_t>, 1) ? cudaGetLastError() : launch(segment_copy_kernel<uint8_t>);
}

// The bulk-eligible, non-empty copies go in batches of up to kMaxBulkBatch;
// every other non-empty copy takes a vector launch of its own. Returns the
// number of launches, or -1 on a launch error (when s is used).
static int segment_copies(const SegCopy* cs, int n, cudaStream_t s, bool launch) {
  const SegCopy* batch[kMaxBulkBatch];
  int nb = 0, launches = 0;
  for (int i = 0; i < n; ++i) {
    if (seg_count(cs[i]) == 0 || cs[i].seg_elems == 0) continue;
    if (!bulk_eligible(cs[i])) {
      ++launches;
      if (launch && launch_vector(cs[i], s) != cudaSuccess) return -1;
      continue;
    }
    batch[nb++] = &cs[i];
    if (nb == kMaxBulkBatch) {
      ++launches;
      if (launch && launch_bulk(batch, nb, s) != cudaSuccess) return -1;
      nb = 0;
    }
  }
  if (nb > 0) {
    ++launches;
    if (launch && launch_bulk(batch, nb, s) != cudaSuccess) return -1;
  }
  return launches;
}

cudaError_t launch_segment_copies(const SegCopy* cs, int n, cudaStream_t s) {
  return segment_copies(cs, n, s, true) < 0 ? cudaErrorLaunchFailure : cudaSuccess;
}

cudaError_t launch_segment_copy(const SegCopy& c, cudaStream_t s) { return launch_segment_copies(&c, 1, s); }

int segment_copy_launches(const SegCopy* cs, int n) { return segment_copies(cs, n, nullptr, false); }

}  // namespace cp
