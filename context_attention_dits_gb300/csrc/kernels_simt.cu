// kernels_simt.cu — the CUDA-core kernels of libcpattn.so:
//   * block attention for fp32 q/k/v (one warp per query row, lanes split D,
//     dot products and the online max/sum reduced with warp shuffles);
//   * the fp32 LSE merge of a block partial into the accumulator
//     (bandwidth-bound, 128-bit loads and stores);
//   * the segment copy behind the Ulysses seq<->head regroups (bandwidth-bound,
//     one warp per contiguous segment, 128-bit vectors).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "cp_internal.h"

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
    for (int key = off; key < off + len; ++key) {
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
// LSE merge. One CTA = kMergeTok consecutive tokens of one batch entry, all H
// heads: the (h, token) weights are computed once into shared memory, then
// the contiguous [kMergeTok, H, D] slab of out rows is streamed as float4.
// ----------------------------------------------------------------------------
constexpr int kMergeTok = 8;
constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads) lse_merge_kernel(float* __restrict__ out_acc, float* __restrict__ lse_acc,
                                                                  const float* __restrict__ out_blk,
                                                                  const float* __restrict__ lse_blk, int H, int S,
                                                                  int D) {
  extern __shared__ float wsm[];  // [2][H][kMergeTok]: weight of acc, weight of blk
  const int b = blockIdx.y;
  const int t0 = blockIdx.x * kMergeTok;
  const int nt = min(kMergeTok, S - t0);
  float* wa = wsm;
  float* wb = wsm + H * kMergeTok;
  for (int idx = threadIdx.x; idx < H * kMergeTok; idx += blockDim.x) {
    const int hh = idx / kMergeTok, tt = idx % kMergeTok;
    if (tt >= nt) continue;
    const int64_t li = (static_cast<int64_t>(b) * H + hh) * S + t0 + tt;
    const float la = lse_acc[li], lb = lse_blk[li];
    const float m = fmaxf(la, lb);
    float ea = 0.f, eb = 0.f, lse = -INFINITY;
    if (m != -INFINITY) {
      const float xa = expf(la - m), xb = expf(lb - m);
      lse = m + logf(xa + xb);
      ea = expf(la - lse);
      eb = expf(lb - lse);
    }
    wa[idx] = ea;
    wb[idx] = eb;
    lse_acc[li] = lse;
  }
  __syncthreads();
  const int64_t base = (static_cast<int64_t>(b) * S + t0) * H * D;
  const int nvec = nt * H * D / 4;
  const int dv = D / 4;
  float4* oa = reinterpret_cast<float4*>(out_acc + base);
  const float4* ob = reinterpret_cast<const float4*>(out_blk + base);
#pragma unroll 4
  for (int v = threadIdx.x; v < nvec; v += kMergeThreads) {
    const int rowi = v / dv;  // (token, head) row within the slab
    const int tt = rowi / H, hh = rowi - tt * H;
    const float x = wa[hh * kMergeTok + tt], y = wb[hh * kMergeTok + tt];
    const float4 p = oa[v], q = ob[v];
    float4 o;
    o.x = x * p.x + y * q.x;
    o.y = x * p.y + y * q.y;
    o.z = x * p.z + y * q.z;
    o.w = x * p.w + y * q.w;
    oa[v] = o;
  }
}

// ----------------------------------------------------------------------------
// Segment copy: warp w copies output segment w (grid-stride), reading the
// input segment at the strided offset. VEC-byte vectors.
// ----------------------------------------------------------------------------
template <typename V>
__global__ void __launch_bounds__(256) segment_copy_kernel(const SegCopy c) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t nseg = c.n0 * c.n1 * c.n2 * c.n3;
  const int64_t seg_bytes = c.seg_elems * c.elem_bytes;
  const int64_t nv = seg_bytes / static_cast<int64_t>(sizeof(V));
  const char* in = static_cast<const char*>(c.in);
  char* out = static_cast<char*>(c.out);
  for (int64_t sg = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); sg < nseg; sg += warps) {
    int64_t rest = sg;
    const int64_t i3 = rest % c.n3;
    rest /= c.n3;
    const int64_t i2 = rest % c.n2;
    rest /= c.n2;
    const int64_t i1 = rest % c.n1;
    const int64_t i0 = rest / c.n1;
    const int64_t src_el = i0 * c.st0 + i1 * c.st1 + i2 * c.st2 + i3 * c.st3;
    const V* src = reinterpret_cast<const V*>(in + src_el * c.elem_bytes);
    V* dst = reinterpret_cast<V*>(out + sg * seg_bytes);
    int64_t v = lane;
    for (; v + 96 < nv; v += 128) {
      const V x0 = src[v], x1 = src[v + 32], x2 = src[v + 64], x3 = src[v + 96];
      dst[v] = x0;
      dst[v + 32] = x1;
      dst[v + 64] = x2;
      dst[v + 96] = x3;
    }
    for (; v < nv; v += 32) dst[v] = src[v];
  }
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
  const size_t smem = 2 * static_cast<size_t>(H) * kMergeTok * sizeof(float);
  dim3 grid((S + kMergeTok - 1) / kMergeTok, B);
  lse_merge_kernel<<<grid, kMergeThreads, smem, s>>>(out_acc, lse_acc, out_blk, lse_blk, H, S, D);
  return cudaGetLastError();
}

cudaError_t launch_segment_copy(const SegCopy& c, cudaStream_t s) {
  const int64_t nseg = c.n0 * c.n1 * c.n2 * c.n3;
  if (nseg == 0 || c.seg_elems == 0) return cudaSuccess;
  const int64_t seg_bytes = c.seg_elems * c.elem_bytes;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (nseg + 7) / 8;                 // 8 warps per CTA, one segment each
  const int blocks = static_cast<int>(want < sms * 8LL ? want : sms * 8LL);
  uint64_t align = static_cast<uint64_t>(seg_bytes) | reinterpret_cast<uintptr_t>(c.in) |
                   reinterpret_cast<uintptr_t>(c.out);
  for (int64_t st : {c.st0, c.st1, c.st2, c.st3}) align |= static_cast<uint64_t>(st * c.elem_bytes);
  if (align % 16 == 0) segment_copy_kernel<uint4><<<blocks, 256, 0, s>>>(c);
  else if (align % 8 == 0) segment_copy_kernel<uint2><<<blocks, 256, 0, s>>>(c);
  else if (align % 4 == 0) segment_copy_kernel<uint32_t><<<blocks, 256, 0, s>>>(c);
  else segment_copy_kernel<uint8_t><<<blocks, 256, 0, s>>>(c);
  return cudaGetLastError();
}

}  // namespace cp
