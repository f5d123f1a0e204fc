// attn_bwd.cu — backward of block / ring attention on CUDA cores (fp32 math).
//
// Gradients of L = sum(out * dout) for out = softmax(scale * q k^T) v, using
// the forward's global lse and delta_i = sum_d dout_id out_id:
//   p_ij  = exp(scale * q_i . k_j - lse_i)
//   dv_j  = sum_i p_ij dout_i
//   ds_ij = p_ij (dout_i . v_j - delta_i)
//   dq_i  = scale * sum_j ds_ij k_j,   dk_j = scale * sum_i ds_ij q_i
// (context parallelism page, Ring Attention and Ulysses Attention sections:
// the plain variants serve training; the variants table marks Ring Anything
// as inference only.)
//
// Three kernels:
//   * delta: one warp per (b, s, h) row, delta[b, h, s] = out_row . dout_row;
//   * dq: a CTA owns 64 query rows of one (b, h) and walks the K/V blocks of
//     its shard's ring lap, (r - t) mod n, in 64-key tiles; dq stays in
//     registers and is stored once;
//   * dk/dv: a CTA owns 64 keys of one (b, h) and walks the query shards in
//     the order its block visits the ranks, (j + t) mod n, in 32-row tiles;
//     dk and dv stay in registers and are stored once.
// Both recompute p from q, k and lse, so neither needs atomics. Tiles live in
// shared memory as fp32, transposed where a product reads them by column, so
// that every inner loop reads 16-byte vectors.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "cp_internal.h"

namespace cp {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBwdThreads = 256;
constexpr int kBT = kBwdTile;  // dq kernel: query rows and keys per tile; dk/dv kernel: keys per CTA
constexpr int kBQ = 32;        // dk/dv kernel: query rows per tile
constexpr int kTP = kBT + 4;   // padded row of a transposed 64-wide tile
constexpr int kTQ = kBQ + 4;   // padded row of a transposed 32-wide tile

__device__ __forceinline__ void load4(const float* p, float x[4]) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  x[0] = v.x;
  x[1] = v.y;
  x[2] = v.z;
  x[3] = v.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float x[4]) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
  x[0] = a.x;
  x[1] = a.y;
  x[2] = b.x;
  x[3] = b.y;
}

// Rows tok0 .. tok0 + nrows - 1 of head h of batch entry b (rows past nrows
// up to `rows` are zero) times `mul`, into shared memory: transposed into
// t[d * tp + j] (lanes along rows, so the scattered stores hit distinct
// banks) and/or row-major into rm[j * D + d] (lanes along d).
template <int D, typename T>
__device__ __forceinline__ void load_tile(const T* base, int64_t bstride, int64_t sstride, int b, int h, int tok0,
                                          int nrows, int rows, float mul, float* t, int tp, float* rm) {
  constexpr int V4 = D / 4;
  const T* src = base + b * bstride + static_cast<int64_t>(tok0) * sstride + h * D;
  if (t != nullptr) {
    for (int e = threadIdx.x; e < rows * V4; e += kBwdThreads) {
      const int j = e % rows, d = (e / rows) * 4;
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      if (j < nrows) load4(src + j * sstride + d, x);
#pragma unroll
      for (int c = 0; c < 4; ++c) t[(d + c) * tp + j] = x[c] * mul;
    }
  }
  if (rm != nullptr) {
    for (int e = threadIdx.x; e < rows * V4; e += kBwdThreads) {
      const int j = e / V4, d = (e % V4) * 4;
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      if (j < nrows) load4(src + j * sstride + d, x);
      *reinterpret_cast<float4*>(rm + j * D + d) = make_float4(x[0] * mul, x[1] * mul, x[2] * mul, x[3] * mul);
    }
  }
}

// lse (times log2 e) and delta of rows tok0 .. tok0 + rows - 1; rows past
// nrows, and rows that saw no key (lse = -inf), get +inf so that p = 0.
__device__ __forceinline__ void load_row_stats(const BwdArgs& a, int b, int h, int tok0, int nrows, int rows,
                                               float* lse2, float* dlt) {
  for (int i = threadIdx.x; i < rows; i += kBwdThreads) {
    float l = INFINITY, dl = 0.f;
    if (i < nrows) {
      const int64_t o = b * a.l_bstride + static_cast<int64_t>(h) * a.S + tok0 + i;
      l = a.lse[o];
      l = l == -INFINITY ? INFINITY : l * kLog2e;
      dl = a.delta[o];
    }
    lse2[i] = l;
    dlt[i] = dl;
  }
}

__device__ __forceinline__ int shard_of(const int* prefix, int n, int item) {
  int r = 0;
  while (r + 1 < n && prefix[r + 1] <= item) ++r;
  return r;
}

// ----------------------------------------------------------------------------
// delta[b, h, s] = sum_d out[b, s, h, d] * dout[b, s, h, d]; one warp per row.
// ----------------------------------------------------------------------------
template <int D, typename T>
__global__ void __launch_bounds__(kBwdThreads) attn_bwd_delta_kernel(const float* __restrict__ out,
                                                                     const T* __restrict__ dout,
                                                                     float* __restrict__ delta, int B, int S, int H) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kBwdThreads / 32) + (threadIdx.x >> 5);
  if (row >= static_cast<int64_t>(B) * S * H) return;
  const int64_t h = row % H, bs = row / H, s = bs % S, b = bs / S;
  float acc = 0.f;
  for (int d = lane * 4; d < D; d += 128) {
    float o[4], g[4];
    load4(out + row * D + d, o);
    load4(dout + row * D + d, g);
#pragma unroll
    for (int c = 0; c < 4; ++c) acc = fmaf(o[c], g[c], acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) delta[(b * H + h) * S + s] = acc;
}

// ----------------------------------------------------------------------------
// dq. Thread t computes the 4 x 4 block (rows 4*(t/16), keys 4*(t%16)) of s
// and dp for each key tile, then 4 rows x D/16 columns of dq.
// ----------------------------------------------------------------------------
template <int D>
constexpr int dq_smem_floats() {
  return 4 * D * kTP + kBT * D + kBT * kTP + 2 * kBT;
}

template <int D, typename T>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_dq_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int CPT = D / 16;  // dq columns per thread
  extern __shared__ __align__(16) float sm[];
  float* Qt = sm;              // [D][kTP] q * scale * log2 e
  float* dOt = Qt + D * kTP;   // [D][kTP]
  float* Kt = dOt + D * kTP;   // [D][kTP]
  float* Vt = Kt + D * kTP;    // [D][kTP]
  float* Kr = Vt + D * kTP;    // [kBT][D]
  float* dSt = Kr + kBT * D;   // [kBT keys][kTP] ds, transposed
  float* lse2 = dSt + kBT * kTP;
  float* dlt = lse2 + kBT;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* dout = static_cast<const T*>(a.dout);
  const int tid = threadIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (bwd_head_is_padding(a, h, b)) return;
  const int r = shard_of(a.q_prefix, a.n, blockIdx.x);
  const int row0 = a.off[r] + (blockIdx.x - a.q_prefix[r]) * kBT;
  const int nrows = min(kBT, a.off[r] + a.len[r] - row0);
  load_tile<D>(q, a.bstride, a.sstride, b, h, row0, nrows, kBT, a.scale * kLog2e, Qt, kTP, nullptr);
  load_tile<D>(dout, a.bstride, a.sstride, b, h, row0, nrows, kBT, 1.f, dOt, kTP, nullptr);
  load_row_stats(a, b, h, row0, nrows, kBT, lse2, dlt);

  const int ti = tid / 16, tj = tid % 16;  // s / dp block
  const int ri = tid / 16, ci = tid % 16;  // dq block
  float acc[4][CPT];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < CPT; ++c) acc[i][c] = 0.f;

  for (int t = 0; t < a.n; ++t) {
    int j = (r - t) % a.n;
    if (j < 0) j += a.n;
    for (int k0 = a.off[j]; k0 < a.off[j] + a.len[j]; k0 += kBT) {
      const int nk = min(kBT, a.off[j] + a.len[j] - k0);
      __syncthreads();  // the previous tile's readers of Kt, Vt, Kr, dSt are done
      load_tile<D>(k, a.bstride, a.sstride, b, h, k0, nk, kBT, 1.f, Kt, kTP, Kr);
      load_tile<D>(v, a.bstride, a.sstride, b, h, k0, nk, kBT, 1.f, Vt, kTP, nullptr);
      __syncthreads();
      float s[4][4], dp[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[i][c] = dp[i][c] = 0.f;
#pragma unroll 4
      for (int d = 0; d < D; ++d) {
        const float4 qa = *reinterpret_cast<const float4*>(Qt + d * kTP + ti * 4);
        const float4 ka = *reinterpret_cast<const float4*>(Kt + d * kTP + tj * 4);
        const float4 ga = *reinterpret_cast<const float4*>(dOt + d * kTP + ti * 4);
        const float4 va = *reinterpret_cast<const float4*>(Vt + d * kTP + tj * 4);
        const float qv[4] = {qa.x, qa.y, qa.z, qa.w}, kv[4] = {ka.x, ka.y, ka.z, ka.w};
        const float gv[4] = {ga.x, ga.y, ga.z, ga.w}, vv[4] = {va.x, va.y, va.z, va.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            s[i][c] = fmaf(qv[i], kv[c], s[i][c]);
            dp[i][c] = fmaf(gv[i], vv[c], dp[i][c]);
          }
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float ds[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float p = tj * 4 + c < nk ? exp2f(s[i][c] - lse2[ti * 4 + i]) : 0.f;
          ds[i] = p * (dp[i][c] - dlt[ti * 4 + i]);
        }
        *reinterpret_cast<float4*>(dSt + (tj * 4 + c) * kTP + ti * 4) = make_float4(ds[0], ds[1], ds[2], ds[3]);
      }
      __syncthreads();
#pragma unroll 4
      for (int jj = 0; jj < kBT; ++jj) {
        const float4 sa = *reinterpret_cast<const float4*>(dSt + jj * kTP + ri * 4);
        const float sv[4] = {sa.x, sa.y, sa.z, sa.w};
        float kr[CPT];
#pragma unroll
        for (int c = 0; c < CPT; c += 4) {
          const float4 kk = *reinterpret_cast<const float4*>(Kr + jj * D + ci * CPT + c);
          kr[c] = kk.x;
          kr[c + 1] = kk.y;
          kr[c + 2] = kk.z;
          kr[c + 3] = kk.w;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c = 0; c < CPT; ++c) acc[i][c] = fmaf(sv[i], kr[c], acc[i][c]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = ri * 4 + i;
    if (row >= nrows) continue;
    float* dst = a.dq + b * a.bstride + static_cast<int64_t>(row0 + row) * a.sstride + h * D + ci * CPT;
#pragma unroll
    for (int c = 0; c < CPT; c += 4)
      *reinterpret_cast<float4*>(dst + c) =
          make_float4(acc[i][c] * a.scale, acc[i][c + 1] * a.scale, acc[i][c + 2] * a.scale, acc[i][c + 3] * a.scale);
  }
}

// ----------------------------------------------------------------------------
// dk / dv. Thread t computes the 2 x 4 block (rows 2*(t/16), keys 4*(t%16))
// of s and dp for each query tile, then 4 keys x D/16 columns of dk and dv.
// ----------------------------------------------------------------------------
template <int D>
constexpr int dkdv_smem_floats() {
  return 2 * D * kTP + 2 * D * kTQ + 2 * kBQ * D + 2 * kBQ * kTP + 2 * kBQ;
}

template <int D, typename T>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_dkdv_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int CPT = D / 16;
  extern __shared__ __align__(16) float sm[];
  float* Kt = sm;              // [D][kTP]
  float* Vt = Kt + D * kTP;    // [D][kTP]
  float* Qt = Vt + D * kTP;    // [D][kTQ] q * scale * log2 e
  float* dOt = Qt + D * kTQ;   // [D][kTQ]
  float* Qr = dOt + D * kTQ;   // [kBQ][D]
  float* dOr = Qr + kBQ * D;   // [kBQ][D]
  float* Pb = dOr + kBQ * D;   // [kBQ][kTP]
  float* dSb = Pb + kBQ * kTP; // [kBQ][kTP]
  float* lse2 = dSb + kBQ * kTP;
  float* dlt = lse2 + kBQ;
  const T* q = static_cast<const T*>(a.q);
  const T* k = static_cast<const T*>(a.k);
  const T* v = static_cast<const T*>(a.v);
  const T* dout = static_cast<const T*>(a.dout);
  const int tid = threadIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (bwd_head_is_padding(a, h, b)) return;
  const int jb = shard_of(a.kv_prefix, a.n, blockIdx.x);
  const int key0 = a.off[jb] + (blockIdx.x - a.kv_prefix[jb]) * kBT;
  const int nk = min(kBT, a.off[jb] + a.len[jb] - key0);
  load_tile<D>(k, a.bstride, a.sstride, b, h, key0, nk, kBT, 1.f, Kt, kTP, nullptr);
  load_tile<D>(v, a.bstride, a.sstride, b, h, key0, nk, kBT, 1.f, Vt, kTP, nullptr);

  const int ti = tid / 16, tj = tid % 16;  // s / dp block: rows 2*ti, keys 4*tj
  const int kj = tid / 16, ci = tid % 16;  // dk / dv block: keys 4*kj, columns CPT*ci
  float dk[4][CPT], dv[4][CPT];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < CPT; ++c) dk[i][c] = dv[i][c] = 0.f;

  for (int t = 0; t < a.n; ++t) {
    const int r = (jb + t) % a.n;  // the rank this block visits at step t
    for (int q0 = a.off[r]; q0 < a.off[r] + a.len[r]; q0 += kBQ) {
      const int nq = min(kBQ, a.off[r] + a.len[r] - q0);
      __syncthreads();  // the previous tile's readers are done
      load_tile<D>(q, a.bstride, a.sstride, b, h, q0, nq, kBQ, a.scale * kLog2e, Qt, kTQ, nullptr);
      load_tile<D>(q, a.bstride, a.sstride, b, h, q0, nq, kBQ, 1.f, nullptr, 0, Qr);
      load_tile<D>(dout, a.bstride, a.sstride, b, h, q0, nq, kBQ, 1.f, dOt, kTQ, dOr);
      load_row_stats(a, b, h, q0, nq, kBQ, lse2, dlt);
      __syncthreads();
      float s[2][4], dp[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[i][c] = dp[i][c] = 0.f;
#pragma unroll 4
      for (int d = 0; d < D; ++d) {
        const float2 qa = *reinterpret_cast<const float2*>(Qt + d * kTQ + ti * 2);
        const float2 ga = *reinterpret_cast<const float2*>(dOt + d * kTQ + ti * 2);
        const float4 ka = *reinterpret_cast<const float4*>(Kt + d * kTP + tj * 4);
        const float4 va = *reinterpret_cast<const float4*>(Vt + d * kTP + tj * 4);
        const float qv[2] = {qa.x, qa.y}, gv[2] = {ga.x, ga.y};
        const float kv[4] = {ka.x, ka.y, ka.z, ka.w}, vv[4] = {va.x, va.y, va.z, va.w};
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            s[i][c] = fmaf(qv[i], kv[c], s[i][c]);
            dp[i][c] = fmaf(gv[i], vv[c], dp[i][c]);
          }
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int row = ti * 2 + i;
        float p[4], ds[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          p[c] = tj * 4 + c < nk ? exp2f(s[i][c] - lse2[row]) : 0.f;
          ds[c] = p[c] * (dp[i][c] - dlt[row]);
        }
        *reinterpret_cast<float4*>(Pb + row * kTP + tj * 4) = make_float4(p[0], p[1], p[2], p[3]);
        *reinterpret_cast<float4*>(dSb + row * kTP + tj * 4) = make_float4(ds[0], ds[1], ds[2], ds[3]);
      }
      __syncthreads();
#pragma unroll 2
      for (int i = 0; i < kBQ; ++i) {
        const float4 pa = *reinterpret_cast<const float4*>(Pb + i * kTP + kj * 4);
        const float4 sa = *reinterpret_cast<const float4*>(dSb + i * kTP + kj * 4);
        const float pv[4] = {pa.x, pa.y, pa.z, pa.w}, sv[4] = {sa.x, sa.y, sa.z, sa.w};
        float g[CPT], x[CPT];
#pragma unroll
        for (int c = 0; c < CPT; c += 4) {
          const float4 gg = *reinterpret_cast<const float4*>(dOr + i * D + ci * CPT + c);
          const float4 qq = *reinterpret_cast<const float4*>(Qr + i * D + ci * CPT + c);
          g[c] = gg.x;
          g[c + 1] = gg.y;
          g[c + 2] = gg.z;
          g[c + 3] = gg.w;
          x[c] = qq.x;
          x[c + 1] = qq.y;
          x[c + 2] = qq.z;
          x[c + 3] = qq.w;
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
          for (int c = 0; c < CPT; ++c) {
            dv[jj][c] = fmaf(pv[jj], g[c], dv[jj][c]);
            dk[jj][c] = fmaf(sv[jj], x[c], dk[jj][c]);
          }
      }
    }
  }
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const int key = kj * 4 + jj;
    if (key >= nk) continue;
    const int64_t o = b * a.bstride + static_cast<int64_t>(key0 + key) * a.sstride + h * D + ci * CPT;
#pragma unroll
    for (int c = 0; c < CPT; c += 4) {
      *reinterpret_cast<float4*>(a.dk + o + c) = make_float4(dk[jj][c] * a.scale, dk[jj][c + 1] * a.scale,
                                                             dk[jj][c + 2] * a.scale, dk[jj][c + 3] * a.scale);
      *reinterpret_cast<float4*>(a.dv + o + c) = make_float4(dv[jj][c], dv[jj][c + 1], dv[jj][c + 2], dv[jj][c + 3]);
    }
  }
}

template <int D, typename T>
cudaError_t launch_bwd_d(const BwdArgs& a, cudaStream_t s) {
  constexpr int dq_bytes = dq_smem_floats<D>() * 4, kv_bytes = dkdv_smem_floats<D>() * 4;
  static_assert(dq_bytes <= 227 * 1024 && kv_bytes <= 227 * 1024, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       dq_bytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, kv_bytes);
  if (e != cudaSuccess) return e;
  if (a.q_prefix[a.n] > 0) {
    attn_bwd_dq_kernel<D, T><<<dim3(a.q_prefix[a.n], a.H, a.B), kBwdThreads, dq_bytes, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (a.kv_prefix[a.n] > 0) {
    attn_bwd_dkdv_kernel<D, T><<<dim3(a.kv_prefix[a.n], a.H, a.B), kBwdThreads, kv_bytes, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int D, typename T>
cudaError_t launch_delta_d(const float* out, const void* dout, float* delta, int B, int S, int H, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(B) * S * H;
  const int64_t blocks = (rows + kBwdThreads / 32 - 1) / (kBwdThreads / 32);
  attn_bwd_delta_kernel<D, T><<<static_cast<unsigned>(blocks), kBwdThreads, 0, s>>>(
      out, static_cast<const T*>(dout), delta, B, S, H);
  return cudaGetLastError();
}

// lse * log2 e and delta of every shard's rows into the padded per-shard
// layout of BwdArgs::lse2p / dltp: element (bh, r, i) for i < lpad.
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const __grid_constant__ BwdArgs a) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  const int64_t per_bh = static_cast<int64_t>(a.n) * a.lpad;
  if (idx >= static_cast<int64_t>(a.B) * a.H * per_bh) return;
  const int64_t bh = idx / per_bh;
  const int rem = static_cast<int>(idx - bh * per_bh);
  const int r = rem / a.lpad, i = rem - r * a.lpad;
  float l2 = INFINITY, dl = 0.f;  // padding: p = 0
  if (i < a.len[r]) {
    const int64_t b = bh / a.H, h = bh - b * a.H;
    const int64_t o = b * a.l_bstride + h * a.S + a.off[r] + i;
    const float l = a.lse[o];
    l2 = l == -INFINITY ? INFINITY : l * 1.4426950408889634f;  // a row that saw no key: p = 0
    dl = a.delta[o];
  }
  a.lse2p[idx] = l2;
  a.dltp[idx] = dl;
}

}  // namespace

cudaError_t launch_attn_bwd_prep(const BwdArgs& a, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(a.B) * a.H * a.n * a.lpad;
  if (n == 0) return cudaSuccess;
  attn_bwd_prep_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const BwdArgs& a, int D, bool bf16, cudaStream_t s) {
  if (D == 128) return bf16 ? launch_bwd_d<128, __nv_bfloat16>(a, s) : launch_bwd_d<128, float>(a, s);
  if (D == 64) return bf16 ? launch_bwd_d<64, __nv_bfloat16>(a, s) : launch_bwd_d<64, float>(a, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_bwd_delta(const float* out, const void* dout, float* delta, int B, int S, int H, int D,
                                  bool bf16, cudaStream_t s) {
  if (static_cast<int64_t>(B) * S * H == 0) return cudaSuccess;
  if (D == 128)
    return bf16 ? launch_delta_d<128, __nv_bfloat16>(out, dout, delta, B, S, H, s)
                : launch_delta_d<128, float>(out, dout, delta, B, S, H, s);
  if (D == 64)
    return bf16 ? launch_delta_d<64, __nv_bfloat16>(out, dout, delta, B, S, H, s)
                : launch_delta_d<64, float>(out, dout, delta, B, S, H, s);
  return cudaErrorInvalidValue;
}

}  // namespace cp
