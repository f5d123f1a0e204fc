// cp_internal.h — launch parameters shared by the kernels and the host driver
// of libcpattn.so. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace cp {

constexpr int kMaxRanks = 16;       // largest ring degree the launch tables hold
constexpr int kTileM = 128;         // query rows per tensor-core tile
constexpr int kTileN = 128;         // keys per K/V tile

// Ring geometry of one launch: the query shards (one per simulated rank) and
// the K/V blocks they visit. Rank r at ring step t attends to block
// (r - t) mod n_kv: its own block first, then the one "received" from its
// predecessor. step >= 0 restricts a launch to that single step; step < 0
// runs the whole lap inside the launch.
struct RingGeom {
  int n_q;
  int q_off[kMaxRanks];
  int q_len[kMaxRanks];
  int cta_prefix[kMaxRanks + 1];   // CUDA-core kernel: 8-row work items per shard, prefix sums
  int pair_prefix[kMaxRanks + 1];  // tensor-core kernel: items with two 128-row Q tiles, prefix sums
  int single_prefix[kMaxRanks + 1];  // tensor-core kernel: items with one Q tile (odd tile count)
  int n_kv;
  int kv_off[kMaxRanks];
  int kv_len[kMaxRanks];
  int step;
};

struct AttnArgs {
  RingGeom g;
  int B;   // batch entries (Ulysses head groups folded in)
  int H;   // heads per batch entry
  int D;   // head dim
  float scale;       // softmax scale applied to q.k
  float scale_log2;  // scale * log2(e)
  // outputs: out[b*o_bstride + s*o_sstride + h*D + d], lse[b*l_bstride + h*l_hstride + s]
  float* out;
  int64_t o_bstride, o_sstride;
  float* lse;
  int64_t l_bstride, l_hstride;
  // raw inputs (element strides) for the CUDA-core fp32 path
  const float* qf;
  const float* kf;
  const float* vf;
  int64_t q_bstride, q_sstride, kv_bstride, kv_sstride;
  // device error word and the bound on each device-side wait
  uint32_t* err;
  uint64_t timeout_ns;
  // ragged head groups (Ulysses Anything): batch entries come in groups of
  // hv_bpg, and groups from hv_short_from on have H - 1 real heads (head H - 1
  // is padding and is skipped). hv_bpg = 1, hv_short_from = INT_MAX: none.
  int hv_bpg;
  int hv_short_from;
  // key-padding mask (nullptr: none): key j of batch entry b takes part iff
  // kmask[(b % km_bmod) * km_bstride + j] != 0 (j indexes the K/V tokens)
  const uint8_t* kmask;
  int64_t km_bstride;
  int km_bmod;
};

// Whether (head h, batch entry b) is padding of a ragged head group.
__host__ __device__ inline bool attn_head_is_padding(const AttnArgs& a, int h, int b) {
  return h == a.H - 1 && b / a.hv_bpg >= a.hv_short_from;
}

// Tensor-core work items of a shard of `rows` query rows: tile pairs, plus one
// single tile when the tile count is odd. All pairs of all shards are launched
// before all singles, so the short items fill the last wave.
inline int tc_tiles_for_rows(int rows) { return (rows + kTileM - 1) / kTileM; }
inline int tc_pairs_for_rows(int rows) { return tc_tiles_for_rows(rows) / 2; }
inline int tc_singles_for_rows(int rows) { return tc_tiles_for_rows(rows) % 2; }
// Work items per shard for the CUDA-core kernel: 8 query rows per CTA.
constexpr int kF32RowsPerCta = 8;
inline int f32_items_for_rows(int rows) { return (rows + kF32RowsPerCta - 1) / kF32RowsPerCta; }

// Backward of a ring lap over n even shards of one sequence (query shards and
// K/V blocks share the table; n = 1 for Ulysses and Ulysses Anything). q, k, v, dout and the outputs dq, dk, dv are
// [B, S, H, D] with element strides (bstride, sstride, 1 per head of D);
// lse and delta are [B, H, S] with batch stride l_bstride.
constexpr int kBwdTile = 64;  // CUDA-core backward: query rows per dq CTA, keys per dk/dv CTA
struct BwdArgs {
  int n;
  int off[kMaxRanks];
  int len[kMaxRanks];
  int q_prefix[kMaxRanks + 1];   // dq CTAs per shard, prefix sums
  int kv_prefix[kMaxRanks + 1];  // dk/dv CTAs per block, prefix sums
  int B, H, S;
  float scale;
  const void* q;
  const void* k;
  const void* v;
  const void* dout;
  int64_t bstride, sstride;
  const float* lse;
  const float* delta;
  int64_t l_bstride;
  float* dq;
  float* dk;
  float* dv;
  // tensor-core kernels: device error word and the bound on each device-side wait
  uint32_t* err;
  uint64_t timeout_ns;
  // ragged head groups (Ulysses Anything), as in AttnArgs: batch entries come
  // in groups of hv_bpg, and groups from hv_short_from on have H - 1 real
  // heads; head H - 1 of those is padding that no kernel touches.
  // hv_bpg = 0: no padding.
  int hv_bpg;
  int hv_short_from;
  // tensor-core dk/dv kernel: per (batch entry, head, shard) the shard's rows'
  // lse * log2 e (+inf where lse = -inf) and delta, each shard padded to lpad
  // rows (a multiple of 64, the padding holding +inf and 0), so that every
  // 64-row piece starts 256-byte aligned for a bulk copy
  float* lse2p;
  float* dltp;
  int lpad;
};

__host__ __device__ inline bool bwd_head_is_padding(const BwdArgs& a, int h, int b) {
  return a.hv_bpg > 0 && h == a.H - 1 && b / a.hv_bpg >= a.hv_short_from;
}
constexpr int kBwdTcTile = 128;  // tensor-core backward: keys (dk/dv) or query rows (dq) per CTA

// Launchers (each returns the launch error, cudaSuccess if none).
// dq, then dk/dv, for D in {64, 128}; bf16 or fp32 inputs.
cudaError_t launch_attn_bwd(const BwdArgs& a, int D, bool bf16, cudaStream_t s);
// Fills a.lse2p and a.dltp (see BwdArgs) from a.lse and a.delta.
cudaError_t launch_attn_bwd_prep(const BwdArgs& a, cudaStream_t s);
// delta[b, h, s] = sum_d out[b, s, h, d] * dout[b, s, h, d] over dense [B, S, H, D].
cudaError_t launch_attn_bwd_delta(const float* out, const void* dout, float* delta, int B, int S, int H, int D,
                                  bool bf16, cudaStream_t s);
// Tensor maps of the tensor-core backward over bf16 q, k, v, dout (128-byte
// swizzle, boxes of 64 columns of one head): boxes of 128 rows for the tiles a
// CTA keeps (K, V in dk/dv; Q, dO in dq) and of 64 rows for the sub-tiles it
// streams (Q, dO in dk/dv; K, V in dq).
struct BwdTensorMaps {
  CUtensorMap q, k, v, o;          // 128-row boxes
  CUtensorMap q64, k64, v64, o64;  // 64-row boxes
};
// Tensor-core backward for bf16: the dk/dv kernel (one CTA per 128 keys,
// kv_prefix) and the dq kernel (one CTA per 128 query rows, q_prefix); dq,
// dk, dv written.
cudaError_t launch_attn_bwd_tc(const BwdArgs& a, int D, const BwdTensorMaps& m, cudaStream_t s);
cudaError_t launch_attn_tc(const AttnArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, cudaStream_t s);
cudaError_t launch_attn_f32(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_lse_merge(float* out_acc, float* lse_acc, const float* out_blk, const float* lse_blk,
                             int B, int H, int S, int D, cudaStream_t s);

// Copy of n0*n1*n2*n3 segments of seg_elems elements each: the input segment
// (i0, i1, i2, i3) starts at element i0*st0 + i1*st1 + i2*st2 + i3*st3. The
// output segment starts at i0*ost0 + i1*ost1 + i2*ost2 + i3*ost3, or, when
// every ost is 0, output segments are contiguous in (i0, i1, i2, i3) order.
struct SegCopy {
  const void* in;
  void* out;
  int64_t n0, n1, n2, n3;
  int64_t st0, st1, st2, st3;
  int64_t seg_elems;
  int elem_bytes;
  int64_t ost0, ost1, ost2, ost3;
};
// One copy: the bulk path when it qualifies (see launch_segment_copies), else
// the widest vector (16, 8, 4 or 1 bytes) that every segment start, the
// segment length and both base pointers allow.
cudaError_t launch_segment_copy(const SegCopy& c, cudaStream_t s);
// n independent copies (no copy reads what another writes; a launch runs its
// copies concurrently): the ones that take the bulk path (16-byte aligned,
// segments of 256 B to 24 KB) share launches, up to 24 per launch; every
// other copy takes a vector launch of its own.
cudaError_t launch_segment_copies(const SegCopy* cs, int n, cudaStream_t s);
// The number of launches launch_segment_copies makes for the same copies
// (pointers need only carry their alignment).
int segment_copy_launches(const SegCopy* cs, int n);

// Device error word of the tensor-core kernel's translation unit.
uint32_t* device_error_word();  // device address on the current device, or nullptr
cudaError_t launch_wait_probe(uint32_t* err, uint64_t timeout_ns, cudaStream_t s);

}  // namespace cp
