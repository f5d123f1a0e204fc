// cp_api.cu — the C ABI of libcpattn.so (declared in include/cp_attn.h):
// argument validation, the ring shard table, tensor-map set-up, and the host
// driver that sequences the regroup, block-attention and merge launches of a
// simulated context-parallel attention forward on one GPU.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "cp_attn.h"
#include "cp_internal.h"

namespace {

using cp::AttnArgs;
using cp::RingGeom;
using cp::SegCopy;

constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // 1 s per device-side wait
constexpr int kMaxDevices = 64;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------------------
// device checks and per-device cached lookups
// ---------------------------------------------------------------------------
struct DeviceInfo {
  int checked = 0;  // 0 unknown, 1 sm_103, -1 other
  uint32_t* err = nullptr;
  int sms = 0;  // multiprocessors
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

cp_status current_device(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CP_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.checked == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return CP_ERR_CUDA;
    d.checked = (major == 10 && minor == 3) ? 1 : -1;
    if (d.checked == 1 && cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      d.checked = 0;
      return CP_ERR_CUDA;
    }
    if (d.checked == 1) {
      d.err = cp::device_error_word();
      if (!d.err) {
        d.checked = 0;
        return CP_ERR_CUDA;
      }
    }
  }
  if (d.checked != 1) return CP_ERR_UNSUPPORTED_DEVICE;
  *out = &d;
  return CP_OK;
}

// ---------------------------------------------------------------------------
// TMA tensor maps (driver entry point fetched through the runtime, so the
// library links no libcuda and loads on machines without a GPU driver)
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// bf16 [Bn, S, H, D] with token stride row and batch stride bstride elements
// (row = H*D for a dense tensor; larger for a range of its heads); box = 64
// columns x 128 tokens of one head, 128-byte swizzle (the K-major operand
// layout the MMA descriptors expect).
bool make_tmap_bf16(CUtensorMap* m, const void* base, int D, int H, int S, int Bn, int64_t row, int64_t bstride,
                    int box_rows = cp::kTileM) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(Bn)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(row) * 2,
                           static_cast<cuuint64_t>(bstride) * 2};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// shard table: balanced split (first S mod n shards one token longer)
// ---------------------------------------------------------------------------
cp_status shard_table(int S, int n, bool uneven_ok, int* off, int* len) {
  if (n < 1 || S < 0) return CP_ERR_INVALID_ARG;
  const int base = S / n, extra = S % n;
  if (extra && !uneven_ok) return CP_ERR_NOT_DIVISIBLE;
  int o = 0;
  for (int r = 0; r < n; ++r) {
    off[r] = o;
    len[r] = base + (r < extra ? 1 : 0);
    o += len[r];
  }
  return CP_OK;
}

void fill_geom(RingGeom* g, cp_dtype dt, int nq, const int* qoff, const int* qlen, int nkv, const int* kvoff,
               const int* kvlen, int step) {
  std::memset(g, 0, sizeof(*g));
  (void)dt;
  g->n_q = nq;
  for (int r = 0; r < nq; ++r) {
    g->q_off[r] = qoff[r];
    g->q_len[r] = qlen[r];
    g->cta_prefix[r + 1] = g->cta_prefix[r] + cp::f32_items_for_rows(qlen[r]);
    g->pair_prefix[r + 1] = g->pair_prefix[r] + cp::tc_pairs_for_rows(qlen[r]);
    g->single_prefix[r + 1] = g->single_prefix[r] + cp::tc_singles_for_rows(qlen[r]);
  }
  g->n_kv = nkv;
  for (int j = 0; j < nkv; ++j) {
    g->kv_off[j] = kvoff[j];
    g->kv_len[j] = kvlen[j];
  }
  g->step = step;
}

// One attention launch over tensors q [Bn, Sq, H, D], k/v [Bn, Skv, H, D].
struct AttnTensors {
  const void* q;
  const void* k;
  const void* v;
  int Bn, H, D, Sq, Skv;
  int64_t q_bstride, kv_bstride;
  float* out;
  int64_t o_bstride;
  float* lse;  // [Bn, H, Sq], head stride Sq
  int hv_bpg = 1;                  // ragged head groups: batch entries per group
  int hv_short_from = INT_MAX;     // first group whose last head is padding
  int64_t row = 0;                 // token stride of q, k, v and out in elements (0: H*D)
  int64_t l_bstride = 0;           // batch stride of lse in elements (0: H*Sq)
  const uint8_t* kmask = nullptr;  // key-padding mask [km_bmod, km_bstride] (nullptr: none)
  int64_t km_bstride = 0;
  int km_bmod = 1;
};

cp_status launch_attention(const AttnTensors& t, const RingGeom& g, float scale, cp_dtype dt, DeviceInfo* dev,
                           cudaStream_t s) {
  AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  a.g = g;
  a.B = t.Bn;
  a.H = t.H;
  a.D = t.D;
  a.scale = scale;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.out = t.out;
  a.o_bstride = t.o_bstride;
  const int64_t row = t.row ? t.row : static_cast<int64_t>(t.H) * t.D;
  a.o_sstride = row;
  a.lse = t.lse;
  a.l_bstride = t.l_bstride ? t.l_bstride : static_cast<int64_t>(t.H) * t.Sq;
  a.l_hstride = t.Sq;
  a.err = dev->err;
  a.timeout_ns = kWaitTimeoutNs;
  a.hv_bpg = t.hv_bpg;
  a.hv_short_from = t.hv_short_from;
  a.kmask = t.kmask;
  a.km_bstride = t.km_bstride;
  a.km_bmod = t.km_bmod > 0 ? t.km_bmod : 1;
  cudaError_t e;
  if (dt == CP_BF16) {
    CUtensorMap tq, tk, tv;
    if (!make_tmap_bf16(&tq, t.q, t.D, t.H, t.Sq, t.Bn, row, t.q_bstride)) return CP_ERR_CUDA;
    const bool kv_empty = t.Skv == 0;
    if (!make_tmap_bf16(&tk, kv_empty ? t.q : t.k, t.D, t.H, kv_empty ? t.Sq : t.Skv, t.Bn, row,
                        kv_empty ? t.q_bstride : t.kv_bstride))
      return CP_ERR_CUDA;
    if (!make_tmap_bf16(&tv, kv_empty ? t.q : t.v, t.D, t.H, kv_empty ? t.Sq : t.Skv, t.Bn, row,
                        kv_empty ? t.q_bstride : t.kv_bstride))
      return CP_ERR_CUDA;
    e = cp::launch_attn_tc(a, tq, tk, tv, s);
  } else {
    a.qf = static_cast<const float*>(t.q);
    a.kf = static_cast<const float*>(t.k);
    a.vf = static_cast<const float*>(t.v);
    a.q_bstride = t.q_bstride;
    a.q_sstride = row;
    a.kv_bstride = t.kv_bstride;
    a.kv_sstride = row;
    e = cp::launch_attn_f32(a, s);
  }
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

int elem_size(cp_dtype dt) { return dt == CP_BF16 ? 2 : 4; }

cp_status check_common(int B, int H, int S, int D, cp_dtype dt) {
  if (B < 0 || H < 1 || S < 0) return CP_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return CP_ERR_INVALID_ARG;
  if (dt != CP_BF16 && dt != CP_F32) return CP_ERR_INVALID_ARG;
  return CP_OK;
}

// Workspace layout of cp_attention_fwd (every piece 256-byte aligned):
// [q_h | k_h | v_h] (Ulysses regroups of the inputs), [out_h | lse_h] (the
// head-sharded result), [out_p | lse_p] (one ring step's partial).
struct WsLayout {
  size_t qh = 0, kh = 0, vh = 0, oh = 0, lh = 0, op = 0, lp = 0, total = 0;
};

WsLayout ws_layout(int B, int H, int S, int D, int R, int U, cp_dtype dt, cp_lap_mode mode) {
  WsLayout w;
  // U head groups of ceil(H/U) heads (the last heads of short groups are padding)
  const size_t Hp = U > 1 ? static_cast<size_t>((H + U - 1) / U) * U : static_cast<size_t>(H);
  const size_t n = static_cast<size_t>(B) * S * Hp * D;
  const size_t nl = static_cast<size_t>(B) * Hp * S;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = round_up(o + bytes, 256);
    return at;
  };
  if (U > 1) {
    w.qh = take(n * elem_size(dt));
    w.kh = take(n * elem_size(dt));
    w.vh = take(n * elem_size(dt));
    w.oh = take(n * 4);
    w.lh = take(nl * 4);
  }
  if (mode == CP_LAP_STEPWISE && R > 1) {
    w.op = take(n * 4);
    w.lp = take(nl * 4);
  }
  w.total = o;
  return w;
}

}  // namespace

extern "C" {

const char* cp_status_string(cp_status s) {
  switch (s) {
    case CP_OK: return "ok";
    case CP_ERR_INVALID_ARG: return "invalid argument";
    case CP_ERR_NOT_DIVISIBLE: return "sequence length or head count not divisible by the parallel degree";
    case CP_ERR_UNSUPPORTED_COMBO: return "unsupported combination of parallel degrees and flags";
    case CP_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
    case CP_ERR_CUDA: return "CUDA error";
    case CP_ERR_TIMEOUT: return "device-side wait timed out";
    case CP_ERR_WORKSPACE: return "workspace missing or too small";
    case CP_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103 (GB300)";
  }
  return "unknown status";
}

int cp_version(void) { return 10000; }

cp_status cp_block_attn_fwd(const void* q, const void* k, const void* v, float* out, float* lse, int B, int H, int Sq,
                            int Skv, int D, float scale, int64_t q_bstride, int64_t kv_bstride, int64_t o_bstride,
                            cp_dtype dt, void* stream) {
  cp_status st = check_common(B, H, Sq, D, dt);
  if (st != CP_OK) return st;
  if (Skv < 0 || !std::isfinite(scale)) return CP_ERR_INVALID_ARG;
  const int64_t row = static_cast<int64_t>(H) * D;
  if (q_bstride == 0) q_bstride = Sq * row;
  if (kv_bstride == 0) kv_bstride = Skv * row;
  if (o_bstride == 0) o_bstride = Sq * row;
  if (q_bstride < Sq * row || kv_bstride < Skv * row || o_bstride < Sq * row) return CP_ERR_INVALID_ARG;
  if (B == 0 || Sq == 0) return CP_OK;
  if (!q || !out || !lse || (Skv > 0 && (!k || !v))) return CP_ERR_INVALID_ARG;
  const int eb = elem_size(dt);
  if (!aligned16(q) || !aligned16(out) || !aligned16(lse) || (Skv > 0 && (!aligned16(k) || !aligned16(v))) ||
      (q_bstride * eb) % 16 || (kv_bstride * eb) % 16 || (o_bstride * 4) % 16)
    return CP_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev)) != CP_OK) return st;
  const int zero = 0;
  RingGeom g;
  fill_geom(&g, dt, 1, &zero, &Sq, 1, &zero, &Skv, 0);
  AttnTensors t{q, k, v, B, H, D, Sq, Skv, q_bstride, kv_bstride, out, o_bstride, lse};
  return launch_attention(t, g, scale, dt, dev, static_cast<cudaStream_t>(stream));
}

cp_status cp_lse_merge(float* out_acc, float* lse_acc, const float* out_blk, const float* lse_blk, int B, int H, int S,
                       int D, void* stream) {
  if (B < 0 || H < 1 || S < 0 || D < 4 || D % 4) return CP_ERR_INVALID_ARG;
  if (B == 0 || S == 0) return CP_OK;
  if (!out_acc || !lse_acc || !out_blk || !lse_blk) return CP_ERR_INVALID_ARG;
  if (!aligned16(out_acc) || !aligned16(out_blk) || (reinterpret_cast<uintptr_t>(lse_acc) & 3) ||
      (reinterpret_cast<uintptr_t>(lse_blk) & 3))
    return CP_ERR_ALIGNMENT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CP_ERR_CUDA;
  return cp::launch_lse_merge(out_acc, lse_acc, out_blk, lse_blk, B, H, S, D, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? CP_OK
             : CP_ERR_CUDA;
}

static cp_status check_permute(const void* in, const void* out, int U, int B, int S, int H, int D, int eb) {
  if (U < 1 || B < 0 || S < 0 || H < 1 || D < 1 || (eb != 1 && eb != 2 && eb != 4 && eb != 8))
    return CP_ERR_INVALID_ARG;
  if (U > H || H % U || S % U) return CP_ERR_INVALID_ARG;
  if (B > 0 && S > 0 && (!in || !out)) return CP_ERR_INVALID_ARG;
  return CP_OK;
}

cp_status cp_ulysses_seq2head(const void* in, void* out, int U, int B, int S, int H, int D, int elem_bytes,
                              void* stream) {
  cp_status st = check_permute(in, out, U, B, S, H, D, elem_bytes);
  if (st != CP_OK) return st;
  if (B == 0 || S == 0) return CP_OK;
  const int64_t Sl = S / U, Hg = H / U;
  // out segments (g, b, u, s) of Hg*D elements <- in[u][b, s, g*Hg : (g+1)*Hg, :]
  SegCopy c{in, out, U, B, U, Sl, Hg * D, Sl * H * D, static_cast<int64_t>(B) * Sl * H * D, H * D,
            Hg * D, elem_bytes};
  return cp::launch_segment_copy(c, static_cast<cudaStream_t>(stream)) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

cp_status cp_ulysses_head2seq(const void* in, void* out, int U, int B, int S, int H, int D, int elem_bytes,
                              void* stream) {
  cp_status st = check_permute(in, out, U, B, S, H, D, elem_bytes);
  if (st != CP_OK) return st;
  if (B == 0 || S == 0) return CP_OK;
  const int64_t Sl = S / U, Hg = H / U;
  // out segments (u, b, s, g) of Hg*D elements <- in[g][b, u*Sl + s, :, :]
  SegCopy c{in, out, U, B, Sl, U, Sl * Hg * D, static_cast<int64_t>(S) * Hg * D, Hg * D,
            static_cast<int64_t>(B) * S * Hg * D, Hg * D, elem_bytes};
  return cp::launch_segment_copy(c, static_cast<cudaStream_t>(stream)) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

// Ulysses Anything regroups over ragged rank blocks and head groups (balanced
// splits of S and H into U). Rank u's block [B, S_u, H, D] starts at element
// B*soff_u*H*D; group g's block [B, S, H_g, D] at element B*S*hoff_g*D.
static cp_status check_anything(const void* in, const void* out, int U, int B, int S, int H, int D, int eb) {
  if (U < 1 || B < 0 || S < 0 || H < 1 || D < 1 || U > H || (eb != 1 && eb != 2 && eb != 4 && eb != 8))
    return CP_ERR_INVALID_ARG;
  if (B > 0 && S > 0 && (!in || !out)) return CP_ERR_INVALID_ARG;
  return CP_OK;
}

static cp_status anything_regroup(const void* in, void* out, int U, int B, int S, int H, int D, int eb,
                                  bool to_heads, void* stream) {
  cp_status st = check_anything(in, out, U, B, S, H, D, eb);
  if (st != CP_OK) return st;
  if (B == 0 || S == 0) return CP_OK;
  std::vector<int> so(U), sl(U), ho(U), hl(U);
  if (shard_table(S, U, true, so.data(), sl.data()) != CP_OK || shard_table(H, U, true, ho.data(), hl.data()) != CP_OK)
    return CP_ERR_INVALID_ARG;
  const char* src = static_cast<const char*>(in);
  char* dst = static_cast<char*>(out);
  const int64_t HD = static_cast<int64_t>(H) * D;
  std::vector<SegCopy> cs;
  for (int g = 0; g < U; ++g) {
    const int64_t gD = static_cast<int64_t>(hl[g]) * D;       // elements of a group row
    const int64_t gbase = static_cast<int64_t>(B) * S * ho[g] * D;
    for (int u = 0; u < U; ++u) {
      if (sl[u] == 0) continue;
      const int64_t rbase = static_cast<int64_t>(B) * so[u] * HD;
      // rank side: rows (b, s) of pitch H*D, batch stride S_u*H*D, head offset hoff_g
      const int64_t r_el = rbase + static_cast<int64_t>(ho[g]) * D, r_b = sl[u] * HD;
      // group side: rows (b, soff_u + s) of pitch H_g*D, batch stride S*H_g*D
      const int64_t g_el = gbase + static_cast<int64_t>(so[u]) * gD, g_b = S * gD;
      cs.push_back(to_heads ? SegCopy{src + r_el * eb, dst + g_el * eb, 1, 1, B, sl[u], 0, 0, r_b, HD, gD, eb,
                                      0, 0, g_b, gD}
                            : SegCopy{src + g_el * eb, dst + r_el * eb, 1, 1, B, sl[u], 0, 0, g_b, gD, gD, eb,
                                      0, 0, r_b, HD});
    }
  }
  // the U * U copies write disjoint ranges: they share launches
  return cp::launch_segment_copies(cs.data(), static_cast<int>(cs.size()), static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? CP_OK
             : CP_ERR_CUDA;
}

cp_status cp_ulysses_anything_seq2head(const void* in, void* out, int U, int B, int S, int H, int D, int elem_bytes,
                                       void* stream) {
  return anything_regroup(in, out, U, B, S, H, D, elem_bytes, true, stream);
}

cp_status cp_ulysses_anything_head2seq(const void* in, void* out, int U, int B, int S, int H, int D, int elem_bytes,
                                       void* stream) {
  return anything_regroup(in, out, U, B, S, H, D, elem_bytes, false, stream);
}

cp_status cp_attention_validate(int B, int H, int S, int D, int ring_degree, int ulysses_degree, int uneven_ok,
                                cp_dtype dt) {
  cp_status st = check_common(B, H, S, D, dt);
  if (st != CP_OK) return st;
  const int R = ring_degree, U = ulysses_degree;
  if (R < 1 || U < 1 || R > cp::kMaxRanks) return CP_ERR_INVALID_ARG;
  // an Anything variant: Ring Anything (R > 1, U == 1) or Ulysses Anything (U > 1, R == 1)
  if (uneven_ok && (R > 1) == (U > 1)) return CP_ERR_UNSUPPORTED_COMBO;
  if (U > H) return CP_ERR_INVALID_ARG;
  if (U == 1) return (S % R && !uneven_ok) ? CP_ERR_NOT_DIVISIBLE : CP_OK;
  if (uneven_ok) return CP_OK;  // Ulysses Anything: any S and H
  if (H % U || S % (static_cast<int64_t>(R) * U)) return CP_ERR_NOT_DIVISIBLE;
  return CP_OK;
}

cp_status cp_ring_shard_table(int S, int n, int uneven_ok, int* offsets, int* lengths) {
  if (!offsets || !lengths) return CP_ERR_INVALID_ARG;
  return shard_table(S, n, uneven_ok != 0, offsets, lengths);
}

size_t cp_attention_workspace_size(int B, int H, int S, int D, int ring_degree, int ulysses_degree, cp_dtype dt,
                                   cp_lap_mode mode) {
  if (B < 0 || H < 1 || S < 0 || D < 1 || ring_degree < 1 || ulysses_degree < 1) return 0;
  return ws_layout(B, H, S, D, ring_degree, ulysses_degree, dt, mode).total;
}

}  // extern "C" (reopened below)

// Copies of the simulated Ulysses all-to-all #1, global [B,S,H,D] -> [U][B,S,Hg,D]
// with Hg = ceil(H/U), for q, k and v (src -> dst). With H % U != 0 the head
// groups are a balanced split and a short group leaves its last head slot
// unwritten (padding).
static void ulysses_in_copies(const void* const src[3], void* const dst[3], int B, int H, int S, int D, int U, int eb,
                              std::vector<SegCopy>* cs) {
  const int Hg = (H + U - 1) / U;
  const int64_t row = static_cast<int64_t>(Hg) * D;
  const int64_t grp = static_cast<int64_t>(B) * S * row;  // elements per head group
  if (H % U == 0) {
    // out segments (g, b, t) of Hg*D elements <- in[b, t, g*Hg : (g+1)*Hg, :]
    for (int i = 0; i < 3; ++i)
      cs->push_back(SegCopy{src[i], dst[i], 1, U, B, S, 0, row, static_cast<int64_t>(S) * H * D,
                            static_cast<int64_t>(H) * D, row, eb});
    return;
  }
  std::vector<int> hoff(U), hlen(U);
  (void)shard_table(H, U, true, hoff.data(), hlen.data());
  for (int i = 0; i < 3; ++i)
    for (int g = 0; g < U; ++g)
      // group g, rows (b, t) of hlen[g]*D elements <- in[b, t, hoff[g] : hoff[g] + hlen[g], :]
      cs->push_back(SegCopy{static_cast<const char*>(src[i]) + static_cast<int64_t>(hoff[g]) * D * eb,
                            static_cast<char*>(dst[i]) + g * grp * eb, 1, 1, B, S, 0, 0,
                            static_cast<int64_t>(S) * H * D, static_cast<int64_t>(H) * D,
                            static_cast<int64_t>(hlen[g]) * D, eb, 0, 0, S * row, row});
}

// Copies of the simulated Ulysses all-to-all #2: out [U][B,S,Hg,D] -> [B,S,H,D]
// and lse [U][B,Hg,S] -> [B,H,S], real heads only.
static void ulysses_out_copies(const float* oa, const float* la, float* out, float* lse, int B, int H, int S, int D,
                               int U, std::vector<SegCopy>* cs) {
  const int Hg = (H + U - 1) / U;
  const int64_t row = static_cast<int64_t>(Hg) * D;
  const int64_t bstride = S * row;
  const int64_t grp = static_cast<int64_t>(B) * bstride;
  if (H % U == 0) {
    cs->push_back(SegCopy{oa, out, 1, B, S, U, 0, bstride, row, static_cast<int64_t>(B) * bstride, row, 4});
    cs->push_back(SegCopy{la, lse, 1, B, U, Hg, 0, static_cast<int64_t>(Hg) * S, static_cast<int64_t>(B) * Hg * S,
                          S, S, 4});
    return;
  }
  std::vector<int> hoff(U), hlen(U);
  (void)shard_table(H, U, true, hoff.data(), hlen.data());
  for (int g = 0; g < U; ++g) {
    // out[b, t, hoff[g] + h, :] <- group g row (b, t)
    cs->push_back(SegCopy{oa + g * grp, out + static_cast<int64_t>(hoff[g]) * D, 1, 1, B, S, 0, 0, S * row, row,
                          static_cast<int64_t>(hlen[g]) * D, 4, 0, 0, static_cast<int64_t>(S) * H * D,
                          static_cast<int64_t>(H) * D});
    // lse[b, hoff[g] + h, :] <- group g lse[b, h, :]
    cs->push_back(SegCopy{la + static_cast<int64_t>(g) * B * Hg * S, lse + static_cast<int64_t>(hoff[g]) * S, 1, 1,
                          B, hlen[g], 0, 0, static_cast<int64_t>(Hg) * S, S, S, 4, 0, 0,
                          static_cast<int64_t>(H) * S, S});
  }
}

extern "C" {

int cp_attention_launch_count(int B, int H, int S, int D, int ring_degree, int ulysses_degree, cp_dtype dt,
                              cp_lap_mode mode) {
  if (B == 0 || S == 0) return 0;
  const int R = ring_degree, U = ulysses_degree;
  int n = (mode == CP_LAP_STEPWISE && R > 1) ? R + (R - 1) : 1;
  if (U > 1 && U <= H && D > 0) {
    // the same copy descriptors as a call makes, on stand-in addresses with
    // the alignment (256 B) of the caller's buffers and the workspace
    const WsLayout w = ws_layout(B, H, S, D, R, U, dt, mode);
    char* base = reinterpret_cast<char*>(uintptr_t{1} << 20);
    const void* src[3] = {base, base, base};
    void* dst[3] = {base + w.qh, base + w.kh, base + w.vh};
    std::vector<SegCopy> in, out;
    ulysses_in_copies(src, dst, B, H, S, D, U, elem_size(dt), &in);
    ulysses_out_copies(reinterpret_cast<float*>(base + w.oh), reinterpret_cast<float*>(base + w.lh),
                       reinterpret_cast<float*>(base), reinterpret_cast<float*>(base), B, H, S, D, U, &out);
    n += cp::segment_copy_launches(in.data(), static_cast<int>(in.size())) +
         cp::segment_copy_launches(out.data(), static_cast<int>(out.size()));
  }
  return n;
}

}  // extern "C" (reopened below)

// cp_attention_fwd with an optional key-padding mask [B, S] (device, nonzero = attend).
static cp_status attention_fwd_impl(const void* q, const void* k, const void* v, const uint8_t* key_mask, float* out,
                                    float* lse, int B, int H, int S, int D, float scale, int ring_degree,
                                    int ulysses_degree, int uneven_ok, void* workspace, size_t ws_bytes, cp_dtype dt,
                                    cp_lap_mode mode, void* stream) {
  cp_status st = cp_attention_validate(B, H, S, D, ring_degree, ulysses_degree, uneven_ok, dt);
  if (st != CP_OK) return st;
  if (!std::isfinite(scale) || (mode != CP_LAP_FUSED && mode != CP_LAP_STEPWISE)) return CP_ERR_INVALID_ARG;
  if (B == 0 || S == 0) return CP_OK;
  if (!q || !k || !v || !out || !lse) return CP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse)) return CP_ERR_ALIGNMENT;
  const int R = ring_degree, U = ulysses_degree;
  const WsLayout w = ws_layout(B, H, S, D, R, U, dt, mode);
  if (w.total > 0 && (!workspace || ws_bytes < w.total)) return CP_ERR_WORKSPACE;
  if (w.total > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255)) return CP_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev)) != CP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const int eb = elem_size(dt);
  // head groups: balanced split of H into U (Ulysses Anything may leave it
  // uneven); each group is stored with Hg = ceil(H/U) heads, the last head of
  // a short group being padding that the attention kernels skip
  const int Hg = (H + U - 1) / U, Bn = B * U;
  const bool ragged = H % U != 0;
  const int64_t row = static_cast<int64_t>(Hg) * D;

  // --- Ulysses all-to-all #1 (simulated): global [B,S,H,D] -> [U][B,S,Hg,D] ---
  const void *qa = q, *ka = k, *va = v;
  float* oa = out;
  float* la = lse;
  if (U > 1) {
    void* dst[3] = {ws + w.qh, ws + w.kh, ws + w.vh};
    const void* src[3] = {q, k, v};
    std::vector<SegCopy> cs;  // disjoint outputs: they share launches
    ulysses_in_copies(src, dst, B, H, S, D, U, eb, &cs);
    if (cp::launch_segment_copies(cs.data(), static_cast<int>(cs.size()), s) != cudaSuccess) return CP_ERR_CUDA;
    qa = dst[0];
    ka = dst[1];
    va = dst[2];
    oa = reinterpret_cast<float*>(ws + w.oh);
    la = reinterpret_cast<float*>(ws + w.lh);
  }

  // --- ring lap over R simulated ranks on every (group, batch) entry ---
  int off[cp::kMaxRanks], len[cp::kMaxRanks];
  if ((st = shard_table(S, R, uneven_ok != 0, off, len)) != CP_OK) return st;
  const int64_t bstride = S * row;
  if (mode == CP_LAP_FUSED || R == 1) {
    RingGeom g;
    fill_geom(&g, dt, R, off, len, R, off, len, -1);
    AttnTensors t{qa, ka, va, Bn, Hg, D, S, S, bstride, bstride, oa, bstride, la};
    if (U > 1 && ragged) {
      t.hv_bpg = B;
      t.hv_short_from = H % U;
    }
    t.kmask = key_mask;  // batch entry (g, b) of a Ulysses group reads mask row b
    t.km_bstride = S;
    t.km_bmod = B;
    if ((st = launch_attention(t, g, scale, dt, dev, s)) != CP_OK) return st;
  } else {
    float* op = reinterpret_cast<float*>(ws + w.op);
    float* lp = reinterpret_cast<float*>(ws + w.lp);
    for (int step = 0; step < R; ++step) {
      RingGeom g;
      fill_geom(&g, dt, R, off, len, R, off, len, step);
      AttnTensors t{qa, ka, va, Bn, Hg, D, S, S, bstride, bstride, step == 0 ? oa : op, bstride, step == 0 ? la : lp};
      t.kmask = key_mask;
      t.km_bstride = S;
      t.km_bmod = B;
      if ((st = launch_attention(t, g, scale, dt, dev, s)) != CP_OK) return st;
      if (step > 0 && cp::launch_lse_merge(oa, la, op, lp, Bn, Hg, S, D, s) != cudaSuccess) return CP_ERR_CUDA;
    }
  }

  // --- Ulysses all-to-all #2 (simulated): [U][B,S,Hg,D] -> [B,S,H,D]; lse [U][B,Hg,S] -> [B,H,S] ---
  if (U > 1) {
    std::vector<SegCopy> cs;
    ulysses_out_copies(oa, la, out, lse, B, H, S, D, U, &cs);
    if (cp::launch_segment_copies(cs.data(), static_cast<int>(cs.size()), s) != cudaSuccess) return CP_ERR_CUDA;
  }
  return CP_OK;
}

extern "C" {

cp_status cp_attention_fwd(const void* q, const void* k, const void* v, float* out, float* lse, int B, int H, int S,
                           int D, float scale, int ring_degree, int ulysses_degree, int uneven_ok, void* workspace,
                           size_t ws_bytes, cp_dtype dt, cp_lap_mode mode, void* stream) {
  return attention_fwd_impl(q, k, v, nullptr, out, lse, B, H, S, D, scale, ring_degree, ulysses_degree, uneven_ok,
                            workspace, ws_bytes, dt, mode, stream);
}

cp_status cp_attention_fwd_masked(const void* q, const void* k, const void* v, const uint8_t* key_mask, float* out,
                                  float* lse, int B, int H, int S, int D, float scale, int ring_degree,
                                  int ulysses_degree, int uneven_ok, void* workspace, size_t ws_bytes, cp_dtype dt,
                                  cp_lap_mode mode, void* stream) {
  // Ring Anything takes no mask ("Ring Anything Attention": attn_mask must be None)
  if (key_mask && uneven_ok && ring_degree > 1) return CP_ERR_UNSUPPORTED_COMBO;
  return attention_fwd_impl(q, k, v, key_mask, out, lse, B, H, S, D, scale, ring_degree, ulysses_degree, uneven_ok,
                            workspace, ws_bytes, dt, mode, stream);
}

// ---------------------------------------------------------------------------
// cp_attention_fwd over host buffers: copies in, attention, copies out, with
// the head range split into chunks whose copies overlap the other chunks'
// attention (two copy streams of the library, one per direction).
// ---------------------------------------------------------------------------
constexpr int kMaxHostChunks = 16;

struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, out_done = nullptr;
  cudaEvent_t in_done[kMaxHostChunks] = {}, comp_done[kMaxHostChunks] = {};
  std::mutex mu;
};
static HostPipe g_pipe[kMaxDevices];

// Device buffer of cp_attention_fwd_host: q, k, v (dt), out, lse (fp32), then
// the workspace of cp_attention_fwd; every piece 256-byte aligned.
struct HostLayout {
  size_t q = 0, k = 0, v = 0, out = 0, lse = 0, ws = 0, ws_bytes = 0, total = 0;
};

static HostLayout host_layout(int B, int H, int S, int D, int R, int U, cp_dtype dt, cp_lap_mode mode) {
  HostLayout h;
  const size_t n = static_cast<size_t>(B) * S * H * D;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = round_up(o + bytes, 256);
    return at;
  };
  h.q = take(n * elem_size(dt));
  h.k = take(n * elem_size(dt));
  h.v = take(n * elem_size(dt));
  h.out = take(n * 4);
  h.lse = take(static_cast<size_t>(B) * H * S * 4);
  h.ws_bytes = ws_layout(B, H, S, D, R, U, dt, mode).total;
  h.ws = take(h.ws_bytes);
  h.total = o;
  return h;
}

}  // extern "C" (reopened below)

static cp_status host_pipe(int dev, HostPipe** out) {
  HostPipe& p = g_pipe[dev];
  if (!p.ready) {
    if (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.out_done, cudaEventDisableTiming) != cudaSuccess)
      return CP_ERR_CUDA;
    for (int j = 0; j < kMaxHostChunks; ++j)
      if (cudaEventCreateWithFlags(&p.in_done[j], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.comp_done[j], cudaEventDisableTiming) != cudaSuccess)
        return CP_ERR_CUDA;
    p.ready = true;
  }
  *out = &p;
  return CP_OK;
}

extern "C" {

size_t cp_attention_host_buffer_size(int B, int H, int S, int D, int ring_degree, int ulysses_degree, cp_dtype dt,
                                     cp_lap_mode mode) {
  if (B < 0 || H < 1 || S < 0 || D < 1 || ring_degree < 1 || ulysses_degree < 1) return 0;
  return host_layout(B, H, S, D, ring_degree, ulysses_degree, dt, mode).total;
}

cp_status cp_attention_fwd_host(const void* q, const void* k, const void* v, float* out, float* lse, int B, int H,
                                int S, int D, float scale, int ring_degree, int ulysses_degree, int uneven_ok,
                                void* dev_buffer, size_t dev_bytes, cp_dtype dt, cp_lap_mode mode, int head_chunks,
                                void* stream) {
  cp_status st = cp_attention_validate(B, H, S, D, ring_degree, ulysses_degree, uneven_ok, dt);
  if (st != CP_OK) return st;
  if (!std::isfinite(scale) || (mode != CP_LAP_FUSED && mode != CP_LAP_STEPWISE) || head_chunks < 1)
    return CP_ERR_INVALID_ARG;
  if (B == 0 || S == 0) return CP_OK;
  if (!q || !k || !v || !out || !lse || !dev_buffer) return CP_ERR_INVALID_ARG;
  const int R = ring_degree, U = ulysses_degree;
  const HostLayout L = host_layout(B, H, S, D, R, U, dt, mode);
  if (dev_bytes < L.total) return CP_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(dev_buffer) & 255) return CP_ERR_ALIGNMENT;
  DeviceInfo* dinfo = nullptr;
  if ((st = current_device(&dinfo)) != CP_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(dev_buffer);
  const int eb = elem_size(dt);
  const size_t n = static_cast<size_t>(B) * S * H * D;
  void* dq = base + L.q;
  void* dk = base + L.k;
  void* dv = base + L.v;
  float* dout = reinterpret_cast<float*>(base + L.out);
  float* dlse = reinterpret_cast<float*>(base + L.lse);
  // chunks of heads only where heads are independent launches: a fused lap
  // (or plain attention) without Ulysses regroups
  int chunks = head_chunks < H ? head_chunks : H;
  if (chunks > kMaxHostChunks) chunks = kMaxHostChunks;
  if (U > 1 || (mode == CP_LAP_STEPWISE && R > 1)) chunks = 1;
  if (chunks == 1) {
    if (cudaMemcpyAsync(dq, q, n * eb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(dk, k, n * eb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(dv, v, n * eb, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return CP_ERR_CUDA;
    if ((st = cp_attention_fwd(dq, dk, dv, dout, dlse, B, H, S, D, scale, R, U, uneven_ok, base + L.ws, L.ws_bytes,
                               dt, mode, stream)) != CP_OK)
      return st;
    if (cudaMemcpyAsync(out, dout, n * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(lse, dlse, static_cast<size_t>(B) * H * S * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return CP_ERR_CUDA;
    return CP_OK;
  }
  HostPipe* p = nullptr;
  std::lock_guard<std::mutex> lk(g_pipe[dev].mu);
  if ((st = host_pipe(dev, &p)) != CP_OK) return st;
  int off[cp::kMaxRanks], len[cp::kMaxRanks];
  if ((st = shard_table(S, R, uneven_ok != 0, off, len)) != CP_OK) return st;
  RingGeom g;
  fill_geom(&g, dt, R, off, len, R, off, len, -1);
  // head chunks: the copies up are the bottleneck. What precedes the first
  // chunk's attention (its copy up) and what follows the last chunk's copy
  // up (its attention, its copy back) is exposed, so those two chunks get
  // about a third of an even share each, and the middle chunks the rest,
  // largest first, each at most one wave of work items (a launch of up to a
  // wave takes one item's time whatever its size). Where the middle chunks
  // cannot hold the rest within a wave each, only the last chunk is small
  // and the others split the rest evenly.
  std::vector<int> ho(chunks), hl(chunks);
  {
    const int n_single = g.single_prefix[g.n_q];
    const int64_t per_head = static_cast<int64_t>(g.pair_prefix[g.n_q] + n_single - n_single / 2) * B;
    const int64_t wave_heads = per_head > 0 ? dinfo->sms / per_head : 0;  // heads per wave of items
    int edge = (H + 3 * chunks / 2) / (3 * chunks);
    if (edge < 1) edge = 1;
    const int mids = chunks - 2, rest = H - 2 * edge;
    if (mids >= 1 && rest >= mids && wave_heads >= 1 && wave_heads * mids >= rest) {
      hl[0] = edge;
      int left = rest;
      for (int j = 1; j <= mids; ++j) {
        hl[j] = static_cast<int>(std::min<int64_t>(wave_heads, left - (mids - j)));
        left -= hl[j];
      }
      hl[chunks - 1] = edge;
      for (int j = 0, o = 0; j < chunks; ++j) {
        ho[j] = o;
        o += hl[j];
      }
    } else {
      int last = edge;
      if (H - last < chunks - 1) last = H - (chunks - 1);
      if (shard_table(H - last, chunks - 1, true, ho.data(), hl.data()) != CP_OK) return CP_ERR_INVALID_ARG;
      ho[chunks - 1] = H - last;
      hl[chunks - 1] = last;
    }
  }
  const size_t row_b = static_cast<size_t>(H) * D * eb, row4 = static_cast<size_t>(H) * D * 4;
  // copies start after everything already queued on the caller's stream
  if (cudaEventRecord(p->start, s) != cudaSuccess || cudaStreamWaitEvent(p->in, p->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(p->out, p->start, 0) != cudaSuccess)
    return CP_ERR_CUDA;
  for (int j = 0; j < chunks; ++j) {
    const size_t hb = static_cast<size_t>(ho[j]) * D;  // element offset of the chunk's first head
    const size_t w_b = static_cast<size_t>(hl[j]) * D * eb, w4 = static_cast<size_t>(hl[j]) * D * 4;
    const void* src[3] = {q, k, v};
    void* dst[3] = {dq, dk, dv};
    for (int i = 0; i < 3; ++i)
      if (cudaMemcpy2DAsync(static_cast<char*>(dst[i]) + hb * eb, row_b, static_cast<const char*>(src[i]) + hb * eb,
                            row_b, w_b, static_cast<size_t>(B) * S, cudaMemcpyHostToDevice, p->in) != cudaSuccess)
        return CP_ERR_CUDA;
    if (cudaEventRecord(p->in_done[j], p->in) != cudaSuccess || cudaStreamWaitEvent(s, p->in_done[j], 0) != cudaSuccess)
      return CP_ERR_CUDA;
    AttnTensors t{static_cast<const char*>(dq) + hb * eb, static_cast<const char*>(dk) + hb * eb,
                  static_cast<const char*>(dv) + hb * eb, B, hl[j], D, S, S,
                  static_cast<int64_t>(S) * H * D, static_cast<int64_t>(S) * H * D, dout + hb,
                  static_cast<int64_t>(S) * H * D, dlse + static_cast<size_t>(ho[j]) * S};
    t.row = static_cast<int64_t>(H) * D;
    t.l_bstride = static_cast<int64_t>(H) * S;
    if ((st = launch_attention(t, g, scale, dt, dinfo, s)) != CP_OK) return st;
    if (cudaEventRecord(p->comp_done[j], s) != cudaSuccess || cudaStreamWaitEvent(p->out, p->comp_done[j], 0) != cudaSuccess)
      return CP_ERR_CUDA;
    if (cudaMemcpy2DAsync(reinterpret_cast<char*>(out) + hb * 4, row4, reinterpret_cast<const char*>(dout + hb), row4,
                          w4, static_cast<size_t>(B) * S, cudaMemcpyDeviceToHost, p->out) != cudaSuccess ||
        cudaMemcpy2DAsync(reinterpret_cast<char*>(lse) + static_cast<size_t>(ho[j]) * S * 4,
                          static_cast<size_t>(H) * S * 4,
                          reinterpret_cast<const char*>(dlse + static_cast<size_t>(ho[j]) * S),
                          static_cast<size_t>(H) * S * 4, static_cast<size_t>(hl[j]) * S * 4, static_cast<size_t>(B),
                          cudaMemcpyDeviceToHost, p->out) != cudaSuccess)
      return CP_ERR_CUDA;
  }
  // the caller's stream resumes once every result is back in host memory
  if (cudaEventRecord(p->out_done, p->out) != cudaSuccess || cudaStreamWaitEvent(s, p->out_done, 0) != cudaSuccess)
    return CP_ERR_CUDA;
  return CP_OK;
}

cp_status cp_check_device_status(void* stream) {
  DeviceInfo* dev = nullptr;
  cp_status st = current_device(&dev);
  if (st != CP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return CP_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, dev->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return CP_ERR_CUDA;
  if (word == 0) return CP_OK;
  if (cudaMemset(dev->err, 0, sizeof(word)) != cudaSuccess) return CP_ERR_CUDA;
  // bit 0: a bounded wait expired; bit 1: a kernel found its shared memory misaligned
  return (word & 1u) ? CP_ERR_TIMEOUT : CP_ERR_CUDA;
}

cp_status cp_debug_bounded_wait_probe(int timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return CP_ERR_INVALID_ARG;
  DeviceInfo* dev = nullptr;
  cp_status st = current_device(&dev);
  if (st != CP_OK) return st;
  return cp::launch_wait_probe(dev->err, static_cast<uint64_t>(timeout_us) * 1000ull,
                               static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CP_OK
             : CP_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// cp_attention_fwd_no_alloc: the workspace is a static device array of this
// file instead of caller memory. Host code sees only a stand-in for the
// array's symbol, so its device address is looked up once per device (with
// that device current) and handed to the kernels as the workspace pointer.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_no_alloc_ws[CP_NO_ALLOC_WORKSPACE_BYTES];

void* g_no_alloc_ws_addr[kMaxDevices];
std::mutex g_no_alloc_mu;

cp_status no_alloc_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CP_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_no_alloc_mu);
  if (!g_no_alloc_ws_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_no_alloc_ws) != cudaSuccess || !p) return CP_ERR_CUDA;
    g_no_alloc_ws_addr[dev] = p;
  }
  *out = g_no_alloc_ws_addr[dev];
  return CP_OK;
}

}  // namespace

extern "C" cp_status cp_attention_fwd_no_alloc(const void* q, const void* k, const void* v, float* out, float* lse,
                                               int B, int H, int S, int D, float scale, int ring_degree,
                                               int ulysses_degree, int uneven_ok, cp_dtype dt, cp_lap_mode mode,
                                               void* stream) {
  cp_status st = cp_attention_validate(B, H, S, D, ring_degree, ulysses_degree, uneven_ok, dt);
  if (st != CP_OK) return st;
  if (mode != CP_LAP_FUSED && mode != CP_LAP_STEPWISE) return CP_ERR_INVALID_ARG;
  const size_t need = cp_attention_workspace_size(B, H, S, D, ring_degree, ulysses_degree, dt, mode);
  if (need > CP_NO_ALLOC_WORKSPACE_BYTES) return CP_ERR_WORKSPACE;
  if (B == 0 || S == 0) return CP_OK;
  DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev)) != CP_OK) return st;
  // a problem that needs no scratch (plain ring, fused lap) never touches the
  // array, so it neither looks the symbol up nor makes a first-call set-up
  if (need == 0)
    return cp_attention_fwd(q, k, v, out, lse, B, H, S, D, scale, ring_degree, ulysses_degree, uneven_ok, nullptr, 0,
                            dt, mode, stream);
  void* ws = nullptr;
  if ((st = no_alloc_workspace(&ws)) != CP_OK) return st;
  return cp_attention_fwd(q, k, v, out, lse, B, H, S, D, scale, ring_degree, ulysses_degree, uneven_ok, ws,
                          CP_NO_ALLOC_WORKSPACE_BYTES, dt, mode, stream);
}

// ----------------------------------------------------------------------------
// Backward (ring, Ulysses, unified; even splits only).
// ----------------------------------------------------------------------------
namespace {

// Workspace layout of cp_attention_bwd (every piece 256-byte aligned):
// delta [B, H, S]; with Ulysses, the head-group copies of q, k, v, dout
// [U][B, S, H/U, D], of lse and delta [U][B, H/U, S], and the head-group
// gradients dq, dk, dv [U][B, S, H/U, D] fp32; for bf16, the tensor-core
// dk/dv kernel's per-shard padded lse * log2 e and delta (BwdArgs::lse2p).
struct BwdWs {
  size_t delta = 0, qh = 0, kh = 0, vh = 0, doh = 0, lh = 0, dlh = 0, dqh = 0, dkh = 0, dvh = 0, l2p = 0, dlp = 0,
         total = 0;
  int lpad = 0;
};

// rows of a shard in the padded lse / delta layout: the longest shard, rounded up to 64
int bwd_lpad(int S, int R) { return (S / R + (S % R ? 1 : 0) + 63) / 64 * 64; }

BwdWs bwd_ws_layout(int B, int H, int S, int D, int R, int U, cp_dtype dt) {
  BwdWs w;
  // U head groups of ceil(H/U) heads (the last head of a short group is padding)
  const size_t Hp = U > 1 ? static_cast<size_t>((H + U - 1) / U) * U : static_cast<size_t>(H);
  const size_t n = static_cast<size_t>(B) * S * Hp * D, nl = static_cast<size_t>(B) * Hp * S;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = round_up(o + bytes, 256);
    return at;
  };
  w.delta = take(static_cast<size_t>(B) * H * S * 4);
  if (U > 1) {
    w.qh = take(n * elem_size(dt));
    w.kh = take(n * elem_size(dt));
    w.vh = take(n * elem_size(dt));
    w.doh = take(n * elem_size(dt));
    w.lh = take(nl * 4);
    w.dlh = take(nl * 4);
    w.dqh = take(n * 4);
    w.dkh = take(n * 4);
    w.dvh = take(n * 4);
  }
  if (dt == CP_BF16 && R >= 1) {
    w.lpad = bwd_lpad(S, R);
    const size_t np = static_cast<size_t>(B) * Hp * R * w.lpad;
    w.l2p = take(np * 4);
    w.dlp = take(np * 4);
  }
  w.total = o;
  return w;
}

cp_status bwd_validate(int B, int H, int S, int D, int R, int U, int uneven_ok, cp_dtype dt) {
  // Ring Anything is inference only; Ulysses Anything has a backward
  if (uneven_ok && R > 1) return CP_ERR_UNSUPPORTED_COMBO;
  return cp_attention_validate(B, H, S, D, R, U, uneven_ok, dt);
}

// Copies of the backward's Ulysses regroups: q, k, v, dout [B,S,H,D] -> [U][B,S,Hg,D]
// and lse, delta [B,H,S] -> [U][B,Hg,S] (in), or dq, dk, dv back (out), with
// Hg = ceil(H/U). With H % U != 0 the head groups are the balanced split and
// a short group's last head slot is left unwritten (padding).
void bwd_in_copies(const void* const src[4], void* const dst[4], const float* lse, const float* delta, float* lh,
                   float* dlh, int B, int H, int S, int D, int U, int eb, std::vector<SegCopy>* cs) {
  const int Hg = (H + U - 1) / U;
  const int64_t row = static_cast<int64_t>(Hg) * D;
  const int64_t grp = static_cast<int64_t>(B) * S * row;  // elements per head group
  const float* ls[2] = {lse, delta};
  float* ld[2] = {lh, dlh};
  if (H % U == 0) {
    for (int i = 0; i < 4; ++i)
      cs->push_back(SegCopy{src[i], dst[i], 1, U, B, S, 0, row, static_cast<int64_t>(S) * H * D,
                            static_cast<int64_t>(H) * D, row, eb});
    // out segments (g, b, h) of S floats <- in[b, g*Hg + h, :]
    for (int i = 0; i < 2; ++i)
      cs->push_back(SegCopy{ls[i], ld[i], 1, U, B, Hg, 0, static_cast<int64_t>(Hg) * S,
                            static_cast<int64_t>(H) * S, S, S, 4});
    return;
  }
  std::vector<int> hoff(U), hlen(U);
  (void)shard_table(H, U, true, hoff.data(), hlen.data());
  for (int i = 0; i < 4; ++i)
    for (int g = 0; g < U; ++g)
      // group g, rows (b, t) of hlen[g]*D elements <- in[b, t, hoff[g] : hoff[g] + hlen[g], :]
      cs->push_back(SegCopy{static_cast<const char*>(src[i]) + static_cast<int64_t>(hoff[g]) * D * eb,
                            static_cast<char*>(dst[i]) + g * grp * eb, 1, 1, B, S, 0, 0,
                            static_cast<int64_t>(S) * H * D, static_cast<int64_t>(H) * D,
                            static_cast<int64_t>(hlen[g]) * D, eb, 0, 0, S * row, row});
  for (int i = 0; i < 2; ++i)
    for (int g = 0; g < U; ++g)
      // group g's [b, h, :] <- in[b, hoff[g] + h, :], h < hlen[g]
      cs->push_back(SegCopy{ls[i] + static_cast<int64_t>(hoff[g]) * S, ld[i] + static_cast<int64_t>(g) * B * Hg * S,
                            1, 1, B, hlen[g], 0, 0, static_cast<int64_t>(H) * S, S, S, 4, 0, 0,
                            static_cast<int64_t>(Hg) * S, S});
}

void bwd_out_copies(const float* const src[3], float* const dst[3], int B, int H, int S, int D, int U,
                    std::vector<SegCopy>* cs) {
  const int Hg = (H + U - 1) / U;
  const int64_t row = static_cast<int64_t>(Hg) * D, bstride = S * row;
  if (H % U == 0) {
    for (int i = 0; i < 3; ++i)
      cs->push_back(
          SegCopy{src[i], dst[i], 1, B, S, U, 0, bstride, row, static_cast<int64_t>(B) * bstride, row, 4});
    return;
  }
  std::vector<int> hoff(U), hlen(U);
  (void)shard_table(H, U, true, hoff.data(), hlen.data());
  for (int i = 0; i < 3; ++i)
    for (int g = 0; g < U; ++g)
      // out[b, t, hoff[g] + h, :] <- group g row (b, t), real heads only
      cs->push_back(SegCopy{src[i] + g * B * bstride, dst[i] + static_cast<int64_t>(hoff[g]) * D, 1, 1, B, S, 0, 0,
                            bstride, row, static_cast<int64_t>(hlen[g]) * D, 4, 0, 0,
                            static_cast<int64_t>(S) * H * D, static_cast<int64_t>(H) * D});
}

}  // namespace

extern "C" {

size_t cp_attention_bwd_workspace_size(int B, int H, int S, int D, int ring_degree, int ulysses_degree, cp_dtype dt) {
  if (B < 0 || H < 1 || S < 0 || D < 1 || ring_degree < 1 || ulysses_degree < 1) return 0;
  return bwd_ws_layout(B, H, S, D, ring_degree, ulysses_degree, dt).total;
}

int cp_attention_bwd_launch_count(int B, int H, int S, int D, int ring_degree, int ulysses_degree, cp_dtype dt) {
  if (B <= 0 || S <= 0 || H < 1 || D < 1 || ring_degree < 1 || ulysses_degree < 1) return 0;
  const int U = ulysses_degree;
  // delta, then the dk/dv and dq kernels: on the CUDA cores (fp32) one launch
  // each; on the tensor cores (bf16) the padded lse / delta copy of the dk/dv
  // CTAs, then one launch of both kinds of CTA
  int n = 3;
  if (U > 1 && U <= H) {
    const BwdWs w = bwd_ws_layout(B, H, S, D, ring_degree, U, dt);
    char* base = reinterpret_cast<char*>(uintptr_t{1} << 20);
    const void* src[4] = {base, base, base, base};
    void* dst[4] = {base + w.qh, base + w.kh, base + w.vh, base + w.doh};
    std::vector<SegCopy> in, out;
    bwd_in_copies(src, dst, reinterpret_cast<float*>(base), reinterpret_cast<float*>(base + w.delta),
                  reinterpret_cast<float*>(base + w.lh), reinterpret_cast<float*>(base + w.dlh), B, H, S, D, U,
                  elem_size(dt), &in);
    const float* gs[3] = {reinterpret_cast<float*>(base + w.dqh), reinterpret_cast<float*>(base + w.dkh),
                          reinterpret_cast<float*>(base + w.dvh)};
    float* gd[3] = {reinterpret_cast<float*>(base), reinterpret_cast<float*>(base), reinterpret_cast<float*>(base)};
    bwd_out_copies(gs, gd, B, H, S, D, U, &out);
    n += cp::segment_copy_launches(in.data(), static_cast<int>(in.size())) +
         cp::segment_copy_launches(out.data(), static_cast<int>(out.size()));
  }
  return n;
}

cp_status cp_attention_bwd(const void* q, const void* k, const void* v, const float* out, const void* dout,
                           const float* lse, float* dq, float* dk, float* dv, int B, int H, int S, int D, float scale,
                           int ring_degree, int ulysses_degree, int uneven_ok, void* workspace, size_t ws_bytes,
                           cp_dtype dt, void* stream) {
  cp_status st = bwd_validate(B, H, S, D, ring_degree, ulysses_degree, uneven_ok, dt);
  if (st != CP_OK) return st;
  if (!std::isfinite(scale)) return CP_ERR_INVALID_ARG;
  if (B == 0 || S == 0) return CP_OK;
  const void* ptrs[9] = {q, k, v, out, dout, lse, dq, dk, dv};
  for (const void* p : ptrs) {
    if (p == nullptr) return CP_ERR_INVALID_ARG;
    if (!aligned16(p)) return CP_ERR_ALIGNMENT;
  }
  const int R = ring_degree, U = ulysses_degree;
  const BwdWs w = bwd_ws_layout(B, H, S, D, R, U, dt);
  if (!workspace || ws_bytes < w.total) return CP_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return CP_ERR_ALIGNMENT;
  DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev)) != CP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const bool bf16 = dt == CP_BF16;
  float* delta = reinterpret_cast<float*>(ws + w.delta);
  if (cp::launch_attn_bwd_delta(out, dout, delta, B, S, H, D, bf16, s) != cudaSuccess) return CP_ERR_CUDA;

  cp::BwdArgs a{};
  a.n = R;
  if ((st = shard_table(S, R, false, a.off, a.len)) != CP_OK) return st;
  a.q_prefix[0] = a.kv_prefix[0] = 0;
  const int tile = bf16 ? cp::kBwdTcTile : cp::kBwdTile;
  for (int r = 0; r < R; ++r) {
    const int tiles = (a.len[r] + tile - 1) / tile;
    a.q_prefix[r + 1] = a.q_prefix[r] + tiles;
    a.kv_prefix[r + 1] = a.kv_prefix[r] + tiles;
  }
  a.S = S;
  a.scale = scale;
  a.err = dev->err;
  a.timeout_ns = kWaitTimeoutNs;
  a.lse2p = reinterpret_cast<float*>(ws + w.l2p);
  a.dltp = reinterpret_cast<float*>(ws + w.dlp);
  a.lpad = w.lpad;
  // bf16: tensor maps over the (possibly head-grouped) q, k, v, dout, then the tensor-core kernels
  auto run = [&](int Bn, int Hx) -> cp_status {
    if (!bf16) return cp::launch_attn_bwd(a, D, false, s) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
    if (cp::launch_attn_bwd_prep(a, s) != cudaSuccess) return CP_ERR_CUDA;
    cp::BwdTensorMaps m;
    const int64_t row = static_cast<int64_t>(Hx) * D;
    if (!make_tmap_bf16(&m.q, a.q, D, Hx, S, Bn, row, a.bstride) ||
        !make_tmap_bf16(&m.k, a.k, D, Hx, S, Bn, row, a.bstride) ||
        !make_tmap_bf16(&m.v, a.v, D, Hx, S, Bn, row, a.bstride) ||
        !make_tmap_bf16(&m.o, a.dout, D, Hx, S, Bn, row, a.bstride) ||
        !make_tmap_bf16(&m.q64, a.q, D, Hx, S, Bn, row, a.bstride, 64) ||
        !make_tmap_bf16(&m.k64, a.k, D, Hx, S, Bn, row, a.bstride, 64) ||
        !make_tmap_bf16(&m.v64, a.v, D, Hx, S, Bn, row, a.bstride, 64) ||
        !make_tmap_bf16(&m.o64, a.dout, D, Hx, S, Bn, row, a.bstride, 64))
      return CP_ERR_CUDA;
    return cp::launch_attn_bwd_tc(a, D, m, s) == cudaSuccess ? CP_OK : CP_ERR_CUDA;
  };
  if (U == 1) {
    a.B = B;
    a.H = H;
    a.q = q;
    a.k = k;
    a.v = v;
    a.dout = dout;
    a.bstride = static_cast<int64_t>(S) * H * D;
    a.sstride = static_cast<int64_t>(H) * D;
    a.lse = lse;
    a.delta = delta;
    a.l_bstride = static_cast<int64_t>(H) * S;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    return run(B, H);
  }
  // Ulysses / unified: regroup to head groups, the ring backward per group, regroup back
  const int eb = elem_size(dt), Hg = (H + U - 1) / U;
  const void* src[4] = {q, k, v, dout};
  void* dst[4] = {ws + w.qh, ws + w.kh, ws + w.vh, ws + w.doh};
  float* lh = reinterpret_cast<float*>(ws + w.lh);
  float* dlh = reinterpret_cast<float*>(ws + w.dlh);
  std::vector<SegCopy> in;
  bwd_in_copies(src, dst, lse, delta, lh, dlh, B, H, S, D, U, eb, &in);
  if (cp::launch_segment_copies(in.data(), static_cast<int>(in.size()), s) != cudaSuccess) return CP_ERR_CUDA;
  float* gq = reinterpret_cast<float*>(ws + w.dqh);
  float* gk = reinterpret_cast<float*>(ws + w.dkh);
  float* gv = reinterpret_cast<float*>(ws + w.dvh);
  a.B = B * U;
  a.H = Hg;
  if (H % U != 0) {  // Ulysses Anything: short head groups' last slot is padding
    a.hv_bpg = B;
    a.hv_short_from = H % U;
  }
  a.q = dst[0];
  a.k = dst[1];
  a.v = dst[2];
  a.dout = dst[3];
  a.bstride = static_cast<int64_t>(S) * Hg * D;
  a.sstride = static_cast<int64_t>(Hg) * D;
  a.lse = lh;
  a.delta = dlh;
  a.l_bstride = static_cast<int64_t>(Hg) * S;
  a.dq = gq;
  a.dk = gk;
  a.dv = gv;
  if ((st = run(B * U, Hg)) != CP_OK) return st;
  const float* gs[3] = {gq, gk, gv};
  float* gd[3] = {dq, dk, dv};
  std::vector<SegCopy> back;
  bwd_out_copies(gs, gd, B, H, S, D, U, &back);
  return cp::launch_segment_copies(back.data(), static_cast<int>(back.size()), s) == cudaSuccess ? CP_OK
                                                                                               : CP_ERR_CUDA;
}

}  // extern "C"
