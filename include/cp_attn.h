/*
 * cp_attn.h — C ABI of libcpattn.so: context-parallel attention forward for
 * diffusion transformers on one GB300 (sm_103a).
 *
 * What it computes (diffusers documentation, "Paralelismo de contexto" page,
 * sections "Atenção em Anel", "Atenção Ulysses", "Atenção Unificada",
 * "Ring Anything Attention", and the "Paralelismo" API page,
 * ContextParallelConfig): non-causal softmax attention of a query shard
 * against the key/value blocks of a ring lap, each block returning an fp32
 * (output, log-sum-exp) partial that is merged online, so that one full lap
 * equals full attention; plus the Ulysses all-to-all regroups between a
 * sequence-sharded and a head-sharded layout. The ranks of the ring and of the
 * Ulysses groups are simulated as shards of one buffer on one GPU: a block
 * "received" from another rank is a pointer offset, and the all-to-all is a
 * regroup kernel that moves the same bytes.
 *
 * Conventions shared by every call
 *   - Layouts: q, k, v, out are [B, S, H, D] row-major (D contiguous, then H,
 *     then S, then B); lse is [B, H, S] float32, natural logarithm of the sum
 *     of exp over the scaled logits scale * q.k. Non-causal, no mask.
 *   - Pointers are DEVICE pointers unless stated. The caller owns every buffer
 *     (inputs, outputs, workspace); the library allocates no device memory
 *     and keeps no per-call state. The one exception is
 *     cp_attention_fwd_no_alloc, whose built-in 64 MiB static device array
 *     (CP_NO_ALLOC_WORKSPACE_BYTES) is shared by all of its calls. Outputs
 *     must not alias inputs unless stated.
 *   - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call is asynchronous on that stream. Arguments are validated on
 *     the host before anything is launched; a failed validation launches
 *     nothing and returns a negative cp_status.
 *   - Supported: D in {64, 128}; q/k/v dtype bf16 (tensor-core path) or f32
 *     (CUDA-core path); out and lse always float32.
 *   - Alignment: every pointer 16-byte aligned; batch strides such that each
 *     batch starts 16-byte aligned. Otherwise CP_ERR_ALIGNMENT.
 *   - Device-side waits are bounded. A kernel whose wait expires records it in
 *     a device error word, releases its resources and returns; read it with
 *     cp_check_device_status().
 */
#ifndef CP_ATTN_H_
#define CP_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CP_OK = 0,
  CP_ERR_INVALID_ARG = -1,       /* bad size, null pointer, unsupported D or dtype, degree > heads */
  CP_ERR_NOT_DIVISIBLE = -2,     /* a length not divisible by a degree that must divide it */
  CP_ERR_UNSUPPORTED_COMBO = -3, /* a flag combination the requirements table rules out */
  CP_ERR_ALIGNMENT = -4,         /* a pointer or stride breaks the 16-byte rule */
  CP_ERR_CUDA = -5,              /* a CUDA launch or runtime call failed */
  CP_ERR_TIMEOUT = -6,           /* a kernel's bounded device wait expired */
  CP_ERR_WORKSPACE = -7,         /* workspace missing or smaller than cp_attention_workspace_size */
  CP_ERR_UNSUPPORTED_DEVICE = -8 /* the current device is not sm_103 */
} cp_status;

typedef enum { CP_BF16 = 0, CP_F32 = 1 } cp_dtype;

/* How cp_attention_fwd runs the ring lap (both give full attention):
 *   CP_LAP_FUSED    one kernel launch; every Q tile walks the K/V blocks in
 *                   ring order (own block first, then its predecessor's, ...)
 *                   and the per-block (out, lse) merge is the running online
 *                   softmax state kept on chip.
 *   CP_LAP_STEPWISE one block-attention launch per ring step over all ranks,
 *                   each writing its fp32 (out, lse) partial, followed by an
 *                   cp_lse_merge launch into the accumulator (steps >= 1). */
typedef enum { CP_LAP_FUSED = 0, CP_LAP_STEPWISE = 1 } cp_lap_mode;

/* Human-readable name of a status code (static string, never NULL). */
const char* cp_status_string(cp_status s);

/* Library version as major*10000 + minor*100 + patch. */
int cp_version(void);

/*
 * Block attention of one query shard against one K/V block ("each device
 * computes attention between its local Q and the KV block it holds": the
 * "Paralelismo" API page, ContextParallelConfig.ring_degree; fp32 output and
 * LSE: ContextParallelConfig.convert_to_fp32).
 *   q    [B, Sq, H, D] (dt), batch stride q_bstride elements (0 = Sq*H*D)
 *   k, v [B, Skv, H, D] (dt), batch stride kv_bstride elements (0 = Skv*H*D)
 *   out  [B, Sq, H, D] float32, batch stride o_bstride elements (0 = Sq*H*D)
 *   lse  [B, H, Sq] float32, dense
 *   out[b,i,h,:] = sum_j softmax_j(scale * q[b,i,h,:].k[b,j,h,:]) v[b,j,h,:]
 *   lse[b,h,i]   = ln sum_j exp(scale * q[b,i,h,:].k[b,j,h,:])
 * Skv == 0 is allowed and yields out = 0, lse = -inf (the merge identity).
 * Sq == 0 or B == 0 launches nothing. Errors: INVALID_ARG, ALIGNMENT, CUDA,
 * UNSUPPORTED_DEVICE.
 */
cp_status cp_block_attn_fwd(const void* q, const void* k, const void* v, float* out, float* lse,
                            int B, int H, int Sq, int Skv, int D, float scale,
                            int64_t q_bstride, int64_t kv_bstride, int64_t o_bstride,
                            cp_dtype dt, void* stream);

/*
 * In-place fp32 LSE merge of a block partial into an accumulator (the step
 * that combines ring partials; "Paralelismo" API page, convert_to_fp32).
 *   out_acc, out_blk [B, S, H, D] float32 dense; lse_acc, lse_blk [B, H, S]
 *   m = max(lse_acc, lse_blk); lse = m + ln(e^(lse_acc-m) + e^(lse_blk-m))
 *   out_acc = e^(lse_acc-lse) out_acc + e^(lse_blk-lse) out_blk; lse_acc = lse
 * Rows where both LSEs are -inf become (0, -inf); merging with (0, -inf)
 * returns the other operand. out_blk/lse_blk must not alias the accumulator.
 * D must be a multiple of 4. Errors: INVALID_ARG, ALIGNMENT, CUDA.
 */
cp_status cp_lse_merge(float* out_acc, float* lse_acc, const float* out_blk, const float* lse_blk,
                       int B, int H, int S, int D, void* stream);

/*
 * Ulysses all-to-all #1, sequence-sharded -> head-sharded ("Atenção Ulysses":
 * the first all-to-all regroups so that each GPU holds every token of a subset
 * of heads). Head group g is heads [g*H/U, (g+1)*H/U); tokens are concatenated
 * in rank order:
 *   in  [U][B, S/U, H, D]   (rank u's sequence shard, ranks stacked)
 *   out [U][B, S, H/U, D]   (group g's heads, groups stacked)
 *   out[g][b, u*S/U + s, h, d] = in[u][b, s, g*H/U + h, d]
 * elem_bytes is the element size (2 for bf16, 4 for f32); a pure byte copy,
 * bit-exact. Errors: INVALID_ARG (H or S not divisible by U, U > H),
 * ALIGNMENT, CUDA.
 */
cp_status cp_ulysses_seq2head(const void* in, void* out, int U, int B, int S, int H, int D,
                              int elem_bytes, void* stream);

/*
 * Ulysses all-to-all #2, the inverse of cp_ulysses_seq2head ("a second
 * all-to-all regroups the results by token"):
 *   in  [U][B, S, H/U, D] -> out [U][B, S/U, H, D]
 *   out[u][b, s, g*H/U + h, d] = in[g][b, u*S/U + s, h, d]
 */
cp_status cp_ulysses_head2seq(const void* in, void* out, int U, int B, int S, int H, int D,
                              int elem_bytes, void* stream);

/*
 * Ulysses Anything regroups ("Paralelismo de contexto", section "Ulysses
 * Anything Attention": the sequence length and the head count need not be
 * divisible by ulysses_degree). Tokens and heads are both split into U
 * balanced shards (this library's reading; cp_ring_shard_table with
 * uneven_ok gives both tables): rank u holds tokens [soff_u, soff_u + S_u),
 * group g holds heads [hoff_g, hoff_g + H_g), the first S mod U ranks and the
 * first H mod U groups one longer.
 *
 * Layouts (both buffers hold B*S*H*D elements of elem_bytes bytes, dense):
 *   sequence-sharded: rank blocks back to back, block u = [B, S_u, H, D]
 *                     starting at element B*soff_u*H*D;
 *   head-grouped:     group blocks back to back, block g = [B, S, H_g, D]
 *                     starting at element B*S*hoff_g*D.
 *   seq2head: grp_g[b, soff_u + s, h, d] = rank_u[b, s, hoff_g + h, d]
 *   head2seq: rank_u[b, s, hoff_g + h, d] = grp_g[b, soff_u + s, h, d]
 * Bit copies (any element type of 1, 2, 4 or 8 bytes). Requires
 * 1 <= U <= H (INVALID_ARG otherwise); in and out must not overlap. With S
 * and H divisible by U the layouts and the result equal cp_ulysses_seq2head /
 * cp_ulysses_head2seq. Asynchronous on `stream`; launch errors -> CP_ERR_CUDA.
 */
cp_status cp_ulysses_anything_seq2head(const void* in, void* out, int U, int B, int S, int H, int D,
                                       int elem_bytes, void* stream);
cp_status cp_ulysses_anything_head2seq(const void* in, void* out, int U, int B, int S, int H, int D,
                                       int elem_bytes, void* stream);

/*
 * Host-only: the status cp_attention_fwd would return for these sizes and
 * flags before touching any pointer (the requirements table of the
 * "Paralelismo de contexto" page):
 *   ring needs S % ring_degree == 0 unless uneven_ok (Ring Anything);
 *   Ulysses needs S and H divisible by ulysses_degree unless uneven_ok
 *   (Ulysses Anything), and ulysses_degree <= H always;
 *   unified (both > 1) needs S % (ring_degree*ulysses_degree) == 0 and
 *   H % ulysses_degree == 0;
 *   uneven_ok selects an Anything variant and needs exactly one of
 *   ring_degree, ulysses_degree > 1 ("Ulysses Anything Attention": not with
 *   Unified, ring_degree 1; ContextParallelConfig.ring_anything:
 *   ulysses_degree 1).
 * Checks, in order: sizes/D/dtype/degrees >= 1 (INVALID_ARG), the uneven_ok
 * combination (UNSUPPORTED_COMBO), ulysses_degree > H (INVALID_ARG), then
 * divisibility (NOT_DIVISIBLE).
 */
cp_status cp_attention_validate(int B, int H, int S, int D, int ring_degree, int ulysses_degree,
                                int uneven_ok, cp_dtype dt);

/*
 * Host-only: the ring shard table ("Ring Anything Attention" pads each rank's
 * K/V to the longest local length; the split itself is this library's
 * reading): contiguous ranges, the first S mod n ranks get ceil(S/n) tokens
 * and the rest floor(S/n). Writes n offsets and n lengths (host arrays).
 * Returns NOT_DIVISIBLE when S % n != 0 and !uneven_ok.
 */
cp_status cp_ring_shard_table(int S, int n, int uneven_ok, int* offsets, int* lengths);

/* Host-only: bytes of device workspace cp_attention_fwd needs (0 if none). */
size_t cp_attention_workspace_size(int B, int H, int S, int D, int ring_degree, int ulysses_degree,
                                   cp_dtype dt, cp_lap_mode mode);

/* Host-only: how many kernels cp_attention_fwd launches for these arguments. */
int cp_attention_launch_count(int B, int H, int S, int D, int ring_degree, int ulysses_degree,
                              cp_dtype dt, cp_lap_mode mode);

/*
 * Context-parallel attention forward over the GLOBAL tensors, with the ranks
 * simulated on this GPU (the variants of the "Paralelismo de contexto" page,
 * configured as in ContextParallelConfig):
 *   q, k, v [B, S, H, D] (dt, dense); out [B, S, H, D] float32; lse [B, H, S]
 *   ulysses_degree == 1: ring lap over ring_degree ranks (ring_degree == 1 is
 *     plain attention); with uneven_ok the shards follow cp_ring_shard_table
 *     (Ring Anything);
 *   ulysses_degree > 1, ring_degree == 1: seq2head of q, k, v into the
 *     workspace, attention per head group over all S tokens, head2seq of out
 *     and lse; with uneven_ok (Ulysses Anything) S and H may be indivisible
 *     by ulysses_degree: the head groups are the balanced split of H, each
 *     stored with ceil(H/U) heads, and the kernels skip a short group's last
 *     (padding) head;
 *   both > 1 (unified): the same regroups, with a ring lap of ring_degree
 *     ranks over each head group's sequence (device (r, u) holds token chunk
 *     r*ulysses_degree + u; ring row r holds tokens [r*S/R, (r+1)*S/R)).
 * The result equals full attention. workspace must hold
 * cp_attention_workspace_size(...) bytes (may be NULL when that is 0).
 * Errors: those of cp_attention_validate, plus INVALID_ARG (null pointers),
 * ALIGNMENT, WORKSPACE, CUDA, UNSUPPORTED_DEVICE.
 */
cp_status cp_attention_fwd(const void* q, const void* k, const void* v, float* out, float* lse,
                           int B, int H, int S, int D, float scale,
                           int ring_degree, int ulysses_degree, int uneven_ok,
                           void* workspace, size_t ws_bytes, cp_dtype dt, cp_lap_mode mode,
                           void* stream);

/*
 * cp_attention_fwd with a key-padding mask: key_mask is a device array of B*S
 * bytes, row-major [B, S]; key j of batch entry b takes part in the softmax
 * of every query and head of that entry iff key_mask[b*S + j] != 0, and a
 * query row whose keys are all masked gets out = 0, lse = -inf. The pages
 * only say that Ring Anything takes no attention mask ("Paralelismo de
 * contexto", Ring Anything Attention: attn_mask must be None); the mask form
 * is this library's reading (a key-padding mask, as for padded text tokens).
 * key_mask == NULL is exactly cp_attention_fwd. Every ring block, Ulysses
 * head group and lap mode reads the mask at the global key position. Errors:
 * those of cp_attention_fwd, plus UNSUPPORTED_COMBO for a mask with
 * uneven_ok and ring_degree > 1 (Ring Anything).
 */
cp_status cp_attention_fwd_masked(const void* q, const void* k, const void* v, const uint8_t* key_mask,
                                  float* out, float* lse, int B, int H, int S, int D, float scale,
                                  int ring_degree, int ulysses_degree, int uneven_ok,
                                  void* workspace, size_t ws_bytes, cp_dtype dt, cp_lap_mode mode,
                                  void* stream);

/*
 * cp_attention_fwd over HOST buffers: q, k, v, out, lse as in
 * cp_attention_fwd but in host memory (page-locked for the copies to overlap;
 * pageable memory works, without overlap). dev_buffer (device, 256-byte
 * aligned, caller-owned) must hold cp_attention_host_buffer_size(...) bytes:
 * device copies of q, k, v, out, lse and the workspace of cp_attention_fwd.
 * With ulysses_degree == 1 and the fused lap (or ring_degree == 1), the
 * heads are split into head_chunks ranges (at most 16). The first and the
 * last range get about a third of an even share each and the middle ranges
 * the rest, largest first, each at most the heads whose work items fill one
 * wave of the device's SMs; where that does not fit, only the last range is
 * small and the others split the rest evenly (at FLUX ring 4, 24 heads: 5
 * chunks -> 2, 8, 8, 4, 2; 4 chunks -> 8, 7, 7, 2). Chunk j's
 * q, k, v are copied in on a library copy stream while chunk j-1 computes on
 * `stream`, and its out, lse are copied back on a second library copy stream
 * while later chunks compute, so the transfers overlap each other and the
 * attention. Heads are independent, so the result equals cp_attention_fwd's
 * on the same inputs bit for bit. Otherwise (Ulysses regroups, or a stepwise
 * ring lap) everything runs in order on `stream` (head_chunks is ignored).
 * All work is ordered after the work already queued on `stream`, and `stream`
 * resumes only after out and lse are in host memory; the call returns without
 * waiting. The host buffers must stay valid and unchanged until then. Calls on
 * one device serialise their enqueueing (the copy streams and their events
 * are the library's, one set per device). Errors: those of cp_attention_fwd,
 * INVALID_ARG for head_chunks < 1 or a null pointer, WORKSPACE when
 * dev_bytes is too small.
 */
size_t cp_attention_host_buffer_size(int B, int H, int S, int D, int ring_degree, int ulysses_degree,
                                     cp_dtype dt, cp_lap_mode mode);
cp_status cp_attention_fwd_host(const void* q, const void* k, const void* v, float* out, float* lse,
                                int B, int H, int S, int D, float scale,
                                int ring_degree, int ulysses_degree, int uneven_ok,
                                void* dev_buffer, size_t dev_bytes, cp_dtype dt, cp_lap_mode mode,
                                int head_chunks, void* stream);

/*
 * Synchronizes stream, then reads and clears the device error word on the
 * current device. Returns CP_OK if no kernel reported a problem since the
 * last call, CP_ERR_TIMEOUT if a kernel's bounded wait expired, CP_ERR_CUDA
 * if a kernel found its shared memory base misaligned (it then did no work)
 * or the read failed.
 */
cp_status cp_check_device_status(void* stream);

/*
 * Test hook for the bounded-wait machinery: launches one small kernel whose
 * threads wait on a shared-memory barrier that nothing completes, through the
 * same bounded wait the attention kernel uses, with a limit of timeout_us
 * microseconds (1..1000000). The kernel then records CP_ERR_TIMEOUT in the
 * device error word and returns; it never faults or hangs.
 */
cp_status cp_debug_bounded_wait_probe(int timeout_us, void* stream);

/*
 * cp_attention_fwd for callers that cannot allocate device memory. The pages
 * have no counterpart to this call; it exists for integrations where device
 * memory belongs to a host framework that gives a plugin no way to allocate,
 * or where the latency and implicit synchronisation of a device allocation in
 * the middle of a step are not acceptable. It takes the same arguments as
 * cp_attention_fwd minus the workspace, and uses instead a workspace of
 * CP_NO_ALLOC_WORKSPACE_BYTES (64 MiB) that the library holds as a static
 * device array: every GPU that loads the library keeps those 64 MiB until the
 * process exits. The first call on a device that needs scratch memory looks
 * the array's device address up (once per device, with that device current);
 * make that first call before any stream capture. A call that needs no
 * scratch (cp_attention_workspace_size(...) == 0, e.g. a plain ring with the
 * fused lap) never touches the array. No part of the array needs to start at zero
 * (every byte used is written before it is read), but all calls share it:
 * calls whose work overlaps on the GPU (other streams, other host threads)
 * race on it and must be serialised by the caller. The call allocates no
 * memory. Returns CP_ERR_WORKSPACE, launching nothing, when
 * cp_attention_workspace_size(...) for these arguments exceeds
 * CP_NO_ALLOC_WORKSPACE_BYTES (e.g. Ulysses at 4608 tokens x 24 heads x 128
 * needs ~141 MB); otherwise the errors of cp_attention_fwd.
 */
#define CP_NO_ALLOC_WORKSPACE_BYTES (64u * 1024u * 1024u)
cp_status cp_attention_fwd_no_alloc(const void* q, const void* k, const void* v, float* out, float* lse,
                                    int B, int H, int S, int D, float scale,
                                    int ring_degree, int ulysses_degree, int uneven_ok,
                                    cp_dtype dt, cp_lap_mode mode, void* stream);

/* ---------------------------------------------------------------------------
 * Backward (training): gradients of L = sum(out * dout) with respect to q, k
 * and v for the attention cp_attention_fwd computes. The context parallelism
 * page (variants table; Ring Attention, Ulysses Attention, Unified Attention
 * sections) lets the plain variants serve training and marks Ring Anything
 * as inference only; it gives no backward formulas. With
 * p_ij = exp(scale q_i.k_j - lse_i) and delta_i = sum_d dout_id out_id:
 *   dv_j = sum_i p_ij dout_i;  ds_ij = p_ij (dout_i.v_j - delta_i);
 *   dq_i = scale sum_j ds_ij k_j;  dk_j = scale sum_i ds_ij q_i.
 * The ring decomposition: each simulated rank's dq sums its lap's blocks in
 * lap order ((r - t) mod R), and each block's dk, dv sum the ranks in the
 * order the block visits them ((j + t) mod R), as dk, dv travel with K/V.
 * -------------------------------------------------------------------------*/

/* Bytes of device workspace cp_attention_bwd needs (256-byte aligned start):
 * delta [B,H,S] fp32, and with ulysses_degree > 1 the head-group copies of
 * q, k, v, dout, lse, delta and the head-group gradients. 0 for invalid sizes. */
size_t cp_attention_bwd_workspace_size(int B, int H, int S, int D, int ring_degree, int ulysses_degree,
                                       cp_dtype dt);

/* Kernel launches one cp_attention_bwd call makes: delta; then for bf16 the
 * padded lse / delta copy and one launch of the dk/dv and dq CTAs, for fp32 a
 * dq and a dk/dv launch; and the Ulysses regroups. 0 for empty or invalid
 * sizes. */
int cp_attention_bwd_launch_count(int B, int H, int S, int D, int ring_degree, int ulysses_degree, cp_dtype dt);

/* Backward of cp_attention_fwd (ring, Ulysses, unified or Ulysses Anything).
 *   q, k, v, dout : device [B, S, H, D] of dt (bf16 or fp32), dense;
 *   out, lse      : the forward's results, fp32 [B, S, H, D] and [B, H, S];
 *   dq, dk, dv    : device fp32 [B, S, H, D], written (not accumulated);
 *   workspace     : device, >= cp_attention_bwd_workspace_size(...) bytes,
 *                   256-byte aligned, owned by the caller.
 * bf16 runs on the tensor cores: bf16 operands (P and dS rounded to bf16
 * for their products), fp32 accumulation. fp32 runs on the CUDA cores in
 * fp32 throughout. Results are deterministic (no atomics). Asynchronous on
 * `stream`.
 * uneven_ok selects Ulysses Anything (ulysses_degree > 1, ring_degree == 1:
 * balanced ragged token shards and head groups, as in cp_attention_fwd).
 * Errors (returned before any launch): the checks of cp_attention_validate;
 * uneven_ok != 0 with ring_degree > 1 -> CP_ERR_UNSUPPORTED_COMBO (Ring
 * Anything is inference only); a null pointer or non-finite scale ->
 * CP_ERR_INVALID_ARG; a pointer not 16-byte aligned -> CP_ERR_ALIGNMENT;
 * workspace missing or short -> CP_ERR_WORKSPACE; launch failure ->
 * CP_ERR_CUDA. B == 0 or S == 0 returns CP_OK without launching. */
cp_status cp_attention_bwd(const void* q, const void* k, const void* v, const float* out, const void* dout,
                           const float* lse, float* dq, float* dk, float* dv, int B, int H, int S, int D,
                           float scale, int ring_degree, int ulysses_degree, int uneven_ok, void* workspace,
                           size_t ws_bytes, cp_dtype dt, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CP_ATTN_H_ */
