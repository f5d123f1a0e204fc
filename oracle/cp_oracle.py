"""Plain float64 CPU oracle for context-parallel attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use this module. It shares no code with the CUDA library.

Sources. The diffusers documentation pages on context parallelism:
  [CP]  "Paralelismo de contexto" / "コンテキスト並列" (optimization/context_parallelism),
        sections Ring Attention, Ulysses Attention, Unified Attention,
        Ring Anything Attention, and the variant/requirements table at the top;
  [API] "Paralelismo" (api/parallel), ContextParallelConfig parameters
        ring_degree, ulysses_degree, convert_to_fp32, ring_anything, mesh.
The pages never write out the attention or merge formulas; where they are
silent the plainest reading is taken and named below (readings R1..R9).

Layouts: q, k, v, out are [B, S, H, D] (D fastest); lse is [B, H, S], natural
log (R1, R2). Inputs may be any float dtype; they are upcast to float64 first,
so the oracle sees exactly the values the GPU sees.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


class NotDivisibleError(ValueError):
    """A length is not divisible by a degree that the variant requires to divide it."""


class UnsupportedComboError(ValueError):
    """A flag combination the requirements table rules out."""


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor: go through float32 (exact for bf16/f32)
        x = x.detach().to("cpu").float().numpy()
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# Block attention: the per-step computation of a ring lap.
# [API] ring_degree: "each device computes attention between its local Q and
# the KV blocks passed around the ring"; [API] convert_to_fp32: the step
# returns an output and an LSE (kept in fp32 for the merge).
# Reading R1: LSE is the natural-log log-sum-exp of the *scaled* logits.
# Reading R3: non-causal, no mask, no dropout ([CP] Ring Anything note:
# inference only, attn_mask must be None).
# ---------------------------------------------------------------------------
def attention(q, k, v, scale: float, row_chunk: int = 1024, key_mask=None):
    """Softmax attention of q against one K/V block, returning (out, lse).

    For each batch b, head h and query row i:
        s_ij   = scale * sum_d q[b,i,h,d] * k[b,j,h,d]
        m_i    = max_j s_ij
        w_ij   = exp(s_ij - m_i),   l_i = sum_j w_ij
        out    = sum_j w_ij v[b,j,h,:] / l_i
        lse    = m_i + ln(l_i)
    An empty block (Skv = 0) gives out = 0 and lse = -inf (reading R6), the
    identity element of ``lse_merge``.

    key_mask: None, or a boolean [B, Skv] array; keys where it is False take
    no part (reading R17: a key-padding mask, the attn_mask the pages rule
    out only for Ring Anything). Here they are simply left out of the sums;
    a batch entry with no key left gets out = 0, lse = -inf (as R6).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    assert k.shape == (B, Skv, H, D) and v.shape == (B, Skv, H, D)
    out = np.zeros((B, Sq, H, D), dtype=np.float64)
    lse = np.full((B, H, Sq), NEG_INF, dtype=np.float64)
    if Skv == 0 or Sq == 0:
        return out, lse
    if key_mask is not None:
        key_mask = np.asarray(key_mask, dtype=bool)
        assert key_mask.shape == (B, Skv)
    for b in range(B):
        keep = slice(None) if key_mask is None else np.nonzero(key_mask[b])[0]
        if key_mask is not None and len(keep) == 0:
            continue
        for h in range(H):
            kt = k[b, keep, h, :].T
            vb = v[b, keep, h, :]
            for i0 in range(0, Sq, row_chunk):
                i1 = min(Sq, i0 + row_chunk)
                s = scale * (q[b, i0:i1, h, :] @ kt)
                m = s.max(axis=1, keepdims=True)
                w = np.exp(s - m)
                l = w.sum(axis=1, keepdims=True)
                out[b, i0:i1, h, :] = (w @ vb) / l
                lse[b, h, i0:i1] = (m + np.log(l))[:, 0]
    return out, lse


def attention_rows(q, k, v, scale: float, rows, key_mask=None):
    """``attention`` for selected query rows only (rows are independent)."""
    q = _f64(q)
    return attention(q[:, np.asarray(rows)], k, v, scale, key_mask=key_mask)


# ---------------------------------------------------------------------------
# LSE merge of two (out, lse) partials.
# [API] convert_to_fp32 ("output and LSE in float32 for the numerical
# stability of ring attention") implies each step yields (out, lse) and the
# steps are combined through the LSE. Reading R4: the merge is the exact
# recombination of two softmax-normalised partials over disjoint key sets:
#     lse = m + ln(e^{lse_a - m} + e^{lse_b - m}),  m = max(lse_a, lse_b)
#     out = e^{lse_a - lse} out_a + e^{lse_b - lse} out_b
# with both-empty rows (m = -inf) giving (0, -inf).
# ---------------------------------------------------------------------------
def lse_merge(out_a, lse_a, out_b, lse_b):
    out_a, lse_a, out_b, lse_b = _f64(out_a), _f64(lse_a), _f64(out_b), _f64(lse_b)
    m = np.maximum(lse_a, lse_b)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    with np.errstate(invalid="ignore"):
        tot = np.exp(lse_a - m_safe) + np.exp(lse_b - m_safe)
        lse = np.where(empty, NEG_INF, m_safe + np.log(np.where(empty, 1.0, tot)))
        lse_safe = np.where(empty, 0.0, lse)
        wa = np.where(empty, 0.0, np.exp(lse_a - lse_safe))
        wb = np.where(empty, 0.0, np.exp(lse_b - lse_safe))
    # weights are per (b, h, s); out rows are (b, s, h, :)
    wa_o = np.transpose(wa, (0, 2, 1))[..., None]
    wb_o = np.transpose(wb, (0, 2, 1))[..., None]
    out = wa_o * out_a + wb_o * out_b
    return out, lse


# ---------------------------------------------------------------------------
# Shard table ([CP] requirements table; Ring Anything section).
# Plain ring needs S % ring_degree == 0. Ring Anything pads each rank's K/V
# to the longest local length and slices each block back to its true length;
# the pages do not say how S is split. Reading R5: balanced split, the first
# S mod N shards get ceil(S/N) tokens and the rest floor(S/N).
# ---------------------------------------------------------------------------
def ring_shard_table(S: int, n: int, uneven_ok: bool):
    """Contiguous token ranges [(offset, length)] of the n ring ranks."""
    if n < 1 or S < 0:
        raise ValueError("ring degree must be >= 1 and S >= 0")
    base, extra = divmod(S, n)
    if extra and not uneven_ok:
        raise NotDivisibleError(f"sequence length {S} is not divisible by ring_degree {n}")
    table, off = [], 0
    for r in range(n):
        ln = base + (1 if r < extra else 0)
        table.append((off, ln))
        off += ln
    return table


# ---------------------------------------------------------------------------
# Ring lap ([CP] Ring Attention: K/V blocks pass around a ring; each GPU
# attends to the block it holds, then passes it on; after a full lap every
# GPU has seen every token's K/V). Reading R7: at step t rank r holds the
# block of rank (r - t) mod N (it receives from its predecessor, own block
# first). The accumulator starts as the t = 0 partial.
# ---------------------------------------------------------------------------
def _ring_lap_rows(q_r, k, v, scale, table, r, key_mask=None):
    n = len(table)
    acc = None
    for t in range(n):
        j = (r - t) % n
        off, ln = table[j]
        km = None if key_mask is None else key_mask[:, off:off + ln]
        part = attention(q_r, k[:, off:off + ln], v[:, off:off + ln], scale, key_mask=km)
        acc = part if acc is None else lse_merge(acc[0], acc[1], part[0], part[1])
    return acc


def ring_attention(q, k, v, scale: float, ring_degree: int, uneven_ok: bool = False, key_mask=None):
    """Simulated ring lap over ``ring_degree`` ranks; returns global (out, lse).
    A key mask travels with its K/V block (each block's slice of it)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, H, D = q.shape
    table = ring_shard_table(S, ring_degree, uneven_ok)
    out = np.zeros((B, S, H, D))
    lse = np.full((B, H, S), NEG_INF)
    for r, (off, ln) in enumerate(table):
        o_r, l_r = _ring_lap_rows(q[:, off:off + ln], k, v, scale, table, r, key_mask)
        out[:, off:off + ln] = o_r
        lse[:, :, off:off + ln] = l_r
    return out, lse


# ---------------------------------------------------------------------------
# Ulysses regroups ([CP] Ulysses Attention: the first all-to-all regroups so
# that each GPU holds every token for a subset of heads; the second regroups
# the results back by token). Reading R8: contiguous head groups
# g*H/U .. (g+1)*H/U - 1; tokens concatenated in rank order.
#   seq2head: out_g[b, u*S/U + s, h, d] = in_u[b, s, g*H/U + h, d]
#   head2seq: out_u[b, s, g*H/U + h, d] = in_g[b, u*S/U + s, h, d]
# Written as explicit index loops (slabs of one head), not as a reshape, so
# that a reshape/transpose formulation can check it independently.
# ---------------------------------------------------------------------------
def seq2head(x_shards):
    """[U][B, S/U, H, D] (sequence-sharded) -> [U][B, S, H/U, D] (head-sharded)."""
    x = np.asarray(x_shards)
    U, B, Sl, H, D = x.shape
    if H % U:
        raise NotDivisibleError(f"heads {H} not divisible by ulysses_degree {U}")
    Hg = H // U
    out = np.empty((U, B, Sl * U, Hg, D), dtype=x.dtype)
    for g in range(U):
        for u in range(U):
            for h in range(Hg):
                out[g, :, u * Sl:(u + 1) * Sl, h, :] = x[u, :, :, g * Hg + h, :]
    return out


def head2seq(x_groups):
    """[U][B, S, H/U, D] (head-sharded) -> [U][B, S/U, H, D] (sequence-sharded)."""
    x = np.asarray(x_groups)
    U, B, S, Hg, D = x.shape
    if S % U:
        raise NotDivisibleError(f"sequence {S} not divisible by ulysses_degree {U}")
    Sl = S // U
    out = np.empty((U, B, Sl, Hg * U, D), dtype=x.dtype)
    for u in range(U):
        for g in range(U):
            for h in range(Hg):
                out[u, :, :, g * Hg + h, :] = x[g, :, u * Sl:(u + 1) * Sl, h, :]
    return out


def head2seq_lse(lse_groups):
    """[U][B, H/U, S] per-group LSE -> [B, H, S]: lse[b, g*H/U + h, s] = lse_g[b, h, s]."""
    x = np.asarray(lse_groups)
    U, B, Hg, S = x.shape
    out = np.empty((B, Hg * U, S), dtype=x.dtype)
    for g in range(U):
        for h in range(Hg):
            out[:, g * Hg + h, :] = x[g, :, h, :]
    return out


def _split_seq(x, n):
    B, S = x.shape[:2]
    Sl = S // n
    return np.stack([x[:, u * Sl:(u + 1) * Sl] for u in range(n)])


def ulysses_attention(q, k, v, scale: float, ulysses_degree: int, key_mask=None):
    """All-to-all, attention over all tokens of a head group, inverse all-to-all.
    A key mask indexes tokens, which every head group holds in full."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, H, D = q.shape
    U = ulysses_degree
    if S % U or H % U:
        raise NotDivisibleError(f"S={S} and H={H} must be divisible by ulysses_degree {U}")
    qh, kh, vh = (seq2head(_split_seq(t, U)) for t in (q, k, v))
    outs, lses = [], []
    for g in range(U):
        o, l = attention(qh[g], kh[g], vh[g], scale, key_mask=key_mask)
        outs.append(o)
        lses.append(l)
    out = np.concatenate(list(head2seq(np.stack(outs))), axis=1)
    lse = head2seq_lse(np.stack(lses))
    return out, lse


# ---------------------------------------------------------------------------
# Ulysses Anything ([CP] Ulysses Anything Attention: drops the requirement
# that the sequence length and the head count be divisible by
# ulysses_degree; it cannot be combined with Unified Attention, so
# ring_degree must be 1; [API] ulysses_anything). The pages do not say how
# the tokens and heads are split. Reading R15: both are split like R5 -
# balanced, the first S mod U ranks hold one token more and the first H mod U
# groups one head more. With uneven shards the regroup buffers are ragged, so
# they are lists of per-rank / per-group arrays:
#   anything_seq2head: out_g[b, soff_u + s, h, d] = in_u[b, s, hoff_g + h, d]
#   anything_head2seq: out_u[b, s, hoff_g + h, d] = in_g[b, soff_u + s, h, d]
# ---------------------------------------------------------------------------
def balanced_split(n: int, parts: int):
    """[(offset, length)] of the balanced split of n items into `parts` (R5, R15)."""
    return ring_shard_table(n, parts, True)


def anything_seq2head(x_ranks):
    """U arrays [B, S_u, H, D] (sequence shards) -> U arrays [B, S, H_g, D] (head groups)."""
    U = len(x_ranks)
    B, _, H, D = x_ranks[0].shape
    S = sum(x.shape[1] for x in x_ranks)
    seq, heads = balanced_split(S, U), balanced_split(H, U)
    if [x.shape[1] for x in x_ranks] != [ln for _, ln in seq]:
        raise ValueError("rank shards are not the balanced split of the sequence")
    out = []
    for g, (ho, hl) in enumerate(heads):
        y = np.empty((B, S, hl, D), dtype=x_ranks[0].dtype)
        for u, (so, sl) in enumerate(seq):
            for h in range(hl):
                y[:, so:so + sl, h, :] = x_ranks[u][:, :, ho + h, :]
        out.append(y)
    return out


def anything_head2seq(x_groups):
    """U arrays [B, S, H_g, D] (head groups) -> U arrays [B, S_u, H, D] (sequence shards)."""
    U = len(x_groups)
    B, S, _, D = x_groups[0].shape
    H = sum(x.shape[2] for x in x_groups)
    seq, heads = balanced_split(S, U), balanced_split(H, U)
    if [x.shape[2] for x in x_groups] != [ln for _, ln in heads]:
        raise ValueError("head groups are not the balanced split of the heads")
    out = []
    for u, (so, sl) in enumerate(seq):
        y = np.empty((B, sl, H, D), dtype=x_groups[0].dtype)
        for g, (ho, hl) in enumerate(heads):
            for h in range(hl):
                y[:, :, ho + h, :] = x_groups[g][:, so:so + sl, h, :]
        out.append(y)
    return out


def anything_head2seq_lse(lse_groups):
    """U arrays [B, H_g, S] -> [B, H, S]: lse[b, hoff_g + h, s] = lse_g[b, h, s]."""
    B, _, S = lse_groups[0].shape
    H = sum(x.shape[1] for x in lse_groups)
    out = np.empty((B, H, S), dtype=lse_groups[0].dtype)
    for (ho, hl), x in zip(balanced_split(H, len(lse_groups)), lse_groups):
        for h in range(hl):
            out[:, ho + h, :] = x[:, h, :]
    return out


def ulysses_anything_attention(q, k, v, scale: float, ulysses_degree: int, key_mask=None):
    """Ulysses with balanced, possibly uneven token shards and head groups."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, H, D = q.shape
    U = ulysses_degree
    if U > H:
        raise ValueError(f"ulysses_degree {U} exceeds the number of heads {H}")
    seq = balanced_split(S, U)
    qh, kh, vh = (anything_seq2head([t[:, so:so + sl] for so, sl in seq]) for t in (q, k, v))
    outs, lses = [], []
    for g in range(U):
        o, l = attention(qh[g], kh[g], vh[g], scale, key_mask=key_mask)
        outs.append(o)
        lses.append(l)
    out = np.concatenate(anything_head2seq(outs), axis=1)
    lse = anything_head2seq_lse(lses)
    return out, lse


# ---------------------------------------------------------------------------
# Unified sequence parallelism ([CP] Unified Attention: an all-to-all
# redistributes heads and tokens, ring attention runs on the result, then the
# all-to-all is reversed; the devices form a 2D ulysses x ring grid with
# orthogonal groups). Reading R9: mesh dims ("ring", "ulysses") as in [API]
# mesh; device (r, u) holds token chunk r*U + u of S/(R*U) tokens; Ulysses
# group r is ring row r, which after its regroup holds tokens
# [r*S/R, (r+1)*S/R) for head group u.
# ---------------------------------------------------------------------------
def unified_attention(q, k, v, scale: float, ring_degree: int, ulysses_degree: int, key_mask=None):
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S, H, D = q.shape
    R, U = ring_degree, ulysses_degree
    if S % (R * U) or H % U:
        raise NotDivisibleError(f"S={S} must be divisible by {R * U} and H={H} by {U}")
    Sr = S // R
    # per ring row r: seq2head inside the Ulysses group -> [U][B, S/R, H/U, D]
    rows = []
    for r in range(R):
        blk = [t[:, r * Sr:(r + 1) * Sr] for t in (q, k, v)]
        rows.append([seq2head(_split_seq(t, U)) for t in blk])
    out = np.zeros((B, S, H, D))
    lse = np.zeros((B, H, S))
    for r in range(R):
        outs, lses = [], []
        for g in range(U):
            acc = None
            for t in range(R):
                j = (r - t) % R
                km = None if key_mask is None else key_mask[:, j * Sr:(j + 1) * Sr]
                part = attention(rows[r][0][g], rows[j][1][g], rows[j][2][g], scale, key_mask=km)
                acc = part if acc is None else lse_merge(acc[0], acc[1], part[0], part[1])
            outs.append(acc[0])
            lses.append(acc[1])
        out[:, r * Sr:(r + 1) * Sr] = np.concatenate(list(head2seq(np.stack(outs))), axis=1)
        lse[:, :, r * Sr:(r + 1) * Sr] = head2seq_lse(np.stack(lses))
    return out, lse


def cp_attention(q, k, v, scale: float, ring_degree: int = 1, ulysses_degree: int = 1,
                 uneven_ok: bool = False, key_mask=None):
    """Dispatch on the ContextParallelConfig degrees ([CP] variants table).

    Ring (ring_degree > 1), Ulysses (ulysses_degree > 1), Unified (both > 1).
    uneven_ok selects an Anything variant: Ring Anything (ring_degree > 1,
    ulysses_degree == 1) or Ulysses Anything (ulysses_degree > 1,
    ring_degree == 1); neither combines with the other degree.
    key_mask: optional boolean [B, S] key-padding mask (R17); Ring Anything
    takes none ([CP] Ring Anything Attention: attn_mask must be None).
    """
    q = _f64(q)
    B, S, H, D = q.shape
    R, U = ring_degree, ulysses_degree
    if R < 1 or U < 1:
        raise ValueError("degrees must be >= 1")
    if uneven_ok and (R > 1) == (U > 1):
        raise UnsupportedComboError("an Anything variant needs exactly one of ring_degree, ulysses_degree > 1")
    if uneven_ok and R > 1 and key_mask is not None:
        raise UnsupportedComboError("Ring Anything takes no attention mask")
    if key_mask is not None:
        key_mask = np.asarray(key_mask, dtype=bool)
    if U > H:
        raise ValueError(f"ulysses_degree {U} exceeds the number of heads {H}")
    if uneven_ok and U > 1:
        return ulysses_anything_attention(q, k, v, scale, U, key_mask)
    if U == 1:
        return ring_attention(q, k, v, scale, R, uneven_ok, key_mask)
    if R == 1:
        return ulysses_attention(q, k, v, scale, U, key_mask)
    return unified_attention(q, k, v, scale, R, U, key_mask)


# ---------------------------------------------------------------------------
# Backward (training). The [CP] variants table and its Ring Anything note mark
# Ring Anything as inference only; the other variants carry no such note, so
# they serve training too. The pages write no backward formulas. Reading R18:
# the gradients are the exact derivatives of L = sum(out * dout) with respect
# to q, k and v for the forward above, in the form that reuses the forward's
# lse. Per batch b and head h, with s_ij = scale * q_i . k_j:
#     p_ij    = exp(s_ij - lse_i)            (the softmax weights)
#     delta_i = sum_d dout_id * out_id      (= sum_j p_ij dp_ij)
#     dv_j    = sum_i p_ij dout_i
#     dp_ij   = dout_i . v_j
#     ds_ij   = p_ij (dp_ij - delta_i)
#     dq_i    = scale * sum_j ds_ij k_j
#     dk_j    = scale * sum_i ds_ij q_i
# In a ring lap the sums over j split over the K/V blocks and the sums over i
# over the query shards: at step t rank r adds block (r - t) mod N's share to
# its dq, and block j's dk and dv collect the shares of the ranks the block
# visits (j, j+1, ... mod N) and travel with it. In float64 the order of these
# additions does not matter.
# ---------------------------------------------------------------------------
def attention_delta(out, dout):
    """delta [B, H, S] = sum over d of out[b, s, h, d] * dout[b, s, h, d]."""
    out, dout = _f64(out), _f64(dout)
    return np.transpose(np.sum(out * dout, axis=3), (0, 2, 1))


def attention_bwd(q, k, v, dout, scale: float, lse, delta):
    """Gradient shares of one query shard against one K/V block.

    q, dout: [B, Sq, H, D]; k, v: [B, Skv, H, D]; lse, delta: [B, H, Sq], the
    global values of the shard's rows (after the whole lap). Returns
    (dq [B, Sq, H, D], dk [B, Skv, H, D], dv [B, Skv, H, D]). A row with
    lse = -inf (it saw no key) has p = 0 and contributes nothing.
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    lse, delta = _f64(lse), _f64(delta)
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    dq = np.zeros((B, Sq, H, D))
    dk = np.zeros((B, Skv, H, D))
    dv = np.zeros((B, Skv, H, D))
    if Sq == 0 or Skv == 0:
        return dq, dk, dv
    for b in range(B):
        for h in range(H):
            qb, kb, vb, gb = q[b, :, h, :], k[b, :, h, :], v[b, :, h, :], dout[b, :, h, :]
            s = scale * (qb @ kb.T)
            live = np.isfinite(lse[b, h])
            p = np.where(live[:, None], np.exp(s - np.where(live, lse[b, h], 0.0)[:, None]), 0.0)
            dv[b, :, h, :] = p.T @ gb
            dp = gb @ vb.T
            ds = p * (dp - delta[b, h][:, None])
            dq[b, :, h, :] = scale * (ds @ kb)
            dk[b, :, h, :] = scale * (ds.T @ qb)
    return dq, dk, dv


def ring_attention_bwd(q, k, v, dout, scale: float, ring_degree: int, out=None, lse=None):
    """Simulated backward ring lap over ``ring_degree`` even shards.

    out, lse: the forward's global results (computed here when omitted).
    Returns (dq, dk, dv), each [B, S, H, D].
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    if out is None:
        out, lse = ring_attention(q, k, v, scale, ring_degree)
    delta = attention_delta(out, dout)
    lse = _f64(lse)
    B, S, H, D = q.shape
    table = ring_shard_table(S, ring_degree, False)
    n = len(table)
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for r, (qo, ql) in enumerate(table):
        rows = slice(qo, qo + ql)
        for t in range(n):
            ko, kl = table[(r - t) % n]
            keys = slice(ko, ko + kl)
            gq, gk, gv = attention_bwd(q[:, rows], k[:, keys], v[:, keys], dout[:, rows], scale,
                                       lse[:, :, rows], delta[:, :, rows])
            dq[:, rows] += gq
            dk[:, keys] += gk
            dv[:, keys] += gv
    return dq, dk, dv


def ulysses_anything_attention_bwd(q, k, v, dout, scale: float, ulysses_degree: int, out, lse):
    """Backward of ``ulysses_anything_attention``: the ragged regroups of q, k,
    v, dout and out (R15), the one-block backward inside each head group with
    the group's slice of lse, and the inverse regroup of dq, dk and dv."""
    q, k, v, dout, out, lse = (_f64(t) for t in (q, k, v, dout, out, lse))
    B, S, H, D = q.shape
    U = ulysses_degree
    seq, heads = balanced_split(S, U), balanced_split(H, U)
    qh, kh, vh, gh, oh = (anything_seq2head([t[:, so:so + sl] for so, sl in seq]) for t in (q, k, v, dout, out))
    grads = [[], [], []]
    for g, (ho, hl) in enumerate(heads):
        res = attention_bwd(qh[g], kh[g], vh[g], gh[g], scale, lse[:, ho:ho + hl, :], attention_delta(oh[g], gh[g]))
        for i in range(3):
            grads[i].append(res[i])
    return tuple(np.concatenate(anything_head2seq(gr), axis=1) for gr in grads)


def cp_attention_bwd(q, k, v, dout, scale: float, ring_degree: int = 1, ulysses_degree: int = 1,
                     uneven_ok: bool = False, out=None, lse=None):
    """Backward of ``cp_attention`` for the training variants (R18).

    Ring: the backward lap above. Ulysses / Unified: the forward's all-to-all
    regroups of q, k, v, dout, out and lse (lse head slices), the ring
    backward inside each head group (ring degree 1 for plain Ulysses), and the
    inverse regroup of dq, dk and dv. Ulysses Anything: the same over ragged
    token shards and head groups (R15). Ring Anything raises
    UnsupportedComboError: it is inference only ([CP] variants table and the
    note closing its section; reading R19).
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, S, H, D = q.shape
    R, U = ring_degree, ulysses_degree
    if R < 1 or U < 1:
        raise ValueError("degrees must be >= 1")
    if uneven_ok and (R > 1) == (U > 1):
        raise UnsupportedComboError("an Anything variant needs exactly one of ring_degree, ulysses_degree > 1")
    if uneven_ok and R > 1:
        raise UnsupportedComboError("Ring Anything is inference only")
    if U > H:
        raise ValueError(f"ulysses_degree {U} exceeds the number of heads {H}")
    if uneven_ok:
        if out is None:
            out, lse = ulysses_anything_attention(q, k, v, scale, U)
        return ulysses_anything_attention_bwd(q, k, v, dout, scale, U, out, lse)
    if S % R:
        raise NotDivisibleError(f"sequence length {S} is not divisible by ring_degree {R}")
    if out is None:
        out, lse = cp_attention(q, k, v, scale, R, U)
    out, lse = _f64(out), _f64(lse)
    if U == 1:
        return ring_attention_bwd(q, k, v, dout, scale, R, out, lse)
    if S % (R * U) or H % U:
        raise NotDivisibleError(f"S={S} must be divisible by {R * U} and H={H} by {U}")
    # head group g holds every token of heads [g*H/U, (g+1)*H/U); within a ring
    # row the seq2head regroup keeps token order, so group g's tokens are in
    # global order and its ring shards are the contiguous S/R ranges
    Hg = H // U
    grads = [np.zeros((U, B, S, Hg, D)) for _ in range(3)]
    groups = [seq2head(_split_seq(t, U)) for t in (q, k, v, dout, out)]
    for g in range(U):
        lse_g = lse[:, g * Hg:(g + 1) * Hg, :]
        res = ring_attention_bwd(groups[0][g], groups[1][g], groups[2][g], groups[3][g], scale, R,
                                 groups[4][g], lse_g)
        for i in range(3):
            grads[i][g] = res[i]
    return tuple(np.concatenate(list(head2seq(gr)), axis=1) for gr in grads)
