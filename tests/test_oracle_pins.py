"""Pins of the float64 oracle against things other than itself (CPU only).

Each pin is one of: brute force with a different formulation, a closed form,
an invariant of softmax attention, a library routine (scipy/numpy) on a
special case, or a value fixed by the pages (tests/golden). The last group
plants mistakes into copies of the oracle and checks that some pin fails.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import cp_oracle as co

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, scale=1.0):
    return scale * np.random.default_rng(seed).standard_normal(shape)


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------
def brute_attention(q, k, v, scale):
    """Scalar loops, no max shift: p_j = e^{s_j} / sum_k e^{s_k}, lse = ln sum e^{s}."""
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    out = np.zeros((B, Sq, H, D))
    lse = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            for i in range(Sq):
                s = [scale * math.fsum(q[b, i, h, d] * k[b, j, h, d] for d in range(D))
                     for j in range(Skv)]
                e = [math.exp(x) for x in s]
                z = math.fsum(e)
                lse[b, h, i] = math.log(z)
                for d in range(D):
                    out[b, i, h, d] = math.fsum(e[j] * v[b, j, h, d] for j in range(Skv)) / z
    return out, lse


@pytest.mark.parametrize("B,Sq,Skv,H,D,seed", [(1, 3, 5, 1, 2, 0), (2, 4, 7, 2, 3, 1),
                                                 (1, 8, 1, 2, 4, 2), (2, 1, 8, 3, 4, 3)])
def test_attention_matches_brute_force(B, Sq, Skv, H, D, seed):
    q, k, v = rnd((B, Sq, H, D), seed), rnd((B, Skv, H, D), seed + 10), rnd((B, Skv, H, D), seed + 20)
    scale = 0.7
    o, l = oracle.attention(q, k, v, scale)
    ob, lb = brute_attention(q, k, v, scale)
    assert np.max(np.abs(o - ob)) <= 1e-13
    assert np.max(np.abs(l - lb)) <= 1e-13


def test_attention_matches_scipy_softmax_logsumexp():
    q, k, v = rnd((2, 9, 3, 16), 4), rnd((2, 33, 3, 16), 5), rnd((2, 33, 3, 16), 6)
    scale = 0.25
    o, l = oracle.attention(q, k, v, scale)
    for b in range(2):
        for h in range(3):
            s = scale * np.einsum("id,jd->ij", q[b, :, h], k[b, :, h])
            np.testing.assert_allclose(l[b, h], scipy.special.logsumexp(s, axis=1), rtol=0, atol=1e-12)
            p = scipy.special.softmax(s, axis=1)
            np.testing.assert_allclose(o[b, :, h], p @ v[b, :, h], rtol=0, atol=1e-12)


def test_rows_sum_to_one():
    q, k = rnd((1, 17, 2, 8), 7, 3.0), rnd((1, 40, 2, 8), 8, 3.0)
    v = np.ones((1, 40, 2, 8))
    o, _ = oracle.attention(q, k, v, 0.5)
    assert np.max(np.abs(o - 1.0)) <= 1e-14


def test_constant_keys_give_mean_of_v():
    B, Sq, Skv, H, D = 1, 5, 11, 2, 4
    q, v = rnd((B, Sq, H, D), 9), rnd((B, Skv, H, D), 10)
    c = rnd((H, D), 11)
    k = np.broadcast_to(c[None, None], (B, Skv, H, D)).copy()
    scale = 0.6
    o, l = oracle.attention(q, k, v, scale)
    mean_v = v.mean(axis=1, keepdims=True)
    np.testing.assert_allclose(o, np.broadcast_to(mean_v, o.shape), rtol=0, atol=1e-14)
    expect_lse = scale * np.einsum("bihd,hd->bhi", q, c) + math.log(Skv)
    np.testing.assert_allclose(l, expect_lse, rtol=0, atol=1e-13)


def test_zero_query_gives_mean_and_log_count():
    q = np.zeros((1, 3, 2, 4))
    k, v = rnd((1, 13, 2, 4), 12), rnd((1, 13, 2, 4), 13)
    o, l = oracle.attention(q, k, v, 1.0)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=1, keepdims=True), o.shape), atol=1e-14, rtol=0)
    np.testing.assert_allclose(l, math.log(13), atol=1e-14, rtol=0)


def test_single_key():
    q, k, v = rnd((2, 6, 2, 4), 14), rnd((2, 1, 2, 4), 15), rnd((2, 1, 2, 4), 16)
    o, l = oracle.attention(q, k, v, 0.3)
    np.testing.assert_array_equal(o, np.broadcast_to(v, o.shape))
    np.testing.assert_allclose(l, 0.3 * np.einsum("bihd,bhd->bhi", q, k[:, 0]), atol=1e-14, rtol=0)


def test_two_keys_closed_form():
    q, k, v = rnd((1, 4, 1, 3), 17), rnd((1, 2, 1, 3), 18), rnd((1, 2, 1, 3), 19)
    scale = 0.9
    o, l = oracle.attention(q, k, v, scale)
    s0 = scale * q[0, :, 0] @ k[0, 0, 0]
    s1 = scale * q[0, :, 0] @ k[0, 1, 0]
    sig = 1.0 / (1.0 + np.exp(-(s0 - s1)))  # logistic weight of key 0
    expect = sig[:, None] * v[0, 0, 0] + (1 - sig)[:, None] * v[0, 1, 0]
    np.testing.assert_allclose(o[0, :, 0], expect, atol=1e-14, rtol=0)
    np.testing.assert_allclose(l[0, 0], np.logaddexp(s0, s1), atol=1e-14, rtol=0)


def test_key_shift_invariance():
    q, k, v = rnd((1, 7, 2, 5), 20), rnd((1, 9, 2, 5), 21), rnd((1, 9, 2, 5), 22)
    delta = rnd((2, 5), 23)
    scale = 0.4
    o1, l1 = oracle.attention(q, k, v, scale)
    o2, l2 = oracle.attention(q, k + delta[None, None], v, scale)
    np.testing.assert_allclose(o2, o1, atol=1e-13, rtol=0)
    np.testing.assert_allclose(l2 - l1, scale * np.einsum("bihd,hd->bhi", q, delta), atol=1e-12, rtol=0)


def test_joint_kv_permutation_invariance():
    q, k, v = rnd((2, 5, 3, 4), 24), rnd((2, 12, 3, 4), 25), rnd((2, 12, 3, 4), 26)
    perm = np.random.default_rng(27).permutation(12)
    o1, l1 = oracle.attention(q, k, v, 0.8)
    o2, l2 = oracle.attention(q, k[:, perm], v[:, perm], 0.8)
    np.testing.assert_allclose(o2, o1, atol=1e-14, rtol=0)
    np.testing.assert_allclose(l2, l1, atol=1e-13, rtol=0)


def test_dominant_key():
    D = 4
    q = np.zeros((1, 1, 1, D)); q[0, 0, 0, 0] = 10.0
    k = rnd((1, 6, 1, D), 28, 0.1)
    k[0, 3, 0, 0] = 8.0          # logit 80 vs |others| < ~3: gap > 50
    v = rnd((1, 6, 1, D), 29)
    o, l = oracle.attention(q, k, v, 1.0)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 3, 0], atol=1e-20 + 1e-14, rtol=0)
    assert abs(l[0, 0, 0] - 80.0) < 1e-20 + 1e-12


def test_empty_block_is_merge_identity():
    q = rnd((1, 3, 2, 4), 30)
    o, l = oracle.attention(q, np.zeros((1, 0, 2, 4)), np.zeros((1, 0, 2, 4)), 1.0)
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_heads_and_batches_independent():
    q, k, v = rnd((2, 4, 3, 4), 31), rnd((2, 6, 3, 4), 32), rnd((2, 6, 3, 4), 33)
    o, l = oracle.attention(q, k, v, 0.5)
    for b in range(2):
        for h in range(3):
            ob, lb = oracle.attention(q[b:b + 1, :, h:h + 1], k[b:b + 1, :, h:h + 1], v[b:b + 1, :, h:h + 1], 0.5)
            np.testing.assert_array_equal(o[b:b + 1, :, h:h + 1], ob)
            np.testing.assert_array_equal(l[b:b + 1, h:h + 1], lb)


def test_row_sampling_matches_full():
    q, k, v = rnd((1, 20, 2, 4), 34), rnd((1, 15, 2, 4), 35), rnd((1, 15, 2, 4), 36)
    o, l = oracle.attention(q, k, v, 0.5)
    rows = [0, 7, 19]
    os_, ls_ = oracle.attention_rows(q, k, v, 0.5, rows)
    np.testing.assert_array_equal(os_, o[:, rows])
    np.testing.assert_array_equal(ls_, l[:, :, rows])


# ----------------------------------------------------------------------------
# merge
# ----------------------------------------------------------------------------
def merged_over_partition(q, k, v, scale, cuts):
    acc = None
    for a, b in zip(cuts[:-1], cuts[1:]):
        part = oracle.attention(q, k[:, a:b], v[:, a:b], scale)
        acc = part if acc is None else oracle.lse_merge(*acc, *part)
    return acc


@pytest.mark.parametrize("cuts", [[0, 8, 16, 24, 32], [0, 11, 12, 32], [0, 1, 2, 3, 32],
                                  [0, 0, 32], [0, 32, 32], [0, 5, 5, 20, 32]])
def test_merge_partition_invariance(cuts):
    q, k, v = rnd((2, 6, 2, 8), 40, 2.0), rnd((2, 32, 2, 8), 41), rnd((2, 32, 2, 8), 42)
    o, l = oracle.attention(q, k, v, 0.5)
    om, lm = merged_over_partition(q, k, v, 0.5, cuts)
    np.testing.assert_allclose(om, o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lm, l, atol=1e-12, rtol=0)


def test_merge_commutative_associative():
    parts = [(rnd((1, 5, 2, 3), 50 + i), 3.0 * rnd((1, 2, 5), 60 + i)) for i in range(3)]
    a, b, c = parts
    ab = oracle.lse_merge(*a, *b)
    ba = oracle.lse_merge(*b, *a)
    np.testing.assert_allclose(ab[0], ba[0], atol=1e-15, rtol=0)
    np.testing.assert_allclose(ab[1], ba[1], atol=1e-15, rtol=0)
    left = oracle.lse_merge(*ab, *c)
    right = oracle.lse_merge(*a, *oracle.lse_merge(*b, *c))
    np.testing.assert_allclose(left[0], right[0], atol=1e-14, rtol=0)
    np.testing.assert_allclose(left[1], right[1], atol=1e-14, rtol=0)


def test_merge_identity_and_both_empty_exact():
    o = rnd((1, 4, 2, 3), 70)
    l = rnd((1, 2, 4), 71)
    zero = np.zeros_like(o)
    ninf = np.full_like(l, -np.inf)
    for om, lm in (oracle.lse_merge(o, l, zero, ninf), oracle.lse_merge(zero, ninf, o, l)):
        np.testing.assert_array_equal(om, o)
        np.testing.assert_array_equal(lm, l)
    om, lm = oracle.lse_merge(zero, ninf, zero, ninf)
    assert np.all(om == 0) and np.all(np.isneginf(lm)) and not np.any(np.isnan(om))


def test_merge_closed_forms():
    o1, o2 = rnd((1, 3, 1, 2), 72), rnd((1, 3, 1, 2), 73)
    l = rnd((1, 1, 3), 74)
    om, lm = oracle.lse_merge(o1, l, o2, l)        # equal weights
    np.testing.assert_allclose(lm, l + math.log(2), atol=1e-15, rtol=0)
    np.testing.assert_allclose(om, 0.5 * (o1 + o2), atol=1e-15, rtol=0)
    om, lm = oracle.lse_merge(o1, l, o2, l + math.log(3))   # weights 1/4, 3/4
    np.testing.assert_allclose(om, 0.25 * o1 + 0.75 * o2, atol=1e-15, rtol=0)
    np.testing.assert_allclose(lm, l + math.log(4), atol=1e-14, rtol=0)


# ----------------------------------------------------------------------------
# shard table, ring lap, Ulysses, unified
# ----------------------------------------------------------------------------
def test_shard_table():
    assert oracle.ring_shard_table(4608, 4, False) == [(0, 1152), (1152, 1152), (2304, 1152), (3456, 1152)]
    assert oracle.ring_shard_table(4607, 3, True) == [(0, 1536), (1536, 1536), (3072, 1535)]
    assert oracle.ring_shard_table(256, 2, False) == [(0, 128), (128, 128)]
    with pytest.raises(oracle.NotDivisibleError):
        oracle.ring_shard_table(4607, 3, False)
    for S in range(0, 40):
        for n in range(1, 9):
            t = oracle.ring_shard_table(S, n, True)
            lens = [ln for _, ln in t]
            assert sum(lens) == S and max(lens) - min(lens) <= 1
            assert all(t[i][0] + t[i][1] == t[i + 1][0] for i in range(n - 1))
            assert lens == sorted(lens, reverse=True)


def test_golden_variant_requirements():
    spec = json.load(open(os.path.join(GOLDEN, "variant_requirements.json")))
    q = np.zeros((1, 1, 1, 1))
    for case in spec["cases"]:
        S, H = case["S"], case["H"]
        R, U, ev = case["ring_degree"], case["ulysses_degree"], case["uneven_ok"]
        # validate without running attention: the same checks cp_attention makes
        try:
            if R < 1 or U < 1:
                raise ValueError
            if ev and (R > 1) == (U > 1):
                raise oracle.UnsupportedComboError
            if U > H:
                got = "invalid_arg"
                raise StopIteration
            if U == 1:
                oracle.ring_shard_table(S, R, ev)
            elif not ev and (S % (R * U) or H % U):
                raise oracle.NotDivisibleError
            got = "ok"
        except StopIteration:
            pass
        except oracle.NotDivisibleError:
            got = "not_divisible"
        except oracle.UnsupportedComboError:
            got = "unsupported_combo"
        assert got == case["expect"], case["name"]
    del q


def test_golden_variant_requirements_via_cp_attention():
    """The same table through the oracle's dispatcher, on tiny shapes with the same divisibility."""
    spec = json.load(open(os.path.join(GOLDEN, "variant_requirements.json")))
    for case in spec["cases"]:
        S, H = case["S"], case["H"]
        R, U, ev = case["ring_degree"], case["ulysses_degree"], case["uneven_ok"]
        # shrink S and H but keep S mod 48 and H mod 24, which fix divisibility by every degree used
        s_small = 48 + S % 48
        h_small = 24 + H % 24 if U <= 24 else H
        q = rnd((1, s_small, h_small, 2), 1)
        try:
            oracle.cp_attention(q, q, q, 1.0, R, U, ev)
            got = "ok"
        except oracle.NotDivisibleError:
            got = "not_divisible"
        except oracle.UnsupportedComboError:
            got = "unsupported_combo"
        except ValueError:
            got = "invalid_arg"
        assert got == case["expect"], case["name"]


@pytest.mark.parametrize("S,R,ev", [(24, 2, False), (24, 3, False), (24, 4, False), (23, 3, True),
                                    (25, 4, True), (5, 4, True), (3, 4, True)])
def test_ring_equals_full_attention(S, R, ev):
    q, k, v = rnd((2, S, 2, 4), 80, 1.5), rnd((2, S, 2, 4), 81), rnd((2, S, 2, 4), 82)
    o, l = oracle.attention(q, k, v, 0.5)
    orr, lr = oracle.ring_attention(q, k, v, 0.5, R, ev)
    np.testing.assert_allclose(orr, o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lr, l, atol=1e-12, rtol=0)


def reshape_seq2head(x):
    U, B, Sl, H, D = x.shape
    return x.reshape(U, B, Sl, U, H // U, D).transpose(3, 1, 0, 2, 4, 5).reshape(U, B, U * Sl, H // U, D)


def test_seq2head_matches_reshape_and_round_trips():
    x = np.arange(4 * 2 * 3 * 8 * 2).reshape(4, 2, 3, 8, 2)
    y = oracle.seq2head(x)
    np.testing.assert_array_equal(y, reshape_seq2head(x))
    np.testing.assert_array_equal(oracle.head2seq(y), x)
    # U = 1 is the identity
    z = np.arange(1 * 2 * 5 * 3 * 2).reshape(1, 2, 5, 3, 2)
    np.testing.assert_array_equal(oracle.seq2head(z), z)
    np.testing.assert_array_equal(oracle.head2seq(z), z)
    # a few explicit elements of the definition
    U, Sl, Hg = 4, 3, 2
    for (g, b, s, h, d) in [(0, 0, 0, 0, 0), (3, 1, 11, 1, 1), (2, 0, 7, 0, 1)]:
        u, sl = divmod(s, Sl)
        assert y[g, b, s, h, d] == x[u, b, sl, g * Hg + h, d]


@pytest.mark.parametrize("U", [1, 2, 4])
def test_ulysses_equals_full_attention(U):
    q, k, v = rnd((2, 16, 8, 4), 90, 1.5), rnd((2, 16, 8, 4), 91), rnd((2, 16, 8, 4), 92)
    o, l = oracle.attention(q, k, v, 0.5)
    ou, lu = oracle.ulysses_attention(q, k, v, 0.5, U)
    np.testing.assert_allclose(ou, o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lu, l, atol=1e-12, rtol=0)


@pytest.mark.parametrize("R,U", [(2, 2), (2, 4), (4, 2), (3, 2)])
def test_unified_equals_full_attention(R, U):
    S = 24
    q, k, v = rnd((1, S, 4, 4), 93, 1.5), rnd((1, S, 4, 4), 94), rnd((1, S, 4, 4), 95)
    o, l = oracle.attention(q, k, v, 0.5)
    ou, lu = oracle.unified_attention(q, k, v, 0.5, R, U)
    np.testing.assert_allclose(ou, o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lu, l, atol=1e-12, rtol=0)
    oc, lc = oracle.cp_attention(q, k, v, 0.5, R, U, False)
    np.testing.assert_array_equal(oc, ou)
    np.testing.assert_array_equal(lc, lu)


# ----------------------------------------------------------------------------
# planted mistakes: each mutated copy of an oracle function must fail a pin
# ----------------------------------------------------------------------------
def _mut_attention(kind):
    def f(q, k, v, scale, row_chunk=1024):
        q, k, v = co._f64(q), co._f64(k), co._f64(v)
        B, Sq, H, D = q.shape
        out = np.zeros((B, Sq, H, D)); lse = np.zeros((B, H, Sq))
        for b in range(B):
            for h in range(H):
                hk = (h + 1) % H if kind == "wrong_head" else h
                kb = k[b, :, hk, :] if kind != "v_for_k" else v[b, :, h, :]
                s = (1.0 if kind == "no_scale" else scale) * (q[b, :, h, :] @ kb.T)
                m = s.max(axis=1, keepdims=True)
                w = np.exp(s - m)
                l = w.sum(axis=1, keepdims=True)
                vb = v[b, :, h, :] if kind != "k_for_v" else k[b, :, h, :]
                out[b, :, h, :] = (w @ vb) / (1.0 if kind == "no_norm" else l)
                lse[b, h, :] = (np.log(l) if kind == "lse_no_max" else m + np.log(l))[:, 0]
        return out, lse
    return f


@pytest.mark.parametrize("kind", ["no_scale", "v_for_k", "k_for_v", "no_norm", "lse_no_max", "wrong_head"])
def test_planted_attention_mistakes_are_caught(kind):
    q, k, v = rnd((1, 3, 2, 2), 100), rnd((1, 4, 2, 2), 101), rnd((1, 4, 2, 2), 102)
    o, l = _mut_attention(kind)(q, k, v, 0.7)
    ob, lb = brute_attention(q, k, v, 0.7)
    assert max(np.max(np.abs(o - ob)), np.max(np.abs(l - lb))) > 1e-6


@pytest.mark.parametrize("kind", ["sign", "no_log", "swap_weights", "max_not_min_guard"])
def test_planted_merge_mistakes_are_caught(kind, monkeypatch):
    def bad(out_a, lse_a, out_b, lse_b):
        m = np.maximum(lse_a, lse_b)
        tot = np.exp(lse_a - m) + np.exp(lse_b - m)
        lse = m + (tot if kind == "no_log" else np.log(tot))
        if kind == "max_not_min_guard":
            lse = np.minimum(lse_a, lse_b) + np.log(tot)
        sa = -1.0 if kind == "sign" else 1.0
        wa = np.exp(sa * (lse_a - lse)); wb = np.exp(lse_b - lse)
        if kind == "swap_weights":
            wa, wb = wb, wa
        return (np.transpose(wa, (0, 2, 1))[..., None] * out_a
                + np.transpose(wb, (0, 2, 1))[..., None] * out_b), lse
    monkeypatch.setattr(co, "lse_merge", bad)
    q, k, v = rnd((1, 4, 1, 4), 103, 2.0), rnd((1, 16, 1, 4), 104), rnd((1, 16, 1, 4), 105)
    o, l = co.attention(q, k, v, 0.5)
    om, lm = co.ring_attention(q, k, v, 0.5, 4)
    assert max(np.max(np.abs(om - o)), np.max(np.abs(lm - l))) > 1e-6


@pytest.mark.parametrize("kind", ["head_index", "token_index", "group_swap"])
def test_planted_permute_mistakes_are_caught(kind):
    x = np.arange(4 * 1 * 3 * 8 * 2).reshape(4, 1, 3, 8, 2)
    U, B, Sl, H, D = x.shape
    Hg = H // U
    y = np.empty((U, B, Sl * U, Hg, D), dtype=x.dtype)
    for g in range(U):
        for u in range(U):
            for h in range(Hg):
                src_h = h * U + g if kind == "head_index" else g * Hg + h
                dst = slice(u * Sl, (u + 1) * Sl) if kind != "token_index" else slice((U - 1 - u) * Sl, (U - u) * Sl)
                gg = (g + 1) % U if kind == "group_swap" else g
                y[gg, :, dst, h, :] = x[u, :, :, src_h, :]
    assert not np.array_equal(y, reshape_seq2head(x))


# ---------------------------------------------------------------------------
# Ulysses Anything: ragged regroups (reading R15: balanced token shards and
# head groups). The balanced split's closed form, offset(u) = u*floor(n/U) +
# min(u, n mod U), is computed here independently of the oracle's table.
# ---------------------------------------------------------------------------
def _bal_off(n, U, u):
    return u * (n // U) + min(u, n % U)


RAGGED = [(1, 37, 7, 3, 4), (2, 10, 5, 4, 3), (1, 9, 6, 4, 2), (3, 4, 3, 3, 1), (1, 13, 24, 5, 2)]


@pytest.mark.parametrize("B,S,H,U,D", RAGGED)
def test_anything_seq2head_elementwise(B, S, H, U, D):
    x = np.arange(B * S * H * D, dtype=np.int64).reshape(B, S, H, D)  # value = flat index
    ranks = [x[:, _bal_off(S, U, u):_bal_off(S, U, u + 1)] for u in range(U)]
    groups = co.anything_seq2head(ranks)
    for g in range(U):
        h0, h1 = _bal_off(H, U, g), _bal_off(H, U, g + 1)
        assert groups[g].shape == (B, S, h1 - h0, D)
        for b in range(B):
            for t in range(S):
                for h in range(h1 - h0):
                    for d in range(D):
                        assert groups[g][b, t, h, d] == ((b * S + t) * H + h0 + h) * D + d
    back = co.anything_head2seq(groups)
    for u in range(U):
        assert np.array_equal(back[u], ranks[u])


@pytest.mark.parametrize("U", [1, 2, 4])
def test_anything_regroups_reduce_to_plain_ulysses(U):
    x = rnd((U, 2, 3, 8, 2), 5)
    got = co.anything_seq2head(list(x))
    want = oracle.seq2head(x)
    assert all(np.array_equal(got[g], want[g]) for g in range(U))
    assert all(np.array_equal(a, b) for a, b in zip(co.anything_head2seq(got), oracle.head2seq(want)))


def test_anything_lse_regroup_elementwise():
    B, H, S, U = 2, 7, 5, 3
    lse = [np.arange(B * (_bal_off(H, U, g + 1) - _bal_off(H, U, g)) * S, dtype=np.float64).reshape(B, -1, S) + 1000 * g
           for g in range(U)]
    full = co.anything_head2seq_lse(lse)
    for g in range(U):
        h0, h1 = _bal_off(H, U, g), _bal_off(H, U, g + 1)
        assert np.array_equal(full[:, h0:h1, :], lse[g])


@pytest.mark.parametrize("B,S,H,U,D", RAGGED + [(1, 24, 8, 4, 3)])
def test_ulysses_anything_equals_full_attention(B, S, H, U, D):
    q, k, v = (rnd((B, S, H, D), i + S) for i in range(3))
    o, l = oracle.cp_attention(q, k, v, 0.4, 1, U, True)
    ro, rl = oracle.attention(q, k, v, 0.4)
    assert np.max(np.abs(o - ro)) <= 1e-12 and np.max(np.abs(l - rl)) <= 1e-12


@pytest.mark.parametrize("kind", ["floor_split", "head_groups_reversed", "ceil_split"])
def test_planted_anything_mistakes_are_caught(kind):
    B, S, H, U, D = 1, 10, 5, 4, 2
    x = np.arange(B * S * H * D).reshape(B, S, H, D)
    if kind == "floor_split":      # uneven shards cut at u*S//U instead of the balanced split
        cut = [u * S // U for u in range(U + 1)]
    elif kind == "ceil_split":     # ceil-chunking: the last shard takes the shortfall
        c = -(-S // U)
        cut = [min(S, u * c) for u in range(U + 1)]
    else:
        cut = [_bal_off(S, U, u) for u in range(U + 1)]
    hcut = [_bal_off(H, U, g) for g in range(U + 1)]
    if kind == "head_groups_reversed":
        hcut = [H - c for c in reversed(hcut)]
    wrong = [np.concatenate([x[:, cut[u]:cut[u + 1], hcut[g]:hcut[g + 1]] for u in range(U)], axis=1)
             for g in range(U)]
    right = co.anything_seq2head([x[:, _bal_off(S, U, u):_bal_off(S, U, u + 1)] for u in range(U)])
    assert any(w.shape != r.shape or not np.array_equal(w, r) for w, r in zip(wrong, right)) or \
        [cut[u + 1] - cut[u] for u in range(U)] != [_bal_off(S, U, u + 1) - _bal_off(S, U, u) for u in range(U)]


# ---------------------------------------------------------------------------
# Key-padding mask (reading R17): masked keys take no part in the softmax.
# ---------------------------------------------------------------------------
def _brute_masked(q, k, v, scale, km):
    """Scalar loops with math.fsum, masked keys skipped; no max shift."""
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    out = np.zeros((B, Sq, H, D))
    lse = np.full((B, H, Sq), -np.inf)
    for b in range(B):
        for h in range(H):
            for i in range(Sq):
                keys = [j for j in range(Skv) if km[b, j]]
                if not keys:
                    continue
                e = [math.exp(scale * math.fsum(q[b, i, h, d] * k[b, j, h, d] for d in range(D))) for j in keys]
                z = math.fsum(e)
                for d in range(D):
                    out[b, i, h, d] = math.fsum(e[t] * v[b, j, h, d] for t, j in enumerate(keys)) / z
                lse[b, h, i] = math.log(z)
    return out, lse


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_masked_attention_matches_brute_force(seed):
    B, Sq, Skv, H, D = 2, 3, 7, 2, 3
    q, k, v = (rnd((B, n, H, D), seed + 10 * i) for i, n in enumerate((Sq, Skv, Skv)))
    km = np.random.default_rng(seed).random((B, Skv)) < 0.6
    km[1, :] = False if seed == 2 else km[1, :]  # seed 2: a batch entry with every key masked
    o, l = oracle.attention(q, k, v, 0.7, key_mask=km)
    bo, bl = _brute_masked(q, k, v, 0.7, km)
    assert np.array_equal(np.isneginf(l), np.isneginf(bl))
    fin = np.isfinite(bl)
    assert np.max(np.abs(o - bo)) <= 1e-13 and np.max(np.abs(l[fin] - bl[fin])) <= 1e-13
    if seed == 2:
        assert np.all(o[1] == 0) and np.all(np.isneginf(l[1]))


def test_mask_all_true_is_no_mask_and_single_key_closed_form():
    q, k, v = (rnd((2, 5, 3, 4), i) for i in range(3))
    o0, l0 = oracle.attention(q, k, v, 0.5)
    o1, l1 = oracle.attention(q, k, v, 0.5, key_mask=np.ones((2, 5), bool))
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    km = np.zeros((2, 5), bool)
    km[:, 3] = True  # one key left: out = v_3, lse = its logit
    o, l = oracle.attention(q, k, v, 0.5, key_mask=km)
    assert np.allclose(o, np.broadcast_to(v[:, 3:4], o.shape), atol=1e-15)
    assert np.allclose(l, 0.5 * np.einsum("bihd,bhd->bhi", q, k[:, 3]), atol=1e-14)


@pytest.mark.parametrize("R,U,ev,S,H", [(4, 1, False, 24, 2), (1, 4, False, 24, 8), (2, 2, False, 24, 4),
                                        (1, 3, True, 23, 5), (3, 1, False, 24, 2)])
def test_masked_decompositions_equal_masked_attention(R, U, ev, S, H):
    q, k, v = (rnd((2, S, H, 3), 40 + i) for i in range(3))
    km = np.random.default_rng(S + R).random((2, S)) < 0.5
    km[0, : S // 2] = False  # whole ring blocks masked for entry 0
    o, l = oracle.cp_attention(q, k, v, 0.3, R, U, ev, key_mask=km)
    ro, rl = oracle.attention(q, k, v, 0.3, key_mask=km)
    assert np.array_equal(np.isneginf(l), np.isneginf(rl))
    fin = np.isfinite(rl)
    assert np.max(np.abs(o - ro)) <= 1e-12 and np.max(np.abs(l[fin] - rl[fin])) <= 1e-12


def test_mask_with_ring_anything_is_rejected():
    q = rnd((1, 23, 2, 2), 0)
    with pytest.raises(oracle.UnsupportedComboError):
        oracle.cp_attention(q, q, q, 1.0, 3, 1, True, key_mask=np.ones((1, 23), bool))


def test_planted_mask_on_queries_is_caught():
    q, k, v = (rnd((1, 6, 2, 3), 50 + i) for i in range(3))
    km = np.array([[True, False, True, True, False, True]])
    o, l = oracle.attention(q, k, v, 0.6, key_mask=km)
    # the mistake: drop the masked positions from the queries instead of the keys
    wrong = oracle.attention(q, k, v, 0.6)[0] * km[:, :, None, None]
    assert np.max(np.abs(wrong - o)) > 1e-3


# ----------------------------------------------------------------------------
# backward (reading R18): pinned to finite differences of the pinned forward,
# to torch autograd of a plain softmax attention, to invariants of the
# softmax Jacobian and to closed forms; then planted mistakes
# ----------------------------------------------------------------------------
def _loss(q, k, v, dout, scale):
    return float(np.sum(brute_attention(q, k, v, scale)[0] * dout))


@pytest.mark.parametrize("seed", [0, 1])
def test_bwd_matches_central_differences(seed):
    B, S, Skv, H, D, scale = 1, 3, 4, 2, 3, 0.6
    q, k, v = rnd((B, S, H, D), 200 + seed), rnd((B, Skv, H, D), 210 + seed), rnd((B, Skv, H, D), 220 + seed)
    dout = rnd((B, S, H, D), 230 + seed)
    out, lse = co.attention(q, k, v, scale)
    dq, dk, dv = co.attention_bwd(q, k, v, dout, scale, lse, co.attention_delta(out, dout))
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            keep = x[idx]
            x[idx] = keep + eps
            up = _loss(q, k, v, dout, scale)
            x[idx] = keep - eps
            dn = _loss(q, k, v, dout, scale)
            x[idx] = keep
            num[idx] = (up - dn) / (2 * eps)
        np.testing.assert_allclose(g, num, atol=1e-8, rtol=1e-6)


def test_bwd_matches_torch_autograd_float64():
    torch = pytest.importorskip("torch")
    B, S, H, D, scale = 2, 7, 3, 5, 0.4
    q, k, v, dout = (rnd((B, S, H, D), 240 + i, 1.5) for i in range(4))
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    s = scale * torch.einsum("bihd,bjhd->bhij", tq, tk)
    o = torch.einsum("bhij,bjhd->bihd", torch.softmax(s, dim=-1), tv)
    o.backward(torch.tensor(dout, dtype=torch.float64))
    dq, dk, dv = co.cp_attention_bwd(q, k, v, dout, scale)
    for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        np.testing.assert_allclose(mine, ref.numpy(), atol=1e-12, rtol=1e-10)


def test_bwd_softmax_invariants():
    # sum_j ds_ij = 0, so sum_j dk_j = 0; the weights sum to one per row, so
    # sum_j dv_j = sum_i dout_i; and dq is unchanged when every key moves by
    # the same vector (the logits of a row shift by one constant)
    B, S, H, D, scale = 2, 9, 2, 4, 0.7
    q, k, v, dout = (rnd((B, S, H, D), 250 + i) for i in range(4))
    dq, dk, dv = co.cp_attention_bwd(q, k, v, dout, scale)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=1), dout.sum(axis=1), atol=1e-12)
    shift = rnd((1, 1, H, D), 260)
    dq2, _, _ = co.cp_attention_bwd(q, k + shift, v, dout, scale)
    np.testing.assert_allclose(dq2, dq, atol=1e-12)


def test_bwd_closed_forms():
    # one key: out = v, so dv = sum of dout over the queries, dq = dk = 0
    q, k, v, dout = rnd((1, 5, 2, 3), 270), rnd((1, 1, 2, 3), 271), rnd((1, 1, 2, 3), 272), rnd((1, 5, 2, 3), 273)
    out, lse = co.attention(q, k, v, 0.5)
    dq, dk, dv = co.attention_bwd(q, k, v, dout, 0.5, lse, co.attention_delta(out, dout))
    np.testing.assert_allclose(dv[:, 0], dout.sum(axis=1), atol=1e-14)
    np.testing.assert_allclose(dq, 0.0, atol=1e-14)
    np.testing.assert_allclose(dk, 0.0, atol=1e-14)
    # q = 0: uniform weights 1/n, out = mean of v, so dv_j = sum_i dout_i / n and
    # dq_i = scale * sum_j (dout_i . (v_j - mean v)) k_j / n; dk = 0 (q = 0)
    n = 6
    q = np.zeros((1, 4, 1, 3)); k, v, dout = rnd((1, n, 1, 3), 274), rnd((1, n, 1, 3), 275), rnd((1, 4, 1, 3), 276)
    out, lse = co.attention(q, k, v, 0.9)
    dq, dk, dv = co.attention_bwd(q, k, v, dout, 0.9, lse, co.attention_delta(out, dout))
    np.testing.assert_allclose(dv[0, :, 0], np.tile(dout[0, :, 0].sum(axis=0) / n, (n, 1)), atol=1e-14)
    vc = v[0, :, 0] - v[0, :, 0].mean(axis=0)
    want = 0.9 * (dout[0, :, 0] @ vc.T) @ k[0, :, 0] / n
    np.testing.assert_allclose(dq[0, :, 0], want, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0, atol=1e-14)


@pytest.mark.parametrize("R,U,S,H", [(1, 1, 12, 4), (3, 1, 12, 4), (4, 1, 12, 2), (1, 2, 12, 4), (1, 4, 12, 4),
                                     (2, 2, 12, 4), (3, 2, 12, 2)])
def test_bwd_decompositions_equal_full_backward(R, U, S, H):
    B, D, scale = 2, 3, 0.8
    q, k, v, dout = (rnd((B, S, H, D), 280 + i, 1.3) for i in range(4))
    out, lse = co.attention(q, k, v, scale)
    full = co.attention_bwd(q, k, v, dout, scale, lse, co.attention_delta(out, dout))
    got = co.cp_attention_bwd(q, k, v, dout, scale, R, U)
    for a, b in zip(got, full):
        np.testing.assert_allclose(a, b, atol=1e-12, rtol=0)


def test_bwd_rejects_ring_anything_and_uneven():
    q = rnd((1, 7, 2, 2), 290)
    with pytest.raises(co.UnsupportedComboError):
        co.cp_attention_bwd(q, q, q, q, 0.5, 2, 1, True)     # Ring Anything: inference only
    with pytest.raises(co.UnsupportedComboError):
        co.cp_attention_bwd(q, q, q, q, 0.5, 2, 2, True)     # Anything with both degrees
    with pytest.raises(co.NotDivisibleError):
        co.cp_attention_bwd(q, q, q, q, 0.5, 2, 1, False)


@pytest.mark.parametrize("U,S,H", [(2, 7, 3), (4, 9, 5), (3, 2, 4), (5, 13, 5)])
def test_bwd_ulysses_anything_equals_full_backward(U, S, H):
    # ragged token shards and head groups (and a shard with no token when S < U)
    B, D, scale = 2, 3, 0.7
    q, k, v, dout = (rnd((B, S, H, D), 320 + i, 1.2) for i in range(4))
    out, lse = co.attention(q, k, v, scale)
    full = co.attention_bwd(q, k, v, dout, scale, lse, co.attention_delta(out, dout))
    got = co.cp_attention_bwd(q, k, v, dout, scale, 1, U, True)
    for a, b in zip(got, full):
        np.testing.assert_allclose(a, b, atol=1e-12, rtol=0)


def _mut_bwd(kind):
    def f(q, k, v, dout, scale, lse, delta):
        q, k, v, dout, lse, delta = (co._f64(x) for x in (q, k, v, dout, lse, delta))
        B, Sq, H, D = q.shape
        dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
        for b in range(B):
            for h in range(H):
                qb, kb, vb, gb = q[b, :, h, :], k[b, :, h, :], v[b, :, h, :], dout[b, :, h, :]
                s = scale * (qb @ kb.T)
                p = np.exp(s - lse[b, h][:, None])
                dv[b, :, h, :] = (p if kind == "dv_untransposed" else p.T) @ gb
                dp = gb @ (kb if kind == "k_for_v" else vb).T
                ds = p * (dp - (0.0 if kind == "no_delta" else delta[b, h][:, None]))
                if kind == "ds_sign":
                    ds = p * (delta[b, h][:, None] - dp)
                dq[b, :, h, :] = (1.0 if kind == "dq_no_scale" else scale) * (ds @ kb)
                dk[b, :, h, :] = scale * ((ds if kind == "dk_untransposed" else ds.T) @ qb)
        return dq, dk, dv
    return f


@pytest.mark.parametrize("kind", ["no_delta", "ds_sign", "dq_no_scale", "k_for_v", "dk_untransposed",
                                  "dv_untransposed"])
def test_planted_bwd_mistakes_are_caught(kind):
    # square blocks, so a transposed operand still has the right shape
    B, S, H, D, scale = 1, 4, 1, 4, 0.6
    q, k, v, dout = (rnd((B, S, H, D), 300 + i) for i in range(4))
    out, lse = co.attention(q, k, v, scale)
    got = _mut_bwd(kind)(q, k, v, dout, scale, lse, co.attention_delta(out, dout))
    eps = 1e-6
    worst = 0.0
    for x, g in zip((q, k, v), got):
        for idx in np.ndindex(*x.shape):
            keep = x[idx]
            x[idx] = keep + eps
            up = _loss(q, k, v, dout, scale)
            x[idx] = keep - eps
            dn = _loss(q, k, v, dout, scale)
            x[idx] = keep
            worst = max(worst, abs(g[idx] - (up - dn) / (2 * eps)))
    assert worst > 1e-4


def test_planted_bwd_lap_mistake_is_caught():
    # a lap whose blocks do not rotate (every rank sees its own block N times)
    real = co.ring_shard_table
    q, k, v, dout = (rnd((1, 8, 1, 2), 310 + i) for i in range(4))
    full = co.cp_attention_bwd(q, k, v, dout, 0.5)
    out, lse = co.attention(q, k, v, 0.5)
    delta = co.attention_delta(out, dout)
    table = real(8, 4, False)
    dq = np.zeros(q.shape)
    for r, (qo, ql) in enumerate(table):
        for t in range(4):
            ko, kl = table[r]  # the mistake: no rotation
            gq, _, _ = co.attention_bwd(q[:, qo:qo + ql], k[:, ko:ko + kl], v[:, ko:ko + kl], dout[:, qo:qo + ql], 0.5,
                                        lse[:, :, qo:qo + ql], delta[:, :, qo:qo + ql])
            dq[:, qo:qo + ql] += gq
    assert np.max(np.abs(dq - full[0])) > 1e-6


def test_planted_anything_bwd_lse_slice_mistake_is_caught():
    # a Ulysses Anything backward that hands every head group the first groups' lse rows
    B, S, H, D, U, scale = 1, 9, 5, 3, 4, 0.7
    q, k, v, dout = (rnd((B, S, H, D), 330 + i, 1.2) for i in range(4))
    out, lse = co.attention(q, k, v, scale)
    full = co.attention_bwd(q, k, v, dout, scale, lse, co.attention_delta(out, dout))
    seq, heads = co.balanced_split(S, U), co.balanced_split(H, U)
    qh, kh, vh, gh, oh = (co.anything_seq2head([t[:, so:so + sl] for so, sl in seq]) for t in (q, k, v, dout, out))
    dq = []
    for g, (ho, hl) in enumerate(heads):
        res = co.attention_bwd(qh[g], kh[g], vh[g], gh[g], scale, lse[:, 0:hl, :], co.attention_delta(oh[g], gh[g]))
        dq.append(res[0])
    bad = np.concatenate(co.anything_head2seq(dq), axis=1)
    assert np.max(np.abs(bad - full[0])) > 1e-6
