"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Tolerances (fixed by the benchmark spec for this path):
  * permutes: bit-exact;
  * merge (fp32 in, fp32 out): max abs error <= 1e-5;
  * attention with bf16 q/k/v, fp32 out/lse: max abs error <= 1e-2 and
    relative L2 error <= 5e-3, on out and on lse;
  * attention with fp32 q/k/v (CUDA-core path, fp32 arithmetic throughout):
    max abs <= 1e-4 and relative L2 <= 1e-5 (derived: ~S ulp-level roundings
    of unit-size values, far inside the bf16 bound).
"""
import numpy as np
import pytest
import torch

import oracle
from synth import WORKLOADS, make_merge_operands, make_qkv

pytestmark = pytest.mark.gpu

BF16_TOL = dict(max_abs=1e-2, rel_l2=5e-3)
F32_TOL = dict(max_abs=1e-4, rel_l2=1e-5)


@pytest.fixture(scope="session", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from context_attention_dits_gb300 import build
    build.build()
    import context_attention_dits_gb300 as cpa
    return cpa


def cpa():
    import context_attention_dits_gb300 as m
    return m


def rel_l2(a, b):
    fin = np.isfinite(b)
    a, b = a[fin], b[fin]
    den = np.sqrt(np.sum(b * b))
    return float(np.sqrt(np.sum((a - b) ** 2)) / max(den, 1e-300))


def assert_close(got, want, max_abs, rel_l2_tol, what):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, what
    # -inf must match exactly (empty rows); everything else finite
    inf_w = np.isneginf(want)
    assert np.array_equal(np.isneginf(got), inf_w), f"{what}: -inf pattern differs"
    assert np.all(np.isfinite(got[~inf_w])), f"{what}: non-finite values"
    err = np.abs(got[~inf_w] - want[~inf_w])
    mx = float(err.max()) if err.size else 0.0
    rl = rel_l2(got[~inf_w], want[~inf_w]) if err.size else 0.0
    assert mx <= max_abs, f"{what}: max abs {mx:.3e} > {max_abs}"
    assert rl <= rel_l2_tol, f"{what}: rel L2 {rl:.3e} > {rel_l2_tol}"
    return mx, rl


def check_attn(out, lse, ro, rl, tol, what):
    assert_close(out.cpu().numpy(), ro, tol["max_abs"], tol["rel_l2"], what + " out")
    assert_close(lse.cpu().numpy(), rl, tol["max_abs"], tol["rel_l2"], what + " lse")


def dev(*ts):
    return [t.cuda() for t in ts]


# ----------------------------------------------------------------------------
# Ulysses permutes: bit-exact
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("U,B,S,H,D,dtype", [
    (4, 1, 4608, 24, 128, torch.bfloat16),   # the FLUX Ulysses-4 regroup
    (4, 1, 4608, 24, 128, torch.float32),
    (4, 2, 64, 8, 64, torch.float32),
    (2, 3, 10, 6, 128, torch.bfloat16),
    (3, 1, 9, 6, 4, torch.float32),
    (1, 2, 7, 3, 64, torch.bfloat16),
    (6, 1, 12, 6, 3, torch.bfloat16),        # 6-byte segments: narrow-vector path
    (2, 1, 6, 128, 128, torch.float32),      # 32 KB segments: larger than a bulk-copy slot
    (4, 3, 520, 8, 64, torch.bfloat16),      # 256-byte segments, ragged last chunk
])
def test_permutes_bit_exact(U, B, S, H, D, dtype):
    g = torch.Generator().manual_seed(U * 1000 + S)
    x = torch.randn((U, B, S // U, H, D), generator=g).to(dtype)
    want = oracle.seq2head(x.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy())
    xd = x.cuda()
    y = torch.empty((U, B, S, H // U, D), dtype=dtype, device="cuda")
    cpa().cp_ulysses_seq2head(xd, y)
    iv = torch.int16 if dtype == torch.bfloat16 else torch.int32
    assert np.array_equal(y.cpu().view(iv).numpy(), want)
    back = torch.empty_like(xd)
    cpa().cp_ulysses_head2seq(y, back)
    assert torch.equal(back.cpu().view(iv), x.view(iv))
    want_back = oracle.head2seq(want)
    assert np.array_equal(back.cpu().view(iv).numpy(), want_back)


# ----------------------------------------------------------------------------
# Ulysses Anything regroups: bit-exact against the ragged oracle permute
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("U,B,S,H,D,dtype", [
    (4, 1, 4481, 24, 128, torch.bfloat16),  # FLUX 1008x1008: tokens 1121/1120/1120/1120
    (5, 1, 4608, 24, 128, torch.float32),   # heads 5/5/5/5/4 (3 KB and 2.5 KB rows)
    (3, 2, 10, 7, 64, torch.float32),
    (4, 1, 9, 5, 128, torch.bfloat16),
    (2, 3, 7, 3, 8, torch.float32),
    (3, 1, 2, 4, 16, torch.bfloat16),       # fewer tokens than ranks: an empty shard
    (6, 2, 1000, 12, 128, torch.bfloat16),  # 36 bulk copies with strided batch rows: two launches of <= 24
    (5, 2, 4481, 24, 128, torch.bfloat16),  # ragged heads and tokens, two batch entries
])
def test_anything_permutes_bit_exact(U, B, S, H, D, dtype):
    from oracle import cp_oracle as co
    iv = torch.int16 if dtype == torch.bfloat16 else torch.int32
    g = torch.Generator().manual_seed(U * 100 + S)
    x = torch.randn((B, S, H, D), generator=g).to(dtype)
    seq = co.balanced_split(S, U)
    ranks = [x[:, o:o + n].contiguous() for o, n in seq]
    flat_in = torch.cat([r.reshape(-1) for r in ranks])
    want_groups = co.anything_seq2head([r.view(iv).numpy() for r in ranks])
    want = np.concatenate([w.reshape(-1) for w in want_groups])
    dx = flat_in.cuda()
    y = torch.empty_like(dx)
    cpa().cp_ulysses_anything_seq2head(dx, y, U, B, S, H, D)
    assert np.array_equal(y.cpu().view(iv).numpy(), want)
    back = torch.empty_like(dx)
    cpa().cp_ulysses_anything_head2seq(y, back, U, B, S, H, D)
    assert torch.equal(back.cpu().view(iv), flat_in.view(iv))


# ----------------------------------------------------------------------------
# LSE merge
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("B,H,S,D,ninf", [(1, 24, 4608, 128, 0), (2, 3, 37, 64, 10), (1, 5, 9, 4, 6), (3, 1, 1, 8, 1)])
def test_lse_merge(B, H, S, D, ninf):
    oa, la, ob, lb = make_merge_operands(B, H, S, D, seed=7 + S, neg_inf_rows=ninf)
    ro, rl = oracle.lse_merge(oa.numpy(), la.numpy(), ob.numpy(), lb.numpy())
    doa, dla, dob, dlb = dev(oa, la, ob, lb)
    cpa().cp_lse_merge(doa, dla, dob, dlb)
    assert_close(doa.cpu().numpy(), ro, 1e-5, 1e-5, "merge out")
    assert_close(dla.cpu().numpy(), rl, 1e-5, 1e-5, "merge lse")


def test_lse_merge_identity_exact():
    oa, la, _, _ = make_merge_operands(1, 4, 33, 128, seed=3)
    ob = torch.zeros_like(oa)
    lb = torch.full_like(la, float("-inf"))
    doa, dla, dob, dlb = dev(oa, la, ob, lb)
    cpa().cp_lse_merge(doa, dla, dob, dlb)
    assert torch.equal(dla.cpu(), la)
    assert torch.equal(doa.cpu(), oa)


# ----------------------------------------------------------------------------
# block attention
# ----------------------------------------------------------------------------
BLOCK_CASES = [
    # B, H, Sq, Skv, D
    (2, 3, 129, 300, 128),
    (1, 2, 1, 1, 64),
    (1, 2, 127, 1535, 128),
    (1, 1, 256, 128, 64),
    (1, 4, 384, 257, 128),     # 3 query tiles: one CTA with two, one with one
    (2, 2, 520, 1000, 64),
    (1, 3, 1152, 1152, 128),   # one FLUX ring block
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,H,Sq,Skv,D", BLOCK_CASES)
def test_block_attention(B, H, Sq, Skv, D, dtype):
    if dtype == torch.float32 and Sq * Skv * H * B > 3_000_000:
        pytest.skip("fp32 CUDA-core path is only exercised on small blocks")
    q, _, _ = make_qkv(B, H, Sq, D, "bf16" if dtype == torch.bfloat16 else "f32", seed=Sq + Skv)
    _, k, v = make_qkv(B, H, Skv, D, "bf16" if dtype == torch.bfloat16 else "f32", seed=Sq * 7 + Skv)
    scale = D ** -0.5
    ro, rl = oracle.attention(q, k, v, scale)
    dq, dk, dv = dev(q, k, v)
    out = torch.empty((B, Sq, H, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    cpa().cp_block_attn_fwd(dq, dk, dv, out, lse, scale)
    check_attn(out, lse, ro, rl, BF16_TOL if dtype == torch.bfloat16 else F32_TOL, f"block {B},{H},{Sq},{Skv},{D}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_block_attention_strided_shard_views(dtype):
    """q, k, v as shard views of larger tensors (batch stride > S*H*D), as a ring step sees them."""
    B, H, S, D = 2, 2, 600, 128
    q, k, v = make_qkv(B, H, S, D, "bf16" if dtype == torch.bfloat16 else "f32", seed=11)
    dq, dk, dv = dev(q, k, v)
    qs, ks, vs = dq[:, 150:350], dk[:, 200:600], dv[:, 200:600]
    outbig = torch.full((B, S, H, D), 7.0, device="cuda")
    o = outbig[:, 150:350]
    lse = torch.empty((B, H, 200), device="cuda")
    cpa().cp_block_attn_fwd(qs, ks, vs, o, lse, 0.1)
    ro, rl = oracle.attention(q[:, 150:350], k[:, 200:600], v[:, 200:600], 0.1)
    check_attn(o, lse, ro, rl, BF16_TOL if dtype == torch.bfloat16 else F32_TOL, "strided")
    # rows outside the view untouched
    assert torch.all(outbig[:, :150] == 7.0) and torch.all(outbig[:, 350:] == 7.0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_block_attention_empty_kv(dtype):
    B, H, Sq, D = 1, 2, 130, 64
    q = torch.randn((B, Sq, H, D)).to(dtype).cuda()
    k = torch.empty((B, 0, H, D), dtype=dtype, device="cuda")
    out = torch.full((B, Sq, H, D), 3.0, device="cuda")
    lse = torch.zeros((B, H, Sq), device="cuda")
    cpa().cp_block_attn_fwd(q, k, k, out, lse, 0.125)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_block_attention_stress_logits():
    """q x 8 (logit std ~8): exercises the rescale path with large max jumps."""
    B, H, S, D = 1, 4, 1000, 128
    q, k, v = make_qkv(B, H, S, D, "bf16", seed=5, q_mult=8.0)
    ro, rl = oracle.attention(q, k, v, D ** -0.5)
    dq, dk, dv = dev(q, k, v)
    out = torch.empty((B, S, H, D), device="cuda")
    lse = torch.empty((B, H, S), device="cuda")
    cpa().cp_block_attn_fwd(dq, dk, dv, out, lse, D ** -0.5)
    check_attn(out, lse, ro, rl, BF16_TOL, "stress")


def test_block_attention_deterministic():
    B, H, S, D = 1, 6, 700, 128
    q, k, v = dev(*make_qkv(B, H, S, D, "bf16", seed=9))
    outs = []
    for _ in range(2):
        out = torch.empty((B, S, H, D), device="cuda")
        lse = torch.empty((B, H, S), device="cuda")
        cpa().cp_block_attn_fwd(q, k, v, out, lse, 0.09)
        outs.append((out, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


# ----------------------------------------------------------------------------
# the full context-parallel forward
# ----------------------------------------------------------------------------
def run_fwd(q, k, v, w, mode):
    B, S, H, D = q.shape
    out = torch.empty((B, S, H, D), device="cuda")
    lse = torch.empty((B, H, S), device="cuda")
    cpa().cp_attention_fwd(q, k, v, out, lse, w.scale, w.ring_degree, w.ulysses_degree, w.uneven_ok, mode=mode)
    torch.cuda.synchronize()
    return out, lse


_ORACLE_CACHE = {}


def workload_reference(name):
    """Inputs and oracle result of a named workload, computed once per session."""
    if name not in _ORACLE_CACHE:
        w = WORKLOADS[name]
        q, k, v = make_qkv(w.B, w.H, w.S, w.D, w.dtype, w.seed, w.q_mult)
        if name == "video_unified":
            rows = np.sort(np.random.default_rng(1234).choice(w.S, size=1024, replace=False))
            ref = (rows,) + oracle.attention_rows(q, k, v, w.scale, rows)
        else:
            ref = oracle.cp_attention(q, k, v, w.scale, w.ring_degree, w.ulysses_degree, w.uneven_ok)
        _ORACLE_CACHE[name] = ((q, k, v), ref)
    return _ORACLE_CACHE[name]


@pytest.mark.parametrize("name", ["tiny_ring", "flux_ring4", "flux_ulysses4", "flux_ulysses4_qx8", "ring_anything3",
                                  "flux1008_ulysses_anything4", "ulysses_anything5_heads"])
@pytest.mark.parametrize("mode", ["fused", "stepwise"])
def test_cp_attention_workloads_full_oracle(name, mode):
    w = WORKLOADS[name]
    (q, k, v), (ro, rl) = workload_reference(name)
    out, lse = run_fwd(*dev(q, k, v), w, mode)
    check_attn(out, lse, ro, rl, BF16_TOL if w.dtype == "bf16" else F32_TOL, f"{name}/{mode}")
    assert cpa().cp_check_device_status() == 0


@pytest.mark.parametrize("mode", ["fused", "stepwise"])
def test_cp_attention_video_unified_sampled_rows(mode):
    w = WORKLOADS["video_unified"]
    (q, k, v), (rows, ro, rl) = workload_reference("video_unified")
    out, lse = run_fwd(*dev(q, k, v), w, mode)
    check_attn(out[:, rows], lse[:, :, rows], ro, rl, BF16_TOL, f"video_unified/{mode} sampled")


@pytest.mark.parametrize("B,H,S,D,R,U,ev", [
    (2, 4, 300, 64, 3, 1, True),      # uneven shards 100/100/100 -> even; ragged tiles
    (1, 2, 301, 128, 4, 1, True),     # 76/75/75/75
    (1, 6, 96, 128, 2, 3, False),     # unified 2 x 3
    (2, 8, 256, 64, 1, 8, False),     # Ulysses 8, one head per group
    (1, 4, 129, 128, 1, 1, False),    # plain attention through the driver
    (1, 2, 3, 64, 4, 1, True),        # more ranks than tokens: one empty shard
    (1, 8, 520, 128, 4, 2, False),    # unified 4 x 2 with ragged tiles (65-token chunks)
    (2, 7, 300, 64, 1, 3, True),      # Ulysses Anything: heads 3/2/2, tokens 100 x 3
    (1, 5, 129, 128, 1, 4, True),     # Ulysses Anything: heads 2/1/1/1, tokens 33/32/32/32
    (1, 24, 130, 128, 1, 5, True),    # Ulysses Anything: heads 5/5/5/5/4, tokens 26 x 5
])
@pytest.mark.parametrize("mode", ["fused", "stepwise"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_cp_attention_small_grid(B, H, S, D, R, U, ev, mode, dtype):
    q, k, v = make_qkv(B, H, S, D, dtype, seed=S + 31 * R + U)

    class W:
        pass
    w = W()
    w.scale, w.ring_degree, w.ulysses_degree, w.uneven_ok = D ** -0.5, R, U, ev
    ro, rl = oracle.cp_attention(q, k, v, w.scale, R, U, ev)
    out, lse = run_fwd(*dev(q, k, v), w, mode)
    check_attn(out, lse, ro, rl, BF16_TOL if dtype == "bf16" else F32_TOL, f"grid {B},{H},{S},{D},{R},{U},{ev}")


# Score patterns for the three branches of the tensor-core softmax after the
# first K/V tile: exponentials with the running maximum kept (row sum <= 2^8);
# row sum above 2^8 with the maximum grown by less than 2^8 (reload, same
# maximum); maximum grown by more than 2^8 (rescale), including growth large
# enough that the first try overflows to inf. q = e_0 for every row and key j
# has k_j = c_j e_0, so the scores are c_j * scale exactly; the tile steps of
# c (in log2 units of the scaled score) are listed per case.
RESCALE_CASES = {
    "kept": [0.0, -1.0, 0.5, -3.0],
    "sum_over_no_rescale": [0.0, 3.0, 3.0, 2.0],
    "rescale": [0.0, 3.0, 20.0, 25.0],
    "overflow_then_rescale": [0.0, 200.0, 150.0, 260.0],
}


@pytest.mark.parametrize("case", sorted(RESCALE_CASES))
@pytest.mark.parametrize("mode", ["fused", "stepwise"])
def test_softmax_rescale_branches(case, mode):
    steps = RESCALE_CASES[case]
    B, H, D = 1, 2, 128
    S = 128 * len(steps) - 37  # ragged last tile
    scale = D ** -0.5
    g = torch.Generator().manual_seed(7)
    # per key: the tile's level (log2 units) minus a spread inside the tile, so
    # that every tile has its own maximum and a range of values below it
    lvl = torch.tensor([steps[j // 128] for j in range(S)], dtype=torch.float64)
    spread = torch.rand(S, generator=g, dtype=torch.float64) * 6.0
    c = (lvl - spread) / (scale * np.log2(np.e))
    q = torch.zeros(B, S, H, D)
    q[..., 0] = 1.0
    k = torch.zeros(B, S, H, D)
    k[..., 0] = c.float()[None, :, None]
    v = torch.randn(B, S, H, D, generator=g)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))

    class W:
        pass
    w = W()
    w.scale, w.ring_degree, w.ulysses_degree, w.uneven_ok = scale, 2, 1, True
    ro, rl = oracle.cp_attention(q, k, v, scale, 2, 1, True)
    out, lse = run_fwd(*dev(q, k, v), w, mode)
    check_attn(out, lse, ro, rl, BF16_TOL, f"rescale/{case}/{mode}")
    assert cpa().cp_check_device_status() == 0


@pytest.mark.parametrize("name,mode,chunks", [
    ("flux_ring4", "fused", 1), ("flux_ring4", "fused", 3), ("flux_ring4", "fused", 4), ("flux_ring4", "fused", 5),
    ("ring_anything3", "fused", 5), ("flux_ulysses4", "fused", 4), ("tiny_ring", "fused", 2),
    ("flux_ring4", "stepwise", 4),
])
def test_attention_fwd_host_equals_device_call(name, mode, chunks):
    """The host-buffer entry point (copies overlapping compute over head chunks) gives the device
    entry point's result bit for bit: heads are independent launches of the same kernel. Five chunks
    at FLUX ring 4 is bench.py's setting (2/8/8/4/2 heads)."""
    w = WORKLOADS[name]
    q, k, v = make_qkv(w.B, w.H, w.S, w.D, w.dtype, w.seed, w.q_mult)
    ref_out, ref_lse = run_fwd(*dev(q, k, v), w, mode)
    qp, kp, vp = (t.pin_memory() for t in (q, k, v))
    out = torch.full((w.B, w.S, w.H, w.D), float("nan")).pin_memory()
    lse = torch.full((w.B, w.H, w.S), float("nan")).pin_memory()
    cpa().cp_attention_fwd_host(qp, kp, vp, out, lse, w.scale, w.ring_degree, w.ulysses_degree, w.uneven_ok,
                                mode=mode, head_chunks=chunks)
    torch.cuda.synchronize()
    assert cpa().cp_check_device_status() == 0
    assert torch.equal(out, ref_out.cpu()) and torch.equal(lse, ref_lse.cpu())


# ----------------------------------------------------------------------------
# key-padding mask (cp_attention_fwd_masked)
# ----------------------------------------------------------------------------
def run_fwd_masked(q, k, v, km, w, mode):
    B, S, H, D = q.shape
    out = torch.empty((B, S, H, D), device="cuda")
    lse = torch.empty((B, H, S), device="cuda")
    cpa().cp_attention_fwd(q, k, v, out, lse, w.scale, w.ring_degree, w.ulysses_degree, w.uneven_ok, mode=mode,
                           key_mask=km.cuda())
    torch.cuda.synchronize()
    assert cpa().cp_check_device_status() == 0
    return out, lse


@pytest.mark.parametrize("mode", ["fused", "stepwise"])
def test_masked_flux_text_padding(mode):
    """FLUX ring 4 with the text part padded: keys 300..511 of the 512 text tokens masked."""
    w = WORKLOADS["flux_ring4"]
    q, k, v = make_qkv(w.B, w.H, w.S, w.D, w.dtype, w.seed)
    km = torch.ones((w.B, w.S), dtype=torch.bool)
    km[:, 300:512] = False
    ro, rl = oracle.cp_attention(q, k, v, w.scale, w.ring_degree, 1, False, key_mask=km.numpy())
    out, lse = run_fwd_masked(*dev(q, k, v), km, w, mode)
    check_attn(out, lse, ro, rl, BF16_TOL, f"masked flux/{mode}")


@pytest.mark.parametrize("B,H,S,D,R,U,ev", [
    (2, 4, 300, 64, 3, 1, False),     # ring 3 (100-token blocks)
    (1, 8, 384, 128, 1, 4, False),    # Ulysses 4
    (1, 8, 520, 128, 4, 2, False),    # unified 4 x 2
    (2, 7, 300, 64, 1, 3, True),      # Ulysses Anything
    (1, 4, 129, 128, 1, 1, False),    # plain attention
])
@pytest.mark.parametrize("mode", ["fused", "stepwise"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_masked_small_grid(B, H, S, D, R, U, ev, mode, dtype):
    q, k, v = make_qkv(B, H, S, D, dtype, seed=S + 7 * R + U)
    g = torch.Generator().manual_seed(S)
    km = torch.rand((B, S), generator=g) < 0.6   # partly masked tiles everywhere
    km[0, : S // 3] = False                      # a run of fully masked tiles / blocks
    if B > 1:
        km[1, :] = False                         # an entry with every key masked: out 0, lse -inf
    class W:
        pass
    w = W()
    w.scale, w.ring_degree, w.ulysses_degree, w.uneven_ok = D ** -0.5, R, U, ev
    ro, rl = oracle.cp_attention(q, k, v, w.scale, R, U, ev, key_mask=km.numpy())
    out, lse = run_fwd_masked(*dev(q, k, v), km, w, mode)
    check_attn(out, lse, ro, rl, BF16_TOL if dtype == "bf16" else F32_TOL, f"masked grid {B},{H},{S},{D},{R},{U}")


def test_mask_all_ones_is_bitwise_unmasked_and_ring_anything_rejects_a_mask():
    w = WORKLOADS["ring_anything3"]
    q, k, v = dev(*make_qkv(w.B, w.H, w.S, w.D, w.dtype, w.seed))
    km = torch.ones((w.B, w.S), dtype=torch.bool, device="cuda")
    out = torch.empty((w.B, w.S, w.H, w.D), device="cuda")
    lse = torch.empty((w.B, w.H, w.S), device="cuda")
    with pytest.raises(cpa().CpError):
        cpa().cp_attention_fwd(q, k, v, out, lse, w.scale, 3, 1, True, key_mask=km)
    w4 = WORKLOADS["flux_ring4"]
    q4, k4, v4 = dev(*make_qkv(w4.B, w4.H, w4.S, w4.D, w4.dtype, w4.seed))
    ref = run_fwd(q4, k4, v4, w4, "fused")
    got = run_fwd_masked(q4, k4, v4, torch.ones((w4.B, w4.S), dtype=torch.bool), w4, "fused")
    assert torch.equal(ref[0], got[0]) and torch.equal(ref[1], got[1])


@pytest.mark.parametrize("B,H,S,D,R,U", [
    (1, 24, 4608, 128, 1, 4),   # FLUX Ulysses 4
    (2, 8, 640, 128, 1, 2),     # two batch entries
    (1, 12, 1024, 64, 2, 2),    # unified 2 x 2 at D = 64
    (1, 30, 516, 128, 1, 6),    # six head groups
])
def test_ulysses_equals_composition_of_public_calls(B, H, S, D, R, U):
    """The fused Ulysses call gives, bit for bit, the plain sequence of the public calls: seq->head
    regroup of the rank shards, attention of the head groups (the ring lap inside, for the unified
    grid), head->seq regroup of out and a permute of lse."""
    q, k, v = dev(*make_qkv(B, H, S, D, "bf16", seed=5 + S + U))
    scale = D ** -0.5
    out = torch.empty((B, S, H, D), device="cuda")
    lse = torch.empty((B, H, S), device="cuda")
    cpa().cp_attention_fwd(q, k, v, out, lse, scale, R, U, mode="fused")
    Hg = H // U

    def to_heads(x):  # global [B, S, H, D] -> the head groups [U, B, S, Hg, D], through the rank shards
        shards = x.view(B, U, S // U, H, D).permute(1, 0, 2, 3, 4).contiguous()
        y = torch.empty((U, B, S, Hg, D), dtype=x.dtype, device="cuda")
        cpa().cp_ulysses_seq2head(shards, y)
        return y

    qh, kh, vh = (to_heads(t).view(U * B, S, Hg, D) for t in (q, k, v))
    oh = torch.empty((U * B, S, Hg, D), device="cuda")
    lh = torch.empty((U * B, Hg, S), device="cuda")
    if R == 1:
        cpa().cp_block_attn_fwd(qh, kh, vh, oh, lh, scale)
    else:
        cpa().cp_attention_fwd(qh, kh, vh, oh, lh, scale, R, 1, mode="fused")
    shards = torch.empty((U, B, S // U, H, D), device="cuda")
    cpa().cp_ulysses_head2seq(oh.view(U, B, S, Hg, D), shards)
    out_seq = shards.permute(1, 0, 2, 3, 4).reshape(B, S, H, D)
    lse_seq = lh.view(U, B, Hg, S).permute(1, 0, 2, 3).reshape(B, H, S)
    torch.cuda.synchronize()
    assert cpa().cp_check_device_status() == 0
    assert torch.equal(out, out_seq) and torch.equal(lse, lse_seq)


@pytest.mark.parametrize("B,H,S,D,U", [(1, 24, 4481, 128, 4), (2, 7, 333, 64, 3), (1, 24, 4608, 128, 5)])
def test_ulysses_anything_equals_composition_of_public_calls(B, H, S, D, U):
    """The same for the ragged groups of Ulysses Anything: the ragged regroups, then the attention of
    each head group on its own (its real heads only), then the ragged regroup back."""
    q, k, v = dev(*make_qkv(B, H, S, D, "bf16", seed=9 + S + U))
    scale = D ** -0.5
    out = torch.empty((B, S, H, D), device="cuda")
    lse = torch.empty((B, H, S), device="cuda")
    cpa().cp_attention_fwd(q, k, v, out, lse, scale, 1, U, True, mode="fused")
    hl = [H // U + (1 if g < H % U else 0) for g in range(U)]
    sl = [S // U + (1 if u < S % U else 0) for u in range(U)]
    so = [sum(sl[:u]) for u in range(U)]
    n = B * S * H * D

    def to_heads(x):  # global [B, S, H, D] -> rank blocks [B, S_u, H, D] -> group blocks [B, S, H_g, D]
        ranks = torch.cat([x[:, so[u]:so[u] + sl[u]].reshape(-1) for u in range(U)])
        y = torch.empty(n, dtype=x.dtype, device="cuda")
        cpa().cp_ulysses_anything_seq2head(ranks, y, U, B, S, H, D)
        return y

    qh, kh, vh = (to_heads(t) for t in (q, k, v))
    oh = torch.empty(n, device="cuda")
    lses = []
    o0 = 0
    for g in range(U):
        m = B * S * hl[g] * D
        blk = [t[o0:o0 + m].view(B, S, hl[g], D) for t in (qh, kh, vh, oh)]
        lg = torch.empty((B, hl[g], S), device="cuda")
        cpa().cp_block_attn_fwd(blk[0], blk[1], blk[2], blk[3], lg, scale)
        lses.append(lg)
        o0 += m
    ranks = torch.empty(n, device="cuda")
    cpa().cp_ulysses_anything_head2seq(oh, ranks, U, B, S, H, D)
    blocks, o0 = [], 0
    for u in range(U):  # rank blocks back to the global [B, S, H, D]
        blocks.append(ranks[o0:o0 + B * sl[u] * H * D].view(B, sl[u], H, D))
        o0 += B * sl[u] * H * D
    out_seq = torch.cat(blocks, dim=1)
    torch.cuda.synchronize()
    assert cpa().cp_check_device_status() == 0
    assert torch.equal(out, out_seq)
    assert torch.equal(lse, torch.cat(lses, dim=1))


def test_cp_attention_modes_agree_and_deterministic():
    w = WORKLOADS["flux_ring4"]
    q, k, v = dev(*make_qkv(w.B, w.H, w.S, w.D, w.dtype, w.seed))
    a = run_fwd(q, k, v, w, "fused")
    b = run_fwd(q, k, v, w, "fused")
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    c = run_fwd(q, k, v, w, "stepwise")
    assert float((a[0] - c[0]).abs().max()) < 2e-3


# ----------------------------------------------------------------------------
# bounded device waits
# ----------------------------------------------------------------------------
def test_bounded_wait_reports_timeout_and_context_survives():
    m = cpa()
    assert m.cp_check_device_status() == 0
    m.cp_debug_bounded_wait_probe(2000)  # 2 ms limit on a barrier nothing completes
    assert m.cp_check_device_status() == m._lib.CP_ERR_TIMEOUT
    assert m.cp_check_device_status() == 0  # the word was cleared
    # the context is still usable
    B, H, S, D = 1, 2, 200, 64
    q, k, v = make_qkv(B, H, S, D, "bf16", seed=1)
    ro, rl = oracle.attention(q, k, v, 0.125)
    dq, dk, dv = dev(q, k, v)
    out = torch.empty((B, S, H, D), device="cuda")
    lse = torch.empty((B, H, S), device="cuda")
    m.cp_block_attn_fwd(dq, dk, dv, out, lse, 0.125)
    check_attn(out, lse, ro, rl, BF16_TOL, "after probe")
