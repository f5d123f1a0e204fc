"""GPU parity of the backward (cp_attention_bwd) against the float64 oracle.

Both sides take the same forward results (out, lse): the oracle's, rounded to
fp32, so the check isolates the backward's arithmetic. fp32 inputs run on the
CUDA cores in fp32: relative L2 <= 1e-4 and max abs <= 1e-3 x max |reference|
(the fp32 forward's bound, loosened for the longer sums of the backward).
bf16 inputs run on the tensor cores: the forward's bf16 bounds (see TOL).
"""
import numpy as np
import pytest
import torch

from oracle import cp_oracle as co
from synth import make_dout, make_qkv

pytestmark = pytest.mark.gpu

# (relative L2, max abs as a fraction of max |reference|) per input dtype. bf16
# runs on the tensor cores with P and dS rounded to bf16 (relative 2^-9) for
# their products: measured ~1.7e-3 relative L2 on random inputs, so the
# forward's bf16 bounds (5e-3 relative L2, 1e-2 max abs at unit scale) apply,
# the max abs taken relative to the gradient's largest entry.
TOL = {"f32": (1e-4, 1e-3), "bf16": (5e-3, 1e-2)}
ZERO_ABS = 1e-4  # where the exact gradient is 0 (one key), only this absolute bound


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from context_attention_dits_gb300 import build
    build.build()


def cpa():
    import context_attention_dits_gb300 as m
    return m


def check(got, want, what, dtype):
    rel_tol, abs_tol = TOL[dtype]
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, what
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - want)
    if float(np.abs(want).max()) == 0.0:
        print(f"{what}: exact zero, max abs {err.max():.3e}")
        assert err.max() <= ZERO_ABS, f"{what}: max abs {err.max():.3e} > {ZERO_ABS} where the gradient is 0"
        return
    scale = float(np.abs(want).max())
    rl = float(np.sqrt(np.sum((got - want) ** 2)) / max(np.sqrt(np.sum(want * want)), 1e-300))
    print(f"{what}: rel L2 {rl:.3e}, max abs / max ref {err.max() / scale:.3e}")
    assert err.max() <= abs_tol * scale, f"{what}: max abs {err.max():.3e} > {abs_tol} x {scale:.3e}"
    assert rl <= rel_tol, f"{what}: rel L2 {rl:.3e} > {rel_tol}"


def run_bwd(q, k, v, out, dout, lse, scale, R, U, ev=False):
    dev = [t.cuda() for t in (q, k, v, out, dout, lse)]
    grads = [torch.empty(q.shape, dtype=torch.float32, device="cuda") for _ in range(3)]
    cpa().cp_attention_bwd(*dev, *grads, scale, R, U, uneven_ok=ev)
    torch.cuda.synchronize()
    return [g.cpu().numpy() for g in grads]


@pytest.mark.parametrize("B,S,H,D,R,U,ev,dtype", [
    (1, 300, 2, 64, 1, 1, False, "f32"),      # single block, ragged last tile (300 = 4 x 64 + 44)
    (2, 256, 4, 128, 2, 1, False, "bf16"),    # ring 2, two batch entries
    (1, 387, 3, 128, 3, 1, False, "bf16"),    # ring 3 over 129-token shards: a 1-row tile per shard
    (1, 512, 4, 64, 1, 2, False, "bf16"),     # Ulysses 2
    (2, 384, 4, 128, 2, 2, False, "f32"),     # unified 2 x 2
    (1, 1, 1, 128, 1, 1, False, "bf16"),      # one token: dq = dk = 0, dv = dout
    (1, 1000, 5, 128, 1, 4, True, "bf16"),    # Ulysses Anything: heads 2/1/1/1, tokens 250 x 4
    (2, 333, 7, 128, 1, 3, True, "bf16"),     # Ulysses Anything: heads 3/2/2, tokens 111 x 3
    (2, 97, 6, 64, 1, 4, True, "f32"),        # Ulysses Anything on the CUDA cores: heads 2/2/1/1, tokens 25/24/24/24
    # the tensor-core kernels walk 64-row sub-steps through 4 (dk/dv) and 6 (dq) streamed slots:
    (1, 130, 2, 128, 1, 1, False, "bf16"),    # an odd count of sub-steps (64 + 64 + 2)
    (1, 700, 3, 128, 2, 1, False, "bf16"),    # 350-token shards: 12 sub-steps per lap, every slot reused
    (1, 1000, 2, 64, 4, 1, False, "bf16"),    # ring 4 over 250-token shards at D = 64: 16 sub-steps
])
def test_bwd_matches_oracle(B, S, H, D, R, U, ev, dtype):
    q, k, v = make_qkv(B, H, S, D, dtype, seed=40 + S)
    dout = make_dout(B, S, H, D, dtype, seed=40 + S)
    scale = D ** -0.5
    out, lse = co.cp_attention(q, k, v, scale, R, U, ev)
    out32 = torch.from_numpy(out).float()
    lse32 = torch.from_numpy(lse).float()
    want = co.cp_attention_bwd(q, k, v, dout, scale, R, U, ev, out=out32.double().numpy(),
                               lse=lse32.double().numpy())
    got = run_bwd(q, k, v, out32, dout, lse32, scale, R, U, ev)
    for name, g, w in zip(("dq", "dk", "dv"), got, want):
        check(g, w, f"{name} B{B} S{S} H{H} D{D} R{R} U{U} ev{int(ev)} {dtype}", dtype)


def test_bwd_flux_ring4_sampled():
    """FLUX ring-4 shape (B=1, S=4608, H=24, D=128, bf16), every head computed on
    the GPU; the oracle checks sampled query rows (dq) and keys (dk, dv) of two
    heads, for which both sides take the oracle's forward (out, lse)."""
    B, S, H, D, R = 1, 4608, 24, 128, 4
    q, k, v = make_qkv(B, H, S, D, "bf16", seed=1)
    dout = make_dout(B, S, H, D, "bf16", seed=1)
    scale = D ** -0.5
    heads = [0, 23]
    # forward results: the library's for all heads, the oracle's for the sampled heads
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty((B, S, H, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    cpa().cp_attention_fwd(qd, kd, vd, out, lse, scale, R, 1)
    sub = [t[:, :, heads] for t in (q, k, v, dout)]
    o_or, l_or = co.attention(sub[0], sub[1], sub[2], scale)
    out[:, :, heads] = torch.from_numpy(o_or).float().cuda()
    lse[:, heads] = torch.from_numpy(l_or).float().cuda()
    o64 = out[:, :, heads].double().cpu().numpy()
    l64 = lse[:, heads].double().cpu().numpy()
    delta = co.attention_delta(o64, sub[3])
    dq, dk, dv = (torch.empty((B, S, H, D), dtype=torch.float32, device="cuda") for _ in range(3))
    cpa().cp_attention_bwd(qd, kd, vd, out, dout.cuda(), lse, dq, dk, dv, scale, R, 1)
    torch.cuda.synchronize()
    dq, dk, dv = (t[:, :, heads].cpu().numpy() for t in (dq, dk, dv))
    # rows and keys at shard and tile boundaries, the ends, and a few inside
    idx = np.array(sorted({0, 1, 63, 64, 1151, 1152, 1153, 2303, 2304, 3455, 3456, 4000, 4606, 4607}))
    gq, _, _ = co.attention_bwd(sub[0][:, idx], sub[1], sub[2], sub[3][:, idx], scale, l64[:, :, idx],
                                delta[:, :, idx])
    _, gk, gv = co.attention_bwd(sub[0], sub[1][:, idx], sub[2][:, idx], sub[3], scale, l64, delta)
    check(dq[:, idx], gq, "dq sampled rows", "bf16")
    check(dk[:, idx], gk, "dk sampled keys", "bf16")
    check(dv[:, idx], gv, "dv sampled keys", "bf16")


def test_bwd_rejects_ring_anything():
    q = torch.zeros((1, 8, 2, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros((1, 8, 2, 64), dtype=torch.float32, device="cuda")
    lse = torch.zeros((1, 2, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(cpa().CpError):
        cpa().cp_attention_bwd(q, q, q, o, q, lse, o, o.clone(), o.clone(), 0.125, 2, 1, uneven_ok=True)
