"""GPU test of cp_attention_fwd_no_alloc, the entry point for callers that
cannot allocate device memory (their device memory belongs to a host framework
that gives plugins no allocator, or they cannot afford an allocation's latency
and implicit synchronisation in the middle of a step). Instead of a caller
workspace it uses the library's built-in 64 MiB device array.

The call goes through the C ABI and its output is compared with that of the
existing entry point, cp_attention_fwd with a caller workspace, and with the
float64 oracle, within the bf16 parity tolerance of the other GPU tests, on two
calls in a row (with different inputs, so stale contents of the shared array
would show). One case needs a workspace just under the array's size; one needs
none and must leave the array alone. The file is named so that pytest collects
it last; it builds what it needs itself, so it passes alone in a fresh process
as well as after the other tests.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import make_qkv

pytestmark = pytest.mark.gpu

TOL_MAX_ABS, TOL_REL_L2 = 1e-2, 5e-3


@pytest.fixture(scope="module")
def cpa():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from context_attention_dits_gb300 import build
    build.build()
    import context_attention_dits_gb300 as m
    return m


def _close(got, want, what):
    got = got.double().cpu().numpy()
    want = want.double().cpu().numpy() if isinstance(want, torch.Tensor) else np.asarray(want, np.float64)
    assert np.array_equal(np.isneginf(got), np.isneginf(want)), what
    fin = np.isfinite(want)
    err = np.abs(got[fin] - want[fin])
    rel = np.sqrt(np.sum(err ** 2) / max(np.sum(want[fin] ** 2), 1e-300))
    assert err.max() <= TOL_MAX_ABS and rel <= TOL_REL_L2, f"{what}: max abs {err.max():.3e}, rel L2 {rel:.3e}"


# (B, H, S, D, ring, ulysses, uneven_ok, mode): each needs workspace
CASES = [
    (1, 8, 512, 128, 1, 4, False, "fused"),      # Ulysses regroups live in the workspace
    (2, 4, 301, 64, 3, 1, True, "stepwise"),     # per-step partials live in the workspace
    (1, 6, 384, 128, 2, 3, False, "stepwise"),   # unified grid, both kinds of scratch
    (1, 8, 6530, 128, 1, 2, False, "fused"),     # Ulysses 2: 99.95% of the built-in array
]


def _oracle_check(q, k, v, scale, R, U, ev, out, lse, what):
    """The float64 oracle on every row when that is cheap, else on 64 seeded rows (rows are independent)."""
    B, S, H, D = q.shape
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    if S <= 1024:
        ro, rl = oracle.cp_attention(qc, kc, vc, scale, R, U, ev)
        _close(out, ro, f"{what} out vs oracle")
        _close(lse, rl, f"{what} lse vs oracle")
        return
    rows = np.sort(np.random.default_rng(S).choice(S, size=64, replace=False))
    ro, rl = oracle.attention_rows(qc, kc, vc, scale, rows)
    _close(out[:, rows], ro, f"{what} out vs oracle (sampled rows)")
    _close(lse[:, :, rows], rl, f"{what} lse vs oracle (sampled rows)")


@pytest.mark.parametrize("B,H,S,D,R,U,ev,mode", CASES)
def test_no_alloc_matches_workspace_entry_point(cpa, B, H, S, D, R, U, ev, mode):
    from context_attention_dits_gb300 import _lib
    L = _lib.lib()
    scale = D ** -0.5
    assert 0 < cpa.cp_attention_workspace_size(B, H, S, D, R, U, torch.bfloat16, mode) <= \
        _lib.CP_NO_ALLOC_WORKSPACE_BYTES
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # two calls in a row on the shared array
        q, k, v = [t.cuda() for t in make_qkv(B, H, S, D, "bf16", seed=100 * call + S + R)]
        ref_out = torch.empty((B, S, H, D), device="cuda")
        ref_lse = torch.empty((B, H, S), device="cuda")
        cpa.cp_attention_fwd(q, k, v, ref_out, ref_lse, scale, R, U, ev, mode=mode)
        out = torch.full((B, S, H, D), float("nan"), device="cuda")
        lse = torch.full((B, H, S), float("nan"), device="cuda")
        st = L.cp_attention_fwd_no_alloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                         B, H, S, D, scale, R, U, int(ev), _lib.CP_BF16,
                                         _lib.CP_LAP_STEPWISE if mode == "stepwise" else _lib.CP_LAP_FUSED, stream)
        assert st == _lib.CP_OK, cpa.cp_status_string(st)
        torch.cuda.synchronize()
        assert cpa.cp_check_device_status() == 0
        _close(out, ref_out, f"call {call} out")
        _close(lse, ref_lse, f"call {call} lse")
        _oracle_check(q, k, v, scale, R, U, ev, out, lse, f"call {call}")


def test_no_alloc_without_scratch(cpa):
    """A plain ring with the fused lap needs no workspace: the call runs without the built-in array."""
    from context_attention_dits_gb300 import _lib
    L = _lib.lib()
    B, H, S, D, R = 1, 4, 640, 128, 4
    assert cpa.cp_attention_workspace_size(B, H, S, D, R, 1, torch.bfloat16, "fused") == 0
    scale = D ** -0.5
    q, k, v = [t.cuda() for t in make_qkv(B, H, S, D, "bf16", seed=31)]
    out = torch.full((B, S, H, D), float("nan"), device="cuda")
    lse = torch.full((B, H, S), float("nan"), device="cuda")
    st = L.cp_attention_fwd_no_alloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                     B, H, S, D, scale, R, 1, 0, _lib.CP_BF16, _lib.CP_LAP_FUSED,
                                     torch.cuda.current_stream().cuda_stream)
    assert st == _lib.CP_OK, cpa.cp_status_string(st)
    torch.cuda.synchronize()
    assert cpa.cp_check_device_status() == 0
    _oracle_check(q, k, v, scale, R, 1, False, out, lse, "no scratch")


def test_no_alloc_rejects_beyond_its_workspace(cpa):
    from context_attention_dits_gb300 import _lib
    L = _lib.lib()
    # Ulysses 4 at FLUX size needs ~141 MB of workspace: more than the built-in 64 MiB
    need = cpa.cp_attention_workspace_size(1, 24, 4608, 128, 1, 4, torch.bfloat16, "fused")
    assert need > _lib.CP_NO_ALLOC_WORKSPACE_BYTES
    p = 1 << 20  # never dereferenced: the call is rejected before any launch
    st = L.cp_attention_fwd_no_alloc(p, p, p, p, p, 1, 24, 4608, 128, 0.088, 1, 4, 0, _lib.CP_BF16,
                                     _lib.CP_LAP_FUSED, None)
    assert st == _lib.CP_ERR_WORKSPACE
