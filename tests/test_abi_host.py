"""Host-side checks of libcpattn.so that need no GPU: the library loads, it
exports every function include/cp_attn.h declares, and the argument checks,
shard table, workspace sizing and launch counts behave as specified. No call
here launches a kernel (all of them fail validation or are host-only)."""
import ctypes
import json
import os
import re

import pytest
import torch

import context_attention_dits_gb300 as cpa
from context_attention_dits_gb300 import _lib
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cp_attn.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "variant_requirements.json")
NAMES = {"ok": 0, "invalid_arg": -1, "not_divisible": -2, "unsupported_combo": -3}


@pytest.fixture(scope="module", autouse=True)
def built_lib():
    from context_attention_dits_gb300 import build
    build.build()
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(cp_[a-z0-9_]+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol(built_lib):
    names = declared_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(built_lib, n), n
    assert set(names) == set(_lib.SIGNATURES), "binding signatures must cover the header exactly"


def test_status_strings_and_version():
    assert cpa.cp_status_string(0) == "ok"
    for code in range(-8, 0):
        assert cpa.cp_status_string(code) != "unknown status"
    assert cpa.cp_version() >= 10000


def test_validate_golden_requirements_table():
    spec = json.load(open(GOLDEN))
    for case in spec["cases"]:
        got = cpa.cp_attention_validate(1, case["H"], case["S"], 128, case["ring_degree"], case["ulysses_degree"],
                                        case["uneven_ok"])
        assert got == NAMES[case["expect"]], case["name"]


def test_validate_argument_errors():
    assert cpa.cp_attention_validate(1, 24, 4608, 96, 4, 1, False) == -1        # D unsupported
    assert cpa.cp_attention_validate(1, 24, 4608, 128, 0, 1, False) == -1      # degree < 1
    assert cpa.cp_attention_validate(1, 24, 4608, 128, 17, 1, False) == -1     # beyond the 16-rank tables
    assert cpa.cp_attention_validate(-1, 24, 4608, 128, 1, 1, False) == -1
    assert cpa.cp_attention_validate(1, 24, 4608, 128, 1, 1, False) == 0
    assert cpa.cp_attention_validate(1, 2, 256, 64, 2, 1, False, torch.float32) == 0


@pytest.mark.parametrize("S", [0, 1, 5, 127, 256, 4607, 4608, 32768])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 16])
def test_shard_table_matches_oracle(S, n):
    want = oracle.ring_shard_table(S, n, True)
    assert cpa.cp_ring_shard_table(S, n, True) == want
    if S % n:
        with pytest.raises(cpa.CpError):
            cpa.cp_ring_shard_table(S, n, False)
    else:
        assert cpa.cp_ring_shard_table(S, n, False) == want


def test_workspace_and_launch_counts():
    f = cpa.cp_attention_workspace_size
    assert f(1, 24, 4608, 128, 4, 1, torch.bfloat16, "fused") == 0
    n = 4608 * 24 * 128
    assert f(1, 24, 4608, 128, 4, 1, torch.bfloat16, "stepwise") >= n * 4 + 24 * 4608 * 4
    assert f(1, 24, 4608, 128, 1, 4, torch.bfloat16, "fused") >= 3 * n * 2 + n * 4 + 24 * 4608 * 4
    c = cpa.cp_attention_launch_count
    assert c(1, 24, 4608, 128, 4, 1, torch.bfloat16, "fused") == 1
    assert c(1, 24, 4608, 128, 4, 1, torch.bfloat16, "stepwise") == 7
    # Ulysses: q, k, v regroups share one bulk launch, out and lse another
    assert c(1, 24, 4608, 128, 1, 4, torch.bfloat16, "fused") == 3
    # 128-byte q, k, v segments take a vector launch each
    assert c(1, 24, 4608, 64, 1, 24, torch.bfloat16, "fused") == 5
    # 128 KB lse rows exceed a ring slot: out and lse launch separately
    assert c(1, 24, 32768, 128, 2, 4, torch.bfloat16, "stepwise") == 3 + 1 + 2


def _raw(fn, *args):
    return getattr(_lib.lib(), fn)(*args)


def test_fwd_rejects_before_any_launch():
    # every call below must fail host validation: none reaches the GPU
    p = 1 << 20  # a fake, 16-byte aligned "device" address that is never dereferenced
    args = lambda **kw: [kw.get("q", p), kw.get("k", p), kw.get("v", p), kw.get("o", p), kw.get("l", p),
                         kw.get("B", 1), kw.get("H", 24), kw.get("S", 4608), kw.get("D", 128), 0.088,
                         kw.get("R", 4), kw.get("U", 1), kw.get("ev", 0), None, 0, kw.get("dt", 0),
                         kw.get("mode", 0), None]
    f = lambda **kw: _raw("cp_attention_fwd", *args(**kw))
    assert f(S=4481) == _lib.CP_ERR_NOT_DIVISIBLE
    assert f(S=4481, U=2, R=2, ev=1) == _lib.CP_ERR_UNSUPPORTED_COMBO
    assert f(D=96) == _lib.CP_ERR_INVALID_ARG
    assert f(q=0) == _lib.CP_ERR_INVALID_ARG
    assert f(q=p + 8) == _lib.CP_ERR_ALIGNMENT
    assert f(R=1, U=4) == _lib.CP_ERR_WORKSPACE            # Ulysses needs workspace
    assert f(mode=7) == _lib.CP_ERR_INVALID_ARG
    assert f(U=32, R=1) == _lib.CP_ERR_INVALID_ARG          # more Ulysses ranks than heads
    assert f(B=0) == _lib.CP_OK                             # empty: nothing to do, nothing launched


def test_block_attn_and_merge_and_permute_reject_before_launch():
    p = 1 << 20
    L = _lib.lib()
    assert L.cp_block_attn_fwd(p, p, p, p, p, 1, 24, 128, 128, 80, 0.1, 0, 0, 0, 0, None) == _lib.CP_ERR_INVALID_ARG
    assert L.cp_block_attn_fwd(p, p, p, p, p + 4, 1, 24, 128, 128, 128, 0.1, 0, 0, 0, 0, None) == _lib.CP_ERR_ALIGNMENT
    assert L.cp_block_attn_fwd(p, p, p, p, p, 1, 24, 128, 128, 128, float("nan"), 0, 0, 0, 0, None) == _lib.CP_ERR_INVALID_ARG
    assert L.cp_block_attn_fwd(p, p, p, p, p, 1, 24, 128, 128, 128, 0.1, 100, 0, 0, 0, None) == _lib.CP_ERR_INVALID_ARG
    assert L.cp_block_attn_fwd(p, p, p, p, p, 2, 24, 0, 128, 128, 0.1, 0, 0, 0, 0, None) == _lib.CP_OK
    assert L.cp_lse_merge(p, p, p, p, 1, 24, 16, 6, None) == _lib.CP_ERR_INVALID_ARG
    assert L.cp_lse_merge(p + 4, p, p, p, 1, 24, 16, 8, None) == _lib.CP_ERR_ALIGNMENT
    assert L.cp_ulysses_seq2head(p, p, 5, 1, 4608, 24, 128, 2, None) == _lib.CP_ERR_INVALID_ARG
    assert L.cp_ulysses_head2seq(p, p, 4, 1, 4607, 24, 128, 2, None) == _lib.CP_ERR_INVALID_ARG
    assert L.cp_ulysses_seq2head(p, p, 32, 1, 4608, 24, 128, 2, None) == _lib.CP_ERR_INVALID_ARG
    assert L.cp_debug_bounded_wait_probe(0, None) == _lib.CP_ERR_INVALID_ARG


def test_masked_host_buffer_and_anything_entry_points_reject_before_launch():
    p = 1 << 20
    L = _lib.lib()
    # cp_attention_fwd_masked: q, k, v, key_mask, out, lse, B, H, S, D, scale, R, U, ev, ws, ws_bytes, dt, mode, stream
    m = lambda **kw: L.cp_attention_fwd_masked(p, p, p, kw.get("km", p), p, p, 1, 24, kw.get("S", 4608),
                                               kw.get("D", 128), 0.088, kw.get("R", 4), kw.get("U", 1),
                                               kw.get("ev", 0), None, 0, 0, 0, None)
    assert m(S=4607, R=3, ev=1) == _lib.CP_ERR_UNSUPPORTED_COMBO   # Ring Anything takes no mask
    assert m(D=96) == _lib.CP_ERR_INVALID_ARG
    assert m(S=4481) == _lib.CP_ERR_NOT_DIVISIBLE
    # cp_attention_fwd_host: q, k, v, out, lse (host), B, H, S, D, scale, R, U, ev, dev_buf, dev_bytes, dt, mode,
    # head_chunks, stream
    need = cpa.cp_attention_host_buffer_size(1, 24, 4608, 128, 4, 1, torch.bfloat16, "fused")
    n = 4608 * 24 * 128
    assert need >= 3 * n * 2 + n * 4 + 24 * 4608 * 4
    hfn = lambda **kw: L.cp_attention_fwd_host(p, p, p, p, p, kw.get("B", 1), 24, 4608, 128, 0.088, 4, 1, 0,
                                               kw.get("buf", p), kw.get("nb", need), 0, 0, kw.get("ch", 4), None)
    assert hfn(ch=0) == _lib.CP_ERR_INVALID_ARG
    assert hfn(nb=need - 1) == _lib.CP_ERR_WORKSPACE
    assert hfn(buf=p + 16) == _lib.CP_ERR_ALIGNMENT
    assert hfn(buf=0) == _lib.CP_ERR_INVALID_ARG
    assert hfn(B=0) == _lib.CP_OK
    # Ulysses Anything regroups: U <= H, element size 1, 2, 4 or 8
    assert L.cp_ulysses_anything_seq2head(p, p, 25, 1, 4481, 24, 128, 2, None) == _lib.CP_ERR_INVALID_ARG
    assert L.cp_ulysses_anything_head2seq(p, p, 4, 1, 4481, 24, 128, 3, None) == _lib.CP_ERR_INVALID_ARG
    assert L.cp_ulysses_anything_seq2head(p, p, 5, 0, 4481, 24, 128, 2, None) == _lib.CP_OK
    # ragged head groups: the 15 per-group q, k, v copies share a launch, the 10 out / lse copies another
    c = cpa.cp_attention_launch_count
    assert c(1, 24, 4608, 128, 1, 5, torch.bfloat16, "fused") == 3
    # 4481-float lse rows are not 16-byte multiples: the lse regroup takes a vector launch
    assert c(1, 24, 4481, 128, 1, 4, torch.bfloat16, "fused") == 4
    assert cpa.cp_attention_validate(1, 24, 4481, 128, 1, 4, True) == 0
    assert cpa.cp_attention_validate(1, 24, 4608, 128, 1, 5, True) == 0


def test_bwd_sizes_counts_and_rejects_before_launch():
    p = 1 << 20
    L = _lib.lib()
    n, nl = 4608 * 24 * 128, 24 * 4608
    ws = cpa.cp_attention_bwd_workspace_size
    assert ws(1, 24, 4608, 128, 4, 1, torch.bfloat16) >= nl * 4                      # delta only
    assert ws(1, 24, 4608, 128, 1, 4, torch.bfloat16) >= nl * 4 + 4 * n * 2 + 2 * nl * 4 + 3 * n * 4
    c = cpa.cp_attention_bwd_launch_count
    assert c(1, 24, 4608, 128, 4, 1, torch.bfloat16) == 3       # delta, padded lse/delta, dk/dv + dq (tensor cores)
    assert c(1, 24, 4608, 128, 4, 1, torch.float32) == 3        # delta, dq, dk/dv on the CUDA cores
    # Ulysses: q, k, v, dout, lse, delta regroups share a launch, dq, dk, dv another
    assert c(1, 24, 4608, 128, 1, 4, torch.bfloat16) == 5
    assert c(0, 24, 4608, 128, 4, 1, torch.bfloat16) == 0
    # Ulysses Anything over 5 head groups: 30 ragged in-copies (two bulk launches of <= 24), 15 out-copies
    assert c(1, 24, 4608, 128, 1, 5, torch.bfloat16) == 3 + 2 + 1
    # 4481-float lse / delta rows are not 16-byte multiples: each of their 10 copies takes a vector launch,
    # the 20 q, k, v, dout copies share one bulk launch
    assert c(1, 24, 4481, 128, 1, 5, torch.bfloat16) == 3 + (1 + 10) + 1
    # 128 KB lse / delta rows exceed a ring slot at 32768 tokens
    assert c(2, 24, 32768, 128, 2, 4, torch.bfloat16) == 3 + (1 + 2) + 1
    # q, k, v, out, dout, lse, dq, dk, dv, B, H, S, D, scale, R, U, ev, ws, ws_bytes, dt, stream
    big = 1 << 34
    f = lambda **kw: L.cp_attention_bwd(kw.get("q", p), p, p, p, p, p, p, p, kw.get("dv", p), 1, 24,
                                        kw.get("S", 4608), kw.get("D", 128), kw.get("scale", 0.088), kw.get("R", 4),
                                        kw.get("U", 1), kw.get("ev", 0), kw.get("ws", p), kw.get("wsb", big), 0, None)
    assert f(ev=1, S=4607, R=3) == _lib.CP_ERR_UNSUPPORTED_COMBO   # Ring Anything: inference only
    assert f(ev=1, S=4481, U=5, R=1, ws=0) == _lib.CP_ERR_WORKSPACE  # Ulysses Anything passes validation
    assert f(ev=1, U=2, R=2) == _lib.CP_ERR_UNSUPPORTED_COMBO
    assert f(S=4607) == _lib.CP_ERR_NOT_DIVISIBLE
    assert f(D=96) == _lib.CP_ERR_INVALID_ARG
    assert f(scale=float("inf")) == _lib.CP_ERR_INVALID_ARG
    assert f(q=0) == _lib.CP_ERR_INVALID_ARG
    assert f(dv=p + 4) == _lib.CP_ERR_ALIGNMENT
    assert f(ws=0) == _lib.CP_ERR_WORKSPACE
    assert f(wsb=16) == _lib.CP_ERR_WORKSPACE
    assert f(ws=p + 16) == _lib.CP_ERR_ALIGNMENT
    # empty problems launch nothing and succeed
    assert L.cp_attention_bwd(p, p, p, p, p, p, p, p, p, 0, 24, 4608, 128, 0.088, 4, 1, 0, None, 0, 0, None) == 0
    assert L.cp_attention_bwd(p, p, p, p, p, p, p, p, p, 1, 24, 0, 128, 0.088, 1, 4, 0, None, 0, 0, None) == 0
    # ragged head groups are stored padded: 24 heads over 5 groups take 5 x 5 head slots
    hp = 25
    assert ws(1, 24, 4608, 128, 1, 5, torch.bfloat16) >= nl * 4 + 4 * (n // 24 * hp) * 2 + 2 * (nl // 24 * hp) * 4 \
        + 3 * (n // 24 * hp) * 4
