"""Host-side checks of the C-ABI library that need no GPU: it builds, loads,
exports every symbol include/ssd.h declares, and rejects bad arguments on
the host before touching CUDA.  Also checks that the oracle and the CUDA path
share no code."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "speculative_decoding_verification_70_gb300")
HEADER = os.path.join(ROOT, "include", "ssd.h")


def _no_gpu():
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:
        return True


# The argument-check tests pass made-up device addresses that only the host
# checks keep from reaching a kernel; they run where no GPU is present, so a
# regressed check can never launch a kernel on such an address.
needs_no_gpu = pytest.mark.skipif(not _no_gpu(), reason="fake device pointers: CPU-only host")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_70_gb300 import build
    path = build.build()
    from speculative_decoding_verification_70_gb300 import _binding
    return _binding.load_library(path)


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^SSD_API\s+[\w\s\*]+?\b(ssd_\w+)\s*\(", text, re.M)))


def test_header_declares_the_five_calls():
    names = declared_symbols()
    for n in ("ssd_softmax_temp", "ssd_verify", "ssd_sample_residual", "ssd_forked_recovery",
              "ssd_spec_cache_lookup"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only",
                          os.path.join(PKG, "libssd_gb300.so")],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (ssd_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(lib, n)


def test_binding_covers_the_header():
    from speculative_decoding_verification_70_gb300._binding import SIGNATURES
    assert sorted(s[0] for s in SIGNATURES) == declared_symbols()


def test_status_strings(lib):
    assert lib.ssd_status_string(0) == b"ok"
    assert lib.ssd_status_string(1) == b"invalid argument"
    assert lib.ssd_status_string(6) == b"workspace too small"
    assert lib.ssd_version() >= 100


def test_workspace_sizes(lib):
    assert lib.ssd_workspace_bytes(0, 5, 100, 0) == 0
    assert lib.ssd_workspace_bytes(1, 32, 100, 0) == 0      # k > 31
    assert lib.ssd_workspace_bytes(1, 5, 100, 17) == 0      # f > 16
    a = lib.ssd_workspace_bytes(512, 7, 151936, 0)
    b = lib.ssd_workspace_bytes(512, 7, 151936, 4)
    assert 0 < a < b
    assert b % 256 == 0
    assert lib.ssd_softmax_workspace_bytes(4, 1000) > 0


def _call_verify(lib, **kw):
    args = dict(Z=1 << 20, zb=0, D=1 << 20, db=0, dt=0, B=1, k=2, V=8, x=1 << 20, T=1 << 20,
                ua=1 << 20, acc=1 << 20, px=None, qx=None, us=None, out=None,
                ws=1 << 20, wsb=1 << 30)
    args.update(kw)
    if args["zb"] == 0:
        args["zb"] = (args["k"] + 1) * args["V"]
    if args["db"] == 0:
        args["db"] = args["k"] * args["V"]
    return lib.ssd_verify(args["Z"], args["zb"], args["D"], args["db"], args["dt"], args["B"],
                          args["k"], args["V"], args["x"], args["T"], args["ua"], args["acc"],
                          args["px"], args["qx"], args["us"], args["out"], args["ws"],
                          args["wsb"], None)


@needs_no_gpu
def test_verify_rejects_bad_arguments_on_host(lib):
    INVALID, DTYPE, WS = 1, 2, 6
    assert _call_verify(lib, Z=None) == INVALID
    assert _call_verify(lib, x=None) == INVALID
    assert _call_verify(lib, B=0) == INVALID
    assert _call_verify(lib, k=0) == INVALID
    assert _call_verify(lib, k=32) == INVALID
    assert _call_verify(lib, V=1) == INVALID
    assert _call_verify(lib, dt=7) == DTYPE
    assert _call_verify(lib, px=1 << 20) == INVALID          # p_at_x without q_at_x
    assert _call_verify(lib, us=1 << 20) == INVALID          # u_smp without out_tok
    assert _call_verify(lib, zb=5) == INVALID                # stride below a batch row
    assert _call_verify(lib, Z=(1 << 20) + 2) == INVALID     # misaligned fp32 pointer
    assert _call_verify(lib, ws=(1 << 20) + 64) == INVALID   # workspace not 256-aligned
    assert _call_verify(lib, wsb=16) == WS


@needs_no_gpu
def test_fork_and_cache_reject_bad_arguments_on_host(lib):
    P = 1 << 20
    # f >= V, f > 16, M > 64
    assert lib.ssd_forked_recovery(P, 8, 0, 1, 2, 4, 4, None, 0, P, P, P, 1 << 30, None) == 1
    assert lib.ssd_forked_recovery(P, 8 * 40, 0, 1, 2, 40, 17, None, 0, P, P, P, 1 << 30, None) == 1
    assert lib.ssd_forked_recovery(P, 8, 0, 1, 2, 4, 2, P, 65, P, P, P, 1 << 30, None) == 1
    assert lib.ssd_forked_recovery(P, 8, 0, 1, 2, 4, 2, None, 1, P, P, P, 1 << 30, None) == 1
    h = ctypes.c_void_p()
    assert lib.ssd_spec_cache_create(100, 7, ctypes.byref(h)) == 1   # not a power of two
    assert lib.ssd_spec_cache_create(64, 0, ctypes.byref(h)) == 1
    assert lib.ssd_spec_cache_create(64, 7, None) == 1
    assert lib.ssd_spec_cache_lookup(None, P, P, P, 4, P, P, None) == 1
    assert lib.ssd_softmax_temp(None, 0, 1, 8, P, None, P, P, P, P, 1 << 30, None) == 1
    assert lib.ssd_selftest_exp2(None, None, None, 4, None) == 1


def test_exp2_table_is_current(tmp_path):
    sys.path.insert(0, os.path.join(PKG, "csrc"))
    try:
        import gen_exp2_table
    finally:
        sys.path.pop(0)
    p = gen_exp2_table.main(str(tmp_path / "t.inc"))
    assert open(p).read() == open(os.path.join(PKG, "csrc", "exp2_table.inc")).read()


def test_exp2_table_values():
    """The table entries are 2^(j/64) split into two binary32 values."""
    import math
    import struct
    text = open(os.path.join(PKG, "csrc", "exp2_table.inc")).read()
    rows = re.findall(r"\{(\S+)f, (\S+)f\}, // j = (-?\d+)", text)
    assert len(rows) == 64
    for hi, lo, j in rows:
        h, l = float.fromhex(hi), float.fromhex(lo)
        assert struct.unpack("f", struct.pack("f", h))[0] == h
        assert abs(h + l - 2.0 ** (int(j) / 64)) <= 2.0 ** (int(j) / 64) * 2e-15


def test_oracle_and_cuda_path_share_no_code():
    """Neither side imports, includes or links the other."""
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".inc")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "ssd_oracle" not in text, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert "speculative_decoding_verification_70_gb300" not in text, f
            assert "ssd.h" not in text, f


@needs_no_gpu
def test_next_rows_reject_bad_arguments_on_host(lib):
    """Draft-side sampling, the drafted verify, the filtered verify and the
    fan-out calls refuse bad arguments before touching CUDA."""
    INVALID, DTYPE, WS = 1, 2, 6
    P = 1 << 20
    big = 1 << 30
    # ssd_draft_sample(D, d_bstride, dt, B, k, V, row0, rows, T, seed, offset, x, x_bstride,
    #                  f, fork_tok, fork_logit, ws, ws_bytes, stream)
    ok = dict(D=P, db=8 * 1000, dt=0, B=2, k=7, V=1000, row0=0, rows=8, T=P, seed=1, off=0,
              x=P, xb=8, f=0, ft=None, fl=None, ws=P, wsb=big)

    def draft(**kw):
        a = dict(ok)
        a.update(kw)
        return lib.ssd_draft_sample(a["D"], a["db"], a["dt"], a["B"], a["k"], a["V"], a["row0"],
                                    a["rows"], a["T"], a["seed"], a["off"], a["x"], a["xb"],
                                    a["f"], a["ft"], a["fl"], a["ws"], a["wsb"], None)
    assert draft(D=None) == INVALID
    assert draft(dt=5) == DTYPE
    assert draft(rows=9) == INVALID                  # row0 + rows > k + 1
    assert draft(row0=-1) == INVALID
    assert draft(db=100) == INVALID                  # stride below the rows read
    assert draft(xb=3) == INVALID                    # x row stride below rows
    assert draft(f=16) == INVALID                    # f + 1 > 16
    assert draft(f=2) == INVALID                     # forks without outputs
    assert draft(wsb=16) == WS
    assert draft(D=P + 2) == INVALID                 # misaligned
    # ssd_verify_topk(Z, zb, D, db, dt, B, k, V, x, T, K, top_p, u_acc, acc, p, q, us, out,
    #                 ws, wsb, stream)

    def topk(K=8, **kw):
        a = dict(Z=P, zb=3 * 1000, D=P, db=2 * 1000, B=2, k=2, V=1000, ws=P, wsb=big)
        a.update(kw)
        return lib.ssd_verify_topk(a["Z"], a["zb"], a["D"], a["db"], 0, a["B"], a["k"], a["V"],
                                   P, P, K, None, P, P, None, None, None, None, a["ws"],
                                   a["wsb"], None)
    assert topk(K=0) == INVALID
    assert topk(K=33, wsb=16) == WS                  # K > 32: the threshold path's workspace
    assert topk(K=8, V=4, zb=12, db=8, wsb=16) == WS  # K > V keeps every token
    assert topk(K=8, zb=10) == INVALID
    assert topk(K=8, wsb=16) == WS
    assert lib.ssd_topk_workspace_bytes(2, 2, 1000, 0) == 0
    n32 = lib.ssd_topk_workspace_bytes(2, 2, 1000, 32)
    n33 = lib.ssd_topk_workspace_bytes(2, 2, 1000, 33)
    assert n32 > 0 and n33 > 0 and n33 != n32
    assert lib.ssd_topk_workspace_bytes(2, 2, 1000, 1 << 30) == lib.ssd_topk_workspace_bytes(2, 2, 1000, 1000)
    assert lib.ssd_topk_workspace_bytes(2, 2, (1 << 21) + 8, 64) == 0   # V beyond the threshold path
    # the drafted verify checks like ssd_verify
    assert lib.ssd_verify_drafted(None, 3000, P, 2000, 0, 2, 2, 1000, P, P, P, P, None, None,
                                  None, None, P, big, None) == INVALID
    # fan-out: F as f
    assert lib.ssd_forked_recovery_fanout(P, 8 * 40, 0, 1, 2, 40, 17, P, None, 0, P, P, P, big,
                                          None) == INVALID


@needs_no_gpu
def test_tree_rejects_bad_arguments_on_host(lib):
    """ssd_verify_tree refuses bad arguments before touching CUDA."""
    INVALID, DTYPE, WS = 1, 2, 6
    P = 1 << 20
    big = 1 << 30
    # ssd_verify_tree(Z, zb, D, db, dt, B, N, V, parent, tok, T, u_acc, u_smp, acc, out_tok,
    #                 out_node, ws, ws_bytes, stream)
    ok = dict(Z=P, zb=5 * 1000, D=P, db=5 * 1000, dt=0, B=2, N=5, V=1000, par=P, tok=P, T=P,
              ua=P, us=P, acc=P, out=P, node=None, ws=P, wsb=big)

    def tree(**kw):
        a = dict(ok)
        a.update(kw)
        return lib.ssd_verify_tree(a["Z"], a["zb"], a["D"], a["db"], a["dt"], a["B"], a["N"],
                                   a["V"], a["par"], a["tok"], a["T"], a["ua"], a["us"],
                                   a["acc"], a["out"], a["node"], a["ws"], a["wsb"], None)
    assert tree(dt=7) == DTYPE
    for key in ("Z", "D", "par", "tok", "T", "ua", "us", "acc", "out", "ws"):
        assert tree(**{key: None}) == INVALID, key
    assert tree(N=0) == INVALID
    assert tree(N=65, zb=65 * 1000, db=65 * 1000) == INVALID   # at most 64 nodes
    assert tree(V=1) == INVALID
    assert tree(zb=4 * 1000) == INVALID                        # stride below N * V
    assert tree(db=4 * 1000) == INVALID
    assert tree(Z=P + 2) == INVALID                            # misaligned
    assert tree(ws=P + 16) == INVALID
    assert tree(wsb=16) == WS
    assert lib.ssd_tree_workspace_bytes(2, 65, 1000) == 0
    assert lib.ssd_tree_workspace_bytes(2, 0, 1000) == 0
    n = lib.ssd_tree_workspace_bytes(2, 5, 1000)
    assert n > 0 and n % 256 == 0
    assert lib.ssd_tree_workspace_bytes(4, 5, 1000) > n


def test_split_override_is_checked_and_restored(lib):
    """ssd_set_split refuses negative values, changes the workspace layout
    while set, and 0 restores the policy."""
    assert lib.ssd_set_split(-1, 0) == 1
    assert lib.ssd_set_split(0, -1) == 1
    n0 = lib.ssd_workspace_bytes(8, 7, 151936, 4)
    try:
        assert lib.ssd_set_split(600, 0) == 0    # more chunks than the policy's 19
        assert lib.ssd_workspace_bytes(8, 7, 151936, 4) > n0
        assert lib.ssd_set_split(1, 0) == 0      # clamped to ceil(V / 256): 256 chunks
        n256 = lib.ssd_workspace_bytes(8, 7, 151936, 4)
        assert lib.ssd_set_split(100000, 0) == 0  # clamped to 32 KB of fp32 logits
        assert lib.ssd_workspace_bytes(8, 7, 151936, 4) <= n0 < n256
    finally:
        assert lib.ssd_set_split(0, 0) == 0
    assert lib.ssd_workspace_bytes(8, 7, 151936, 4) == n0
