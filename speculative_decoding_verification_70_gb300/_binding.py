"""ctypes binding of libssd_gb300.so (include/ssd.h).

Argument marshalling only: torch supplies device memory and the current
stream; every step of the verify-and-recover path runs in the library's CUDA
kernels.  There is no CPU fallback: if the library is missing or a tensor is
not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssd_gb300.so")

SSD_F32 = 0
SSD_BF16 = 1
STATUS = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED_DTYPE",
          3: "SSD_ERR_CUDA", 4: "SSD_ERR_CACHE_FULL", 5: "SSD_ERR_TIMEOUT",
          6: "SSD_ERR_WORKSPACE"}
DEVERR_BAD_TEMPERATURE = 0x1
DEVERR_BAD_LOGITS = 0x2
DEVERR_BAD_TOKEN = 0x4
DEVERR_CACHE_FULL = 0x8
DEVERR_TIMEOUT = 0x10
DEVERR_FILTER_BAND = 0x20

# (name, restype, argtypes)
_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_Z = ctypes.c_size_t
SIGNATURES = [
    ("ssd_status_string", ctypes.c_char_p, [_I]),
    ("ssd_version", _I, []),
    ("ssd_workspace_bytes", _Z, [_I, _I, _I, _I]),
    ("ssd_softmax_workspace_bytes", _Z, [_I, _I]),
    ("ssd_workspace_init", _I, [_P, _Z, _P]),
    ("ssd_get_device_error", _I, [_P, _P, _P, _I]),
    ("ssd_softmax_temp", _I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _Z, _P]),
    ("ssd_verify", _I, [_P, _L, _P, _L, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P,
                        _P, _Z, _P]),
    ("ssd_sample_residual", _I, [_P, _L, _P, _L, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                                 _Z, _P]),
    ("ssd_forked_recovery", _I, [_P, _L, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P, _Z, _P]),
    ("ssd_verify_fork", _I, [_P, _L, _P, _L, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                             _P, _I, _P, _I, _P, _P, _P, _Z, _P]),
    ("ssd_forked_recovery_fanout", _I, [_P, _L, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P,
                                        _Z, _P]),
    ("ssd_verify_fork_fanout", _I, [_P, _L, _P, _L, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                                    _P, _P, _I, _P, _P, _I, _P, _P, _P, _Z, _P]),
    ("ssd_draft_sample", _I, [_P, _L, _I, _I, _I, _I, _I, _I, _P, ctypes.c_uint64,
                              ctypes.c_uint32, _P, _L, _I, _P, _P, _P, _Z, _P]),
    ("ssd_verify_drafted", _I, [_P, _L, _P, _L, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                _P, _P, _Z, _P]),
    ("ssd_topk_workspace_bytes", _Z, [_I, _I, _I, _I]),
    ("ssd_verify_topk", _I, [_P, _L, _P, _L, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P, _P,
                             _P, _P, _P, _Z, _P]),
    ("ssd_tree_workspace_bytes", _Z, [_I, _I, _I]),
    ("ssd_verify_tree", _I, [_P, _L, _P, _L, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P,
                             _P, _Z, _P]),
    ("ssd_verify_fork_cache", _I, [_P, _L, _P, _L, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                   _P, _I, _P, _I, _P, _P, _P, _I, _P, _P, _P, _P, _Z, _P]),
    ("ssd_spec_cache_create", _I, [_I, _I, _P]),
    ("ssd_spec_cache_destroy", None, [_P]),
    ("ssd_spec_cache_clear", _I, [_P, _P]),
    ("ssd_spec_cache_insert", _I, [_P, _P, _P, _P, _P, _I, _P]),
    ("ssd_spec_cache_lookup", _I, [_P, _P, _P, _P, _I, _P, _P, _P]),
    ("ssd_spec_cache_insert_forks", _I, [_P, _P, _I, _I, _I, _P, _P]),
    ("ssd_spec_cache_lookup_outcome", _I, [_P, _P, _P, _I, _I, _P, _P, _P]),
    ("ssd_spec_cache_get_error", _I, [_P, _P, _P, _I]),
    ("ssd_spec_cache_capacity", _I, [_P]),
    ("ssd_spec_cache_depth", _I, [_P]),
    ("ssd_selftest_exp2", _I, [_P, _P, _P, _I, _P]),
    ("ssd_verify_noalloc", _I, [_P, _L, _P, _L, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                _P, _P]),
    ("ssd_set_split", _I, [_I, _I]),
    ("ssd_set_chain_batch", _I, [_I]),
    ("ssd_set_step_schedule", _I, [_I, _I]),
    ("ssd_profile_begin", _I, [_I]),
    ("ssd_profile_end", _I, [_P, _I, _P]),
]


class ProfileEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 40), ("launches", ctypes.c_int),
                ("timed", ctypes.c_int), ("total_ms", ctypes.c_double)]

_lib = None


def load_library(path: Optional[str] = None):
    """Load the C-ABI library (raises if it is missing)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            "libssd_gb300.so is not built (%s); run __graft_entry__.build() or "
            "python -m speculative_decoding_verification_70_gb300.build" % p)
    lib = ctypes.CDLL(p)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


class SSDError(RuntimeError):
    def __init__(self, name: str, status: int):
        lib = load_library()
        msg = lib.ssd_status_string(status).decode()
        super().__init__("%s failed: %s (%s)" % (name, STATUS.get(status, status), msg))
        self.status = status


def _check(name: str, status: int):
    if status != 0:
        raise SSDError(name, status)


def _dev(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (the library has no CPU path)" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _opt(t: Optional[torch.Tensor], name: str):
    return None if t is None else _dev(t, name)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSD_F32
    if t.dtype == torch.bfloat16:
        return SSD_BF16
    raise TypeError("logits must be float32 or bfloat16, got %s" % t.dtype)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream if hasattr(s, "cuda_stream") else int(s)


def _want(t: torch.Tensor, dtype: torch.dtype, name: str):
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))


# ---------------------------------------------------------------------------
# workspace
# ---------------------------------------------------------------------------
def workspace_bytes(B: int, k: int, V: int, f: int = 0) -> int:
    return int(load_library().ssd_workspace_bytes(B, k, V, f))


def softmax_workspace_bytes(rows: int, V: int) -> int:
    return int(load_library().ssd_softmax_workspace_bytes(rows, V))


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled device workspace (torch memory, 256-byte aligned)."""
    if nbytes <= 0:
        raise ValueError("invalid workspace size")
    return torch.zeros(int(nbytes) + 256, dtype=torch.uint8, device=device)


def _ws_ptr(ws: torch.Tensor):
    p = _dev(ws, "ws")
    off = (-p) % 256
    return p + off, ws.numel() - off


def get_device_error(ws: torch.Tensor, clear: bool = False, stream=None) -> int:
    p, _ = _ws_ptr(ws)
    out = ctypes.c_int32(0)
    _check("ssd_get_device_error",
           load_library().ssd_get_device_error(p, _stream(stream), ctypes.byref(out), int(clear)))
    return int(out.value)


# ---------------------------------------------------------------------------
# the five calls
# ---------------------------------------------------------------------------
def ssd_softmax_temp(logits: torch.Tensor, T: torch.Tensor, want_probs: bool = True, *,
                     ws: Optional[torch.Tensor] = None, stream=None) -> Dict[str, torch.Tensor]:
    """Temperature softmax per row of a [rows, V] tensor (T == 0: greedy)."""
    lib = load_library()
    rows, V = logits.shape
    _want(T, torch.float32, "T")
    dev = logits.device
    if ws is None:
        ws = new_workspace(softmax_workspace_bytes(rows, V), dev)
    wp, wn = _ws_ptr(ws)
    probs = torch.empty((rows, V), dtype=torch.float32, device=dev) if want_probs else None
    m = torch.empty(rows, dtype=torch.float32, device=dev)
    s = torch.empty(rows, dtype=torch.float32, device=dev)
    a = torch.empty(rows, dtype=torch.int32, device=dev)
    _check("ssd_softmax_temp", lib.ssd_softmax_temp(
        _dev(logits, "logits"), _dtype_code(logits), rows, V, _dev(T, "T"),
        _opt(probs, "probs"), _dev(m, "row_max"), _dev(s, "row_sum"), _dev(a, "row_argmax"),
        wp, wn, _stream(stream)))
    return {"probs": probs, "row_max": m, "row_sum": s, "row_argmax": a, "ws": ws}


def _verify_outputs(B, k, dev, out, sample: bool, f: int = 0, P: int = 0):
    out = {} if out is None else out
    if "accept_len" not in out:
        out["accept_len"] = torch.empty(B, dtype=torch.int32, device=dev)
        out["p_at_x"] = torch.empty((B, k), dtype=torch.float32, device=dev)
        out["q_at_x"] = torch.empty((B, k), dtype=torch.float32, device=dev)
        out["out_tok"] = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if f and "fork_tok" not in out:
        out["fork_tok"] = torch.empty((B, P, f), dtype=torch.int32, device=dev)
        out["fork_logit"] = torch.empty((B, P, f), dtype=torch.float32, device=dev)
    return out


def ssd_verify(Z: torch.Tensor, D: torch.Tensor, x: torch.Tensor, T: torch.Tensor,
               u_acc: torch.Tensor, u_smp: Optional[torch.Tensor] = None, *,
               drafted: bool = False, ws: Optional[torch.Tensor] = None,
               out: Optional[dict] = None, stream=None) -> Dict[str, torch.Tensor]:
    """Acceptance, first-reject prefix and (if u_smp is given) the recovery or
    bonus draw.  Z [B,k+1,V], D [B,>=k,V] (same dtype), x [B,k] int32,
    T [B], u_acc [B,k], u_smp [B] float32.  drafted: the draft rows'
    statistics are already in ws (ssd_draft_sample with the same ws)."""
    lib = load_library()
    B, kp1, V = Z.shape
    k = kp1 - 1
    if D.dim() != 3 or D.shape[0] != B or D.shape[2] != V or D.shape[1] < k:
        raise ValueError("D must be [B, >=k, V]")
    if Z.dtype != D.dtype:
        raise TypeError("Z and D must share a dtype")
    for t, n in ((x, "x"),):
        _want(t, torch.int32, n)
    for t, n in ((T, "T"), (u_acc, "u_acc")):
        _want(t, torch.float32, n)
    dev = Z.device
    if drafted and ws is None:
        raise ValueError("drafted=True needs the workspace of ssd_draft_sample")
    if ws is None:
        ws = new_workspace(workspace_bytes(B, k, V, 0), dev)
    wp, wn = _ws_ptr(ws)
    o = _verify_outputs(B, k, dev, out, u_smp is not None)
    fn = lib.ssd_verify_drafted if drafted else lib.ssd_verify
    _check("ssd_verify_drafted" if drafted else "ssd_verify", fn(
        _dev(Z, "Z"), kp1 * V, _dev(D, "D"), D.shape[1] * V, _dtype_code(Z), B, k, V,
        _dev(x, "x"), _dev(T, "T"), _dev(u_acc, "u_acc"), _dev(o["accept_len"], "accept_len"),
        _dev(o["p_at_x"], "p_at_x"), _dev(o["q_at_x"], "q_at_x"), _opt(u_smp, "u_smp"),
        _dev(o["out_tok"], "out_tok"), wp, wn, _stream(stream)))
    o["ws"] = ws
    return o


def ssd_sample_residual(Z: torch.Tensor, D: torch.Tensor, x: torch.Tensor, T: torch.Tensor,
                        accept_len: torch.Tensor, u_smp: torch.Tensor, ws: torch.Tensor, *,
                        out_tok: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The recovery/bonus draw after an ssd_verify call (u_smp=None) that used
    the same workspace."""
    lib = load_library()
    B, kp1, V = Z.shape
    k = kp1 - 1
    _want(accept_len, torch.int32, "accept_len")
    if out_tok is None:
        out_tok = torch.empty((B, k + 1), dtype=torch.int32, device=Z.device)
    wp, wn = _ws_ptr(ws)
    _check("ssd_sample_residual", lib.ssd_sample_residual(
        _dev(Z, "Z"), kp1 * V, _dev(D, "D"), D.shape[1] * V, _dtype_code(Z), B, k, V,
        _dev(x, "x"), _dev(T, "T"), _dev(accept_len, "accept_len"), _dev(u_smp, "u_smp"),
        _dev(out_tok, "out_tok"), wp, wn, _stream(stream)))
    return out_tok


def ssd_forked_recovery(L: torch.Tensor, f: int, mask: Optional[torch.Tensor] = None, *,
                        fanout: Optional[torch.Tensor] = None,
                        ws: Optional[torch.Tensor] = None, out: Optional[dict] = None,
                        stream=None) -> Dict[str, torch.Tensor]:
    """Top-f forked recovery tokens per (b, j) of L [B,P,V], skipping the
    tokens in mask [B,P,M] (int32, -1 = none).  fanout [P] int32 (device)
    keeps f_j <= f tokens at position j."""
    lib = load_library()
    B, P, V = L.shape
    dev = L.device
    M = 0 if mask is None else mask.shape[2]
    if mask is not None:
        _want(mask, torch.int32, "mask")
    if ws is None:
        ws = new_workspace(workspace_bytes(B, P - 1, V, f), dev)
    wp, wn = _ws_ptr(ws)
    out = {} if out is None else out
    if "fork_tok" not in out:
        out["fork_tok"] = torch.empty((B, P, f), dtype=torch.int32, device=dev)
        out["fork_logit"] = torch.empty((B, P, f), dtype=torch.float32, device=dev)
    if fanout is None:
        _check("ssd_forked_recovery", lib.ssd_forked_recovery(
            _dev(L, "L"), P * V, _dtype_code(L), B, P, V, f, _opt(mask, "mask"), M,
            _dev(out["fork_tok"], "fork_tok"), _dev(out["fork_logit"], "fork_logit"), wp, wn,
            _stream(stream)))
    else:
        _want(fanout, torch.int32, "fanout")
        if fanout.numel() != P:
            raise ValueError("fanout must hold P values")
        _check("ssd_forked_recovery_fanout", lib.ssd_forked_recovery_fanout(
            _dev(L, "L"), P * V, _dtype_code(L), B, P, V, f, _dev(fanout, "fanout"),
            _opt(mask, "mask"), M, _dev(out["fork_tok"], "fork_tok"),
            _dev(out["fork_logit"], "fork_logit"), wp, wn, _stream(stream)))
    out["ws"] = ws
    return out


def ssd_verify_fork_cache(Z: torch.Tensor, D: torch.Tensor, x: torch.Tensor, T: torch.Tensor,
                          u_acc: torch.Tensor, u_smp: Optional[torch.Tensor], f: int,
                          mask: Optional[torch.Tensor], cache: "SpecCache",
                          payload: torch.Tensor, *, clear: bool = True,
                          ws: Optional[torch.Tensor] = None, out: Optional[dict] = None,
                          stream=None) -> Dict[str, torch.Tensor]:
    """One SSD round step: ssd_verify_fork, the forks inserted into `cache`
    (cleared first when clear) with payload [B*(k+1)*f, depth], and each
    row's realised outcome looked up: out["hit"] [B], out["tok_out"]
    [B, depth]."""
    lib = load_library()
    B, kp1, V = Z.shape
    k = kp1 - 1
    if tuple(D.shape) != (B, kp1, V):
        raise ValueError("D must be [B, k+1, V] for the fused call")
    if Z.dtype != D.dtype:
        raise TypeError("Z and D must share a dtype")
    _want(x, torch.int32, "x")
    _want(payload, torch.int32, "payload")
    if tuple(payload.shape) != (B * kp1 * f, cache.depth):
        raise ValueError("payload must be [B*(k+1)*f, depth]")
    M = 0 if mask is None else mask.shape[2]
    dev = Z.device
    if ws is None:
        ws = new_workspace(workspace_bytes(B, k, V, f), dev)
    wp, wn = _ws_ptr(ws)
    o = _verify_outputs(B, k, dev, out, True, f, kp1)
    if "hit" not in o:
        o["hit"] = torch.empty(B, dtype=torch.int32, device=dev)
        o["tok_out"] = torch.empty((B, cache.depth), dtype=torch.int32, device=dev)
    _check("ssd_verify_fork_cache", lib.ssd_verify_fork_cache(
        _dev(Z, "Z"), kp1 * V, _dev(D, "D"), kp1 * V, _dtype_code(Z), B, k, V,
        _dev(x, "x"), _dev(T, "T"), _dev(u_acc, "u_acc"), _dev(o["accept_len"], "accept_len"),
        _dev(o["p_at_x"], "p_at_x"), _dev(o["q_at_x"], "q_at_x"), _opt(u_smp, "u_smp"),
        _dev(o["out_tok"], "out_tok"), f, _opt(mask, "mask"), M,
        _dev(o["fork_tok"], "fork_tok"), _dev(o["fork_logit"], "fork_logit"), cache._h,
        int(clear), _dev(payload, "payload"), _dev(o["hit"], "hit"),
        _dev(o["tok_out"], "tok_out"), wp, wn, _stream(stream)))
    o["ws"] = ws
    return o


def ssd_verify_fork(Z: torch.Tensor, D: torch.Tensor, x: torch.Tensor, T: torch.Tensor,
                    u_acc: torch.Tensor, u_smp: Optional[torch.Tensor], f: int,
                    mask: Optional[torch.Tensor] = None, *,
                    fanout: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                    out: Optional[dict] = None, stream=None) -> Dict[str, torch.Tensor]:
    """ssd_verify plus the forked recovery over the SSD draft D [B,k+1,V] in
    one pass over the logits (fanout [k+1] int32: f_j <= f forks at j)."""
    lib = load_library()
    B, kp1, V = Z.shape
    k = kp1 - 1
    if tuple(D.shape) != (B, kp1, V):
        raise ValueError("D must be [B, k+1, V] for the fused call")
    if Z.dtype != D.dtype:
        raise TypeError("Z and D must share a dtype")
    _want(x, torch.int32, "x")
    M = 0 if mask is None else mask.shape[2]
    dev = Z.device
    if ws is None:
        ws = new_workspace(workspace_bytes(B, k, V, f), dev)
    wp, wn = _ws_ptr(ws)
    o = _verify_outputs(B, k, dev, out, u_smp is not None, f, kp1)
    head = (_dev(Z, "Z"), kp1 * V, _dev(D, "D"), kp1 * V, _dtype_code(Z), B, k, V,
            _dev(x, "x"), _dev(T, "T"), _dev(u_acc, "u_acc"), _dev(o["accept_len"], "accept_len"),
            _dev(o["p_at_x"], "p_at_x"), _dev(o["q_at_x"], "q_at_x"), _opt(u_smp, "u_smp"),
            _dev(o["out_tok"], "out_tok"), f)
    tail = (_opt(mask, "mask"), M, _dev(o["fork_tok"], "fork_tok"),
            _dev(o["fork_logit"], "fork_logit"), wp, wn, _stream(stream))
    if fanout is None:
        _check("ssd_verify_fork", lib.ssd_verify_fork(*head, *tail))
    else:
        _want(fanout, torch.int32, "fanout")
        if fanout.numel() != kp1:
            raise ValueError("fanout must hold k+1 values")
        _check("ssd_verify_fork_fanout",
               lib.ssd_verify_fork_fanout(*head, _dev(fanout, "fanout"), *tail))
    o["ws"] = ws
    return o


def ssd_draft_sample(D: torch.Tensor, T: torch.Tensor, k: int, seed: int, offset: int, *,
                     row0: int = 0, rows: Optional[int] = None, f: int = 0,
                     ws: Optional[torch.Tensor] = None, out: Optional[dict] = None,
                     stream=None) -> Dict[str, torch.Tensor]:
    """Draw the drafter's tokens for rows [row0, row0 + rows) of D [B, Pd, V]
    (Gumbel-max with Philox4x32-10 uniforms; argmax at T == 0) and keep the
    rows' statistics in ws for ssd_verify(..., drafted=True).  With f > 0
    also the f forks per row (top-f logits other than the drafted token)."""
    lib = load_library()
    B, Pd, V = D.shape
    rows = Pd - row0 if rows is None else rows
    _want(T, torch.float32, "T")
    dev = D.device
    if ws is None:
        ws = new_workspace(workspace_bytes(B, k, V, f + 1 if f > 0 else 0), dev)
    wp, wn = _ws_ptr(ws)
    out = {} if out is None else out
    if "x" not in out:
        out["x"] = torch.empty((B, rows), dtype=torch.int32, device=dev)
        if f > 0:
            out["fork_tok"] = torch.empty((B, rows, f), dtype=torch.int32, device=dev)
            out["fork_logit"] = torch.empty((B, rows, f), dtype=torch.float32, device=dev)
    _check("ssd_draft_sample", lib.ssd_draft_sample(
        _dev(D, "D"), Pd * V, _dtype_code(D), B, k, V, row0, rows, _dev(T, "T"),
        seed & 0xFFFFFFFFFFFFFFFF, offset & 0xFFFFFFFF, _dev(out["x"], "x"), rows, f,
        _opt(out.get("fork_tok"), "fork_tok"), _opt(out.get("fork_logit"), "fork_logit"),
        wp, wn, _stream(stream)))
    out["ws"] = ws
    return out


def ssd_verify_topk(Z: torch.Tensor, D: torch.Tensor, x: torch.Tensor, T: torch.Tensor,
                    K: int, top_p: Optional[torch.Tensor], u_acc: torch.Tensor,
                    u_smp: Optional[torch.Tensor] = None, *, ws: Optional[torch.Tensor] = None,
                    out: Optional[dict] = None, stream=None) -> Dict[str, torch.Tensor]:
    """ssd_verify over top-K / top-p filtered target and draft distributions
    (any K >= 1, K >= V for top-p over the whole vocabulary; top_p [B]
    float32 or None)."""
    lib = load_library()
    B, kp1, V = Z.shape
    k = kp1 - 1
    if D.dim() != 3 or D.shape[0] != B or D.shape[2] != V or D.shape[1] < k:
        raise ValueError("D must be [B, >=k, V]")
    if Z.dtype != D.dtype:
        raise TypeError("Z and D must share a dtype")
    _want(x, torch.int32, "x")
    if top_p is not None:
        _want(top_p, torch.float32, "top_p")
    dev = Z.device
    if ws is None:
        n = lib.ssd_topk_workspace_bytes(B, k, V, K)
        if n == 0:
            raise SSDError("ssd_topk_workspace_bytes", 1)
        ws = new_workspace(n, dev)
    wp, wn = _ws_ptr(ws)
    o = _verify_outputs(B, k, dev, out, u_smp is not None)
    _check("ssd_verify_topk", lib.ssd_verify_topk(
        _dev(Z, "Z"), kp1 * V, _dev(D, "D"), D.shape[1] * V, _dtype_code(Z), B, k, V,
        _dev(x, "x"), _dev(T, "T"), K, _opt(top_p, "top_p"), _dev(u_acc, "u_acc"),
        _dev(o["accept_len"], "accept_len"), _dev(o["p_at_x"], "p_at_x"),
        _dev(o["q_at_x"], "q_at_x"), _opt(u_smp, "u_smp"), _dev(o["out_tok"], "out_tok"),
        wp, wn, _stream(stream)))
    o["ws"] = ws
    return o


def ssd_verify_tree(Z: torch.Tensor, D: torch.Tensor, parent: torch.Tensor,
                    tok: torch.Tensor, T: torch.Tensor, u_acc: torch.Tensor,
                    u_smp: torch.Tensor, *, ws: Optional[torch.Tensor] = None,
                    out: Optional[dict] = None, stream=None) -> Dict[str, torch.Tensor]:
    """Verify a draft token tree per batch row (multi-step speculative
    sampling; greedy at T == 0).  Z, D: [B, N, V] target and draft logits at
    the N nodes (a leaf's draft row is not read); parent, tok: [B, N] int32
    (parent[:, 0] == -1, parent[:, j] < j); u_acc: [B, N] float32 (entry j
    tests node j), u_smp: [B].

    Returns accept_len [B], out_tok [B, N] (accepted tokens, the final
    token, then -1) and out_node [B, N] (accepted node ids, then -1)."""
    lib = load_library()
    if Z.dim() != 3 or D.shape != Z.shape:
        raise ValueError("Z and D must both be [B, N, V]")
    if Z.dtype != D.dtype:
        raise TypeError("Z and D must share a dtype")
    B, N, V = Z.shape
    for t, name in ((parent, "parent"), (tok, "tok")):
        _want(t, torch.int32, name)
        if t.shape != (B, N):
            raise ValueError("%s must be [B, N]" % name)
    _want(T, torch.float32, "T")
    _want(u_acc, torch.float32, "u_acc")
    _want(u_smp, torch.float32, "u_smp")
    dev = Z.device
    if ws is None:
        n = lib.ssd_tree_workspace_bytes(B, N, V)
        if n == 0:
            raise SSDError("ssd_tree_workspace_bytes", 1)
        ws = new_workspace(n, dev)
    wp, wn = _ws_ptr(ws)
    o = {} if out is None else out
    if "accept_len" not in o:
        o["accept_len"] = torch.empty(B, dtype=torch.int32, device=dev)
        o["out_tok"] = torch.empty((B, N), dtype=torch.int32, device=dev)
        o["out_node"] = torch.empty((B, N), dtype=torch.int32, device=dev)
    _check("ssd_verify_tree", lib.ssd_verify_tree(
        _dev(Z, "Z"), N * V, _dev(D, "D"), N * V, _dtype_code(Z), B, N, V,
        _dev(parent, "parent"), _dev(tok, "tok"), _dev(T, "T"), _dev(u_acc, "u_acc"),
        _dev(u_smp, "u_smp"), _dev(o["accept_len"], "accept_len"),
        _dev(o["out_tok"], "out_tok"), _dev(o["out_node"], "out_node"), wp, wn,
        _stream(stream)))
    o["ws"] = ws
    return o


class SpecCache:
    """Device speculation cache: key (b, position, token) -> depth tokens."""

    def __init__(self, capacity: int, depth: int):
        self._lib = load_library()
        h = ctypes.c_void_p()
        _check("ssd_spec_cache_create",
               self._lib.ssd_spec_cache_create(capacity, depth, ctypes.byref(h)))
        self._h = h
        self.capacity = capacity
        self.depth = depth

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            self._lib.ssd_spec_cache_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def clear(self, stream=None):
        _check("ssd_spec_cache_clear", self._lib.ssd_spec_cache_clear(self._h, _stream(stream)))

    def insert(self, b, pos, tok, payload, stream=None):
        n = b.numel()
        _check("ssd_spec_cache_insert", self._lib.ssd_spec_cache_insert(
            self._h, _dev(b, "b"), _dev(pos, "pos"), _dev(tok, "tok"), _dev(payload, "payload"),
            n, _stream(stream)))

    def insert_forks(self, fork_tok, payload, stream=None):
        B, P, f = fork_tok.shape
        _check("ssd_spec_cache_insert_forks", self._lib.ssd_spec_cache_insert_forks(
            self._h, _dev(fork_tok, "fork_tok"), B, P, f, _dev(payload, "payload"),
            _stream(stream)))

    def lookup(self, b, pos, tok, out=None, stream=None):
        n = b.numel()
        dev = b.device
        out = out or {"hit": torch.empty(n, dtype=torch.int32, device=dev),
                      "tok_out": torch.empty((n, self.depth), dtype=torch.int32, device=dev)}
        _check("ssd_spec_cache_lookup", self._lib.ssd_spec_cache_lookup(
            self._h, _dev(b, "b"), _dev(pos, "pos"), _dev(tok, "tok"), n,
            _dev(out["hit"], "hit"), _dev(out["tok_out"], "tok_out"), _stream(stream)))
        return out

    def lookup_outcome(self, accept_len, out_tok, out=None, stream=None):
        B, kp1 = out_tok.shape
        dev = out_tok.device
        out = out or {"hit": torch.empty(B, dtype=torch.int32, device=dev),
                      "tok_out": torch.empty((B, self.depth), dtype=torch.int32, device=dev)}
        _check("ssd_spec_cache_lookup_outcome", self._lib.ssd_spec_cache_lookup_outcome(
            self._h, _dev(accept_len, "accept_len"), _dev(out_tok, "out_tok"), B, kp1 - 1,
            _dev(out["hit"], "hit"), _dev(out["tok_out"], "tok_out"), _stream(stream)))
        return out

    def error(self, clear: bool = False, stream=None) -> int:
        v = ctypes.c_int32(0)
        _check("ssd_spec_cache_get_error", self._lib.ssd_spec_cache_get_error(
            self._h, _stream(stream), ctypes.byref(v), int(clear)))
        return int(v.value)


def selftest_exp2(x_hi: torch.Tensor, x_lo: torch.Tensor, stream=None) -> torch.Tensor:
    out = torch.empty(x_hi.numel(), dtype=torch.float64, device=x_hi.device)
    _check("ssd_selftest_exp2", load_library().ssd_selftest_exp2(
        _dev(x_hi, "x_hi"), _dev(x_lo, "x_lo"), _dev(out, "out"), x_hi.numel(), _stream(stream)))
    return out


def set_split(chunk_elems: int = 0, chunks_per_cta: int = 0):
    """Override the vocabulary split (elements per chunk, chunks per
    statistics CTA; 0 = the library's policy) for later calls in this
    process.  Integer results do not depend on it."""
    _check("ssd_set_split", load_library().ssd_set_split(int(chunk_elems), int(chunks_per_cta)))


def set_chain_batch(max_b: int = -1):
    """Largest batch whose verify tail (finalisation, draw, cache step) runs
    as the one cluster kernel; 0 disables it, negative restores the default
    (16).  Process-wide, for later calls."""
    _check("ssd_set_chain_batch", load_library().ssd_set_chain_batch(int(max_b)))


def set_step_schedule(max_b: int = -1, max_grid: int = 0):
    """Largest batch whose whole verify call runs as the one cooperative
    kernel (0 disables it, negative restores the default of 4; at most 8),
    and a cap on that kernel's CTAs (0: as many as the GPU holds).
    Process-wide, for later calls."""
    _check("ssd_set_step_schedule",
           load_library().ssd_set_step_schedule(int(max_b), int(max_grid)))


def profile_begin(max_launches: int = 4096):
    """Start bracketing every library kernel launch with CUDA events."""
    _check("ssd_profile_begin", load_library().ssd_profile_begin(max_launches))


def profile_end() -> Dict[str, dict]:
    """Stop profiling; returns {kernel: {launches, timed, total_ms}}."""
    arr = (ProfileEntry * 64)()
    n = ctypes.c_int(0)
    _check("ssd_profile_end", load_library().ssd_profile_end(arr, 64, ctypes.byref(n)))
    return {arr[i].name.decode(): {"launches": arr[i].launches, "timed": arr[i].timed,
                                   "total_ms": arr[i].total_ms} for i in range(n.value)}
