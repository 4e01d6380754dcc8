"""CPU oracle for the speculative-decoding verify-and-recover step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (the CUDA library and its Python binding) never imports it and has no
CPU fallback.

The arithmetic lives in ``ssd_oracle.c`` (scalar C, double precision, plain
loops in the method's own order); this module only compiles and loads it
with ``gcc`` and marshals numpy arrays.  The speculation-cache oracle is a
Python ``dict``: the plain definition of an exact-key map.

Sources followed (cited by page title and section):
  * "tanishqkumar/ssd" summary page, module notes: greedy/stochastic sampler
    selected by temperature; forked recovery tokens by top-k over logits with
    masking for cache hits.
  * "SSD: drafting and verification on separate GPUs", "What changes in SSD":
    verify the draft in one pass; exactness; speculation cache (roadmap).
  * speculative-sampling summary (sourcepulse project 1842340), "How It
    Works": accept, then regenerate from the point of divergence.
  * Leviathan et al. 2023 / Chen et al. 2023: the min(1, p/q) acceptance,
    the norm(max(0, p - q)) residual and the bonus draw from p.
  * "tanishqkumar/ssd" summary page, module notes on tree decoding, with
    SpecInfer's multi-step speculative sampling (Miao et al. 2024) as the
    rule for verifying a token tree.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssd_oracle.so")

F32 = 0
BF16 = 1

_lib = None


def build(force: bool = False) -> str:
    """Compile ssd_oracle.c into libssd_oracle.so next to it (gcc, -O2,
    strict IEEE: no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    i32 = ctypes.c_int
    lib.oracle_softmax_temp.argtypes = [P, i32, i32, i64, P, P, P, P, P]
    lib.oracle_softmax_temp.restype = i32
    lib.oracle_verify_recover.argtypes = [P, i64, P, i64, i32, i32, i32, i64,
                                          P, P, P, P, P, P, P, P]
    lib.oracle_verify_recover.restype = i32
    lib.oracle_verify_recover_f64.argtypes = lib.oracle_verify_recover.argtypes
    lib.oracle_verify_recover_f64.restype = i32
    lib.oracle_forked_topf.argtypes = [P, i64, i32, i32, i32, i64, i32, P, i32,
                                       P, P]
    lib.oracle_forked_topf.restype = i32
    lib.oracle_verify_recover_filtered.argtypes = [P, i64, P, i64, i32, i32, i32, i64, P, P,
                                                   i32, P, P, P, i32, P, P, P, P]
    lib.oracle_verify_recover_filtered.restype = i32
    lib.oracle_verify_tree.argtypes = [P, i64, P, i64, i32, i32, i32, i64, P, P, P, P, P,
                                       P, P, P]
    lib.oracle_verify_tree.restype = i32
    lib.oracle_verify_tree_f64.argtypes = lib.oracle_verify_tree.argtypes
    lib.oracle_verify_tree_f64.restype = i32
    lib.oracle_philox4x32_10.argtypes = [P, P, P]
    lib.oracle_philox4x32_10.restype = None
    u32 = ctypes.c_uint32
    lib.oracle_draft_sample.argtypes = [P, i64, i32, i32, i32, i64, i32, i32, P, u32, u32, u32,
                                        P, i64]
    lib.oracle_draft_sample.restype = i32
    _lib = lib
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a) -> Tuple[np.ndarray, int]:
    """Accept a numpy float32 array, a numpy uint16 array holding bf16 bit
    patterns, or a CPU torch tensor (float32 or bfloat16)."""
    try:
        import torch  # noqa: F401  (only for tensor inputs)
        if isinstance(a, torch.Tensor):
            t = a.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16), BF16
            if t.dtype == torch.float32:
                return t.numpy(), F32
            raise TypeError("oracle takes float32 or bfloat16 logits")
    except ImportError:
        pass
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError("oracle takes float32 logits or bf16 bit patterns (uint16)")


def _check(rc: int, name: str):
    if rc != 0:
        raise RuntimeError("%s failed with oracle status %d" % (name, rc))


def softmax_temp(logits, T) -> Dict[str, np.ndarray]:
    """Temperature softmax per row of a [rows, V] array.

    Returns probs [rows, V] (float64), row_max, row_sum, row_argmax.
    T == 0 rows give a one-hot at the argmax with row_sum 1.
    """
    z, dt = _logits(logits)
    rows, V = z.shape[0], z.shape[-1]
    T = np.ascontiguousarray(T, dtype=np.float32).reshape(rows)
    probs = np.empty((rows, V), dtype=np.float64)
    m = np.empty(rows, dtype=np.float64)
    s = np.empty(rows, dtype=np.float64)
    a = np.empty(rows, dtype=np.int32)
    _check(_load().oracle_softmax_temp(_ptr(z), dt, rows, V, _ptr(T), _ptr(probs),
                                       _ptr(m), _ptr(s), _ptr(a)), "softmax_temp")
    return {"probs": probs, "row_max": m, "row_sum": s, "row_argmax": a}


def verify_recover(Z, D, x, T, u_acc, u_smp, f64_uniforms: bool = False
                   ) -> Dict[str, np.ndarray]:
    """One verify-and-recover step.

    Z: [B, k+1, V] target logits.  D: [B, Pd, V] draft logits with Pd >= k
    (only rows 0..k-1 are read).  x: [B, k] int32 draft tokens.  T: [B].
    u_acc: [B, k], u_smp: [B] uniforms in [0, 1), binary32 as the GPU
    library takes them, or double when f64_uniforms (used to pin the oracle by
    exact enumeration).

    Returns accept_len [B], p_at_x / q_at_x [B, k] (float64) and
    out_tok [B, k+1].
    """
    z, dt = _logits(Z)
    d, dt2 = _logits(D)
    if dt != dt2:
        raise TypeError("Z and D must share a dtype")
    B, kp1, V = z.shape
    k = kp1 - 1
    Pd = d.shape[1]
    if d.shape[0] != B or d.shape[2] != V or Pd < k:
        raise ValueError("D must be [B, >=k, V]")
    x = np.ascontiguousarray(x, dtype=np.int32).reshape(B, k)
    T = np.ascontiguousarray(T, dtype=np.float32).reshape(B)
    udt = np.float64 if f64_uniforms else np.float32
    u_acc = np.ascontiguousarray(u_acc, dtype=udt).reshape(B, k)
    u_smp = np.ascontiguousarray(u_smp, dtype=udt).reshape(B)
    acc = np.empty(B, dtype=np.int32)
    pax = np.empty((B, k), dtype=np.float64)
    qax = np.empty((B, k), dtype=np.float64)
    out = np.empty((B, k + 1), dtype=np.int32)
    fn = _load().oracle_verify_recover_f64 if f64_uniforms else _load().oracle_verify_recover
    _check(fn(
        _ptr(z), kp1 * V, _ptr(d), Pd * V, dt, B, k, V, _ptr(x), _ptr(T),
        _ptr(u_acc), _ptr(u_smp), _ptr(acc), _ptr(pax), _ptr(qax), _ptr(out)),
        "verify_recover")
    return {"accept_len": acc, "p_at_x": pax, "q_at_x": qax, "out_tok": out}


def verify_recover_filtered(Z, D, x, T, K: int, top_p, u_acc, u_smp,
                            f64_uniforms: bool = False) -> Dict[str, np.ndarray]:
    """verify_recover over top-k / top-p filtered target and draft
    distributions (same K and top_p for both; top_p [B] or None): the tokens
    ordered by (logit desc, index asc), the first K kept, then the shortest
    prefix holding >= top_p of their mass, renormalised."""
    z, dt = _logits(Z)
    d, dt2 = _logits(D)
    if dt != dt2:
        raise TypeError("Z and D must share a dtype")
    B, kp1, V = z.shape
    k = kp1 - 1
    Pd = d.shape[1]
    x = np.ascontiguousarray(x, dtype=np.int32).reshape(B, k)
    T = np.ascontiguousarray(T, dtype=np.float32).reshape(B)
    tp = None if top_p is None else np.ascontiguousarray(top_p, dtype=np.float32).reshape(B)
    udt = np.float64 if f64_uniforms else np.float32
    u_acc = np.ascontiguousarray(u_acc, dtype=udt).reshape(B, k)
    u_smp = np.ascontiguousarray(u_smp, dtype=udt).reshape(B)
    acc = np.empty(B, dtype=np.int32)
    pax = np.empty((B, k), dtype=np.float64)
    qax = np.empty((B, k), dtype=np.float64)
    out = np.empty((B, k + 1), dtype=np.int32)
    _check(_load().oracle_verify_recover_filtered(
        _ptr(z), kp1 * V, _ptr(d), Pd * V, dt, B, k, V, _ptr(x), _ptr(T), K, _ptr(tp),
        _ptr(u_acc), _ptr(u_smp), int(f64_uniforms), _ptr(acc), _ptr(pax), _ptr(qax),
        _ptr(out)), "verify_recover_filtered")
    return {"accept_len": acc, "p_at_x": pax, "q_at_x": qax, "out_tok": out}


def verify_tree(Z, D, parent, tok, T, u_acc, u_smp, f64_uniforms: bool = False
                ) -> Dict[str, np.ndarray]:
    """Token-tree verification (multi-step speculative sampling over a tree
    whose children at a node were drawn from the draft's q there).

    Z, D: [B, N, V] target and draft logits at the N nodes (a leaf's draft
    row is not read).  parent, tok:
    [B, N] int32 (parent[:, 0] == -1, parent[:, j] < j; tok[:, 0] unused).
    T: [B].  u_acc: [B, N] (entry j tests node j), u_smp: [B]: binary32 as
    the GPU library takes them, or double when f64_uniforms.

    Returns accept_len [B], out_tok [B, N] (accepted tokens, the final
    token, then -1) and out_node [B, N] (accepted node ids, then -1).
    """
    z, dt = _logits(Z)
    d, dt2 = _logits(D)
    if dt != dt2:
        raise TypeError("Z and D must share a dtype")
    B, N, V = z.shape
    if d.shape != z.shape:
        raise ValueError("D must be [B, N, V] like Z")
    parent = np.ascontiguousarray(parent, dtype=np.int32).reshape(B, N)
    tok = np.ascontiguousarray(tok, dtype=np.int32).reshape(B, N)
    T = np.ascontiguousarray(T, dtype=np.float32).reshape(B)
    udt = np.float64 if f64_uniforms else np.float32
    u_acc = np.ascontiguousarray(u_acc, dtype=udt).reshape(B, N)
    u_smp = np.ascontiguousarray(u_smp, dtype=udt).reshape(B)
    acc = np.empty(B, dtype=np.int32)
    out = np.empty((B, N), dtype=np.int32)
    node = np.empty((B, N), dtype=np.int32)
    fn = _load().oracle_verify_tree_f64 if f64_uniforms else _load().oracle_verify_tree
    _check(fn(
        _ptr(z), N * V, _ptr(d), N * V, dt, B, N, V, _ptr(parent), _ptr(tok), _ptr(T),
        _ptr(u_acc), _ptr(u_smp), _ptr(acc), _ptr(out), _ptr(node)), "verify_tree")
    return {"accept_len": acc, "out_tok": out, "out_node": node}


def forked_topf(L, f: int, mask=None, fanout=None) -> Dict[str, np.ndarray]:
    """Top-f forked recovery tokens per (b, j) of L [B, P, V], skipping the
    tokens listed in mask [B, P, M] (-1 = no entry).

    fanout [P] (variable fan-out, "tanishqkumar/ssd" summary, module notes:
    forked recovery tokens selected by fan-out strategy): position j keeps
    f_j = min(max(fanout[j], 0), f) tokens -- by definition the first f_j of
    its top-f list, since the order is total -- and pads the rest with
    (-1, -inf)."""
    l, dt = _logits(L)
    B, P, V = l.shape
    if mask is None:
        mask = np.full((B, P, 0), -1, dtype=np.int32)
    mask = np.ascontiguousarray(mask, dtype=np.int32)
    M = mask.shape[2]
    tok = np.empty((B, P, f), dtype=np.int32)
    lg = np.empty((B, P, f), dtype=np.float64)
    _check(_load().oracle_forked_topf(_ptr(l), P * V, dt, B, P, V, f,
                                      _ptr(mask) if M > 0 else None, M,
                                      _ptr(tok), _ptr(lg)), "forked_topf")
    if fanout is not None:
        keep = np.clip(np.asarray(fanout, dtype=np.int64).reshape(P), 0, f)
        drop = np.arange(f)[None, :] >= keep[:, None]          # [P, f]
        tok[:, drop] = -1
        lg[:, drop] = -np.inf
    return {"fork_tok": tok, "fork_logit": lg}


def philox4x32_10(ctr, key) -> np.ndarray:
    """Philox4x32-10 of a counter (4 x uint32) and key (2 x uint32)."""
    c = np.ascontiguousarray(ctr, dtype=np.uint32).reshape(4)
    k = np.ascontiguousarray(key, dtype=np.uint32).reshape(2)
    out = np.empty(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def draft_sample(D, T, seed: int, offset: int, row0: int = 0,
                 rows: Optional[int] = None) -> np.ndarray:
    """The drafter's tokens for rows [row0, row0 + rows) of D [B, Pd, V]:
    Gumbel-max draws from softmax(D / T) with Philox4x32-10 uniforms
    (counter (v / 4, row, b, offset), key = the 64-bit seed); argmax at
    T == 0; -1 for invalid T or rows.  Returns x [B, rows] int32."""
    d, dt = _logits(D)
    B, Pd, V = d.shape
    rows = Pd - row0 if rows is None else rows
    T = np.ascontiguousarray(T, dtype=np.float32).reshape(B)
    x = np.empty((B, rows), dtype=np.int32)
    _check(_load().oracle_draft_sample(_ptr(d), Pd * V, dt, B, Pd, V, row0, rows, _ptr(T),
                                       seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF,
                                       offset & 0xFFFFFFFF, _ptr(x), rows), "draft_sample")
    return x


class SpecCacheOracle:
    """The speculation cache as an exact-key map (summary page: cache hits
    and misses; "SSD: drafting and verification on separate GPUs", roadmap:
    speculation cache).  Key (b, position, token) -> the draft continuation.
    Inserts apply in input order, so the last duplicate wins."""

    def __init__(self, depth: int):
        self.depth = depth
        self.table: Dict[Tuple[int, int, int], Tuple[int, ...]] = {}

    def clear(self):
        self.table.clear()

    def insert(self, b: Sequence[int], pos: Sequence[int], tok: Sequence[int],
               payload: np.ndarray):
        payload = np.asarray(payload).reshape(len(b), self.depth)
        for i in range(len(b)):
            self.table[(int(b[i]), int(pos[i]), int(tok[i]))] = tuple(
                int(v) for v in payload[i])

    def lookup(self, b: Sequence[int], pos: Sequence[int], tok: Sequence[int]):
        n = len(b)
        hit = np.zeros(n, dtype=np.int32)
        out = np.full((n, self.depth), -1, dtype=np.int32)
        for i in range(n):
            key = (int(b[i]), int(pos[i]), int(tok[i]))
            if key in self.table:
                hit[i] = 1
                out[i] = self.table[key]
        return hit, out

    def __len__(self):
        return len(self.table)
