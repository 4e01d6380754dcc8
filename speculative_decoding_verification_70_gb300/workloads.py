"""Seeded synthetic inputs for the verify-and-recover step.

This module only draws random numbers in the shapes of the pages' workloads;
it holds none of the method's arithmetic (no softmax, acceptance, residual or
top-f).  Both the CUDA path and the CPU oracle read the tensors it returns.

Workloads (vocabulary sizes stand in for the Llama-3 and Qwen3 families that
"tanishqkumar/ssd" (sourcepulse summary, "Highlighted Details") supports; k,
f, batch and temperature follow the README bench commands quoted on the
Chinese README translation page, "基准测试" section):

  tiny      B=1,   k=4, f=2, V=1000,   fp32, Z~N(0,2), D=Z+N(0,0.5), T=1
  llama_sd  B=1,   k=6,      V=128256, bf16, Z~N(0,3)+5 peaks(+8), D=Z+N(0,1)
  ssd_fork  B=1,   k=7, f=3, V=128256, bf16, as llama_sd, D has k+1 rows
  qwen_b64  B=64,  k=5, f=3, V=151936, bf16, D=Z+N(0,sigma_b),
            sigma_b in {0.3,1,3}, T=0.7
  mixed512  B=512, k=7, f=4, V=151936, fp32, peaks at Zipf(1.1) ranks,
            T=0 on half the rows (seeded permutation), U(0.5,1.2) elsewhere

Draft tokens are drawn from softmax(D/T) with the Gumbel-max trick
(argmax(D/T + G), G standard Gumbel), which needs no softmax; at T = 0 they
are the draft argmax.  In SSD mode the draft holds k+1 rows and the extra
token x_k (drawn from draft row k) is the mask at position k.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np
import torch

# N(0, s): s is the standard deviation.


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    k: int
    f: int            # 0: no forked recovery (sync SD)
    V: int
    dtype: str        # "f32" | "bf16"
    z_std: float
    d_std: float      # draft noise std (qwen_b64 overrides per row)
    peaks: int
    peak_boost: float
    peak_place: str   # "uniform" | "zipf"
    temp: str         # a number, "mixed" (half 0, half U(0.5,1.2)) or
                      # "stochastic" (all U(0.5,1.2))
    ssd: bool         # draft logits carry k+1 rows

    @property
    def Pd(self) -> int:
        return self.k + 1 if self.ssd else self.k

    def algorithmic_bytes(self) -> Dict[str, int]:
        s = 4 if self.dtype == "f32" else 2
        verify = self.B * (2 * self.k + 1) * self.V * s
        fork = self.B * self.V * s if self.f > 0 else 0
        return {"verify": verify, "fork": fork, "residual_max": 2 * self.B * self.V * s}


WORKLOADS = {
    "tiny": Workload("tiny", 1, 4, 2, 1000, "f32", 2.0, 0.5, 0, 0.0, "uniform", "1.0", True),
    "llama_sd": Workload("llama_sd", 1, 6, 0, 128256, "bf16", 3.0, 1.0, 5, 8.0, "uniform", "1.0", False),
    "ssd_fork": Workload("ssd_fork", 1, 7, 3, 128256, "bf16", 3.0, 1.0, 5, 8.0, "uniform", "1.0", True),
    "qwen_b64": Workload("qwen_b64", 64, 5, 3, 151936, "bf16", 3.0, -1.0, 5, 8.0, "uniform", "0.7", True),
    "mixed512": Workload("mixed512", 512, 7, 4, 151936, "f32", 3.0, 1.0, 5, 8.0, "zipf", "mixed", True),
}
ORDER = ["tiny", "llama_sd", "ssd_fork", "qwen_b64", "mixed512"]
SEED_BASE = 1234


def workload(name: str, **overrides) -> Workload:
    return dataclasses.replace(WORKLOADS[name], **overrides)


def default_seed(name: str) -> int:
    return SEED_BASE + ORDER.index(name) + 1 if name in ORDER else SEED_BASE


def _peak_indices(w: Workload, rows: int, rng: np.random.Generator) -> np.ndarray:
    if w.peaks == 0:
        return np.zeros((rows, 0), dtype=np.int64)
    if w.peak_place == "uniform":
        return rng.integers(0, w.V, size=(rows, w.peaks))
    out = np.empty((rows, w.peaks), dtype=np.int64)
    for r in range(rows):
        for j in range(w.peaks):
            while True:
                v = int(rng.zipf(1.1)) - 1
                if v < w.V:
                    out[r, j] = v
                    break
    return out


def temperatures(w: Workload, seed: int, temp: Optional[str] = None) -> torch.Tensor:
    rng = np.random.default_rng(seed + 7)
    t = temp if temp is not None else w.temp
    if t in ("mixed", "stochastic"):
        T = rng.uniform(0.5, 1.2, size=w.B).astype(np.float32)
        if t == "mixed":  # exactly half the rows greedy
            zero = rng.permutation(w.B)[: w.B // 2]
            T[zero] = 0.0
    else:
        T = np.full(w.B, float(t), dtype=np.float32)
    return torch.from_numpy(T)


def make_inputs(w: Workload, device="cpu", seed: Optional[int] = None,
                temp: Optional[str] = None, b_block: int = 32) -> Dict[str, torch.Tensor]:
    """Draw one batch of the workload on ``device``.

    Returns Z [B,k+1,V], D [B,Pd,V] (float32 or bfloat16), x [B,k] int32,
    x_next [B] int32 (the draft token at position k in SSD mode, else -1),
    mask [B,k+1,1] int32, T [B] f32, u_acc [B,k] f32, u_smp [B] f32.
    Rows are generated in blocks of ``b_block`` batch rows to bound the
    temporaries.
    """
    seed = default_seed(w.name) if seed is None else seed
    device = torch.device(device)
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    B, k, V, Pd = w.B, w.k, w.V, w.Pd
    rng = np.random.default_rng(seed)
    peaks = torch.from_numpy(_peak_indices(w, B * (k + 1), rng)).to(device)
    if w.d_std < 0:
        sig = rng.choice(np.array([0.3, 1.0, 3.0]), size=B).astype(np.float32)
    else:
        sig = np.full(B, w.d_std, dtype=np.float32)
    T = temperatures(w, seed, temp)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    Z = torch.empty((B, k + 1, V), dtype=dt, device=device)
    D = torch.empty((B, Pd, V), dtype=dt, device=device)
    x_all = torch.empty((B, Pd), dtype=torch.int32, device=device)
    sig_t = torch.from_numpy(sig).to(device)
    T_dev = T.to(device)
    for b0 in range(0, B, b_block):
        b1 = min(B, b0 + b_block)
        nb = b1 - b0
        z = torch.randn((nb, k + 1, V), generator=gen, device=device) * w.z_std
        if w.peaks:
            pk = peaks[b0 * (k + 1):b1 * (k + 1)].view(nb, k + 1, w.peaks)
            z.scatter_add_(2, pk, torch.full(pk.shape, w.peak_boost, device=device))
        zq = z.to(dt)
        Z[b0:b1] = zq
        # draft rows: target row i plus noise (row k of the target seeds the
        # extra SSD draft row, as the other rows do)
        src = zq[:, :Pd].float() if Pd <= k + 1 else None
        d = src + torch.randn((nb, Pd, V), generator=gen, device=device) * sig_t[b0:b1].view(nb, 1, 1)
        dq = d.to(dt)
        D[b0:b1] = dq
        # draft tokens: Gumbel-max sample from softmax(D/T); argmax at T = 0
        tb = T_dev[b0:b1].view(nb, 1, 1)
        u = torch.rand((nb, Pd, V), generator=gen, device=device)
        g = -torch.log(-torch.log(u.clamp_min(1e-38)))
        score = torch.where(tb > 0, dq.float() / torch.where(tb > 0, tb, torch.ones_like(tb)) + g,
                            dq.float())
        x_all[b0:b1] = torch.argmax(score, dim=2).to(torch.int32)
        del z, zq, d, dq, u, g, score
    u_acc = torch.rand((B, k), generator=gen, device=device)
    u_smp = torch.rand((B,), generator=gen, device=device)
    x = x_all[:, :k].contiguous()
    if w.ssd:
        x_next = x_all[:, k].contiguous()
        mask = x_all[:, :, None].contiguous()
    else:
        x_next = torch.full((B,), -1, dtype=torch.int32, device=device)
        mask = torch.cat([x, x_next[:, None]], dim=1)[:, :, None].contiguous()
    return {"Z": Z, "D": D, "x": x, "x_next": x_next, "mask": mask,
            "T": T_dev.contiguous(), "u_acc": u_acc.contiguous(),
            "u_smp": u_smp.contiguous()}


# ---------------------------------------------------------------------------
# token trees (tree decoding: "tanishqkumar/ssd" summary, module notes)
# ---------------------------------------------------------------------------
def tree_parents(widths) -> np.ndarray:
    """Parents of a level-ordered tree in which every node of level l has
    widths[l] children (node 0 the root): e.g. (4, 2, 1) gives 1 + 4 + 8 + 8
    = 21 nodes."""
    par = [-1]
    level = [0]
    for w in widths:
        nxt = []
        for u in level:
            for _ in range(w):
                par.append(u)
                nxt.append(len(par) - 1)
        level = nxt
    return np.asarray(par, dtype=np.int32)


def random_tree_parents(B: int, N: int, seed: int) -> np.ndarray:
    """[B, N] parents of random recursive trees (node j hangs below a
    uniformly drawn earlier node)."""
    rng = np.random.default_rng(seed)
    par = np.full((B, N), -1, dtype=np.int32)
    for j in range(1, N):
        par[:, j] = rng.integers(0, j, size=B)
    return par


# The tree benchmark workload: Qwen3-sized vocabulary, bf16, 64 batch rows,
# trees of widths (4, 2, 1) = 21 nodes, per-row draft noise as qwen_b64.
TREE_B64 = dict(B=64, widths=(4, 2, 1), V=151936, dtype="bf16", z_std=3.0, d_std=-1.0,
                peaks=5, peak_boost=8.0, temp="0.7")


def make_tree_inputs(B: int, parent, V: int, dtype: str = "f32", temp="1.0",
                     z_std: float = 3.0, d_std: float = 1.0, peaks: int = 5,
                     peak_boost: float = 8.0, seed: int = 4242, device="cpu",
                     b_block: int = 16) -> Dict[str, torch.Tensor]:
    """Draw one batch of token trees.

    parent: [N] (the same tree in every batch row) or [B, N] int32.
    Z [B,N,V] ~ N(0, z_std) plus `peaks` logits raised by `peak_boost` at
    uniform indices; D = Z + N(0, d_std) (d_std < 0: per-row std drawn from
    {0.3, 1, 3}).  temp: a number, "mixed" or "stochastic" (as the chain
    workloads).  Node j's token is drawn from softmax(D[parent[j]] / T) by
    Gumbel-max (so that siblings are independent draws from the parent's
    q); on T == 0 rows from softmax(D[parent[j]]) with the first child of
    every node forced to the draft argmax.  u_acc [B,N], u_smp [B] uniform.
    """
    device = torch.device(device)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    par = np.asarray(parent, dtype=np.int32)
    par = np.repeat(par[None], B, axis=0) if par.ndim == 1 else par.copy()
    par = np.ascontiguousarray(par, dtype=np.int32)
    N = par.shape[1]
    rng = np.random.default_rng(seed)
    pk_idx = torch.from_numpy(rng.integers(0, V, size=(B * N, max(peaks, 1)))).to(device)
    sig = (rng.choice(np.array([0.3, 1.0, 3.0]), size=B) if d_std < 0
           else np.full(B, d_std)).astype(np.float32)
    w = Workload("tree", B, 1, 0, V, dtype, z_std, d_std, peaks, peak_boost, "uniform",
                 str(temp), False)
    T = temperatures(w, seed, str(temp)).to(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    Z = torch.empty((B, N, V), dtype=dt, device=device)
    D = torch.empty((B, N, V), dtype=dt, device=device)
    tok = torch.zeros((B, N), dtype=torch.int32, device=device)
    par_t = torch.from_numpy(par.astype(np.int64)).to(device)
    sig_t = torch.from_numpy(sig).to(device)
    first = np.zeros((B, N), dtype=bool)
    for j in range(1, N):
        first[:, j] = ~(par[:, 1:j] == par[:, j:j + 1]).any(axis=1)
    first_t = torch.from_numpy(first).to(device)
    for b0 in range(0, B, b_block):
        b1 = min(B, b0 + b_block)
        nb = b1 - b0
        z = torch.randn((nb, N, V), generator=gen, device=device) * z_std
        if peaks:
            pk = pk_idx[b0 * N:b1 * N].view(nb, N, -1)
            z.scatter_add_(2, pk, torch.full(pk.shape, peak_boost, device=device))
        zq = z.to(dt)
        Z[b0:b1] = zq
        d = zq.float() + torch.randn((nb, N, V), generator=gen, device=device) * \
            sig_t[b0:b1].view(nb, 1, 1)
        dq = d.to(dt)
        D[b0:b1] = dq
        # each node's token from its parent's draft row
        pd = torch.gather(dq.float(), 1, par_t[b0:b1].clamp_min(0)[:, :, None].expand(nb, N, V))
        tb = T[b0:b1].view(nb, 1, 1)
        u = torch.rand((nb, N, V), generator=gen, device=device)
        g = -torch.log(-torch.log(u.clamp_min(1e-38)))
        score = pd / torch.where(tb > 0, tb, torch.ones_like(tb)) + g
        t = torch.argmax(score, dim=2)
        am = torch.argmax(pd, dim=2)
        t = torch.where((tb.view(nb, 1) == 0) & first_t[b0:b1], am, t)
        tok[b0:b1] = t.to(torch.int32)
        del z, zq, d, dq, pd, u, g, score
    tok[:, 0] = 0
    u_acc = torch.rand((B, N), generator=gen, device=device)
    u_smp = torch.rand((B,), generator=gen, device=device)
    return {"Z": Z, "D": D, "parent": torch.from_numpy(par).to(device), "tok": tok,
            "T": T.contiguous(), "u_acc": u_acc.contiguous(), "u_smp": u_smp.contiguous()}


def cache_workload(fork_tok: torch.Tensor, depth: int, V: int, n_queries: int,
                   seed: int) -> Dict[str, torch.Tensor]:
    """Speculation-cache traffic for the SSD workload: one entry per forked
    recovery token (b, j, fork_tok[b,j,r]) with a random depth-token payload,
    plus ``n_queries`` lookups, half of them inserted keys and half keys that
    were never inserted.  All tensors on the CPU (int32)."""
    rng = np.random.default_rng(seed)
    ft = fork_tok.detach().cpu().numpy()
    B, P, f = ft.shape
    bb, jj, rr = np.meshgrid(np.arange(B), np.arange(P), np.arange(f), indexing="ij")
    ins_b = bb.reshape(-1).astype(np.int32)
    ins_pos = jj.reshape(-1).astype(np.int32)
    ins_tok = ft.reshape(-1).astype(np.int32)
    keep = ins_tok >= 0
    ins_b, ins_pos, ins_tok = ins_b[keep], ins_pos[keep], ins_tok[keep]
    payload = rng.integers(0, V, size=(len(ins_b), depth)).astype(np.int32)
    inserted = set(zip(ins_b.tolist(), ins_pos.tolist(), ins_tok.tolist()))
    half = n_queries // 2
    pick = rng.integers(0, len(ins_b), size=half)
    qb = list(ins_b[pick]); qp = list(ins_pos[pick]); qt = list(ins_tok[pick])
    while len(qb) < n_queries:
        cand = (int(rng.integers(0, B)), int(rng.integers(0, P)), int(rng.integers(0, V)))
        if cand in inserted:
            continue
        qb.append(cand[0]); qp.append(cand[1]); qt.append(cand[2])
    order = rng.permutation(n_queries)
    as_t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.int32)[order].copy())
    return {"ins_b": torch.from_numpy(ins_b), "ins_pos": torch.from_numpy(ins_pos),
            "ins_tok": torch.from_numpy(ins_tok), "payload": torch.from_numpy(payload),
            "q_b": as_t(qb), "q_pos": as_t(qp), "q_tok": as_t(qt)}
