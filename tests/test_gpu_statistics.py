"""Statistical checks of the CUDA path (through the C ABI): the output law of
the verify-and-recover step equals the target law (exactness: "SSD: drafting
and verification on separate GPUs", "What changes in SSD"), and the
acceptance rate at a position equals sum_x min(p(x), q(x)) (the
speculative-sampling rule of Leviathan et al. / Chen et al. that the
speculative-sampling summary's "How It Works" describes).

10^6 independent trials of V = 8, k = 2 run as one call with B = 10^6 batch
rows (more than one grid's 65535 batch rows, so the launch loops are
exercised).  The target and draft logits are the same in every row; the
draft tokens and the uniforms differ.  The expected laws are computed here
in float64 from the closed form of the softmax, not by the oracle; the GPU's
tokens are also compared with the oracle's on the same inputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import Report, compare_verify

pytestmark = pytest.mark.gpu
scipy_stats = pytest.importorskip("scipy.stats")


def _softmax64(z, T):
    a = np.exp((z.astype(np.float64) - z.max(axis=-1, keepdims=True)) / T)
    return a / a.sum(axis=-1, keepdims=True)


def _draw_from(probs, u):
    c = np.cumsum(probs)
    return np.minimum((u[:, None] >= c[None, :]).sum(-1), len(probs) - 1)


@pytest.fixture(scope="module")
def million(gpu_lib):
    rng = np.random.default_rng(77)
    V, k, N, T = 8, 2, 1_000_000, 0.9
    Z = (rng.standard_normal((k + 1, V)) * 1.2).astype(np.float32)
    D = (Z[:k] + rng.standard_normal((k, V)) * 0.8).astype(np.float32)
    p, q = _softmax64(Z, T), _softmax64(D, T)
    x = np.stack([_draw_from(q[i], rng.random(N)) for i in range(k)], axis=1).astype(np.int32)
    ua = rng.random((N, k)).astype(np.float32)
    us = rng.random(N).astype(np.float32)
    host = {"Z": torch.from_numpy(np.broadcast_to(Z, (N, k + 1, V)).copy()),
            "D": torch.from_numpy(np.broadcast_to(D, (N, k, V)).copy()),
            "x": torch.from_numpy(x), "T": torch.full((N,), T, dtype=torch.float32),
            "u_acc": torch.from_numpy(ua), "u_smp": torch.from_numpy(us)}
    dev = {key: v.cuda() for key, v in host.items()}
    out = gpu_lib.ssd_verify(dev["Z"], dev["D"], dev["x"], dev["T"], dev["u_acc"], dev["u_smp"])
    torch.cuda.synchronize()
    assert gpu_lib.get_device_error(out["ws"]) == 0
    got = {key: out[key].cpu() for key in ("accept_len", "out_tok", "p_at_x", "q_at_x")}
    # complete every row to 3 tokens with independent draws from the target
    n = got["accept_len"].numpy()
    tok = got["out_tok"].numpy()
    seq = np.full((N, 3), -1, dtype=np.int64)
    for j in range(3):
        have = j <= n
        seq[have, j] = tok[have, j]
        seq[~have, j] = _draw_from(p[j], rng.random(int((~have).sum())))
    return {"p": p, "q": q, "n": n, "seq": seq, "N": N, "V": V, "host": host, "got": got}


def test_gpu_output_law_equals_target_law(million):
    p, seq, N, V = million["p"], million["seq"], million["N"], million["V"]
    assert (seq >= 0).all() and (seq < V).all()
    idx = seq[:, 0] * V * V + seq[:, 1] * V + seq[:, 2]
    obs = np.bincount(idx, minlength=V ** 3).astype(np.float64)
    exp = np.einsum("i,j,k->ijk", p[0], p[1], p[2]).reshape(-1) * N
    small = exp < 5
    o = np.append(obs[~small], obs[small].sum())
    e = np.append(exp[~small], exp[small].sum())
    if e[-1] == 0:
        o, e = o[:-1], e[:-1]
    assert scipy_stats.chisquare(o, e).pvalue > 1e-3
    first = np.bincount(seq[:, 0], minlength=V)
    assert scipy_stats.chisquare(first, p[0] * N).pvalue > 1e-3


def test_gpu_acceptance_rate_closed_form(million):
    p, q, n, N = million["p"], million["q"], million["n"], million["N"]
    for i in range(2):
        rate = np.minimum(p[: i + 1], q[: i + 1]).sum(axis=1).prod()
        emp = (n >= i + 1).mean()
        sigma = math.sqrt(rate * (1 - rate) / N)
        assert abs(emp - rate) < 5 * sigma, (i, emp, rate)


def test_gpu_tokens_match_oracle_on_a_million_rows(million):
    host, got = million["host"], million["got"]
    ref = oracle.verify_recover(host["Z"], host["D"], host["x"], host["T"], host["u_acc"],
                                host["u_smp"])
    diff = (ref["accept_len"] != got["accept_len"].numpy()) | \
        (ref["out_tok"] != got["out_tok"].numpy()).any(axis=1)
    bad = np.nonzero(diff)[0]
    assert len(bad) <= 1e-4 * million["N"], len(bad)
    if len(bad):
        sub = {key: ref[key][bad] for key in ("accept_len", "out_tok", "p_at_x", "q_at_x")}
        rep = compare_verify(host, got, bad, sub, Report())
        assert not rep.failures, rep.failures[:5]
    dp = np.abs(ref["p_at_x"] - got["p_at_x"].numpy()).max()
    dq = np.abs(ref["q_at_x"] - got["q_at_x"].numpy()).max()
    assert dp <= 1e-5 and dq <= 1e-5


def test_gpu_draft_sampler_law_on_a_million_rows(gpu_lib):
    """The drafter's Gumbel-max draws follow softmax(z / T): 10^6 rows of the
    same logits (distinct batch rows, so distinct Philox counters), one call;
    every row also equals the oracle's draw."""
    V, N, T = 8, 1_000_000, 0.9
    z = torch.tensor([0.4, -0.7, 1.9, 0.0, 1.2, -2.5, 0.9, 0.1])
    D = z.reshape(1, 1, V).expand(N, 1, V).contiguous()
    Tv = torch.full((N,), T)
    out = gpu_lib.ssd_draft_sample(D.cuda(), Tv.cuda(), 1, 0xABCDEF, 2)
    torch.cuda.synchronize()
    x = out["x"][:, 0].cpu().numpy()
    p = _softmax64(z.numpy()[None], T)[0]
    assert scipy_stats.chisquare(np.bincount(x, minlength=V), p * N).pvalue > 1e-3
    ref = oracle.draft_sample(D, Tv, 0xABCDEF, 2)[:, 0]
    assert (ref != x).sum() <= 1e-4 * N


def test_gpu_tree_law_on_a_million_rows(gpu_lib):
    """Token-tree verification keeps the target law (multi-step speculative
    sampling; tree decoding, "tanishqkumar/ssd" summary, module notes):
    10^6 trees (root with three children drawn from the root's q, each with
    two children drawn from that child's q), V = 5, one call.  The first two
    tokens (completed from the target when one is produced) follow
    p_root(t1) * p_t1(t2); every row equals the oracle's."""
    rng = np.random.default_rng(91)
    B, V, T = 1_000_000, 5, 1.0
    Zr = (rng.standard_normal(V) * 1.5).astype(np.float32)
    Dr = (Zr + rng.standard_normal(V) * 1.5).astype(np.float32)
    Zc = (rng.standard_normal((V, V)) * 1.5).astype(np.float32)
    Dc = (Zc + rng.standard_normal((V, V)) * 1.5).astype(np.float32)
    pr, qr = _softmax64(Zr[None], T)[0], _softmax64(Dr[None], T)[0]
    pc, qc = _softmax64(Zc, T), _softmax64(Dc, T)
    par = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3], np.int32)
    N = len(par)
    tok = np.zeros((B, N), np.int32)
    for j in range(1, 4):
        tok[:, j] = _draw_from(qr, rng.random(B))
    for j in range(4, N):
        pt = tok[:, par[j]]
        tok[:, j] = np.minimum((np.cumsum(qc[pt], axis=1) <= rng.random(B)[:, None]).sum(1), V - 1)
    Z = np.empty((B, N, V), np.float32)
    D = np.empty((B, N, V), np.float32)
    Z[:, 0], D[:, 0] = Zr, Dr
    Z[:, 1:], D[:, 1:] = Zc[tok[:, 1:]], Dc[tok[:, 1:]]
    ua = rng.random((B, N)).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    host = {"Z": torch.from_numpy(Z), "D": torch.from_numpy(D),
            "parent": torch.from_numpy(np.repeat(par[None], B, axis=0)),
            "tok": torch.from_numpy(tok), "T": torch.full((B,), T),
            "u_acc": torch.from_numpy(ua), "u_smp": torch.from_numpy(us)}
    dev = {k: v.cuda() for k, v in host.items()}
    out = gpu_lib.ssd_verify_tree(dev["Z"], dev["D"], dev["parent"], dev["tok"], dev["T"],
                                  dev["u_acc"], dev["u_smp"])
    torch.cuda.synchronize()
    assert gpu_lib.get_device_error(out["ws"]) == 0
    n = out["accept_len"].cpu().numpy()
    o = out["out_tok"].cpu().numpy()
    assert (n >= 0).all() and (n >= 1).mean() > 0.3 and (n == 2).any()
    t1 = o[:, 0].astype(np.int64)
    t2 = np.where(n >= 1, o[:, 1],
                  np.minimum((np.cumsum(pc[t1], axis=1) <= rng.random(B)[:, None]).sum(1), V - 1))
    obs = np.bincount(t1 * V + t2, minlength=V * V)
    assert scipy_stats.chisquare(obs, (pr[:, None] * pc).reshape(-1) * B).pvalue > 1e-3
    ref = oracle.verify_tree(Z, D, host["parent"].numpy(), tok, host["T"].numpy(), ua, us)
    diff = (ref["accept_len"] != n) | (ref["out_tok"] != o).any(axis=1)
    assert diff.sum() <= 1e-4 * B, int(diff.sum())
