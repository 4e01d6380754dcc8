"""Verify over top-k / top-p filtered distributions on the GPU (through the
C ABI) against the oracle (reading R9: the target and the draft filtered
alike -- the first K tokens by logit, then the shortest prefix holding
>= top_p of their mass -- and the speculative-sampling rule applied to the
filtered p and q)."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import to_np
from speculative_decoding_verification_70_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _draft_tokens_in_topk(D, k, K, seed):
    """Draft tokens drawn uniformly among each draft row's K best logits (so
    most of them survive the filter and acceptance is exercised)."""
    g = torch.Generator(device=D.device).manual_seed(seed)
    top = torch.topk(D[:, :k].float(), K, dim=2).indices            # [B, k, K]
    pick = torch.randint(0, K, top.shape[:2] + (1,), generator=g, device=D.device)
    return top.gather(2, pick)[..., 0].to(torch.int32).contiguous()


def _check(inp, x, K, top_p, out):
    ref = oracle.verify_recover_filtered(inp["Z"].cpu(), inp["D"].cpu(), x.cpu(), inp["T"].cpu(),
                                         K, None if top_p is None else top_p.cpu(),
                                         inp["u_acc"].cpu(), inp["u_smp"].cpu())
    assert np.array_equal(to_np(out["accept_len"]), ref["accept_len"])
    assert np.array_equal(to_np(out["out_tok"]), ref["out_tok"])
    ok = ref["accept_len"] >= 0
    for key in ("p_at_x", "q_at_x"):
        g, r = to_np(out[key])[ok], ref[key][ok]
        assert np.max(np.abs(g - r), initial=0.0) <= 1e-5, key
    return ref


CASES = [("tiny", {}, None, 5, 0.9), ("tiny", {"B": 12}, "stochastic", 1, None),
         ("llama_sd", {}, "1.0", 32, None), ("llama_sd", {}, "0", 32, 0.5),
         ("ssd_fork", {"B": 3}, "1.0", 8, 0.95), ("qwen_b64", {"B": 8}, None, 20, 0.8),
         ("mixed512", {"B": 8}, None, 32, "rows")]


@pytest.mark.parametrize("name,over,temp,K,tp", CASES)
def test_verify_topk_matches_oracle(gpu_lib, name, over, temp, K, tp):
    w = W.workload(name, **over)
    inp = W.make_inputs(w, device=DEV, seed=W.default_seed(name) + 300, temp=temp)
    x = _draft_tokens_in_topk(inp["D"], w.k, min(K, 4) if K > 1 else 1, 5)
    if tp == "rows":
        top_p = torch.linspace(0.2, 1.0, w.B, device=DEV)
    elif tp is None:
        top_p = None
    else:
        top_p = torch.full((w.B,), tp, device=DEV)
    out = gpu_lib.ssd_verify_topk(inp["Z"], inp["D"][:, : w.k].contiguous(), x, inp["T"], K,
                                  top_p, inp["u_acc"], inp["u_smp"])
    torch.cuda.synchronize()
    inp = dict(inp, D=inp["D"][:, : w.k].contiguous())
    ref = _check(inp, x, K, top_p, out)
    assert gpu_lib.get_device_error(out["ws"]) == 0
    if temp != "0" and w.B >= 8:
        assert (ref["accept_len"] > 0).any()   # acceptance is exercised


def test_verify_topk_edges(gpu_lib):
    """Sentinels, rows with fewer than K finite logits, ties, an unaligned
    row length (scalar path) and K = V; K up to 16 and K above 16 take the
    two candidate-selection paths of the pass kernel."""
    B, k, V = 8, 3, 37
    g = torch.Generator().manual_seed(11)
    Z = torch.randint(-3, 4, (B, k + 1, V), generator=g).float()    # many ties
    D = torch.randint(-3, 4, (B, k, V), generator=g).float()
    Z[1, :, 5:] = float("-inf")                                        # 5 finite logits
    D[1, :, 7:] = float("-inf")
    Z[2, 1, 3] = float("nan")
    x = torch.randint(0, 5, (B, k), generator=g, dtype=torch.int32)
    x[3, 0] = V                                                       # bad token
    T = torch.tensor([1.0, 0.8, 1.0, 1.0, -1.0, 0.0, 1.5, 0.7])
    ua = torch.rand((B, k), generator=g)
    us = torch.rand(B, generator=g)
    inp = {"Z": Z, "D": D, "T": T, "u_acc": ua, "u_smp": us}
    for K, tp in ((6, None), (V, None), (3, 0.6), (32, None), (20, 0.6), (17, None)):
        if K > 32:
            continue
        top_p = None if tp is None else torch.full((B,), tp)
        out = gpu_lib.ssd_verify_topk(Z.to(DEV), D.to(DEV), x.to(DEV), T.to(DEV), K,
                                      None if top_p is None else top_p.to(DEV), ua.to(DEV),
                                      us.to(DEV))
        torch.cuda.synchronize()
        ref = _check(inp, x, K, top_p, out)
        assert ref["accept_len"][2] == -1 and ref["accept_len"][3] == -2
        assert ref["accept_len"][4] == -1
        gpu_lib.get_device_error(out["ws"], clear=True)


def test_verify_topk_full_vocab_equals_plain_verify(gpu_lib):
    """K = V (V <= 32) and no top-p is no filter: same results as ssd_verify."""
    B, k, V = 64, 4, 32
    g = torch.Generator().manual_seed(2)
    Z = (torch.randn((B, k + 1, V), generator=g) * 2).to(DEV)
    D = (Z[:, :k] + torch.randn((B, k, V), generator=g).to(DEV)).contiguous()
    x = torch.randint(0, V, (B, k), generator=g, dtype=torch.int32).to(DEV)
    T = (torch.rand(B, generator=g) + 0.5).to(DEV)
    ua = torch.rand((B, k), generator=g).to(DEV)
    us = torch.rand(B, generator=g).to(DEV)
    a = gpu_lib.ssd_verify_topk(Z, D, x, T, V, None, ua, us)
    b = gpu_lib.ssd_verify(Z, D, x, T, ua, us)
    assert torch.equal(a["accept_len"], b["accept_len"])
    assert torch.equal(a["out_tok"], b["out_tok"])
    assert torch.allclose(a["p_at_x"], b["p_at_x"], atol=1e-6)


def test_verify_topk_clustered_top_logits(gpu_lib):
    """Top logits packed into one thread's vectors: certification from the
    threads' top-4 lists fails and the pass takes its second chance (row 0:
    six top logits at indices 0-3, 1024, 2048) or, when one thread holds
    hundreds of them, its last resort (row 1: every index = 0..3 mod 1024)."""
    B, k, V, K = 4, 2, 151936, 32
    g = torch.Generator().manual_seed(9)
    Z = torch.randn((B, k + 1, V), generator=g)
    D = torch.randn((B, k, V), generator=g)
    hot0 = torch.tensor([0, 1, 2, 3, 1024, 2048])
    idx = torch.arange(V)
    hot1 = idx[(idx % 1024) < 4]
    for t in (Z, D):
        t[0, :, hot0] = 20.0 + torch.arange(len(hot0)).float() * 0.01
        t[1, :, hot1] = 10.0 + torch.rand((t.shape[1], len(hot1)), generator=g)
    x = torch.stack([hot0[:k], hot1[5:5 + k], torch.tensor([7, 9]), torch.tensor([11, 13])]).int()
    T = torch.tensor([1.0, 0.8, 1.0, 0.6])
    ua = torch.rand((B, k), generator=g)
    us = torch.rand(B, generator=g)
    inp = {"Z": Z, "D": D, "T": T, "u_acc": ua, "u_smp": us}
    for tp in (None, 0.7):
        top_p = None if tp is None else torch.full((B,), tp)
        out = gpu_lib.ssd_verify_topk(Z.to(DEV), D.to(DEV), x.to(DEV), T.to(DEV), K,
                                      None if top_p is None else top_p.to(DEV), ua.to(DEV),
                                      us.to(DEV))
        torch.cuda.synchronize()
        _check(inp, x, K, top_p, out)
        assert gpu_lib.get_device_error(out["ws"]) == 0


def test_verify_topk_last_resort(gpu_lib):
    """B = 512 makes a CTA cover a whole row (593 elements per thread); in
    row 3 one thread holds all 596 top logits (every index = 0..3 mod 1024),
    more than the second-chance buffer takes, so the exact K-round re-scan
    runs.  Rows 3 and 100 are compared with the oracle."""
    B, k, V, K = 512, 2, 151936, 32
    g = torch.Generator(device=DEV).manual_seed(4)
    Z = torch.randn((B, k + 1, V), generator=g, device=DEV)
    D = torch.randn((B, k, V), generator=g, device=DEV)
    idx = torch.arange(V, device=DEV)
    hot = idx[(idx % 1024) < 4]
    Z[3, :, hot] = 10.0 + torch.rand((k + 1, len(hot)), generator=g, device=DEV)
    D[3, :, hot] = 10.0 + torch.rand((k, len(hot)), generator=g, device=DEV)
    x = torch.randint(0, V, (B, k), generator=g, device=DEV, dtype=torch.int32)
    x[3] = hot[:k].int()
    T = torch.full((B,), 0.9, device=DEV)
    ua = torch.rand((B, k), generator=g, device=DEV)
    us = torch.rand(B, generator=g, device=DEV)
    out = gpu_lib.ssd_verify_topk(Z, D, x, T, K, None, ua, us)
    torch.cuda.synchronize()
    rows = [3, 100]
    sub = {"Z": Z[rows].cpu(), "D": D[rows].cpu(), "T": T[rows].cpu(), "u_acc": ua[rows].cpu(),
           "u_smp": us[rows].cpu()}
    got = {key: out[key][rows] for key in ("accept_len", "out_tok", "p_at_x", "q_at_x")}
    _check(sub, x[rows].cpu(), K, None, got)
    assert gpu_lib.get_device_error(out["ws"]) == 0


# ---------------------------------------------------------------------------
# K above the in-register lists and top-p over the whole vocabulary: each
# row's kept set is a threshold on the token order, found from histograms
# (ssd_filter.cu).  Same rules as above: decisions and tokens identical to
# the oracle, p(x), q(x) within 1e-5.
# ---------------------------------------------------------------------------
BIG = [("qwen_b64", {"B": 8}, None, 50, None), ("qwen_b64", {"B": 8}, None, 50, 0.9),
       ("qwen_b64", {"B": 8}, None, 256, 0.95), ("qwen_b64", {"B": 8}, None, "V", 0.9),
       ("qwen_b64", {"B": 8}, None, "V", 0.95), ("qwen_b64", {"B": 6}, None, 1024, None),
       ("mixed512", {"B": 8}, None, 50, 0.9), ("mixed512", {"B": 8}, None, 256, None),
       ("mixed512", {"B": 8}, None, "V", 0.9), ("mixed512", {"B": 8}, None, "V", 0.95),
       ("mixed512", {"B": 6}, "stochastic", 2000, 0.5), ("llama_sd", {"B": 4}, "1.0", "V", 0.8),
       ("tiny", {"B": 12}, "stochastic", 33, None), ("tiny", {"B": 12}, "stochastic", "V", 0.7)]


@pytest.mark.parametrize("name,over,temp,K,tp", BIG)
def test_verify_filtered_large_k_and_nucleus(gpu_lib, name, over, temp, K, tp):
    w = W.workload(name, **over)
    K = w.V if K == "V" else K
    inp = W.make_inputs(w, device=DEV, seed=W.default_seed(name) + 600, temp=temp)
    x = _draft_tokens_in_topk(inp["D"], w.k, 4, 6)
    top_p = None if tp is None else torch.full((w.B,), tp, device=DEV)
    D = inp["D"][:, : w.k].contiguous()
    out = gpu_lib.ssd_verify_topk(inp["Z"], D, x, inp["T"], K, top_p, inp["u_acc"], inp["u_smp"])
    torch.cuda.synchronize()
    ref = _check(dict(inp, D=D), x, K, top_p, out)
    assert gpu_lib.get_device_error(out["ws"]) == 0
    if w.B >= 8 and temp != "0":
        assert (ref["accept_len"] > 0).any()


def test_verify_filtered_nucleus_every_row_of_a_batch(gpu_lib):
    """Top-p 0.9 over the whole vocabulary (K = V) on 256 stochastic rows of
    the large-batch shape (fp32, V = 151936), per-row top_p, every row
    against the oracle."""
    w = W.workload("mixed512", B=256)
    inp = W.make_inputs(w, device=DEV, seed=6061, temp="stochastic")
    x = _draft_tokens_in_topk(inp["D"], w.k, 8, 7)
    top_p = torch.linspace(0.5, 0.99, w.B, device=DEV)
    D = inp["D"][:, : w.k].contiguous()
    out = gpu_lib.ssd_verify_topk(inp["Z"], D, x, inp["T"], w.V, top_p, inp["u_acc"],
                                  inp["u_smp"])
    torch.cuda.synchronize()
    _check(dict(inp, D=D), x, w.V, top_p, out)
    assert gpu_lib.get_device_error(out["ws"]) == 0


def test_verify_filtered_no_filter_equals_plain_verify(gpu_lib):
    """K >= V and no top-p keeps every token: the threshold path then gives
    what ssd_verify gives (same draws: the kept mass is the row's exact
    mass)."""
    w = W.workload("qwen_b64", B=16)
    inp = W.make_inputs(w, device=DEV, seed=71)
    D = inp["D"][:, : w.k].contiguous()
    a = gpu_lib.ssd_verify_topk(inp["Z"], D, inp["x"], inp["T"], 10 * w.V, None, inp["u_acc"],
                                inp["u_smp"])
    b = gpu_lib.ssd_verify(inp["Z"], D, inp["x"], inp["T"], inp["u_acc"], inp["u_smp"])
    assert torch.equal(a["accept_len"], b["accept_len"])
    assert torch.equal(a["out_tok"], b["out_tok"])
    assert torch.allclose(a["p_at_x"], b["p_at_x"], atol=1e-6)


def test_verify_filtered_edges(gpu_lib):
    """Rows the threshold path must get right: thousands of equal logits
    (the cut's bins overflow the candidate buffer: bisection), ties at the
    cut, -0 and +0 logits, rows with fewer finite logits than K, NaN and
    +inf rows, a bad token, greedy rows, top_p = 0 (one token kept), top_p
    just below 1, K just below V; an unaligned row length takes the scalar
    path."""
    for V in (5000, 5001):
        B, k = 10, 3
        g = torch.Generator().manual_seed(V)
        Z = torch.randn((B, k + 1, V), generator=g) * 2
        D = Z[:, :k] + torch.randn((B, k, V), generator=g) * 0.7
        Z[0] = 1.5                                            # constant rows
        D[0] = 1.5
        Z[1] = torch.randint(-2, 3, (k + 1, V), generator=g).float()  # five values: ties
        D[1] = torch.randint(-2, 3, (k, V), generator=g).float()
        Z[2, :, ::2] = 0.0                                    # +0 and -0
        Z[2, :, 1::2] = -0.0
        D[2, :, ::3] = -0.0
        Z[3, :, 40:] = float("-inf")                           # 40 finite logits
        D[3, :, 60:] = float("-inf")
        Z[4, 1, 17] = float("nan")
        D[5, 0, 3] = float("inf")
        x = torch.randint(0, 40, (B, k), generator=g, dtype=torch.int32)
        x[6, 1] = V                                           # bad token
        T = torch.tensor([1.0, 0.9, 1.1, 0.8, 1.0, 1.0, 1.0, 0.0, 0.7, 1.3])
        ua = torch.rand((B, k), generator=g)
        us = torch.rand(B, generator=g)
        inp = {"Z": Z, "D": D, "T": T, "u_acc": ua, "u_smp": us}
        for K, tp in ((V, 0.9), (1000, None), (V - 1, 0.3), (100, 0.999999), (64, 0.0),
                      (V, float(np.nextafter(np.float32(1), np.float32(0))))):
            top_p = None if tp is None else torch.full((B,), tp)
            out = gpu_lib.ssd_verify_topk(Z.to(DEV), D.to(DEV), x.to(DEV), T.to(DEV), K,
                                          None if top_p is None else top_p.to(DEV),
                                          ua.to(DEV), us.to(DEV))
            torch.cuda.synchronize()
            ref = _check(inp, x, K, top_p, out)
            assert ref["accept_len"][4] == -1 and ref["accept_len"][5] == -1
            assert ref["accept_len"][6] == -2
            err = gpu_lib.get_device_error(out["ws"], clear=True)
            assert not err & gpu_lib.DEVERR_FILTER_BAND, (V, K, tp, err)
