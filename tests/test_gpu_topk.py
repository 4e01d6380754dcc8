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
    row length (scalar path) and K = V."""
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
    for K, tp in ((6, None), (V, None), (3, 0.6)):
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
