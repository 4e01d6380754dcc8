"""Draft-side sampling on the GPU (through the C ABI) against the oracle:
the drafter's tokens (Gumbel-max draws with Philox4x32-10 uniforms, argmax
at T = 0), the forks with the drafted token masked, and the verify call that
reuses the draft rows' statistics ("tanishqkumar/ssd" summary, module notes:
sampler greedy at temperature 0, forked recovery by top-k with masking;
speculative-sampling summary, "How It Works": the small model proposes the
draft)."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import Report, compare_verify, oracle_rows, to_np
from speculative_decoding_verification_70_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
SEED = 0x5EED_0000_1234


def _check_forks(D, x, f, got_tok, got_logit, rows):
    B = D.shape[0]
    ref = oracle.forked_topf(D[:, :rows].cpu(), f, x.reshape(B, rows, 1).cpu())
    assert np.array_equal(ref["fork_tok"], to_np(got_tok))
    rl = ref["fork_logit"].astype(np.float32)
    gl = to_np(got_logit)
    assert np.all((rl == gl) | (np.isnan(rl) & np.isnan(gl)))


CASES = [("tiny", {}, None), ("tiny", {"B": 9}, "stochastic"), ("llama_sd", {}, "1.0"),
         ("llama_sd", {}, "0"), ("ssd_fork", {}, "1.0"), ("qwen_b64", {"B": 6}, None),
         ("mixed512", {"B": 8}, None)]


@pytest.mark.parametrize("name,over,temp", CASES)
def test_draft_sample_matches_oracle(gpu_lib, name, over, temp):
    w = W.workload(name, **over)
    inp = W.make_inputs(w, device=DEV, seed=W.default_seed(name) + 77, temp=temp)
    D, T = inp["D"], inp["T"]
    rows = D.shape[1]
    f = 3
    for offset in (0, 5):
        out = gpu_lib.ssd_draft_sample(D, T, w.k, SEED, offset, f=f)
        torch.cuda.synchronize()
        ref = oracle.draft_sample(D.cpu(), T.cpu(), SEED, offset)
        assert np.array_equal(to_np(out["x"]), ref), (np.argwhere(to_np(out["x"]) != ref)[:5])
        _check_forks(D, out["x"], f, out["fork_tok"], out["fork_logit"], rows)
        assert gpu_lib.get_device_error(out["ws"]) == 0


def test_draft_sample_rows_and_sentinels(gpu_lib):
    """A sub-range of rows, an unaligned row stride (scalar path), invalid
    temperatures and a NaN row."""
    B, Pd, V = 5, 4, 1001
    g = torch.Generator().manual_seed(3)
    D = (torch.randn((B, Pd, V), generator=g) * 2).to(DEV)
    D[2, 2, 17] = float("nan")
    T = torch.tensor([1.0, 0.0, 0.9, -1.0, float("nan")], device=DEV)
    out = gpu_lib.ssd_draft_sample(D, T, Pd - 1, SEED, 9, row0=1, rows=3, f=2)
    torch.cuda.synchronize()
    ref = oracle.draft_sample(D.cpu(), T.cpu(), SEED, 9, row0=1, rows=3)
    assert np.array_equal(to_np(out["x"]), ref)
    assert ref[2, 1] == -1 and (ref[3] == -1).all() and (ref[4] == -1).all()
    err = gpu_lib.get_device_error(out["ws"], clear=True)
    assert err & gpu_lib.DEVERR_BAD_TEMPERATURE and err & gpu_lib.DEVERR_BAD_LOGITS
    _check_forks(D[:, 1:], out["x"], 2, out["fork_tok"], out["fork_logit"], 3)


@pytest.mark.parametrize("name,over,temp", [("tiny", {"B": 7}, None), ("llama_sd", {}, "1.0"),
                                            ("ssd_fork", {}, "1.0"), ("qwen_b64", {"B": 8}, None),
                                            ("mixed512", {"B": 16}, None)])
def test_verify_after_draft_sample_matches_oracle(gpu_lib, name, over, temp):
    """The draft tokens come from ssd_draft_sample (rows 0..k-1, one call per
    row as a drafter would make them); ssd_verify_drafted then reads only the
    target rows."""
    w = W.workload(name, **over)
    inp = W.make_inputs(w, device=DEV, seed=W.default_seed(name) + 91, temp=temp)
    ws = gpu_lib.new_workspace(gpu_lib.workspace_bytes(w.B, w.k, w.V, 0), DEV)
    x = torch.empty((w.B, w.k), dtype=torch.int32, device=DEV)
    for i in range(w.k):
        o = gpu_lib.ssd_draft_sample(inp["D"], inp["T"], w.k, SEED, 11, row0=i, rows=1, ws=ws)
        x[:, i] = o["x"][:, 0]
    inp = dict(inp, x=x)
    out = gpu_lib.ssd_verify(inp["Z"], inp["D"], x, inp["T"], inp["u_acc"], inp["u_smp"],
                             drafted=True, ws=ws)
    torch.cuda.synchronize()
    ref_x = oracle.draft_sample(inp["D"][:, : w.k].cpu(), inp["T"].cpu(), SEED, 11)
    assert np.array_equal(to_np(x), ref_x)
    bs = np.arange(w.B)
    rep = compare_verify(inp, out, bs, oracle_rows(inp, bs), Report())
    assert not rep.failures, rep.failures[:5]
    assert rep.sampled_mismatch == 0
    # the same tokens through the plain verify: the same probabilities
    plain = gpu_lib.ssd_verify(inp["Z"], inp["D"], x, inp["T"], inp["u_acc"], inp["u_smp"])
    assert torch.allclose(plain["p_at_x"], out["p_at_x"], atol=1e-6, rtol=0)
    assert torch.allclose(plain["q_at_x"], out["q_at_x"], atol=1e-6, rtol=0)
    assert gpu_lib.get_device_error(out["ws"]) == 0
