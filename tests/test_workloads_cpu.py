"""The seeded input generators (CPU): shapes, determinism, and the
statistical property the exactness tests rely on -- draft tokens, and a tree
node's children, are draws from the draft's law at their position
(softmax(D / T) by the Gumbel-max trick; greedy rows take the argmax).

The laws are computed here with scipy's softmax, independently of the
oracle and of the CUDA path."""
import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

from speculative_decoding_verification_70_gb300 import workloads as W


def test_tree_parents_shapes():
    assert W.tree_parents(()).tolist() == [-1]
    assert W.tree_parents((3,)).tolist() == [-1, 0, 0, 0]
    par = W.tree_parents((4, 2, 1))
    assert len(par) == 1 + 4 + 8 + 8
    assert par[0] == -1 and all(0 <= par[j] < j for j in range(1, len(par)))
    kids = np.bincount(par[1:], minlength=len(par))
    assert kids[0] == 4 and (kids[1:5] == 2).all() and (kids[5:13] == 1).all()
    assert (kids[13:] == 0).all()
    rp = W.random_tree_parents(50, 17, seed=3)
    assert rp.shape == (50, 17) and (rp[:, 0] == -1).all()
    for j in range(1, 17):
        assert ((rp[:, j] >= 0) & (rp[:, j] < j)).all()


def test_make_tree_inputs_shapes_and_determinism():
    par = W.tree_parents((2, 2))
    a = W.make_tree_inputs(5, par, 64, dtype="bf16", temp="mixed", seed=11)
    b = W.make_tree_inputs(5, par, 64, dtype="bf16", temp="mixed", seed=11)
    N = len(par)
    assert a["Z"].shape == (5, N, 64) and a["Z"].dtype == torch.bfloat16
    assert a["D"].shape == a["Z"].shape and a["parent"].shape == (5, N)
    assert a["parent"].is_contiguous() and a["parent"].numpy().flags.writeable
    assert a["tok"].dtype == torch.int32 and (a["tok"][:, 0] == 0).all()
    assert ((a["tok"] >= 0) & (a["tok"] < 64)).all()
    for k in a:
        assert torch.equal(a[k], b[k]), k
    assert (a["T"] == 0).sum() == 2          # "mixed": half the rows greedy (rounded down)


def test_tree_children_follow_the_parents_draft_law():
    """10^5 trees with a root of two children: each child's token is a draw
    from softmax(D[root] / T) (chi-square), the two independent."""
    B, V, T = 100_000, 6, 0.8
    inp = W.make_tree_inputs(B, W.tree_parents((2,)), V, temp=str(T), seed=5, d_std=0.0,
                             peaks=0, b_block=25_000)
    D0 = inp["D"][:, 0].double().numpy()
    # the root's draft row differs per tree: test the law of the rank of the
    # drawn token's probability via the probability integral transform
    q = scipy.special.softmax(D0 / T, axis=1)
    for j in (1, 2):
        x = inp["tok"][:, j].long().numpy()
        cdf_hi = np.cumsum(q, axis=1)[np.arange(B), x]
        cdf_lo = cdf_hi - q[np.arange(B), x]
        # a randomised PIT value is U(0,1) when x ~ q
        u = cdf_lo + np.random.default_rng(j).random(B) * (cdf_hi - cdf_lo)
        assert scipy.stats.kstest(u, "uniform").pvalue > 1e-3
    same = (inp["tok"][:, 1] == inp["tok"][:, 2]).double().mean().item()
    expect = (q ** 2).sum(axis=1).mean()
    assert abs(same - expect) < 5 * np.sqrt(expect * (1 - expect) / B)


def test_greedy_rows_take_the_draft_argmax_first():
    inp = W.make_tree_inputs(64, W.tree_parents((3,)), 50, temp="0", seed=9, peaks=0)
    am = torch.argmax(inp["D"][:, 0].float(), dim=1)
    assert torch.equal(inp["tok"][:, 1].long(), am)     # the first child of the root


@pytest.mark.parametrize("name", ["tiny", "llama_sd", "ssd_fork"])
def test_chain_draft_tokens_follow_the_draft_law(name):
    """The chain workloads' draft tokens are draws from softmax(D / T):
    randomised probability integral transform over many batch rows."""
    w = W.workload(name, B=4000, V=300)
    inp = W.make_inputs(w, device="cpu", seed=21, temp="1.0", b_block=1000)
    D = inp["D"][:, 0].double().numpy()
    q = scipy.special.softmax(D, axis=1)
    x = inp["x"][:, 0].long().numpy()
    B = len(x)
    cdf_hi = np.cumsum(q, axis=1)[np.arange(B), x]
    cdf_lo = cdf_hi - q[np.arange(B), x]
    u = cdf_lo + np.random.default_rng(0).random(B) * (cdf_hi - cdf_lo)
    assert scipy.stats.kstest(u, "uniform").pvalue > 1e-3
