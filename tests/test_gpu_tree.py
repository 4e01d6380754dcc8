"""Parity of the token-tree verification (ssd_verify_tree, through the C ABI)
with the oracle: greedy rows, sentinels and accepted node ids exactly; rows
that sample identical unless a decision of the oracle's walk lies within
1e-6 of its uniform (an acceptance ratio r(x)/q(x) or a boundary of the
final draw's normalised CDF).

The rule is SpecInfer's multi-step speculative sampling over a tree (tree
decoding, "tanishqkumar/ssd" summary, module notes); inputs come from the
seeded tree generator (children drawn from their parent's draft law).
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import to_np
from speculative_decoding_verification_70_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
BOUNDARY = 1e-6


def _probs(row, T):
    return oracle.softmax_temp(row[None], [T])["probs"][0]


def _boundary_distance(inp, b):
    """Smallest distance between a uniform and the decision it is compared
    with along the oracle's walk of row b (recomputed from the oracle's
    softmax; the residual update written out in numpy)."""
    Z, D = inp["Z"][b].float().numpy(), inp["D"][b].float().numpy()
    par, tok = inp["parent"][b].numpy(), inp["tok"][b].numpy()
    T = float(inp["T"][b])
    ua, us = inp["u_acc"][b].numpy(), float(inp["u_smp"][b])
    N = len(par)
    cur, r, best = 0, _probs(Z[0], T), 1.0
    while True:
        moved = 0
        q = None
        for c in range(cur + 1, N):
            if par[c] != cur:
                continue
            if q is None:
                q = _probs(D[cur], T)
            x = tok[c]
            if q[x] > 0:
                best = min(best, abs(float(ua[c]) - r[x] / q[x]))
                acc = ua[c] < r[x] / q[x]
            else:
                acc = r[x] > 0
            if acc:
                moved = c
                break
            w = np.maximum(r - q, 0.0)
            if w.sum() > 0:
                r = w / w.sum()
        if not moved:
            cdf = np.cumsum(r) / r.sum()
            return min(best, float(np.min(np.abs(cdf - us))))
        cur, r = moved, _probs(Z[moved], T)


def _run(gpu_lib, inp):
    dev = {k: v.to(DEV) for k, v in inp.items()}
    out = gpu_lib.ssd_verify_tree(dev["Z"], dev["D"], dev["parent"], dev["tok"], dev["T"],
                                  dev["u_acc"], dev["u_smp"])
    torch.cuda.synchronize()
    return out


def _compare(inp, out, rows=None):
    B = inp["T"].shape[0]
    rows = np.arange(B) if rows is None else np.asarray(rows)
    sub = {k: v[rows] for k, v in inp.items()}
    ref = oracle.verify_tree(sub["Z"], sub["D"], sub["parent"], sub["tok"], sub["T"],
                             sub["u_acc"], sub["u_smp"])
    g_acc = to_np(out["accept_len"])[rows]
    g_tok = to_np(out["out_tok"])[rows]
    g_node = to_np(out["out_node"])[rows]
    T = sub["T"].numpy()
    mism = 0
    for i, b in enumerate(rows):
        same = (g_acc[i] == ref["accept_len"][i] and np.array_equal(g_tok[i], ref["out_tok"][i])
                and np.array_equal(g_node[i], ref["out_node"][i]))
        if same:
            continue
        assert T[i] > 0 and ref["accept_len"][i] >= 0, \
            "row %d (greedy or sentinel) differs: gpu %d %s oracle %d %s" % (
                b, g_acc[i], g_tok[i], ref["accept_len"][i], ref["out_tok"][i])
        dist = _boundary_distance(sub, i)
        assert dist <= BOUNDARY, "row %d differs %.3g from a boundary: gpu %s oracle %s" % (
            b, dist, g_tok[i], ref["out_tok"][i])
        mism += 1
    return ref, mism


CASES = [
    # dtype, V, B, tree, temp
    ("f32", 1000, 64, "random12", "mixed"),
    ("bf16", 4096, 32, (4, 2, 1), "stochastic"),
    ("f32", 151936, 6, (3, 2), "0.7"),
    ("bf16", 128256, 4, "random24", "1.0"),
    ("f32", 999, 16, "random8", "mixed"),         # V not a multiple of 4: scalar loads
    ("bf16", 1003, 16, (2, 2), "stochastic"),     # V not a multiple of 8
    ("f32", 3000, 32, "single", "stochastic"),    # N = 1: the bonus draw only
]


def _parents(tree, B, seed):
    if tree == "single":
        return np.full((B, 1), -1, np.int32)
    if isinstance(tree, str) and tree.startswith("random"):
        return W.random_tree_parents(B, int(tree[6:]), seed)
    return W.tree_parents(tree)


@pytest.mark.parametrize("dtype,V,B,tree,temp", CASES)
def test_tree_matches_oracle(gpu_lib, dtype, V, B, tree, temp):
    seed = 900 + V % 97 + B
    inp = W.make_tree_inputs(B, _parents(tree, B, seed), V, dtype=dtype, temp=temp, seed=seed,
                             d_std=-1.0)
    out = _run(gpu_lib, inp)
    assert gpu_lib.get_device_error(out["ws"]) == 0
    ref, mism = _compare(inp, out)
    assert mism <= max(1, B // 1000)
    if tree != "single" and (inp["T"] > 0).sum() >= 8:
        assert (ref["accept_len"] > 0).any()       # acceptance is exercised


def test_tree_deep_chain_and_many_siblings(gpu_lib):
    """A 64-node chain with q close to p (long accepted paths), and a root
    with 40 children whose draft law avoids the target's mass (every child
    rejected: 40 residual updates, then the draw)."""
    B, V = 8, 2000
    chain = np.arange(-1, 63, dtype=np.int32)
    inp = W.make_tree_inputs(B, chain, V, temp="1.0", seed=77, d_std=0.05, peaks=0)
    out = _run(gpu_lib, inp)
    ref, _ = _compare(inp, out)
    assert ref["accept_len"].max() >= 10
    star = np.zeros(41, np.int32)
    star[0] = -1
    inp = W.make_tree_inputs(B, star, V, temp="0.8", seed=78, d_std=3.0)
    g = torch.Generator().manual_seed(5)
    Dr = torch.randn((B, V), generator=g) * 3
    inp["D"][:, 0] = Dr                              # q unrelated to p at the root
    inp["tok"][:, 1:] = torch.argsort(Dr, dim=1, descending=True)[:, :40].to(torch.int32)
    out = _run(gpu_lib, inp)
    ref, _ = _compare(inp, out)
    assert (ref["accept_len"] == 0).any()


def test_tree_edges(gpu_lib):
    """Sentinels (invalid T, NaN in a draft row with children, bad parent,
    token out of range), a NaN in a leaf's draft row (not read), children
    with q(x) = 0, duplicate sibling tokens and greedy rows with ties."""
    B, V = 12, 40
    par = W.tree_parents((3, 2))
    inp = W.make_tree_inputs(B, par, V, temp="mixed", seed=31, peaks=0)
    Z, D = inp["Z"], inp["D"]
    inp["T"][0] = -1.0
    D[1, 1, 3] = float("nan")                        # node 1 has children
    D[7, 7, 3] = float("nan")                        # node 7 is a leaf: not read
    inp["parent"][2, 5] = 5                          # parent not before the node
    inp["tok"][3, 4] = V                             # token out of range
    inp["T"][4] = 0.9
    D[4, 0, inp["tok"][4, 1]] = float("-inf")        # q(x) = 0 for the first child
    inp["T"][5] = 1.1
    inp["tok"][5, 2] = inp["tok"][5, 1]              # duplicate siblings
    inp["T"][6] = 0.0
    Z[6] = torch.round(Z[6])                         # ties for the argmax
    inp["tok"][6, 1:4] = torch.argmax(Z[6, 0]).to(torch.int32)
    out = _run(gpu_lib, inp)
    ref, _ = _compare(inp, out)
    assert list(ref["accept_len"][:4]) == [-1, -1, -2, -2]
    assert ref["accept_len"][7] >= 0
    assert ref["accept_len"][6] >= 1 and to_np(out["out_node"])[6, 0] == 1
    gpu_lib.get_device_error(out["ws"], clear=True)


def test_tree_benchmark_workload_sampled(gpu_lib):
    """The benchmark's tree workload (B = 64, widths (4, 2, 1) = 21 nodes,
    V = 151936, bf16): every fourth row against the oracle."""
    cfg = W.TREE_B64
    par = W.tree_parents(cfg["widths"])
    inp = W.make_tree_inputs(cfg["B"], par, cfg["V"], dtype=cfg["dtype"], temp=cfg["temp"],
                             z_std=cfg["z_std"], d_std=cfg["d_std"], peaks=cfg["peaks"],
                             peak_boost=cfg["peak_boost"], seed=4242, device=DEV)
    out = _run(gpu_lib, {k: v for k, v in inp.items()})
    host = {k: v.cpu() for k, v in inp.items()}
    ref, mism = _compare(host, out, rows=np.arange(0, cfg["B"], 4))
    assert mism <= 1
    assert (ref["accept_len"] >= 2).any()


def test_tree_graph_replay(gpu_lib):
    """The call is capture-safe: replays of a captured call give the eager
    results."""
    B, V = 16, 2048
    inp = W.make_tree_inputs(B, W.tree_parents((3, 2, 1)), V, temp="mixed", seed=12)
    dev = {k: v.to(DEV) for k, v in inp.items()}
    eager = gpu_lib.ssd_verify_tree(dev["Z"], dev["D"], dev["parent"], dev["tok"], dev["T"],
                                    dev["u_acc"], dev["u_smp"])
    torch.cuda.synchronize()
    ref = {k: eager[k].clone() for k in ("accept_len", "out_tok", "out_node")}
    out = dict(eager)
    for k in ("accept_len", "out_tok", "out_node"):
        out[k].fill_(-7)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            gpu_lib.ssd_verify_tree(dev["Z"], dev["D"], dev["parent"], dev["tok"], dev["T"],
                                    dev["u_acc"], dev["u_smp"], ws=eager["ws"], out=out)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for k in ref:
        assert torch.equal(out[k], ref[k]), k


def test_tree_golden_cases(gpu_lib):
    """The hand-derived cases of tests/golden/tree_cases.json on the GPU."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "tree_cases.json")) as fh:
        cases = json.load(fh)["cases"]
    for case in cases:
        Z = np.log(np.array(case["target_weights"], dtype=np.float64)).astype(np.float32)[None]
        D = np.log(np.array(case["draft_weights"], dtype=np.float64)).astype(np.float32)[None]
        t = lambda a, dt: torch.tensor(a, dtype=dt, device=DEV)
        out = gpu_lib.ssd_verify_tree(t(Z, torch.float32), t(D, torch.float32),
                                      t([case["parent"]], torch.int32),
                                      t([case["tok"]], torch.int32),
                                      t([case["T"]], torch.float32),
                                      t([case["u_acc"]], torch.float32),
                                      t([case["u_smp"]], torch.float32))
        torch.cuda.synchronize()
        assert int(out["accept_len"][0]) == case["accept_len"], case["name"]
        assert to_np(out["out_tok"])[0].tolist() == case["out_tok"], case["name"]
        assert to_np(out["out_node"])[0].tolist() == case["out_node"], case["name"]
