"""The B = 1 SSD step as a CUDA graph.  The pages' engine runs its decode loop
with CUDA graphs ("tanishqkumar/ssd" summary: optimized kernels with CUDA
graphs; SSD project summary, "Highlighted Details": CUDAgraphs), and at
B = 1 the step is launch-bound, so the library's calls must be capturable:
capture once with static buffers, then replay with new inputs copied in.
Each replay is checked against the oracle and the dict cache."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import Report, compare_forks, compare_verify, oracle_rows
from speculative_decoding_verification_70_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEPTH = 7


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("temp", ["1.0", "0"])
def test_graph_replay_of_the_b1_ssd_step(gpu_lib, temp):
    w = W.workload("ssd_fork")
    static = W.make_inputs(w, device="cuda", seed=100, temp=temp)
    ws = gpu_lib.new_workspace(gpu_lib.workspace_bytes(w.B, w.k, w.V, w.f), "cuda")
    out, look = {}, {}
    cache = gpu_lib.SpecCache(64, DEPTH)
    payload = torch.arange(w.B * (w.k + 1) * w.f * DEPTH, dtype=torch.int32,
                           device="cuda").reshape(-1, DEPTH)

    def step():
        o = gpu_lib.ssd_verify_fork(static["Z"], static["D"], static["x"], static["T"],
                                    static["u_acc"], static["u_smp"], w.f, static["mask"],
                                    ws=ws, out=out)
        cache.clear()
        cache.insert_forks(o["fork_tok"], payload)
        r = cache.lookup_outcome(o["accept_len"], o["out_tok"], out=look or None)
        look.update(r)

    g = _capture(step)
    rep = Report()
    for seed in range(5):
        new = W.make_inputs(w, device="cuda", seed=200 + seed, temp=temp)
        for key in static:
            static[key].copy_(new[key])
        g.replay()
        torch.cuda.synchronize()
        ref = oracle_rows(new, np.arange(w.B))
        compare_verify(new, out, np.arange(w.B), ref, rep)
        rf = oracle.forked_topf(new["D"].cpu(), w.f, new["mask"].cpu())
        compare_forks(rf, out["fork_tok"], out["fork_logit"])
        # the realised outcome hits the cache iff it is one of the forks
        c = oracle.SpecCacheOracle(DEPTH)
        ft = rf["fork_tok"]
        bb = np.repeat(np.arange(w.B), (w.k + 1) * w.f)
        pp = np.tile(np.repeat(np.arange(w.k + 1), w.f), w.B)
        c.insert(bb, pp, ft.reshape(-1), payload.cpu().numpy())
        n = ref["accept_len"]
        hit, tok = c.lookup(np.arange(w.B), n, ref["out_tok"][np.arange(w.B), n])
        assert np.array_equal(look["hit"].cpu().numpy(), hit)
        assert np.array_equal(look["tok_out"].cpu().numpy(), tok)
    assert not rep.failures, rep.failures[:3]
    assert rep.sampled_mismatch == 0
    assert cache.error() == 0
    cache.close()


def test_graph_replays_keep_last_insert_wins(gpu_lib):
    """Duplicates across replays of one captured insert: the later replay's
    payload wins even when its duplicate sits at a lower input index."""
    n = 8
    b = torch.zeros(n, dtype=torch.int32, device="cuda")
    pos = torch.zeros(n, dtype=torch.int32, device="cuda")
    tok = torch.arange(n, dtype=torch.int32, device="cuda") + 100
    pay = torch.zeros((n, 2), dtype=torch.int32, device="cuda")
    qb = torch.zeros(1, dtype=torch.int32, device="cuda")
    qtok = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    cache = gpu_lib.SpecCache(64, 2)
    look = {}

    def step():
        cache.insert(b, pos, tok, pay)
        r = cache.lookup(qb, qb, qtok, out=look or None)
        look.update(r)

    g = _capture(step)   # capture runs the warm-up inserts too; their keys are 100..107
    for rep, idx in enumerate([7, 0, 5, 1]):
        t = torch.arange(n, dtype=torch.int32) + 1000 * (rep + 1)
        t[idx] = 7                       # the duplicate key, at a different index each time
        tok.copy_(t)
        pay.fill_(rep)
        g.replay()
        torch.cuda.synchronize()
        assert int(look["hit"][0]) == 1
        assert look["tok_out"][0].tolist() == [rep, rep]
    cache.close()
