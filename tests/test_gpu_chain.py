"""The small-batch schedule of the verify step.

After the statistics pass, a batch of at most a few rows runs its
finalisation (row merges, acceptance min(1, p/q), the first-reject prefix,
the forked top-f), the recovery / bonus draw and, in the SSD round step, the
cache insert of its forks and the lookup of its realised outcome as one
kernel: one thread-block cluster per batch row.  Larger batches run the
same steps as separate batched kernels.

These tests run both schedules on the same inputs (ssd_set_chain_batch picks
one) and check that accept lengths, p(x), q(x), forks, drawn tokens and cache
lookups are the same bits, and that both agree with the oracle: on short and
long vocabularies, unaligned rows, the largest k and f, batches of more
clusters than fit the GPU at once, CUDA graph replays of the B = 1 round
step, and the draw's degenerate rows (near-equal target and draft rows, whose
sign split overflows; u at the ends; greedy, invalid and NaN rows).
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import Report, compare_forks, compare_verify, oracle_rows, to_np
from speculative_decoding_verification_70_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
CHAIN, BATCHED = 1 << 20, 0


@pytest.fixture
def schedule(gpu_lib):
    yield gpu_lib.set_chain_batch
    gpu_lib.set_chain_batch(-1)


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t


def _same(a, b, keys):
    for key in keys:
        assert torch.equal(_bits(a[key]), _bits(b[key])), key


def _verify(gpu_lib, w, inp):
    if w.f > 0:
        out = gpu_lib.ssd_verify_fork(inp["Z"], inp["D"], inp["x"], inp["T"], inp["u_acc"],
                                      inp["u_smp"], w.f, inp["mask"])
    else:
        out = gpu_lib.ssd_verify(inp["Z"], inp["D"], inp["x"], inp["T"], inp["u_acc"],
                                 inp["u_smp"])
    torch.cuda.synchronize()
    res = {k: v.clone() for k, v in out.items() if k != "ws"}
    res["err"] = gpu_lib.get_device_error(out["ws"], clear=True)
    return res


KEYS = ("accept_len", "out_tok", "p_at_x", "q_at_x")
FORK_KEYS = ("fork_tok", "fork_logit")

CASES = [
    ("tiny", {"B": 8, "V": 8000}, "mixed"),
    ("ssd_fork", {}, "1.0"),
    ("ssd_fork", {}, "0"),
    ("llama_sd", {}, "1.0"),
    ("llama_sd", {"B": 4}, "stochastic"),
    ("qwen_b64", {"B": 16}, None),
    ("mixed512", {"B": 12}, None),
    # 40 clusters of 8 CTAs: more than the GPU holds at once
    ("mixed512", {"B": 40, "V": 50000}, "stochastic"),
    # odd V (scalar loads), the largest k and f
    ("tiny", {"B": 5, "V": 1001, "k": 31, "f": 16}, "1.0"),
    ("tiny", {"B": 3, "V": 2, "k": 1, "f": 1}, "1.0"),
    ("tiny", {"B": 4, "V": 4099, "dtype": "bf16", "f": 5}, "stochastic"),
]


@pytest.mark.parametrize("name,over,temp", CASES)
def test_chain_equals_batched_and_oracle(gpu_lib, schedule, name, over, temp):
    w = W.workload(name, **over)
    inp = W.make_inputs(w, device=DEV, seed=W.default_seed(name) + 311, temp=temp)
    schedule(CHAIN)
    a = _verify(gpu_lib, w, inp)
    schedule(BATCHED)
    b = _verify(gpu_lib, w, inp)
    _same(a, b, KEYS + (FORK_KEYS if w.f > 0 else ()))
    assert a["err"] == b["err"]
    bs = np.arange(w.B)
    rep = compare_verify(inp, a, bs, oracle_rows(inp, bs), Report())
    assert not rep.failures, rep.failures[:3]
    if w.f > 0:
        rf = oracle.forked_topf(inp["D"].cpu(), w.f, inp["mask"].cpu())
        compare_forks(rf, a["fork_tok"], a["fork_logit"], name)


def _round(gpu_lib, w, inp, cache, payload, clear):
    out = gpu_lib.ssd_verify_fork_cache(inp["Z"], inp["D"], inp["x"], inp["T"], inp["u_acc"],
                                        inp["u_smp"], w.f, inp["mask"], cache, payload,
                                        clear=clear)
    torch.cuda.synchronize()
    return {k: v.clone() for k, v in out.items() if k != "ws"}


@pytest.mark.parametrize("name,over", [("ssd_fork", {}), ("qwen_b64", {"B": 8}),
                                       ("tiny", {"B": 8, "V": 8000, "temp": "mixed"})])
def test_chain_round_step_equals_batched(gpu_lib, schedule, name, over):
    """Two SSD round steps into one cache, the second without a clear: the
    later call's payload wins for keys both calls insert, whichever schedule
    ran each call."""
    w = W.workload(name, **over)
    inp = W.make_inputs(w, device=DEV, seed=W.default_seed(name) + 97)
    depth = 4
    n = w.B * (w.k + 1) * w.f
    cap = 1 << max(6, (4 * n - 1).bit_length())
    pay = torch.arange(n * depth, dtype=torch.int32, device=DEV).reshape(n, depth)
    results = {}
    for order in ((CHAIN, CHAIN), (BATCHED, BATCHED), (CHAIN, BATCHED), (BATCHED, CHAIN)):
        cache = gpu_lib.SpecCache(cap, depth)
        outs = []
        for rep, sched in enumerate(order):
            schedule(sched)
            outs.append(_round(gpu_lib, w, inp, cache, pay + 1000 * rep, clear=rep == 0))
        assert cache.error() == 0
        cache.close()
        results[order] = outs
    ref = results[(BATCHED, BATCHED)]
    for order, outs in results.items():
        for r in range(2):
            _same(outs[r], ref[r], KEYS + FORK_KEYS + ("hit", "tok_out"))
    # against the dict cache: the second call's entries replace the first's
    out = ref[1]
    c = oracle.SpecCacheOracle(depth)
    ft = to_np(out["fork_tok"]).reshape(-1)
    bb = np.repeat(np.arange(w.B), (w.k + 1) * w.f)
    pp = np.tile(np.repeat(np.arange(w.k + 1), w.f), w.B)
    keep = ft >= 0  # empty fork slots are not inserted
    for rep in range(2):
        c.insert(bb[keep], pp[keep], ft[keep], (pay + 1000 * rep).cpu().numpy()[keep])
    nacc = to_np(out["accept_len"])
    ot = to_np(out["out_tok"])
    tok = np.array([ot[b, nacc[b]] if 0 <= nacc[b] <= w.k else -1 for b in range(w.B)])
    hit, tout = c.lookup(np.arange(w.B), nacc, tok)
    assert np.array_equal(to_np(out["hit"]), hit)
    assert np.array_equal(to_np(out["tok_out"]), tout)


def test_chain_degenerate_rows(gpu_lib, schedule):
    """Rows the draw treats specially, through both schedules and the oracle:
    near-equal target and draft rows rejected at position 0 (every element's
    sign is ambiguous, so the split overflows and the residual is summed
    directly), u = 0 and the largest u below 1 in the draw, greedy, invalid
    temperature, out-of-range token and NaN rows."""
    B, k, V = 8, 3, 151936
    g = torch.Generator().manual_seed(5)
    Z = 3.0 * torch.randn((B, k + 1, V), generator=g)
    D = Z[:, :k] + 0.7 * torch.randn((B, k, V), generator=g)
    x = torch.randint(0, V, (B, k), generator=g, dtype=torch.int32)
    T = torch.ones(B)
    u_acc = torch.rand((B, k), generator=g)
    u_smp = torch.rand(B, generator=g)
    # row 0: D = Z up to 1e-4 noise, the drafted token raised by 0.5 so that
    # p/q ~ 0.6 there, and u = 0.9 rejects it
    D[0] = Z[0, :k] + 1e-4 * torch.randn((k, V), generator=g)
    D[0, 0, int(x[0, 0])] += 0.5
    u_acc[0, 0] = 0.9
    u_smp[1] = 0.0                                   # row 1: u = 0
    u_smp[2] = float(np.nextafter(np.float32(1), np.float32(0)))  # row 2: largest u < 1
    T[3] = 0.0                                       # row 3: greedy
    T[4] = -1.0                                      # row 4: invalid temperature
    x[5, 2] = V                                      # row 5: token out of range
    Z[6, 1, 12345] = float("nan")                    # row 6: NaN target logit
    inp = {"Z": Z.to(DEV), "D": D.contiguous().to(DEV), "x": x.to(DEV), "T": T.to(DEV),
           "u_acc": u_acc.to(DEV), "u_smp": u_smp.to(DEV)}
    w = W.workload("tiny", B=B, k=k, V=V, f=0)
    schedule(CHAIN)
    a = _verify(gpu_lib, w, inp)
    schedule(BATCHED)
    b = _verify(gpu_lib, w, inp)
    _same(a, b, KEYS)
    assert a["err"] == b["err"]
    assert a["err"] == (gpu_lib.DEVERR_BAD_TEMPERATURE | gpu_lib.DEVERR_BAD_TOKEN |
                        gpu_lib.DEVERR_BAD_LOGITS)
    acc = to_np(a["accept_len"])
    assert acc[0] == 0 and list(acc[4:7]) == [-1, -2, -1]
    ref = oracle_rows(inp, np.arange(B))
    rep = compare_verify(inp, a, np.arange(B), ref, Report())
    assert not rep.failures, rep.failures[:3]
    assert rep.sampled_mismatch == 0


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


@pytest.mark.parametrize("temp", ["1.0", "0"])
def test_chain_round_step_graph_replay(gpu_lib, schedule, temp):
    """The B = 1 round step (one statistics pass, then the cluster kernel
    with the cache clear, insert and lookup) captured once and replayed with
    new inputs: each replay against the oracle and the dict cache."""
    schedule(-1)  # the default schedule: B = 1 takes the cluster kernel
    w = W.workload("ssd_fork")
    depth = 7
    static = W.make_inputs(w, device=DEV, seed=400, temp=temp)
    ws = gpu_lib.new_workspace(gpu_lib.workspace_bytes(w.B, w.k, w.V, w.f), DEV)
    cache = gpu_lib.SpecCache(64, depth)
    n = w.B * (w.k + 1) * w.f
    payload = torch.arange(n * depth, dtype=torch.int32, device=DEV).reshape(n, depth)
    out = {}

    def step():
        r = gpu_lib.ssd_verify_fork_cache(static["Z"], static["D"], static["x"], static["T"],
                                          static["u_acc"], static["u_smp"], w.f, static["mask"],
                                          cache, payload, ws=ws, out=out or None)
        out.update(r)

    graph = _capture(step)
    rep = Report()
    for seed in range(4):
        new = W.make_inputs(w, device=DEV, seed=500 + seed, temp=temp)
        for key in static:
            static[key].copy_(new[key])
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle_rows(new, np.arange(w.B))
        compare_verify(new, out, np.arange(w.B), ref, rep)
        rf = oracle.forked_topf(new["D"].cpu(), w.f, new["mask"].cpu())
        compare_forks(rf, out["fork_tok"], out["fork_logit"])
        c = oracle.SpecCacheOracle(depth)
        c.insert(np.zeros(n, dtype=np.int64), np.repeat(np.arange(w.k + 1), w.f),
                 rf["fork_tok"].reshape(-1), payload.cpu().numpy())
        nacc = ref["accept_len"]
        hit, tok = c.lookup(np.arange(w.B), nacc, ref["out_tok"][np.arange(w.B), nacc])
        assert np.array_equal(to_np(out["hit"]), hit)
        assert np.array_equal(to_np(out["tok_out"]), tok)
    assert not rep.failures, rep.failures[:3]
    assert rep.sampled_mismatch == 0
    assert cache.error() == 0
    cache.close()
