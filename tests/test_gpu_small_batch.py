"""The small-batch schedules of the verify step.

A verify call of a few batch rows moves a few MB; its time is its chain of
dependent launches.  Two schedules shorten that chain:
  - step: the whole call (statistics pass, row merges and forks, acceptance,
    the draw's exact passes, select, cache clear / insert / lookup) as one
    cooperative kernel whose CTAs meet at grid-wide barriers (B <= 8);
  - chain: after the statistics pass, one thread-block cluster per batch
    row does the finalisation, the draw and the cache step (one launch).
Larger batches run the same steps as separate batched kernels.

These tests run every schedule on the same inputs (ssd_set_step_schedule
and ssd_set_chain_batch pick one) and check that accept lengths, p(x), q(x),
forks, drawn tokens and cache lookups are the same bits as the batched
kernels', and that they agree with the oracle: on short and long
vocabularies, unaligned rows, the largest k and f, batches of more clusters
than fit the GPU at once, a step grid far smaller than the work (many units
per CTA), CUDA graph replays of the B = 1 round step, the draw's degenerate
rows (near-equal target and draft rows; u at the ends; greedy, invalid and
NaN rows), and a barrier wait that runs out (the kernel reports
SSD_DEVERR_TIMEOUT and leaves the workspace usable).
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import Report, compare_forks, compare_verify, oracle_rows, to_np
from speculative_decoding_verification_70_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"

# (step max batch, step grid cap, chain max batch)
SCHEDULES = {
    "step": (8, 0, 0),
    "step_g40": (8, 40, 0),      # 40 CTAs: several statistics units per CTA, long ranges
    "chain": (0, 0, 1 << 20),
    "batched": (0, 0, 0),
}


@pytest.fixture
def schedule(gpu_lib):
    def pick(name):
        mb, grid, chain = SCHEDULES[name]
        gpu_lib.set_step_schedule(mb, grid)
        gpu_lib.set_chain_batch(chain)
    yield pick
    gpu_lib.set_step_schedule(-1, 0)
    gpu_lib.set_chain_batch(-1)


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t


def _same(a, b, keys, label=""):
    for key in keys:
        assert torch.equal(_bits(a[key]), _bits(b[key])), (label, key)


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
def test_schedules_agree_and_match_oracle(gpu_lib, schedule, name, over, temp):
    w = W.workload(name, **over)
    inp = W.make_inputs(w, device=DEV, seed=W.default_seed(name) + 311, temp=temp)
    outs = {}
    for sched in SCHEDULES:
        schedule(sched)
        outs[sched] = _verify(gpu_lib, w, inp)
    ref = outs["batched"]
    for sched, o in outs.items():
        _same(o, ref, KEYS + (FORK_KEYS if w.f > 0 else ()), sched)
        assert o["err"] == ref["err"], sched
    bs = np.arange(w.B)
    rep = compare_verify(inp, ref, bs, oracle_rows(inp, bs), Report())
    assert not rep.failures, rep.failures[:3]
    if w.f > 0:
        rf = oracle.forked_topf(inp["D"].cpu(), w.f, inp["mask"].cpu())
        compare_forks(rf, ref["fork_tok"], ref["fork_logit"], name)


def _round(gpu_lib, w, inp, cache, payload, clear):
    out = gpu_lib.ssd_verify_fork_cache(inp["Z"], inp["D"], inp["x"], inp["T"], inp["u_acc"],
                                        inp["u_smp"], w.f, inp["mask"], cache, payload,
                                        clear=clear)
    torch.cuda.synchronize()
    return {k: v.clone() for k, v in out.items() if k != "ws"}


@pytest.mark.parametrize("name,over", [("ssd_fork", {}), ("qwen_b64", {"B": 8}),
                                       ("tiny", {"B": 8, "V": 8000, "temp": "mixed"})])
def test_round_step_schedules_agree(gpu_lib, schedule, name, over):
    """Two SSD round steps into one cache, the second without a clear: the
    later call's payload wins for keys both calls insert, whichever schedule
    ran each call (the schedules share the cache's call counter)."""
    w = W.workload(name, **over)
    inp = W.make_inputs(w, device=DEV, seed=W.default_seed(name) + 97)
    depth = 4
    n = w.B * (w.k + 1) * w.f
    cap = 1 << max(6, (4 * n - 1).bit_length())
    pay = torch.arange(n * depth, dtype=torch.int32, device=DEV).reshape(n, depth)
    results = {}
    for order in (("batched", "batched"), ("step", "step"), ("chain", "chain"),
                  ("step", "batched"), ("batched", "step"), ("chain", "step"),
                  ("step_g40", "chain")):
        cache = gpu_lib.SpecCache(cap, depth)
        outs = []
        for rep, sched in enumerate(order):
            schedule(sched)
            outs.append(_round(gpu_lib, w, inp, cache, pay + 1000 * rep, clear=rep == 0))
        assert cache.error() == 0
        cache.close()
        results[order] = outs
    ref = results[("batched", "batched")]
    for order, outs in results.items():
        for r in range(2):
            _same(outs[r], ref[r], KEYS + FORK_KEYS + ("hit", "tok_out"), order)
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


def test_degenerate_rows_every_schedule(gpu_lib, schedule):
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
    outs = {}
    for sched in SCHEDULES:
        schedule(sched)
        outs[sched] = _verify(gpu_lib, w, inp)
    a = outs["batched"]
    for sched, o in outs.items():
        _same(o, a, KEYS, sched)
        assert o["err"] == a["err"], sched
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


@pytest.mark.parametrize("sched,temp", [("step", "1.0"), ("step", "0"), ("chain", "1.0")])
def test_round_step_graph_replay(gpu_lib, schedule, sched, temp):
    """The B = 1 round step (verify, forks, cache clear, insert and lookup)
    captured once as a CUDA graph and replayed with new inputs: each replay
    against the oracle and the dict cache."""
    schedule(sched)
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


def test_step_barrier_timeout_is_reported(gpu_lib, schedule):
    """A grid barrier whose wait cannot end: the workspace's first arrival
    sub-counter is planted at a value the count never reaches, so no CTA
    completes the first barrier.  Every wait gives up after its time limit,
    the call reports SSD_DEVERR_TIMEOUT, the kernel's exit puts the barrier
    words back to zero, and the next call on the same workspace is right."""
    schedule("step")
    w = W.workload("tiny", B=2, V=4096, temp="1.0")
    inp = W.make_inputs(w, device=DEV, seed=8)
    ws = gpu_lib.new_workspace(gpu_lib.workspace_bytes(w.B, w.k, w.V, w.f), DEV)
    base = (-ws.data_ptr()) % 256          # the binding aligns the workspace to 256 bytes
    bar = ws[base + 256: base + 260]       # sub-counter 0 of the barrier words
    bar.copy_(torch.tensor([0x00, 0x00, 0x00, 0x40], dtype=torch.uint8, device=DEV))
    args = (inp["Z"], inp["D"], inp["x"], inp["T"], inp["u_acc"], inp["u_smp"], w.f, inp["mask"])
    gpu_lib.ssd_verify_fork(*args, ws=ws)
    torch.cuda.synchronize()
    assert gpu_lib.get_device_error(ws, clear=True) & gpu_lib.DEVERR_TIMEOUT
    assert int(bar.sum()) == 0
    out = gpu_lib.ssd_verify_fork(*args, ws=ws)
    torch.cuda.synchronize()
    assert gpu_lib.get_device_error(ws, clear=True) == 0
    ref = oracle_rows(inp, np.arange(w.B))
    rep = compare_verify(inp, out, np.arange(w.B), ref, Report())
    assert not rep.failures, rep.failures[:3]
