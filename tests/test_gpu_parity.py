"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Inputs are the seeded synthetic workloads; the oracle reads host copies of the
same tensors.  Sizes span several chunks and a ragged last chunk (V = 128256
and 151936 are not multiples of the chunk size), plus the edge cases of the
method: sentinels, infinities, ties, the smallest and largest sizes.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import Report, compare_forks, compare_verify, oracle_rows, to_np
from speculative_decoding_verification_70_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_verify(ssd, inp, fork_f=0, sample=True):
    if fork_f:
        return ssd.ssd_verify_fork(inp["Z"], inp["D"], inp["x"], inp["T"], inp["u_acc"],
                                   inp["u_smp"] if sample else None, fork_f, inp["mask"])
    return ssd.ssd_verify(inp["Z"], inp["D"], inp["x"], inp["T"], inp["u_acc"],
                          inp["u_smp"] if sample else None)


# ---------------------------------------------------------------------------
def test_exp2_extended_precision(gpu_lib):
    rng = np.random.default_rng(0)
    xh = np.concatenate([-rng.random(20000) * 124.0, -rng.random(20000) * 2.0,
                         [0.0, -0.5, -1.0, -124.9]]).astype(np.float32)
    xl = (rng.standard_normal(xh.size) * np.abs(xh) * 2e-8).astype(np.float32)
    xl[-4:] = 0
    out = to_np(gpu_lib.selftest_exp2(torch.from_numpy(xh).to(DEV), torch.from_numpy(xl).to(DEV)))
    ref = np.exp2(xh.astype(np.float64) + xl.astype(np.float64))
    rel = np.abs(out - ref) / ref
    # ~1e-9 relative down to 2^-100 (below that the low half of the pair is
    # subnormal; such weights are < 1e-30 of the row maximum and vanish from
    # every sum)
    normal = xh >= -100
    assert rel[normal].max() < 1e-9, rel[normal].max()
    assert np.abs(out - ref)[~normal].max() < 2.0 ** -120


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("V,dtype", [(1000, torch.float32), (1001, torch.float32),
                                     (128256, torch.bfloat16), (151936, torch.float32),
                                     (7, torch.bfloat16)])
def test_softmax_temp_parity(gpu_lib, V, dtype):
    g = torch.Generator().manual_seed(V)
    rows = 6
    z = (torch.randn((rows, V), generator=g) * 3).to(dtype)
    z[1, V // 3] = float("-inf")
    z[4] = float("-inf")             # all -inf: invalid at T > 0
    z[5, V // 2] = float("nan")      # NaN: invalid
    T = torch.tensor([1.0, 0.7, 0.0, -1.0, 1.0, 1.0])
    r = gpu_lib.ssd_softmax_temp(z.to(DEV), T.to(DEV))
    ref = oracle.softmax_temp(z, T)
    assert np.array_equal(to_np(r["row_argmax"]), ref["row_argmax"])
    gm, rm = to_np(r["row_max"]), ref["row_max"].astype(np.float32)
    assert np.array_equal(np.isnan(gm), np.isnan(rm))
    assert np.array_equal(gm[~np.isnan(gm)], rm[~np.isnan(rm)])
    gs = to_np(r["row_sum"]).astype(np.float64)
    ok = ~np.isnan(ref["row_sum"])
    assert np.array_equal(np.isnan(gs), ~ok)
    assert np.all(np.abs(gs[ok] - ref["row_sum"][ok]) <= 1e-5 * ref["row_sum"][ok])
    gp = to_np(r["probs"]).astype(np.float64)
    assert np.array_equal(np.isnan(gp), np.isnan(ref["probs"]))
    fin = ~np.isnan(gp)
    assert np.max(np.abs(gp[fin] - ref["probs"][fin])) <= 1e-5
    err = gpu_lib.get_device_error(r["ws"], clear=True)
    assert err & gpu_lib.DEVERR_BAD_TEMPERATURE and err & gpu_lib.DEVERR_BAD_LOGITS


def test_softmax_temp_more_rows_than_one_grid(gpu_lib):
    """70000 rows: the launches loop over batches of 65535 grid rows."""
    g = torch.Generator().manual_seed(70000)
    rows, V = 70000, 24
    z = torch.randn((rows, V), generator=g) * 2
    T = torch.rand(rows, generator=g) + 0.5
    T[::7] = 0.0
    r = gpu_lib.ssd_softmax_temp(z.to(DEV), T.to(DEV))
    assert torch.equal(r["row_argmax"].cpu().long(), torch.argmax(z, dim=1))
    assert torch.equal(r["row_max"].cpu(), z.max(dim=1).values)
    sel = np.r_[0:50, 65500:65600, rows - 50:rows]
    ref = oracle.softmax_temp(z[sel], T[sel])
    gp = to_np(r["probs"])[sel].astype(np.float64)
    assert np.max(np.abs(gp - ref["probs"])) <= 1e-5
    assert gpu_lib.get_device_error(r["ws"]) == 0


# ---------------------------------------------------------------------------
CASES = [
    ("tiny", {}, None, 0), ("tiny", {"B": 16}, None, 3),
    ("llama_sd", {}, "0", 0), ("llama_sd", {}, "1.0", 0), ("llama_sd", {"B": 3}, "1.0", 7),
    ("ssd_fork", {}, "0", 0), ("ssd_fork", {}, "1.0", 0), ("ssd_fork", {"B": 2}, "1.0", 11),
    ("qwen_b64", {"B": 4}, None, 0), ("mixed512", {"B": 8}, None, 0),
]


@pytest.mark.parametrize("name,over,temp,dseed", CASES)
def test_verify_parity(gpu_lib, name, over, temp, dseed):
    w = W.workload(name, **over)
    seed = W.default_seed(name) + dseed
    inp = W.make_inputs(w, device=DEV, seed=seed, temp=temp)
    f = w.f if w.ssd and w.f else 0
    out = run_verify(gpu_lib, inp, fork_f=f)
    torch.cuda.synchronize()
    bs = np.arange(w.B)
    ref = oracle_rows(inp, bs)
    rep = compare_verify(inp, out, bs, ref, Report())
    assert not rep.failures, rep.failures[:5]
    assert rep.sampled_mismatch == 0 or rep.sampled_rows >= 10000, rep.summary()
    if f:
        rf = oracle.forked_topf(inp["D"].cpu(), f, inp["mask"].cpu())
        compare_forks(rf, out["fork_tok"], out["fork_logit"], name)
    assert gpu_lib.get_device_error(out["ws"]) == 0


def test_fused_equals_separate_calls(gpu_lib):
    w = W.workload("qwen_b64", B=6)
    inp = W.make_inputs(w, device=DEV, seed=99)
    fused = run_verify(gpu_lib, inp, fork_f=3)
    sep = run_verify(gpu_lib, inp)
    forks = gpu_lib.ssd_forked_recovery(inp["D"], 3, inp["mask"])
    for key in ("accept_len", "out_tok", "p_at_x", "q_at_x"):
        assert torch.equal(fused[key], sep[key]), key
    assert torch.equal(fused["fork_tok"], forks["fork_tok"])
    assert torch.equal(fused["fork_logit"], forks["fork_logit"])


def test_sample_residual_standalone(gpu_lib):
    w = W.workload("qwen_b64", B=5)
    inp = W.make_inputs(w, device=DEV, seed=7)
    a = run_verify(gpu_lib, inp, sample=False)
    tok = gpu_lib.ssd_sample_residual(inp["Z"], inp["D"], inp["x"], inp["T"], a["accept_len"],
                                      inp["u_smp"], a["ws"])
    b = run_verify(gpu_lib, inp, sample=True)
    assert torch.equal(tok, b["out_tok"])
    # a caller-chosen prefix length: n = 0 everywhere draws from the residual of row 0
    n0 = torch.zeros_like(a["accept_len"])
    tok0 = gpu_lib.ssd_sample_residual(inp["Z"], inp["D"], inp["x"], inp["T"], n0,
                                       inp["u_smp"], a["ws"])
    Zc, Dc = inp["Z"].cpu().float().numpy(), inp["D"].cpu().float().numpy()
    us, T = to_np(inp["u_smp"]), to_np(inp["T"])
    for r in range(w.B):
        p = oracle.softmax_temp(Zc[r, :1], [T[r]])["probs"][0]
        q = oracle.softmax_temp(Dc[r, :1], [T[r]])["probs"][0]
        wv = np.maximum(0, p - q)
        C = np.cumsum(wv)
        j = int(tok0[r, 0])
        t = us[r] * C[-1]
        assert (C[j - 1] if j else 0) - 1e-12 <= t < C[j] + 1e-12


def test_forked_recovery_ties_masks_nan(gpu_lib):
    B, P, V, f = 3, 5, 5000, 16
    g = torch.Generator().manual_seed(3)
    L = torch.randint(-8, 8, (B, P, V), generator=g).float() / 2  # heavy ties
    L[0, 1, 100] = float("nan")
    L[1, 2] = float("-inf")
    L[1, 2, 4999] = 1.0
    mask = torch.randint(-1, V, (B, P, 4), generator=g, dtype=torch.int32)
    for dtype in (torch.float32, torch.bfloat16):
        Lt = L.to(dtype)
        r = gpu_lib.ssd_forked_recovery(Lt.to(DEV), f, mask.to(DEV))
        ref = oracle.forked_topf(Lt, f, mask)
        compare_forks(ref, r["fork_tok"], r["fork_logit"], str(dtype))


@pytest.mark.parametrize("name,over,fan", [
    ("ssd_fork", {}, [3, 2, 2, 1, 1, 1, 0, 3]),
    ("mixed512", {"B": 8}, [4, 4, 3, 3, 2, 2, 1, 0]),
    ("qwen_b64", {"B": 5}, [0, 1, 2, 3, 1, 2]),
])
def test_variable_fanout(gpu_lib, name, over, fan):
    """Per-position fan-out f_j: standalone and fused calls against the
    oracle; padded slots are skipped by the cache insert."""
    w = W.workload(name, **over)
    inp = W.make_inputs(w, device=DEV, seed=W.default_seed(name) + 40)
    fanout = torch.tensor(fan, dtype=torch.int32, device=DEV)
    ref = oracle.forked_topf(inp["D"].cpu(), w.f, inp["mask"].cpu(), fanout=fan)
    alone = gpu_lib.ssd_forked_recovery(inp["D"], w.f, inp["mask"], fanout=fanout)
    compare_forks(ref, alone["fork_tok"], alone["fork_logit"], name)
    fused = gpu_lib.ssd_verify_fork(inp["Z"], inp["D"], inp["x"], inp["T"], inp["u_acc"],
                                    inp["u_smp"], w.f, inp["mask"], fanout=fanout)
    compare_forks(ref, fused["fork_tok"], fused["fork_logit"], name)
    plain = run_verify(gpu_lib, inp, fork_f=w.f)
    for key in ("accept_len", "out_tok", "p_at_x", "q_at_x"):
        assert torch.equal(fused[key], plain[key]), key
    cache = gpu_lib.SpecCache(256 if w.B * (w.k + 1) * w.f < 128 else 4096, 2)
    pay = torch.arange(w.B * (w.k + 1) * w.f * 2, dtype=torch.int32, device=DEV).reshape(-1, 2)
    cache.insert_forks(fused["fork_tok"], pay)
    bb = torch.arange(w.B, device=DEV, dtype=torch.int32).repeat_interleave((w.k + 1) * w.f)
    pp = torch.arange(w.k + 1, device=DEV, dtype=torch.int32).repeat_interleave(w.f).repeat(w.B)
    tt = fused["fork_tok"].reshape(-1)
    valid = tt >= 0
    look = cache.lookup(bb[valid].contiguous(), pp[valid].contiguous(), tt[valid].contiguous())
    assert bool((look["hit"] == 1).all())
    assert torch.equal(look["tok_out"], pay[valid])
    assert cache.error() == 0
    cache.close()


def test_forked_recovery_constant_rows_use_exact_fallback(gpu_lib):
    """Rows whose logits are all equal put every element at the candidate
    bound, overflowing the candidate buffer: the exact fallback must still
    return the lowest unmasked indices."""
    B, P, V, f = 2, 3, 40000, 16
    L = torch.zeros((B, P, V))
    L[0, 1] = float("-inf")
    L[1, 2, ::7] = 2.5
    mask = torch.tensor([[[0, 3], [1, -1], [5, 9]], [[2, 2], [7, 14], [0, 21]]], dtype=torch.int32)
    for dtype in (torch.float32, torch.bfloat16):
        Lt = L.to(dtype)
        r = gpu_lib.ssd_forked_recovery(Lt.to(DEV), f, mask.to(DEV))
        ref = oracle.forked_topf(Lt, f, mask)
        compare_forks(ref, r["fork_tok"], r["fork_logit"], str(dtype))


# ---------------------------------------------------------------------------
def test_spec_cache_ssd_workload(gpu_lib):
    w = W.workload("ssd_fork")
    inp = W.make_inputs(w, device=DEV, temp="1.0")
    out = run_verify(gpu_lib, inp, fork_f=3)
    depth, cap = 7, 64
    cw = W.cache_workload(out["fork_tok"], depth, w.V, 10000, seed=5)
    cache = gpu_lib.SpecCache(cap, depth)
    ref = oracle.SpecCacheOracle(depth)
    d = lambda t: t.to(DEV)
    cache.insert(d(cw["ins_b"]), d(cw["ins_pos"]), d(cw["ins_tok"]), d(cw["payload"]))
    ref.insert(cw["ins_b"], cw["ins_pos"], cw["ins_tok"], cw["payload"].numpy())
    got = cache.lookup(d(cw["q_b"]), d(cw["q_pos"]), d(cw["q_tok"]))
    hit, tok = ref.lookup(cw["q_b"], cw["q_pos"], cw["q_tok"])
    assert np.array_equal(to_np(got["hit"]), hit)
    assert np.array_equal(to_np(got["tok_out"]), tok)
    assert 0.45 < hit.mean() < 0.55
    # the realised outcome of the verify step, looked up on the device
    oc = cache.lookup_outcome(out["accept_len"], out["out_tok"])
    n = int(out["accept_len"][0])
    h2, t2 = ref.lookup([0], [n], [int(out["out_tok"][0, n])])
    assert int(oc["hit"][0]) == h2[0] and np.array_equal(to_np(oc["tok_out"])[0], t2[0])
    # insert_forks builds the same keys as the explicit insert
    cache2 = gpu_lib.SpecCache(cap, depth)
    pay = torch.arange(w.B * (w.k + 1) * 3 * depth, dtype=torch.int32).view(-1, depth)
    cache2.insert_forks(out["fork_tok"], pay.to(DEV))
    ft = to_np(out["fork_tok"]).reshape(-1)
    qb = torch.zeros(ft.size, dtype=torch.int32)
    qp = torch.arange(w.k + 1, dtype=torch.int32).repeat_interleave(3)
    g2 = cache2.lookup(d(qb), d(qp), torch.from_numpy(ft).to(DEV))
    ref2 = oracle.SpecCacheOracle(depth)
    ref2.insert(qb.numpy(), qp.numpy(), ft, pay.numpy())
    h3, t3 = ref2.lookup(qb.numpy(), qp.numpy(), ft)
    assert np.array_equal(to_np(g2["hit"]), h3) and np.array_equal(to_np(g2["tok_out"]), t3)
    assert cache.error() == 0
    cache.clear()
    got = cache.lookup(d(cw["q_b"]), d(cw["q_pos"]), d(cw["q_tok"]))
    assert int(got["hit"].sum()) == 0


@pytest.mark.parametrize("name,over", [("ssd_fork", {}), ("mixed512", {"B": 64}),
                                       ("qwen_b64", {})])
def test_fused_round_step_equals_separate_calls(gpu_lib, name, over):
    """ssd_verify_fork_cache (the forks inserted on a side stream while the
    draw runs, for B >= 32) gives what the separate calls give."""
    w = W.workload(name, **over)
    inp = W.make_inputs(w, device=DEV, seed=W.default_seed(name) + 55)
    depth = 5
    n = w.B * (w.k + 1) * w.f
    cap = 1 << max(6, (2 * n - 1).bit_length())
    pay = torch.arange(n * depth, dtype=torch.int32, device=DEV).reshape(n, depth)
    c1, c2 = gpu_lib.SpecCache(cap, depth), gpu_lib.SpecCache(cap, depth)
    for rep in range(2):  # the second round also checks the clear
        fused = gpu_lib.ssd_verify_fork_cache(inp["Z"], inp["D"], inp["x"], inp["T"], inp["u_acc"],
                                              inp["u_smp"], w.f, inp["mask"], c1, pay + rep)
        sep = run_verify(gpu_lib, inp, fork_f=w.f)
        c2.clear()
        c2.insert_forks(sep["fork_tok"], pay + rep)
        look = c2.lookup_outcome(sep["accept_len"], sep["out_tok"])
        torch.cuda.synchronize()
        for key in ("accept_len", "out_tok", "p_at_x", "q_at_x", "fork_tok", "fork_logit"):
            assert torch.equal(fused[key], sep[key]), key
        assert torch.equal(fused["hit"], look["hit"])
        assert torch.equal(fused["tok_out"], look["tok_out"])
    assert c1.error() == 0
    c1.close()
    c2.close()


def test_spec_cache_duplicates_and_overflow(gpu_lib):
    cache = gpu_lib.SpecCache(8, 2)
    b = torch.tensor([0, 0, 0, 1], dtype=torch.int32, device=DEV)
    pos = torch.tensor([1, 1, 1, 1], dtype=torch.int32, device=DEV)
    tok = torch.tensor([5, 5, 5, 5], dtype=torch.int32, device=DEV)
    pay = torch.tensor([[1, 1], [2, 2], [3, 3], [4, 4]], dtype=torch.int32, device=DEV)
    cache.insert(b, pos, tok, pay)
    r = cache.lookup(b[:2], pos[:2], tok[:2])
    assert to_np(r["tok_out"]).tolist() == [[3, 3], [3, 3]]
    cache.insert(b[:1], pos[:1], tok[:1], pay[3:4] * 10)   # a later call wins
    assert to_np(cache.lookup(b[:1], pos[:1], tok[:1])["tok_out"]).tolist() == [[40, 40]]
    # 20 distinct keys into 8 slots: 6 more fit, the rest are dropped
    n = 20
    kb = torch.arange(n, dtype=torch.int32, device=DEV) + 10
    cache.insert(kb, torch.zeros_like(kb), torch.zeros_like(kb),
                 torch.zeros((n, 2), dtype=torch.int32, device=DEV))
    assert cache.error(clear=True) & gpu_lib.DEVERR_CACHE_FULL
    hits = cache.lookup(kb, torch.zeros_like(kb), torch.zeros_like(kb))["hit"]
    assert int(hits.sum()) == 6
    assert cache.error() == 0


# ---------------------------------------------------------------------------
def test_edge_cases_sentinels(gpu_lib):
    B, k, V = 6, 3, 2048
    g = torch.Generator().manual_seed(1)
    Z = torch.randn((B, k + 1, V), generator=g)
    D = Z[:, :k] + 0.5 * torch.randn((B, k, V), generator=g)
    x = torch.randint(0, V, (B, k), generator=g, dtype=torch.int32)
    T = torch.tensor([1.0, -0.5, 1.0, 1.0, 0.0, 1.0])
    x[2, 1] = V                        # bad token: -2
    Z[3, 2, 17] = float("nan")         # NaN: -1
    Z[4, 0] = float("-inf")            # greedy row, all -inf: still valid
    Z[5, 1, :] = float("-inf")
    Z[5, 1, 3] = 0.0                   # mostly -inf: valid
    inp = {"Z": Z.to(DEV), "D": D.contiguous().to(DEV), "x": x.to(DEV), "T": T.to(DEV),
           "u_acc": torch.rand((B, k), generator=g).to(DEV),
           "u_smp": torch.rand(B, generator=g).to(DEV)}
    out = run_verify(gpu_lib, inp)
    ref = oracle_rows(inp, np.arange(B))
    assert list(to_np(out["accept_len"])[:4]) == [int(v) for v in ref["accept_len"][:4]]
    assert list(ref["accept_len"][1:4]) == [-1, -2, -1]
    rep = compare_verify(inp, out, np.arange(B), ref, Report())
    assert not rep.failures, rep.failures
    err = gpu_lib.get_device_error(out["ws"], clear=True)
    assert err == (gpu_lib.DEVERR_BAD_TEMPERATURE | gpu_lib.DEVERR_BAD_TOKEN |
                   gpu_lib.DEVERR_BAD_LOGITS)
    assert gpu_lib.get_device_error(out["ws"]) == 0


@pytest.mark.parametrize("B,k,V,f,dtype", [(3, 1, 2, 1, torch.float32),
                                           (2, 31, 1001, 16, torch.float32),
                                           (2, 4, 4099, 5, torch.bfloat16)])
def test_extreme_sizes(gpu_lib, B, k, V, f, dtype):
    g = torch.Generator().manual_seed(V)
    Z = (torch.randn((B, k + 1, V), generator=g) * 2).to(dtype)
    D = (Z.float() + torch.randn((B, k + 1, V), generator=g)).to(dtype)
    x = torch.randint(0, V, (B, k), generator=g, dtype=torch.int32)
    x[:, : k // 2] = torch.argmax(Z.float()[:, : k // 2], dim=2).int()
    T = torch.tensor([1.0, 0.0, 0.8][:B])
    mask = torch.cat([x, x[:, :1]], dim=1)[:, :, None].contiguous()
    inp = {"Z": Z.to(DEV), "D": D.to(DEV), "x": x.to(DEV), "T": T.to(DEV), "mask": mask.to(DEV),
           "u_acc": torch.rand((B, k), generator=g).to(DEV),
           "u_smp": torch.rand(B, generator=g).to(DEV)}
    out = run_verify(gpu_lib, inp, fork_f=f)
    ref = oracle_rows(inp, np.arange(B))
    rep = compare_verify(inp, out, np.arange(B), ref, Report())
    assert not rep.failures, rep.failures
    compare_forks(oracle.forked_topf(D, f, mask), out["fork_tok"], out["fork_logit"])


def test_unaligned_rows_use_scalar_path(gpu_lib):
    # a batch stride that is not a multiple of 4 floats forces scalar loads
    B, k, V = 3, 2, 3001
    g = torch.Generator().manual_seed(2)
    Zbig = torch.randn((B, (k + 1) * V + 1), generator=g)
    Z = Zbig[:, : (k + 1) * V].reshape(B, k + 1, V)
    D = (Z[:, :k] + torch.randn((B, k, V), generator=g)).contiguous()
    x = torch.randint(0, V, (B, k), generator=g, dtype=torch.int32)
    T = torch.tensor([1.0, 0.9, 0.0])
    lib = gpu_lib.load_library()
    Zd = Zbig.to(DEV)
    ws = gpu_lib.new_workspace(gpu_lib.workspace_bytes(B, k, V, 0), DEV)
    wp = ws.data_ptr() + ((-ws.data_ptr()) % 256)
    acc = torch.empty(B, dtype=torch.int32, device=DEV)
    pq = torch.empty((2, B, k), device=DEV)
    out = torch.empty((B, k + 1), dtype=torch.int32, device=DEV)
    Dd, xd, Td = D.to(DEV), x.to(DEV), T.to(DEV)
    ua, us = torch.rand((B, k), generator=g).to(DEV), torch.rand(B, generator=g).to(DEV)
    st = lib.ssd_verify(Zd.data_ptr(), (k + 1) * V + 1, Dd.data_ptr(), k * V, 0, B, k, V,
                        xd.data_ptr(), Td.data_ptr(), ua.data_ptr(), acc.data_ptr(),
                        pq[0].data_ptr(), pq[1].data_ptr(), us.data_ptr(), out.data_ptr(), wp,
                        ws.numel() - 256, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    inp = {"Z": Z.contiguous(), "D": D, "x": x, "T": T, "u_acc": ua.cpu(), "u_smp": us.cpu()}
    ref = oracle_rows(inp, np.arange(B))
    gpu = {"accept_len": acc, "out_tok": out, "p_at_x": pq[0], "q_at_x": pq[1]}
    rep = compare_verify(inp, gpu, np.arange(B), ref, Report())
    assert not rep.failures, rep.failures


# ---------------------------------------------------------------------------
def test_full_size_bench_workload_sampled(gpu_lib):
    """mixed512 at full size in the benchmark's launch configuration: a sample
    of batch rows against the oracle, every row against invariants."""
    w = W.workload("mixed512")
    inp = W.make_inputs(w, device=DEV)
    out = run_verify(gpu_lib, inp, fork_f=w.f)
    torch.cuda.synchronize()
    bs = np.linspace(0, w.B - 1, 12).astype(int)
    ref = oracle_rows(inp, bs)
    rep = compare_verify(inp, out, bs, ref, Report())
    assert not rep.failures, rep.failures
    rf = oracle.forked_topf(inp["D"][bs].cpu(), w.f, inp["mask"][bs].cpu())
    compare_forks(rf, out["fork_tok"][bs], out["fork_logit"][bs])
    # invariants on every row
    acc = out["accept_len"]
    assert int(acc.min()) >= 0 and int(acc.max()) <= w.k
    ar = torch.arange(w.k + 1, device=DEV)[None]
    prefix = ar[:, :w.k] < acc[:, None]
    assert torch.equal(torch.where(prefix, inp["x"], 0), torch.where(prefix, out["out_tok"][:, :w.k], 0))
    assert bool((out["out_tok"].gather(1, acc[:, None].long()) >= 0).all())
    greedy = inp["T"] == 0
    am = torch.argmax(inp["Z"].float(), dim=2)          # first maximum on ties
    match = (inp["x"] == am[:, :w.k]).int()
    n_ref = torch.cumprod(match, dim=1).sum(1)
    assert torch.equal(acc[greedy].long(), n_ref[greedy])
    tok_ref = am.gather(1, n_ref[:, None])[:, 0]
    assert torch.equal(out["out_tok"].gather(1, acc[:, None].long())[greedy, 0].long(), tok_ref[greedy])
    assert gpu_lib.get_device_error(out["ws"]) == 0


def test_full_size_qwen_batch(gpu_lib):
    w = W.workload("qwen_b64")
    inp = W.make_inputs(w, device=DEV)
    out = run_verify(gpu_lib, inp, fork_f=w.f)
    bs = np.arange(w.B)
    ref = oracle_rows(inp, bs)
    rep = compare_verify(inp, out, bs, ref, Report())
    assert not rep.failures, rep.failures
    compare_forks(oracle.forked_topf(inp["D"].cpu(), w.f, inp["mask"].cpu()),
                  out["fork_tok"], out["fork_logit"])


def test_residual_extremes_large_chunks(gpu_lib):
    """Residual draws at the largest chunk sums and with overflowing
    ambiguous-sign lists (bf16, B=64: chunks of ~15K elements).
    Rows 0 mod 4: flat target (p uniform) against a peaked draft, so nearly
    every element sits on the positive side of p - q.  Rows 1 mod 4: the draft
    equals the target except at the draft token, a token of target
    probability ~1e-4 raised by 0.25, so |p - q| is below 1e-3 (p + q) on
    every other element.  u_acc = 0.999 rejects early."""
    w = W.workload("qwen_b64", temp="1.0")
    inp = W.make_inputs(w, device=DEV, seed=321)
    Z, D, x = inp["Z"].clone(), inp["D"].clone(), inp["x"].clone()
    Z[0::4] = 1.0
    for b in range(1, w.B, 4):
        for j in range(w.k):
            lp = torch.log_softmax(Z[b, j].float(), dim=0)
            v = int(torch.argmin((lp - np.log(1e-4)).abs()))
            x[b, j] = v
            D[b, j] = Z[b, j]
            D[b, j, v] += 0.25
    inp["Z"], inp["D"], inp["x"] = Z, D, x
    inp["u_acc"] = torch.full_like(inp["u_acc"], 0.999)
    out = run_verify(gpu_lib, inp, fork_f=w.f)
    torch.cuda.synchronize()
    bs = np.concatenate([np.arange(0, w.B, 4)[:8], np.arange(1, w.B, 4)[:8], [2, 3]])
    ref = oracle_rows(inp, bs)
    assert (ref["accept_len"][:16] < w.k).all()
    rep = compare_verify(inp, out, bs, ref, Report())
    assert not rep.failures, rep.failures[:5]
    assert rep.sampled_mismatch == 0, rep.summary()
    assert gpu_lib.get_device_error(out["ws"]) == 0


def test_sampled_token_agreement_rate(gpu_lib):
    """>= 99.99% identical draws over 12288 stochastic rows, every mismatch
    traced to a uniform within 1e-6 of a CDF boundary."""
    rep = Report()
    for s in range(3):
        w = W.Workload("rate32k", 4096, 1, 0, 32000, "f32", 3.0, 1.0, 5, 8.0, "uniform",
                       "stochastic", False)
        inp = W.make_inputs(w, device=DEV, seed=500 + s)
        out = run_verify(gpu_lib, inp)
        bs = np.arange(w.B)
        compare_verify(inp, out, bs, oracle_rows(inp, bs), rep)
    assert not rep.failures, rep.failures[:5]
    assert rep.sampled_rows >= 10000
    assert rep.sampled_mismatch <= 1e-4 * rep.rows, rep.summary()
    print(rep.summary())


@pytest.mark.parametrize("u", [0.0, float(np.nextafter(np.float32(1.0), np.float32(0.0)))])
def test_uniforms_at_the_ends(gpu_lib, u):
    """u = 0 and the largest binary32 below 1, for every acceptance and draw:
    u = 0 accepts every draft token with p(x) > 0 and draws the first token
    of positive weight (exact on both sides); u just below 1 rejects unless
    p(x)/q(x) >= 1 and draws near the end of the CDF (compared with the
    boundary rule)."""
    w = W.workload("llama_sd", B=12)
    inp = W.make_inputs(w, device=DEV, seed=515, temp="stochastic")
    inp["u_acc"].fill_(u)
    inp["u_smp"].fill_(u)
    out = run_verify(gpu_lib, inp)
    torch.cuda.synchronize()
    ref = oracle_rows(inp, np.arange(w.B))
    if u == 0.0:
        assert np.array_equal(to_np(out["accept_len"]), ref["accept_len"])
        assert np.array_equal(to_np(out["out_tok"]), ref["out_tok"])
        assert (ref["accept_len"] == w.k).all()
    rep = compare_verify(inp, out, np.arange(w.B), ref, Report())
    assert not rep.failures, rep.failures
    tr = W.make_tree_inputs(12, W.tree_parents((3, 2)), 4096, temp="stochastic", seed=516,
                            device=DEV)
    tr["u_acc"].fill_(u)
    tr["u_smp"].fill_(u)
    to = gpu_lib.ssd_verify_tree(tr["Z"], tr["D"], tr["parent"], tr["tok"], tr["T"],
                                 tr["u_acc"], tr["u_smp"])
    torch.cuda.synchronize()
    tc = {k: v.cpu() for k, v in tr.items()}
    rt = oracle.verify_tree(tc["Z"], tc["D"], tc["parent"], tc["tok"], tc["T"], tc["u_acc"],
                            tc["u_smp"])
    if u == 0.0:
        for key in ("accept_len", "out_tok", "out_node"):
            assert np.array_equal(to_np(to[key]), rt[key]), key
        assert (rt["accept_len"] == 2).all()      # the first child at every level
