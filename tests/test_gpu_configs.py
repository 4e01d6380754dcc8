"""Every configuration of the workload table at full size, element by element
against the oracle, in the launch configuration the benchmark times.

For each configuration, batches drawn with fresh seeds until at least 10^4
stochastic batch rows have been compared (greedy rows on top where the
configuration has them), each through the call that configuration's
benchmark line times:

  llama_sd   B = 1 per call (ssd_verify), V = 128256 bf16, T = 1 and T = 0
  ssd_fork   B = 1 per call (ssd_verify_fork_cache: forks, cache clear /
             insert / outcome lookup), V = 128256 bf16, T = 1 and T = 0
  qwen_b64   B = 64 per call (ssd_verify_fork_cache), V = 151936 bf16, T = 0.7
  mixed512   B = 512 per call (ssd_verify_fork_cache), V = 151936 fp32,
             half the rows greedy

Rules (exactness of speculative sampling, "SSD: drafting and verification
on separate GPUs", "What changes in SSD"; the matching rules of the
workload table): greedy tokens and accept lengths bit-exact; p(x), q(x)
within 1e-5; sampled rows identical on >= 99.99% of the stochastic rows,
every difference traced to a uniform within 1e-6 of the decision it flips;
forked tokens, their logits and the cache lookups bit-exact.  The oracle runs
on the host cores (threads; its C entry points release the GIL).
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import (Report, compare_forks, compare_verify, host_threads,
                         oracle_forks_host, oracle_verify_host, to_np)
from speculative_decoding_verification_70_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
DEPTH = 7                  # speculation-cache payload tokens per entry
MIN_STOCHASTIC = 10000     # stochastic rows compared per configuration
RATE = 1e-4                # at most this fraction of stochastic rows may differ


def _cache_oracle(fork_tok, payload, accept_len, out_tok, b_ids):
    """The dict cache: insert every forked token (b, j, tok) -> its payload
    row in input order (the insert skips token -1), then look up each row's
    realised outcome (b, n, out_tok[b, n])."""
    B, P, f = fork_tok.shape
    c = oracle.SpecCacheOracle(payload.shape[1])
    bb = np.repeat(b_ids, P * f)
    pp = np.tile(np.repeat(np.arange(P), f), B)
    ft = fork_tok.reshape(-1)
    keep = ft >= 0
    c.insert(bb[keep], pp[keep], ft[keep], payload[keep])
    n = accept_len
    tok = np.where(n >= 0, out_tok[np.arange(B), np.clip(n, 0, None)], -1)
    return c.lookup(b_ids, n, tok)


def _account(name, rep, extra=""):
    stoch = rep.sampled_rows + rep.accept_flips
    differ = rep.sampled_mismatch + rep.accept_flips
    print("PARITY %s: %s stochastic %d differing %d (%.2e)%s"
          % (name, rep.summary(), stoch, differ, differ / max(1, stoch), extra))
    assert not rep.failures, rep.failures[:5]
    return stoch, differ


def _check_rate(stoch, differ, need):
    assert stoch >= need, stoch
    assert differ <= RATE * stoch, (differ, stoch)


def _per_row_calls(ssd, w, inp, forks, cache, payload):
    """One B = 1 call per batch row (the single-sequence launch shape),
    writing into slices of batch-sized outputs; one workspace for all."""
    B, k = w.B, w.k
    out = {"accept_len": torch.empty(B, dtype=torch.int32, device=DEV),
           "p_at_x": torch.empty((B, k), device=DEV),
           "q_at_x": torch.empty((B, k), device=DEV),
           "out_tok": torch.empty((B, k + 1), dtype=torch.int32, device=DEV)}
    if forks:
        out["fork_tok"] = torch.empty((B, k + 1, w.f), dtype=torch.int32, device=DEV)
        out["fork_logit"] = torch.empty((B, k + 1, w.f), device=DEV)
        out["hit"] = torch.empty(B, dtype=torch.int32, device=DEV)
        out["tok_out"] = torch.empty((B, DEPTH), dtype=torch.int32, device=DEV)
    ws = ssd.new_workspace(ssd.workspace_bytes(1, k, w.V, w.f if forks else 0), DEV)
    per = (k + 1) * w.f
    for b in range(B):
        sl = slice(b, b + 1)
        o = {key: v[sl] for key, v in out.items()}
        if forks:
            ssd.ssd_verify_fork_cache(inp["Z"][sl], inp["D"][sl], inp["x"][sl], inp["T"][sl],
                                      inp["u_acc"][sl], inp["u_smp"][sl], w.f, inp["mask"][sl],
                                      cache, payload[b * per:(b + 1) * per], ws=ws, out=o)
        else:
            ssd.ssd_verify(inp["Z"][sl], inp["D"][sl], inp["x"][sl], inp["T"][sl],
                           inp["u_acc"][sl], inp["u_smp"][sl], ws=ws, out=o)
    out["ws"] = ws
    return out


def _compare_batch(w, cpu, out, rep, forks, payload, per_row):
    bs = np.arange(w.B)
    ref = oracle_verify_host(cpu)
    compare_verify(cpu, out, bs, ref, rep)
    if not forks:
        return
    rf = oracle_forks_host(cpu["D"], w.f, cpu["mask"])
    compare_forks(rf, out["fork_tok"], out["fork_logit"], w.name)
    # the cache sees the GPU's own outcome (compare_verify has checked it)
    acc, otok = to_np(out["accept_len"]), to_np(out["out_tok"])
    pay = to_np(payload)
    if per_row:   # each call cleared the cache and used batch index 0
        per = (w.k + 1) * w.f
        hits, toks = [], []
        for b in range(w.B):
            h, t = _cache_oracle(rf["fork_tok"][b:b + 1], pay[b * per:(b + 1) * per],
                                 acc[b:b + 1], otok[b:b + 1], np.zeros(1, dtype=np.int64))
            hits.append(h)
            toks.append(t)
        hit, tok = np.concatenate(hits), np.concatenate(toks)
    else:
        hit, tok = _cache_oracle(rf["fork_tok"], pay, acc, otok, bs)
    assert np.array_equal(to_np(out["hit"]), hit)
    assert np.array_equal(to_np(out["tok_out"]), tok)


CONFIGS = [
    # name, per-call B, temperature override, batches, batch rows per batch, stochastic
    ("llama_sd", 1, "1.0", 40, 256, True),
    ("llama_sd", 1, "0", 4, 256, False),
    ("ssd_fork", 1, "1.0", 40, 256, True),
    ("ssd_fork", 1, "0", 4, 256, False),
    ("qwen_b64", 64, None, 160, 64, True),
    ("mixed512", 512, None, 40, 512, True),
]


@pytest.mark.parametrize("name,call_B,temp,batches,rows,stochastic", CONFIGS)
def test_config_full_size_against_oracle(gpu_lib, name, call_B, temp, batches, rows, stochastic):
    ssd = gpu_lib
    w = W.workload(name, B=rows)
    forks = w.ssd and w.f > 0
    per_row = call_B == 1
    cache = ssd.SpecCache(1 << max(6, (2 * call_B * (w.k + 1) * w.f - 1).bit_length()),
                          DEPTH) if forks else None
    rep = Report()
    g = torch.Generator(device=DEV).manual_seed(4000 + W.ORDER.index(name))
    for i in range(batches):
        seed = W.default_seed(name) + 1000 * (i + 1) + (0 if stochastic else 777)
        inp = W.make_inputs(w, device=DEV, seed=seed, temp=temp)
        payload = torch.randint(0, w.V, (rows * (w.k + 1) * max(w.f, 1), DEPTH), generator=g,
                                device=DEV, dtype=torch.int32)
        if per_row:
            out = _per_row_calls(ssd, w, inp, forks, cache, payload)
        elif forks:
            out = ssd.ssd_verify_fork_cache(inp["Z"], inp["D"], inp["x"], inp["T"],
                                            inp["u_acc"], inp["u_smp"], w.f, inp["mask"], cache,
                                            payload)
        else:
            out = ssd.ssd_verify(inp["Z"], inp["D"], inp["x"], inp["T"], inp["u_acc"],
                                 inp["u_smp"])
        torch.cuda.synchronize()
        assert ssd.get_device_error(out["ws"]) == 0
        cpu = {key: v.cpu() for key, v in inp.items()}
        del inp
        _compare_batch(w, cpu, out, rep, forks, payload, per_row)
        del cpu, out
    if cache is not None:
        assert cache.error() == 0
        cache.close()
    stoch, differ = _account("%s T=%s B/call=%d" % (name, temp or w.temp, call_B), rep,
                             " threads %d" % host_threads())
    if stochastic:
        _check_rate(stoch, differ, MIN_STOCHASTIC)
    else:
        assert rep.greedy_rows == batches * rows
