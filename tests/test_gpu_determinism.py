"""Determinism of the CUDA path: repeated calls give bit-identical outputs,
and the vocabulary split (chunks per row, chunks per statistics CTA) does
not change any integer result.

Partial statistics are merged in chunk order and everything the draw sums
above a thread is exact fixed point, so the accept lengths, the output
tokens, the forked tokens and their logits, and the cache lookups are the
same for one chunk per row and for up to 256.  The float outputs p(x), q(x)
come from per-chunk float sums that round differently under another split,
so they are compared within 1e-6 (the parity tolerance is 1e-5).
"""
import numpy as np
import pytest
import torch

from parity_util import Report, compare_verify, oracle_rows
from speculative_decoding_verification_70_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
INT_KEYS = ("accept_len", "out_tok", "fork_tok", "fork_logit")


@pytest.fixture
def split(gpu_lib):
    yield gpu_lib.set_split
    gpu_lib.set_split(0, 0)


def _run(ssd, inp, f):
    out = ssd.ssd_verify_fork(inp["Z"], inp["D"], inp["x"], inp["T"], inp["u_acc"],
                              inp["u_smp"], f, inp["mask"])
    torch.cuda.synchronize()
    return {k: v.clone() for k, v in out.items() if k != "ws"}


def test_repeated_calls_are_bit_identical(gpu_lib):
    w = W.workload("mixed512", B=32)
    inp = W.make_inputs(w, device=DEV, seed=77)
    a = _run(gpu_lib, inp, w.f)
    b = _run(gpu_lib, inp, w.f)
    for key in a:
        assert torch.equal(a[key], b[key]), key


# (workload, overrides, splits: (chunk elements, chunks per CTA))
CASES = [
    # V = 8000 fp32: one chunk per row (8000 elements) up to 125 chunks of 64
    ("tiny", {"B": 24, "V": 8000, "temp": "mixed"},
     [(0, 0), (8000, 1), (1000, 1), (1000, 8), (64, 1), (64, 4), (200, 40)]),
    # the vocabulary of the large workloads: 10 to 254 chunks per row
    ("qwen_b64", {"B": 6}, [(0, 0), (16384, 1), (16384, 10), (2048, 4), (600, 1), (600, 32)]),
]


@pytest.mark.parametrize("name,over,splits", CASES)
def test_split_does_not_change_results(gpu_lib, split, name, over, splits):
    w = W.workload(name, **over)
    inp = W.make_inputs(w, device=DEV, seed=91)
    f = w.f
    outs = []
    for ch, g in splits:
        split(ch, g)
        outs.append(_run(gpu_lib, inp, f))
    ref = outs[0]
    for (ch, g), o in zip(splits[1:], outs[1:]):
        for key in INT_KEYS:
            assert torch.equal(o[key], ref[key]), (ch, g, key)
        ok = ref["accept_len"] >= 0
        for key in ("p_at_x", "q_at_x"):
            d = (o[key][ok] - ref[key][ok]).abs().max().item() if ok.any() else 0.0
            assert d <= 1e-6, (ch, g, key, d)
    # and the default split agrees with the oracle on these rows
    bs = np.arange(w.B)
    rep = compare_verify(inp, ref, bs, oracle_rows(inp, bs), Report())
    assert not rep.failures, rep.failures[:3]

