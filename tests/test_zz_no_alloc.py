"""ssd_verify_noalloc: the verify call for callers that cannot allocate device
memory (for example code running inside a framework that owns every
allocation).  It uses a static device array as its scratch instead of a
caller-supplied workspace.  These tests call it through the C ABI and check
that it returns exactly what ssd_verify returns, on two calls in a row (the
array keeps the previous call's contents), that its results agree with the
oracle under the parity rules (it runs a one-stream schedule of its own),
and that sizes beyond the array are refused on the host.

This file is collected last so that a failure here leaves every other test
already run.
"""
import numpy as np
import pytest
import torch

from parity_util import Report, compare_verify, oracle_rows
from speculative_decoding_verification_70_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SSD_ERR_WORKSPACE = 6
SCRATCH_BYTES = 8 << 20


def _noalloc(lib, inp):
    Z, D = inp["Z"], inp["D"]
    B, kp1, V = Z.shape
    k = kp1 - 1
    dev = Z.device
    out = {"accept_len": torch.full((B,), -7, dtype=torch.int32, device=dev),
           "p_at_x": torch.full((B, k), -7.0, device=dev),
           "q_at_x": torch.full((B, k), -7.0, device=dev),
           "out_tok": torch.full((B, k + 1), -7, dtype=torch.int32, device=dev)}
    st = lib.ssd_verify_noalloc(
        Z.data_ptr(), kp1 * V, D.data_ptr(), D.shape[1] * V, 1 if Z.dtype == torch.bfloat16 else 0,
        B, k, V, inp["x"].data_ptr(), inp["T"].data_ptr(), inp["u_acc"].data_ptr(),
        out["accept_len"].data_ptr(), out["p_at_x"].data_ptr(), out["q_at_x"].data_ptr(),
        inp["u_smp"].data_ptr(), out["out_tok"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    return st, out


def test_noalloc_matches_verify_twice(gpu_lib):
    lib = gpu_lib.load_library()
    cases = [(W.workload("qwen_b64", B=8), 31), (W.workload("mixed512", B=6), 32)]
    for w, seed in cases:
        inp = W.make_inputs(w, device="cuda", seed=seed)
        assert gpu_lib.workspace_bytes(w.B, w.k, w.V, 0) <= SCRATCH_BYTES
        ref = gpu_lib.ssd_verify(inp["Z"], inp["D"], inp["x"], inp["T"], inp["u_acc"],
                                 inp["u_smp"])
        st, got = _noalloc(lib, inp)
        torch.cuda.synchronize()
        assert st == 0
        assert torch.equal(got["accept_len"], ref["accept_len"])
        assert torch.equal(got["out_tok"], ref["out_tok"])
        both = ref["accept_len"] >= 0
        assert torch.allclose(got["p_at_x"][both], ref["p_at_x"][both], atol=1e-5, rtol=0)
        assert torch.allclose(got["q_at_x"][both], ref["q_at_x"][both], atol=1e-5, rtol=0)
        # and directly against the oracle on the same rows
        bs = np.arange(w.B)
        rep = compare_verify(inp, got, bs, oracle_rows(inp, bs), Report())
        assert not rep.failures, rep.failures[:3]
        assert rep.sampled_mismatch == 0, rep.summary()


def test_noalloc_refuses_sizes_beyond_the_array(gpu_lib):
    lib = gpu_lib.load_library()
    B, k, V = 4096, 7, 151936
    assert gpu_lib.workspace_bytes(B, k, V, 0) > SCRATCH_BYTES
    # no device pointer at all: the size check refuses first, and were it
    # ever to pass, the null-pointer check would refuse before any launch
    st = lib.ssd_verify_noalloc(None, (k + 1) * V, None, k * V, 0, B, k, V, None, None, None,
                                None, None, None, None, None, None)
    assert st == SSD_ERR_WORKSPACE
    assert lib.ssd_verify_noalloc(None, 3 * 1000, None, 2 * 1000, 0, 2, 2, 1000, None, None, None,
                                  None, None, None, None, None, None) == 1  # null pointers
    assert lib.ssd_verify_noalloc(None, 0, None, 0, 0, 0, 2, 1000, None, None, None, None, None,
                                  None, None, None, None) == 1              # B = 0
