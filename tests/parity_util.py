"""Comparison of the CUDA path with the oracle under the parity rules:
greedy tokens and accept lengths bit-exact; probabilities within 1e-5
absolute; sampled decisions identical unless the uniform lies within 1e-6 of
the decision boundary (p/q for an acceptance, a CDF boundary for a draw);
top-f and cache results bit-exact."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle

PROB_ATOL = 1e-5
BOUNDARY = 1e-6


def to_np(t):
    return t.detach().cpu().numpy() if hasattr(t, "detach") else np.asarray(t)


def oracle_rows(inp, bs):
    """Run the oracle on batch rows `bs` of a workload's inputs."""
    sel = lambda k: inp[k][bs].cpu()
    return oracle.verify_recover(sel("Z"), sel("D"), sel("x"), sel("T"), sel("u_acc"),
                                 sel("u_smp"))


def host_threads():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def _slices(B, per_task):
    return [(b0, min(B, b0 + per_task)) for b0 in range(0, B, per_task)]


def oracle_verify_host(cpu, per_task=8, threads=None):
    """The oracle's verify_recover on every batch row of host tensors `cpu`
    (Z, D, x, T, u_acc, u_smp), spread over the host cores: the oracle is a
    C library called through ctypes, which releases the GIL, so each thread
    runs the oracle on its own slice of rows."""
    B = cpu["Z"].shape[0]
    oracle.build()  # compile (if needed) once, before the threads load it

    def one(sl):
        b0, b1 = sl
        return oracle.verify_recover(cpu["Z"][b0:b1], cpu["D"][b0:b1], cpu["x"][b0:b1],
                                     cpu["T"][b0:b1], cpu["u_acc"][b0:b1], cpu["u_smp"][b0:b1])
    with ThreadPoolExecutor(threads or host_threads()) as ex:
        parts = list(ex.map(one, _slices(B, per_task)))
    return {key: np.concatenate([q[key] for q in parts]) for key in parts[0]}


def oracle_forks_host(D, f, mask, per_task=8, threads=None):
    """oracle.forked_topf over every batch row of host tensors, threaded."""
    B = D.shape[0]
    oracle.build()

    def one(sl):
        b0, b1 = sl
        return oracle.forked_topf(D[b0:b1], f, mask[b0:b1])
    with ThreadPoolExecutor(threads or host_threads()) as ex:
        parts = list(ex.map(one, _slices(B, per_task)))
    return {key: np.concatenate([q[key] for q in parts]) for key in parts[0]}


def draw_weights(Zrow, Drow, T, n, k):
    """The oracle's draw weights for a row (recomputed with the oracle's
    softmax): residual max(0, p - q) for n < k (p if all zero), p for n == k."""
    p = oracle.softmax_temp(Zrow[None], [T])["probs"][0]
    if n == k:
        return p
    q = oracle.softmax_temp(Drow[None], [T])["probs"][0]
    w = np.maximum(0.0, p - q)
    return w if w.sum() > 0 else p


class Report:
    def __init__(self):
        self.rows = 0
        self.greedy_rows = 0
        self.sampled_rows = 0
        self.sampled_mismatch = 0
        self.accept_flips = 0
        self.max_prob_err = 0.0
        self.failures = []

    def fail(self, msg):
        self.failures.append(msg)

    def summary(self):
        return ("rows %d greedy %d sampled %d sampled_mismatch %d accept_flips %d "
                "max|dp| %.2e failures %d" % (self.rows, self.greedy_rows, self.sampled_rows,
                                              self.sampled_mismatch, self.accept_flips,
                                              self.max_prob_err, len(self.failures)))


def compare_verify(inp, gpu, bs, ref, report, sampled=True):
    """Compare GPU outputs for batch rows `bs` with oracle outputs `ref`."""
    k = inp["x"].shape[1]
    g_acc = to_np(gpu["accept_len"])[bs]
    g_out = to_np(gpu["out_tok"])[bs]
    g_p = to_np(gpu["p_at_x"])[bs]
    g_q = to_np(gpu["q_at_x"])[bs]
    T = to_np(inp["T"])[bs]
    ua = to_np(inp["u_acc"])[bs]
    us = to_np(inp["u_smp"])[bs]
    x = to_np(inp["x"])[bs]
    for r in range(len(bs)):
        report.rows += 1
        b = int(bs[r])
        n_o, n_g = int(ref["accept_len"][r]), int(g_acc[r])
        greedy = not (T[r] > 0)
        if n_o < 0 or greedy:
            report.greedy_rows += 1
            if n_o != n_g or not np.array_equal(ref["out_tok"][r], g_out[r]):
                report.fail("b=%d greedy/sentinel mismatch: oracle n=%d %s gpu n=%d %s"
                            % (b, n_o, ref["out_tok"][r], n_g, g_out[r]))
            continue
        # probabilities at the draft tokens
        dp = max(np.max(np.abs(ref["p_at_x"][r] - g_p[r])), np.max(np.abs(ref["q_at_x"][r] - g_q[r])))
        report.max_prob_err = max(report.max_prob_err, float(dp))
        if not dp <= PROB_ATOL:
            report.fail("b=%d |dp| %.3e" % (b, dp))
        if n_o != n_g:
            i = min(n_o, n_g)  # first position whose decision differs
            ratio = ref["p_at_x"][r, i] / ref["q_at_x"][r, i] if ref["q_at_x"][r, i] > 0 else np.inf
            report.accept_flips += 1
            if not abs(float(ua[r, i]) - ratio) < BOUNDARY:
                report.fail("b=%d acceptance at %d differs: u=%.9f p/q=%.9f" % (b, i, ua[r, i], ratio))
            continue
        if not np.array_equal(ref["out_tok"][r, :n_o], g_out[r, :n_o]) or np.any(g_out[r, n_o + 1:] != -1):
            report.fail("b=%d prefix mismatch" % b)
            continue
        if not sampled:
            continue
        report.sampled_rows += 1
        jo, jg = int(ref["out_tok"][r, n_o]), int(g_out[r, n_o])
        if jo == jg:
            continue
        report.sampled_mismatch += 1
        if jg < 0:
            report.fail("b=%d no token drawn" % b)
            continue
        w = draw_weights(to_np(inp["Z"][b, n_o].float()), to_np(inp["D"][b, n_o].float())
                         if n_o < k else None, float(T[r]), n_o, k)
        C = np.cumsum(w) / np.sum(w)
        lo, hi = min(jo, jg), max(jo, jg)
        d = max(abs(float(us[r]) - C[lo]), abs(float(us[r]) - C[hi - 1]))
        if not d < BOUNDARY:
            report.fail("b=%d draw differs: oracle %d gpu %d, u=%.9f, C[%d]=%.9f C[%d]=%.9f"
                        % (b, jo, jg, us[r], lo, C[lo], hi - 1, C[hi - 1]))
    return report


def compare_forks(ref, g_tok, g_logit, label=""):
    g_tok, g_logit = to_np(g_tok), to_np(g_logit)
    assert np.array_equal(ref["fork_tok"], g_tok), label
    rl = ref["fork_logit"].astype(np.float32)
    same = (rl == g_logit) | (np.isnan(rl) & np.isnan(g_logit))
    assert np.all(same), label
