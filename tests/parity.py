"""Comparison of GPU verification results with the fp64 oracle.

Greedy and tree results must be bit-exact.  Sampling follows the parity
contract: accept counts and tokens match exactly, except where the oracle's
own decision margin is below MARGIN -- |u_i - p_i(x_i)/q_i(x_i)| for an accept
decision, or u's distance to the oracle's CDF interval of the token the GPU
picked for the final sample.  Such excused differences are counted; anything
else is a failure.
"""
from __future__ import annotations

import numpy as np

MARGIN = 1e-4
LOGPROB_RTOL = 1e-5


def compare_sample(gpu_tok, gpu_acc, ref, x, u, gpu_lp=None, check_lp=True):
    """Returns dict(failures=[...], excused=int, exact=int, rows=int, events=[...]);
    events lists each excused difference as (kind, sequence, position, margin)."""
    B, g1 = gpu_tok.shape
    g = g1 - 1
    fails, excused, exact = [], 0, 0
    events = []
    for b in range(B):
        ko, kg = int(ref["accepted"][b]), int(gpu_acc[b])
        if ko < 0 or kg < 0:
            if ko != kg or not (gpu_tok[b] == -1).all():
                fails.append((b, "bad-input handling", ko, kg))
            continue
        # the GPU's own output must be well formed
        if not (0 <= kg <= g) or not (gpu_tok[b, :kg] == x[b, :kg]).all() or \
                not (gpu_tok[b, kg + 1:] == -1).all() or gpu_tok[b, kg] < 0:
            fails.append((b, "malformed output", gpu_tok[b].tolist(), kg))
            continue
        if ko != kg:
            i = min(ko, kg)                           # first differing decision
            m = abs(float(u[b, i]) - float(ref["ratio"][b, i]))
            if m < MARGIN:
                excused += 1
                events.append(("accept", b, i, m))
            else:
                fails.append((b, "accept decision", i, float(u[b, i]), float(ref["ratio"][b, i])))
            continue
        to, tg = int(ref["tokens"][b, ko]), int(gpu_tok[b, kg])
        if to == tg:
            exact += 1
            continue
        cdf = ref["cdf"][b]
        lo = cdf[tg - 1] if tg > 0 else 0.0
        hi = cdf[tg]
        uu = float(u[b, g])
        dist = max(0.0, lo - uu, uu - hi)
        if dist < MARGIN:
            excused += 1
            events.append(("final", b, ko, dist))
        else:
            fails.append((b, "final token", to, tg, uu, lo, hi))
    if gpu_lp is not None and check_lp:
        lp_ref = ref["logprob"]
        ok = ref["accepted"] >= 0
        for b in np.nonzero(ok)[0]:
            pg = np.exp(gpu_lp[b].astype(np.float64))
            pr = np.exp(lp_ref[b])
            tiny = (pg < 1e-30) & (pr < 1e-30)
            rel = np.abs(pg - pr) / np.maximum(pr, 1e-300)
            bad = (~tiny) & (rel > LOGPROB_RTOL)
            if bad.any():
                fails.append((int(b), "logprob", float(rel[bad].max())))
    return {"failures": fails, "excused": excused, "exact": exact, "rows": B * g1,
            "events": events}


def compare_exact(name, got, want):
    got = np.asarray(got)
    want = np.asarray(want)
    if got.shape != want.shape:
        return [(name, "shape", got.shape, want.shape)]
    bad = np.argwhere(got != want)
    if bad.size:
        i = tuple(bad[0])
        return [(name, "first mismatch at", i, int(got[i]), int(want[i]), int(bad.shape[0]))]
    return []
