"""Sampled full-size parity: the oracle's layer for a sample of tokens, computed expert by expert.

Test infrastructure (host side, no GPU).  A full-size layer (decode, prefill, skewed) is too large for
the oracle to compute whole, but every routed pair's values depend only on its own token: quantisation is
per token, the GEMMs are row-wise and the permutation only moves rows.  So for a sample of tokens the
oracle computes, for each expert, exactly the rows the whole layer would hold for those tokens' pairs:

* the w13 stage on the device's quantised rows (bit-identical to the oracle's own, which the caller
  asserts first), compared with the device's Y13 rows at the stage tolerance;
* the SiLU-and-Mul requantisation of the device's Y13 rows, compared code by code with the device's;
* the w2 stage on the device's Hq rows, compared with the device's Y2 rows at the stage tolerance;
* the oracle's own chain for the pair (its Y13 -> its Hq -> its Y2), whose routing-weighted combine per
  token is the end-to-end reference.

Experts are independent, so a spawn-started process pool spreads them over the host's cores (a pool
started by fork after CUDA initialisation can hang; spawn starts clean interpreters).
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

import oracle
from helpers import moe_experts


def pick_tokens(T, n, seed, ids, E, extra=()):
    """A seeded sample of n distinct tokens (all of them if n >= T), always holding tokens 0 and T - 1 and
    the tokens listed in `extra`."""
    if n >= T:
        return np.arange(T)
    must = sorted({0, T - 1, *[int(t) for t in extra]})
    rng = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(T), must)
    take = rng.choice(rest, size=max(0, n - len(must)), replace=False)
    return np.sort(np.concatenate([np.asarray(must, np.int64), take.astype(np.int64)]))


def skew_extremes(ids, E, per_expert=4, n_cold=8):
    """Tokens routed to the most popular expert (up to per_expert of them) and to the least popular experts
    that hold any pair (all tokens of up to n_cold such experts): the hot and near-empty ends of a skewed
    routing."""
    flat = np.asarray(ids).reshape(-1)
    k = np.asarray(ids).shape[1]
    counts = np.bincount(flat, minlength=E)
    hot = int(np.argmax(counts))
    toks = list(np.nonzero(flat == hot)[0][:per_expert] // k)
    used = np.nonzero(counts > 0)[0]
    cold = used[np.argsort(counts[used], kind="stable")][:n_cold]
    for e in cold:
        toks.extend(np.nonzero(flat == e)[0] // k)
    return sorted({int(t) for t in toks}), hot, [int(e) for e in cold]


def _expert_job(job):
    """Oracle rows of one expert's sampled pairs (runs in a pool worker)."""
    seed, cfg, e, xq, xs, y13_dev, hq_dev, hs_dev, y2_dev = job
    w13, w2 = moe_experts(seed, cfg)
    W13, S13 = w13.w(e), w13.s(e)
    y13_ref = oracle.round_bf16(oracle.w4a8_gemm(xq, xs, W13, S13))
    del W13
    rhq, rhs = oracle.silu_mul_requant(y13_dev)
    hq_o, hs_o = oracle.silu_mul_requant(y13_ref)
    m = xq.shape[0]
    W2, S2 = w2.w(e), w2.s(e)
    both = oracle.round_bf16(oracle.w4a8_gemm(np.concatenate([hq_dev, hq_o]), np.concatenate([hs_dev, hs_o]),
                                              W2, S2))
    y2_ref, y2_o = both[:m], both[m:]
    deq_dev, deq_ref = oracle.dequant(hq_dev, hs_dev), oracle.dequant(rhq, rhs)
    return dict(
        e=e,
        y13=(float(np.sum((y13_dev - y13_ref) ** 2)), float(np.sum(y13_ref ** 2))),
        y2=(float(np.sum((y2_dev - y2_ref) ** 2)), float(np.sum(y2_ref ** 2))),
        hq_mismatch=int(np.count_nonzero(hq_dev != rhq)), hq_total=int(hq_dev.size),
        hq_deq=(float(np.sum((deq_dev - deq_ref) ** 2)), float(np.sum(deq_ref ** 2))),
        y2_chain=y2_o.astype(np.float32),  # bf16 values: exact in float32
    )


def pool_size():
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(16, n))


def sampled_layer_check(seed, cfg, sample, logits, rows):
    """Stage and end-to-end comparison for the sampled tokens.

    rows: the device's rows of the sampled pairs, as a dict of arrays indexed by a flat pair position
    p = s * k + j (s the sample index, j the slot): xq uint8 [n, H], xs fp32 [n, H/128], y13 float [n, 2I],
    hq uint8 [n, I], hs fp32 [n, I/128], y2 float [n, H].  The routed expert of each pair comes from the
    oracle's routing of the sampled tokens (the caller checks the device's ids against it).
    Returns (stats, out_ref): relative Frobenius errors of the stages, the SiLU code mismatch fraction, and
    the oracle's layer output rows for the sample (float64 bf16 values, [n_sample, H]).
    """
    k = cfg["k"]
    ids, w = oracle.route_topk(logits[sample], k)
    flat = ids.reshape(-1)
    jobs = []
    for e in np.unique(flat):
        pos = np.nonzero(flat == e)[0]
        jobs.append((seed, cfg, int(e), rows["xq"][pos], rows["xs"][pos], rows["y13"][pos], rows["hq"][pos],
                     rows["hs"][pos], rows["y2"][pos]))
    ctx = mp.get_context("spawn")
    with ctx.Pool(pool_size()) as pool:
        res = pool.map(_expert_job, jobs, chunksize=1)
    H = rows["y2"].shape[1]
    y2_chain = np.zeros((flat.size, H), np.float64)
    acc = {n: [0.0, 0.0] for n in ("y13", "y2", "hq_deq")}
    mism = tot = 0
    for r in res:
        pos = np.nonzero(flat == r["e"])[0]
        y2_chain[pos] = r["y2_chain"]
        for n in acc:
            acc[n][0] += r[n][0]
            acc[n][1] += r[n][1]
        mism += r["hq_mismatch"]
        tot += r["hq_total"]
    out_ref = oracle.round_bf16(oracle.unpermute_combine(y2_chain, np.arange(flat.size), w, len(sample), k))
    stats = {n: float(np.sqrt(a / b)) if b > 0 else 0.0 for n, (a, b) in acc.items()}
    stats["hq_mismatch"] = mism / max(tot, 1)
    return stats, out_ref
