"""Shared test helpers: seeded inputs, oracle runs, GPU <-> oracle comparisons."""
from __future__ import annotations

import math

import numpy as np

import kvsynth
import oracle

D = 128
ASSIGN_TIE_REL = 1e-5     # assignment may differ where the oracle's top-2 relative gap is below this
TOPK_TIE_REL = 1e-5       # top-k may differ for clusters within this of the k-th score
OUT_REL_L2 = 2e-3         # attention output relative L2 per (unit, head)


def params_of(w, iters=None) -> oracle.IndexParams:
    return oracle.IndexParams(seg_len=w.seg_len, clusters_per_seg=w.clusters_per_seg,
                              iters=w.iters if iters is None else iters, n_sink=w.n_sink,
                              local_window=w.local_window, budget_frac=w.budget_frac, budget_k=w.budget_k)


def small(name="tiny-8k", **kw):
    return kvsynth.get_workload(name).with_(**kw)


def gen(w, step=0):
    """bf16 bit arrays (k, v, q) and their float64 values (K, V [units][n][d], Q [units][g][d])."""
    k, v = kvsynth.kv_cache(w)
    q = kvsynth.queries(w, step=step)
    K = oracle.bf16_from_bits(k).reshape(w.units, w.n_ctx, D)
    V = oracle.bf16_from_bits(v).reshape(w.units, w.n_ctx, D)
    Q = oracle.bf16_from_bits(q).reshape(w.units, w.group, D)
    return k, v, q, K, V, Q


def index_arrays(idx):
    """Oracle index (list of per-unit dicts) -> arrays for wi_index_import."""
    counts = np.ascontiguousarray(np.stack([i["counts"] for i in idx]).astype(np.int32))
    perm = np.ascontiguousarray(np.stack([i["perm"] for i in idx]).astype(np.int32))
    mu = np.ascontiguousarray(np.stack([oracle.bf16_to_bits(i["mu"]) for i in idx]).view(np.int16))
    vs = np.ascontiguousarray(np.stack([i["valsum"] for i in idx]).astype(np.float32))
    return counts, perm, mu, vs


def rel_l2(got, ref):
    return np.linalg.norm(got - ref, axis=-1) / np.maximum(np.linalg.norm(ref, axis=-1), 1e-300)


def check_topk(gpu_ids, gpu_cnt, scores, nonempty, k):
    """GPU selection equals the oracle's except for clusters within TOPK_TIE_REL of the k-th score."""
    ids = np.nonzero(nonempty)[0]
    kk = min(k, ids.size)
    assert gpu_cnt == kk
    got = np.asarray(gpu_ids[:kk])
    assert np.all(np.diff(got) > 0), "ids must be ascending and distinct"
    assert np.all(gpu_ids[kk:] == -1)
    assert np.all(nonempty[got]), "an empty cluster was selected"
    ref = oracle.select_topk(scores, nonempty, k)
    sym = np.setxor1d(got, ref)
    if sym.size:
        s_k = np.sort(scores[ids])[::-1][kk - 1]
        band = TOPK_TIE_REL * max(abs(s_k), 1e-30)
        assert np.all(np.abs(scores[sym] - s_k) <= band), (sym, scores[sym], s_k)
    return sym.size


def assignment_from_index(counts, perm, n, n_sink):
    """Per-position cluster id from (counts, perm) of one unit (-1 for steady)."""
    a = np.full(n, -1, np.int64)
    owner = np.repeat(np.arange(counts.size), counts)
    a[perm] = owner
    return a


def near_tie(K_rows, c_hat):
    """Relative gap (s1 - s2)/|s1| of the two best centroid scores per row (float64)."""
    s = K_rows @ c_hat.T
    top2 = -np.sort(-s, axis=1)[:, :2]
    return (top2[:, 0] - top2[:, 1]) / np.maximum(np.abs(top2[:, 0]), 1e-300)


def compare_assignment(a_gpu, a_ref, K, centroids_of_segment, S, Cs):
    """Assignments agree except at near ties; returns the number of disagreements."""
    diff = np.nonzero(a_gpu != a_ref)[0]
    for p in diff:
        assert a_ref[p] >= 0 and a_gpu[p] >= 0, f"steady/clustered mismatch at {p}"
        s = p // S
        assert a_gpu[p] // Cs == s, "assigned outside its segment"
        gap = near_tie(K[p][None], centroids_of_segment(s))[0]
        assert gap < ASSIGN_TIE_REL, f"position {p}: gpu {a_gpu[p]} oracle {a_ref[p]} gap {gap:.2e}"
    return diff.size


def bf16_ulp(x):
    """Spacing of bf16 values at |x| (x float64)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 7), 2.0 ** -133)
