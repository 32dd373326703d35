"""Decode-time index maintenance on the GPU against the oracle.

Appended tokens join the local window; once an append leaves the window with
local_window + seg_len rows, its oldest seg_len rows become one more segment
(oracle.grow_unit_index).  The GPU grows the index inside the appending step.
Checked at steps around each growth:
  * the grown segment's clustering against the oracle's from the same seeds
    (one round: assignment identical except near ties, counts / mean keys /
    value sums per agreed cluster);
  * the decode output against oracle.decode_unit given the GPU's own index
    (exported, growth included), step after step;
  * the exported index's invariants (every grown slot once, inside its segment).
"""
import numpy as np
import pytest
import torch

import kvsynth
import oracle
from helpers import (OUT_REL_L2, bf16_ulp, check_topk, compare_assignment, gen, index_arrays, params_of, rel_l2,
                     small)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def wi():
    import clustered_sparse_kv_gb300 as m
    return m


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV)


def index_from_export(exp, u, w, appended):
    """The GPU index of unit u as an oracle index dict (growth included)."""
    S = w.seg_len
    grown = appended // S
    C = w.clusters + grown * w.clusters_per_seg     # clusters held so far (the rest is room, empty)
    assert np.all(exp["counts"][u][C:] == 0)
    counts = exp["counts"][u][:C].astype(np.int64)
    filled = w.n_ctx - w.n_sink - w.local_window + grown * S
    perm = exp["perm"][u][:filled]
    assert counts.sum() == filled
    a = np.full(w.n_ctx + appended, -1, np.int64)
    a[perm] = np.repeat(np.arange(C), counts)
    return {"counts": counts, "assignment": a, "grown": grown,
            "mu": oracle.bf16_from_bits(exp["mu"][u].view(np.uint16)).reshape(-1, 128)[:C],
            "valsum": exp["valsum"][u][:C].astype(np.float64)}


def run_growth(wi, w, T, checks, imported, seg_parity):
    k, v, q, K, V, Q = gen(w)
    p = params_of(w)
    n, S, Cs = w.n_ctx, w.seg_len, w.clusters_per_seg
    cfg = wi.config_from_workload(w, max_append=T)
    kt, vt = dev16(k), dev16(v)
    idx0 = oracle.build_index(K, V, p) if (imported or seg_parity) else None
    if imported:
        ix = wi.WaveIndex.adopt(cfg, kt, vt, *index_arrays(idx0))
    else:
        ix = wi.WaveIndex.build(cfg, kt, vt)
    Gmax = T // S
    Cb = w.clusters
    assert ix.clusters == Cb + Gmax * Cs
    ka, va = kvsynth.kv_cache(w, p0=n, p1=n + T)
    KA = oracle.bf16_from_bits(ka).reshape(w.units, T, 128)
    VA = oracle.bf16_from_bits(va).reshape(w.units, T, 128)
    checked = 0
    for t in range(T):
        qb = kvsynth.queries(w, step=t)
        check = t in checks
        if check:   # the index this step attends with (growth from earlier appends included)
            exp = {name: a.cpu().numpy() for name, a in ix.export().items()}
        out = ix.decode(dev16(qb), dev16(ka[:, :, :, t]), dev16(va[:, :, :, t]))
        if not check:
            continue
        ids, cnt = ix.selection()
        torch.cuda.synchronize()
        ix.check()
        got = out.cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64)
        Qt = oracle.bf16_from_bits(qb).reshape(w.units, w.group, 128)
        grown = t // S
        for u in range(w.units):
            gi = index_from_export(exp, u, w, t)
            K_all = np.concatenate([K[u], KA[u, :t]])
            V_all = np.concatenate([V[u], VA[u, :t]])
            w0 = n - w.local_window
            for g in range(grown):   # every grown slot once, inside its segment
                pos = np.sort(exp["perm"][u][w.n_ctx - w.n_sink - w.local_window + g * S:][:S])
                np.testing.assert_array_equal(pos, w0 + g * S + np.arange(S))
            if seg_parity and grown:
                ref = oracle.grow_unit_index(idx0[u], K_all, V_all, n, p)
                for g in range(grown):
                    pos = w0 + g * S + np.arange(S)
                    c_init = oracle.init_centroids(K_all[pos], p)
                    a_ref = ref["assignment"].copy()
                    a_gpu = gi["assignment"].copy()
                    dis = compare_assignment(a_gpu[pos] - Cb - g * Cs + 0, a_ref[pos] - Cb - g * Cs + 0,
                                             K_all[pos], lambda s: c_init, S, Cs)
                    assert dis <= max(1, 1e-3 * S)
                    if dis == 0:
                        sl = slice(Cb + g * Cs, Cb + (g + 1) * Cs)
                        np.testing.assert_array_equal(gi["counts"][sl], ref["counts"][sl])
                        ne = ref["counts"][sl] > 0
                        mr, mg = ref["mu"][sl][ne], gi["mu"][sl][ne]
                        assert np.all(np.abs(mg - mr) <= bf16_ulp(mr) * 1.0000001)
                        vr, vg = ref["valsum"][sl][ne], gi["valsum"][sl][ne]
                        assert np.linalg.norm(vg - vr) <= 1e-5 * np.linalg.norm(vr)
            ref_o, info = oracle.decode_unit(Qt[u], K[u], V[u], gi, p, KA[u, :t], VA[u, :t], details=True)
            err = rel_l2(got[u], ref_o)
            assert err.max() <= OUT_REL_L2, (t, u, err.max())
            kk = oracle.budget_k(gi["counts"].size, p)
            ne = gi["counts"] > 0
            for h in range(w.group):
                check_topk(ids.cpu().numpy()[u, h], cnt.cpu().numpy()[u, h], info[h]["scores"], ne, kk)
        checked += 1
    assert checked == len(checks)
    ix.free()


def test_growth_imported_index_one_round(wi):
    """One k-means round: the grown segments' clustering is compared with the oracle's from the
    same default seeds, and every checked step's output with the oracle given the GPU's index."""
    w = small(batch=1, n_q_heads=8, n_kv_heads=2, n_ctx=2048, seg_len=256, clusters_per_seg=16, iters=1,
              n_sink=4, local_window=8, budget_k=0, budget_frac=0.05, seed=95)
    run_growth(wi, w, T=600, checks={0, 255, 256, 257, 400, 511, 512, 599}, imported=True, seg_parity=True)


@pytest.mark.parametrize("n_sink,window", [(4, 0), (2, 300)])
def test_growth_built_index_three_rounds(wi, n_sink, window):
    """A GPU-built index with three k-means rounds; no local window at all, and a window wider
    than a segment (the first grown segment lies wholly in the build's window)."""
    w = small(batch=2, n_q_heads=4, n_kv_heads=1, n_ctx=4096, seg_len=256, clusters_per_seg=32, iters=3,
              n_sink=n_sink, local_window=window, budget_k=0, budget_frac=0.03, seed=96)
    run_growth(wi, w, T=530, checks={255, 256, 300, 512, 529}, imported=False, seg_parity=False)
