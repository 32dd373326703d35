"""Index-build parity: the CUDA segmented spherical k-means against the
float64 oracle on the same seeded keys.

Per round (wi_kmeans_step) both sides start from the same bf16 centroids;
for the final index both run their last assignment from the same centroids
(wi_build_index seeded with the oracle's centroids, one round).  A full
default build is checked by invariants that hold at any size."""
import numpy as np
import pytest
import torch

import kvsynth
import oracle
from helpers import (assignment_from_index, bf16_ulp, compare_assignment, gen, near_tie, params_of, small)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def wi():
    import clustered_sparse_kv_gb300 as m
    return m


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV)


def from16(t):
    return oracle.bf16_from_bits(t.cpu().numpy().view(np.uint16))


def seg_centroids(idx, t):
    """Centroids of round t of every unit and segment: [units][nseg][Cs][d] (float64)."""
    return np.stack([np.stack([h[t] for h in i["histories"]]) for i in idx])


def check_kmeans_step(wi, w, K, k, idx, t):
    p = params_of(w)
    c_in = seg_centroids(idx, t)
    cbits = oracle.bf16_to_bits(c_in)
    assign = torch.empty((w.units, w.n_ctx), dtype=torch.int32, device=DEV)
    new_c = torch.empty(cbits.shape, dtype=torch.int16, device=DEV)
    cfg = wi.config_from_workload(w)
    wi.wi_kmeans_step(cfg, dev16(k), dev16(cbits), assign, new_c)
    torch.cuda.synchronize()
    a_gpu = assign.cpu().numpy().astype(np.int64)
    c_gpu = from16(new_c).reshape(c_in.shape)
    steady = oracle.steady_positions(w.n_ctx, p)
    disagree = 0
    for u in range(w.units):
        a_ref = np.full(w.n_ctx, -1, np.int64)
        for s in range(w.n_segments):
            seg = np.arange(s * w.seg_len, (s + 1) * w.seg_len)
            loc = np.setdiff1d(seg, steady) - s * w.seg_len
            a_ref[s * w.seg_len + loc] = s * w.clusters_per_seg + oracle.assign(K[u][s * w.seg_len + loc], c_in[u, s])
        disagree += compare_assignment(a_gpu[u], a_ref, K[u], lambda s: c_in[u, s], w.seg_len, w.clusters_per_seg)
        # the update from the oracle's assignment, cluster by cluster where both sides hold the same members
        for s in range(w.n_segments):
            seg = np.arange(s * w.seg_len, (s + 1) * w.seg_len)
            loc = np.setdiff1d(seg, steady)
            a_loc = a_ref[loc] - s * w.clusters_per_seg
            c_ref = oracle.update(K[u][loc], a_loc, c_in[u, s])
            bad = set(np.unique(a_gpu[u][loc][a_gpu[u][loc] != a_ref[loc]] - s * w.clusters_per_seg))
            bad |= set(np.unique(a_loc[a_gpu[u][loc] != a_ref[loc]]))
            ok = np.array([j not in bad for j in range(w.clusters_per_seg)])
            diff = np.abs(c_gpu[u, s][ok] - c_ref[ok])
            assert np.all(diff <= bf16_ulp(c_ref[ok]) * 1.0000001), diff.max()
    total = w.units * (w.n_ctx - w.n_sink - w.local_window)
    assert disagree <= 1e-3 * total
    return disagree


@pytest.mark.parametrize("t", [0, 2])
def test_kmeans_step_parity_small(wi, t):
    w = small(batch=2, n_q_heads=4, n_kv_heads=2, n_ctx=4096, seg_len=1024, clusters_per_seg=64, iters=3,
              budget_k=4, seed=71)
    k, v, q, K, V, Q = gen(w)
    idx = oracle.build_index(K, V, params_of(w))
    check_kmeans_step(wi, w, K, k, idx, t)


def test_kmeans_step_parity_tiny_workload(wi):
    w = kvsynth.get_workload("tiny-8k").with_(iters=4)
    k, v, q, K, V, Q = gen(w)
    idx = oracle.build_index(K, V, params_of(w))
    for t in range(4):
        check_kmeans_step(wi, w, K, k, idx, t)


def check_index(w, K, V, k_perm, v_perm, exp, ref, c_last):
    """GPU-exported index `exp` against the oracle index `ref` of one round from the same centroids."""
    p = params_of(w)
    U = w.units
    n_idx = w.n_ctx - w.n_sink - w.local_window
    counts = exp["counts"].cpu().numpy()
    perm = exp["perm"].cpu().numpy()
    offs = exp["offsets"].cpu().numpy()
    mu = from16(exp["mu"]).reshape(U, w.clusters, 128)
    vs = exp["valsum"].cpu().numpy().astype(np.float64)
    kp = oracle.bf16_from_bits(k_perm).reshape(U, w.n_ctx, 128)
    vp = oracle.bf16_from_bits(v_perm).reshape(U, w.n_ctx, 128)
    steady = oracle.steady_positions(w.n_ctx, p)
    for u in range(U):
        # invariants: conservation, bijection, segments, offsets, position order
        assert counts[u].sum() == n_idx
        np.testing.assert_array_equal(offs[u], w.n_sink + np.concatenate([[0], np.cumsum(counts[u])]))
        np.testing.assert_array_equal(np.sort(perm[u]), oracle.indexed_positions(w.n_ctx, p))
        a_gpu = assignment_from_index(counts[u], perm[u], w.n_ctx, w.n_sink)
        assert np.all(a_gpu[perm[u]] // w.clusters_per_seg == perm[u] // w.seg_len)
        owner = np.repeat(np.arange(w.clusters), counts[u])
        assert np.all((np.diff(perm[u]) > 0) | (np.diff(owner) != 0))
        # the cache rows were permuted in place: slot r holds the row of position perm[r]
        np.testing.assert_array_equal(kp[u][w.n_sink:w.n_ctx - w.local_window], K[u][perm[u]])
        np.testing.assert_array_equal(vp[u][w.n_sink:w.n_ctx - w.local_window], V[u][perm[u]])
        np.testing.assert_array_equal(kp[u][steady], K[u][steady])
        # parity with the oracle's assignment from the same centroids
        dis = compare_assignment(a_gpu, ref[u]["assignment"], K[u], lambda s: c_last[u, s], w.seg_len,
                                 w.clusters_per_seg)
        assert dis <= 1e-3 * n_idx
        same = np.ones(w.clusters, bool)
        moved = a_gpu != ref[u]["assignment"]
        same[np.unique(a_gpu[moved])] = False
        same[np.unique(ref[u]["assignment"][moved])] = False
        if dis == 0:
            np.testing.assert_array_equal(counts[u], ref[u]["counts"])
            np.testing.assert_array_equal(perm[u], ref[u]["perm"])
        np.testing.assert_array_equal(counts[u][same], ref[u]["counts"][same])
        ne = same & (counts[u] > 0)
        assert np.all(np.abs(mu[u][ne] - ref[u]["mu"][ne]) <= bf16_ulp(ref[u]["mu"][ne]) * 1.0000001)
        num = np.linalg.norm(vs[u][ne] - ref[u]["valsum"][ne])
        assert num <= 1e-5 * np.linalg.norm(ref[u]["valsum"][ne])


def seeded_build_case(wi, w, zero_rows=None):
    """Oracle clusters with T rounds; both sides then run the final round from the oracle's last centroids.
    zero_rows: (unit, position) pairs whose key is set to zero on both sides first."""
    k, v, q, K, V, Q = gen(w)
    if zero_rows:
        shape = k.shape
        k = k.copy().reshape(w.units, w.n_ctx, 128)
        for u, pos in zero_rows:
            k[u, pos] = 0
        k = k.reshape(shape)
        K = oracle.bf16_from_bits(k).reshape(w.units, w.n_ctx, 128)
    p = params_of(w)
    full = oracle.build_index(K, V, p)
    c_last = seg_centroids(full, w.iters - 1)
    ref = [oracle.build_unit_index(K[u], V[u], p, c_init=list(c_last[u]), iters=1) for u in range(w.units)]
    cfg = wi.config_from_workload(w, iters=1)
    kt, vt = dev16(k), dev16(v)
    ix = wi.WaveIndex.build(cfg, kt, vt, init_centroids=dev16(oracle.bf16_to_bits(c_last)))
    exp = ix.export()
    torch.cuda.synchronize()
    ix.check()
    k_perm = kt.cpu().numpy().view(np.uint16)
    v_perm = vt.cpu().numpy().view(np.uint16)
    check_index(w, K, V, k_perm, v_perm, exp, ref, c_last)
    ix.free()


def test_seeded_build_parity_small(wi):
    w = small(batch=2, n_q_heads=4, n_kv_heads=2, n_ctx=4096, seg_len=1024, clusters_per_seg=64, iters=3,
              budget_k=4, seed=81)
    seeded_build_case(wi, w)


def test_seeded_build_parity_tiny_workload(wi):
    seeded_build_case(wi, kvsynth.get_workload("tiny-8k"))


def test_seeded_build_parity_ragged_steady(wi):
    w = small(n_ctx=2048, seg_len=512, clusters_per_seg=32, iters=2, n_q_heads=1, n_sink=600, local_window=700,
              budget_k=3, seed=82)
    seeded_build_case(wi, w)


@pytest.mark.parametrize("seg,cs,nseg", [(128, 16, 16), (256, 32, 16), (1024, 128, 16), (768, 384, 4),
                                         (3968, 496, 2), (16384, 512, 2)])
def test_seeded_build_parity_small_geometries(wi, seg, cs, nseg):
    """The smallest segment and cluster counts the configuration admits (128-token segments, 16
    clusters: 8 tokens per cluster), a tensor-core one, large cluster counts outside the
    tensor-core set (384, 496: the SIMT assignment), and the longest segment admitted (16384 tokens),
    several segments each."""
    w = small(batch=1, layers=2, n_q_heads=4, n_kv_heads=2, n_ctx=nseg * seg, seg_len=seg, clusters_per_seg=cs,
              iters=2, budget_k=4, seed=84 + cs)
    seeded_build_case(wi, w)


def test_seeded_build_parity_zero_keys(wi):
    """Keys of norm 0 (padding-like rows): seed positions, clustered positions and a sink.  They add
    nothing to a centroid's sum, a zero seed gives the zero centroid, every score against it is 0."""
    w = small(batch=1, n_q_heads=4, n_kv_heads=2, n_ctx=4096, seg_len=1024, clusters_per_seg=64, iters=3,
              budget_k=4, seed=88)
    rng = np.random.default_rng(88)
    rows = [(u, p) for u in range(w.units) for p in (0, 16, 1024 + 32, 2048 + 5 * 16)]       # sink and seeds
    rows += [(u, int(p)) for u in range(w.units) for p in rng.choice(np.arange(8, 4000), 60, replace=False)]
    seeded_build_case(wi, w, zero_rows=rows)


def test_default_build_invariants_and_quality(wi):
    """Full default build (10 rounds from the default seeds) on the tiny workload:
    invariants of the index, and a clustering objective within 1% of the oracle's."""
    w = kvsynth.get_workload("tiny-8k")
    k, v, q, K, V, Q = gen(w)
    p = params_of(w)
    ref = oracle.build_index(K, V, p)
    cfg = wi.config_from_workload(w)
    kt, vt = dev16(k), dev16(v)
    ix = wi.WaveIndex.build(cfg, kt, vt)
    exp = ix.export()
    torch.cuda.synchronize()
    ix.check()
    counts = exp["counts"].cpu().numpy()[0]
    perm = exp["perm"].cpu().numpy()[0]
    n_idx = w.n_ctx - 68
    assert counts.sum() == n_idx
    np.testing.assert_array_equal(np.sort(perm), oracle.indexed_positions(w.n_ctx, p))
    a_gpu = assignment_from_index(counts, perm, w.n_ctx, w.n_sink)

    def objective(a):
        I = oracle.indexed_positions(w.n_ctx, p)
        kh = K[0][I] / np.linalg.norm(K[0][I], axis=1, keepdims=True)
        tot = 0.0
        for j in np.unique(a[I]):
            m = kh[a[I] == j]
            tot += np.linalg.norm(m.sum(0))
        return tot

    og, orf = objective(a_gpu), objective(ref[0]["assignment"])
    assert abs(og - orf) <= 0.01 * orf, (og, orf)
    ix.free()


# ------------------------------------------------- B1 seeding, tie rule ----

@pytest.mark.parametrize("shape", [dict(n_ctx=4096, seg_len=1024, clusters_per_seg=64),
                                   dict(n_ctx=16384, seg_len=8192, clusters_per_seg=512),
                                   dict(n_ctx=1536, seg_len=768, clusters_per_seg=48)])
def test_default_seeds_match_oracle_init(wi, shape):
    """k_init_centroids (the centroids of the first round when none are given) element by
    element against oracle.init_centroids, within one bf16 step (fp32 vs float64 norm)."""
    w = small(batch=2, layers=2, n_q_heads=4, n_kv_heads=2, iters=1, budget_k=4, seed=83, **shape)
    default_seeds_case(wi, w)


def test_default_seeds_zero_keys(wi):
    """Keys of norm 0 at seed positions give zero centroids, exactly; a zero key ties every centroid
    at score 0 and goes to the segment's first; the one-round build still follows the oracle."""
    w = small(batch=1, n_q_heads=4, n_kv_heads=2, n_ctx=4096, seg_len=1024, clusters_per_seg=64, iters=1,
              budget_k=4, seed=86)
    stride = w.seg_len // w.clusters_per_seg
    rng = np.random.default_rng(86)
    rows = [(u, s * w.seg_len + j * stride) for u in range(w.units) for s in range(w.n_segments)
            for j in (0, 3, 17, w.clusters_per_seg - 1)]
    rows += [(u, int(p)) for u in range(w.units) for p in rng.choice(w.n_ctx, 80, replace=False)]
    c = default_seeds_case(wi, w, zero_rows=rows)
    for u, pos in rows:
        s, j = divmod(pos, w.seg_len)
        if j % stride == 0:
            assert not c[u, s, j // stride].any(), (u, pos)


def default_seeds_case(wi, w, zero_rows=()):
    k, v, q, K, V, Q = gen(w)
    if zero_rows:
        shape = k.shape
        k = k.copy().reshape(w.units, w.n_ctx, 128)
        for u, pos in zero_rows:
            k[u, pos] = 0
        k = k.reshape(shape)
        K = oracle.bf16_from_bits(k).reshape(w.units, w.n_ctx, 128)
    p = params_of(w)
    cfg = wi.config_from_workload(w)
    c = torch.empty((w.units, w.n_segments, w.clusters_per_seg, 128), dtype=torch.int16, device=DEV)
    wi.wi_init_centroids(cfg, dev16(k), c)
    torch.cuda.synchronize()
    got = from16(c).reshape(w.units, w.n_segments, w.clusters_per_seg, 128)
    ref = np.stack([np.stack([oracle.init_centroids(K[u][s * w.seg_len:(s + 1) * w.seg_len], p)
                              for s in range(w.n_segments)]) for u in range(w.units)])
    diff = np.abs(got - ref)
    assert np.all(diff <= bf16_ulp(ref) * 1.0000001), diff.max()
    assert np.mean(diff == 0) > 0.99   # rounding differences are rare
    # and the default one-round build assigns by exactly those seeds
    ix = wi.WaveIndex.build(cfg, dev16(k), dev16(v))
    exp = ix.export()
    torch.cuda.synchronize()
    ix.check()
    for u in range(w.units):
        a_gpu = assignment_from_index(exp["counts"][u].cpu().numpy(), exp["perm"][u].cpu().numpy(), w.n_ctx,
                                      w.n_sink)
        a_ref = oracle.build_unit_index(K[u], V[u], p, iters=1)["assignment"]
        dis = compare_assignment(a_gpu, a_ref, K[u], lambda s: ref[u, s], w.seg_len, w.clusters_per_seg)
        assert dis <= 1e-3 * (w.n_ctx - w.n_sink - w.local_window)
    ix.free()
    return got


@pytest.mark.parametrize("cs,base,seg", [(512, 128, 1024), (256, 64, 1024), (64, 16, 1024), (48, 16, 768)])
def test_assignment_ties_go_to_lowest_id_exactly(wi, cs, base, seg):
    """Centroid j repeats centroid j mod `base`: every score has exact ties, across the
    accumulator halves and column groups of the tensor-core epilogue (Cs = 512, 256) and in
    the SIMT path (Cs = 48).  Every token must take the lowest id of its best centroid --
    no near-tie excuse -- and equal the oracle (first maximum) wherever the best distinct
    centroid leads by a relative 1e-5."""
    w = small(batch=1, n_q_heads=1, n_kv_heads=1, n_ctx=2 * seg, seg_len=seg, clusters_per_seg=cs, iters=1,
              budget_k=2, seed=84)
    k, v, q, K, V, Q = gen(w)
    p = params_of(w)
    rng = np.random.default_rng(85)
    distinct = oracle.bf16_round(rng.standard_normal((w.units, w.n_segments, base, 128)) / np.sqrt(128))
    c = distinct[:, :, np.arange(cs) % base]
    cfg = wi.config_from_workload(w)
    assign = torch.empty((w.units, w.n_ctx), dtype=torch.int32, device=DEV)
    new_c = torch.empty(c.shape, dtype=torch.int16, device=DEV)
    wi.wi_kmeans_step(cfg, dev16(k), dev16(oracle.bf16_to_bits(c)), assign, new_c)
    torch.cuda.synchronize()
    a_gpu = assign.cpu().numpy().astype(np.int64)[0]
    steady = oracle.steady_positions(w.n_ctx, p)
    I = oracle.indexed_positions(w.n_ctx, p)
    assert np.all(a_gpu[steady] == -1)
    loc = a_gpu[I] - (I // w.seg_len) * cs
    assert np.all((loc >= 0) & (loc < base)), "a tie went to a higher duplicate id"
    for s in range(w.n_segments):
        pos = I[I // w.seg_len == s]
        a_ref = oracle.assign(K[0][pos], c[0, s])
        assert np.all(a_ref < base)
        gap = near_tie(K[0][pos], distinct[0, s])
        firm = gap >= 1e-5
        np.testing.assert_array_equal((a_gpu[pos] - s * cs)[firm], a_ref[firm])
        assert firm.mean() > 0.99
