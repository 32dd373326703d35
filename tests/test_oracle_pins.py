"""Pins of the CPU oracle to facts outside itself (CPU only).

Each test ties an oracle function to mathematics or to an independent
routine: textbook softmax attention, closed forms of the estimation zone,
Jensen's inequality, exhaustive search on tiny inputs, torch's bf16 cast,
conservation laws.  A plausible slip in the oracle (dropped n_j factor, wrong
centroid in the estimate, off-by-one zone, reversed tie-break, transposed
operand) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import kvsynth
import oracle
from oracle import IndexParams

D = 128
LAM = 1.0 / math.sqrt(D)


def textbook_attention(q, K, V):
    """softmax(q K^T / sqrt(d)) V over all rows, written independently of the oracle."""
    l = (K @ q) / math.sqrt(K.shape[1])
    w = np.exp(l - l.max())
    return (w @ V) / w.sum()


def bf16_keys(rng, n, d=D, scale=1.0):
    return oracle.bf16_round(scale * rng.standard_normal((n, d)))


def tiny_workload(n, S, Cs, g=1, iters=4, n_sink=4, window=8, budget_k=2, topics=8, seed=5):
    return kvsynth.get_workload("tiny-8k").with_(
        n_ctx=n, seg_len=S, clusters_per_seg=Cs, iters=iters, n_sink=n_sink, local_window=window,
        budget_k=budget_k, n_topics=topics, n_q_heads=g, n_kv_heads=1, seed=seed)


def gen_unit(w, step=0):
    k, v = kvsynth.kv_cache(w)
    q = kvsynth.queries(w, step=step)
    K = oracle.bf16_from_bits(k).reshape(w.units, w.n_ctx, D)
    V = oracle.bf16_from_bits(v).reshape(w.units, w.n_ctx, D)
    Q = oracle.bf16_from_bits(q).reshape(w.units, w.group, D)
    return K, V, Q


def params_of(w):
    return IndexParams(seg_len=w.seg_len, clusters_per_seg=w.clusters_per_seg, iters=w.iters, n_sink=w.n_sink,
                       local_window=w.local_window, budget_frac=w.budget_frac, budget_k=w.budget_k)


# ------------------------------------------------------------------ bf16 ----

def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(0)
    x32 = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.bf16_round(x32.astype(np.float64)), ref)


def test_bf16_round_hand_values():
    # ulp of bf16 at 1.0 is 2**-7; halfway cases round to the even significand
    assert oracle.bf16_round(1 + 2.0 ** -8) == 1.0
    assert oracle.bf16_round(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6
    assert oracle.bf16_round(1 + 2.0 ** -8 + 2.0 ** -30) == 1 + 2.0 ** -7
    assert oracle.bf16_round(-3.0) == -3.0
    bits = oracle.bf16_to_bits(np.array([1.0, -2.0, 0.5]))
    assert list(bits) == [0x3F80, 0xC000, 0x3F00]
    np.testing.assert_array_equal(oracle.bf16_from_bits(bits), [1.0, -2.0, 0.5])


def test_generator_rounding_agrees_with_oracle_rounding():
    rng = np.random.default_rng(1)
    xs = rng.standard_normal(2000) * 10
    for x in xs:
        assert oracle.bf16_from_bits(np.uint16(kvsynth.bf16_bits(x))) == oracle.bf16_round(x)


def test_generator_splitmix_published_value():
    # SplitMix64 seeded with 0: first output 0xE220A8397B1DCDAF (Steele et al. reference sequence)
    assert kvsynth.draw(0, 0) == 0xE220A8397B1DCDAF


# ---------------------------------------------------------- P1 all = full ----

@pytest.mark.parametrize("g", [1, 4])
def test_all_clusters_selected_is_full_attention(g):
    w = tiny_workload(n=512, S=128, Cs=8, g=g, budget_k=10 ** 6)
    K, V, Q = gen_unit(w)
    p = params_of(w)
    idx = oracle.build_index(K, V, p)
    o = oracle.decode(Q, K, V, idx, p, g)
    for h in range(g):
        np.testing.assert_allclose(o[0, h], textbook_attention(Q[0, h], K[0], V[0]), rtol=0, atol=1e-12)


def test_all_clusters_selected_with_appended_tokens():
    w = tiny_workload(n=512, S=128, Cs=8, budget_k=10 ** 6)
    K, V, Q = gen_unit(w)
    ka, va = kvsynth.kv_cache(w, p0=512, p1=517)
    KA = oracle.bf16_from_bits(ka).reshape(1, 5, D)
    VA = oracle.bf16_from_bits(va).reshape(1, 5, D)
    p = params_of(w)
    idx = oracle.build_index(K, V, p)
    o = oracle.decode(Q, K, V, idx, p, 1, k_app=KA, v_app=VA)
    ref = textbook_attention(Q[0, 0], np.concatenate([K[0], KA[0]]), np.concatenate([V[0], VA[0]]))
    np.testing.assert_allclose(o[0, 0], ref, rtol=0, atol=1e-12)


# ----------------------------------------------------- P2 singletons exact ----

@pytest.mark.parametrize("k", [1, 3, 7])
def test_singleton_clusters_make_estimation_exact(k):
    rng = np.random.default_rng(2)
    n, S = 64, 32
    K = bf16_keys(rng, n)[None]
    V = bf16_keys(rng, n)[None]
    q = bf16_keys(rng, 1, scale=0.5)
    p = IndexParams(seg_len=S, clusters_per_seg=S, iters=3, n_sink=2, local_window=4, budget_k=k)
    idx = oracle.build_index(K, V, p)
    c = idx[0]["counts"]
    # every clustered token sits alone; steady seeds leave their cluster empty
    assert set(np.unique(c)) <= {0, 1}
    assert c.sum() == n - 6
    o = oracle.decode(q[None], K, V, idx, p, 1)
    np.testing.assert_allclose(o[0, 0], textbook_attention(q[0], K[0], V[0]), rtol=0, atol=1e-12)


# -------------------------------------------------------- P3 Jensen bound ----

def test_estimate_is_jensen_lower_bound_per_cluster():
    w = tiny_workload(n=1024, S=256, Cs=16, g=4, budget_k=3)
    K, V, Q = gen_unit(w)
    p = params_of(w)
    idx = oracle.build_index(K, V, p)[0]
    a = idx["assignment"]
    d_est_total = d_exact_total = 0.0
    for h in range(4):
        q = Q[0, h]
        for j in np.nonzero(idx["counts"] > 0)[0]:
            members = K[0][a == j]
            exact = np.exp(LAM * members @ q).sum()
            est = idx["counts"][j] * np.exp(LAM * idx["mu"][j] @ q)
            mean = members.mean(axis=0)
            slack = math.exp(LAM * np.linalg.norm(q) * np.linalg.norm(idx["mu"][j] - mean))
            assert est <= exact * slack * (1 + 1e-12)
            # with the exact mean the inequality holds without slack
            assert len(members) * np.exp(LAM * mean @ q) <= exact * (1 + 1e-12)
            d_est_total += est / slack
            d_exact_total += exact
    assert d_est_total <= d_exact_total


# ------------------------------------------------- P4 cosh closed form ----

def test_two_token_cluster_estimate_closed_form():
    """Cluster B = {mu + delta, mu - delta}, estimated: its exact share over its
    estimated share is cosh(lam q.delta), and the output is the closed form."""
    rng = np.random.default_rng(3)
    d = 4
    lam = 1 / math.sqrt(d)
    # rows: 0 sink | 1, 2 cluster A (retrieved) | 3, 4 cluster B (estimated) | 5 window
    muB = np.array([0.5, -0.25, 1.0, 0.75])
    delta = np.array([0.25, 0.5, -0.125, 0.0])
    K = np.stack([[1.0, 0, 0, 0], [2.0, 2.0, 2.0, 1.0], [2.0, 1.0, 2.0, 2.0], muB + delta, muB - delta,
                  [0, 1.0, 0, 0]])
    V = rng.standard_normal((6, d))
    q = np.array([0.5, 1.0, 0.25, -0.5])
    idx = {"assignment": np.array([-1, 0, 0, 1, 1, -1]), "counts": np.array([2, 2]),
           "mu": np.array([(K[1] + K[2]) / 2, muB]), "valsum": np.array([V[1] + V[2], V[3] + V[4]])}
    assert idx["mu"][0] @ q > muB @ q
    p = IndexParams(seg_len=6, clusters_per_seg=2, n_sink=1, local_window=1, budget_k=1)
    o = oracle.decode_unit(q[None], K, V, idx, p)[0]
    exact_rows = [0, 1, 2, 5]
    l = lam * K[exact_rows] @ q
    eB = lam * muB @ q
    N = np.exp(l) @ V[exact_rows] + math.exp(eB) * (V[3] + V[4])
    Dn = np.exp(l).sum() + 2 * math.exp(eB)
    np.testing.assert_allclose(o, N / Dn, rtol=1e-13, atol=0)
    exact_B = math.exp(lam * K[3] @ q) + math.exp(lam * K[4] @ q)
    np.testing.assert_allclose(exact_B / (2 * math.exp(eB)), math.cosh(lam * q @ delta), rtol=1e-14)


# ----------------------------------------------------- P5 brute force ----

def brute_assign(k_idx, c):
    out = []
    for i in range(k_idx.shape[0]):
        best, bj = -math.inf, -1
        for j in range(c.shape[0]):
            s = sum(float(k_idx[i, e]) * float(c[j, e]) for e in range(k_idx.shape[1]))
            if s > best:          # strict: the first (lowest) j keeps a tie
                best, bj = s, j
        out.append(bj)
    return np.array(out)


def brute_decode(q, K, V, idx, n_sink, window, k):
    n, d = K.shape
    lam = 1 / math.sqrt(d)
    counts, mu, vs, a = idx["counts"], idx["mu"], idx["valsum"], idx["assignment"]
    ids = [j for j in range(len(counts)) if counts[j] > 0]
    scored = sorted(ids, key=lambda j: (-float(mu[j] @ q), j))
    R = set(scored[:min(k, len(ids))])
    num = np.zeros(d)
    den = 0.0
    for i in range(n):
        if i < n_sink or i >= n - window or a[i] in R:
            wgt = math.exp(lam * sum(q[e] * K[i, e] for e in range(d)))
            den += wgt
            num += wgt * V[i]
    for j in ids:
        if j not in R:
            wgt = math.exp(lam * float(mu[j] @ q))
            den += counts[j] * wgt
            num += wgt * vs[j]
    return num / den, sorted(R)


def test_brute_force_tiny():
    rng = np.random.default_rng(4)
    n, S, Cs, d = 96, 32, 4, 16
    K = oracle.bf16_round(rng.standard_normal((n, d)) + np.repeat(rng.standard_normal((12, d)) * 2, 8, axis=0))
    V = oracle.bf16_round(rng.standard_normal((n, d)))
    q = oracle.bf16_round(rng.standard_normal(d))
    p = IndexParams(seg_len=S, clusters_per_seg=Cs, iters=3, n_sink=4, local_window=8, budget_k=3)
    idx = oracle.build_unit_index(K, V, p)
    # assignment of each segment's last iteration against exhaustive search
    steady = np.zeros(n, bool)
    steady[oracle.steady_positions(n, p)] = True
    for s in range(n // S):
        seg = np.arange(s * S, (s + 1) * S)
        loc = np.nonzero(~steady[seg])[0]
        c_last = idx["histories"][s][-1]
        np.testing.assert_array_equal(idx["assignment"][seg[loc]] - s * Cs, brute_assign(K[seg[loc]], c_last))
    o, info = oracle.decode_unit(q[None], K, V, idx, p, details=True)
    ob, Rb = brute_decode(q, K, V, idx, 4, 8, 3)
    np.testing.assert_array_equal(info[0]["selected"], Rb)
    np.testing.assert_allclose(o[0], ob, rtol=1e-12, atol=1e-14)


# ----------------------------------------------------- P6 k-means sanity ----

def test_planted_clusters_recovered():
    rng = np.random.default_rng(6)
    S, Cs, d = 256, 16, D
    dirs = rng.standard_normal((Cs, d))
    dirs /= np.linalg.norm(dirs, axis=1, keepdims=True)
    label = np.arange(S) // (S // Cs)          # seed 16*j lands in planted cluster j
    K = oracle.bf16_round(10 * dirs[label] + 0.05 * rng.standard_normal((S, d)))
    p = IndexParams(seg_len=S, clusters_per_seg=Cs, iters=5, n_sink=0, local_window=0)
    a, _ = oracle.spherical_kmeans(K, np.arange(S), p)
    np.testing.assert_array_equal(a, label)


def _axis_keys(norms, d=D):
    """Keys norms[i] * e_i (exactly representable in bf16 for the norms used below)."""
    k = np.zeros((len(norms), d))
    for i, s in enumerate(norms):
        k[i, i] = s
    return k


def test_update_sums_unit_vectors_hand_value():
    """Spherical update (RetroInfer fr 2.A.2, spherical k-means): the new centroid is the
    normalised sum of the members' UNIT vectors, rounded to bf16.

    Members 3 e0, 0.5 e1, 2 e2 have unequal norms.  Their unit vectors sum to
    (1, 1, 1), normalised 1/sqrt(3) = 0.57735... per coordinate, binary
    0.10010011|1101...: eight significant bits round up to 0.10010100 = 148/256.
    Two members 3 e0 and e1 give (1, 1)/sqrt(2) = 0.70710678... = 0.10110101|0000...,
    which rounds down to 181/256.  A sum of the raw keys would give (3, .5, 2)/|.|
    and (3, 1)/|.| instead."""
    c_prev = oracle.bf16_round(np.random.default_rng(61).standard_normal((2, D)))
    k3 = _axis_keys([3.0, 0.5, 2.0])
    c = oracle.update(k3, np.zeros(3, np.int64), c_prev)
    want = np.zeros(D)
    want[:3] = 148.0 / 256.0
    np.testing.assert_array_equal(c[0], want)
    k2 = _axis_keys([3.0, 1.0])
    c = oracle.update(k2, np.array([1, 1]), c_prev)
    want = np.zeros(D)
    want[:2] = 181.0 / 256.0
    np.testing.assert_array_equal(c[1], want)


def test_update_empty_cluster_keeps_previous_centroid():
    """A cluster with no member keeps its centroid bit for bit (neither zeroed nor renormalised)."""
    rng = np.random.default_rng(62)
    c_prev = oracle.bf16_round(0.37 * rng.standard_normal((4, D)))   # deliberately not unit-norm
    k = oracle.bf16_round(rng.standard_normal((5, D)))
    a = np.array([0, 0, 3, 3, 0])
    c = oracle.update(k, a, c_prev)
    np.testing.assert_array_equal(c[1], c_prev[1])
    np.testing.assert_array_equal(c[2], c_prev[2])
    for j in (0, 3):   # members' unit vectors, summed and normalised (exact sum order is irrelevant at bf16)
        u = sum(k[i] / np.linalg.norm(k[i]) for i in np.nonzero(a == j)[0])
        np.testing.assert_array_equal(c[j], oracle.bf16_round(u / np.linalg.norm(u)))


def test_zero_keys_have_no_direction():
    """A key of norm 0 adds nothing to its cluster's spherical sum: members {3 e0, 0} give e0
    exactly, as {3 e0} alone; a cluster whose members are all zero, or whose unit vectors cancel
    ({2 e1, -5 e1}), gets the zero centroid; a zero seed gives the zero centroid, which scores 0
    against every key (so a key with all scores <= 0 ties at 0 and goes to the lowest such id)."""
    e = np.eye(D)
    k = np.stack([3 * e[0], np.zeros(D), np.zeros(D), 2 * e[1], -5 * e[1]])
    a = np.array([0, 0, 1, 2, 2])
    c_prev = oracle.bf16_round(np.ones((3, D)) / np.sqrt(D))
    c = oracle.update(k, a, c_prev)
    np.testing.assert_array_equal(c[0], e[0])
    np.testing.assert_array_equal(c[1], np.zeros(D))
    np.testing.assert_array_equal(c[2], np.zeros(D))
    assert np.all(np.isfinite(c))
    # segment 0, 2 e1, -e0-e1, 3 e2 with 2 clusters seeded at positions 0 and 2 (stride 2): the first seed
    # is the zero key, so c0 = 0; c1 = bf16(-(e0 + e1)/sqrt 2) = -181/256 on axes 0 and 1.  Scores
    # (K_i . c0, K_i . c1): 0 -> (0, 0), tie, 0; 2 e1 -> (0, -1.41), 0; -e0-e1 -> (0, 1.41), 1;
    # 3 e2 -> (0, 0), tie, 0.
    K = np.stack([np.zeros(D), 2 * e[1], -e[0] - e[1], 3 * e[2]])
    p = IndexParams(seg_len=4, clusters_per_seg=2, iters=1, n_sink=0, local_window=0)
    c0 = oracle.init_centroids(K, p)
    np.testing.assert_array_equal(c0[0], np.zeros(D))
    np.testing.assert_array_equal(c0[1], -(181 / 256) * (e[0] + e[1]))
    assert list(oracle.assign(K, c0)) == [0, 0, 1, 0]


def test_kmeans_second_round_centroid_hand_value():
    """Inside spherical_kmeans the second round's centroids come from the first round's
    assignment by the same spherical update.  Segment of 4 keys 3 e0, 0.5 e1, 2 e2, 4 e3 and
    2 clusters seeded at positions 0 and 2 (stride 2): centroids e0 and e2.  Key 3 e0 scores
    (3, 0) and joins cluster 0; 0.5 e1 and 4 e3 score (0, 0), a tie that goes to the lowest
    id, 0; 2 e2 scores (0, 2) and joins cluster 1.  Cluster 0 = {3 e0, 0.5 e1, 4 e3}: unit
    sum e0 + e1 + e3, normalised 1/sqrt(3) -> 148/256 on those axes; cluster 1 = {2 e2}
    -> e2 exactly."""
    K = _axis_keys([3.0, 0.5, 2.0, 4.0])
    p = IndexParams(seg_len=4, clusters_per_seg=2, iters=2, n_sink=0, local_window=0)
    a, hist = oracle.spherical_kmeans(K, np.arange(4), p)
    e = np.eye(D)
    np.testing.assert_array_equal(hist[0], np.stack([e[0], e[2]]))
    want0 = np.zeros(D)
    want0[[0, 1, 3]] = 148.0 / 256.0
    np.testing.assert_array_equal(hist[1][0], want0)
    np.testing.assert_array_equal(hist[1][1], e[2])


def test_kmeans_objective_non_decreasing():
    w = tiny_workload(n=2048, S=2048, Cs=64, iters=8)
    K, V, _ = gen_unit(w)
    p = params_of(w)
    steady = oracle.steady_positions(w.n_ctx, p)
    loc = np.setdiff1d(np.arange(w.n_ctx), steady)
    khat = K[0][loc] / np.linalg.norm(K[0][loc], axis=1, keepdims=True)
    _, hist = oracle.spherical_kmeans(K[0], loc, p)
    objs = []
    for c in hist:
        a = oracle.assign(K[0][loc], c)
        objs.append(float((khat * c[a]).sum()))
    # exact arithmetic gives a non-decreasing objective; bf16 centroids add
    # at most about 2**-8 relative per cluster
    for t in range(1, len(objs)):
        assert objs[t] >= objs[t - 1] - 4e-3 * abs(objs[t - 1]) / math.sqrt(len(loc))
    assert objs[-1] > objs[0]


def test_segments_are_clustered_independently():
    w = tiny_workload(n=1024, S=512, Cs=16)
    K, V, _ = gen_unit(w)
    p = params_of(w)
    a1 = oracle.build_unit_index(K[0], V[0], p)["assignment"]
    K2 = K[0].copy()
    K2[600:900] = oracle.bf16_round(K2[600:900] * -1.5)
    a2 = oracle.build_unit_index(K2, V[0], p)["assignment"]
    np.testing.assert_array_equal(a1[:512], a2[:512])


# ----------------------------------------------------- P7 conservation ----

def test_index_conservation():
    w = tiny_workload(n=4096, S=1024, Cs=64, g=1)
    K, V, _ = gen_unit(w)
    p = params_of(w)
    idx = oracle.build_unit_index(K[0], V[0], p)
    n = w.n_ctx
    I = oracle.indexed_positions(n, p)
    c = idx["counts"]
    assert c.sum() == I.size
    np.testing.assert_array_equal(np.sort(idx["perm"]), I)            # bijection on I
    np.testing.assert_array_equal(idx["offsets"], p.n_sink + np.concatenate([[0], np.cumsum(c)]))
    np.testing.assert_allclose(idx["valsum"].sum(0), V[0][I].sum(0), rtol=0, atol=1e-4)
    for j in np.nonzero(c)[0]:
        rows = idx["perm"][idx["offsets"][j] - p.n_sink: idx["offsets"][j + 1] - p.n_sink]
        seg = j // p.clusters_per_seg
        assert np.all(rows // p.seg_len == seg)                        # cluster inside its segment
        assert np.all(np.diff(rows) > 0)                                # position order inside a cluster
        assert np.all(idx["assignment"][rows] == j)
        np.testing.assert_array_equal(idx["mu"][j], oracle.bf16_round(K[0][rows].mean(0)))
        np.testing.assert_array_equal(idx["valsum"][j], oracle.fp32_round(V[0][rows].sum(0)))
    # cluster-contiguous slots: slot offsets of segment s start at the segment start
    for s in range(1, n // p.seg_len):
        assert idx["offsets"][s * p.clusters_per_seg] == s * p.seg_len


# ------------------------------------------------------- P8 LSE merge ----

def test_lse_merge_associative():
    rng = np.random.default_rng(8)
    n = 300
    K = bf16_keys(rng, n, scale=2.0)
    V = bf16_keys(rng, n)
    q = bf16_keys(rng, 1)[0]
    single = textbook_attention(q, K, V)
    for trial in range(5):
        cuts = np.sort(rng.choice(np.arange(1, n), size=trial + 1, replace=False))
        parts = [oracle.zone_partial(q, K[a:b], V[a:b], LAM) for a, b in zip([0, *cuts], [*cuts, n])]
        parts.append(oracle.zone_partial(q, K[:0], V[:0], LAM))        # an empty chunk
        np.testing.assert_allclose(oracle.lse_merge(parts), single, rtol=0, atol=1e-13)


# ------------------------------------------------------------- P9 ties ----

def test_ties_go_to_lowest_id():
    rng = np.random.default_rng(9)
    c = oracle.bf16_round(rng.standard_normal((6, D)))
    c[4] = c[1]                                    # duplicated centroid
    k = np.stack([c[1] * 3, c[4] * 2, c[0]])
    a = oracle.assign(k, c)
    assert a[0] == 1 and a[1] == 1 and a[2] == 0
    scores = np.array([1.0, 5.0, 5.0, 2.0, 5.0, 0.5])
    ne = np.array([True, True, True, True, True, False])
    np.testing.assert_array_equal(oracle.select_topk(scores, ne, 2), [1, 2])
    np.testing.assert_array_equal(oracle.select_topk(scores, ne, 4), [1, 2, 3, 4])
    # empty clusters are never selected, and k is capped at the non-empty count
    np.testing.assert_array_equal(oracle.select_topk(scores, ne, 10), [0, 1, 2, 3, 4])


def test_budget_matches_configured_counts():
    p = IndexParams()
    assert oracle.budget_k(512, p) == 10
    assert oracle.budget_k(8192, p) == 148
    assert oracle.budget_k(7680, p) == 139
    assert oracle.budget_k(65536, p) == 1180
    assert oracle.budget_k(16384, p) == 295


def test_steady_zone_partition():
    p = IndexParams(n_sink=4, local_window=64)
    n = 8192
    s = oracle.steady_positions(n, p)
    i = oracle.indexed_positions(n, p)
    assert s.size == 68 and i.size == n - 68
    assert np.intersect1d(s, i).size == 0
    np.testing.assert_array_equal(np.sort(np.concatenate([s, i])), np.arange(n))


# ------------------------------------------------- full-attention oracle ----

def test_full_attention_equals_wave_index_with_every_cluster_retrieved():
    """The comparator's oracle against the (separately pinned) tripartite decode with a budget
    above the cluster count, appended tokens included: two different computations of one value."""
    w = tiny_workload(n=512, S=128, Cs=8, g=4, budget_k=10 ** 6)
    K, V, Q = gen_unit(w)
    ka, va = kvsynth.kv_cache(w, p0=512, p1=515)
    KA = oracle.bf16_from_bits(ka).reshape(1, 3, D)
    VA = oracle.bf16_from_bits(va).reshape(1, 3, D)
    p = params_of(w)
    idx = oracle.build_index(K, V, p)
    wave = oracle.decode(Q, K, V, idx, p, 4, k_app=KA, v_app=VA)
    np.testing.assert_allclose(oracle.full_attention(Q, K, V, KA, VA), wave, rtol=0, atol=1e-12)


def test_full_attention_closed_forms():
    rng = np.random.default_rng(3)
    V = rng.standard_normal((1, 40, D))
    Q = rng.standard_normal((1, 2, D))
    # one row: the weights are {1}, the output is that value row
    np.testing.assert_allclose(oracle.full_attention(Q, rng.standard_normal((1, 1, D)), V[:, :1]),
                               np.repeat(V[:, :1], 2, axis=1), rtol=0, atol=1e-15)
    # identical keys: uniform weights, the output is the mean value row
    Kc = np.repeat(rng.standard_normal((1, 1, D)), 40, axis=1)
    np.testing.assert_allclose(oracle.full_attention(Q, Kc, V), np.repeat(V.mean(axis=1, keepdims=True), 2, axis=1),
                               rtol=0, atol=1e-13)
    # attention is a set function of the (key, value) rows: any row order gives the same output
    K = rng.standard_normal((1, 40, D))
    perm = rng.permutation(40)
    np.testing.assert_allclose(oracle.full_attention(Q, K[:, perm], V[:, perm]), oracle.full_attention(Q, K, V),
                               rtol=0, atol=1e-13)


# ------------------------------------------------ group-shared retrieval ----

def test_group_topk_variant_pins():
    """The variant in which a kv head's query heads share the top-k of their summed scores:
    one head reduces to the default decode; the shared selection is the brute-force top-k of
    sum_h q_h . mu_j (explicit loops, full sort, ties to the lowest id) for every head; with every
    cluster retrieved it is full attention."""
    w = tiny_workload(n=1024, S=256, Cs=16, g=4, budget_k=5, seed=17)
    K, V, Q = gen_unit(w)
    p = params_of(w)
    idx = oracle.build_index(K, V, p)
    # one head: identical to the per-head definition
    o1 = oracle.decode(Q[:, :1], K, V, idx, p, 1, group_topk=True)
    np.testing.assert_array_equal(o1, oracle.decode(Q[:, :1], K, V, idx, p, 1))
    # the shared selection, brute force
    out, info = oracle.decode_unit(Q[0], K[0], V[0], idx[0], p, details=True, group_topk=True)
    counts, mu = idx[0]["counts"], idx[0]["mu"]
    summed = [(-sum(float(np.dot(Q[0, h], mu[j])) for h in range(4)), j) for j in range(mu.shape[0]) if counts[j] > 0]
    want = sorted(j for _, j in sorted(summed)[:5])
    for h in range(4):
        assert list(info[h]["selected"]) == want
    # the heads' own selections differ from the shared one somewhere (the variant is not the default)
    _, own = oracle.decode_unit(Q[0], K[0], V[0], idx[0], p, details=True)
    assert any(list(own[h]["selected"]) != want for h in range(4))
    assert not np.allclose(out, oracle.decode_unit(Q[0], K[0], V[0], idx[0], p))
    # every cluster retrieved: full attention
    wa = tiny_workload(n=1024, S=256, Cs=16, g=4, budget_k=10 ** 6, seed=17)
    np.testing.assert_allclose(oracle.decode(Q, K, V, idx, params_of(wa), 4, group_topk=True),
                               oracle.full_attention(Q, K, V), rtol=0, atol=1e-12)


# ------------------------------------------- decode-time index maintenance ----

def grown_case(n=2048, S=256, Cs=16, W=8, n_sink=4, appended=600, iters=3, seed=12, budget_k=3):
    w = tiny_workload(n=n, S=S, Cs=Cs, g=2, iters=iters, n_sink=n_sink, window=W, budget_k=budget_k, seed=seed)
    K, V, Q = gen_unit(w)
    ka, va = kvsynth.kv_cache(w, p0=n, p1=n + appended)
    KA = oracle.bf16_from_bits(ka).reshape(appended, D)
    VA = oracle.bf16_from_bits(va).reshape(appended, D)
    p = params_of(w)
    idx = oracle.build_unit_index(K[0], V[0], p)
    K_all, V_all = np.concatenate([K[0], KA]), np.concatenate([V[0], VA])
    return w, p, K[0], V[0], Q[0], KA, VA, K_all, V_all, idx


def test_grown_segment_equals_build_of_that_segment_alone():
    """A segment added during decode is clustered exactly like a build segment of its own
    (segments are independent, de/fr/zh 2.A): its counts, mean keys, value sums, member order
    and assignment equal build_unit_index run on those seg_len rows alone (no steady zone)."""
    w, p, K, V, Q, KA, VA, K_all, V_all, idx = grown_case()
    n, S, Cs = w.n_ctx, p.seg_len, p.clusters_per_seg
    assert oracle.grown_segments(600, p) == 2
    gi = oracle.grow_unit_index(idx, K_all, V_all, n, p)
    C0 = idx["counts"].shape[0]
    assert gi["counts"].shape[0] == C0 + 2 * Cs and gi["grown"] == 2
    w0 = n - p.local_window
    p_alone = IndexParams(seg_len=S, clusters_per_seg=Cs, iters=p.iters, n_sink=0, local_window=0)
    n_idx = idx["perm"].size
    for g in range(2):
        pos = w0 + g * S + np.arange(S)
        ref = oracle.build_unit_index(K_all[pos], V_all[pos], p_alone)
        sl = slice(C0 + g * Cs, C0 + (g + 1) * Cs)
        np.testing.assert_array_equal(gi["counts"][sl], ref["counts"])
        np.testing.assert_array_equal(gi["mu"][sl], ref["mu"])
        np.testing.assert_array_equal(gi["valsum"][sl], ref["valsum"])
        np.testing.assert_array_equal(gi["assignment"][pos], C0 + g * Cs + ref["assignment"])
        np.testing.assert_array_equal(gi["perm"][n_idx + g * S:n_idx + (g + 1) * S], pos[ref["perm"]])
        np.testing.assert_array_equal(gi["offsets"][sl], n + g * S + ref["offsets"][:-1])
    # the build's part is untouched; the window past the grown segments is not clustered
    np.testing.assert_array_equal(gi["counts"][:C0], idx["counts"])
    np.testing.assert_array_equal(gi["assignment"][:w0], idx["assignment"][:w0])
    assert np.all(gi["assignment"][w0 + 2 * S:] == -1)
    assert gi["counts"].sum() == idx["counts"].sum() + 2 * S


def test_all_clusters_after_growth_is_full_attention():
    """Every cluster retrieved after growth: the zones partition the n + appended tokens, so the
    output is textbook softmax attention over all of them (1e-12)."""
    w, p, K, V, Q, KA, VA, K_all, V_all, idx = grown_case(budget_k=10 ** 6)
    gi = oracle.grow_unit_index(idx, K_all, V_all, w.n_ctx, p)
    o = oracle.decode_unit(Q, K, V, gi, p, KA, VA)
    for h in range(Q.shape[0]):
        np.testing.assert_allclose(o[h], textbook_attention(Q[h], K_all, V_all), rtol=1e-12, atol=1e-14)


def test_singleton_grown_clusters_make_estimation_exact():
    """clusters_per_seg = seg_len: every cluster, grown ones included, holds one token, so the
    estimate is exact for any budget and the output is full attention."""
    w, p, K, V, Q, KA, VA, K_all, V_all, idx = grown_case(n=1024, S=128, Cs=128, appended=300, budget_k=2)
    gi = oracle.grow_unit_index(idx, K_all, V_all, w.n_ctx, p)
    assert gi["grown"] == 2 and gi["counts"].max() == 1
    o = oracle.decode_unit(Q, K, V, gi, p, KA, VA)
    for h in range(Q.shape[0]):
        np.testing.assert_allclose(o[h], textbook_attention(Q[h], K_all, V_all), rtol=1e-10, atol=1e-12)


def test_budget_counts_grown_clusters():
    """k = ceil(budget_frac * C) counts the grown segments' clusters too."""
    w, p, K, V, Q, KA, VA, K_all, V_all, idx = grown_case(budget_k=0)
    p = IndexParams(seg_len=p.seg_len, clusters_per_seg=p.clusters_per_seg, iters=p.iters, n_sink=p.n_sink,
                    local_window=p.local_window, budget_frac=0.05)
    gi = oracle.grow_unit_index(idx, K_all, V_all, w.n_ctx, p)
    _, info = oracle.decode_unit(Q, K, V, gi, p, KA, VA, details=True)
    C = gi["counts"].shape[0]
    assert len(info[0]["selected"]) == math.ceil(0.05 * C) == math.ceil(0.05 * (128 + 32))


@pytest.mark.parametrize("W,appended", [(8, 0), (8, 247), (8, 248), (8, 600), (300, 0), (300, 211), (300, 512)])
def test_window_keeps_between_w_and_w_plus_s_rows(W, appended):
    """READING (decode-time growth): the local window never holds fewer than W rows nor W + S: an
    append that would leave W + S rows turns the oldest S into a segment.  Checked on the zones the
    decode uses: with one cluster retrieved, a head's exact rows are the sinks, the window and that
    cluster's rows, and every clustered row belongs to the build or to a grown segment."""
    S = 256
    w, p, K, V, Q, KA, VA, K_all, V_all, idx = grown_case(n=2048, S=S, Cs=16, W=W, appended=appended, budget_k=1)
    gi = oracle.grow_unit_index(idx, K_all, V_all, w.n_ctx, p)
    _, info = oracle.decode_unit(Q, K, V, gi, p, KA, VA, details=True)
    for h in range(Q.shape[0]):
        (j,) = info[h]["selected"]
        window = info[h]["exact_rows"] - p.n_sink - int(gi["counts"][j])
        assert W <= window < W + S, (W, appended, window)
    # the rows not in the steady zone are exactly the clustered ones
    assert int(gi["counts"].sum()) == w.n_ctx + appended - p.n_sink - (W + appended % S)
