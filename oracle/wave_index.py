"""Wave index, stated plainly in float64 -- TEST INFRASTRUCTURE ONLY.

Sources (the RetroInfer technical summaries; "de", "fr", "zh" name the
gist.science pages of arXiv 2505.02922, "abstract" the chatpaper.ai page):
  * tripartite attention approximation: de/fr/zh section 2.A (steady zone,
    retrieval zone, estimation zone);
  * estimation zone: clusters not retrieved contribute through their
    centroid and precomputed sum of values, a lower bound by Jensen's
    inequality (zh 2.A, "estimation zone"; fr 2.A.3);
  * spherical k-means as the clustering behind the retrieval zone (fr 2.A.2);
  * segmented clustering: the context is cut into segments clustered
    independently (de 2.A closing paragraph, fr 2.A, zh 2.A);
  * retrieval budget of about 1.8% of the index (zh section 3).

Where the pages are silent the plainest reading is taken; each is marked
READING below:
  * the steady zone is the first n_sink and the last `window` positions (plus
    tokens appended during decode); clustering covers every other position,
    so the three zones partition the context;
  * centroid initialisation: the first token of each stride-(S/C_s) block of
    the segment, normalised and rounded to bf16;
  * a zero vector normalises to zero (a key of norm 0 adds nothing to a
    centroid sum; a zero seed or a zero sum gives the zero centroid);
  * spherical k-means on unit-normalised keys; centroids are rounded to bf16
    before every assignment; ties go to the lowest centroid id; empty clusters
    keep their centroid; the index keeps the T-th assignment;
  * the index stores, per cluster, the count n_j, the arithmetic mean of the
    raw keys mu_j (bf16) and the sum of values (fp32); decode scores and
    estimates with mu_j (the Jensen bound holds for the arithmetic mean);
  * top-k per query head over non-empty clusters, ties to the lowest cluster
    id, k = ceil(budget_frac * C) capped at the number of non-empty clusters;
  * logits scaled by 1/sqrt(d); zones merged by log-sum-exp (one softmax).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from .bf16 import bf16_round, fp32_round


@dataclass(frozen=True)
class IndexParams:
    seg_len: int = 8192
    clusters_per_seg: int = 512
    iters: int = 10
    n_sink: int = 4
    local_window: int = 64
    budget_frac: float = 0.018
    budget_k: int = 0          # >0 overrides budget_frac

    @property
    def init_stride(self) -> int:
        return self.seg_len // self.clusters_per_seg


# ----------------------------------------------------------------- zones ----

def steady_positions(n: int, p: IndexParams) -> np.ndarray:
    """Steady zone of a context of n tokens: first n_sink and last window.

    Summaries de/fr/zh 2.A, "steady zone": tokens that matter because of where
    they sit, at the start and the end of the context; computed exactly.
    """
    lo = np.arange(min(p.n_sink, n))
    hi = np.arange(max(n - p.local_window, p.n_sink), n)
    return np.concatenate([lo, hi])


def window_start(n: int, p: IndexParams) -> int:
    """First position of the build's local window (the steady zone's tail)."""
    return max(n - p.local_window, min(p.n_sink, n))


def indexed_positions(n: int, p: IndexParams) -> np.ndarray:
    """Positions that are clustered: the complement of the steady zone."""
    mask = np.ones(n, bool)
    mask[steady_positions(n, p)] = False
    return np.nonzero(mask)[0]


def budget_k(n_clusters: int, p: IndexParams) -> int:
    """Retrieval budget: clusters fetched exactly per query head (zh section 3, ~1.8%)."""
    if p.budget_k > 0:
        return p.budget_k
    return int(math.ceil(p.budget_frac * n_clusters))


# ------------------------------------------------------ spherical k-means ----

def _unit_rows(x: np.ndarray) -> np.ndarray:
    """Rows scaled to unit length.  READING (pages silent): a zero row has no direction and stays
    zero, so a key of norm 0 adds nothing to a spherical sum, and a zero seed or a zero sum gives
    the zero centroid (which scores 0 against every key)."""
    nrm = np.linalg.norm(x, axis=1, keepdims=True)
    return np.divide(x, nrm, out=np.zeros_like(x), where=nrm > 0)


def init_centroids(k_seg: np.ndarray, p: IndexParams) -> np.ndarray:
    """Initial centroids of one segment: bf16(normalise(K[seg_start + stride*j])).

    k_seg holds every position of the segment (steady ones included), so the
    seeds are taken at absolute positions.  READING (pages silent).
    """
    seeds = k_seg[np.arange(p.clusters_per_seg) * p.init_stride]
    return bf16_round(_unit_rows(seeds))


def assign(k_idx: np.ndarray, c_hat: np.ndarray) -> np.ndarray:
    """Spherical assignment: a_i = argmax_j K_i . c_j, ties to the lowest j.

    Summary fr 2.A.2: clustering by spherical k-means.  argmax of the raw dot
    product equals argmax of the cosine because |K_i| is fixed per token.
    np.argmax returns the first maximum, i.e. the lowest j on ties.
    """
    if k_idx.shape[0] == 0:          # a segment that lies wholly in the steady zone
        return np.zeros(0, np.int64)
    scores = k_idx @ c_hat.T
    return np.argmax(scores, axis=1)


def update(k_idx: np.ndarray, a: np.ndarray, c_prev: np.ndarray) -> np.ndarray:
    """Spherical centroid update: c_j = bf16(u_j / |u_j|), u_j = sum_{a_i=j} K_i/|K_i|.

    Empty clusters keep their previous centroid.
    """
    u = np.zeros_like(c_prev)
    np.add.at(u, a, _unit_rows(k_idx))
    c = c_prev.copy()
    counts = np.bincount(a, minlength=c_prev.shape[0])
    ne = counts > 0
    c[ne] = bf16_round(_unit_rows(u[ne]))
    return c


def spherical_kmeans(k_seg: np.ndarray, idx_local: np.ndarray, p: IndexParams,
                     c_init: np.ndarray | None = None, iters: int | None = None):
    """T rounds of (assign, update) on one segment; returns (a, centroid history).

    k_seg: all rows of the segment; idx_local: positions (relative to the
    segment start) that are clustered.  The returned assignment is the T-th;
    history[t] is the centroid set the t-th assignment used.
    """
    iters = p.iters if iters is None else iters
    c = init_centroids(k_seg, p) if c_init is None else c_init
    k_idx = k_seg[idx_local]
    history = []
    a = None
    for t in range(iters):
        history.append(c)
        a = assign(k_idx, c)
        if t + 1 < iters:
            c = update(k_idx, a, c)
    return a, history


# ------------------------------------------------------------- the index ----

def build_unit_index(K: np.ndarray, V: np.ndarray, p: IndexParams, c_init: list | None = None,
                     iters: int | None = None) -> dict:
    """Segmented clustering of one (sequence, layer, kv head) and its index.

    Segments of seg_len tokens are clustered independently (segmented
    clustering, de/fr/zh 2.A); global cluster id = segment * C_s + j.  Per
    cluster: count n_j, mu_j = bf16(mean of raw keys), valsum_j = fp32(sum of
    values) -- the precomputed value sum of the estimation zone (zh 2.A).
    Tokens are listed cluster by cluster, by position inside a cluster
    (`perm`); `offsets` are their row numbers in the cluster-contiguous
    layout, which starts at row n_sink.
    """
    n, d = K.shape
    S, Cs = p.seg_len, p.clusters_per_seg
    nseg = n // S
    C = nseg * Cs
    steady = np.zeros(n, bool)
    steady[steady_positions(n, p)] = True
    assignment = np.full(n, -1, np.int64)
    histories = []
    for s in range(nseg):
        seg = np.arange(s * S, (s + 1) * S)
        idx_local = np.nonzero(~steady[seg])[0]
        ci = None if c_init is None else c_init[s]
        a, hist = spherical_kmeans(K[seg], idx_local, p, c_init=ci, iters=iters)
        assignment[seg[idx_local]] = s * Cs + a
        histories.append(hist)
    idx = np.nonzero(assignment >= 0)[0]
    counts = np.bincount(assignment[idx], minlength=C).astype(np.int64)
    # stable sort by cluster id keeps position order inside each cluster
    perm = idx[np.argsort(assignment[idx], kind="stable")]
    offsets = p.n_sink + np.concatenate([[0], np.cumsum(counts)])
    ksum = np.zeros((C, d))
    vsum = np.zeros((C, d))
    np.add.at(ksum, assignment[idx], K[idx])
    np.add.at(vsum, assignment[idx], V[idx])
    mu = np.zeros((C, d))
    ne = counts > 0
    mu[ne] = bf16_round(ksum[ne] / counts[ne, None])
    return {
        "assignment": assignment, "counts": counts, "offsets": offsets, "perm": perm,
        "mu": mu, "valsum": fp32_round(vsum), "histories": histories,
    }


def grown_segments(n_appended: int, p: IndexParams) -> int:
    """Segments added during decode after n_appended appended tokens.

    READING (decode-time index maintenance; the pages describe the index at
    prefill only): appended tokens join the local window; once a step's append
    leaves the window holding local_window + seg_len rows, its oldest seg_len
    rows become one more segment, so the window is back to local_window rows.
    That happens after every seg_len appended tokens.
    """
    return n_appended // p.seg_len


def grow_unit_index(index: dict, K_all: np.ndarray, V_all: np.ndarray, n: int, p: IndexParams) -> dict:
    """The index of one unit after decode-time growth (see grown_segments).

    K_all, V_all hold the n built rows followed by every appended row.
    Grown segment g covers positions [w0 + g*S, w0 + (g+1)*S), w0 = the
    build's window start; it is clustered on its own like a build segment
    (segmented clustering, de/fr/zh 2.A: the seeds, the spherical rounds and
    the per-cluster count, mean key and value sum), every position of it
    clustered, and its clusters are numbered after all existing ones.  Its
    slots are numbered from row n + g*S (the build's slots end below row n).
    """
    S, Cs = p.seg_len, p.clusters_per_seg
    grown = grown_segments(K_all.shape[0] - n, p)
    w0 = window_start(n, p)
    C0 = index["counts"].shape[0]
    d = K_all.shape[1]
    counts = [index["counts"]]
    mus, vss, perms, offs = [index["mu"]], [index["valsum"]], [index["perm"]], [index["offsets"][:-1]]
    assignment = np.full(K_all.shape[0], -1, np.int64)
    assignment[:n] = index["assignment"][:n]
    for g in range(grown):
        pos = w0 + g * S + np.arange(S)
        a, _ = spherical_kmeans(K_all[pos], np.arange(S), p)
        ids = C0 + g * Cs + a
        assignment[pos] = ids
        cnt = np.bincount(a, minlength=Cs).astype(np.int64)
        order = np.argsort(a, kind="stable")        # by cluster, by position inside a cluster
        ksum = np.zeros((Cs, d))
        vsum = np.zeros((Cs, d))
        np.add.at(ksum, a, K_all[pos])
        np.add.at(vsum, a, V_all[pos])
        mu = np.zeros((Cs, d))
        ne = cnt > 0
        mu[ne] = bf16_round(ksum[ne] / cnt[ne, None])
        counts.append(cnt)
        mus.append(mu)
        vss.append(fp32_round(vsum))
        perms.append(pos[order])
        offs.append(n + g * S + np.concatenate([[0], np.cumsum(cnt)[:-1]]))
    out = dict(index)
    out.update({"counts": np.concatenate(counts), "mu": np.concatenate(mus), "valsum": np.concatenate(vss),
                "perm": np.concatenate(perms), "assignment": assignment, "grown": grown})
    offsets = np.concatenate(offs)
    out["offsets"] = np.concatenate([offsets, [offsets[-1] + out["counts"][-1]]])
    return out


def build_index(K: np.ndarray, V: np.ndarray, p: IndexParams, **kw) -> list:
    """Index of every unit; K, V shaped [units][n][d] (float64)."""
    return [build_unit_index(K[u], V[u], p, **kw) for u in range(K.shape[0])]


# ---------------------------------------------------------------- decode ----

def select_topk(scores: np.ndarray, nonempty: np.ndarray, k: int) -> np.ndarray:
    """Retrieval zone: the k non-empty clusters of highest score, ties to the
    lowest cluster id, returned in ascending id order (de/fr/zh 2.A, retrieval zone)."""
    ids = np.nonzero(nonempty)[0]
    k = min(k, ids.size)
    order = np.lexsort((ids, -scores[ids]))    # by score descending, then id ascending
    return np.sort(ids[order[:k]])


def zone_partial(q: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray, scale: float):
    """(m, Z, N) of exact softmax over some rows: m = max logit,
    Z = sum exp(l - m), N = sum exp(l - m) V."""
    if k_rows.shape[0] == 0:
        return -np.inf, 0.0, np.zeros(q.shape[0])
    l = scale * (k_rows @ q)
    m = l.max()
    w = np.exp(l - m)
    return m, w.sum(), w @ v_rows


def lse_merge(parts) -> np.ndarray:
    """Merge zone partials (m, Z, N) into one softmax output by log-sum-exp."""
    M = max(m for m, _, _ in parts)
    Z = sum(z * math.exp(m - M) for m, z, _ in parts if m > -np.inf)
    N = sum(n * math.exp(m - M) for m, _, n in parts if m > -np.inf)
    return N / Z


def decode_unit(q_heads: np.ndarray, K: np.ndarray, V: np.ndarray, index: dict, p: IndexParams,
                k_app: np.ndarray | None = None, v_app: np.ndarray | None = None, details: bool = False,
                group_topk: bool = False):
    """Tripartite attention of the g query heads of one kv head.

    For each head h (summaries de/fr/zh 2.A; zones merged into one softmax):
      scores s_j = q . mu_j over non-empty clusters;  R = top-k clusters;
      exact set X = steady zone (+ appended tokens) + members of R,
        l_i = q . K_i / sqrt(d);
      estimated set E = non-empty clusters not in R,
        e_j = q . mu_j / sqrt(d), contributing n_j exp(e_j) to the
        denominator and exp(e_j) valsum_j to the numerator;
      o = N / D with M = max over both zones (single sum, float64).
    group_topk: the variant in which the g heads share one retrieval zone, the top-k of the
    summed scores sum_h q_h . mu_j (each head still has its own logits and estimate).
    """
    n, d = K.shape
    scale = 1.0 / math.sqrt(d)
    counts, mu, vs, a = index["counts"], index["mu"], index["valsum"], index["assignment"]
    C = counts.shape[0]
    nonempty = counts > 0
    k = budget_k(C, p)
    if k_app is not None and k_app.shape[0] > 0:
        K = np.concatenate([K, k_app])
        V = np.concatenate([V, v_app])
    if a.shape[0] < K.shape[0]:      # appended positions not clustered (yet)
        a = np.concatenate([a, np.full(K.shape[0] - a.shape[0], -1)])
    # steady zone: the sinks, and the local window from its start (past any grown segment) to the
    # last appended token
    w = window_start(n, p) + index.get("grown", 0) * p.seg_len
    steady = np.concatenate([np.arange(min(p.n_sink, n)), np.arange(w, K.shape[0])])
    ks = K[steady]
    vsd = V[steady]
    out = np.zeros((q_heads.shape[0], d))
    info = []
    R_group = select_topk(mu @ q_heads.sum(axis=0), nonempty, k) if group_topk else None
    for h in range(q_heads.shape[0]):
        q = q_heads[h]
        s = mu @ q
        R = R_group if group_topk else select_topk(s, nonempty, k)
        member = np.isin(a, R)
        kx = np.concatenate([ks, K[member]])
        vx = np.concatenate([vsd, V[member]])
        l = scale * (kx @ q)
        E = nonempty.copy()
        E[R] = False
        e = scale * s[E]
        nE = counts[E].astype(np.float64)
        M = l.max()
        if e.size:
            M = max(M, (e + np.log(nE)).max())
        D = np.exp(l - M).sum() + (nE * np.exp(e - M)).sum()
        N = np.exp(l - M) @ vx + np.exp(e - M) @ vs[E]
        out[h] = N / D
        if details:
            info.append({"scores": s, "selected": R, "exact_rows": int(kx.shape[0])})
    return (out, info) if details else out


def decode(Q: np.ndarray, K: np.ndarray, V: np.ndarray, indexes: list, p: IndexParams, group: int,
           k_app=None, v_app=None, details: bool = False, group_topk: bool = False):
    """Decode over all units. Q [units][g][d]; K, V [units][n][d]; appended rows [units][t][d]."""
    outs, infos = [], []
    for u in range(K.shape[0]):
        ka = None if k_app is None else k_app[u]
        va = None if v_app is None else v_app[u]
        r = decode_unit(Q[u], K[u], V[u], indexes[u], p, ka, va, details=details, group_topk=group_topk)
        if details:
            outs.append(r[0])
            infos.append(r[1])
        else:
            outs.append(r)
    o = np.stack(outs)
    return (o, infos) if details else o


# ------------------------------------------------------ full attention ----

def full_attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, k_app=None, v_app=None) -> np.ndarray:
    """Full (dense) attention, the baseline the summaries measure the wave index against
    (de/fr/zh 2.A: the tripartite approximation stands in for attention over every cached
    token; zh section 3 reports the speed-up over it).

    For every unit u and query head h: softmax(q K^T / sqrt(d)) V over all n context rows of
    the unit followed by its appended rows, in float64.  Q [units][g][d]; K, V [units][n][d];
    appended rows [units][t][d] or None.  Returns [units][g][d]."""
    U, n, d = K.shape
    scale = 1.0 / math.sqrt(d)
    out = np.zeros((U, Q.shape[1], d))
    for u in range(U):
        Ku, Vu = K[u], V[u]
        if k_app is not None and k_app.shape[1] > 0:
            Ku = np.concatenate([Ku, k_app[u]])
            Vu = np.concatenate([Vu, v_app[u]])
        for h in range(Q.shape[1]):
            logits = (Ku @ Q[u, h]) * scale
            w = np.exp(logits - logits.max())
            out[u, h] = (w @ Vu) / w.sum()
    return out
