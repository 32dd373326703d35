"""Decode parity: the CUDA decode step against the float64 oracle, both given
the oracle's index (wi_index_import), on the same seeded input bytes."""
import numpy as np
import pytest
import torch

import kvsynth
import oracle
from helpers import (OUT_REL_L2, check_topk, gen, index_arrays, params_of, rel_l2, small)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def wi():
    import clustered_sparse_kv_gb300 as m
    return m


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV)


def run_case(wi, w, idx=None, steps=1, append=False, kv=None, strict_ids=False):
    """Import the oracle index, decode `steps` steps (with append if asked), compare every step.
    strict_ids: the selection must equal the oracle's exactly (ties included)."""
    k, v, q, K, V, Q = gen(w)
    if kv is not None:
        k, v = kv
        K = oracle.bf16_from_bits(k).reshape(w.units, w.n_ctx, 128)
        V = oracle.bf16_from_bits(v).reshape(w.units, w.n_ctx, 128)
    p = params_of(w)
    if idx is None:
        idx = oracle.build_index(K, V, p)
    cfg = wi.config_from_workload(w, max_append=steps if append else 0)
    kt, vt = dev16(k), dev16(v)
    ix = wi.WaveIndex.adopt(cfg, kt, vt, *index_arrays(idx))
    worst = 0.0
    if append:
        ka, va = kvsynth.kv_cache(w, p0=w.n_ctx, p1=w.n_ctx + steps)
        KA = oracle.bf16_from_bits(ka).reshape(w.units, steps, 128)
        VA = oracle.bf16_from_bits(va).reshape(w.units, steps, 128)
    for t in range(steps):
        qb = kvsynth.queries(w, step=t)
        Qt = oracle.bf16_from_bits(qb).reshape(w.units, w.group, 128)
        kn = vn = None
        if append:
            kn, vn = dev16(ka[:, :, :, t]), dev16(va[:, :, :, t])
        out = ix.decode(dev16(qb), kn, vn)
        ids, cnt = ix.selection()
        torch.cuda.synchronize()
        ix.check()
        got = out.cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64)
        kap = KA[:, :t] if append else None
        vap = VA[:, :t] if append else None
        ref, info = oracle.decode(Qt, K, V, idx, p, w.group, k_app=kap, v_app=vap, details=True)
        err = rel_l2(got, ref)
        assert err.max() <= OUT_REL_L2, (t, err.max())
        worst = max(worst, float(err.max()))
        ids, cnt = ids.cpu().numpy(), cnt.cpu().numpy()
        for u in range(w.units):
            ne = idx[u]["counts"] > 0
            kk = oracle.budget_k(w.clusters, p)
            for h in range(w.group):
                check_topk(ids[u, h], cnt[u, h], info[u][h]["scores"], ne, kk)
                if strict_ids:
                    ref_ids = np.sort(oracle.select_topk(info[u][h]["scores"], ne, kk))
                    assert np.array_equal(ids[u, h][:cnt[u, h]], ref_ids), (u, h)
    ix.free()
    return worst


@pytest.mark.parametrize("g", [1, 2, 3, 4, 5, 6, 7, 8])
def test_decode_parity_group_sizes(wi, g):
    """Every group size the kernels are instantiated for (1-8 query heads per kv head: different
    head packings in the scores MMA and the estimation's lane layout)."""
    w = small(n_ctx=4096, seg_len=1024, clusters_per_seg=64, iters=3, n_q_heads=g, n_kv_heads=1, budget_k=6)
    assert run_case(wi, w) < 1e-4


def test_decode_parity_zero_keys(wi):
    """Keys of norm 0 throughout the context (steady and clustered), with the oracle's index."""
    w = small(batch=1, n_q_heads=8, n_kv_heads=2, n_ctx=4096, seg_len=1024, clusters_per_seg=64, iters=2,
              budget_k=6, seed=89)
    k, v, q, K, V, Q = gen(w)
    rng = np.random.default_rng(89)
    shape = k.shape
    k = k.copy().reshape(w.units, w.n_ctx, 128)
    for u in range(w.units):
        k[u, rng.choice(w.n_ctx, 300, replace=False)] = 0
        k[u, :2] = 0                       # two sinks
        k[u, w.n_ctx - 5:] = 0             # the window's last rows
    assert run_case(wi, w, kv=(k.reshape(shape), v)) < 1e-4


@pytest.mark.parametrize("seg,cs", [(128, 16), (256, 32)])
def test_decode_parity_small_geometries(wi, seg, cs):
    """128- and 256-token segments with 16 and 32 clusters (the smallest the configuration admits):
    many segments, few tokens per cluster, a budget of a fifth of the clusters."""
    w = small(batch=2, n_q_heads=8, n_kv_heads=2, n_ctx=32 * seg, seg_len=seg, clusters_per_seg=cs, iters=2,
              budget_k=(32 * cs) // 5, seed=40 + cs)
    assert run_case(wi, w, steps=2, append=True) < 1e-4


@pytest.mark.parametrize("g", [3, 5, 8])
def test_decode_parity_group_sizes_multi_unit(wi, g):
    """The odd group sizes with several units and an appending step."""
    w = small(batch=2, n_q_heads=2 * g, n_kv_heads=2, n_ctx=4096, seg_len=1024, clusters_per_seg=64, iters=2,
              budget_k=7, seed=30 + g)
    assert run_case(wi, w, steps=2, append=True) < 1e-4


def test_decode_parity_multi_unit(wi):
    w = small(batch=2, layers=2, n_q_heads=8, n_kv_heads=2, n_ctx=2048, seg_len=512, clusters_per_seg=32, iters=2,
              budget_k=5, seed=11)
    assert run_case(wi, w) < 1e-4


def test_decode_tiny_workload_full_size(wi):
    w = kvsynth.get_workload("tiny-8k")
    assert run_case(wi, w) < 1e-4


def test_all_clusters_selected_is_full_attention(wi):
    w = small(n_ctx=2048, seg_len=512, clusters_per_seg=32, iters=2, n_q_heads=4, budget_k=128)
    k, v, q, K, V, Q = gen(w)
    p = params_of(w)
    idx = oracle.build_index(K, V, p)
    cfg = wi.config_from_workload(w)
    ix = wi.WaveIndex.adopt(cfg, dev16(k), dev16(v), *index_arrays(idx))
    out = ix.decode(dev16(q)).cpu().numpy().reshape(1, 4, 128)
    for h in range(4):
        l = K[0] @ Q[0, h] / np.sqrt(128)
        wgt = np.exp(l - l.max())
        full = wgt @ V[0] / wgt.sum()
        assert rel_l2(out[0, h], full) < 1e-5
    ix.free()


def degenerate_kv(w, lo, hi):
    """Generator cache with positions [lo, hi) overwritten by copies of one key row:
    one giant cluster, duplicated seeds (ties to the lowest id) and many empty clusters."""
    k, v = kvsynth.kv_cache(w)
    k[:, :, :, lo:hi] = k[:, :, :, lo:lo + 1]
    return k, v


def test_decode_ragged_clusters(wi):
    w = small(n_ctx=2048, seg_len=1024, clusters_per_seg=64, iters=4, n_q_heads=4, budget_k=7, seed=21)
    k, v = degenerate_kv(w, 100, 900)
    K = oracle.bf16_from_bits(k).reshape(1, w.n_ctx, 128)
    V = oracle.bf16_from_bits(v).reshape(1, w.n_ctx, 128)
    idx = oracle.build_index(K, V, params_of(w))
    c = idx[0]["counts"]
    assert (c == 0).sum() > 40 and c.max() >= 800
    assert run_case(wi, w, idx=idx, kv=(k, v)) < 1e-4


def test_decode_budget_above_nonempty(wi):
    w = small(n_ctx=2048, seg_len=1024, clusters_per_seg=64, iters=4, n_q_heads=4, budget_k=100, seed=22)
    k, v = degenerate_kv(w, 50, 1000)
    K = oracle.bf16_from_bits(k).reshape(1, w.n_ctx, 128)
    V = oracle.bf16_from_bits(v).reshape(1, w.n_ctx, 128)
    idx = oracle.build_index(K, V, params_of(w))
    assert (idx[0]["counts"] > 0).sum() < 100
    assert run_case(wi, w, idx=idx, kv=(k, v)) < 1e-4


def tied_index(w, pattern):
    """Oracle index whose mean keys are overwritten so that scores tie: `pattern(j)` picks, per
    cluster j, which of two fixed mean-key rows it gets (equal rows give bitwise-equal scores)."""
    k, v, q, K, V, Q = gen(w)
    idx = oracle.build_index(K, V, params_of(w))
    for u in range(w.units):
        mu = idx[u]["mu"]
        rows = [mu[0].copy(), mu[1].copy()]
        for j in range(mu.shape[0]):
            mu[j] = rows[pattern(j)]
    return idx


def test_topk_all_scores_tied(wi):
    # every score equal: more tied keys than top-k threads, the k lowest non-empty ids win
    w = small(n_ctx=8192, seg_len=1024, clusters_per_seg=128, iters=1, n_q_heads=4, budget_k=100, seed=31)
    idx = tied_index(w, lambda j: 0)
    assert (idx[0]["counts"] > 0).sum() > 600
    assert run_case(wi, w, idx=idx, strict_ids=True) < 1e-4


def test_topk_half_tied(wi):
    # two score levels, each shared by half the clusters: the threshold level holds ~512 ties
    w = small(n_ctx=8192, seg_len=1024, clusters_per_seg=128, iters=1, n_q_heads=4, budget_k=100, seed=32)
    idx = tied_index(w, lambda j: j & 1)
    assert run_case(wi, w, idx=idx, strict_ids=True) < 1e-4


@pytest.mark.parametrize("n_ctx,budget", [(131072, 0), (81920, 37)])
def test_topk_large_cluster_count(wi, n_ctx, budget):
    """Above 32768 clusters per kv head the top-k keeps 16-bit distance bins in shared memory
    instead of the keys: C = 65536 (k = 1180, the million-token budget) and C = 40960."""
    w = small(n_ctx=n_ctx, seg_len=1024, clusters_per_seg=512, iters=1, n_q_heads=4, budget_k=budget,
              budget_frac=0.018, seed=34)
    assert w.clusters > 32768
    assert run_case(wi, w, strict_ids=False) < 1e-4


def test_topk_cluster_count_at_the_key_cache_limit(wi):
    """C = 32768, the most clusters whose keys the top-k keeps in shared memory (k = 590, above the
    list capacity), and the same count with every score tied (the radix path over the cached keys)."""
    w = small(n_ctx=65536, seg_len=1024, clusters_per_seg=512, iters=1, n_q_heads=4, budget_k=0,
              budget_frac=0.018, seed=37)
    assert w.clusters == 32768
    assert run_case(wi, w, strict_ids=False) < 1e-4
    w = w.with_(budget_k=100, seed=38)
    assert run_case(wi, w, idx=tied_index(w, lambda j: 0), strict_ids=True) < 1e-4


def test_topk_large_cluster_count_ties(wi):
    """Every score tied at C = 65536 (more ties than ranking threads: the radix path over keys read
    from global memory) and two score levels at C = 40960; the selection must equal the oracle's."""
    w = small(n_ctx=131072, seg_len=1024, clusters_per_seg=512, iters=1, n_q_heads=4, budget_k=100, seed=35)
    assert run_case(wi, w, idx=tied_index(w, lambda j: 0), strict_ids=True) < 1e-4
    w = small(n_ctx=81920, seg_len=1024, clusters_per_seg=512, iters=1, n_q_heads=4, budget_k=300, seed=36)
    assert run_case(wi, w, idx=tied_index(w, lambda j: (j * 7) % 3 == 0), strict_ids=True) < 1e-4


def test_decode_large_budget(wi):
    # k above the top-k's list capacity (512): the selection goes through per-chunk bit masks
    w = small(n_ctx=16384, seg_len=1024, clusters_per_seg=128, iters=2, n_q_heads=4, budget_k=700, seed=33)
    assert run_case(wi, w, strict_ids=False) < 1e-4


def test_decode_largest_budget(wi):
    # k = 4096, the largest budget the configuration admits, over C = 8192 clusters
    w = small(n_ctx=65536, seg_len=1024, clusters_per_seg=128, iters=1, n_q_heads=4, budget_k=4096, seed=39)
    assert w.clusters == 8192
    assert run_case(wi, w, strict_ids=False) < 1e-4


@pytest.mark.parametrize("n_sink,window", [(0, 16), (8, 0), (4, 64)])
def test_decode_steady_zone_shapes(wi, n_sink, window):
    w = small(n_ctx=2048, seg_len=512, clusters_per_seg=32, iters=2, n_q_heads=4, n_sink=n_sink,
              local_window=window, budget_k=4, seed=31)
    assert run_case(wi, w) < 1e-4


def test_decode_with_append(wi):
    w = small(batch=2, n_ctx=2048, seg_len=512, clusters_per_seg=32, iters=2, n_q_heads=7, n_kv_heads=1,
              budget_k=5, append=True, decode_steps=6, seed=41)
    assert run_case(wi, w, steps=6, append=True) < 1e-4


def test_append_buffer_full(wi):
    w = small(n_ctx=1024, seg_len=512, clusters_per_seg=32, iters=1, n_q_heads=1, budget_k=2)
    k, v, q, K, V, Q = gen(w)
    cfg = wi.config_from_workload(w, max_append=1)
    ix = wi.WaveIndex.build(cfg, dev16(k), dev16(v))
    kn = torch.zeros((1, 1, 1, 128), dtype=torch.int16, device=DEV)
    ix.decode(dev16(q), kn, kn)
    with pytest.raises(wi.WiError) as e:
        ix.decode(dev16(q), kn, kn)
    assert e.value.code == wi.WI_EFULL
    ix.decode(dev16(q))  # without append still fine
    torch.cuda.synchronize()
    ix.free()


def test_host_buffer_variant_matches(wi):
    w = small(n_ctx=2048, seg_len=512, clusters_per_seg=32, iters=2, n_q_heads=4, budget_k=4, seed=51)
    k, v, q, K, V, Q = gen(w)
    cfg = wi.config_from_workload(w)
    ix = wi.WaveIndex.build(cfg, dev16(k), dev16(v))
    ref = ix.decode(dev16(q)).cpu()
    qh = torch.from_numpy(q.view(np.int16)).pin_memory()
    oh = torch.empty((1, 1, 4, 128), dtype=torch.float32).pin_memory()
    wi.wi_decode_step_host(ix.handle, qh, oh)  # pinned buffers: the captured graph
    assert torch.equal(oh, ref)
    # other pinned buffers and other queries through the same graph (its copy addresses are reset
    # at every call), and pageable buffers (direct launches)
    for t in (1, 2):
        qt = kvsynth.queries(w, step=t)
        want = ix.decode(dev16(qt)).cpu()
        qh2 = torch.from_numpy(qt.view(np.int16).copy()).pin_memory()
        oh2 = torch.full((1, 1, 4, 128), float("nan"), dtype=torch.float32).pin_memory()
        wi.wi_decode_step_host(ix.handle, qh2, oh2)
        assert torch.equal(oh2, want)
        oh3 = torch.full((1, 1, 4, 128), float("nan"), dtype=torch.float32)
        wi.wi_decode_step_host(ix.handle, torch.from_numpy(qt.view(np.int16).copy()), oh3)
        assert torch.equal(oh3, want)
    ix.free()


def test_graph_replay_matches_direct(wi):
    w = small(n_ctx=4096, seg_len=1024, clusters_per_seg=64, iters=2, n_q_heads=4, budget_k=6, seed=61)
    k, v, q, K, V, Q = gen(w)
    cfg = wi.config_from_workload(w)
    ix = wi.WaveIndex.build(cfg, dev16(k), dev16(v))
    qbuf = dev16(q)
    out = torch.empty((1, 1, 4, 128), dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ix.decode(qbuf, out=out, stream=s)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        ix.decode(qbuf, out=out, stream=s)
    for t in range(3):
        qn = kvsynth.queries(w, step=t + 1)
        qbuf.copy_(dev16(qn))
        graph.replay()
        torch.cuda.synchronize()
        got = out.clone()
        direct = ix.decode(dev16(qn))
        torch.cuda.synchronize()
        assert torch.equal(got, direct)
    ix.free()



def test_single_kernel_launches_repeat_the_step(wi):
    """wi_decode_kernel (the benchmark's kernel-alone timing) launches one kernel of the step; run
    after a whole step, each kernel repeats its part, so the output is bit-identical."""
    w = small(n_ctx=8192, seg_len=2048, clusters_per_seg=128, iters=2, n_q_heads=8, n_kv_heads=2, budget_k=9,
              seed=62)
    k, v, q, K, V, Q = gen(w)
    ix = wi.WaveIndex.build(wi.config_from_workload(w), dev16(k), dev16(v))
    qd = dev16(q)
    with pytest.raises(wi.WiError):
        wi.wi_decode_kernel(ix.handle, 2, qd, torch.empty(1, device=DEV))  # no whole step yet
    ref = ix.decode(qd)
    torch.cuda.synchronize()
    for order in ([2], [1, 2], [0, 1, 2], [2, 2]):
        out = torch.full_like(ref, float("nan"))
        for kid in order:
            wi.wi_decode_kernel(ix.handle, kid, qd, out)
        torch.cuda.synchronize()
        ix.check()
        assert torch.equal(out, ref), order
    ix.free()


@pytest.mark.parametrize("rows", [32, 64])
@pytest.mark.parametrize("splits", [1, 5, 12])
def test_exact_split_counts(wi, monkeypatch, splits, rows):
    """The exact-attention rows cut into 1, 5 or 12 row-balanced splits per head (plus the steady
    CTA), streamed through 32- or 64-row stages, give the oracle's output; the layout query reports
    the split count in use."""
    w = small(batch=2, n_q_heads=8, n_kv_heads=2, n_ctx=4096, seg_len=1024, clusters_per_seg=64, iters=2,
              budget_k=12, seed=5)
    k, v, q, K, V, Q = gen(w)
    p = params_of(w)
    idx = oracle.build_index(K, V, p)
    monkeypatch.setenv("WI_D3_SPLITS", str(splits))
    monkeypatch.setenv("WI_D3_STAGE_ROWS", str(rows))
    ix = wi.WaveIndex.adopt(wi.config_from_workload(w), dev16(k), dev16(v), *index_arrays(idx))
    assert wi.wi_decode_layout(ix.handle)["exact_splits"] == splits
    for t in range(2):
        qb = kvsynth.queries(w, step=t)
        out = ix.decode(dev16(qb)).cpu().numpy()
        ix.check()
        Qt = oracle.bf16_from_bits(qb).reshape(w.units, w.group, 128)
        ref = oracle.decode(Qt, K, V, idx, p, w.group)
        err = rel_l2(out.reshape(w.units, w.group, 128).astype(np.float64), ref)
        assert err.max() <= OUT_REL_L2, (t, err.max())
    ix.free()


@pytest.mark.parametrize("est_first,pe", [(0, 3), (1, 3), (1, 1)])
def test_select_estimate_block_orders(wi, monkeypatch, est_first, pe):
    """The top-k / estimation launch with either role first in block order, and 1 or 3 estimation
    CTAs per unit, gives the oracle's output."""
    w = small(batch=2, n_q_heads=8, n_kv_heads=2, n_ctx=4096, seg_len=1024, clusters_per_seg=64, iters=2,
              budget_k=12, seed=6)
    k, v, q, K, V, Q = gen(w)
    p = params_of(w)
    idx = oracle.build_index(K, V, p)
    monkeypatch.setenv("WI_ESTIMATE_FIRST", str(est_first))
    monkeypatch.setenv("WI_ESTIMATE_CTAS_PER_UNIT", str(pe))
    ix = wi.WaveIndex.adopt(wi.config_from_workload(w), dev16(k), dev16(v), *index_arrays(idx))
    assert wi.wi_decode_layout(ix.handle)["estimate_ctas"] == pe
    for t in range(2):
        qb = kvsynth.queries(w, step=t)
        out = ix.decode(dev16(qb)).cpu().numpy()
        ix.check()
        Qt = oracle.bf16_from_bits(qb).reshape(w.units, w.group, 128)
        ref = oracle.decode(Qt, K, V, idx, p, w.group)
        err = rel_l2(out.reshape(w.units, w.group, 128).astype(np.float64), ref)
        assert err.max() <= OUT_REL_L2, (t, err.max())
    ix.free()


@pytest.mark.parametrize("pe", [1, 2])
def test_estimation_depth_does_not_change_results(wi, monkeypatch, pe):
    """Two or three value-sum tiles in flight per estimation CTA (four and two tiles per CTA here):
    the same bits out, and the oracle's output."""
    w = small(batch=1, n_q_heads=8, n_kv_heads=2, n_ctx=8192, seg_len=1024, clusters_per_seg=64, iters=2,
              budget_k=12, seed=7)
    k, v, q, K, V, Q = gen(w)
    p = params_of(w)
    idx = oracle.build_index(K, V, p)
    monkeypatch.setenv("WI_ESTIMATE_CTAS_PER_UNIT", str(pe))
    outs = []
    for depth in (2, 3):
        monkeypatch.setenv("WI_ESTIMATE_DEPTH", str(depth))
        ix = wi.WaveIndex.adopt(wi.config_from_workload(w), dev16(k), dev16(v), *index_arrays(idx))
        outs.append([ix.decode(dev16(kvsynth.queries(w, step=t))).clone() for t in range(2)])
        torch.cuda.synchronize()
        ix.check()
        ix.free()
    for t in range(2):
        assert torch.equal(outs[0][t], outs[1][t]), t
        Qt = oracle.bf16_from_bits(kvsynth.queries(w, step=t)).reshape(w.units, w.group, 128)
        ref = oracle.decode(Qt, K, V, idx, p, w.group)
        err = rel_l2(outs[0][t].cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64), ref)
        assert err.max() <= OUT_REL_L2, (t, err.max())


def _bf16_valsum_index(idx):
    """The bf16 value-sum variant's definition: the stored fp32 value sums rounded to bf16."""
    return [{**d, "valsum": oracle.bf16_round(oracle.fp32_round(d["valsum"]))} for d in idx]


@pytest.mark.parametrize("g", [4, 7])
def test_valsum_bf16_variant_imported_index(wi, g):
    w = small(n_ctx=8192, seg_len=1024, clusters_per_seg=64, iters=2, n_q_heads=2 * g, n_kv_heads=2, budget_k=8,
              seed=21)
    k, v, q, K, V, Q = gen(w)
    p = params_of(w)
    idx = oracle.build_index(K, V, p)
    cfg = wi.config_from_workload(w)
    cfg.valsum_bf16 = 1
    ix = wi.WaveIndex.adopt(cfg, dev16(k), dev16(v), *index_arrays(idx))
    for t in range(2):
        qb = kvsynth.queries(w, step=t)
        out = ix.decode(dev16(qb)).cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64)
        ix.check()
        Qt = oracle.bf16_from_bits(qb).reshape(w.units, w.group, 128)
        ref = oracle.decode(Qt, K, V, _bf16_valsum_index(idx), p, w.group)
        err = rel_l2(out, ref)
        assert err.max() <= OUT_REL_L2, (t, err.max())
    ix.free()


@pytest.mark.parametrize("g", [4, 7])
def test_group_topk_with_bf16_value_sums(wi, g):
    """Both variants at once: group-shared retrieval over an index whose value sums are read as
    bf16, with appended tokens; parity with the oracle's group variant on the bf16-rounded sums."""
    w = small(n_ctx=8192, seg_len=1024, clusters_per_seg=64, iters=2, n_q_heads=2 * g, n_kv_heads=2, budget_k=8,
              seed=23)
    k, v, q, K, V, Q = gen(w)
    p = params_of(w)
    idx = oracle.build_index(K, V, p)
    T = 2
    cfg = wi.config_from_workload(w, max_append=T)
    cfg.valsum_bf16 = 1
    cfg.group_topk = 1
    ix = wi.WaveIndex.adopt(cfg, dev16(k), dev16(v), *index_arrays(idx))
    ka, va = kvsynth.kv_cache(w, p0=w.n_ctx, p1=w.n_ctx + T)
    KA = oracle.bf16_from_bits(ka).reshape(w.units, T, 128)
    VA = oracle.bf16_from_bits(va).reshape(w.units, T, 128)
    for t in range(T):
        qb = kvsynth.queries(w, step=t)
        out = ix.decode(dev16(qb), dev16(ka[:, :, :, t]), dev16(va[:, :, :, t]))
        out = out.cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64)
        ix.check()
        Qt = oracle.bf16_from_bits(qb).reshape(w.units, w.group, 128)
        ref = oracle.decode(Qt, K, V, _bf16_valsum_index(idx), p, w.group, k_app=KA[:, :t], v_app=VA[:, :t],
                            group_topk=True)
        err = rel_l2(out, ref)
        assert err.max() <= OUT_REL_L2, (t, err.max())
    ix.free()


def test_valsum_bf16_with_64_row_stages(wi, monkeypatch):
    """The bf16 value-sum instance of the exact kernel with 64-row stages (the layout of launches
    in several waves), forced on a small index: parity with the oracle."""
    w = small(n_ctx=8192, seg_len=1024, clusters_per_seg=64, iters=2, n_q_heads=8, n_kv_heads=2, budget_k=8,
              seed=25)
    k, v, q, K, V, Q = gen(w)
    p = params_of(w)
    idx = oracle.build_index(K, V, p)
    monkeypatch.setenv("WI_D3_STAGE_ROWS", "64")
    cfg = wi.config_from_workload(w)
    cfg.valsum_bf16 = 1
    ix = wi.WaveIndex.adopt(cfg, dev16(k), dev16(v), *index_arrays(idx))
    qb = kvsynth.queries(w, step=0)
    out = ix.decode(dev16(qb)).cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64)
    ix.check()
    Qt = oracle.bf16_from_bits(qb).reshape(w.units, w.group, 128)
    ref = oracle.decode(Qt, K, V, _bf16_valsum_index(idx), p, w.group)
    assert rel_l2(out, ref).max() <= OUT_REL_L2
    ix.free()


def test_valsum_bf16_variant_built_index(wi):
    """The library's own build with the variant: the decode matches the oracle on the exported
    index with its value sums rounded to bf16."""
    w = small(batch=2, n_q_heads=8, n_kv_heads=2, n_ctx=4096, seg_len=1024, clusters_per_seg=64, iters=3,
              budget_k=8, seed=23)
    k, v, q, K, V, Q = gen(w)
    p = params_of(w)
    cfg = wi.config_from_workload(w)
    cfg.valsum_bf16 = 1
    kt, vt = dev16(k), dev16(v)
    ix = wi.WaveIndex.build(cfg, kt, vt)
    exp = {n: t.cpu().numpy() for n, t in ix.export().items()}
    out = ix.decode(dev16(q)).cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64)
    ix.check()
    from helpers import assignment_from_index
    idx = [{"counts": exp["counts"][u].astype(np.int64),
            "mu": oracle.bf16_from_bits(exp["mu"][u].view(np.uint16)).reshape(w.clusters, 128),
            "valsum": exp["valsum"][u].astype(np.float64),
            "assignment": assignment_from_index(exp["counts"][u], exp["perm"][u], w.n_ctx, p.n_sink)}
           for u in range(w.units)]
    ref = oracle.decode(Q, K, V, _bf16_valsum_index(idx), p, w.group)
    assert rel_l2(out, ref).max() <= OUT_REL_L2
    # information: how far the variant moves the output from the fp32 value sums' definition
    print(f"bf16 value sums vs fp32, relative L2 max {rel_l2(out, oracle.decode(Q, K, V, idx, p, w.group)).max():.2e}")
    ix.free()


@pytest.mark.parametrize("g", [2, 4, 7, 8])
def test_group_topk_variant(wi, g):
    """Group-shared retrieval: every query head of a kv head takes the top-k of the heads' summed
    scores (the same ids for all of them), with its own logits, estimate and retrieved-term
    weights; parity with the oracle's variant over three steps with appended tokens."""
    w = small(batch=2, n_q_heads=2 * g, n_kv_heads=2, n_ctx=8192, seg_len=1024, clusters_per_seg=64, iters=2,
              budget_k=8, seed=29)
    k, v, q, K, V, Q = gen(w)
    p = params_of(w)
    idx = oracle.build_index(K, V, p)
    T = 3
    cfg = wi.config_from_workload(w, max_append=T)
    cfg.group_topk = 1
    ix = wi.WaveIndex.adopt(cfg, dev16(k), dev16(v), *index_arrays(idx))
    ka, va = kvsynth.kv_cache(w, p0=w.n_ctx, p1=w.n_ctx + T)
    KA = oracle.bf16_from_bits(ka).reshape(w.units, T, 128)
    VA = oracle.bf16_from_bits(va).reshape(w.units, T, 128)
    kk = oracle.budget_k(w.clusters, p)
    for t in range(T):
        qb = kvsynth.queries(w, step=t)
        out = ix.decode(dev16(qb), dev16(ka[:, :, :, t]), dev16(va[:, :, :, t]))
        ids, cnt = ix.selection()
        torch.cuda.synchronize()
        ix.check()
        Qt = oracle.bf16_from_bits(qb).reshape(w.units, w.group, 128)
        ref = oracle.decode(Qt, K, V, idx, p, w.group, k_app=KA[:, :t], v_app=VA[:, :t], group_topk=True)
        got = out.cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64)
        assert rel_l2(got, ref).max() <= OUT_REL_L2, t
        ids, cnt = ids.cpu().numpy(), cnt.cpu().numpy()
        for u in range(w.units):
            summed = idx[u]["mu"] @ Qt[u].sum(axis=0)
            for h in range(w.group):
                np.testing.assert_array_equal(ids[u, h], ids[u, 0])
                check_topk(ids[u, h], cnt[u, h], summed, idx[u]["counts"] > 0, kk)
    ix.free()
