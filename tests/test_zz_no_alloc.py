"""wi_kmeans_step_noalloc: the clustering round for callers that may not
allocate device memory (a serving process whose KV-cache pool holds nearly
all GPU memory, or a host that allows device memory only through its own
arena).  Its scratch is a fixed device array inside the library, so it must
give exactly what the allocating wi_kmeans_step gives, call after call, and
refuse problems larger than that array.

This file is collected last on purpose: a run that stops at the first
failure has run every other test before it."""
import ctypes

import numpy as np
import pytest

import kvsynth
import oracle


@pytest.fixture(scope="module")
def wi():
    import clustered_sparse_kv_gb300 as m
    return m


def workload():
    return kvsynth.get_workload("tiny-8k").with_(batch=2, n_q_heads=4, n_kv_heads=2, n_ctx=4096, seg_len=1024,
                                                 clusters_per_seg=64, iters=2, budget_k=4, seed=91)


def test_rejects_problem_beyond_the_fixed_scratch(wi):
    w = kvsynth.get_workload("llama3-8b-131k").with_(batch=4)   # 4M tokens: far beyond 8 MiB of scratch
    cfg = wi.config_from_workload(w)
    rc = wi.lib.wi_kmeans_step_noalloc(ctypes.byref(cfg), 16, 16, 16, 16, None)
    assert rc == wi.WI_EINVAL
    assert "scratch" in wi.lib.wi_last_error().decode()


@pytest.mark.gpu
def test_noalloc_round_matches_allocating_round(wi):
    import torch

    dev = "cuda:0"
    w = workload()
    k, _ = kvsynth.kv_cache(w)
    K = oracle.bf16_from_bits(k).reshape(w.units, w.n_ctx, 128)
    p = oracle.IndexParams(seg_len=w.seg_len, clusters_per_seg=w.clusters_per_seg)
    c0 = np.stack([np.stack([oracle.init_centroids(K[u][s * w.seg_len:(s + 1) * w.seg_len], p)
                             for s in range(w.n_segments)]) for u in range(w.units)])
    kt = torch.from_numpy(k.view(np.int16)).to(dev)
    cur = torch.from_numpy(oracle.bf16_to_bits(c0).view(np.int16)).to(dev)
    cfg = wi.config_from_workload(w)
    for call in range(2):
        a_ref = torch.empty((w.units, w.n_ctx), dtype=torch.int32, device=dev)
        c_ref = torch.empty_like(cur)
        wi.wi_kmeans_step(cfg, kt, cur, a_ref, c_ref)
        a_na = torch.full((w.units, w.n_ctx), -7, dtype=torch.int32, device=dev)
        c_na = torch.zeros_like(cur)
        wi.wi_kmeans_step_noalloc(cfg, kt, cur, a_na, c_na)
        torch.cuda.synchronize()
        # integer assignment: bit-exact; centroids: the same kernels in the same order, so bit-exact too
        assert torch.equal(a_na, a_ref), call
        assert torch.equal(c_na, c_ref), call
        assert int((a_na >= 0).sum()) == w.units * (w.n_ctx - w.n_sink - w.local_window)
        cur = c_na.clone()
