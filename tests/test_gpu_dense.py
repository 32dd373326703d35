"""The dense comparator (full attention over every cached and appended token) against the
float64 oracle's full attention, on the same input bytes: small cases with several group
sizes and units, appended tokens, and the Llama-3-8B-shaped 131K workload (library-built
index, every unit checked)."""
import numpy as np
import pytest
import torch

import kvsynth
import oracle
from helpers import OUT_REL_L2, gen, index_arrays, params_of, rel_l2, small

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def wi():
    import clustered_sparse_kv_gb300 as m
    return m


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV)


def check(w, got, Q, K, V, KA=None, VA=None):
    ref = oracle.full_attention(Q, K, V, KA, VA)
    got = got.cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64)
    err = rel_l2(got, ref)
    assert err.max() <= OUT_REL_L2, err.max()
    return err.max()


@pytest.mark.parametrize("g,kv", [(1, 1), (2, 2), (3, 1), (4, 2), (5, 1), (6, 2), (7, 1), (8, 1)])
def test_dense_parity_group_sizes(wi, g, kv):
    w = small(n_ctx=4096, seg_len=1024, clusters_per_seg=64, iters=2, n_q_heads=g * kv, n_kv_heads=kv,
              budget_k=6, seed=3 + g)
    k, v, q, K, V, Q = gen(w)
    idx = oracle.build_index(K, V, params_of(w))
    ix = wi.WaveIndex.adopt(wi.config_from_workload(w), dev16(k), dev16(v), *index_arrays(idx))
    out = ix.dense_decode(dev16(q))
    torch.cuda.synchronize()
    ix.check()
    assert check(w, out, Q, K, V) < 1e-5
    ix.free()


def test_dense_includes_appended_tokens(wi):
    w = small(batch=2, n_q_heads=8, n_kv_heads=2, n_ctx=2048, seg_len=512, clusters_per_seg=32, iters=2,
              budget_k=5, seed=9)
    T = 70  # more than one 64-row stage of appended rows
    k, v, q, K, V, Q = gen(w)
    idx = oracle.build_index(K, V, params_of(w))
    ix = wi.WaveIndex.adopt(wi.config_from_workload(w, max_append=T), dev16(k), dev16(v), *index_arrays(idx))
    ka, va = kvsynth.kv_cache(w, p0=w.n_ctx, p1=w.n_ctx + T)
    KA = oracle.bf16_from_bits(ka).reshape(w.units, T, 128)
    VA = oracle.bf16_from_bits(va).reshape(w.units, T, 128)
    for t in range(T):
        qb = dev16(kvsynth.queries(w, step=t))
        ix.decode(qb, dev16(ka[:, :, :, t]), dev16(va[:, :, :, t]))
        if t in (0, 63, T - 1):
            out = ix.dense_decode(qb)  # t + 1 tokens appended now
            torch.cuda.synchronize()
            ix.check()
            Qt = oracle.bf16_from_bits(kvsynth.queries(w, step=t)).reshape(w.units, w.group, 128)
            check(w, out, Qt, K, V, KA[:, :t + 1], VA[:, :t + 1])
    ix.free()


def test_dense_fullsize_131k(wi):
    """Every unit of the 131K workload; the index is the library's own build (the context rows are
    read in its permuted order, which attention does not depend on)."""
    w = kvsynth.get_workload("llama3-8b-131k")
    k, v = kvsynth.kv_cache(w)
    q = kvsynth.queries(w, step=0)
    kt, vt = dev16(k), dev16(v)
    ix = wi.WaveIndex.build(wi.config_from_workload(w), kt, vt)
    out = ix.dense_decode(dev16(q))
    wave = ix.decode(dev16(q))
    torch.cuda.synchronize()
    ix.check()
    K = oracle.bf16_from_bits(k).reshape(w.units, w.n_ctx, 128)
    V = oracle.bf16_from_bits(v).reshape(w.units, w.n_ctx, 128)
    Q = oracle.bf16_from_bits(q).reshape(w.units, w.group, 128)
    check(w, out, Q, K, V)
    # information only (approximation quality is not pinned): the wave index against full attention
    approx = rel_l2(wave.cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64),
                    out.cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64))
    print(f"wave index vs full attention, relative L2: max {approx.max():.3e} mean {approx.mean():.3e}")
    ix.free()
