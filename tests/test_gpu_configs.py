"""Full-size decode parity for the batch-16 workload (Llama-3-8B shape, 122880
tokens, 128 units), the grouped-query append workload (Qwen2.5-7B shape,
batch 8, 262144 tokens, 7 query heads per kv head, 64 decode steps that each
append a token) and one kv head of the million-token workload (C = 65536
clusters, k = 1180: the top-k without a shared-memory key cache and above its
list capacity), in the launch configuration of the default build.

The oracle cannot cluster these sizes, so the library builds its own index
(ten rounds); the index is checked by its invariants, and the oracle decodes
sampled (unit, step) pairs with the exported index (same counts, members,
mean keys and value sums), which pins every decode step (scores, top-k,
estimation, exact attention, merge, append) at full size."""
import numpy as np
import pytest
import torch

import kvsynth
import oracle
from helpers import OUT_REL_L2, assignment_from_index, check_topk, params_of, rel_l2
from test_gpu_build import dev16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wi():
    import clustered_sparse_kv_gb300 as m
    return m


def build_and_export(wi, w):
    k, v = kvsynth.kv_cache(w)
    cfg = wi.config_from_workload(w)
    kt, vt = dev16(k), dev16(v)
    ix = wi.WaveIndex.build(cfg, kt, vt)
    exp = {name: t.cpu().numpy() for name, t in ix.export().items()}
    torch.cuda.synchronize()
    ix.check()
    return k, v, kt, vt, ix, exp


def check_invariants(w, k, kt, exp, units):
    p = params_of(w)
    I = oracle.indexed_positions(w.n_ctx, p)
    kp = kt.reshape(w.units, w.n_ctx, 128)
    kf = k.reshape(w.units, w.n_ctx, 128)
    for u in units:
        counts, perm = exp["counts"][u], exp["perm"][u]
        assert counts.sum() == I.size
        np.testing.assert_array_equal(np.sort(perm), I)
        owner = np.repeat(np.arange(w.clusters), counts) // w.clusters_per_seg
        assert np.all(perm // w.seg_len == owner)  # every cluster inside its segment
        rows = kp[u, w.n_sink:w.n_ctx - w.local_window].cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(rows, kf[u][perm])  # the permuted rows are the members' keys
        np.testing.assert_array_equal(exp["offsets"][u][:-1], w.n_sink + np.concatenate([[0], np.cumsum(counts)[:-1]]))


def oracle_index(w, exp, u):
    p = params_of(w)
    return {
        "counts": exp["counts"][u].astype(np.int64),
        "mu": oracle.bf16_from_bits(exp["mu"][u].view(np.uint16)).reshape(w.clusters, 128),
        "valsum": exp["valsum"][u].astype(np.float64),
        "assignment": assignment_from_index(exp["counts"][u], exp["perm"][u], w.n_ctx, p.n_sink),
    }


def check_step(w, u_list, k, v, exp, qb, got, ids, cnt, k_app=None, v_app=None):
    p = params_of(w)
    kk = oracle.budget_k(w.clusters, p)
    Q = oracle.bf16_from_bits(qb).reshape(w.units, w.group, 128)
    kf = k.reshape(w.units, w.n_ctx, 128)
    vf = v.reshape(w.units, w.n_ctx, 128)
    for u in u_list:
        idx = oracle_index(w, exp, u)
        K = oracle.bf16_from_bits(kf[u]).reshape(w.n_ctx, 128)
        V = oracle.bf16_from_bits(vf[u]).reshape(w.n_ctx, 128)
        ka = None if k_app is None else k_app[u]
        va = None if v_app is None else v_app[u]
        ref, info = oracle.decode_unit(Q[u], K, V, idx, p, ka, va, details=True)
        err = rel_l2(got[u], ref)
        assert err.max() <= OUT_REL_L2, (u, err.max())
        ne = idx["counts"] > 0
        for h in range(w.group):
            check_topk(ids[u, h], cnt[u, h], info[h]["scores"], ne, kk)


def test_batch16_120k(wi):
    w = kvsynth.get_workload("llama3-8b-b16-120k")
    assert (w.units, w.clusters, oracle.budget_k(w.clusters, params_of(w))) == (128, 7680, 139)
    k, v, kt, vt, ix, exp = build_and_export(wi, w)
    sample = [0, 77, 127]
    check_invariants(w, k, kt, exp, sample)
    qb = kvsynth.queries(w, step=0)
    out = ix.decode(dev16(qb))
    ids, cnt = ix.selection()
    torch.cuda.synchronize()
    ix.check()
    got = out.cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64)
    assert np.isfinite(got).all()
    check_step(w, sample, k, v, exp, qb, got, ids.cpu().numpy(), cnt.cpu().numpy())
    ix.free()


def test_gqa7_262k_append_64_steps(wi):
    w = kvsynth.get_workload("qwen2.5-7b-b8-262k")
    assert (w.units, w.group, w.clusters, oracle.budget_k(w.clusters, params_of(w))) == (32, 7, 16384, 295)
    k, v, kt, vt, ix, exp = build_and_export(wi, w)
    sample = [0, 13, 31]
    check_invariants(w, k, kt, exp, sample)
    T = w.decode_steps
    ka, va = kvsynth.kv_cache(w, p0=w.n_ctx, p1=w.n_ctx + T)
    KA = oracle.bf16_from_bits(ka).reshape(w.units, T, 128)
    VA = oracle.bf16_from_bits(va).reshape(w.units, T, 128)
    checked = 0
    for t in range(T):
        qb = kvsynth.queries(w, step=t)
        out = ix.decode(dev16(qb), dev16(ka[:, :, :, t]), dev16(va[:, :, :, t]))
        if t in (0, 1, 31, T - 1):
            ids, cnt = ix.selection()
            torch.cuda.synchronize()
            ix.check()
            got = out.cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64)
            assert np.isfinite(got).all()
            check_step(w, sample, k, v, exp, qb, got, ids.cpu().numpy(), cnt.cpu().numpy(),
                       KA[:, :t], VA[:, :t])
            checked += 1
    torch.cuda.synchronize()
    ix.check()
    assert checked == 4
    ix.free()


def test_one_million_tokens_one_kv_head(wi):
    w = kvsynth.get_workload("llama3-8b-1m-32l").with_(layers=1, n_kv_heads=1, n_q_heads=4)
    assert (w.units, w.clusters, oracle.budget_k(w.clusters, params_of(w))) == (1, 65536, 1180)
    k, v, kt, vt, ix, exp = build_and_export(wi, w)
    check_invariants(w, k, kt, exp, [0])
    for step in range(2):
        qb = kvsynth.queries(w, step=step)
        out = ix.decode(dev16(qb))
        ids, cnt = ix.selection()
        torch.cuda.synchronize()
        ix.check()
        got = out.cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64)
        check_step(w, [0], k, v, exp, qb, got, ids.cpu().numpy(), cnt.cpu().numpy())
    ix.free()


def test_one_million_tokens_32_layers_full_size(wi):
    """The million-token, 32-layer workload at full size (256 units, 137 GB generated on the
    device), built by the library and decoded in the launch configuration the benchmark times;
    two sampled units (layer 0 kv head 0, layer 31 kv head 7) checked against the oracle given the
    exported index, on two steps.  The build permutes the cache in place, so the sampled units'
    original rows are kept aside first."""
    w = kvsynth.get_workload("llama3-8b-1m-32l")
    assert (w.units, w.clusters) == (256, 65536)
    gen = kvsynth.DeviceGen(w)
    kt, vt = gen.kv_cache()
    sample = [0, 255]
    k_orig = [kt.view(w.units, w.n_ctx, 128)[u].cpu().numpy().view(np.uint16) for u in sample]
    v_orig = [vt.view(w.units, w.n_ctx, 128)[u].cpu().numpy().view(np.uint16) for u in sample]
    ix = wi.WaveIndex.build(wi.config_from_workload(w), kt, vt)
    torch.cuda.synchronize()
    ix.check()
    layout = wi.wi_decode_layout(ix.handle)
    assert layout == {"score_ctas": 1, "estimate_ctas": 1, "exact_splits": 1}
    p = params_of(w)
    kk = oracle.budget_k(w.clusters, p)
    I = oracle.indexed_positions(w.n_ctx, p)
    # the sampled units' index, exported one array at a time (full-size device copies, then sliced)
    exp = {}
    for name, shape, dt in (("counts", (w.units, w.clusters), torch.int32),
                            ("perm", (w.units, w.n_ctx - w.n_sink - w.local_window), torch.int32),
                            ("mu", (w.units, w.clusters, 128), torch.int16),
                            ("valsum", (w.units, w.clusters, 128), torch.float32)):
        t = torch.empty(shape, dtype=dt, device="cuda")
        wi.wi_index_export(ix.handle, **{name: t})
        torch.cuda.synchronize()
        exp[name] = [t[u].cpu().numpy() for u in sample]
        del t
        torch.cuda.empty_cache()
    idx = []
    for i in range(len(sample)):
        counts, perm_u = exp["counts"][i], exp["perm"][i]
        assert counts.sum() == I.size
        np.testing.assert_array_equal(np.sort(perm_u), I)
        idx.append({"counts": counts.astype(np.int64), "valsum": exp["valsum"][i].astype(np.float64),
                    "mu": oracle.bf16_from_bits(exp["mu"][i].view(np.uint16)).reshape(w.clusters, 128),
                    "assignment": assignment_from_index(counts, perm_u, w.n_ctx, p.n_sink)})
    KV = [(oracle.bf16_from_bits(k_orig[i]), oracle.bf16_from_bits(v_orig[i])) for i in range(len(sample))]
    for step in range(2):
        qd = gen.queries(step)
        out = ix.decode(qd)
        ids, cnt = ix.selection()
        torch.cuda.synchronize()
        ix.check()
        got = out.cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64)
        assert np.isfinite(got).all()
        Q = oracle.bf16_from_bits(qd.cpu().numpy().view(np.uint16)).reshape(w.units, w.group, 128)
        ids, cnt = ids.cpu().numpy(), cnt.cpu().numpy()
        for i, u in enumerate(sample):
            ref, info = oracle.decode_unit(Q[u], KV[i][0], KV[i][1], idx[i], p, details=True)
            err = rel_l2(got[u], ref)
            assert err.max() <= OUT_REL_L2, (step, u, err.max())
            ne = idx[i]["counts"] > 0
            for h in range(w.group):
                check_topk(ids[u, h], cnt[u, h], info[h]["scores"], ne, kk)
    ix.free()
    del kt, vt
    torch.cuda.empty_cache()
