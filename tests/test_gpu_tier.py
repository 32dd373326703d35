"""The host memory tier (wave buffer) on the GPU.

Two indexes are made from the same oracle index and the same input bytes; one gets the tier.  The
tiered one must give the untiered one's outputs bit for bit at every step (where a row is read from
-- a cached page or host memory -- cannot change the stages the attention kernel sees), with the
caller's K/V overwritten after attach (so they are provably not read).  With rounds run on request,
the device's page table after every round must equal the oracle's LRU rounds fed the pages the step
read, and the pages stamped must be exactly the pages of the retrieved clusters' rows.
"""
import numpy as np
import pytest
import torch

import kvsynth
import oracle
from helpers import OUT_REL_L2, gen, index_arrays, params_of, rel_l2, small

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
PAGE = 16
NAN16 = 0x7FC0  # a bf16 NaN: any read of the overwritten caller K/V would poison the output


@pytest.fixture(scope="module")
def wi():
    import clustered_sparse_kv_gb300 as m
    return m


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV)


def workload(seed, max_append=0, **kw):
    base = dict(batch=1, n_q_heads=8, n_kv_heads=2, n_ctx=8192, seg_len=1024, clusters_per_seg=64, iters=2,
                budget_k=24, seed=seed)
    base.update(kw)
    return small(**base)


def pair(wi, w, max_append=0):
    """Two indexes adopted from the oracle's index on copies of the same bytes."""
    k, v, q, K, V, Q = gen(w)
    idx = oracle.build_index(K, V, params_of(w))
    cfg = wi.config_from_workload(w, max_append=max_append)
    a = wi.WaveIndex.adopt(cfg, dev16(k), dev16(v), *index_arrays(idx))
    b = wi.WaveIndex.adopt(cfg, dev16(k), dev16(v), *index_arrays(idx))
    return a, b, idx, K, V


def selected_pages(wi, ix, exp, units):
    """Per unit: the pages of the rows of every cluster some head retrieved in the last step, and
    the retrieved rows summed over heads."""
    ids, cnt = ix.selection()
    ids, cnt = ids.cpu().numpy(), cnt.cpu().numpy()
    out, rows = [], 0
    for u in range(units):
        pages = set()
        for h in range(ids.shape[1]):
            for j in ids[u, h, :cnt[u, h]]:
                r0, n = int(exp["offsets"][u][j]), int(exp["counts"][u][j])
                pages.update(oracle.pages_of_rows(r0, n, PAGE))
                rows += n
        out.append(sorted(pages))
    return out, rows


@pytest.mark.parametrize("slots_frac,admit", [(0.25, 64), (1.0, 1000), (0.0, 8), (0.05, 4)])
def test_tier_rounds_match_oracle_and_outputs_are_unchanged(wi, slots_frac, admit):
    w = workload(41)
    a, b, idx, K, V = pair(wi, w)
    exp = {n: t.cpu().numpy() for n, t in a.export().items()}
    pages = w.n_ctx // PAGE
    slots = int(slots_frac * pages)
    b.attach_tier(slots, admit, async_rounds=False)
    b.k.fill_(NAN16)
    b.v.fill_(NAN16)
    refs = [oracle.LruPagePolicy(pages, slots, admit) for _ in range(w.units)]
    rows_sel = 0
    hits = misses = 0
    for t in range(12):
        qb = kvsynth.queries(w, step=t // 3)   # each query three times: pages recur
        qd = dev16(qb)
        oa = a.decode(qd).clone()
        ob = b.decode(qd).clone()
        torch.cuda.synchronize()
        assert torch.equal(oa, ob), t
        sel, nrows = selected_pages(wi, a, exp, w.units)
        rows_sel += nrows
        b.tier_round()
        slot_of, use = (x.numpy() for x in b.tier_tables())
        for u in range(w.units):
            touched = np.nonzero(use[u] == t)[0].tolist()
            assert touched == sel[u], (t, u)
            hits += sum(p in refs[u].slot_of for p in touched)
            misses += sum(p not in refs[u].slot_of for p in touched)
            refs[u].round(touched, t)
            want = np.full(pages, -1, np.int32)
            for p, s in refs[u].slot_of.items():
                want[p] = s
            np.testing.assert_array_equal(slot_of[u], want)
        if t == 0:  # the parity proper: the tiered output against the oracle
            Qt = oracle.bf16_from_bits(qb).reshape(w.units, w.group, 128)
            ref = oracle.decode(Qt, K, V, idx, params_of(w), w.group)
            err = rel_l2(ob.cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64), ref)
            assert err.max() <= OUT_REL_L2
    st = b.tier_stats()
    assert st["rounds"] == 12
    assert st["page_hits"] == hits and st["page_misses"] == misses
    assert st["pages_read"] == hits + misses
    assert st["rows_from_cache"] + st["rows_from_host"] == rows_sel
    if slots == 0:
        assert st["rows_from_cache"] == 0 and st["admitted"] == 0
    if slots_frac == 1.0:
        assert st["evicted"] == 0 and st["rows_from_cache"] > 0
    a.check()
    b.check()
    a.free()
    b.free()


def test_tier_async_rounds_and_appends(wi):
    """Rounds on the library's thread while steps run, with tokens appended every step: outputs
    equal the untiered index's bit for bit; the page table stays a valid partial map."""
    T = 40
    w = workload(42)
    a, b, idx, K, V = pair(wi, w, max_append=T)
    pages = w.n_ctx // PAGE
    b.attach_tier(pages // 8, 32, async_rounds=True)
    b.k.fill_(NAN16)
    b.v.fill_(NAN16)
    ka, va = kvsynth.kv_cache(w, p0=w.n_ctx, p1=w.n_ctx + T)
    for t in range(T):
        qd = dev16(kvsynth.queries(w, step=t // 4))
        kn, vn = dev16(ka[:, :, :, t]), dev16(va[:, :, :, t])
        oa = a.decode(qd, kn, vn).clone()
        ob = b.decode(qd, kn, vn).clone()
        torch.cuda.synchronize()   # the thread gets its rounds in between
        assert torch.equal(oa, ob), t
    st = b.tier_stats()
    assert st["rounds"] >= 1 and st["admitted"] > 0
    assert st["page_hits"] + st["page_misses"] == st["pages_read"]
    assert st["evicted"] <= st["admitted"]
    # a round on request while the thread runs them too: it waits for the thread's round, then runs
    b.tier_round()
    assert b.tier_stats()["rounds"] == st["rounds"] + 1
    ob = b.decode(dev16(kvsynth.queries(w, step=T)))
    oa = a.decode(dev16(kvsynth.queries(w, step=T)))
    torch.cuda.synchronize()
    assert torch.equal(oa, ob)
    slot_of, use = (x.numpy() for x in b.tier_tables())
    for u in range(w.units):
        used = slot_of[u][slot_of[u] >= 0]
        assert len(used) == len(set(used.tolist())) <= pages // 8
        assert np.all(use[u][slot_of[u] >= 0] >= 0)   # only pages some step read are cached
    a.check()
    b.check()
    a.free()
    b.free()


def test_tier_refusals(wi):
    w = workload(43)
    a, b, idx, K, V = pair(wi, w)
    pages = w.n_ctx // PAGE
    with pytest.raises(wi.WiError) as e:
        b.attach_tier(pages + 1, 4)
    assert e.value.code == wi.WI_EINVAL
    b.attach_tier(16, 4, async_rounds=False)
    with pytest.raises(wi.WiError) as e:
        b.attach_tier(16, 4)
    assert e.value.code == wi.WI_EINVAL
    q = dev16(kvsynth.queries(w, step=0))
    with pytest.raises(wi.WiError) as e:
        b.dense_decode(q)
    assert e.value.code == wi.WI_EUNSUPPORTED
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with pytest.raises(wi.WiError) as e:
            with torch.cuda.graph(g, stream=s):
                b.decode(q, stream=s)
    assert e.value.code == wi.WI_EUNSUPPORTED
    a.free()
    b.free()
    # an index that grows, and the bf16 value-sum variant, are refused
    wg = workload(44, seg_len=512, clusters_per_seg=32)
    k, v, q, K, V, Q = gen(wg)
    ig = oracle.build_index(K, V, params_of(wg))
    grow = wi.WaveIndex.adopt(wi.config_from_workload(wg, max_append=600), dev16(k), dev16(v), *index_arrays(ig))
    with pytest.raises(wi.WiError) as e:
        grow.attach_tier(8, 4)
    assert e.value.code == wi.WI_EUNSUPPORTED
    grow.free()
    cfg = wi.config_from_workload(wg)
    cfg.valsum_bf16 = 1
    vb = wi.WaveIndex.adopt(cfg, dev16(k), dev16(v), *index_arrays(ig))
    with pytest.raises(wi.WiError) as e:
        vb.attach_tier(8, 4)
    assert e.value.code == wi.WI_EUNSUPPORTED
    vb.free()


def test_tier_allocation_failure_leaves_the_index_usable(wi, monkeypatch):
    """Every allocation of the tier refused in turn: attach reports WI_ENOMEM, the index decodes as
    before (untiered, from the caller's K/V), and a later attach succeeds."""
    w = workload(45)
    a, b, idx, K, V = pair(wi, w)
    q = dev16(kvsynth.queries(w, step=0))
    ref = a.decode(q).clone()
    for n in range(1, 15):   # nine device allocations, five page-locked host ones
        monkeypatch.setenv("WI_FAIL_TIER_ALLOC_AT", str(n))
        with pytest.raises(wi.WiError) as e:
            b.attach_tier(32, 16)
        assert e.value.code == wi.WI_ENOMEM, n
        assert "WI_FAIL_TIER_ALLOC_AT" in str(e.value)
        assert torch.equal(b.decode(q), ref), n
    monkeypatch.setenv("WI_FAIL_TIER_ALLOC_AT", "15")   # past the last allocation: nothing refused
    b.attach_tier(32, 16, async_rounds=False)
    monkeypatch.delenv("WI_FAIL_TIER_ALLOC_AT")
    b.k.fill_(NAN16)
    b.v.fill_(NAN16)
    assert torch.equal(b.decode(q), ref)
    b.check()
    a.free()
    b.free()


def test_tier_with_64_row_stages(wi, monkeypatch):
    """The tier instance of the exact kernel with 64-row stages (the layout of launches in several
    waves), forced: the same bits as the untiered index with the same stages, every step."""
    monkeypatch.setenv("WI_D3_STAGE_ROWS", "64")
    w = workload(47)
    a, b, idx, K, V = pair(wi, w)
    pages = w.n_ctx // PAGE
    b.attach_tier(pages // 4, 64, async_rounds=False)
    b.k.fill_(NAN16)
    b.v.fill_(NAN16)
    for t in range(6):
        qd = dev16(kvsynth.queries(w, step=t // 2))
        oa = a.decode(qd).clone()
        ob = b.decode(qd).clone()
        torch.cuda.synchronize()
        assert torch.equal(oa, ob), t
        b.tier_round()
    st = b.tier_stats()
    assert st["rows_from_cache"] > 0 and st["rows_from_host"] > 0
    a.check()
    b.check()
    a.free()
    b.free()


@pytest.mark.parametrize("group_topk", [0, 1])
def test_tier_host_buffers_and_group_retrieval(wi, group_topk):
    """The host-buffer entry point (query and output in page-locked host memory) and group-shared
    retrieval through the tier: the same bits as the untiered index."""
    w = workload(46)
    k, v, q, K, V, Q = gen(w)
    idx = oracle.build_index(K, V, params_of(w))
    cfg = wi.config_from_workload(w)
    cfg.group_topk = group_topk
    a = wi.WaveIndex.adopt(cfg, dev16(k), dev16(v), *index_arrays(idx))
    b = wi.WaveIndex.adopt(cfg, dev16(k), dev16(v), *index_arrays(idx))
    b.attach_tier(w.n_ctx // PAGE // 4, 64, async_rounds=True)
    b.k.fill_(NAN16)
    b.v.fill_(NAN16)
    oh_a = torch.empty((w.batch, w.layers, w.n_q_heads, 128), dtype=torch.float32).pin_memory()
    oh_b = torch.empty_like(oh_a).pin_memory()
    for t in range(6):
        qh = torch.from_numpy(kvsynth.queries(w, step=t // 2).view(np.int16)).pin_memory()
        wi.wi_decode_step_host(a.handle, qh, oh_a)
        wi.wi_decode_step_host(b.handle, qh, oh_b)
        assert torch.equal(oh_a, oh_b), t
    st = b.tier_stats()
    assert st["rows_from_cache"] + st["rows_from_host"] > 0
    a.check()
    b.check()
    a.free()
    b.free()
