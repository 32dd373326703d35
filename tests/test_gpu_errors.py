"""Error paths on the GPU without faulting it: a device allocation refused partway through
making an index (the WI_FAIL_ALLOC_AT hook) is reported as WI_ENOMEM with everything already
allocated released, and the next index is made and decodes normally; the kernels' bounded wait,
run on a barrier nothing completes, gives up, records its error bit and leaves the context usable."""
import ctypes

import numpy as np
import pytest
import torch

import kvsynth
import oracle
from helpers import OUT_REL_L2, gen, index_arrays, params_of, rel_l2, small

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wi():
    import clustered_sparse_kv_gb300 as m
    return m


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to("cuda:0")


@pytest.mark.parametrize("n", [1, 7, 20])
def test_refused_allocation_is_reported_and_released(wi, monkeypatch, n):
    w = small(n_ctx=2048, seg_len=512, clusters_per_seg=32, iters=2, n_q_heads=4, budget_k=4, seed=51)
    k, v, q, K, V, Q = gen(w)
    kt, vt = dev16(k), dev16(v)
    cfg = wi.config_from_workload(w)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    monkeypatch.setenv("WI_FAIL_ALLOC_AT", str(n))
    out = ctypes.c_void_p(123)
    rc = wi.lib.wi_build_index(ctypes.byref(cfg), ctypes.c_void_p(kt.data_ptr()), ctypes.c_void_p(vt.data_ptr()),
                               None, None, ctypes.byref(out))
    assert rc == wi.WI_ENOMEM and out.value is None
    assert "WI_FAIL_ALLOC_AT" in wi.lib.wi_last_error().decode()
    monkeypatch.delenv("WI_FAIL_ALLOC_AT")
    torch.cuda.synchronize()
    assert abs(torch.cuda.mem_get_info()[0] - free0) < (64 << 20)  # nothing kept
    # the next index works: the oracle's index imported, one decode step at parity
    p = params_of(w)
    idx = oracle.build_index(K, V, p)
    ix = wi.WaveIndex.adopt(cfg, kt, vt, *index_arrays(idx))
    got = ix.decode(dev16(q)).cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64)
    ix.check()
    assert rel_l2(got, oracle.decode(Q, K, V, idx, p, w.group)).max() <= OUT_REL_L2
    ix.free()


def test_bounded_wait_gives_up_and_the_context_stays_usable(wi):
    r = wi.wi_selftest_wait_timeout()    # about one second: the wait's cycle bound
    assert r["wait_returned"] == 1         # returned without the barrier completing
    assert r["device_error"] == 16         # the timeout bit, nothing else
    w = small(n_ctx=2048, seg_len=512, clusters_per_seg=32, iters=2, n_q_heads=4, budget_k=4, seed=52)
    k, v, q, K, V, Q = gen(w)
    p = params_of(w)
    idx = oracle.build_index(K, V, p)
    ix = wi.WaveIndex.adopt(wi.config_from_workload(w), dev16(k), dev16(v), *index_arrays(idx))
    got = ix.decode(dev16(q)).cpu().numpy().reshape(w.units, w.group, 128).astype(np.float64)
    ix.check()
    assert rel_l2(got, oracle.decode(Q, K, V, idx, p, w.group)).max() <= OUT_REL_L2
    ix.free()
