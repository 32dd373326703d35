"""The device generator (kvsynth_cuda.cu) against the host generator (kvsynth.c):
the same seeded draws, transforms and rounding, so the same bf16 bytes except
where the device's double log / sin / cos (within a couple of ulps of the
host's libm) move a value across a bf16 rounding boundary -- expected to
happen to almost no element, and then by one bf16 step."""
import numpy as np
import pytest
import torch

import kvsynth

pytestmark = pytest.mark.gpu


def compare(dev_bits, host_bits, max_frac=1e-6):
    a = dev_bits.cpu().numpy().view(np.uint16).astype(np.int64)
    b = np.asarray(host_bits).view(np.uint16).astype(np.int64)
    assert a.shape == b.shape
    diff = a != b
    n = int(diff.sum())
    assert n <= max(1, max_frac * a.size), f"{n} of {a.size} differ"
    if n:   # one bf16 step (same sign, adjacent bit patterns)
        assert np.all(np.abs(a[diff] - b[diff]) == 1)
    return n


def test_device_cache_and_queries_match_host_small():
    w = kvsynth.get_workload("tiny-8k").with_(batch=2, layers=2, n_q_heads=8, n_kv_heads=2, n_ctx=4096, seed=17)
    g = kvsynth.DeviceGen(w)
    kd, vd = g.kv_cache()
    kh, vh = kvsynth.kv_cache(w)
    torch.cuda.synchronize()
    compare(kd, kh)
    compare(vd, vh)
    for step in (0, 5):
        compare(g.queries(step), kvsynth.queries(w, step=step))
    # appended positions (beyond the context) continue the same chain
    ka, va = g.kv_cache(p0=w.n_ctx, p1=w.n_ctx + 70)
    kah, vah = kvsynth.kv_cache(w, p0=w.n_ctx, p1=w.n_ctx + 70)
    compare(ka, kah)
    compare(va, vah)


def test_device_cache_matches_host_at_million_token_positions():
    """Rows near position 2^20 of the million-token workload (the largest rotation angles),
    every unit of its 32 layers x 8 kv heads, and its queries."""
    w = kvsynth.get_workload("llama3-8b-1m-32l")
    g = kvsynth.DeviceGen(w)
    p0, p1 = w.n_ctx - 96, w.n_ctx
    kd, vd = g.kv_cache(p0=p0, p1=p1)
    kh, vh = kvsynth.kv_cache(w, p0=p0, p1=p1)
    torch.cuda.synchronize()
    compare(kd, kh)
    compare(vd, vh)
    compare(g.queries(3), kvsynth.queries(w, step=3))
    # sinks of the first rows
    kd, vd = g.kv_cache(p0=0, p1=8)
    kh, vh = kvsynth.kv_cache(w, p0=0, p1=8)
    compare(kd, kh)
    compare(vd, vh)
