"""GB300 wave-index hot path: Python binding of ``libwaveindex.so``.

Argument marshalling only: every step of the index build and of the decode
step runs in the CUDA kernels of ``csrc/`` behind the C ABI declared in
``include/wave_index.h``.  The functions keep the C names; tensors are torch
tensors (device memory unless a function says host), passed by data pointer
together with torch's current CUDA stream.  There is no CPU fallback: if the
library has not been built, importing this package raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libwaveindex.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")

lib = ctypes.CDLL(_LIB_PATH)

WI_OK, WI_EINVAL, WI_ENOMEM, WI_ECUDA, WI_EUNSUPPORTED, WI_EDEVICE, WI_EFULL = 0, -1, -2, -3, -4, -5, -6
_NAMES = {-1: "WI_EINVAL", -2: "WI_ENOMEM", -3: "WI_ECUDA", -4: "WI_EUNSUPPORTED", -5: "WI_EDEVICE",
          -6: "WI_EFULL"}


class WiError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_NAMES.get(code, code)}: {msg}")
        self.code = code


class wi_config(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int), ("layers", ctypes.c_int), ("n_q_heads", ctypes.c_int),
        ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("n_ctx", ctypes.c_longlong),
        ("seg_len", ctypes.c_int), ("clusters_per_seg", ctypes.c_int), ("iters", ctypes.c_int),
        ("n_sink", ctypes.c_int), ("local_window", ctypes.c_int), ("max_append", ctypes.c_int),
        ("budget_frac", ctypes.c_double), ("budget_k", ctypes.c_int),
        ("valsum_bf16", ctypes.c_int),
        ("group_topk", ctypes.c_int),
        ("reserved", ctypes.c_int * 1),
    ]


_vp = ctypes.c_void_p
_ip = ctypes.POINTER(ctypes.c_int)
_cfgp = ctypes.POINTER(wi_config)
_SIGS = {
    "wi_build_index": [_cfgp, _vp, _vp, _vp, _vp, ctypes.POINTER(_vp)],
    "wi_index_import": [_cfgp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.POINTER(_vp)],
    "wi_index_export": [_vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "wi_decode_step": [_vp, _vp, _vp, _vp, _vp, _vp],
    "wi_decode_step_host": [_vp, _vp, _vp, _vp, _vp, _vp],
    "wi_dense_decode": [_vp, _vp, _vp, _vp],
    "wi_decode_kernel": [_vp, ctypes.c_int, _vp, _vp, _vp],
    "wi_last_selection": [_vp, _vp, _vp, _vp],
    "wi_index_shape": [_vp, _ip, _ip, _ip, _ip, _ip],
    "wi_decode_layout": [_vp, _ip, _ip, _ip],
    "wi_kmeans_step": [_cfgp, _vp, _vp, _vp, _vp, _vp],
    "wi_kmeans_step_noalloc": [_cfgp, _vp, _vp, _vp, _vp, _vp],
    "wi_init_centroids": [_cfgp, _vp, _vp, _vp],
    "wi_check_device": [_vp],
    "wi_selftest_wait_timeout": [_ip, _ip],
    "wi_profile_begin": [_vp, ctypes.c_int],
    "wi_index_build_stats": [_vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double), _ip],
    "wi_profile_read": [_vp, ctypes.POINTER(ctypes.c_double), _ip, ctypes.POINTER(ctypes.c_ulonglong)],
    "wi_tier_attach": [_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp],
    "wi_tier_round": [_vp, _vp],
    "wi_tier_stats": [_vp, ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_ulonglong), _ip, _ip],
    "wi_tier_tables": [_vp, _vp, _vp],
    "wi_lru_round": [_vp, _vp, ctypes.c_int, ctypes.c_longlong, _vp, _vp, _ip, _vp, _vp, _ip],
}
for _name, _args in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
lib.wi_free.argtypes = [_vp]
lib.wi_free.restype = None
lib.wi_last_error.argtypes = []
lib.wi_last_error.restype = ctypes.c_char_p
lib.wi_lru_new.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
lib.wi_lru_new.restype = _vp
lib.wi_lru_free.argtypes = [_vp]
lib.wi_lru_free.restype = None

EXPORTED = sorted([*_SIGS, "wi_free", "wi_last_error", "wi_lru_new", "wi_lru_free"])


def _check(rc: int):
    if rc != WI_OK:
        raise WiError(rc, lib.wi_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        return t.data_ptr()
    if hasattr(t, "__array_interface__"):  # numpy array: host memory
        if not t.flags["C_CONTIGUOUS"]:
            raise ValueError("arrays must be C-contiguous")
        return t.ctypes.data
    return int(t)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def make_config(batch, layers, n_q_heads, n_kv_heads, n_ctx, seg_len=8192, clusters_per_seg=512, iters=10,
                n_sink=4, local_window=64, max_append=0, budget_frac=0.018, budget_k=0, head_dim=128,
                valsum_bf16=0) -> wi_config:
    c = wi_config()
    c.batch, c.layers, c.n_q_heads, c.n_kv_heads, c.head_dim = batch, layers, n_q_heads, n_kv_heads, head_dim
    c.n_ctx, c.seg_len, c.clusters_per_seg, c.iters = n_ctx, seg_len, clusters_per_seg, iters
    c.n_sink, c.local_window, c.max_append = n_sink, local_window, max_append
    c.budget_frac, c.budget_k = budget_frac, budget_k
    c.valsum_bf16 = valsum_bf16
    return c


def config_from_workload(w, max_append: int | None = None, iters: int | None = None) -> wi_config:
    return make_config(w.batch, w.layers, w.n_q_heads, w.n_kv_heads, w.n_ctx, w.seg_len, w.clusters_per_seg,
                       w.iters if iters is None else iters, w.n_sink, w.local_window,
                       (w.decode_steps if w.append else 0) if max_append is None else max_append,
                       w.budget_frac, w.budget_k, w.head_dim)


# ----------------------------------------------------------- C-named calls ----

def wi_build_index(cfg: wi_config, k: torch.Tensor, v: torch.Tensor, init_centroids=None, stream=None) -> int:
    out = _vp()
    _check(lib.wi_build_index(ctypes.byref(cfg), _ptr(k), _ptr(v), _ptr(init_centroids), _stream(stream),
                              ctypes.byref(out)))
    return out.value


def wi_index_import(cfg: wi_config, k, v, counts, perm, mu, valsum, stream=None) -> int:
    out = _vp()
    _check(lib.wi_index_import(ctypes.byref(cfg), _ptr(k), _ptr(v), _ptr(counts), _ptr(perm), _ptr(mu),
                               _ptr(valsum), _stream(stream), ctypes.byref(out)))
    return out.value


def wi_index_export(ix: int, counts=None, offsets=None, perm=None, mu=None, valsum=None, stream=None):
    _check(lib.wi_index_export(ix, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(mu), _ptr(valsum),
                               _stream(stream)))


def wi_decode_step(ix: int, q, out, k_new=None, v_new=None, stream=None):
    _check(lib.wi_decode_step(ix, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out), _stream(stream)))


def wi_dense_decode(ix: int, q, out, stream=None):
    _check(lib.wi_dense_decode(ix, _ptr(q), _ptr(out), _stream(stream)))


def wi_decode_kernel(ix: int, kernel: int, q, out, stream=None):
    """One decode kernel alone (0 scores, 1 top-k + estimation, 2 exact + merge), for timing."""
    _check(lib.wi_decode_kernel(ix, kernel, _ptr(q), _ptr(out), _stream(stream)))


def wi_decode_step_host(ix: int, q_host, out_host, k_new_host=None, v_new_host=None, stream=None):
    _check(lib.wi_decode_step_host(ix, _ptr(q_host), _ptr(k_new_host), _ptr(v_new_host), _ptr(out_host),
                                   _stream(stream)))


def wi_last_selection(ix: int, ids, counts=None, stream=None):
    _check(lib.wi_last_selection(ix, _ptr(ids), _ptr(counts), _stream(stream)))


def wi_index_shape(ix: int) -> dict:
    vals = [ctypes.c_int() for _ in range(5)]
    _check(lib.wi_index_shape(ix, *[ctypes.byref(x) for x in vals]))
    return dict(zip(["units", "clusters", "k_max", "group", "appended"], [x.value for x in vals]))


def wi_decode_layout(ix: int) -> dict:
    vals = [ctypes.c_int() for _ in range(3)]
    _check(lib.wi_decode_layout(ix, *[ctypes.byref(x) for x in vals]))
    return dict(zip(["score_ctas", "estimate_ctas", "exact_splits"], [x.value for x in vals]))


def wi_kmeans_step(cfg: wi_config, k, centroids, assign, new_centroids, stream=None):
    _check(lib.wi_kmeans_step(ctypes.byref(cfg), _ptr(k), _ptr(centroids), _ptr(assign), _ptr(new_centroids),
                              _stream(stream)))


def wi_init_centroids(cfg: wi_config, k, centroids, stream=None):
    _check(lib.wi_init_centroids(ctypes.byref(cfg), _ptr(k), _ptr(centroids), _stream(stream)))


def wi_kmeans_step_noalloc(cfg: wi_config, k, centroids, assign, new_centroids, stream=None):
    """wi_kmeans_step with its scratch in the library's fixed device array (no allocation)."""
    _check(lib.wi_kmeans_step_noalloc(ctypes.byref(cfg), _ptr(k), _ptr(centroids), _ptr(assign),
                                      _ptr(new_centroids), _stream(stream)))


def wi_check_device(ix: int):
    _check(lib.wi_check_device(ix))


def wi_selftest_wait_timeout() -> dict:
    """Run the kernels' bounded wait on a barrier nothing completes (test hook; about one second)."""
    err, ret = ctypes.c_int(), ctypes.c_int()
    _check(lib.wi_selftest_wait_timeout(ctypes.byref(err), ctypes.byref(ret)))
    return {"device_error": err.value, "wait_returned": ret.value}


WI_NUM_DECODE_KERNELS = 3
DECODE_KERNELS = ["scores", "select_estimate", "exact_merge"]


def wi_profile_begin(ix: int, max_steps: int):
    _check(lib.wi_profile_begin(ix, max_steps))


def wi_profile_read(ix: int, times: bool = True):
    """(per-kernel summed ms, filled slots, exact rows).  times=False skips the event
    timings (use it before the recorded steps have run, e.g. right after a graph capture)."""
    ms = (ctypes.c_double * WI_NUM_DECODE_KERNELS)()
    steps = ctypes.c_int()
    rows = ctypes.c_ulonglong()
    _check(lib.wi_profile_read(ix, ms if times else None, ctypes.byref(steps), ctypes.byref(rows)))
    return dict(zip(DECODE_KERNELS, list(ms))) if times else None, steps.value, rows.value


def wi_index_build_stats(ix: int) -> dict:
    b, a, n = ctypes.c_double(), ctypes.c_double(), ctypes.c_int()
    _check(lib.wi_index_build_stats(ix, ctypes.byref(b), ctypes.byref(a), ctypes.byref(n)))
    return {"build_ms": b.value, "assign_ms": a.value, "assign_launches": n.value}


def wi_free(ix: int):
    lib.wi_free(ix)


TIER_COUNTERS = ["rounds", "pages_read", "page_hits", "page_misses", "admitted", "evicted"]


def wi_tier_attach(ix: int, slots_per_unit: int, admit_per_round: int, async_rounds: bool = True, stream=None):
    _check(lib.wi_tier_attach(ix, slots_per_unit, admit_per_round, 1 if async_rounds else 0, _stream(stream)))


def wi_tier_round(ix: int, stream=None):
    _check(lib.wi_tier_round(ix, _stream(stream)))


def wi_tier_stats(ix: int) -> dict:
    c = (ctypes.c_longlong * 6)()
    r = (ctypes.c_ulonglong * 2)()
    slots, pages = ctypes.c_int(), ctypes.c_int()
    _check(lib.wi_tier_stats(ix, c, r, ctypes.byref(slots), ctypes.byref(pages)))
    d = dict(zip(TIER_COUNTERS, list(c)))
    d.update(rows_from_cache=r[0], rows_from_host=r[1], slots=slots.value, pages=pages.value)
    return d


def wi_tier_tables(ix: int, slot_of=None, use=None):
    _check(lib.wi_tier_tables(ix, _ptr(slot_of), _ptr(use)))


class LruPolicy:
    """The tier's page replacement policy alone, run on the host (wi_lru_*)."""

    def __init__(self, pages: int, slots: int, admit_max: int):
        self.h = lib.wi_lru_new(pages, slots, admit_max)
        if not self.h:
            raise ValueError("bad policy sizes")

    def round(self, touched, t: int):
        import numpy as np
        tp = np.ascontiguousarray(np.asarray(list(touched), dtype=np.int32))
        n = max(int(tp.size), 1)
        ep, es, ap, as_ = (np.empty(n, np.int32) for _ in range(4))
        ne, na = ctypes.c_int(), ctypes.c_int()
        _check(lib.wi_lru_round(self.h, tp.ctypes.data if tp.size else None, int(tp.size), t, ep.ctypes.data,
                                es.ctypes.data, ctypes.byref(ne), ap.ctypes.data, as_.ctypes.data, ctypes.byref(na)))
        return ([(int(ep[i]), int(es[i])) for i in range(ne.value)],
                [(int(ap[i]), int(as_[i])) for i in range(na.value)])

    def __del__(self):
        if getattr(self, "h", None):
            lib.wi_lru_free(self.h)
            self.h = None


# ------------------------------------------------------------ convenience ----

class WaveIndex:
    """Owns one index handle; tensors stay torch tensors on the current device."""

    def __init__(self, cfg: wi_config, k: torch.Tensor, v: torch.Tensor, handle: int):
        self.cfg, self.k, self.v, self.handle = cfg, k, v, handle
        s = wi_index_shape(handle)
        self.units, self.clusters, self.k_max, self.group = s["units"], s["clusters"], s["k_max"], s["group"]

    @classmethod
    def build(cls, cfg: wi_config, k: torch.Tensor, v: torch.Tensor, init_centroids=None, stream=None):
        return cls(cfg, k, v, wi_build_index(cfg, k, v, init_centroids, stream))

    @classmethod
    def adopt(cls, cfg: wi_config, k, v, counts, perm, mu, valsum, stream=None):
        return cls(cfg, k, v, wi_index_import(cfg, k, v, counts, perm, mu, valsum, stream))

    def decode(self, q: torch.Tensor, k_new=None, v_new=None, out=None, stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty((self.cfg.batch, self.cfg.layers, self.cfg.n_q_heads, 128), dtype=torch.float32,
                              device=q.device)
        wi_decode_step(self.handle, q, out, k_new, v_new, stream)
        return out

    def dense_decode(self, q: torch.Tensor, out=None, stream=None) -> torch.Tensor:
        """Full attention over every cached and appended token (the comparator)."""
        if out is None:
            out = torch.empty((self.cfg.batch, self.cfg.layers, self.cfg.n_q_heads, 128), dtype=torch.float32,
                              device=q.device)
        wi_dense_decode(self.handle, q, out, stream)
        return out

    @property
    def perm_slots(self) -> int:
        """Slots per unit in perm: the build's clustered tokens plus room for the segments that
        appends may grow (max_append // seg_len of seg_len tokens)."""
        c = self.cfg
        return c.n_ctx - c.n_sink - c.local_window + (c.max_append // c.seg_len) * c.seg_len

    def export(self, stream=None) -> dict:
        U, C = self.units, self.clusters
        n_idx = self.perm_slots
        dev = self.k.device
        r = {
            "counts": torch.empty((U, C), dtype=torch.int32, device=dev),
            "offsets": torch.empty((U, C + 1), dtype=torch.int32, device=dev),
            "perm": torch.empty((U, n_idx), dtype=torch.int32, device=dev),
            "mu": torch.empty((U, C, 128), dtype=torch.int16, device=dev),
            "valsum": torch.empty((U, C, 128), dtype=torch.float32, device=dev),
        }
        wi_index_export(self.handle, r["counts"], r["offsets"], r["perm"], r["mu"], r["valsum"], stream)
        return r

    def selection(self, stream=None):
        ids = torch.empty((self.units, self.group, self.k_max), dtype=torch.int32, device=self.k.device)
        cnt = torch.empty((self.units, self.group), dtype=torch.int32, device=self.k.device)
        wi_last_selection(self.handle, ids, cnt, stream)
        return ids, cnt

    def check(self):
        wi_check_device(self.handle)

    def attach_tier(self, slots_per_unit: int, admit_per_round: int, async_rounds: bool = True, stream=None):
        """Move the K/V rows to host memory behind a device page cache (after this, no call reads
        this index's k / v tensors)."""
        wi_tier_attach(self.handle, slots_per_unit, admit_per_round, async_rounds, stream)

    def tier_round(self, stream=None):
        wi_tier_round(self.handle, stream)

    def tier_stats(self) -> dict:
        return wi_tier_stats(self.handle)

    def tier_tables(self):
        s = wi_tier_stats(self.handle)
        slot_of = torch.empty((self.units, s["pages"]), dtype=torch.int32)
        use = torch.empty((self.units, s["pages"]), dtype=torch.int32)
        wi_tier_tables(self.handle, slot_of, use)
        return slot_of, use

    def free(self):
        if self.handle:
            wi_free(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass

