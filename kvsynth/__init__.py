"""Seeded synthetic KV-cache / query generator (input generation only).

Shared by the CPU oracle and the CUDA path: both consume the bf16 bytes made
here.  Holds none of the wave-index arithmetic.  The C source ``kvsynth.c``
documents the distribution (topic Markov chain, rotate-half RoPE, sinks) and
the counter-based random numbers (SplitMix64 draws, Box-Muller normals).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .workloads import WORKLOADS, Workload, get_workload  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvsynth.c")
_LIB_PATH = os.path.join(_HERE, "libkvsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``kvsynth.c`` into ``libkvsynth.so`` beside it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Params(ctypes.Structure):
    _fields_ = [
        ("seed", ctypes.c_uint64),
        ("d", ctypes.c_int),
        ("n_topics", ctypes.c_int),
        ("n_sink", ctypes.c_int),
        ("p_stay", ctypes.c_double),
        ("sigma_k", ctypes.c_double),
        ("sink_scale", ctypes.c_double),
        ("theta", ctypes.c_double),
        ("q_scale", ctypes.c_double),
        ("sigma_q", ctypes.c_double),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u16p = ctypes.POINTER(ctypes.c_uint16)
            lib.kvs_cache.argtypes = [ctypes.POINTER(_Params), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_long, ctypes.c_long, u16p, u16p]
            lib.kvs_cache.restype = ctypes.c_int
            lib.kvs_queries.argtypes = [ctypes.POINTER(_Params), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_long, ctypes.c_int, u16p]
            lib.kvs_queries.restype = ctypes.c_int
            lib.kvs_bf16.argtypes = [ctypes.c_double]
            lib.kvs_bf16.restype = ctypes.c_uint16
            lib.kvs_draw.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.kvs_draw.restype = ctypes.c_uint64
            lib.kvs_mix64.argtypes = [ctypes.c_uint64]
            lib.kvs_mix64.restype = ctypes.c_uint64
            lib.kvs_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.kvs_normal.restype = ctypes.c_double
            _lib = lib
    return _lib


def _params(w: Workload, seed: int) -> _Params:
    return _Params(seed, w.head_dim, w.n_topics, w.n_sink, w.p_stay, w.sigma_k, w.sink_scale,
                   w.rope_theta, w.q_scale, w.sigma_q)


def _u16p(a: np.ndarray):
    assert a.dtype == np.uint16 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def kv_cache(w: Workload, seed: int | None = None, p0: int = 0, p1: int | None = None,
             out_k: np.ndarray | None = None, out_v: np.ndarray | None = None):
    """Keys and values as bf16 bit patterns, shape [B][L][Hkv][p1-p0][d] (uint16).

    Positions default to the whole context [0, n_ctx).  Rows for positions at or
    beyond n_ctx continue the same topic chain (used for appended tokens).
    """
    lib = _load()
    seed = w.seed if seed is None else seed
    p1 = w.n_ctx if p1 is None else p1
    shape = (w.batch, w.layers, w.n_kv_heads, p1 - p0, w.head_dim)
    k = np.empty(shape, np.uint16) if out_k is None else out_k
    v = np.empty(shape, np.uint16) if out_v is None else out_v
    assert k.shape == shape and v.shape == shape
    prm = _params(w, seed)
    rc = lib.kvs_cache(ctypes.byref(prm), w.batch, w.layers, w.n_kv_heads, p0, p1, _u16p(k), _u16p(v))
    if rc != 0:
        raise MemoryError("kvsynth: allocation failed")
    return k, v


def queries(w: Workload, step: int = 0, seed: int | None = None) -> np.ndarray:
    """Decode queries for step ``step`` at position n_ctx + step, bf16 bits [B][L][Hq][d]."""
    lib = _load()
    seed = w.seed if seed is None else seed
    q = np.empty((w.batch, w.layers, w.n_q_heads, w.head_dim), np.uint16)
    prm = _params(w, seed)
    rc = lib.kvs_queries(ctypes.byref(prm), w.batch, w.layers, w.n_q_heads, w.n_kv_heads,
                         w.n_ctx + step, step, _u16p(q))
    if rc != 0:
        raise MemoryError("kvsynth: allocation failed")
    return q


# ----------------------------------------------------------- on the GPU ----
# kvsynth_cuda.cu: the same generator as CUDA kernels (same draws, transforms and rounding),
# for caches too large to generate on the host.  Built by build_cuda(); needs a CUDA device.

_CU_SRC = os.path.join(_HERE, "kvsynth_cuda.cu")
_CU_LIB_PATH = os.path.join(_HERE, "libkvsynth_cuda.so")
_cu_lib = None


def build_cuda(force: bool = False) -> str:
    """Compile ``kvsynth_cuda.cu`` into ``libkvsynth_cuda.so`` beside it (nvcc, sm_103a, no FMA
    contraction so that every double operation rounds like the host build)."""
    if force or not os.path.exists(_CU_LIB_PATH) or os.path.getmtime(_CU_LIB_PATH) < os.path.getmtime(_CU_SRC):
        import shutil
        nvcc = next((c for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc")
                     if c and os.path.exists(c)), None)
        if nvcc is None:
            raise RuntimeError("nvcc not found")
        tmp = _CU_LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-fmad=false", "-Xcompiler", "-fPIC",
               "-shared", "-o", tmp, _CU_SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _CU_LIB_PATH)
    return _CU_LIB_PATH


def _load_cuda():
    global _cu_lib
    with _lock:
        if _cu_lib is None:
            lib = ctypes.CDLL(build_cuda())
            vp = ctypes.c_void_p
            pp = ctypes.POINTER(_Params)
            lib.kvs_topics_dev.argtypes = [pp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp]
            lib.kvs_cache_dev.argtypes = [pp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_long, ctypes.c_long,
                                          vp, vp, vp, vp]
            lib.kvs_queries_dev.argtypes = [pp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_long, ctypes.c_int, vp, vp, vp]
            for f in (lib.kvs_topics_dev, lib.kvs_cache_dev, lib.kvs_queries_dev):
                f.restype = ctypes.c_int
            _cu_lib = lib
    return _cu_lib


class DeviceGen:
    """The generator of one workload and seed on a CUDA device: topic centres computed once,
    then key/value rows of any position range and the queries of any step, as int16 torch
    tensors holding bf16 bits (same shapes as kv_cache / queries)."""

    def __init__(self, w: Workload, seed: int | None = None, device="cuda", stream=None):
        import torch
        self.w, self.seed = w, (w.seed if seed is None else seed)
        self.torch, self.device = torch, torch.device(device)
        self.prm = _params(w, self.seed)
        self.lib = _load_cuda()
        self.topics = torch.empty((w.units, w.n_topics, w.head_dim), dtype=torch.float64, device=self.device)
        self._call(self.lib.kvs_topics_dev, ctypes.byref(self.prm), w.batch, w.layers, w.n_kv_heads,
                   self.topics.data_ptr(), self._stream(stream))

    def _stream(self, stream):
        torch = self.torch
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        return s.cuda_stream if isinstance(s, torch.cuda.Stream) else int(s)

    @staticmethod
    def _call(f, *args):
        rc = f(*args)
        if rc != 0:
            raise RuntimeError(f"kvsynth (device): CUDA error {rc}")

    def kv_cache(self, p0: int = 0, p1: int | None = None, out_k=None, out_v=None, stream=None):
        w, torch = self.w, self.torch
        p1 = w.n_ctx if p1 is None else p1
        shape = (w.batch, w.layers, w.n_kv_heads, p1 - p0, w.head_dim)
        k = torch.empty(shape, dtype=torch.int16, device=self.device) if out_k is None else out_k
        v = torch.empty(shape, dtype=torch.int16, device=self.device) if out_v is None else out_v
        assert tuple(k.shape) == shape and tuple(v.shape) == shape and k.is_contiguous() and v.is_contiguous()
        self._call(self.lib.kvs_cache_dev, ctypes.byref(self.prm), w.batch, w.layers, w.n_kv_heads, p0, p1,
                   self.topics.data_ptr(), k.data_ptr(), v.data_ptr(), self._stream(stream))
        return k, v

    def queries(self, step: int = 0, out=None, stream=None):
        w, torch = self.w, self.torch
        shape = (w.batch, w.layers, w.n_q_heads, w.head_dim)
        q = torch.empty(shape, dtype=torch.int16, device=self.device) if out is None else out
        self._call(self.lib.kvs_queries_dev, ctypes.byref(self.prm), w.batch, w.layers, w.n_q_heads, w.n_kv_heads,
                   w.n_ctx + step, step, self.topics.data_ptr(), q.data_ptr(), self._stream(stream))
        return q


def bf16_bits(x: float) -> int:
    """The generator's own double -> bf16 rounding (used to pin it in tests)."""
    return int(_load().kvs_bf16(float(x)))


def draw(state: int, i: int) -> int:
    """i-th 64-bit draw of the SplitMix64 sequence started from ``state``."""
    return int(_load().kvs_draw(state, i))


def normal(key: int, i: int) -> float:
    return float(_load().kvs_normal(key, i))
