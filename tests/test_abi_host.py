"""The C ABI library loads, exports every declared entry point, and rejects
bad arguments on the host with the documented codes (no GPU needed)."""
import ctypes
import os
import re

import pytest

import __graft_entry__

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_build = __graft_entry__._load_build_module()
HEADER = os.path.join(ROOT, "include", "wave_index.h")


@pytest.fixture(scope="module")
def wi():
    _build.build()
    import clustered_sparse_kv_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(wi_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_path(wi):
    names = declared_functions()
    for must in ["wi_build_index", "wi_decode_step", "wi_free", "wi_index_import", "wi_index_export",
                 "wi_kmeans_step", "wi_last_error"]:
        assert must in names


def test_library_exports_every_declared_symbol(wi):
    lib = ctypes.CDLL(_build.LIB)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert sorted(wi.EXPORTED) == declared_functions()


def good_cfg(wi, **kw):
    base = dict(batch=1, layers=1, n_q_heads=4, n_kv_heads=1, n_ctx=2048, seg_len=1024, clusters_per_seg=64,
                iters=2, n_sink=4, local_window=64, max_append=0, budget_frac=0.018, budget_k=0)
    base.update(kw)
    return wi.make_config(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=64), -1),
    (dict(n_q_heads=6, n_kv_heads=4), -1),
    (dict(seg_len=1000, n_ctx=2000), -1),
    (dict(n_ctx=3000), -1),
    (dict(clusters_per_seg=8), -1),
    (dict(clusters_per_seg=1024, seg_len=2048, n_ctx=2048), -1),
    (dict(iters=0), -1),
    (dict(n_sink=0, local_window=0), -1),
    (dict(n_sink=1024, local_window=1024), -1),
    (dict(budget_k=10 ** 6), -1),
    (dict(batch=0), -1),
    (dict(n_q_heads=16, n_kv_heads=1), -4),
    (dict(seg_len=32768, n_ctx=32768, clusters_per_seg=512), -4),
])
def test_build_rejects_bad_config(wi, kw, code):
    cfg = good_cfg(wi, **kw)
    out = ctypes.c_void_p(123)
    rc = wi.lib.wi_build_index(ctypes.byref(cfg), 16, 16, None, None, ctypes.byref(out))
    assert rc == code, wi.lib.wi_last_error()
    assert out.value is None
    assert wi.lib.wi_last_error().decode() != ""


def test_reserved_fields_must_be_zero(wi):
    cfg = good_cfg(wi)
    cfg.reserved[0] = 7
    out = ctypes.c_void_p()
    assert wi.lib.wi_build_index(ctypes.byref(cfg), 16, 16, None, None, ctypes.byref(out)) == -1


@pytest.mark.parametrize("field", ["valsum_bf16", "group_topk"])
def test_variant_flags_are_zero_or_one(wi, field):
    cfg = good_cfg(wi)
    setattr(cfg, field, 2)
    out = ctypes.c_void_p()
    assert wi.lib.wi_build_index(ctypes.byref(cfg), 16, 16, None, None, ctypes.byref(out)) == -1
    assert field in wi.lib.wi_last_error().decode()


def test_null_and_misaligned_pointers_rejected(wi):
    cfg = good_cfg(wi)
    out = ctypes.c_void_p()
    assert wi.lib.wi_build_index(ctypes.byref(cfg), None, 16, None, None, ctypes.byref(out)) == -1
    assert wi.lib.wi_build_index(ctypes.byref(cfg), 18, 16, None, None, ctypes.byref(out)) == -1
    assert wi.lib.wi_build_index(None, 16, 16, None, None, ctypes.byref(out)) == -1
    assert wi.lib.wi_build_index(ctypes.byref(cfg), 16, 16, None, None, None) == -1
    assert wi.lib.wi_index_import(ctypes.byref(cfg), 16, 16, None, None, None, None, None, ctypes.byref(out)) == -1


def test_calls_on_null_index(wi):
    assert wi.lib.wi_decode_step(None, 16, None, None, 16, None) == -1
    assert wi.lib.wi_decode_step_host(None, 16, None, None, 16, None) == -1
    assert wi.lib.wi_index_export(None, None, None, None, None, None, None) == -1
    assert wi.lib.wi_last_selection(None, 16, None, None) == -1
    assert wi.lib.wi_index_shape(None, None, None, None, None, None) == -1
    assert wi.lib.wi_check_device(None) == -1
    assert wi.lib.wi_tier_attach(None, 8, 8, 0, None) == -1
    assert wi.lib.wi_tier_round(None, None) == -1
    assert wi.lib.wi_tier_stats(None, None, None, None, None) == -1
    assert wi.lib.wi_tier_tables(None, None, None) == -1
    assert "no host memory tier" in wi.lib.wi_last_error().decode() or "NULL" in wi.lib.wi_last_error().decode()
    assert wi.lib.wi_lru_new(0, 4, 4) is None     # bad sizes: no policy
    assert wi.lib.wi_lru_round(None, None, 0, 0, None, None, None, None, None, None) == -1
    wi.lib.wi_lru_free(None)  # no-op
    wi.lib.wi_free(None)  # no-op
    assert wi.lib.wi_selftest_wait_timeout(None, None) == -1   # checked before any device work
    cfg = good_cfg(wi)
    assert wi.lib.wi_kmeans_step(ctypes.byref(cfg), None, 16, 16, 16, None) == -1
    assert wi.lib.wi_kmeans_step(ctypes.byref(good_cfg(wi, head_dim=96)), 16, 16, 16, 16, None) == -1


def test_error_is_thread_local(wi):
    import threading
    cfg = good_cfg(wi, head_dim=64)
    out = ctypes.c_void_p()
    wi.lib.wi_build_index(ctypes.byref(cfg), 16, 16, None, None, ctypes.byref(out))
    seen = {}

    def other():
        seen["msg"] = wi.lib.wi_last_error().decode()

    t = threading.Thread(target=other)
    t.start()
    t.join()
    assert seen["msg"] == ""
    assert "head_dim" in wi.lib.wi_last_error().decode()


def test_header_is_c_and_config_layout_matches_binding(wi, tmp_path):
    """The header compiles as plain C99, and wi_config has the same size and field offsets in C as
    in the ctypes binding (a mismatch would pass wrong shapes silently)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [name for name, _ in wi.wi_config._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "wave_index.h"\nint main(void) {\n'
                   '  printf("size %zu\\n", sizeof(wi_config));\n'
                   + "".join(f'  printf("{f} %zu\\n", offsetof(wi_config, {f}));\n' for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)],
                   check=True)
    out = dict(line.split() for line in subprocess.run([str(exe)], check=True, capture_output=True,
                                                       text=True).stdout.splitlines())
    assert int(out["size"]) == ctypes.sizeof(wi.wi_config)
    for f in fields:
        assert int(out[f]) == getattr(wi.wi_config, f).offset, f
