"""The C-ABI library without a GPU: it builds, loads, exports every function
include/dllm_kv.h declares, and rejects bad arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "dllm_kv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:dllm_status|const char\s*\*)\s*(\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from denoising_step_kv_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        from denoising_step_kv_gb300 import build
        build.build()
    return _lib.lib()


def test_header_declares_the_step(lib):
    names = _declared()
    for n in ("dllm_cache_init", "kv_refresh", "block_attn", "lmhead_conf", "stab_update"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from denoising_step_kv_gb300 import _lib
    names = _declared()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # the Python binding wraps every one of them under the same name
    assert sorted(set(_lib.EXPORTS)) == names


def _cfg(**kw):
    from denoising_step_kv_gb300 import _lib
    from workloads import configs as C
    c = _lib.make_cfg(C.get("mid_bf16"))
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("field,value,status", [
    ("batch", 0, 1), ("block_len", 65, 1), ("swd_K", 9, 1), ("dtype", 7, 1),
    ("head_dim", 96, 5), ("ffn", 100, 5), ("rope_theta", -1.0, 1),
])
def test_init_rejects_bad_shapes_without_cuda(lib, field, value, status):
    h = ctypes.c_void_p()
    st = lib.dllm_cache_init(ctypes.byref(_cfg(**{field: value})), None, ctypes.byref(h))
    assert st == status
    assert not h.value
    assert lib.dllm_last_error()


def test_null_handle_is_einval(lib):
    assert lib.kv_refresh(None, 0, None, None, None, None, None, None, 0, None) == 1
    assert lib.block_attn(None, 0, 0, 1, None, None) == 1
    assert lib.lmhead_conf(None, None, None, 1, 2, 2, 0, None, None, None, None) == 1
    assert lib.stab_update(None, None, None, None, None, 0, 0, 0, 0, None, None, None) == 1
    assert b"null" in lib.dllm_last_error()


def test_python_binding_has_no_fallback(monkeypatch, tmp_path):
    from denoising_step_kv_gb300 import _lib
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        _lib.lib()


def _header_code():
    src = open(os.path.join(ROOT, "include", "dllm_kv.h")).read()
    return re.sub(r"/\*.*?\*/", "", src, flags=re.S)


def test_binding_matches_the_header():
    """The ctypes mirror of dllm_cache_cfg lists the header's fields in the
    header's order with the header's C types, and the binding's field, kernel
    and error constants carry the header's values."""
    from denoising_step_kv_gb300 import _lib as K
    src = _header_code()
    body = re.search(r"typedef struct \{(.*?)\} dllm_cache_cfg;", src, flags=re.S).group(1)
    want = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        ctype, names = decl.split(None, 1)
        want += [(n.strip(), ctype) for n in names.split(",")]
    got = [(n, {ctypes.c_int: "int", ctypes.c_float: "float"}[t]) for n, t in K.CacheCfg._fields_]
    assert got == want
    fields = dict(re.findall(r"DLLM_FIELD_(\w+)\s*=\s*(\d+)", src))
    assert fields and {k: int(v) for k, v in fields.items()} == {
        k[len("FIELD_"):]: getattr(K, k) for k in dir(K) if k.startswith("FIELD_")}
    errs = dict(re.findall(r"#define DLLM_ERR_(\w+)\s+(0x[0-9a-fA-F]+)u", src))
    assert errs and {k: int(v, 16) for k, v in errs.items()} == {
        k[len("ERR_"):]: getattr(K, k) for k in dir(K) if k.startswith("ERR_")}
    profs = dict(re.findall(r"DLLM_PROF_(\w+)\s*=\s*(\d+)", src))
    assert profs and {k: int(v) for k, v in profs.items()} == {
        k[len("PROF_"):]: getattr(K, k) for k in dir(K) if k.startswith("PROF_")}
