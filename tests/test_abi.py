"""The C-ABI library builds for sm_103a, loads, and exports every function
include/ar.h declares; argument checks that return before any CUDA call are
exercised here without a GPU."""
import ctypes

import pytest

from shot_allreduce_ranks_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_header_declares_the_contract():
    names = _lib.header_functions()
    for required in ("ar_create", "ar_allreduce", "ar_destroy", "ar_set_variant",
                     "ar_get_device_status", "ar_status_string"):
        assert required in names


def test_every_declared_function_is_exported(lib):
    missing = [n for n in _lib.header_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_the_header():
    assert sorted(_lib.PROTOTYPES) == _lib.header_functions()


def test_status_and_variant_names(lib):
    for code in range(6):
        assert lib.ar_status_string(code)
    assert lib.ar_status_string(99) == b"unknown status"
    for name, v in _lib.VARIANTS.items():
        assert lib.ar_variant_name(v).decode() == name
    assert lib.ar_variant_name(42) == b"?"


def test_create_rejects_bad_arguments_before_touching_the_device(lib):
    h = ctypes.c_void_p(1)
    assert lib.ar_create(0, 16, 0, ctypes.byref(h)) == _lib.AR_ERR_INVALID_ARG
    assert h.value is None
    assert lib.ar_create(_lib.AR_MAX_RANKS + 1, 16, 0, ctypes.byref(h)) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_create(8, 0, 0, ctypes.byref(h)) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_create(8, 16, 0, None) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_create(8, 16, 3, ctypes.byref(h)) == _lib.AR_ERR_UNSUPPORTED
    assert lib.ar_create(8, 16, -1, ctypes.byref(h)) == _lib.AR_ERR_UNSUPPORTED


def test_null_handle_calls(lib):
    assert lib.ar_allreduce(None, 1, 1, 8, None) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_allreduce_host(None, 1, 1, 8, None) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_reduce_scatter(None, 1, 1, 8, None) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_all_gather(None, 1, 1, 8, None) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_allreduce_fused_noalloc(0, 1, 1, 8, None) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_destroy(None) == _lib.AR_OK
    assert lib.ar_set_variant(None, 0) == _lib.AR_ERR_INVALID_ARG
    v = ctypes.c_int()
    assert lib.ar_select(None, 8, ctypes.byref(v)) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_set_launch(None, 1, 0, 0) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_set_spin_limit_ns(None, 10 ** 6) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_get_device_status(None, None) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_last_timeout(None, None, None, None) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_debug_check_guards(None, None) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_query(None, None) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_reserve_host_staging(None) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_debug_skip_producer(None, 0) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_debug_set_epoch(None, 1) == _lib.AR_ERR_INVALID_ARG
    assert lib.ar_debug_get_epoch(None, None) == _lib.AR_ERR_INVALID_ARG


def test_build_targets_sm103a_only():
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert "--use_fast_math" not in build.NVCC_FLAGS
    assert "-ftz=false" in build.NVCC_FLAGS and "-fmad=false" in build.NVCC_FLAGS


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load(str(tmp_path / "libar_gb300.so"))


def _prototype_comment(text, name):
    """The comment block that ends right before `name`'s prototype."""
    import re
    for m in re.finditer(r"/\*(.*?)\*/", text, re.S):
        after = text[m.end():m.end() + 1200]
        # skip preprocessor lines (with their continuations) between the two
        after = re.sub(r"\A(\s*#(?:[^\n]*\\\n)*[^\n]*\n)+", "", after)
        decl = re.match(r"\s*[A-Za-z_][\w \t*]*?\b(\w+)\s*\(", after)
        if decl and decl.group(1) == name:
            return m.group(1)
    return ""


def test_core_entry_points_cite_their_source_passage():
    """Every core call of the boundary names the page (and section) that
    defines the operation, or says that the pages have none."""
    text = open(_lib.HEADER).read()
    cites = ("#1910", "#245", "#3850", "#254", "no counterpart", "define no such")
    for name in ("ar_create", "ar_allreduce", "ar_destroy", "ar_set_variant",
                 "ar_get_device_status", "ar_status_string",
                 "ar_allreduce_fused_noalloc", "ar_last_timeout"):
        comment = _prototype_comment(text, name)
        assert comment, name
        assert "Source:" in comment or "no counterpart" in comment, name
        assert any(c in comment for c in cites), name
