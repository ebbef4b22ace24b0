"""Host-side checks of the C-ABI library that need no GPU: it builds, loads,
exports every entry point that include/lora.h declares, answers host-only
calls, rejects bad arguments before touching the device, and the product
package never reaches the oracle."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lora.h")


@pytest.fixture(scope="module")
def lib():
    from tenant_composite_lora_gb300 import build, native
    build.build()
    return native.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("lora_pool_create", "lora_pool_register", "lora_build_mapping", "lora_delta_apply",
                 "lora_mapping_status", "lora_pool_destroy", "lora_mapping_destroy"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    from tenant_composite_lora_gb300 import native
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(native.EXPORTS) == names


def test_host_only_calls(lib):
    from tenant_composite_lora_gb300 import native
    assert native.status_string(0) == "ok"
    assert "not supported" in native.status_string(5)
    assert "sm_103a" in native.lora_version()
    # the dispatch table: decode batches, long prefill batches, the middle
    assert native.lora_dispatch_choose(32, 96, 8, 4096, 4096) == native.LORA_PATH_DECODE
    assert native.lora_dispatch_choose(256, 512, 64, 4096, 1024) == native.LORA_PATH_DECODE
    assert native.lora_dispatch_choose(3250, 6500, 16, 4096, 4096) == native.LORA_PATH_MMA
    assert native.lora_dispatch_choose(300, 900, 16, 4096, 4096) == native.LORA_PATH_SPLIT


def test_bad_arguments_rejected_before_device(lib):
    out = ctypes.c_void_p()
    assert lib.lora_pool_create(0, 64, 8, 4, ctypes.byref(out)) == 1
    assert lib.lora_pool_create(64, 64, 8, 4, None) == 1
    assert lib.lora_pool_create(100, 64, 8, 4, ctypes.byref(out)) == 5   # not a multiple of 64
    assert lib.lora_pool_create(64, 64, 65, 4, ctypes.byref(out)) == 5   # rank above the limit
    assert lib.lora_pool_create(64, 64, 8, 49153, ctypes.byref(out)) == 5
    assert lib.lora_mapping_create(-1, 4, 4, ctypes.byref(out)) == 1
    assert lib.lora_mapping_create(4, 4, 0, ctypes.byref(out)) == 1
    assert lib.lora_build_mapping(None, None, None, None, 1, 1, None) == 1
    assert lib.lora_delta_apply(None, None, None, None, None, None) == 1
    assert lib.lora_pool_register(None, 0, None, None, 1, None) == 1
    assert lib.lora_pool_destroy(None) == 0
    assert lib.lora_mapping_destroy(None) == 0


def test_missing_library_fails_loudly(tmp_path):
    from tenant_composite_lora_gb300 import native
    saved = native._lib
    native._lib = None
    try:
        with pytest.raises(RuntimeError, match="no CPU or Python fallback"):
            native.load(str(tmp_path / "nope.so"))
    finally:
        native._lib = saved


def test_product_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "tenant_composite_lora_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.lower(), f
                assert "lora_oracle" not in src
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            src = open(os.path.join(ROOT, "oracle", f)).read()
            assert "tenant_composite_lora_gb300" not in src
