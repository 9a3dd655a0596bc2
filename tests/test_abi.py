"""The C-ABI library builds for sm_103a, loads, and exports every entry point
that include/sdv.h declares; argument checks that need no GPU behave as
documented.  No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdv.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sdv_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from draft_verification_sdv_gb300 import binding
    return binding.load(build=True)


def test_header_declares_the_api():
    names = _declared_functions()
    for required in ("sdv_create", "sdv_verify", "sdv_verify_ex", "sdv_verify_host",
                     "sdv_sync", "sdv_last_error", "sdv_destroy"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from draft_verification_sdv_gb300 import binding
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert name in binding.SIGNATURES, "binding misses " + name


def test_argument_errors_without_gpu(lib):
    from draft_verification_sdv_gb300 import binding as bd
    ctx = ctypes.c_void_p()
    # shape / dtype / alignment checks return before any CUDA call
    assert lib.sdv_create(None, 1, 1, 1, 32, bd.SDV_F32, None) == bd.SDV_ERR_ARG
    for B, K, G, V, dt in [(0, 1, 4, 32, bd.SDV_F32), (1, 0, 4, 32, bd.SDV_F32),
                           (1, 1, 0, 32, bd.SDV_F32), (1, 1, 4, 0, bd.SDV_F32),
                           (1, 1, 4, 30, bd.SDV_BF16), (1, 1, 4, 5, bd.SDV_F32),
                           (1, 1, 4, 32, 7)]:
        assert lib.sdv_create(ctypes.byref(ctx), B, K, G, V, dt, None) == bd.SDV_ERR_ARG
        assert ctx.value is None
    assert lib.sdv_verify(None, None, None, None, 1.0, 0, None, None, None) == bd.SDV_ERR_ARG
    assert lib.sdv_verify_qstat(None, None, None, None, None, None, 1.0, None, 0, None, None, None,
                                None, None) == bd.SDV_ERR_ARG
    # path search with statistics: shape and limit checks come before any CUDA call
    for B, G, mmax, beam in [(0, 4, 8, 3), (1, 0, 8, 3), (1, 4, 0, 3), (1, 4, 17, 3), (1, 4, 8, 0),
                             (1, 4, 8, 17)]:
        assert lib.sdv_cps_ex(B, G, 64, bd.SDV_BF16, None, None, 1.0, None, 0.8, mmax, beam, -1,
                              None, None, None, None, None, None, None, None,
                              None) == bd.SDV_ERR_ARG
    # the allocation-free entry point: alignment of the int32 / float arrays is
    # checked before anything touches the device (fake, never dereferenced
    # addresses: 16-byte aligned logits, then one 4-byte array off by 2)
    base = [0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000]
    for i in range(2, 6):
        ptrs = list(base)
        ptrs[i] += 2
        assert lib.sdv_verify_static(2, 2, 3, 64, bd.SDV_BF16, None, ptrs[0], ptrs[1], ptrs[2], 1.0,
                                     None, 0, ptrs[3], ptrs[4], ptrs[5]) == bd.SDV_ERR_ARG
    assert lib.sdv_verify_static(2, 2, 3, 64, bd.SDV_BF16, None, base[0], base[1], base[2], 1.0,
                                 0x70002, 0, base[3], base[4], base[5]) == bd.SDV_ERR_ARG
    assert lib.sdv_set_test_hooks(None, 0) == bd.SDV_ERR_ARG
    assert lib.sdv_sync(None) == bd.SDV_ERR_ARG
    assert lib.sdv_last_error(None) == b"null context"
    lib.sdv_destroy(None)


def test_product_path_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "draft_verification_sdv_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "sdvo_" not in text and "sdv_oracle" not in text, f
