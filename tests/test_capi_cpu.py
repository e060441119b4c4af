"""The C-ABI library without a GPU: it builds, loads, exports every function
include/qre_moe.h declares, and its host-side checks answer as documented
(no call here launches a kernel)."""
import ctypes
import os
import re

import pytest

from oracle import formats as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def capi():
    from quantized_routed_expert_route_gb300 import build
    if not os.path.exists(build.lib_path()):
        build.build()
    from quantized_routed_expert_route_gb300 import capi as c
    return c


def _declared_functions():
    txt = open(os.path.join(ROOT, "include", "qre_moe.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", txt)))


def test_every_declared_symbol_is_exported(capi):
    decl = _declared_functions()
    assert len(decl) >= 13
    lib = capi.library()
    for name in decl:
        assert hasattr(lib, name), name
    assert sorted(capi.EXPORTS) == decl


def test_row_bytes_agree_with_the_oracle(capi):
    for t in sorted(F.TYPE_NAMES):
        for k in (32, 96, 256, 768, 2048, 4096, 100):
            assert capi.moe_row_bytes(t, k) == F.row_bytes(t, k), (t, k)
    # 16 is a kernel-side variant of NVFP4, not a type
    assert capi.moe_row_bytes(16, 256) == 0


def test_host_argument_checks(capi):
    lib = capi.library()
    g = capi.moe_layer_geom(256, 128, 8, 2, capi.MOE_Q8_0, capi.MOE_Q8_0)
    out = ctypes.c_void_p()
    # null rows, wrong byte counts, bad geometry: refused before any CUDA call
    assert lib.moe_bank_create(ctypes.byref(g), None, 0, None, 0, None, 0, None, ctypes.byref(out)) == capi.MOE_EINVAL
    buf = (ctypes.c_uint8 * 16)()
    assert lib.moe_bank_create(ctypes.byref(g), buf, 16, buf, 16, None, 0, None, ctypes.byref(out)) == capi.MOE_EINVAL
    bad = capi.moe_layer_geom(256, 128, 8, 9, capi.MOE_Q8_0, capi.MOE_Q8_0)     # top_k > E
    assert lib.moe_bank_create(ctypes.byref(bad), buf, 16, buf, 16, None, 0, None, ctypes.byref(out)) == capi.MOE_EINVAL
    bad = capi.moe_layer_geom(300, 128, 8, 2, capi.MOE_Q4_K, capi.MOE_Q8_0)     # H not a whole super-block
    assert lib.moe_bank_create(ctypes.byref(bad), buf, 16, buf, 16, None, 0, None, ctypes.byref(out)) == capi.MOE_EINVAL
    assert out.value is None
    assert lib.moe_decode(None, None, 1, None, None, None, None, 0, None) == capi.MOE_EINVAL
    assert lib.moe_quantize_q8_1(None, 32, None, None) == capi.MOE_EINVAL
    assert lib.moe_debug_block_dots(capi.MOE_BF16, buf, 1, 32, buf, buf, None) == capi.MOE_EINVAL
    assert lib.moe_workspace_bytes(None, 4) == 0
    assert lib.moe_bank_destroy(None) == capi.MOE_OK
    assert capi.status_string(capi.MOE_EDEVICE) == "device-side error flag set"


def test_host_argument_checks_of_the_newer_entry_points(capi):
    """moe_linear, the GLU field, the s_down fold, the prompt modes and the
    expert cache refuse bad arguments before any CUDA call."""
    lib = capi.library()
    buf = (ctypes.c_uint8 * 64)()
    out = ctypes.c_void_p()
    # moe_linear: T = 0 is a no-op; nulls, sizes, types and alignment are refused
    assert lib.moe_linear(capi.MOE_NVFP4, buf, 4, 256, None, buf, 0, buf, None, None) == capi.MOE_OK
    assert lib.moe_linear(capi.MOE_NVFP4, None, 4, 256, None, buf, 1, buf, None, None) == capi.MOE_EINVAL
    assert lib.moe_linear(capi.MOE_BF16, buf, 4, 256, None, buf, 1, buf, None, None) == capi.MOE_EUNSUPPORTED
    assert lib.moe_linear(capi.MOE_NVFP4, buf, 4, 256, None, buf, capi.MOE_LINEAR_MAX_T + 1, buf, None,
                          None) == capi.MOE_EUNSUPPORTED
    assert lib.moe_linear(capi.MOE_Q4_K, buf, 4, 96, None, buf, 1, buf, None, None) == capi.MOE_EINVAL
    assert lib.moe_linear(capi.MOE_F16, buf, 4, 256, None, buf, 1, buf, None, None) == capi.MOE_EUNSUPPORTED
    assert lib.moe_linear(13, buf, 4, 256, None, buf, 1, buf, None, None) == capi.MOE_EINVAL
    assert lib.moe_linear(capi.MOE_NVFP4, ctypes.addressof(buf) + 1, 4, 256, None, buf, 1, buf, None,
                          None) == capi.MOE_EINVAL
    # geometry: an unknown GLU or type is refused
    g = capi.moe_layer_geom(256, 128, 8, 2, capi.MOE_Q8_0, capi.MOE_Q8_0, 2)
    assert lib.moe_bank_create(ctypes.byref(g), buf, 64, buf, 64, None, 0, None, ctypes.byref(out)) == capi.MOE_EINVAL
    g = capi.moe_layer_geom(256, 128, 8, 2, capi.MOE_MXFP4 + 1, capi.MOE_Q8_0)
    assert lib.moe_bank_create(ctypes.byref(g), buf, 64, buf, 64, None, 0, None, ctypes.byref(out)) == capi.MOE_EINVAL
    # fold, prompt modes, cache
    assert lib.moe_bank_fold_down_scale(None, buf, capi.MOE_SRC_HOST, None) == capi.MOE_EINVAL
    assert lib.moe_prefill_workspace_bytes(None, 16, capi.MOE_PREFILL_FP16) == 0
    assert lib.moe_prefill_grouped(None, buf, 1, buf, buf, 3, buf, buf, 64, None) == capi.MOE_EINVAL
    g = capi.moe_layer_geom(256, 256, 8, 2, capi.MOE_Q4_K, capi.MOE_Q4_K)
    assert lib.moe_cache_create(ctypes.byref(g), 0, None, ctypes.byref(out)) == capi.MOE_EINVAL
    assert lib.moe_cache_create(None, 4, None, ctypes.byref(out)) == capi.MOE_EINVAL
    assert lib.moe_cache_bank(None) is None
    assert lib.moe_cache_acquire(None, 0, buf, buf, None, 8, None, 0, None, None, None) == capi.MOE_EINVAL
    assert lib.moe_cache_destroy(None) == capi.MOE_OK
    assert lib.moe_slot_table_create(0, ctypes.byref(out)) == capi.MOE_EINVAL
    assert out.value is None
    slots = (ctypes.c_int64 * 1)()
    assert lib.moe_cache_plan(-1, 1, (ctypes.c_int64 * 1)(5), (ctypes.c_int64 * 1)(1), slots) == capi.MOE_EINVAL
    assert lib.moe_cache_plan(100, 1, (ctypes.c_int64 * 1)(0), (ctypes.c_int64 * 1)(1), slots) == capi.MOE_EINVAL


def test_wait_timeout_hook_argument_checks(capi):
    """The failure-detection hook rejects bad modes, limits and pointers on
    the host, before any device work."""
    lib = capi.library()
    buf = ctypes.create_string_buffer(64)
    addr = ctypes.addressof(buf)
    assert lib.moe_debug_wait_timeout(2, 4, addr, None) == capi.MOE_EINVAL
    assert lib.moe_debug_wait_timeout(0, 0, addr, None) == capi.MOE_EINVAL
    assert lib.moe_debug_wait_timeout(1, capi.MOE_DEBUG_WAIT_MAX + 1, addr, None) == capi.MOE_EINVAL
    assert lib.moe_debug_wait_timeout(0, 4, None, None) == capi.MOE_EINVAL
    assert lib.moe_debug_wait_timeout(0, 4, addr + 1, None) == capi.MOE_EINVAL
