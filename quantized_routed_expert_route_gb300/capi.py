"""Thin ctypes binding of the C ABI in include/qre_moe.h (same names, same arguments).

Pointers are passed as Python ints (device or host addresses), streams as
ints (a cudaStream_t; 0 = the legacy default stream).  Nothing here computes:
every step of the decode path runs in the library's kernels.  Importing this
module fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

from .build import lib_path

MOE_BF16, MOE_Q8_0, MOE_Q4_K, MOE_NVFP4, MOE_Q6_K, MOE_Q4_0 = 0, 1, 2, 3, 4, 5
MOE_Q4_1, MOE_Q5_0, MOE_Q5_1, MOE_Q5_K, MOE_MXFP4, MOE_F16, MOE_F32 = 6, 7, 8, 9, 10, 11, 12
MOE_OK, MOE_EINVAL, MOE_EUNSUPPORTED, MOE_ENOMEM, MOE_ECUDA, MOE_EDEVICE = 0, -1, -2, -3, -4, -5
MOE_DEVERR_BAD_ID, MOE_DEVERR_TIMEOUT = 1, 2
MOE_SRC_HOST, MOE_SRC_DEVICE, MOE_SRC_DEVICE_BORROW = 0, 1, 2
MOE_MAX_E, MOE_MAX_TOPK, MOE_DECODE_T_CHUNK, MOE_LINEAR_MAX_T = 1024, 32, 64, 8
MOE_PREFILL_W4A4, MOE_PREFILL_W4A8, MOE_PREFILL_FP16, MOE_PREFILL_W4A4_FIXED = 0, 1, 2, 3
MOE_GLU_SILU, MOE_GLU_GELU_TANH = 0, 1
MOE_NOALLOC_WS_BYTES = 4 << 20
MOE_DEBUG_WAIT_MAX = 64

# every symbol include/qre_moe.h declares
EXPORTS = (
    "moe_row_bytes", "moe_bank_create", "moe_bank_destroy", "moe_bank_geometry", "moe_bank_fold_down_scale",
    "moe_workspace_bytes", "moe_workspace_init", "moe_decode", "moe_get_error",
    "moe_status_string", "moe_last_cuda_error", "moe_quantize_q8_1",
    "moe_debug_block_dots", "moe_debug_decode_stages", "moe_decode_noalloc", "moe_debug_tc_gemm",
    "moe_debug_wait_timeout", "moe_debug_fp4_gemm",
    "moe_prefill_workspace_bytes", "moe_prefill_grouped", "moe_debug_prefill_stages",
    "moe_decode_kernel_count", "moe_decode_io_bytes", "moe_decode_io_offsets", "moe_decode_host",
    "moe_linear", "moe_cache_plan", "moe_slot_table_create", "moe_slot_table_destroy", "moe_slot_table_acquire",
    "moe_slot_table_stats", "moe_cache_create", "moe_cache_destroy", "moe_cache_bank", "moe_cache_acquire",
    "moe_cache_stats", "moe_slot_table_invalidate", "moe_cache_invalidate", "moe_cache_bytes", "moe_cache_create_at",
    "moe_overlay_bytes", "moe_overlay_create", "moe_overlay_destroy", "moe_overlay_bank", "moe_overlay_load",
)


class moe_layer_geom(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("gate_up_type", ctypes.c_int32), ("down_type", ctypes.c_int32),
                ("glu", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {status_string(status)}"
        if status == MOE_ECUDA:
            msg += f" ({_lib.moe_last_cuda_error().decode()})"
        super().__init__(msg)


def _load() -> ctypes.CDLL:
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"the CUDA library {path} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    vp, sz, i32, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
    sig = {
        "moe_row_bytes": (sz, [i32, i64]),
        "moe_bank_create": (ctypes.c_int, [ctypes.POINTER(moe_layer_geom), vp, sz, vp, sz, vp, i32, vp,
                                           ctypes.POINTER(vp)]),
        "moe_bank_destroy": (ctypes.c_int, [vp]),
        "moe_bank_geometry": (ctypes.c_int, [vp, ctypes.POINTER(moe_layer_geom)]),
        "moe_bank_fold_down_scale": (ctypes.c_int, [vp, vp, i32, vp]),
        "moe_workspace_bytes": (sz, [vp, i32]),
        "moe_workspace_init": (ctypes.c_int, [vp, sz, vp]),
        "moe_decode": (ctypes.c_int, [vp, vp, i32, vp, vp, vp, vp, sz, vp]),
        "moe_get_error": (ctypes.c_int, [vp, sz, vp, ctypes.POINTER(i32)]),
        "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "moe_last_cuda_error": (ctypes.c_char_p, []),
        "moe_quantize_q8_1": (ctypes.c_int, [vp, i64, vp, vp]),
        "moe_debug_block_dots": (ctypes.c_int, [i32, vp, i32, i32, vp, vp, vp]),
        "moe_debug_decode_stages": (ctypes.c_int, [vp, vp, i32, vp, vp, vp, vp, sz, vp, vp, vp, vp]),
        "moe_decode_noalloc": (ctypes.c_int, [vp, vp, i32, vp, vp, vp, vp]),
        "moe_debug_tc_gemm": (ctypes.c_int, [vp, vp, i32, i32, vp, vp, vp]),
        "moe_debug_wait_timeout": (ctypes.c_int, [i32, i32, vp, vp]),
        "moe_debug_fp4_gemm": (ctypes.c_int, [vp, vp, vp, vp, i32, i32, vp, vp, vp]),
        "moe_linear": (ctypes.c_int, [i32, vp, i32, i32, vp, vp, i32, vp, vp, vp]),
        "moe_cache_plan": (ctypes.c_int, [i64, i32, vp, vp, vp]),
        "moe_slot_table_create": (ctypes.c_int, [i32, ctypes.POINTER(vp)]),
        "moe_slot_table_destroy": (ctypes.c_int, [vp]),
        "moe_slot_table_acquire": (ctypes.c_int, [vp, i32, vp, i32, i32, vp, vp, vp, vp]),
        "moe_slot_table_stats": (ctypes.c_int, [vp, vp, vp]),
        "moe_cache_create": (ctypes.c_int, [ctypes.POINTER(moe_layer_geom), i32, vp, ctypes.POINTER(vp)]),
        "moe_cache_destroy": (ctypes.c_int, [vp]),
        "moe_cache_bank": (vp, [vp]),
        "moe_cache_acquire": (ctypes.c_int, [vp, i32, vp, vp, vp, i32, vp, i32, vp, vp, vp]),
        "moe_cache_stats": (ctypes.c_int, [vp, vp, vp, vp]),
        "moe_slot_table_invalidate": (ctypes.c_int, [vp]),
        "moe_cache_invalidate": (ctypes.c_int, [vp]),
        "moe_cache_bytes": (sz, [ctypes.POINTER(moe_layer_geom), i32]),
        "moe_cache_create_at": (ctypes.c_int, [ctypes.POINTER(moe_layer_geom), i32, vp, sz, vp, ctypes.POINTER(vp)]),
        "moe_overlay_bytes": (sz, [ctypes.POINTER(moe_layer_geom)]),
        "moe_overlay_create": (ctypes.c_int, [ctypes.POINTER(moe_layer_geom), vp, sz, vp, ctypes.POINTER(vp)]),
        "moe_overlay_destroy": (ctypes.c_int, [vp]),
        "moe_overlay_bank": (vp, [vp]),
        "moe_overlay_load": (ctypes.c_int, [vp, vp, i32, vp, vp, vp, vp]),
        "moe_prefill_workspace_bytes": (sz, [vp, i32, i32]),
        "moe_decode_kernel_count": (ctypes.c_int, [vp, i32]),
        "moe_decode_io_bytes": (sz, [vp, i32]),
        "moe_decode_io_offsets": (i32, [vp, i32, vp]),
        "moe_decode_host": (ctypes.c_int, [vp, vp, i32, vp, vp, vp, vp, sz, vp, sz, vp]),
        "moe_prefill_grouped": (ctypes.c_int, [vp, vp, i32, vp, vp, i32, vp, vp, sz, vp]),
        "moe_debug_prefill_stages": (ctypes.c_int, [vp, vp, i32, vp, vp, i32, vp, vp, sz, vp, vp, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    return _lib


def status_string(status: int) -> str:
    return _lib.moe_status_string(status).decode()


def _check(status: int, what: str) -> int:
    if status != MOE_OK:
        raise MoeError(status, what)
    return status


def moe_row_bytes(wtype: int, k: int) -> int:
    return int(_lib.moe_row_bytes(wtype, k))


def moe_bank_create(geom: moe_layer_geom, gate_up: int, gate_up_bytes: int, down: int, down_bytes: int,
                    scale_bank: int | None, src_kind: int, stream: int = 0) -> int:
    out = ctypes.c_void_p()
    _check(_lib.moe_bank_create(ctypes.byref(geom), gate_up, gate_up_bytes, down, down_bytes,
                                scale_bank or None, src_kind, stream or None, ctypes.byref(out)),
           "moe_bank_create")
    return out.value


def moe_bank_destroy(bank: int) -> None:
    _check(_lib.moe_bank_destroy(bank), "moe_bank_destroy")


def moe_bank_geometry(bank: int) -> moe_layer_geom:
    g = moe_layer_geom()
    _check(_lib.moe_bank_geometry(bank, ctypes.byref(g)), "moe_bank_geometry")
    return g


def moe_bank_fold_down_scale(bank: int, per_expert_scale: int, src_kind: int, stream: int = 0) -> None:
    """s_down[e] *= per_expert_scale[e] (fp32) in the bank's scale bank."""
    _check(_lib.moe_bank_fold_down_scale(bank, per_expert_scale, src_kind, stream or None),
           "moe_bank_fold_down_scale")


def moe_workspace_bytes(bank: int, max_tokens: int) -> int:
    return int(_lib.moe_workspace_bytes(bank, max_tokens))


def moe_workspace_init(ws: int, ws_bytes: int, stream: int = 0) -> None:
    _check(_lib.moe_workspace_init(ws, ws_bytes, stream or None), "moe_workspace_init")


def moe_decode(bank: int, x: int, T: int, topk_ids: int, topk_w: int, out: int, ws: int, ws_bytes: int,
               stream: int = 0) -> None:
    _check(_lib.moe_decode(bank, x, T, topk_ids, topk_w, out, ws, ws_bytes, stream or None), "moe_decode")


def moe_decode_noalloc(bank: int, x: int, T: int, topk_ids: int, topk_w: int, out: int, stream: int = 0) -> None:
    """moe_decode on the library's fixed device workspace (allocates nothing)."""
    _check(_lib.moe_decode_noalloc(bank, x, T, topk_ids, topk_w, out, stream or None), "moe_decode_noalloc")


def moe_get_error(ws: int, ws_bytes: int, stream: int = 0) -> int:
    """Returns the device error bits (0 if none) and clears them."""
    v = ctypes.c_int32(0)
    st = _lib.moe_get_error(ws, ws_bytes, stream or None, ctypes.byref(v))
    if st not in (MOE_OK, MOE_EDEVICE):
        raise MoeError(st, "moe_get_error")
    return int(v.value)


def moe_quantize_q8_1(x: int, n: int, out_blocks: int, stream: int = 0) -> None:
    _check(_lib.moe_quantize_q8_1(x, n, out_blocks, stream or None), "moe_quantize_q8_1")


def moe_debug_block_dots(wtype: int, rows: int, nrows: int, k: int, act_blocks: int, out: int,
                         stream: int = 0) -> None:
    _check(_lib.moe_debug_block_dots(wtype, rows, nrows, k, act_blocks, out, stream or None),
           "moe_debug_block_dots")


def moe_debug_decode_stages(bank: int, x: int, T: int, topk_ids: int, topk_w: int, out: int, ws: int,
                            ws_bytes: int, stream: int = 0, x_blocks: int | None = None,
                            inter: int | None = None, inter_blocks: int | None = None) -> None:
    _check(_lib.moe_debug_decode_stages(bank, x, T, topk_ids, topk_w, out, ws, ws_bytes, stream or None,
                                        x_blocks or None, inter or None, inter_blocks or None),
           "moe_debug_decode_stages")


def moe_linear(wtype: int, rows: int, N: int, K: int, row_scale: int | None, x: int, T: int, out: int,
               dev_err: int | None = None, stream: int = 0) -> None:
    """out[T, N] (bf16) = row_scale * (q8_1(x[T, K]) @ W[N, K]^T) for quantized rows W."""
    _check(_lib.moe_linear(wtype, rows, N, K, row_scale or None, x, T, out, dev_err or None, stream or None),
           "moe_linear")


def moe_cache_plan(budget_bytes: int, expert_bytes, selections) -> list:
    """Slots per geometry for a byte budget (see include/qre_moe.h)."""
    n = len(expert_bytes)
    eb = (ctypes.c_int64 * n)(*expert_bytes)
    sel = (ctypes.c_int64 * n)(*selections)
    out = (ctypes.c_int64 * n)()
    _check(_lib.moe_cache_plan(budget_bytes, n, eb, sel, out), "moe_cache_plan")
    return [int(v) for v in out]


class SlotTable:
    """The host LRU state of one slot pool (moe_slot_table)."""

    def __init__(self, nslots: int):
        h = ctypes.c_void_p()
        _check(_lib.moe_slot_table_create(nslots, ctypes.byref(h)), "moe_slot_table_create")
        self.h, self.nslots = h.value, nslots

    def acquire(self, layer: int, ids, E: int):
        """(slot per id, [(slot, expert) to fill]) for one request."""
        n = len(ids)
        a = (ctypes.c_int32 * max(n, 1))(*ids)
        slots = (ctypes.c_int32 * max(n, 1))()
        fs = (ctypes.c_int32 * self.nslots)()
        fe = (ctypes.c_int32 * self.nslots)()
        nf = ctypes.c_int32(0)
        _check(_lib.moe_slot_table_acquire(self.h, layer, a, n, E, slots, fs, fe, ctypes.byref(nf)),
               "moe_slot_table_acquire")
        return [int(slots[i]) for i in range(n)], [(int(fs[i]), int(fe[i])) for i in range(nf.value)]

    def stats(self):
        h, m = ctypes.c_int64(0), ctypes.c_int64(0)
        _check(_lib.moe_slot_table_stats(self.h, ctypes.byref(h), ctypes.byref(m)), "moe_slot_table_stats")
        return int(h.value), int(m.value)

    def invalidate(self):
        _check(_lib.moe_slot_table_invalidate(self.h), "moe_slot_table_invalidate")

    def close(self):
        if self.h:
            _lib.moe_slot_table_destroy(self.h)
            self.h = None


def moe_cache_create(geom: moe_layer_geom, nslots: int, stream: int = 0) -> int:
    out = ctypes.c_void_p()
    _check(_lib.moe_cache_create(ctypes.byref(geom), nslots, stream or None, ctypes.byref(out)), "moe_cache_create")
    return out.value


def moe_cache_destroy(cache: int) -> None:
    _check(_lib.moe_cache_destroy(cache), "moe_cache_destroy")


def moe_cache_bytes(geom: moe_layer_geom, nslots: int) -> int:
    return int(_lib.moe_cache_bytes(ctypes.byref(geom), nslots))


def moe_cache_create_at(geom: moe_layer_geom, nslots: int, base: int, nbytes: int, stream: int = 0) -> int:
    """A pool carved from caller device memory [base, base + nbytes)."""
    out = ctypes.c_void_p()
    _check(_lib.moe_cache_create_at(ctypes.byref(geom), nslots, base, nbytes, stream or None, ctypes.byref(out)),
           "moe_cache_create_at")
    return out.value


def moe_cache_invalidate(cache: int) -> None:
    _check(_lib.moe_cache_invalidate(cache), "moe_cache_invalidate")


def moe_overlay_bytes(geom: moe_layer_geom) -> int:
    return int(_lib.moe_overlay_bytes(ctypes.byref(geom)))


def moe_overlay_create(geom: moe_layer_geom, base: int, nbytes: int, stream: int = 0) -> int:
    out = ctypes.c_void_p()
    _check(_lib.moe_overlay_create(ctypes.byref(geom), base, nbytes, stream or None, ctypes.byref(out)),
           "moe_overlay_create")
    return out.value


def moe_overlay_destroy(overlay: int) -> None:
    _check(_lib.moe_overlay_destroy(overlay), "moe_overlay_destroy")


def moe_overlay_bank(overlay: int) -> int:
    return _lib.moe_overlay_bank(overlay)


def moe_overlay_load(overlay: int, pools, gate_up: int, down: int, scales: int | None, stream: int = 0) -> None:
    """Invalidate the overlapping pools, then copy one layer's rows into the overlay."""
    arr = (ctypes.c_void_p * max(len(pools), 1))(*pools)
    _check(_lib.moe_overlay_load(overlay, arr, len(pools), gate_up, down, scales or None, stream or None),
           "moe_overlay_load")


def moe_cache_bank(cache: int) -> int:
    return _lib.moe_cache_bank(cache)


def moe_cache_acquire(cache: int, layer: int, gate_up: int, down: int, scales: int | None, E: int, ids,
                      stream: int = 0):
    """Slot ids for one request's expert ids (host list) and the number of misses."""
    n = len(ids)
    a = (ctypes.c_int32 * max(n, 1))(*ids)
    slots = (ctypes.c_int32 * max(n, 1))()
    nf = ctypes.c_int32(0)
    _check(_lib.moe_cache_acquire(cache, layer, gate_up, down, scales or None, E, a, n, slots, ctypes.byref(nf),
                                  stream or None), "moe_cache_acquire")
    return [int(slots[i]) for i in range(n)], int(nf.value)


def moe_cache_stats(cache: int):
    h, m, b = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
    _check(_lib.moe_cache_stats(cache, ctypes.byref(h), ctypes.byref(m), ctypes.byref(b)), "moe_cache_stats")
    return int(h.value), int(m.value), int(b.value)


def moe_debug_wait_timeout(mode: int, limit: int, dev_err: int, stream: int = 0) -> None:
    """A bounded wait that runs out (failure-detection check); see include/qre_moe.h."""
    _check(_lib.moe_debug_wait_timeout(mode, limit, dev_err, stream or None), "moe_debug_wait_timeout")


def moe_debug_fp4_gemm(A: int, sA: int, B: int, sB: int, K: int, N: int, D: int, dev_err: int,
                       stream: int = 0) -> None:
    """One block-scaled FP4 tensor-core tile (see include/qre_moe.h)."""
    _check(_lib.moe_debug_fp4_gemm(A, sA, B, sB, K, N, D, dev_err, stream or None), "moe_debug_fp4_gemm")


def moe_debug_tc_gemm(A: int, B: int, K: int, N: int, D: int, dev_err: int, stream: int = 0) -> None:
    """D[128, N] = A[128, K] @ B[N, K]^T (fp16 in, fp32 out) on the tcgen05 tensor cores."""
    _check(_lib.moe_debug_tc_gemm(A, B, K, N, D, dev_err, stream or None), "moe_debug_tc_gemm")


def moe_prefill_workspace_bytes(bank: int, T: int, mode: int) -> int:
    return int(_lib.moe_prefill_workspace_bytes(bank, T, mode))


def moe_prefill_grouped(bank: int, x: int, T: int, topk_ids: int, topk_w: int, mode: int, out: int, ws: int,
                        ws_bytes: int, stream: int = 0) -> None:
    _check(_lib.moe_prefill_grouped(bank, x, T, topk_ids, topk_w, mode, out, ws, ws_bytes, stream or None),
           "moe_prefill_grouped")


def moe_debug_prefill_stages(bank: int, x: int, T: int, topk_ids: int, topk_w: int, mode: int, out: int, ws: int,
                             ws_bytes: int, stream: int = 0, xq: int | None = None, off: int | None = None,
                             perm: int | None = None, i16: int | None = None) -> None:
    _check(_lib.moe_debug_prefill_stages(bank, x, T, topk_ids, topk_w, mode, out, ws, ws_bytes, stream or None,
                                         xq or None, off or None, perm or None, i16 or None),
           "moe_debug_prefill_stages")


def moe_decode_kernel_count(bank: int, T: int) -> int:
    n = int(_lib.moe_decode_kernel_count(bank, T))
    if n < 0:
        raise MoeError(n, "moe_decode_kernel_count")
    return n


def moe_decode_io_bytes(bank: int, T: int) -> int:
    return int(_lib.moe_decode_io_bytes(bank, T))


def moe_decode_io_offsets(bank: int, T: int) -> tuple:
    """(ids, weights, out) byte offsets of the host-buffer staging layout; x is at 0."""
    offs = (ctypes.c_size_t * 3)()
    _check(_lib.moe_decode_io_offsets(bank, T, ctypes.addressof(offs)), "moe_decode_io_offsets")
    return int(offs[0]), int(offs[1]), int(offs[2])


def moe_decode_host(bank: int, x: int, T: int, topk_ids: int, topk_w: int, out: int, io: int, io_bytes: int, ws: int,
                    ws_bytes: int, stream: int = 0) -> None:
    """moe_decode with x, ids, weights and out in (pinned) host memory; io is device staging."""
    _check(_lib.moe_decode_host(bank, x, T, topk_ids, topk_w, out, io, io_bytes, ws, ws_bytes, stream or None),
           "moe_decode_host")
