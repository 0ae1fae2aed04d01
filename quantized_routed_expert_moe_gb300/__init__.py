"""Python binding of the GB300 routed-MoE library (ctypes over ``include/moe.h``).

Argument marshalling only: every step of the computation runs in the CUDA
library ``_build/libmoe_gb300.so``. Importing this module does not build or
fall back to anything; calling into it without the built library raises.

Functions keep the C names (``moe_layer_create``, ``moe_route``,
``moe_decode``, ``moe_prefill_chunk``, ``moe_decode_tokens_host``,
``moe_cache_stage`` ...). Pointer arguments accept a torch tensor (its
``data_ptr()``), a numpy array, a raw integer address or None.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libmoe_gb300.so")

MOE_ABI_VERSION = 1
MOE_F32, MOE_BF16 = 0, 1
MOE_W_F32, MOE_W_Q8G64, MOE_W_Q4G64, MOE_W_Q2G64 = 0, 1, 2, 3
STATUS = {0: "MOE_OK", 1: "MOE_E_INVALID", 2: "MOE_E_UNSUPPORTED", 3: "MOE_E_NOMEM",
          4: "MOE_E_CUDA", 5: "MOE_E_TIMEOUT", 6: "MOE_E_STATE", 7: "MOE_E_SOURCE"}

# every symbol include/moe.h declares
EXPORTS = ("moe_layer_create", "moe_layer_destroy", "moe_expert_record_bytes", "moe_pack_expert_record",
           "moe_layer_device_bytes", "moe_layer_set_next", "moe_layer_set_router_scoring", "moe_route", "moe_layer_selection", "moe_decode", "moe_decode_static_scratch", "moe_prefill_chunk",
           "moe_decode_tokens_host", "moe_cache_stage", "moe_cache_prefetch", "moe_cache_prefetch_stats", "moe_cache_stats", "moe_cache_residency", "moe_cache_usage", "moe_cache_pin", "moe_hottest", "moe_cache_pin_hottest", "moe_lfu_trace", "moe_lfu_trace_pinned",
           "moe_profile_start", "moe_profile_stop", "moe_layer_set_option", "moe_layer_check", "moe_trace_read_split",
           "moe_status_str", "moe_last_error")

MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID = 0, 1
MOE_STATIC_SCRATCH_BYTES = 256 * 1024
MOE_OPT_TEST_STALL_SHARED, MOE_OPT_TRACE = 2, 3
MOE_OPT_HOST_TIMEOUT_MS, MOE_OPT_TEST_STALL_COPIES_MS, MOE_OPT_CACHE_DEVICE = 4, 5, 6
MOE_MAX_TOP_K = 8


class MoEError(RuntimeError):
    def __init__(self, status: int, call: str, detail: str):
        self.status = status
        super().__init__(f"{call}: {STATUS.get(status, status)}: {detail}")


class moe_qmat(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("bias", ctypes.c_void_p)]


class moe_expert(ctypes.Structure):
    _fields_ = [("gate", moe_qmat), ("up", moe_qmat), ("down", moe_qmat)]


class moe_router(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("q", moe_qmat)]


class moe_layer_desc(ctypes.Structure):
    _fields_ = [("abi_version", ctypes.c_uint32), ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("router_fmt", ctypes.c_int32), ("expert_fmt", ctypes.c_int32), ("group", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32), ("max_tokens", ctypes.c_int32), ("cache_slots", ctypes.c_int32)]


class moe_cache_stats_t(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_uint64), ("hits", ctypes.c_uint64), ("misses", ctypes.c_uint64),
                ("bytes_h2d", ctypes.c_uint64), ("stage_ns", ctypes.c_uint64)]


class moe_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_uint64), ("total_ms", ctypes.c_double)]


SOURCE_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t)

_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"CUDA library not built ({LIB_PATH} missing): run "
                    "`python -m quantized_routed_expert_moe_gb300.build` or __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            st = ctypes.c_int
            L.moe_layer_create.restype = st
            L.moe_layer_create.argtypes = [ctypes.POINTER(moe_layer_desc), ctypes.POINTER(moe_router), vp,
                                           ctypes.POINTER(moe_expert), ctypes.POINTER(moe_expert), vp,
                                           SOURCE_FN, vp, i32, ctypes.POINTER(vp)]
            L.moe_layer_destroy.restype = None
            L.moe_layer_destroy.argtypes = [vp]
            L.moe_expert_record_bytes.restype = sz
            L.moe_expert_record_bytes.argtypes = [ctypes.POINTER(moe_layer_desc)]
            L.moe_pack_expert_record.restype = st
            L.moe_pack_expert_record.argtypes = [ctypes.POINTER(moe_layer_desc), ctypes.POINTER(moe_expert), vp]
            L.moe_layer_device_bytes.restype = sz
            L.moe_layer_device_bytes.argtypes = [vp]
            L.moe_route.restype = st
            L.moe_route.argtypes = [vp, vp, i32, vp, vp, vp]
            L.moe_decode.restype = st
            L.moe_decode.argtypes = [vp, vp, vp, vp, vp]
            L.moe_decode_static_scratch.restype = st
            L.moe_decode_static_scratch.argtypes = [vp, vp, vp, vp, vp]
            L.moe_prefill_chunk.restype = st
            L.moe_prefill_chunk.argtypes = [vp, vp, i32, vp, vp, vp]
            L.moe_decode_tokens_host.restype = st
            L.moe_decode_tokens_host.argtypes = [vp, vp, i32, vp, vp]
            L.moe_cache_stage.restype = st
            L.moe_cache_stage.argtypes = [vp, vp, i32, vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]
            L.moe_cache_prefetch.restype = st
            L.moe_cache_prefetch.argtypes = [vp, vp, vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]
            L.moe_cache_prefetch_stats.restype = st
            L.moe_cache_prefetch_stats.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64)]
            L.moe_cache_stats.restype = st
            L.moe_cache_stats.argtypes = [vp, ctypes.POINTER(moe_cache_stats_t)]
            L.moe_cache_residency.restype = st
            L.moe_cache_residency.argtypes = [vp, vp]
            L.moe_cache_usage.restype = st
            L.moe_cache_usage.argtypes = [vp, vp]
            L.moe_cache_pin.restype = st
            L.moe_cache_pin.argtypes = [vp, vp, ctypes.c_int32]
            L.moe_hottest.restype = st
            L.moe_hottest.argtypes = [vp, i32, i32, vp]
            L.moe_cache_pin_hottest.restype = st
            L.moe_cache_pin_hottest.argtypes = [vp, i32]
            L.moe_lfu_trace.restype = st
            L.moe_lfu_trace.argtypes = [i32, i32, i32, i32, vp, vp, vp]
            L.moe_lfu_trace_pinned.restype = st
            L.moe_lfu_trace_pinned.argtypes = [i32, i32, i32, i32, vp, vp, i32, vp, vp, vp]
            L.moe_profile_start.restype = st
            L.moe_profile_start.argtypes = [vp, i32]
            L.moe_profile_stop.restype = st
            L.moe_profile_stop.argtypes = [vp, ctypes.POINTER(moe_kernel_time), i32, ctypes.POINTER(i32)]
            L.moe_layer_set_option.restype = st
            L.moe_layer_set_option.argtypes = [vp, i32, ctypes.c_int64]
            L.moe_layer_set_next.restype = st
            L.moe_layer_set_next.argtypes = [vp, vp]
            L.moe_layer_set_router_scoring.restype = st
            L.moe_layer_set_router_scoring.argtypes = [vp, i32, ctypes.c_float]
            L.moe_layer_check.restype = st
            L.moe_layer_check.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
            L.moe_layer_selection.restype = st
            L.moe_layer_selection.argtypes = [vp, i32, vp, vp, vp]
            L.moe_trace_read_split.restype = st
            L.moe_trace_read_split.argtypes = [vp, vp, i32]
            L.moe_status_str.restype = ctypes.c_char_p
            L.moe_status_str.argtypes = [st]
            L.moe_last_error.restype = ctypes.c_char_p
            L.moe_last_error.argtypes = []
            _lib = L
    return _lib


def _addr(a) -> int | None:
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    if hasattr(a, "ctypes"):
        return a.ctypes.data
    raise TypeError(f"cannot take the address of {type(a)}")


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream if hasattr(s, "cuda_stream") else int(s)


def _check(status: int, call: str):
    if status != 0:
        raise MoEError(status, call, moe_last_error())


def moe_status_str(status: int) -> str:
    return lib().moe_status_str(status).decode()


def moe_last_error() -> str:
    return lib().moe_last_error().decode()


# ---------------------------------------------------------------------------
# marshalling of canonical weights
# ---------------------------------------------------------------------------

def _qmat(m) -> moe_qmat:
    for a in (m.codes, m.scale, m.bias):
        assert a.flags["C_CONTIGUOUS"]
    return moe_qmat(_addr(m.codes), _addr(m.scale), _addr(m.bias))


def _expert(e) -> moe_expert:
    return moe_expert(_qmat(e.gate), _qmat(e.up), _qmat(e.down))


def make_desc(hidden, inter, n_experts, top_k=8, n_shared=1, router_fmt="f32", act="bf16",
              max_tokens=1, cache_slots=0, expert_bits=4) -> moe_layer_desc:
    return moe_layer_desc(MOE_ABI_VERSION, hidden, inter, n_experts, top_k, n_shared,
                          MOE_W_F32 if router_fmt == "f32" else MOE_W_Q8G64,
                          MOE_W_Q2G64 if expert_bits == 2 else MOE_W_Q4G64, 64,
                          MOE_BF16 if act == "bf16" else MOE_F32, max_tokens, cache_slots)


def desc_from_spec(spec, max_tokens=1, cache_slots=0) -> moe_layer_desc:
    return make_desc(spec.hidden, spec.inter, spec.n_experts, spec.top_k, spec.n_shared,
                     spec.router_fmt, spec.act, max_tokens, cache_slots, getattr(spec, "expert_bits", 4))


def moe_expert_record_bytes(desc: moe_layer_desc) -> int:
    return int(lib().moe_expert_record_bytes(ctypes.byref(desc)))


def moe_pack_expert_record(desc: moe_layer_desc, expert, dst) -> None:
    ce = _expert(expert)
    _check(lib().moe_pack_expert_record(ctypes.byref(desc), ctypes.byref(ce), _addr(dst)),
           "moe_pack_expert_record")


def moe_layer_create(desc: moe_layer_desc, router, router_bias=None, shared=None, experts=None,
                     records=None, source=None, source_user=None, device: int = 0) -> int:
    """Create a layer from canonical host arrays; returns the opaque handle."""
    r = moe_router()
    if router.fmt == "f32":
        assert router.w.flags["C_CONTIGUOUS"]
        r.w = _addr(router.w)
    else:
        r.q = _qmat(router.q)
    sh = _expert(shared) if shared is not None else None
    ex_arr = None
    if experts is not None:
        ex_arr = (moe_expert * len(experts))(*[_expert(e) for e in experts])
    rec_arr = None
    if records is not None:
        rec_arr = (ctypes.c_void_p * len(records))(*[_addr(p) for p in records])
    src = source if source is not None else SOURCE_FN()
    out = ctypes.c_void_p()
    st = lib().moe_layer_create(ctypes.byref(desc), ctypes.byref(r), _addr(router_bias),
                                ctypes.byref(sh) if sh is not None else None, ex_arr,
                                ctypes.cast(rec_arr, ctypes.c_void_p) if rec_arr is not None else None,
                                src, _addr(source_user), device, ctypes.byref(out))
    _check(st, "moe_layer_create")
    return out.value


def moe_layer_destroy(handle) -> None:
    lib().moe_layer_destroy(handle)


def moe_layer_device_bytes(handle) -> int:
    return int(lib().moe_layer_device_bytes(handle))


def moe_route(handle, x, T, ids, w, stream=None) -> None:
    _check(lib().moe_route(handle, _addr(x), T, _addr(ids), _addr(w), _stream(stream)), "moe_route")


def moe_decode(handle, x, y, y_f32=None, stream=None) -> None:
    _check(lib().moe_decode(handle, _addr(x), _addr(y), _addr(y_f32), _stream(stream)), "moe_decode")


def moe_decode_static_scratch(handle, x, y, y_f32=None, stream=None) -> None:
    """moe_decode over the library's fixed per-device scratch region; the
    library allocates nothing (the caller passes buffers it already owns)."""
    _check(lib().moe_decode_static_scratch(handle, _addr(x), _addr(y), _addr(y_f32), _stream(stream)),
           "moe_decode_static_scratch")


def moe_prefill_chunk(handle, x, T, y, y_f32=None, stream=None) -> None:
    _check(lib().moe_prefill_chunk(handle, _addr(x), T, _addr(y), _addr(y_f32), _stream(stream)),
           "moe_prefill_chunk")


def moe_decode_tokens_host(handle, x_host, T, y_host, stream=None) -> None:
    _check(lib().moe_decode_tokens_host(handle, _addr(x_host), T, _addr(y_host), _stream(stream)),
           "moe_decode_tokens_host")


def moe_cache_prefetch(handle, x, stream=None) -> tuple[int, int]:
    """Router lookahead on a streamed layer; returns (predicted already resident, fills issued)."""
    r, f = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().moe_cache_prefetch(handle, _addr(x), _stream(stream), ctypes.byref(r), ctypes.byref(f)),
           "moe_cache_prefetch")
    return r.value, f.value


def moe_cache_prefetch_stats(handle) -> dict:
    out = (ctypes.c_uint64 * 4)()
    _check(lib().moe_cache_prefetch_stats(handle, out), "moe_cache_prefetch_stats")
    return {"calls": out[0], "resident": out[1], "fills": out[2], "bytes_h2d": out[3]}


def moe_cache_stage(handle, ids, n, stream=None) -> tuple[int, int]:
    h, m = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().moe_cache_stage(handle, _addr(ids), n, _stream(stream), ctypes.byref(h), ctypes.byref(m)),
           "moe_cache_stage")
    return h.value, m.value


def moe_cache_stats(handle) -> dict:
    s = moe_cache_stats_t()
    _check(lib().moe_cache_stats(handle, ctypes.byref(s)), "moe_cache_stats")
    return {f: int(getattr(s, f)) for f, _ in moe_cache_stats_t._fields_}


def moe_lfu_trace(slots: int, n_experts: int, ids):
    """Host-only run of the cache policy: ids int32 [n_tokens][k] -> (slot, hit) arrays."""
    import numpy as _np
    ids = _np.ascontiguousarray(ids, dtype=_np.int32)
    n_tokens, k = ids.shape
    slot = _np.empty((n_tokens, k), _np.int32)
    hit = _np.empty((n_tokens, k), _np.uint8)
    _check(lib().moe_lfu_trace(slots, n_experts, k, n_tokens, ids.ctypes.data, slot.ctypes.data, hit.ctypes.data),
           "moe_lfu_trace")
    return slot, hit


def moe_lfu_trace_pinned(slots: int, n_experts: int, ids, pinned):
    """Host-only run of the cache policy with pinned experts: -> (slot, hit, usage)."""
    import numpy as _np
    ids = _np.ascontiguousarray(ids, dtype=_np.int32)
    pin = _np.ascontiguousarray(_np.asarray(pinned, dtype=_np.int32))
    n_tokens, k = ids.shape
    slot = _np.empty((n_tokens, k), _np.int32)
    hit = _np.empty((n_tokens, k), _np.uint8)
    usage = _np.zeros(n_experts, _np.uint64)
    _check(lib().moe_lfu_trace_pinned(slots, n_experts, k, n_tokens, ids.ctypes.data,
                                      pin.ctypes.data if len(pin) else None, len(pin), slot.ctypes.data,
                                      hit.ctypes.data, usage.ctypes.data), "moe_lfu_trace_pinned")
    return slot, hit, usage


def moe_cache_residency(handle, slots: int) -> list[int]:
    arr = (ctypes.c_int32 * slots)()
    _check(lib().moe_cache_residency(handle, ctypes.cast(arr, ctypes.c_void_p)), "moe_cache_residency")
    return list(arr)


def moe_cache_usage(handle, n_experts: int):
    """Per-expert selection counts of a streamed layer (numpy uint64 [n_experts])."""
    import numpy as np
    out = np.zeros(n_experts, np.uint64)
    _check(lib().moe_cache_usage(handle, ctypes.c_void_p(out.ctypes.data)), "moe_cache_usage")
    return out


def moe_cache_pin(handle, experts) -> None:
    """Pin these experts (the learning cache); an empty list unpins all."""
    import numpy as np
    ids = np.ascontiguousarray(np.asarray(experts, dtype=np.int32))
    _check(lib().moe_cache_pin(handle, ctypes.c_void_p(ids.ctypes.data) if len(ids) else None, len(ids)),
           "moe_cache_pin")


def moe_hottest(counts, n: int):
    """The n experts with the largest counts, the lower id first among equal
    counts (the library's ordering, host only)."""
    import numpy as np
    c = np.ascontiguousarray(np.asarray(counts, dtype=np.uint64))
    out = np.zeros(max(n, 0), np.int32)
    _check(lib().moe_hottest(ctypes.c_void_p(c.ctypes.data), len(c), n, ctypes.c_void_p(out.ctypes.data)),
           "moe_hottest")
    return out


def moe_cache_pin_hottest(handle, n: int) -> None:
    """Pin the n most used experts of a streamed layer so far."""
    _check(lib().moe_cache_pin_hottest(handle, n), "moe_cache_pin_hottest")


def moe_profile_start(handle, max_launches: int) -> None:
    _check(lib().moe_profile_start(handle, max_launches), "moe_profile_start")


def moe_profile_stop(handle) -> dict:
    """{kernel name: (launches, total_ms)} since moe_profile_start."""
    cap = 32
    arr = (moe_kernel_time * cap)()
    n = ctypes.c_int32()
    _check(lib().moe_profile_stop(handle, arr, cap, ctypes.byref(n)), "moe_profile_stop")
    return {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms)) for i in range(min(n.value, cap))}


def moe_layer_set_option(handle, option: int, value: int) -> None:
    _check(lib().moe_layer_set_option(handle, option, value), "moe_layer_set_option")


def moe_layer_set_next(handle, next_handle) -> None:
    _check(lib().moe_layer_set_next(handle, next_handle), "moe_layer_set_next")


def moe_layer_set_router_scoring(handle, scoring: int, routed_scaling: float = 1.0) -> None:
    _check(lib().moe_layer_set_router_scoring(handle, scoring, routed_scaling), "moe_layer_set_router_scoring")


def moe_layer_check(handle) -> tuple[int, int]:
    """(status, error bits) of device-side bounded waits since the last check."""
    bits = ctypes.c_uint32()
    st = lib().moe_layer_check(handle, ctypes.byref(bits))
    return st, bits.value


def moe_layer_selection(handle, T, ids, w, stream=None):
    """Copy the selection the last route / decode / prefill call used into
    device buffers ids int32 [T][k] and w fp32 [T][k] (enqueued on stream)."""
    _check(lib().moe_layer_selection(handle, T, _addr(ids), _addr(w), _stream(stream)), "moe_layer_selection")


MOE_TRACE_MAX_CTAS = 1024
MOE_TRACE_KERNELS = 5
SPLIT_TRACE_KERNELS = ("router", "gateup", "down", "prefill_gemm_gateup", "prefill_gemm_down")
SPLIT_TRACE_POINTS = ("start", "dependency", "main_done", "end")
PREFILL_WAIT_ROLES = ("copy", "dequant", "mma", "total")


def moe_trace_read_split(handle):
    """[kernel][cta][4]: decode stamps (ns) for kernels 0..2; for the prefill
    GEMMs (kernels 3..4) the cycles the copy, dequantiser and MMA roles waited
    and the CTA's total cycles."""
    cap = MOE_TRACE_KERNELS * MOE_TRACE_MAX_CTAS * 4
    buf = (ctypes.c_uint64 * cap)()
    _check(lib().moe_trace_read_split(handle, ctypes.cast(buf, ctypes.c_void_p), cap), "moe_trace_read_split")
    v = list(buf)
    return [[v[(kk * MOE_TRACE_MAX_CTAS + c) * 4:(kk * MOE_TRACE_MAX_CTAS + c) * 4 + 4]
             for c in range(MOE_TRACE_MAX_CTAS)] for kk in range(MOE_TRACE_KERNELS)]


class MoELayer:
    """Owns one layer handle; ``layer`` is any object with ``spec``, ``router``,
    ``router_bias``, ``shared`` and ``experts`` attributes in canonical form."""

    def __init__(self, layer, device: int = 0, max_tokens: int = 1, cache_slots: int = 0,
                 records=None, source=None):
        self.spec = layer.spec
        self.desc = desc_from_spec(layer.spec, max_tokens=max_tokens, cache_slots=cache_slots)
        self._records = records
        self._source = source
        self.handle = moe_layer_create(self.desc, layer.router, layer.router_bias, layer.shared,
                                       None if cache_slots else layer.experts, records=records,
                                       source=source, device=device)
        if getattr(layer.spec, "router_score", "softmax") == "sigmoid":
            moe_layer_set_router_scoring(self.handle, MOE_SCORE_SIGMOID, layer.spec.routed_scaling)

    def close(self):
        if getattr(self, "handle", None):
            moe_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def route(self, x, T, ids, w, stream=None):
        moe_route(self.handle, x, T, ids, w, stream)

    def decode(self, x, y, y_f32=None, stream=None):
        moe_decode(self.handle, x, y, y_f32, stream)

    def selection(self, T, ids, w, stream=None):
        moe_layer_selection(self.handle, T, ids, w, stream)

    def decode_static_scratch(self, x, y, y_f32=None, stream=None):
        moe_decode_static_scratch(self.handle, x, y, y_f32, stream)

    def prefill_chunk(self, x, T, y, y_f32=None, stream=None):
        moe_prefill_chunk(self.handle, x, T, y, y_f32, stream)

    def decode_tokens_host(self, x_host, T, y_host, stream=None):
        moe_decode_tokens_host(self.handle, x_host, T, y_host, stream)

    def cache_stage(self, ids, n, stream=None):
        return moe_cache_stage(self.handle, ids, n, stream)

    def cache_prefetch(self, x, stream=None):
        return moe_cache_prefetch(self.handle, x, stream)

    def prefetch_stats(self):
        return moe_cache_prefetch_stats(self.handle)

    def cache_stats(self):
        return moe_cache_stats(self.handle)

    def residency(self):
        return moe_cache_residency(self.handle, self.desc.cache_slots)

    def cache_usage(self):
        return moe_cache_usage(self.handle, self.desc.n_experts)

    def cache_pin(self, experts):
        moe_cache_pin(self.handle, experts)

    def pin_hottest(self, n):
        """Pin the n most used experts so far (ties: the lower id first)."""
        moe_cache_pin_hottest(self.handle, n)

    def set_option(self, option, value):
        moe_layer_set_option(self.handle, option, value)

    def set_next(self, other):
        moe_layer_set_next(self.handle, other.handle if other is not None else None)

    def set_router_scoring(self, scoring, routed_scaling=1.0):
        moe_layer_set_router_scoring(self.handle, scoring, routed_scaling)

    def check(self):
        return moe_layer_check(self.handle)

    @property
    def device_bytes(self):
        return moe_layer_device_bytes(self.handle)
