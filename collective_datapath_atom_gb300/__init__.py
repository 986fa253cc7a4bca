"""Thin Python binding of ``libpurlin.so`` (the C ABI in ``include/purlin.h``).

Argument marshalling only: every step of a collective runs in the library's
CUDA kernels.  There is no fallback: if the shared library is missing or
cannot be loaded, importing this package raises.

Buffers may be given as torch CUDA tensors or as integer device addresses.
Function names match the C ABI; a non-OK status raises :class:`PurlinError`.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpurlin.so")

PURLIN_MAX_RANKS = 64

PURLIN_F32, PURLIN_BF16 = 0, 1
PURLIN_COPY, PURLIN_SUM = 0, 1
PURLIN_PACKED, PURLIN_SCATTERED, PURLIN_TRANSPOSED = 0, 1, 2

PURLIN_OK = 0
PURLIN_ERR_INVALID_ARG = 1
PURLIN_ERR_ALIGNMENT = 2
PURLIN_ERR_UNSUPPORTED = 3
PURLIN_ERR_ALIAS = 4
PURLIN_ERR_OOM = 5
PURLIN_ERR_CUDA = 6
PURLIN_ERR_TIMEOUT = 7

(PURLIN_OPT_VARIANT, PURLIN_OPT_CROSSOVER_BYTES, PURLIN_OPT_AR_MODE, PURLIN_OPT_CHUNK_BYTES,
 PURLIN_OPT_STAGES, PURLIN_OPT_CTAS, PURLIN_OPT_SPIN_TIMEOUT_NS, PURLIN_OPT_DROP_NOTIFY,
 PURLIN_OPT_LAT_CTAS, PURLIN_OPT_LAT_BLOCK, PURLIN_OPT_CONSUMER_WARPS,
 PURLIN_OPT_COPY_STORES) = range(12)

(PURLIN_COLL_ALL_REDUCE, PURLIN_COLL_REDUCE_SCATTER, PURLIN_COLL_ALL_GATHER,
 PURLIN_COLL_ALL_TO_ALL, PURLIN_COLL_ALL_GATHER_V, PURLIN_COLL_REDUCE_SCATTER_V,
 PURLIN_COLL_ALL_TO_ALL_V) = range(7)

# The one legal (op, layout) pair of each collective
# ("Purlin: Separating Orchestration from the Datapath of Collectives" §3.1).
LAYOUTS = {
    "all_reduce": (PURLIN_SUM, (PURLIN_SCATTERED, PURLIN_SCATTERED)),
    "reduce_scatter": (PURLIN_SUM, (PURLIN_SCATTERED, PURLIN_PACKED)),
    "all_gather": (PURLIN_COPY, (PURLIN_PACKED, PURLIN_SCATTERED)),
    "all_to_all": (PURLIN_COPY, (PURLIN_SCATTERED, PURLIN_TRANSPOSED)),
    "all_gather_v": (PURLIN_COPY, (PURLIN_PACKED, PURLIN_SCATTERED)),
    "reduce_scatter_v": (PURLIN_SUM, (PURLIN_SCATTERED, PURLIN_PACKED)),
    "all_to_all_v": (PURLIN_COPY, (PURLIN_SCATTERED, PURLIN_TRANSPOSED)),
}


class purlin_layout(ctypes.Structure):
    _fields_ = [("in_", ctypes.c_int32), ("out", ctypes.c_int32)]


class purlin_launch_info(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("grid", ctypes.c_int32), ("block", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("chunk_bytes", ctypes.c_int64),
                ("chunks", ctypes.c_int64), ("units", ctypes.c_int64),
                ("segments", ctypes.c_int64), ("smem_bytes", ctypes.c_int64),
                ("epoch", ctypes.c_uint64), ("epoch_next", ctypes.c_uint64)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class purlin_segment(ctypes.Structure):
    _fields_ = [("src_off", ctypes.c_uint64), ("dst_off", ctypes.c_uint64),
                ("bytes", ctypes.c_uint64), ("src_rank", ctypes.c_int32),
                ("dst_rank", ctypes.c_int32), ("skip_rank", ctypes.c_int32),
                ("src_is_dst", ctypes.c_int32), ("sync", ctypes.c_int32), ("tma", ctypes.c_int32),
                ("shift", ctypes.c_int32), ("head_bytes", ctypes.c_uint64), ("tail_bytes", ctypes.c_uint64),
                ("chunk_begin", ctypes.c_uint64), ("chunk_bytes", ctypes.c_uint64),
                ("unit_begin", ctypes.c_uint64)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class purlin_device_coll(ctypes.Structure):
    """A collective compiled for device-side calls (include/purlin.h)."""
    _fields_ = [("src", ctypes.c_void_p * PURLIN_MAX_RANKS),
                ("dst", ctypes.c_void_p * PURLIN_MAX_RANKS),
                ("segs", ctypes.c_void_p), ("flags", ctypes.c_void_p),
                ("epochs", ctypes.c_void_p), ("err", ctypes.c_void_p),
                ("nchunks", ctypes.c_uint64), ("nunits", ctypes.c_uint64),
                ("epoch_inc", ctypes.c_uint64), ("timeout_ns", ctypes.c_int64),
                ("drop_notify", ctypes.c_int64), ("flag_slots", ctypes.c_uint32),
                ("stages", ctypes.c_uint32), ("slot_stride", ctypes.c_uint32),
                ("workspace_bytes", ctypes.c_uint32), ("nseg", ctypes.c_int32),
                ("R", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("vector_copies", ctypes.c_int32), ("blocks", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("composed", ctypes.c_int32),
                ("coll", ctypes.c_int32), ("ragged", ctypes.c_int32),
                ("owner", ctypes.c_void_p)]


class purlin_packet_channel(ctypes.Structure):
    """A payload+flag packet channel between CTAs of one launch (include/purlin.h)."""
    _fields_ = [("staging", ctypes.c_void_p), ("state", ctypes.c_void_p),
                ("capacity", ctypes.c_uint64), ("timeout_ns", ctypes.c_int64),
                ("drop_unit", ctypes.c_int64), ("ctas", ctypes.c_int32),
                ("pad", ctypes.c_int32), ("owner", ctypes.c_void_p)]


class PurlinError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = int(status)
        super().__init__(f"{what}: {status_string(status)} (status {status})")


# Exported symbols and their C signatures (kept in step with include/purlin.h).
_VPP = ctypes.POINTER(ctypes.c_void_p)
_SZP = ctypes.POINTER(ctypes.c_size_t)
_CTX = ctypes.c_void_p
_SIGNATURES = {
    "purlin_init": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(_CTX)]),
    "purlin_finalize": (ctypes.c_int, [_CTX]),
    "purlin_set_stream": (ctypes.c_int, [_CTX, ctypes.c_void_p]),
    "purlin_all_reduce": (ctypes.c_int, [_CTX, _VPP, _VPP, ctypes.c_size_t, ctypes.c_int,
                                         ctypes.c_int, purlin_layout]),
    "purlin_reduce_scatter": (ctypes.c_int, [_CTX, _VPP, _VPP, ctypes.c_size_t, ctypes.c_int,
                                             ctypes.c_int, purlin_layout]),
    "purlin_all_gather": (ctypes.c_int, [_CTX, _VPP, _VPP, ctypes.c_size_t, ctypes.c_int,
                                         ctypes.c_int, purlin_layout]),
    "purlin_all_to_all": (ctypes.c_int, [_CTX, _VPP, _VPP, ctypes.c_size_t, ctypes.c_int,
                                         ctypes.c_int, purlin_layout]),
    "purlin_all_gather_v": (ctypes.c_int, [_CTX, _VPP, _VPP, _SZP, ctypes.c_int, ctypes.c_int,
                                           purlin_layout]),
    "purlin_reduce_scatter_v": (ctypes.c_int, [_CTX, _VPP, _VPP, _SZP, ctypes.c_int,
                                               ctypes.c_int, purlin_layout]),
    "purlin_all_to_all_v": (ctypes.c_int, [_CTX, _VPP, _VPP, _SZP, ctypes.c_int, ctypes.c_int,
                                           purlin_layout]),
    "purlin_all_gather_v_device_counts": (ctypes.c_int, [
        _CTX, _VPP, _VPP, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int,
        ctypes.c_int, purlin_layout]),
    "purlin_reduce_scatter_v_device_counts": (ctypes.c_int, [
        _CTX, _VPP, _VPP, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int,
        ctypes.c_int, purlin_layout]),
    "purlin_all_to_all_v_device_counts": (ctypes.c_int, [
        _CTX, _VPP, _VPP, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int,
        ctypes.c_int, purlin_layout]),
    "purlin_all_reduce_noalloc": (ctypes.c_int, [ctypes.c_int, _VPP, _VPP, ctypes.c_size_t,
                                                 ctypes.c_int, ctypes.c_int, purlin_layout,
                                                 ctypes.c_void_p]),
    "purlin_noalloc_check": (ctypes.c_int, [ctypes.c_void_p]),
    "purlin_empty_launch": (ctypes.c_int, [ctypes.c_void_p]),
    "purlin_touch_launch": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "purlin_check": (ctypes.c_int, [_CTX]),
    "purlin_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "purlin_set_option": (ctypes.c_int, [_CTX, ctypes.c_int, ctypes.c_int64]),
    "purlin_get_option": (ctypes.c_int, [_CTX, ctypes.c_int, ctypes.POINTER(ctypes.c_int64)]),
    "purlin_last_launch": (ctypes.c_int, [_CTX, ctypes.POINTER(purlin_launch_info)]),
    "purlin_plan_inspect": (ctypes.c_int, [
        ctypes.c_int, ctypes.c_int, _VPP, _VPP, ctypes.c_size_t, _SZP, ctypes.c_int, ctypes.c_int,
        purlin_layout, ctypes.c_int, ctypes.c_int, ctypes.c_uint64,
        ctypes.POINTER(purlin_segment), ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t),
        ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]),
    "purlin_device_prepare": (ctypes.c_int, [
        _CTX, ctypes.c_int, _VPP, _VPP, ctypes.c_size_t, _SZP, ctypes.c_int, ctypes.c_int,
        purlin_layout, ctypes.c_int, ctypes.c_uint32, ctypes.POINTER(purlin_device_coll)]),
    "purlin_device_check": (ctypes.c_int, [ctypes.POINTER(purlin_device_coll), ctypes.c_void_p]),
    "purlin_device_release": (ctypes.c_int, [_CTX, ctypes.POINTER(purlin_device_coll)]),
    "purlin_device_coll_size": (ctypes.c_size_t, []),
    "purlin_packet_channel_create": (ctypes.c_int, [_CTX, ctypes.c_size_t, ctypes.c_int,
                                                    ctypes.POINTER(purlin_packet_channel)]),
    "purlin_packet_channel_check": (ctypes.c_int, [ctypes.POINTER(purlin_packet_channel),
                                                   ctypes.c_void_p]),
    "purlin_packet_channel_release": (ctypes.c_int, [_CTX, ctypes.POINTER(purlin_packet_channel)]),
}


def _load_library():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
            "g.build()'); this package has no fallback path")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load_library()


def status_string(status: int) -> str:
    return lib.purlin_status_string(int(status)).decode()


def _ok(status: int, what: str):
    if status != PURLIN_OK:
        raise PurlinError(status, what)


def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _ptr_array(bufs: Sequence):
    arr = (ctypes.c_void_p * max(1, len(bufs)))()
    for i, b in enumerate(bufs):
        arr[i] = _addr(b)
    return ctypes.cast(arr, _VPP), arr


def _size_array(xs):
    xs = [int(x) for x in xs]
    arr = (ctypes.c_size_t * max(1, len(xs)))(*xs)
    return ctypes.cast(arr, _SZP), arr


def _layout(layout):
    return purlin_layout(int(layout[0]), int(layout[1]))


def _stream_handle(stream) -> int:
    if stream is None:
        return 0
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


class Context:
    """Owns one ``purlin_ctx*``; calls ``purlin_finalize`` on close."""

    def __init__(self, handle: int, R: int):
        self.handle = ctypes.c_void_p(handle)
        self.R = R

    def close(self):
        if self.handle:
            _ok(lib.purlin_finalize(self.handle), "purlin_finalize")
            self.handle = ctypes.c_void_p(0)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False


# ----------------------------------------------------------- C ABI names ---

def purlin_init(R: int, stream=None) -> Context:
    h = ctypes.c_void_p(0)
    _ok(lib.purlin_init(int(R), ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(h)),
        "purlin_init")
    return Context(h.value, int(R))


def purlin_finalize(ctx: Context):
    ctx.close()


def purlin_set_stream(ctx: Context, stream):
    _ok(lib.purlin_set_stream(ctx.handle, ctypes.c_void_p(_stream_handle(stream))),
        "purlin_set_stream")


def _uniform(fn, name, ctx, src, dst, n, dtype, op, layout):
    dflt_op, dflt_layout = LAYOUTS[name]
    op = dflt_op if op is None else op
    layout = dflt_layout if layout is None else layout
    ps, _keep1 = _ptr_array(src)
    pd, _keep2 = _ptr_array(dst)
    _ok(fn(ctx.handle, ps, pd, int(n), int(dtype), int(op), _layout(layout)), f"purlin_{name}")


def _varlen(fn, name, ctx, src, dst, counts, dtype, op, layout):
    dflt_op, dflt_layout = LAYOUTS[name]
    op = dflt_op if op is None else op
    layout = dflt_layout if layout is None else layout
    ps, _keep1 = _ptr_array(src)
    pd, _keep2 = _ptr_array(dst)
    pc, _keep3 = _size_array(counts)
    _ok(fn(ctx.handle, ps, pd, pc, int(dtype), int(op), _layout(layout)), f"purlin_{name}")


def purlin_all_reduce(ctx, src, dst, n, dtype, op=None, layout=None):
    _uniform(lib.purlin_all_reduce, "all_reduce", ctx, src, dst, n, dtype, op, layout)


def purlin_reduce_scatter(ctx, src, dst, n, dtype, op=None, layout=None):
    _uniform(lib.purlin_reduce_scatter, "reduce_scatter", ctx, src, dst, n, dtype, op, layout)


def purlin_all_gather(ctx, src, dst, n, dtype, op=None, layout=None):
    _uniform(lib.purlin_all_gather, "all_gather", ctx, src, dst, n, dtype, op, layout)


def purlin_all_to_all(ctx, src, dst, n, dtype, op=None, layout=None):
    _uniform(lib.purlin_all_to_all, "all_to_all", ctx, src, dst, n, dtype, op, layout)


def purlin_all_gather_v(ctx, src, dst, counts, dtype, op=None, layout=None):
    _varlen(lib.purlin_all_gather_v, "all_gather_v", ctx, src, dst, counts, dtype, op, layout)


def purlin_reduce_scatter_v(ctx, src, dst, counts, dtype, op=None, layout=None):
    _varlen(lib.purlin_reduce_scatter_v, "reduce_scatter_v", ctx, src, dst, counts, dtype, op,
            layout)


def purlin_all_to_all_v(ctx, src, dst, counts, dtype, op=None, layout=None):
    """``counts``: R*R element counts, row s = source, column d = destination."""
    _varlen(lib.purlin_all_to_all_v, "all_to_all_v", ctx, src, dst, counts, dtype, op, layout)


def _device_counts(fn, name, ctx, src, dst, counts, in_capacity, out_capacity, dtype, op,
                   layout):
    dflt_op, dflt_layout = LAYOUTS[name]
    op = dflt_op if op is None else op
    layout = dflt_layout if layout is None else layout
    ps, _keep1 = _ptr_array(src)
    pd, _keep2 = _ptr_array(dst)
    _ok(fn(ctx.handle, ps, pd, ctypes.c_void_p(_addr(counts)), int(in_capacity),
           int(out_capacity), int(dtype), int(op), _layout(layout)),
        f"purlin_{name}_device_counts")


def purlin_all_gather_v_device_counts(ctx, src, dst, counts, in_capacity, out_capacity, dtype,
                                      op=None, layout=None):
    """AllGatherV with the R counts in device memory (a tensor of int64 or a
    device address)."""
    _device_counts(lib.purlin_all_gather_v_device_counts, "all_gather_v", ctx, src, dst, counts,
                   in_capacity, out_capacity, dtype, op, layout)


def purlin_reduce_scatter_v_device_counts(ctx, src, dst, counts, in_capacity, out_capacity,
                                          dtype, op=None, layout=None):
    _device_counts(lib.purlin_reduce_scatter_v_device_counts, "reduce_scatter_v", ctx, src, dst,
                   counts, in_capacity, out_capacity, dtype, op, layout)


def purlin_all_to_all_v_device_counts(ctx, src, dst, counts, in_capacity, out_capacity, dtype,
                                      op=None, layout=None):
    """AllToAllV with the R*R count matrix (row = source) in device memory."""
    _device_counts(lib.purlin_all_to_all_v_device_counts, "all_to_all_v", ctx, src, dst, counts,
                   in_capacity, out_capacity, dtype, op, layout)


def purlin_all_reduce_noalloc(R, src, dst, n, dtype, op=None, layout=None, stream=None):
    """AllReduce with no device allocation (static scratch inside the
    library); see include/purlin.h for its limits."""
    dflt_op, dflt_layout = LAYOUTS["all_reduce"]
    op = dflt_op if op is None else op
    layout = dflt_layout if layout is None else layout
    ps, _keep1 = _ptr_array(src)
    pd, _keep2 = _ptr_array(dst)
    _ok(lib.purlin_all_reduce_noalloc(int(R), ps, pd, int(n), int(dtype), int(op),
                                      _layout(layout), ctypes.c_void_p(_stream_handle(stream))),
        "purlin_all_reduce_noalloc")


def purlin_noalloc_check(stream=None):
    """Synchronize `stream` and raise if a device-side wait of an
    allocation-free AllReduce expired since the last check."""
    _ok(lib.purlin_noalloc_check(ctypes.c_void_p(_stream_handle(stream))), "purlin_noalloc_check")


def purlin_empty_launch(stream=None):
    _ok(lib.purlin_empty_launch(ctypes.c_void_p(_stream_handle(stream))), "purlin_empty_launch")


def purlin_touch_launch(src_ptr: int, dst_ptr: int, stream=None):
    _ok(lib.purlin_touch_launch(ctypes.c_void_p(src_ptr), ctypes.c_void_p(dst_ptr),
                                ctypes.c_void_p(_stream_handle(stream))), "purlin_touch_launch")


def purlin_check(ctx) -> int:
    """Synchronise and return the device status (raises on non-OK)."""
    _ok(lib.purlin_check(ctx.handle), "purlin_check")
    return PURLIN_OK


def purlin_check_status(ctx) -> int:
    """Like :func:`purlin_check` but returns the status instead of raising."""
    return int(lib.purlin_check(ctx.handle))


def purlin_set_option(ctx, opt: int, value: int):
    _ok(lib.purlin_set_option(ctx.handle, int(opt), int(value)), "purlin_set_option")


def purlin_get_option(ctx, opt: int) -> int:
    v = ctypes.c_int64(0)
    _ok(lib.purlin_get_option(ctx.handle, int(opt), ctypes.byref(v)), "purlin_get_option")
    return v.value


def purlin_last_launch(ctx) -> dict:
    info = purlin_launch_info()
    _ok(lib.purlin_last_launch(ctx.handle, ctypes.byref(info)), "purlin_last_launch")
    return info.as_dict()


def purlin_plan_inspect(coll: int, R: int, src, dst, n: int, counts, dtype: int, op: int,
                        layout, variant: int, ar_mode: int = 0, chunk_bytes: int = 0,
                        cap: int = 8192):
    """Validate + compile one call on the host.  Returns
    ``(status, segments, nchunks, nunits)``; never touches a GPU."""
    ps, _k1 = _ptr_array(src)
    pd, _k2 = _ptr_array(dst)
    if counts is None:
        pc, _k3 = None, None
    else:
        pc, _k3 = _size_array(counts)
    segs = (purlin_segment * cap)()
    nseg = ctypes.c_size_t(0)
    nch = ctypes.c_uint64(0)
    nun = ctypes.c_uint64(0)
    st = lib.purlin_plan_inspect(int(coll), int(R), ps, pd, int(n), pc, int(dtype), int(op),
                                 _layout(layout), int(variant), int(ar_mode), int(chunk_bytes),
                                 segs, cap, ctypes.byref(nseg), ctypes.byref(nch),
                                 ctypes.byref(nun))
    out = [segs[i].as_dict() for i in range(min(nseg.value, cap))] if st == PURLIN_OK else []
    return int(st), out, nch.value, nun.value


# ------------------------------------------------------ device-side API ---

COLL_NAMES = ["all_reduce", "reduce_scatter", "all_gather", "all_to_all", "all_gather_v",
              "reduce_scatter_v", "all_to_all_v"]


def purlin_device_prepare(ctx, coll: int, src, dst, n: int = 0, counts=None, dtype: int = 0,
                          op=None, layout=None, blocks: int = 1,
                          max_workspace_bytes: int = 0) -> purlin_device_coll:
    """Compile a collective for kernels that call it themselves; returns the
    descriptor to pass to them (see include/purlin.h)."""
    dflt_op, dflt_layout = LAYOUTS[COLL_NAMES[int(coll)]]
    op = dflt_op if op is None else op
    layout = dflt_layout if layout is None else layout
    ps, _k1 = _ptr_array(src)
    pd, _k2 = _ptr_array(dst)
    pc, _k3 = (None, None) if counts is None else _size_array(counts)
    d = purlin_device_coll()
    _ok(lib.purlin_device_prepare(ctx.handle, int(coll), ps, pd, int(n), pc, int(dtype), int(op),
                                  _layout(layout), int(blocks), int(max_workspace_bytes),
                                  ctypes.byref(d)), "purlin_device_prepare")
    return d


def purlin_device_check(desc: purlin_device_coll, stream=None) -> int:
    """Wait for the stream, then read and clear the descriptor's error word
    (returns the status; does not raise)."""
    return int(lib.purlin_device_check(ctypes.byref(desc),
                                       ctypes.c_void_p(_stream_handle(stream))))


def purlin_device_release(ctx, desc: purlin_device_coll):
    _ok(lib.purlin_device_release(ctx.handle, ctypes.byref(desc)), "purlin_device_release")


def purlin_packet_channel_create(ctx, capacity_bytes: int, ctas: int) -> purlin_packet_channel:
    ch = purlin_packet_channel()
    _ok(lib.purlin_packet_channel_create(ctx.handle, int(capacity_bytes), int(ctas),
                                         ctypes.byref(ch)), "purlin_packet_channel_create")
    return ch


def purlin_packet_channel_check(ch: purlin_packet_channel, stream=None) -> int:
    """Wait for the stream, then read and clear the channel's error word
    (returns the status; does not raise)."""
    return int(lib.purlin_packet_channel_check(ctypes.byref(ch),
                                               ctypes.c_void_p(_stream_handle(stream))))


def purlin_packet_channel_release(ctx, ch: purlin_packet_channel):
    _ok(lib.purlin_packet_channel_release(ctx.handle, ctypes.byref(ch)),
        "purlin_packet_channel_release")
