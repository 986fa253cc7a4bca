"""Binding of ``libpurlin_examples.so``: kernels written against the
device-side API (``include/purlin_device.cuh``), launched through the C entry
points of ``device_examples.h``.  Argument marshalling only."""
from __future__ import annotations

import ctypes
import os

from .. import (_addr, _ok, _ptr_array, _stream_handle, _VPP, purlin_device_coll,
                purlin_packet_channel)

LIB_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "libpurlin_examples.so")

_DC = ctypes.POINTER(purlin_device_coll)
_SIGNATURES = {
    "purlin_example_collective": (ctypes.c_int, [_DC, ctypes.c_int, ctypes.c_void_p]),
    "purlin_example_relu_collective": (ctypes.c_int, [_DC, ctypes.c_size_t, ctypes.c_int,
                                                      ctypes.c_void_p]),
    "purlin_example_subset": (ctypes.c_int, [_DC, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                                             ctypes.c_int, ctypes.c_void_p]),
    "purlin_example_atom_copy": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                                ctypes.c_size_t, ctypes.c_void_p,
                                                ctypes.c_void_p]),
    "purlin_example_atom_reduce": (ctypes.c_int, [ctypes.c_void_p, _VPP, ctypes.c_int,
                                                  ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int,
                                                  ctypes.c_void_p, ctypes.c_void_p]),
    "purlin_example_atom_smem_bytes": (ctypes.c_size_t, []),
    "purlin_example_packet_stream": (ctypes.c_int, [
        ctypes.POINTER(purlin_packet_channel), _VPP, _VPP, ctypes.c_int, ctypes.c_size_t,
        ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "purlin_example_packet_stream_threads": (ctypes.c_int, []),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build the package first")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()


def collective(desc, threads: int = 0, stream=None):
    _ok(lib.purlin_example_collective(ctypes.byref(desc), int(threads),
                                      ctypes.c_void_p(_stream_handle(stream))),
        "purlin_example_collective")


def relu_collective(desc, n: int, threads: int = 0, stream=None):
    _ok(lib.purlin_example_relu_collective(ctypes.byref(desc), int(n), int(threads),
                                           ctypes.c_void_p(_stream_handle(stream))),
        "purlin_example_relu_collective")


def subset(desc, extra_blocks: int, fill, words: int, threads: int = 0, stream=None):
    _ok(lib.purlin_example_subset(ctypes.byref(desc), int(extra_blocks),
                                  ctypes.c_void_p(_addr(fill)), int(words), int(threads),
                                  ctypes.c_void_p(_stream_handle(stream))),
        "purlin_example_subset")


def atom_copy(dst, src, nbytes: int, bytes_per_block: int, status, stream=None):
    _ok(lib.purlin_example_atom_copy(ctypes.c_void_p(_addr(dst)), ctypes.c_void_p(_addr(src)),
                                     int(nbytes), int(bytes_per_block),
                                     ctypes.c_void_p(_addr(status)),
                                     ctypes.c_void_p(_stream_handle(stream))),
        "purlin_example_atom_copy")


def atom_reduce(dst, srcs, elems: int, elems_per_block: int, dtype: int, status, stream=None):
    ps, _keep = _ptr_array(srcs)
    _ok(lib.purlin_example_atom_reduce(ctypes.c_void_p(_addr(dst)), ps, len(srcs), int(elems),
                                       int(elems_per_block), int(dtype),
                                       ctypes.c_void_p(_addr(status)),
                                       ctypes.c_void_p(_stream_handle(stream))),
        "purlin_example_atom_reduce")


def atom_smem_bytes() -> int:
    return int(lib.purlin_example_atom_smem_bytes())


def packet_stream(ch, src, dst, n: int, dtype: int, relu: bool = True, stream=None):
    """Producer CTAs compute the rank-order sum of relu(src) per 8-byte unit
    and stream it through the packet channel; consumer CTAs write it to every
    dst (device_examples.h)."""
    ps, _k1 = _ptr_array(src)
    pd, _k2 = _ptr_array(dst)
    _ok(lib.purlin_example_packet_stream(ctypes.byref(ch), ps, pd, len(src), int(n), int(dtype),
                                         1 if relu else 0,
                                         ctypes.c_void_p(_stream_handle(stream))),
        "purlin_example_packet_stream")


def packet_stream_threads() -> int:
    return int(lib.purlin_example_packet_stream_threads())
