"""CPU oracle for the Purlin collectives -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``collective_datapath_atom_gb300``) never imports, links or executes it, and
this package imports nothing from the product.

The arithmetic lives in ``purlin_oracle.c`` (plain C99, nested per-rank
loops, one binary32 addition per step); this module only builds that file
with gcc and marshals numpy arrays into it.  Every function cites the
passage of "Purlin: Separating Orchestration from the Datapath of
Collectives" (§2.1, §3.1, §3.3, §C.4) or of the
"Purlin" project README that it follows; see the C file's header.

Arrays: each rank buffer is a 1-D numpy array.  fp32 data is ``np.float32``;
bf16 data is carried as its raw bits in ``np.uint16``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Sequence

import numpy as np

F32 = 0
BF16 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "purlin_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_CFLAGS = ["-O2", "-std=c99", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared"]


_OMP_LIB_PATH = os.path.join(_HERE, "liboracle_omp.so")


def build(force: bool = False, openmp: bool = False) -> str:
    """Compile ``purlin_oracle.c`` into ``liboracle.so`` beside it, or with
    ``openmp`` into ``liboracle_omp.so``: the same loops, their element
    ranges split over the host's cores (the CPU baseline's second leg)."""
    path = _OMP_LIB_PATH if openmp else _LIB_PATH
    if force or not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
        tmp = path + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, *(["-fopenmp"] if openmp else []), "-o", tmp,
                               _SRC])
        os.replace(tmp, path)
    return path


def _bind(lib):
    vpp = ctypes.POINTER(ctypes.c_void_p)
    szp = ctypes.POINTER(ctypes.c_size_t)
    lib.oracle_bf16_to_f32_bits.restype = ctypes.c_uint32
    lib.oracle_bf16_to_f32_bits.argtypes = [ctypes.c_uint16]
    lib.oracle_f32_bits_to_bf16.restype = ctypes.c_uint16
    lib.oracle_f32_bits_to_bf16.argtypes = [ctypes.c_uint32]
    lib.oracle_f32_bits_to_bf16_n.restype = None
    lib.oracle_f32_bits_to_bf16_n.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t]
    for name in ("oracle_all_gather", "oracle_reduce_scatter", "oracle_all_reduce",
                 "oracle_all_to_all"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_int, ctypes.c_size_t, ctypes.c_int, vpp, vpp]
    for name in ("oracle_all_gather_v", "oracle_reduce_scatter_v", "oracle_all_to_all_v"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_int, szp, ctypes.c_int, vpp, vpp]
    lib.oracle_threads.restype = ctypes.c_int
    lib.oracle_threads.argtypes = [ctypes.c_int]
    lib.oracle_all_reduce_one.restype = ctypes.c_int
    lib.oracle_all_reduce_one.argtypes = [ctypes.c_int, ctypes.c_size_t, ctypes.c_int, vpp,
                                          ctypes.c_void_p]
    lib.oracle_reduce_at.restype = ctypes.c_int
    lib.oracle_reduce_at.argtypes = [ctypes.c_int, ctypes.c_int, vpp, ctypes.c_size_t,
                                     ctypes.c_void_p]
    lib.oracle_all_to_all_v_source.restype = ctypes.c_int
    lib.oracle_all_to_all_v_source.argtypes = [
        ctypes.c_int, szp, ctypes.c_int, ctypes.c_size_t,
        ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_size_t)]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile a (test-modified) copy of the oracle source to ``out_path``.

    Used only by the tests that plant a mistake in the oracle to show that
    its pins catch it."""
    c_path = out_path + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", *_CFLAGS, "-o", out_path, c_path])
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


class openmp:
    """Context manager: route this module's functions to the OpenMP build
    with ``threads`` threads (0: the runtime's default) inside a ``with``
    block; ``.threads`` is the count the element loops then use."""

    def __init__(self, threads: int = 0):
        self._want = threads
        self._saved = None
        self.threads = 1

    def __enter__(self):
        global _lib
        self._saved = _lib
        _lib = _bind(ctypes.CDLL(build(openmp=True)))
        self.threads = int(_lib.oracle_threads(self._want))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


class use_library:
    """Context manager: route this module's functions to another build of the
    oracle (a planted-mistake variant) for the duration of a ``with`` block."""

    def __init__(self, path: str):
        self._path = path
        self._saved = None

    def __enter__(self):
        global _lib
        self._saved = _lib
        _lib = _bind(ctypes.CDLL(self._path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _np_dtype(dtype: int):
    return np.float32 if dtype == F32 else np.uint16


def _ptrs(arrays: Sequence[np.ndarray]):
    arr = (ctypes.c_void_p * max(1, len(arrays)))()
    for k, a in enumerate(arrays):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("oracle buffers must be contiguous")
        arr[k] = a.ctypes.data
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))


def _sizes(xs: Sequence[int]):
    arr = (ctypes.c_size_t * max(1, len(xs)))(*[int(x) for x in xs])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_size_t))


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments of {what}")


def _outs(R: int, length: int, dtype: int):
    return [np.zeros(length, dtype=_np_dtype(dtype)) for _ in range(R)]


# ---------------------------------------------------------------- codec ----

def f32_bits_to_bf16(bits: int) -> int:
    """Round-to-nearest-even binary32 -> bf16 on raw bit patterns."""
    return int(_load().oracle_f32_bits_to_bf16(int(bits) & 0xFFFFFFFF))


def f32_bits_to_bf16_array(bits: np.ndarray) -> np.ndarray:
    """Vector form of :func:`f32_bits_to_bf16` (uint32 in, uint16 out)."""
    src = np.ascontiguousarray(bits, dtype=np.uint32)
    out = np.empty(src.size, dtype=np.uint16)
    _load().oracle_f32_bits_to_bf16_n(src.ctypes.data, out.ctypes.data, src.size)
    return out


def bf16_to_f32_bits(b: int) -> int:
    return int(_load().oracle_bf16_to_f32_bits(int(b) & 0xFFFF))


# ---------------------------------------------------------- collectives ----

def all_gather(inputs: Sequence[np.ndarray], dtype: int) -> list[np.ndarray]:
    """out_d[s*n + i] = in_s[i] for every d (§2.1, §3.1 packed -> scattered)."""
    R, n = len(inputs), int(inputs[0].size)
    out = _outs(R, R * n, dtype)
    _check(_load().oracle_all_gather(R, n, dtype, _ptrs(inputs), _ptrs(out)), "all_gather")
    return out


def all_gather_v(inputs: Sequence[np.ndarray], counts: Sequence[int], dtype: int):
    """out_d[D_s + i] = in_s[i], D = exclusive prefix of counts (§2.1, §C.4)."""
    R = len(inputs)
    out = _outs(R, int(sum(counts)), dtype)
    _check(_load().oracle_all_gather_v(R, _sizes(counts), dtype, _ptrs(inputs), _ptrs(out)),
           "all_gather_v")
    return out


def reduce_scatter(inputs: Sequence[np.ndarray], dtype: int) -> list[np.ndarray]:
    """out_r[i] = rnd(sum_s in_s[r*M + i]) in rank order (§3.1, §3.3)."""
    R, n = len(inputs), int(inputs[0].size)
    out = _outs(R, n // R if R else 0, dtype)
    _check(_load().oracle_reduce_scatter(R, n, dtype, _ptrs(inputs), _ptrs(out)),
           "reduce_scatter")
    return out


def reduce_scatter_v(inputs: Sequence[np.ndarray], counts: Sequence[int], dtype: int):
    """out_r[i] = rnd(sum_s in_s[D_r + i]), i < counts[r] (§C.4, §3.3)."""
    R = len(inputs)
    out = [np.zeros(int(c), dtype=_np_dtype(dtype)) for c in counts]
    _check(_load().oracle_reduce_scatter_v(R, _sizes(counts), dtype, _ptrs(inputs), _ptrs(out)),
           "reduce_scatter_v")
    return out


def all_reduce(inputs: Sequence[np.ndarray], dtype: int) -> list[np.ndarray]:
    """out_d[i] = rnd(sum_s in_s[i]) for every d (§3.1 scattered -> scattered)."""
    R, n = len(inputs), int(inputs[0].size)
    out = _outs(R, n, dtype)
    _check(_load().oracle_all_reduce(R, n, dtype, _ptrs(inputs), _ptrs(out)), "all_reduce")
    return out


def all_reduce_one(inputs: Sequence[np.ndarray], dtype: int) -> np.ndarray:
    """One AllReduce output, rnd(sum_s in_s[i]): every destination's value."""
    R, n = len(inputs), int(inputs[0].size)
    out = np.zeros(n, dtype=_np_dtype(dtype))
    _check(_load().oracle_all_reduce_one(R, n, dtype, _ptrs(inputs),
                                         ctypes.c_void_p(out.ctypes.data)), "all_reduce_one")
    return out


def all_to_all(inputs: Sequence[np.ndarray], dtype: int) -> list[np.ndarray]:
    """out_d[s*M + i] = in_s[d*M + i] (§3.1 scattered -> transposed)."""
    R, n = len(inputs), int(inputs[0].size)
    out = _outs(R, n, dtype)
    _check(_load().oracle_all_to_all(R, n, dtype, _ptrs(inputs), _ptrs(out)), "all_to_all")
    return out


def all_to_all_v(inputs: Sequence[np.ndarray], C: np.ndarray, dtype: int):
    """out_d[Q_d[s] + i] = in_s[S_s[d] + i], i < C[s][d] (§2.1, §C.4)."""
    R = len(inputs)
    C = np.ascontiguousarray(np.asarray(C, dtype=np.uint64).reshape(R, R))
    out = [np.zeros(int(C[:, d].sum()), dtype=_np_dtype(dtype)) for d in range(R)]
    _check(_load().oracle_all_to_all_v(R, _sizes(C.reshape(-1).tolist()), dtype,
                                       _ptrs(inputs), _ptrs(out)), "all_to_all_v")
    return out


# -------------------------------------------------------- point checks ----

def reduce_at(inputs: Sequence[np.ndarray], dtype: int, idx: int):
    """One reduced element rnd(sum_s in_s[idx]) as a numpy scalar of the dtype."""
    out = np.zeros(1, dtype=_np_dtype(dtype))
    _check(_load().oracle_reduce_at(len(inputs), dtype, _ptrs(inputs), int(idx),
                                    ctypes.c_void_p(out.ctypes.data)), "reduce_at")
    return out[0]


def all_to_all_v_source(C: np.ndarray, d: int, j: int) -> tuple[int, int]:
    """(source rank, source index) of AllToAllV output element out_d[j]."""
    C = np.asarray(C, dtype=np.uint64).reshape(-1)
    R = int(round(len(C) ** 0.5))
    s, i = ctypes.c_int(), ctypes.c_size_t()
    _check(_load().oracle_all_to_all_v_source(R, _sizes(C.tolist()), int(d), int(j),
                                              ctypes.byref(s), ctypes.byref(i)),
           "all_to_all_v_source")
    return s.value, i.value
