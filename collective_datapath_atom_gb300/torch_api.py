"""Tensor-level calls in the shape of the "Purlin" project README's Python API
("Using Purlin", Python: ``initialize``, ``all_reduce(x, out, handle,
stream)``, ``finalize``; "Deterministic Reduction": ``reduction_mode``).

One GPU holds all R ranks here, so ``x`` and ``out`` are sequences of R
tensors (rank r's input and output), not one tensor per process.  Sizes and
dtypes are read from the tensors; everything else is the C ABI through the
ctypes binding, so this module only marshals arguments.

    h = initialize(8, stream=torch.cuda.current_stream())
    all_reduce(xs, outs, h)                  # every outs[r] = sum over s of xs[s]
    finalize(h)
"""
from __future__ import annotations

import enum
from typing import Sequence

from . import (PURLIN_BF16, PURLIN_F32, Context, _stream_handle, purlin_all_gather,
               purlin_all_gather_v, purlin_all_reduce, purlin_all_to_all, purlin_all_to_all_v,
               purlin_check, purlin_finalize, purlin_init, purlin_reduce_scatter,
               purlin_reduce_scatter_v, purlin_set_stream)


class ReductionMode(enum.Enum):
    """The README's reduction modes.  Only the deterministic one exists on one
    GPU (no NVLink SHARP): sums are taken in rank order in binary32 and
    rounded once."""
    DETERMINISTIC = "deterministic"
    NON_DETERMINISTIC = "non_deterministic"


def _dtype_of(tensors: Sequence) -> int:
    import torch

    kinds = {t.dtype for t in tensors}
    if len(kinds) != 1:
        raise TypeError(f"all rank tensors must share one dtype, got {sorted(map(str, kinds))}")
    dt = kinds.pop()
    if dt == torch.float32:
        return PURLIN_F32
    if dt in (torch.bfloat16, torch.int16):   # bf16, or its raw bits
        return PURLIN_BF16
    raise TypeError(f"unsupported dtype {dt}: float32, bfloat16 (or its int16 bits)")


def _check(xs: Sequence, outs: Sequence, handle: Context):
    if len(xs) != handle.R or len(outs) != handle.R:
        raise ValueError(f"expected {handle.R} input and output tensors, got {len(xs)} and "
                         f"{len(outs)}")
    for t in list(xs) + list(outs):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("rank tensors must be contiguous CUDA tensors")
    d = _dtype_of(list(xs) + list(outs))
    return d


def _uniform_numel(xs: Sequence) -> int:
    n = {int(t.numel()) for t in xs}
    if len(n) != 1:
        raise ValueError("every rank's input must hold the same number of elements")
    return n.pop()


def _on(handle: Context, stream):
    """Switch the handle to `stream` if it names another stream (the switch
    waits for the previous stream, so it is skipped when nothing changes)."""
    if stream is None:
        return
    h = _stream_handle(stream)
    if h != getattr(handle, "stream_handle", None):
        purlin_set_stream(handle, stream)
        handle.stream_handle = h


def initialize(R: int, stream=None) -> Context:
    """A context for R rank buffers on the current CUDA device."""
    handle = purlin_init(R, stream)
    handle.stream_handle = _stream_handle(stream)
    return handle


def finalize(handle: Context, stream=None):
    _on(handle, stream)
    purlin_finalize(handle)


def check(handle: Context) -> None:
    """Wait for the handle's stream and raise if a device-side wait expired."""
    purlin_check(handle)


def all_reduce(xs, outs, handle, stream=None, reduction_mode=ReductionMode.DETERMINISTIC):
    if reduction_mode is not ReductionMode.DETERMINISTIC:
        raise NotImplementedError("only the deterministic reduction exists on one GPU")
    d = _check(xs, outs, handle)
    n = _uniform_numel(xs)
    if any(int(o.numel()) != n for o in outs):
        raise ValueError("AllReduce outputs hold as many elements as the inputs")
    _on(handle, stream)
    purlin_all_reduce(handle, xs, outs, n, d)


def reduce_scatter(xs, outs, handle, stream=None, reduction_mode=ReductionMode.DETERMINISTIC):
    if reduction_mode is not ReductionMode.DETERMINISTIC:
        raise NotImplementedError("only the deterministic reduction exists on one GPU")
    d = _check(xs, outs, handle)
    n = _uniform_numel(xs)
    if n % handle.R or any(int(o.numel()) != n // handle.R for o in outs):
        raise ValueError("ReduceScatter: inputs of n elements (n divisible by R), outputs of n/R")
    _on(handle, stream)
    purlin_reduce_scatter(handle, xs, outs, n, d)


def all_gather(xs, outs, handle, stream=None):
    d = _check(xs, outs, handle)
    n = _uniform_numel(xs)
    if any(int(o.numel()) != handle.R * n for o in outs):
        raise ValueError("AllGather outputs hold R times the input elements")
    _on(handle, stream)
    purlin_all_gather(handle, xs, outs, n, d)


def all_to_all(xs, outs, handle, stream=None):
    d = _check(xs, outs, handle)
    n = _uniform_numel(xs)
    if n % handle.R or any(int(o.numel()) != n for o in outs):
        raise ValueError("AllToAll: inputs and outputs of n elements, n divisible by R")
    _on(handle, stream)
    purlin_all_to_all(handle, xs, outs, n, d)


def all_gather_v(xs, outs, handle, stream=None):
    """Rank r contributes xs[r] (any length); every output holds all of them."""
    d = _check(xs, outs, handle)
    counts = [int(t.numel()) for t in xs]
    if any(int(o.numel()) != sum(counts) for o in outs):
        raise ValueError("AllGatherV outputs hold the sum of the input lengths")
    _on(handle, stream)
    purlin_all_gather_v(handle, xs, outs, counts, d)


def reduce_scatter_v(xs, outs, handle, stream=None, reduction_mode=ReductionMode.DETERMINISTIC):
    """outs[r] receives the rank-order sum of block r; block lengths are the
    output lengths, and every input holds their total."""
    if reduction_mode is not ReductionMode.DETERMINISTIC:
        raise NotImplementedError("only the deterministic reduction exists on one GPU")
    d = _check(xs, outs, handle)
    counts = [int(o.numel()) for o in outs]
    if any(int(t.numel()) != sum(counts) for t in xs):
        raise ValueError("ReduceScatterV inputs hold the sum of the output lengths")
    _on(handle, stream)
    purlin_reduce_scatter_v(handle, xs, outs, counts, d)


def all_to_all_v(xs, outs, counts, handle, stream=None):
    """counts: R x R element counts (row = source, column = destination), as a
    nested sequence or a flat one of R*R entries."""
    d = _check(xs, outs, handle)
    R = handle.R
    flat = [int(c) for row in counts for c in (row if hasattr(row, "__iter__") else [row])]
    if len(flat) != R * R:
        raise ValueError(f"AllToAllV needs {R * R} counts")
    for s in range(R):
        if int(xs[s].numel()) < sum(flat[s * R:(s + 1) * R]):
            raise ValueError(f"input {s} is shorter than its row of counts")
    for dd in range(R):
        if int(outs[dd].numel()) < sum(flat[s * R + dd] for s in range(R)):
            raise ValueError(f"output {dd} is shorter than its column of counts")
    _on(handle, stream)
    purlin_all_to_all_v(handle, xs, outs, flat, d)
