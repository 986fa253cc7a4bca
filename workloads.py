"""Seeded synthetic inputs for the Purlin collectives.

This module only draws inputs.  It holds none of the collectives' arithmetic,
so both the CPU oracle and the CUDA path can take their inputs from it.

Recipe (every array is drawn rank-major, rank 0 first, from one
``numpy.random.default_rng(seed)`` stream per workload):

* fp32 inputs are drawn directly.
* bf16 inputs are binary32 normals rounded to bf16 (nearest-even) by torch's
  CPU conversion; they are carried as raw bits in ``np.uint16``.
* The AllToAllV count matrix of the MoE-dispatch workload takes, for each
  source rank in order, ``multinomial(tokens, p)`` with Zipf destination
  weights ``p_d ~ (d+1)^-1.2``; the payload normals continue the same stream.

The workloads are the ones "Purlin: Separating Orchestration from the Datapath of Collectives"
§2.1 names (throughput-bound
prefill payloads and latency-bound decode messages) and the MoE dispatch
pattern of Table 2, shaped as single-GPU rank buffers.
"""
from __future__ import annotations

import dataclasses

import numpy as np

F32 = 0
BF16 = 1
ELEM_BYTES = {F32: 4, BF16: 2}

HIDDEN = 4096          # decode/prefill AllReduce message = batch x 4096 hidden
MOE_TOKENS = 16384     # tokens held by each rank in the AllToAllV dispatch
MOE_HIDDEN = 7168      # hidden size of each dispatched token
ZIPF_S = 1.2


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    collective: str    # all_reduce | all_gather | reduce_scatter | all_to_all_v ...
    dtype: int
    R: int
    n: int             # elements per rank input buffer
    seed: int


# The five workloads.  Names state what they are and their sizes.
AR_F32_R8_4096 = Workload("allreduce_f32_R8_n4096_intvalues", "all_reduce", F32, 8, 4096, 0)
AG_BF16_R8_8MI = Workload("allgather_bf16_R8_n8Mi", "all_gather", BF16, 8, 8 << 20, 1)
RS_BF16_R8_128MI = Workload("reducescatter_bf16_R8_n128Mi", "reduce_scatter", BF16, 8,
                            128 << 20, 2)
A2AV_BF16_R8_MOE = Workload("alltoallv_bf16_R8_16384tok_x7168_zipf1.2", "all_to_all_v", BF16,
                            8, MOE_TOKENS * MOE_HIDDEN, 3)
AR_BF16_SWEEP_BATCHES = [1 << k for k in range(16)]   # 1, 2, 4, ..., 32768


def ar_sweep_workload(batch: int) -> Workload:
    return Workload(f"allreduce_bf16_R8_b{batch}x{HIDDEN}", "all_reduce", BF16, 8,
                    batch * HIDDEN, 4)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round binary32 values to bf16 (nearest-even, torch CPU) and return raw bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def int_values_f32(seed: int, R: int, n: int, lo: int = -8, hi: int = 8) -> list[np.ndarray]:
    """Uniform integers in [lo, hi] as fp32 (sums stay exact)."""
    rng = np.random.default_rng(seed)
    return [rng.integers(lo, hi + 1, size=n).astype(np.float32) for _ in range(R)]


def int_values_bf16(seed: int, R: int, n: int, lo: int = -8, hi: int = 8) -> list[np.ndarray]:
    return [to_bf16_bits(x) for x in int_values_f32(seed, R, n, lo, hi)]


def normals(seed: int, R: int, n: int, dtype: int, rng=None) -> list[np.ndarray]:
    """R rank buffers of n N(0,1) values, rank 0 first."""
    rng = np.random.default_rng(seed) if rng is None else rng
    out = []
    for _ in range(R):
        x = rng.standard_normal(n, dtype=np.float32)
        out.append(x if dtype == F32 else to_bf16_bits(x))
    return out


def ragged_counts(seed: int, R: int, total: int, skew: float = 1.0) -> list[int]:
    """R non-negative counts summing to ``total`` (multinomial, Zipf-weighted)."""
    rng = np.random.default_rng(seed)
    w = (np.arange(R) + 1.0) ** (-skew)
    return [int(c) for c in rng.multinomial(total, w / w.sum())]


def zipf_weights(R: int, s: float = ZIPF_S) -> np.ndarray:
    w = (np.arange(R, dtype=np.float64) + 1.0) ** (-s)
    return w / w.sum()


def moe_dispatch(seed: int = 3, R: int = 8, tokens: int = MOE_TOKENS, hidden: int = MOE_HIDDEN,
                 dtype: int = BF16, payload: bool = True):
    """MoE-dispatch AllToAllV input.

    Returns ``(C_tokens, inputs)``: the R x R count matrix in tokens (row s =
    source, column d = destination; each row sums to ``tokens``) and the R
    input buffers of ``tokens * hidden`` elements each (``None`` when
    ``payload`` is false).  Element counts are ``C_tokens * hidden``.
    """
    rng = np.random.default_rng(seed)
    p = zipf_weights(R)
    C = np.stack([rng.multinomial(tokens, p) for _ in range(R)]).astype(np.int64)
    inputs = normals(seed, R, tokens * hidden, dtype, rng=rng) if payload else None
    return C, inputs


def zipf_partition(total: int, R: int = 8, s: float = 0.125) -> list[int]:
    """The V-collective split of "Purlin: Separating Orchestration from the Datapath of Collectives"
    §C.4: rank r's share of a
    total of `total` elements has weight (r+1)^-s; floor each share and give
    the remainder to rank 0, so the split preserves the total.  Totals of at
    most 2 KiB of bf16 (1024 elements) are split uniformly, as the section
    states.  (With s = 0.125 the largest share is 1.176x the mean; the page
    quotes 1.125x, which these weights do not give.)"""
    if total <= 1024:
        part = [total // R] * R
        part[0] += total - sum(part)
        return part
    w = (np.arange(R, dtype=np.float64) + 1.0) ** (-s)
    part = [int(np.floor(total * (x / w.sum()))) for x in w]
    part[0] += total - sum(part)
    return part


def rotated_counts(part: list[int]) -> np.ndarray:
    """AllToAllV count matrix that rotates a partition: C[s][d] = part[(d - s) mod R], so every
    rank sends and receives the whole total (§C.4)."""
    R = len(part)
    return np.array([[part[(d - src) % R] for d in range(R)] for src in range(R)], dtype=np.int64)


def ar_sweep_inputs(batch: int, R: int = 8, seed: int = 4, max_batch: int | None = None):
    """AllReduce sweep input for one batch size: the first R*n values of the
    workload's single stream, split rank-major (n = batch x 4096)."""
    n = batch * HIDDEN
    rng = np.random.default_rng(seed)
    flat = rng.standard_normal(R * n, dtype=np.float32)
    return [to_bf16_bits(flat[r * n:(r + 1) * n]) for r in range(R)]


def inputs_for(w: Workload):
    """Inputs of one named workload (A2AV returns ``(C_tokens, inputs)``)."""
    if w.collective == "all_to_all_v":
        return moe_dispatch(w.seed, w.R)
    if w is AR_F32_R8_4096:
        return int_values_f32(w.seed, w.R, w.n)
    if w.name.startswith("allreduce_bf16_R8_b"):
        return ar_sweep_inputs(w.n // HIDDEN, w.R, w.seed)
    return normals(w.seed, w.R, w.n, w.dtype)
