"""Seeded synthetic inputs for MLA absorbed decode.

This module is shared by the CPU oracle (``oracle/``) and the CUDA path
(``mla_latent_kv_72_b300``).  It holds only random draws, the storage
rounding of those draws (f64 -> f32 -> bf16, round-to-nearest-even) and the
workload table.  None of the attention arithmetic lives here: RoPE, the
absorption, softmax and the FP8 cache quantisation are implemented
separately by each side.

Recipe (one generator stream per purpose, so that any single sequence can be
regenerated on its own):

* ``numpy.random.default_rng([seed, TAG, b])``: per-sequence cache rows.
  ``c_kv`` [L_b, d_c] and the *unrotated* RoPE key pre-image ``k_rope`` [L_b, d_r],
  both standard normal.
* ``default_rng([seed, TAG_Q])``: ``q_nope`` [B, h, d_nope] and the unrotated
  ``q_rope`` [B, h, d_r], standard normal.
* ``default_rng([seed, TAG_W])``: ``w_uk`` and ``w_uv`` [h, d_v, d_c], normal
  with variance 1/fan_in, fan_in = d_c.
* ``default_rng([seed, TAG_L])``: sequence lengths (variable-length workload).
* ``default_rng([seed, TAG_P])``: the physical-block permutation of the
  paged workload.
* ``default_rng([seed, TAG_QM, q_len])``: queries of q_len new tokens per
  sequence (multi-token decode).
* ``default_rng([seed, TAG_H, d_model, d_cq])``: the hidden state and the
  linear layers around the step (query compression and output projection).
* ``default_rng([seed, TAG_PF, b])``: the prompt queries of sequence b (prefill).

All draws are float64; storage dtype "bf16" rounds f64 -> f32 -> bf16 with
round-to-nearest-even at each step, "f32" rounds f64 -> f32.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

TAG_SEQ = 11
TAG_Q = 12
TAG_W = 13
TAG_L = 14
TAG_P = 15
TAG_QM = 16
TAG_H = 17
TAG_PF = 18


# ----------------------------------------------------------------------------
# storage rounding of the synthetic draws
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round-to-nearest-even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r = r.copy()
        r[nan] = 0x7FC0
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def to_storage(x64: np.ndarray, dtype: str) -> np.ndarray:
    """Storage form of a float64 draw.

    dtype "bf16" -> uint16 bit patterns, "f32" -> float32 array.
    """
    x32 = np.asarray(x64, dtype=np.float64).astype(np.float32)
    if dtype == "f32":
        return x32
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    raise ValueError(f"unknown storage dtype {dtype!r}")


def storage_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of a storage array."""
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    raise ValueError(f"unknown storage dtype {dtype!r}")


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode workload: shapes, storage dtypes and cache structure."""

    name: str
    index: int          # 1-based position in the workload table
    B: int
    h: int
    L: int | None       # uniform length; None => drawn per sequence
    L_range: tuple[int, int] | None
    dtype: str          # query / weight / rope-key storage: "f32" or "bf16"
    latent_dtype: str   # "f32", "bf16" or "fp8e4m3"
    layout: str         # "contiguous" (identity block table) or "paged" (permuted)
    d_c: int = 512
    d_r: int = 64
    d_nope: int = 128
    d_v: int = 128
    block_size: int = 64
    theta: float = 10000.0
    lens: tuple[int, ...] | None = None   # explicit lengths (edge-case tests), else L / L_range

    @property
    def seed(self) -> int:
        return 7200 + self.index

    @property
    def d_qk(self) -> int:
        return self.d_c + self.d_r


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_fp32_b1_h16_l512", 1, B=1, h=16, L=512, L_range=None,
                 dtype="f32", latent_dtype="f32", layout="contiguous"),
        Workload("small_bf16_b64_h16_l4096", 2, B=64, h=16, L=4096, L_range=None,
                 dtype="bf16", latent_dtype="bf16", layout="contiguous"),
        Workload("v3_bf16_b64_h128_l8192", 3, B=64, h=128, L=8192, L_range=None,
                 dtype="bf16", latent_dtype="bf16", layout="contiguous"),
        Workload("paged_bf16_b128_h128_lvar", 4, B=128, h=128, L=None, L_range=(1024, 32768),
                 dtype="bf16", latent_dtype="bf16", layout="paged"),
        Workload("longctx_fp8_b4_h128_l131072", 5, B=4, h=128, L=131072, L_range=None,
                 dtype="bf16", latent_dtype="fp8e4m3", layout="contiguous"),
    ]
}

WORKLOAD_ORDER = [w.name for w in sorted(WORKLOADS.values(), key=lambda w: w.index)]


def workload(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[WORKLOAD_ORDER[name_or_index - 1]]
    return WORKLOADS[name_or_index]


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(w, **changes)


# ----------------------------------------------------------------------------
# draws
# ----------------------------------------------------------------------------

def lengths(w: Workload) -> np.ndarray:
    """Cached length L_b of every sequence (int64 [B])."""
    if w.lens is not None:
        assert len(w.lens) == w.B
        return np.asarray(w.lens, dtype=np.int64)
    if w.L is not None:
        return np.full(w.B, w.L, dtype=np.int64)
    lo, hi = w.L_range
    rng = np.random.default_rng([w.seed, TAG_L])
    return rng.integers(lo, hi, endpoint=True, size=w.B).astype(np.int64)


def blocks_per_seq(w: Workload, lens: np.ndarray | None = None) -> np.ndarray:
    lens = lengths(w) if lens is None else lens
    return (lens + w.block_size - 1) // w.block_size


def block_table(w: Workload, lens: np.ndarray | None = None) -> tuple[np.ndarray, int]:
    """Block table int32 [B, max_blocks] and the number of physical blocks.

    Contiguous layout: sequence b owns physical blocks
    [sum_{b'<b} nb_{b'}, ... ) in order (identity table).  Paged layout: the
    same logical blocks land on a seeded random permutation of the pool.
    Unused table entries are -1.
    """
    lens = lengths(w) if lens is None else lens
    nb = blocks_per_seq(w, lens)
    total = int(nb.sum())
    maxb = int(nb.max()) if len(nb) else 0
    phys = np.arange(total, dtype=np.int64)
    if w.layout == "paged":
        rng = np.random.default_rng([w.seed, TAG_P])
        phys = rng.permutation(total)
    table = np.full((w.B, max(maxb, 1)), -1, dtype=np.int32)
    start = 0
    for b in range(w.B):
        table[b, : nb[b]] = phys[start : start + nb[b]]
        start += nb[b]
    return table, total


def sequence_f64(w: Workload, b: int, L: int) -> tuple[np.ndarray, np.ndarray]:
    """Raw float64 draws of sequence b: c_kv [L, d_c], unrotated k_rope [L, d_r]."""
    rng = np.random.default_rng([w.seed, TAG_SEQ, b])
    c = rng.standard_normal((L, w.d_c))
    kr = rng.standard_normal((L, w.d_r))
    return c, kr


def latent_source_dtype(w: Workload) -> str:
    """Storage dtype of the latent rows handed to the cache writer.

    The FP8 cache is written from bf16 rows (the model emits bf16 latents).
    """
    return "f32" if w.latent_dtype == "f32" else "bf16"


def sequence(w: Workload, b: int, L: int) -> tuple[np.ndarray, np.ndarray]:
    """Storage form of sequence b's rows (latent source dtype, rope dtype)."""
    c, kr = sequence_f64(w, b, L)
    return to_storage(c, latent_source_dtype(w)), to_storage(kr, w.dtype)


def queries_multi(w: Workload, q_len: int) -> tuple[np.ndarray, np.ndarray]:
    """Storage form of q_nope [B, q_len, h, d_nope] and unrotated q_rope
    [B, q_len, h, d_r] for q_len new tokens per sequence, standard normal."""
    rng = np.random.default_rng([w.seed, TAG_QM, q_len])
    qn = rng.standard_normal((w.B, q_len, w.h, w.d_nope))
    qr = rng.standard_normal((w.B, q_len, w.h, w.d_r))
    return to_storage(qn, w.dtype), to_storage(qr, w.dtype)


def query_positions_multi(w: Workload, q_len: int, lens: np.ndarray | None = None) -> np.ndarray:
    """Positions [B, q_len] of the new tokens: L_b - q_len + j."""
    lens = lengths(w) if lens is None else lens
    return (lens[:, None] - q_len + np.arange(q_len)[None, :]).astype(np.int32)


def sequence_last_row(w: Workload, b: int, L: int) -> tuple[np.ndarray, np.ndarray]:
    """Storage form of the last row (index L - 1) of sequence(w, b, L)."""
    c, kr = sequence(w, b, L)
    return c[L - 1], kr[L - 1]


def queries(w: Workload) -> tuple[np.ndarray, np.ndarray]:
    """Storage form of q_nope [B, h, d_nope] and unrotated q_rope [B, h, d_r]."""
    rng = np.random.default_rng([w.seed, TAG_Q])
    qn = rng.standard_normal((w.B, w.h, w.d_nope))
    qr = rng.standard_normal((w.B, w.h, w.d_r))
    return to_storage(qn, w.dtype), to_storage(qr, w.dtype)


def weights(w: Workload) -> tuple[np.ndarray, np.ndarray]:
    """Storage form of W_UK and W_UV, both [h, d_v, d_c], variance 1/d_c."""
    rng = np.random.default_rng([w.seed, TAG_W])
    s = 1.0 / math.sqrt(w.d_c)
    wuk = rng.standard_normal((w.h, w.d_nope, w.d_c)) * s
    wuv = rng.standard_normal((w.h, w.d_v, w.d_c)) * s
    return to_storage(wuk, w.dtype), to_storage(wuv, w.dtype)


def prefill_queries(w: Workload, lens: np.ndarray | None = None) -> tuple[np.ndarray, np.ndarray]:
    """Storage form of the prompt's queries, packed by sequence: q_nope
    [T, h, d_nope] and unrotated q_rope [T, h, d_r], T = sum of the lengths,
    standard normal (one stream per sequence)."""
    lens = lengths(w) if lens is None else lens
    qn, qr = [], []
    for b, L in enumerate(lens):
        rng = np.random.default_rng([w.seed, TAG_PF, b])
        qn.append(rng.standard_normal((int(L), w.h, w.d_nope)))
        qr.append(rng.standard_normal((int(L), w.h, w.d_r)))
    return to_storage(np.concatenate(qn), w.dtype), to_storage(np.concatenate(qr), w.dtype)


def hidden_inputs(w: Workload, d_model: int, d_cq: int) -> dict:
    """Storage form of the hidden-state side of a step: x [B, d_model] ~ N(0,1)
    and the linear layers stored [out, in] with variance 1/fan_in: w_dq
    [d_cq, d_model], w_uq [h * d_nope, d_cq], w_qr [h * d_r, d_cq], w_o
    [d_model, h * d_v]."""
    rng = np.random.default_rng([w.seed, TAG_H, d_model, d_cq])
    x = rng.standard_normal((w.B, d_model))
    wdq = rng.standard_normal((d_cq, d_model)) / math.sqrt(d_model)
    wuq = rng.standard_normal((w.h * w.d_nope, d_cq)) / math.sqrt(d_cq)
    wqr = rng.standard_normal((w.h * w.d_r, d_cq)) / math.sqrt(d_cq)
    wo = rng.standard_normal((d_model, w.h * w.d_v)) / math.sqrt(w.h * w.d_v)
    return {k: to_storage(v, w.dtype) for k, v in
            {"x": x, "w_dq": wdq, "w_uq": wuq, "w_qr": wqr, "w_o": wo}.items()}


def query_positions(w: Workload, lens: np.ndarray | None = None) -> np.ndarray:
    """Position of the decoded token: the last cached slot, L_b - 1."""
    lens = lengths(w) if lens is None else lens
    return (lens - 1).astype(np.int32)
