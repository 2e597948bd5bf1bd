"""CPU oracle for MLA decode with a latent KV cache.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU
baseline and ``--impl reference`` arm) may import this module.  The CUDA path
never calls it and shares no code with it.

Everything is float64 numpy, written in the order the pages state the method:

* The attention definition (kexue.fm "From MHA, MQA, GQA to MLA", the MHA
  equation in section "MHA"): o_t^(s) = sum_i exp(q_t^(s) k_i^(s)T) v_i^(s) /
  sum_i exp(q_t^(s) k_i^(s)T), summed over cached positions i <= t.
* The released MLA form with decoupled RoPE (same page, section "Part 2",
  the hybrid equation, and section "Part 3", eq. mla-mha):
  k_i^(s) = [c_i W_kc^(s), x_i W_kr R_i], v_i^(s) = c_i W_v^(s),
  q^(s) = [q_c^(s), q_r^(s) R_t].  The cache holds c_i and the rotated
  x_i W_kr R_i only.
* The score scale 1/sqrt(d_nope + d_r) (iotdigitaltwinplm.com "MLA vs GQA vs
  MQA", the absorbed-decode listing in section "A latent KV projection in
  PyTorch"; intvml.com "DL0107 MLA", the paragraph giving an effective head
  dimension of 192).
* RoPE with interleaved (even, odd) pairs and inverse frequency
  theta^(-2i/d) (iotdigitaltwinplm.com, the ``rope`` helper of the same
  section).

``decode_reference`` is the non-absorbed definition (per-head K and V are
rebuilt from the latent).  ``decode_absorbed`` is the decode-time MQA form
(kexue.fm, section "Part 3", eq. mla-mqa): W_UK folded into the query, scores
over the 576-d concatenation [c_i, k_R,i], probabilities applied to c_i, W_UV
applied after attention.  The two must agree (absorption identity, kexue.fm
section "Part 1", the equation q k^T = x (W_q W_k^T) c^T); the tests pin the
oracle with that identity, RoPE's closed forms, special cases of softmax
attention, brute-force scalar loops and the cache-size arithmetic printed on
iotdigitaltwinplm.com ("Worked numbers from real configs").

Weight layout: w_uk[s, d, c] and w_uv[s, v, c] ([h, d_v, d_c]), i.e. row s,d of
the up-projection as stored by the ``uk``/``uv`` linear layers of the
iotdigitaltwinplm.com listing.  k^(s)_i[d] = sum_c c_i[c] w_uk[s, d, c].
"""
from __future__ import annotations

import math

import numpy as np

ROPE_THETA = 10000.0


# ----------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------

def rope_inv_freq(d_r: int, theta: float = ROPE_THETA) -> np.ndarray:
    """omega_i = theta^(-2i/d_r), i = 0 .. d_r/2 - 1 (iotdigitaltwinplm.com, ``rope``)."""
    i = np.arange(d_r // 2, dtype=np.float64)
    return theta ** (-2.0 * i / d_r)


def rope(x: np.ndarray, pos, theta: float = ROPE_THETA) -> np.ndarray:
    """Rotate the last axis of x by position pos (broadcast over leading axes).

    Pair i is (x[2i], x[2i+1]); it is rotated by angle pos * omega_i:
    (a, b) -> (a cos - b sin, a sin + b cos).  This is the block-diagonal
    rotation R_pos of kexue.fm section "Part 2" (R_m R_n^T = R_{m-n}).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty(np.broadcast_shapes(x.shape, ang.shape[:-1] + (d,)), dtype=np.float64)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


def rope_matrix(d: int, pos: float, theta: float = ROPE_THETA) -> np.ndarray:
    """The d x d matrix R_pos with rope(x, pos) == x @ R_pos (row-vector convention)."""
    return rope(np.eye(d), pos, theta)


def score_scale(d_nope: int, d_r: int) -> float:
    """1 / sqrt(d_nope + d_r): the scale of the 192-d per-head score."""
    return 1.0 / math.sqrt(d_nope + d_r)


# ----------------------------------------------------------------------------
# exact softmax attention
# ----------------------------------------------------------------------------

def softmax_with_lse(z: np.ndarray):
    """Exact softmax over the last axis and its log-sum-exp (natural log)."""
    m = np.max(z, axis=-1, keepdims=True)
    e = np.exp(z - m)
    ssum = np.sum(e, axis=-1, keepdims=True)
    return e / ssum, (m + np.log(ssum))[..., 0]


def decode_reference(q_nope, q_rope, q_pos, w_uk, w_uv, seqs, *, heads=None,
                     scale=None, theta=ROPE_THETA, k_pos=None):
    """Non-absorbed MLA decode of one query token per sequence.

    q_nope [B, h, d_nope], q_rope [B, h, d_r] (unrotated), q_pos [B],
    w_uk [h, d_nope, d_c], w_uv [h, d_v, d_c], seqs: list of B pairs
    (c_kv [L_b, d_c], k_rope [L_b, d_r] unrotated pre-images).
    heads: optional list of head indices to evaluate (default all).
    k_pos: optional list of B position arrays for the keys (default 0..L_b-1).

    Returns dict with out [B, H, d_v] (after W_UV), o_lat [B, H, d_c]
    (probabilities applied to the latent) and lse [B, H] (log-sum-exp of the
    scaled scores), H = len(heads).
    """
    q_nope = np.asarray(q_nope, dtype=np.float64)
    q_rope = np.asarray(q_rope, dtype=np.float64)
    w_uk = np.asarray(w_uk, dtype=np.float64)
    w_uv = np.asarray(w_uv, dtype=np.float64)
    B, h, d_nope = q_nope.shape
    d_r = q_rope.shape[-1]
    d_v = w_uv.shape[1]
    d_c = w_uk.shape[2]
    heads = list(range(h)) if heads is None else list(heads)
    H = len(heads)
    sc = score_scale(d_nope, d_r) if scale is None else scale
    out = np.zeros((B, H, d_v))
    o_lat = np.zeros((B, H, d_c))
    lse = np.zeros((B, H))
    for b in range(B):
        c = np.asarray(seqs[b][0], dtype=np.float64)
        kr_pre = np.asarray(seqs[b][1], dtype=np.float64)
        L = c.shape[0]
        pos = np.arange(L) if k_pos is None else np.asarray(k_pos[b], dtype=np.float64)
        k_r = rope(kr_pre, pos, theta)                      # shared rotated key [L, d_r]
        for j, s in enumerate(heads):
            k_c = c @ w_uk[s].T                             # per-head content key [L, d_nope]
            v = c @ w_uv[s].T                               # per-head value [L, d_v]
            q_r = rope(q_rope[b, s], q_pos[b], theta)       # rotated query part [d_r]
            k = np.concatenate([k_c, k_r], axis=1)          # [L, d_nope + d_r]
            q = np.concatenate([q_nope[b, s], q_r])         # [d_nope + d_r]
            z = (k @ q) * sc
            p, l = softmax_with_lse(z)
            out[b, j] = p @ v
            o_lat[b, j] = p @ c
            lse[b, j] = l
    return {"out": out, "o_lat": o_lat, "lse": lse}


def decode_reference_multi(q_nope, q_rope, w_uk, w_uv, seqs, *, heads=None, scale=None,
                           theta=ROPE_THETA):
    """Non-absorbed MLA decode of q_len new tokens per sequence (multi-token
    prediction or speculative decoding verify several tokens in one step).

    The L_b cached rows of sequence b include its q_len new tokens, so token j
    sits at position L_b - q_len + j and, as in the MHA equation of kexue.fm
    (keys i <= t), attends to the cached rows 0 .. L_b - q_len + j.  Token j's
    output is ``decode_reference`` of its own query over those rows.

    q_nope [B, q_len, h, d_nope], q_rope [B, q_len, h, d_r] (unrotated),
    seqs as in ``decode_reference``.  Returns out [B, q_len, H, d_v],
    o_lat [B, q_len, H, d_c], lse [B, q_len, H]; a token that sees no row
    (L_b - q_len + j < 0) gets out = o_lat = 0 and lse = -inf.
    """
    q_nope = np.asarray(q_nope, dtype=np.float64)
    q_rope = np.asarray(q_rope, dtype=np.float64)
    B, q_len, h = q_nope.shape[:3]
    H = h if heads is None else len(heads)
    d_v, d_c = np.asarray(w_uv).shape[1], np.asarray(w_uk).shape[2]
    out = np.zeros((B, q_len, H, d_v))
    o_lat = np.zeros((B, q_len, H, d_c))
    lse = np.full((B, q_len, H), -np.inf)
    for b in range(B):
        c, kr = seqs[b]
        L = np.asarray(c).shape[0]
        for j in range(q_len):
            n = L - q_len + j + 1          # rows visible to token j
            if n <= 0:
                continue
            r = decode_reference(q_nope[b:b + 1, j], q_rope[b:b + 1, j], [n - 1], w_uk, w_uv,
                                 [(c[:n], kr[:n])], heads=heads, scale=scale, theta=theta)
            out[b, j], o_lat[b, j], lse[b, j] = r["out"][0], r["o_lat"][0], r["lse"][0]
    return {"out": out, "o_lat": o_lat, "lse": lse}


def prefill_reference(q_nope, q_rope, w_uk, w_uv, c, k_rope, *, heads=None, scale=None,
                      theta=ROPE_THETA):
    """Prefill of one sequence in the MHA form (kexue.fm "Part 3", eq. mla-mha,
    used for training and prefill; iotdigitaltwinplm.com "Prefill versus
    decode"): per head the keys k_i = [c_i W_kc^(s), RoPE(k_R,i, i)] (192-d)
    and values v_i = c_i W_v^(s) (128-d) are formed, and every token t
    attends causally to the tokens i <= t with its query
    [q_nope,t, RoPE(q_R,t, t)] and the scale 1/sqrt(192).

    q_nope [T, h, d_nope], q_rope [T, h, d_r] (unrotated, position t = row t),
    c [T, d_c], k_rope [T, d_r] (unrotated pre-images).  Returns out
    [T, H, d_v] and lse [T, H] (natural log of the causal softmax's
    denominator).
    """
    q_nope = np.asarray(q_nope, dtype=np.float64)
    q_rope = np.asarray(q_rope, dtype=np.float64)
    c = np.asarray(c, dtype=np.float64)
    w_uk = np.asarray(w_uk, dtype=np.float64)
    w_uv = np.asarray(w_uv, dtype=np.float64)
    T, h, d_nope = q_nope.shape
    d_r = q_rope.shape[-1]
    heads = list(range(h)) if heads is None else list(heads)
    sc = score_scale(d_nope, d_r) if scale is None else scale
    pos = np.arange(T)
    k_r = rope(np.asarray(k_rope, dtype=np.float64), pos, theta)          # [T, d_r]
    causal = pos[None, :] <= pos[:, None]                                 # [t, i]
    out = np.zeros((T, len(heads), w_uv.shape[1]))
    lse = np.zeros((T, len(heads)))
    for j, s in enumerate(heads):
        k = np.concatenate([c @ w_uk[s].T, k_r], axis=1)                 # [T, 192]
        v = c @ w_uv[s].T                                                 # [T, d_v]
        q = np.concatenate([q_nope[:, s], rope(q_rope[:, s], pos, theta)], axis=1)
        z = np.where(causal, (q @ k.T) * sc, -np.inf)
        p, l = softmax_with_lse(z)
        out[:, j] = p @ v
        lse[:, j] = l
    return {"out": out, "lse": lse}


def decode_absorbed(q_nope, q_rope, q_pos, w_uk, w_uv, seqs, *, heads=None,
                    scale=None, theta=ROPE_THETA):
    """Absorbed (MQA-form) MLA decode in float64.

    q_cat^(s) = [q_nope^(s) W_UK^(s), RoPE(q_rope^(s), q_pos)] in R^(d_c+d_r);
    k_i = [c_i, RoPE(k_rope_i, i)] shared by all heads; scores q_cat k_i^T
    times the same 1/sqrt(d_nope+d_r); o_lat^(s) = sum_i p_i c_i;
    out^(s) = o_lat^(s) W_UV^(s)T.  Same arguments and outputs as
    ``decode_reference``.
    """
    q_nope = np.asarray(q_nope, dtype=np.float64)
    q_rope = np.asarray(q_rope, dtype=np.float64)
    w_uk = np.asarray(w_uk, dtype=np.float64)
    w_uv = np.asarray(w_uv, dtype=np.float64)
    B, h, d_nope = q_nope.shape
    d_r = q_rope.shape[-1]
    heads = list(range(h)) if heads is None else list(heads)
    sc = score_scale(d_nope, d_r) if scale is None else scale
    q_abs = np.einsum("bsd,sdc->bsc", q_nope[:, heads], w_uk[heads])       # [B, H, d_c]
    q_r = rope(q_rope[:, heads], np.asarray(q_pos, dtype=np.float64)[:, None], theta)
    q_cat = np.concatenate([q_abs, q_r], axis=-1)                          # [B, H, d_c+d_r]
    H = len(heads)
    o_lat = np.zeros((B, H, w_uk.shape[2]))
    lse = np.zeros((B, H))
    for b in range(B):
        c = np.asarray(seqs[b][0], dtype=np.float64)
        k_r = rope(np.asarray(seqs[b][1], dtype=np.float64), np.arange(c.shape[0]), theta)
        kcat = np.concatenate([c, k_r], axis=1)                            # [L, d_c+d_r]
        z = (q_cat[b] @ kcat.T) * sc                                       # [H, L]
        p, l = softmax_with_lse(z)
        o_lat[b] = p @ c
        lse[b] = l
    out = np.einsum("bsc,svc->bsv", o_lat, w_uv[heads])
    return {"out": out, "o_lat": o_lat, "lse": lse, "q_cat": q_cat}


def absorb_query(q_nope, q_rope, q_pos, w_uk, theta=ROPE_THETA):
    """q_cat [B, h, d_c + d_r] of the absorbed form (the first decode step)."""
    q_nope = np.asarray(q_nope, dtype=np.float64)
    q_abs = np.einsum("bsd,sdc->bsc", q_nope, np.asarray(w_uk, dtype=np.float64))
    q_r = rope(np.asarray(q_rope, dtype=np.float64),
               np.asarray(q_pos, dtype=np.float64)[:, None], theta)
    return np.concatenate([q_abs, q_r], axis=-1)


def output_projection(o_lat, w_uv):
    """out[b, s, v] = sum_c o_lat[b, s, c] w_uv[s, v, c] (W_UV applied after attention)."""
    return np.einsum("bsc,svc->bsv", np.asarray(o_lat, dtype=np.float64),
                     np.asarray(w_uv, dtype=np.float64))


def query_from_hidden(x, w_dq, w_uq, w_qr, h):
    """Per-head queries from the hidden state through the compressed query
    (kexue.fm "Part 3": c'_t = x_t W_c'; every head's content query
    c'_t W_qc^(s) and rotary query c'_t W_qr^(s) are read off it).

    x [B, d_model]; weights stored [out, in] as linear layers: w_dq
    [d_cq, d_model], w_uq [h * d_nope, d_cq], w_qr [h * d_r, d_cq].
    Returns q_nope [B, h, d_nope] and the unrotated q_rope [B, h, d_r].
    """
    x = np.asarray(x, dtype=np.float64)
    c = x @ np.asarray(w_dq, dtype=np.float64).T
    qn = c @ np.asarray(w_uq, dtype=np.float64).T
    qr = c @ np.asarray(w_qr, dtype=np.float64).T
    B = x.shape[0]
    return qn.reshape(B, h, -1), qr.reshape(B, h, -1)


def output_to_hidden(out, w_o):
    """y_t = [o^(1), ..., o^(h)] W_O^T: the heads' value outputs [B, h, d_v]
    concatenated and projected back to the hidden size (w_o [d_model, h * d_v])."""
    out = np.asarray(out, dtype=np.float64)
    return out.reshape(out.shape[0], -1) @ np.asarray(w_o, dtype=np.float64).T


def fold_uv_into_o(w_uv, w_o):
    """The output projection with W_UV merged in (kexue.fm "Part 1": W_v moves
    into the projection after attention): w_fold[n, s * d_c + c] =
    sum_v w_o[n, s * d_v + v] w_uv[s, v, c], so that y = o_lat w_fold^T."""
    w_uv = np.asarray(w_uv, dtype=np.float64)
    w_o = np.asarray(w_o, dtype=np.float64)
    h, d_v, d_c = w_uv.shape
    d_model = w_o.shape[0]
    fold = np.einsum("nsv,svc->nsc", w_o.reshape(d_model, h, d_v), w_uv)
    return fold.reshape(d_model, h * d_c)


def decode_from_hidden(x, w_dq, w_uq, w_qr, w_uk, w_uv, w_o, q_pos, seqs, *, theta=ROPE_THETA):
    """The whole decode step at the hidden-state boundary, non-absorbed:
    queries from x (``query_from_hidden``), attention as ``decode_reference``,
    output through W_UV and W_O (``output_to_hidden``).  Returns y [B, d_model]
    and the intermediate dict of ``decode_reference``."""
    h = np.asarray(w_uk).shape[0]
    qn, qr = query_from_hidden(x, w_dq, w_uq, w_qr, h)
    r = decode_reference(qn, qr, q_pos, w_uk, w_uv, seqs, theta=theta)
    return output_to_hidden(r["out"], w_o), r


def merge_partials(o_parts, lses):
    """Merge attention computed over disjoint key ranges.

    o_parts [J, ..., d] are each range's normalised output, lses [J, ...] each
    range's log-sum-exp; a range with no keys has lse = -inf and weight 0.
    The result equals attention over the union of the ranges (the softmax
    denominator is the sum of the ranges' exp(lse)).
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    m = np.max(lses, axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lses), np.exp(lses - m_safe), 0.0)
    wsum = np.sum(w, axis=0)
    o = np.sum(w[..., None] * o_parts, axis=0) / np.where(wsum > 0, wsum, 1.0)[..., None]
    lse = np.where(finite, m_safe + np.log(np.where(wsum > 0, wsum, 1.0)), -np.inf)
    return o, lse


# ----------------------------------------------------------------------------
# cache arithmetic (iotdigitaltwinplm.com, "The Cache Arithmetic")
# ----------------------------------------------------------------------------

def cache_elements_per_token_layer(scheme: str, *, n_h=None, d_h=None, n_g=None,
                                   d_c=None, d_r=None) -> int:
    """Elements cached per token per layer: MHA 2 n_h d_h, MQA 2 d_h,
    GQA 2 n_g d_h, MLA d_c + d_r."""
    if scheme == "mha":
        return 2 * n_h * d_h
    if scheme == "mqa":
        return 2 * d_h
    if scheme == "gqa":
        return 2 * n_g * d_h
    if scheme == "mla":
        return d_c + d_r
    raise ValueError(scheme)


def mla_cache_bytes_per_token(latent_dtype: str, rope_dtype: str, d_c: int, d_r: int,
                              block_size: int) -> float:
    """Bytes one cached token occupies in the paged layout (scale amortised per block)."""
    width = {"f32": 4, "bf16": 2, "fp8e4m3": 1}
    b = d_c * width[latent_dtype] + d_r * width[rope_dtype]
    if latent_dtype == "fp8e4m3":
        b += 4.0 / block_size
    return b


# ----------------------------------------------------------------------------
# FP8 e4m3 storage of the latent (iotdigitaltwinplm.com "Interaction with
# quantisation and paging": the latent may be stored in FP8)
# ----------------------------------------------------------------------------
#
# e4m3 (OCP 8-bit floating point, "E4M3"): 1 sign bit, 4 exponent bits with
# bias 7, 3 mantissa bits; exponent field 0 encodes subnormals m/8 * 2^-6;
# S.1111.111 is NaN and there is no infinity, so the largest finite value is
# 1.75 * 2^8 = 448.

E4M3_MAX = 448.0


def e4m3_value_table() -> np.ndarray:
    """float64 value of every code 0..255 (NaN codes -> nan)."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = sign * (m / 8.0) * 2.0 ** (1 - 7)
        else:
            vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


def e4m3_encode(v) -> np.ndarray:
    """Round values to the nearest finite e4m3 code, ties to even mantissa,
    saturating to +-448 (values are exact float64 numbers, e.g. float32 quotients)."""
    v = np.asarray(v, dtype=np.float64)
    table = e4m3_value_table()
    pos_codes = np.arange(0, 0x7F)            # 0x00 .. 0x7E: all finite non-negative codes
    pos_vals = table[pos_codes]               # strictly increasing
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.searchsorted(pos_vals, a, side="left")      # first value >= a
    hi = np.clip(hi, 0, len(pos_vals) - 1)
    lo = np.clip(hi - 1, 0, len(pos_vals) - 1)
    d_hi = pos_vals[hi] - a
    d_lo = a - pos_vals[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (pos_codes[hi] % 2 == 0))
    exact = pos_vals[hi] == a
    code = np.where(exact | pick_hi, pos_codes[hi], pos_codes[lo]).astype(np.uint8)
    # the sign survives rounding, as in IEEE arithmetic: a negative value that
    # rounds to zero is the code of -0 (0x80)
    code = np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)
    return code


def e4m3_decode(codes) -> np.ndarray:
    return e4m3_value_table()[np.asarray(codes, dtype=np.uint8)]


def fp8_quantize_block(x) -> tuple[np.ndarray, np.float32]:
    """Quantise one cache block of latent rows [rows, d_c] to e4m3 with one scale.

    scale = amax / 448 in float32 (1 when amax is 0); code = e4m3(x / scale)
    where the quotient is the correctly rounded float32 division.  The
    dequantised value is e4m3_decode(code) * scale.
    """
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0.0)
    scale = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
    q = (x32 / scale).astype(np.float32)
    return e4m3_encode(q.astype(np.float64)), scale


def fp8_dequantize(codes, scale) -> np.ndarray:
    return e4m3_decode(codes) * np.float64(scale)


def quantized_latent_f64(c_src32: np.ndarray, block_size: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Quantise a sequence's latent rows block by block.

    Returns (codes [L, d_c] uint8, scales [nblocks] float32, dequantised [L, d_c] f64).
    """
    L = c_src32.shape[0]
    nb = (L + block_size - 1) // block_size
    codes = np.zeros(c_src32.shape, dtype=np.uint8)
    scales = np.zeros(nb, dtype=np.float32)
    deq = np.zeros(c_src32.shape, dtype=np.float64)
    for j in range(nb):
        rows = slice(j * block_size, min(L, (j + 1) * block_size))
        cj, sj = fp8_quantize_block(c_src32[rows])
        codes[rows] = cj
        scales[j] = sj
        deq[rows] = fp8_dequantize(cj, sj)
    return codes, scales, deq


def fp8_append_row(codes, scale, c_new):
    """Append one latent row to an FP8 block that already holds len(codes) rows.

    The cache keeps only the e4m3 codes and the block's float32 scale, so the
    block's earlier values are known only in dequantised form.  Reading of
    iotdigitaltwinplm.com "Interaction with quantisation and paging" (the
    latent is stored in FP8 and the cache grows by one token per decode step):

    * an empty block (the token lands in slot 0) is quantised on its own, as
      ``fp8_quantize_block`` does for one row;
    * otherwise, with a = max|c_new| and s the block's scale, the scale stays
      when a <= 448 s (float32 product): the new row's code is e4m3(c / s);
    * when a > 448 s the scale grows to s' = a / 448 (float32 quotient), every
      earlier code is re-quantised from its dequantised value,
      e4m3((e4m3(code) * s) / s') (each step a float32 operation), and the new
      row's code is e4m3(c / s').

    codes [rows, d_c] uint8, scale float32, c_new [d_c] (float32 values).
    Returns (codes [rows + 1, d_c], new scale).
    """
    codes = np.asarray(codes, dtype=np.uint8).reshape(-1, np.asarray(c_new).shape[-1])
    x = np.asarray(c_new, dtype=np.float32)
    if codes.shape[0] == 0:
        c, sc = fp8_quantize_block(x[None, :])
        return c, sc
    s_old = np.float32(scale)
    a = np.float32(np.max(np.abs(x)))
    if a > np.float32(E4M3_MAX) * s_old:
        s_new = np.float32(a / np.float32(E4M3_MAX))
        deq = (e4m3_decode(codes).astype(np.float32) * s_old).astype(np.float32)
        old = e4m3_encode((deq / s_new).astype(np.float32).astype(np.float64))
    else:
        s_new = s_old
        old = codes
    new = e4m3_encode((x / s_new).astype(np.float32).astype(np.float64))
    return np.concatenate([old, new[None, :]], axis=0), s_new


def quantized_latent_appended(c_src32, block_size, n_fill):
    """FP8 latent of a sequence whose first n_fill rows were written block by
    block (``fp8_quantize_block`` over each block's rows) and whose remaining
    rows were appended one at a time (``fp8_append_row``).

    Returns (codes [L, d_c] uint8, scales [nblocks] float32, dequantised [L, d_c] f64).
    """
    c_src32 = np.asarray(c_src32, dtype=np.float32)
    L = c_src32.shape[0]
    nb = (L + block_size - 1) // block_size
    codes = np.zeros(c_src32.shape, dtype=np.uint8)
    scales = np.zeros(nb, dtype=np.float32)
    for j in range(nb):
        r0, r1 = j * block_size, min(L, (j + 1) * block_size)
        f1 = min(r1, max(r0, n_fill))                # rows [r0, f1) come from the fill
        if f1 > r0:
            blk, sc = fp8_quantize_block(c_src32[r0:f1])
        else:
            blk, sc = np.zeros((0, c_src32.shape[1]), dtype=np.uint8), np.float32(1.0)
        for r in range(f1, r1):
            blk, sc = fp8_append_row(blk, sc, c_src32[r])
        codes[r0:r1] = blk
        scales[j] = sc
    deq = np.zeros(c_src32.shape, dtype=np.float64)
    for j in range(nb):
        r0, r1 = j * block_size, min(L, (j + 1) * block_size)
        deq[r0:r1] = fp8_dequantize(codes[r0:r1], scales[j])
    return codes, scales, deq


# ----------------------------------------------------------------------------
# paged cache, logical view
# ----------------------------------------------------------------------------

def paged_gather(pool: np.ndarray, table_row: np.ndarray, L: int, block_size: int) -> np.ndarray:
    """Logical rows 0..L-1 of one sequence from a pool [nblk, block_size, ...]."""
    rows = []
    for j in range((L + block_size - 1) // block_size):
        n = min(block_size, L - j * block_size)
        rows.append(pool[int(table_row[j]), :n])
    return np.concatenate(rows, axis=0) if rows else pool[:0, 0]


# ----------------------------------------------------------------------------
# the oracle's view of a seeded workload
# ----------------------------------------------------------------------------

def sequence_view(w, b: int, L: int, n_fill: int | None = None):
    """(c_kv f64 [L, d_c], unrotated k_rope f64 [L, d_r]) exactly as the cache holds them.

    bf16 / f32 latents are the stored values; an FP8 latent is the
    dequantised value of the per-block e4m3 codes (``quantized_latent_f64``,
    or ``quantized_latent_appended`` when only the first n_fill rows were
    written block by block and the rest appended one at a time).
    """
    import mla_inputs as mi
    c_st, kr_st = mi.sequence(w, b, L)
    kr = mi.storage_to_f64(kr_st, w.dtype)
    src = mi.latent_source_dtype(w)
    if w.latent_dtype == "fp8e4m3":
        c32 = mi.storage_to_f64(c_st, src).astype(np.float32)
        if n_fill is None or n_fill >= L:
            _, _, c = quantized_latent_f64(c32, w.block_size)
        else:
            _, _, c = quantized_latent_appended(c32, w.block_size, n_fill)
    else:
        c = mi.storage_to_f64(c_st, src)
    return c, kr


def workload_inputs_f64(w):
    """Query, weights and positions of a workload as float64 (exact storage values)."""
    import mla_inputs as mi
    qn, qr = mi.queries(w)
    wuk, wuv = mi.weights(w)
    lens = mi.lengths(w)
    return {
        "q_nope": mi.storage_to_f64(qn, w.dtype),
        "q_rope": mi.storage_to_f64(qr, w.dtype),
        "w_uk": mi.storage_to_f64(wuk, w.dtype),
        "w_uv": mi.storage_to_f64(wuv, w.dtype),
        "q_pos": mi.query_positions(w, lens),
        "lens": lens,
    }
