"""ctypes binding of libmla72.so (see include/mla72.h for the contract).

Functions carry the C names and take torch tensors; they pass data pointers,
sizes and ``torch.cuda.current_stream()`` to the library and raise
``MLAError`` on a non-zero status.  No arithmetic of the method happens here.
"""
from __future__ import annotations

import ctypes
import os

import torch

MLA_F32 = 0
MLA_BF16 = 1
MLA_FP8E4M3 = 2

MLA_DECODE_AUTO = 0
MLA_DECODE_FORCE_SIMT = 1
MLA_DECODE_TEST_WAIT_TIMEOUT = 2

MLA_DEV_OK = 0
MLA_DEV_BAD_BLOCK = 1
MLA_DEV_BAD_LENGTH = 2
MLA_DEV_WAIT_TIMEOUT = 3

MLA_MAX_PARTS = 1024
MLA_MAX_Q_LEN = 8

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

EXPORTED_SYMBOLS = (
    "mla_status_string", "mla_version", "mla_cache_bytes_per_token", "mla_absorb_q",
    "mla_decode_num_partials", "mla_decode_fwd", "mla_decode_fwd_multi", "mla_combine", "mla_combine_out_proj", "mla_decode_attend_noalloc",
    "mla_out_proj", "mla_cache_fill", "mla_cache_append", "mla_paged_gather",
    "mla_linear_workspace_bytes", "mla_linear", "mla_fold_uv_into_o", "mla_prefill_query",
    "mla_prefill_fwd",
)


class MLAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: status {status} ({mla_status_string(status)})")


class KVCache(ctypes.Structure):
    """ctypes mirror of ``mla_kv_cache`` (tensors kept alive on ``self.tensors``)."""

    _fields_ = [
        ("latent", ctypes.c_void_p),
        ("rope", ctypes.c_void_p),
        ("scale", ctypes.c_void_p),
        ("latent_stride", ctypes.c_int64),
        ("rope_stride", ctypes.c_int64),
        ("latent_dtype", ctypes.c_int32),
        ("rope_dtype", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("d_c", ctypes.c_int32),
        ("d_r", ctypes.c_int32),
    ]

    @classmethod
    def packed(cls, pool: torch.Tensor, d_c: int, d_r: int) -> "KVCache":
        """Packed float pool [num_blocks, block_size, d_c + d_r] (latent then rope)."""
        assert pool.dim() == 3 and pool.shape[2] == d_c + d_r and pool.is_contiguous()
        dt = dtype_code(pool.dtype)
        kv = cls(pool.data_ptr(), pool.data_ptr() + d_c * pool.element_size(), None,
                 d_c + d_r, d_c + d_r, dt, dt, pool.shape[0], pool.shape[1], d_c, d_r)
        kv.tensors = (pool,)
        return kv

    @classmethod
    def split(cls, latent: torch.Tensor, rope: torch.Tensor,
              scale: torch.Tensor | None = None) -> "KVCache":
        """Separate pools: latent [nblk, bs, d_c] (bf16/f32, or uint8 e4m3 codes with
        a float32 scale [nblk]) and rope [nblk, bs, d_r]."""
        assert latent.is_contiguous() and rope.is_contiguous()
        ldt = MLA_FP8E4M3 if latent.dtype in (torch.uint8, torch.float8_e4m3fn) else dtype_code(latent.dtype)
        kv = cls(latent.data_ptr(), rope.data_ptr(), scale.data_ptr() if scale is not None else None,
                 latent.shape[2], rope.shape[2], ldt, dtype_code(rope.dtype), latent.shape[0],
                 latent.shape[1], latent.shape[2], rope.shape[2])
        kv.tensors = (latent, rope, scale)
        return kv


def library_path() -> str:
    return os.path.join(_HERE, "libmla72.so")


def lib() -> ctypes.CDLL:
    """Load libmla72.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m mla_latent_kv_72_b300.build`")
    L = ctypes.CDLL(path)
    vp, i32, i64, f32, f64, u32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                   ctypes.c_double, ctypes.c_uint)
    kvp = ctypes.POINTER(KVCache)
    sig = {
        "mla_status_string": (ctypes.c_char_p, [i32]),
        "mla_version": (i32, []),
        "mla_cache_bytes_per_token": (f64, [i32, i32, i32, i32, i32]),
        "mla_absorb_q": (i32, [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f64, vp]),
        "mla_decode_num_partials": (i32, [i32, i32]),
        "mla_decode_fwd": (i32, [vp, i32, kvp, vp, i32, vp, i32, i32, i32, f32, vp, vp, vp, u32, vp]),
        "mla_decode_fwd_multi": (i32, [vp, i32, kvp, vp, i32, vp, i32, i32, i32, i32, f32, vp, vp,
                                       vp, u32, vp]),
        "mla_combine": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, i32, vp, vp]),
        "mla_combine_out_proj": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, i32, vp, i32,
                                       vp, i32, vp, vp, vp]),
        "mla_decode_attend_noalloc": (i32, [vp, i32, kvp, vp, i32, vp, i32, i32, i32, f32, vp, i32,
                                            vp, vp, vp]),
        "mla_out_proj": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]),
        "mla_cache_fill": (i32, [vp, vp, i32, vp, i32, i32, vp, i32, kvp, f64, vp, vp]),
        "mla_cache_append": (i32, [vp, vp, i32, vp, i32, vp, i32, kvp, f64, vp, vp]),
        "mla_linear_workspace_bytes": (ctypes.c_size_t, [i32, i32, i32]),
        "mla_linear": (i32, [vp, vp, vp, i32, i32, i32, i32, vp, ctypes.c_size_t, vp]),
        "mla_fold_uv_into_o": (i32, [vp, vp, vp, i32, i32, i32, i32, vp]),
        "mla_prefill_query": (i32, [vp, vp, vp, i32, i32, i32, f64, vp, vp]),
        "mla_prefill_fwd": (i32, [vp, vp, vp, vp, vp, i32, i32, i64, i32, f32, vp, i32, vp, vp,
                                  vp]),
        "mla_paged_gather": (i32, [kvp, vp, i32, vp, i32, i32, vp, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = L
    return L


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return MLA_F32
    if dt == torch.bfloat16:
        return MLA_BF16
    if dt in (torch.uint8, torch.float8_e4m3fn):
        return MLA_FP8E4M3
    raise TypeError(f"unsupported dtype {dt}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise MLAError(fn, status)


def mla_status_string(status: int) -> str:
    return lib().mla_status_string(status).decode()


def mla_version() -> int:
    return lib().mla_version()


def mla_cache_bytes_per_token(latent_dtype: int, rope_dtype: int, d_c: int, d_r: int,
                              block_size: int) -> float:
    return lib().mla_cache_bytes_per_token(latent_dtype, rope_dtype, d_c, d_r, block_size)


def mla_absorb_q(q_nope, q_rope, q_pos, w_uk, q_cat, rope_theta=10000.0, stream=None):
    """q_cat[B, h, d_c + d_r] <- [q_nope W_UK, RoPE(q_rope, q_pos)] (see mla72.h)."""
    B, h, d_nope = q_nope.shape
    d_r = q_rope.shape[2]
    d_c = w_uk.shape[2]
    _check("mla_absorb_q", lib().mla_absorb_q(
        _ptr(q_nope), _ptr(q_rope), _ptr(q_pos), _ptr(w_uk), _ptr(q_cat), B, h, d_nope, d_c, d_r,
        dtype_code(q_nope.dtype), float(rope_theta), _stream(stream)))
    return q_cat


def mla_decode_num_partials(B: int, num_parts: int) -> int:
    n = lib().mla_decode_num_partials(B, num_parts)
    if n < 0:
        raise MLAError("mla_decode_num_partials", n)
    return n


def default_num_parts(device=None) -> int:
    """One part per CTA pair of the device (half its SM count)."""
    props = torch.cuda.get_device_properties(device if device is not None else torch.cuda.current_device())
    return max(1, props.multi_processor_count // 2)


def mla_decode_fwd(q_cat, kv: KVCache, block_table, seq_lens, num_parts, o_part, lse_part, *,
                   softmax_scale=0.0, dev_status=None, flags=MLA_DECODE_AUTO, stream=None):
    """Partials o_part [B + num_parts - 1, h, d_c], lse_part [B + num_parts - 1, h]
    over the balanced part partition of the block stream (see mla72.h)."""
    B, h, _ = q_cat.shape
    _check("mla_decode_fwd", lib().mla_decode_fwd(
        _ptr(q_cat), dtype_code(q_cat.dtype), ctypes.byref(kv), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, h, int(num_parts), float(softmax_scale),
        _ptr(o_part), _ptr(lse_part), _ptr(dev_status), int(flags), _stream(stream)))


def mla_decode_fwd_multi(q_cat, kv: KVCache, block_table, seq_lens, num_parts, o_part, lse_part,
                         *, softmax_scale=0.0, dev_status=None, flags=MLA_DECODE_AUTO,
                         stream=None):
    """Partials of q_len new tokens per sequence; q_cat [B, q_len, h, d_c + d_r],
    o_part [slots, q_len * h, d_c], lse_part [slots, q_len * h] (see mla72.h)."""
    B, q_len, h, _ = q_cat.shape
    _check("mla_decode_fwd_multi", lib().mla_decode_fwd_multi(
        _ptr(q_cat), dtype_code(q_cat.dtype), ctypes.byref(kv), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, q_len, h, int(num_parts), float(softmax_scale),
        _ptr(o_part), _ptr(lse_part), _ptr(dev_status), int(flags), _stream(stream)))


def mla_combine(o_part, lse_part, seq_lens, block_size, max_blocks_per_seq, num_parts, o_lat,
                lse=None, stream=None):
    """o_lat [B, h, d_c], lse [B, h] from the partials of mla_decode_fwd (see mla72.h)."""
    B, h, d_c = o_lat.shape
    _check("mla_combine", lib().mla_combine(
        _ptr(o_part), _ptr(lse_part), _ptr(seq_lens), int(block_size), int(max_blocks_per_seq),
        B, h, d_c, int(num_parts), _ptr(o_lat), dtype_code(o_lat.dtype), _ptr(lse),
        _stream(stream)))
    return o_lat


def mla_combine_out_proj(o_part, lse_part, seq_lens, block_size, max_blocks_per_seq, num_parts,
                         w_uv, out, o_lat=None, lse=None, dev_status=None, stream=None):
    """out [B, h, d_v] = the merged partials through W_UV (see mla72.h); o_lat
    [B, h, d_c] and lse [B, h] are written when given."""
    B, h, d_v = out.shape
    d_c = w_uv.shape[2]
    _check("mla_combine_out_proj", lib().mla_combine_out_proj(
        _ptr(o_part), _ptr(lse_part), _ptr(seq_lens), int(block_size), int(max_blocks_per_seq),
        B, h, d_c, int(num_parts), _ptr(w_uv), d_v, _ptr(out), dtype_code(out.dtype),
        _ptr(o_lat), dtype_code(o_lat.dtype) if o_lat is not None else 0, _ptr(lse),
        _ptr(dev_status), _stream(stream)))
    return out


def mla_decode_attend_noalloc(q_cat, kv: KVCache, block_table, seq_lens, num_parts, o_lat,
                              lse=None, *, softmax_scale=0.0, dev_status=None, stream=None):
    """mla_decode_fwd + mla_combine with the partials in the library's own
    device array, for callers that cannot allocate (see mla72.h)."""
    B, h, _ = q_cat.shape
    _check("mla_decode_attend_noalloc", lib().mla_decode_attend_noalloc(
        _ptr(q_cat), dtype_code(q_cat.dtype), ctypes.byref(kv), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, h, int(num_parts), float(softmax_scale),
        _ptr(o_lat), dtype_code(o_lat.dtype), _ptr(lse), _ptr(dev_status), _stream(stream)))
    return o_lat


def mla_out_proj(o_lat, w_uv, out, stream=None):
    """out[b, s, v] = sum_c o_lat[b, s, c] w_uv[s, v, c] (see mla72.h)."""
    B, h, d_c = o_lat.shape
    d_v = w_uv.shape[1]
    _check("mla_out_proj", lib().mla_out_proj(
        _ptr(o_lat), _ptr(w_uv), _ptr(out), B, h, d_c, d_v, dtype_code(o_lat.dtype),
        dtype_code(out.dtype), _stream(stream)))
    return out


def mla_cache_fill(c_kv, k_rope, cu_seqlens, max_len, block_table, kv: KVCache,
                   rope_theta=10000.0, dev_status=None, stream=None):
    """Write rows of B sequences into the paged cache (see mla72.h)."""
    B = cu_seqlens.shape[0] - 1
    _check("mla_cache_fill", lib().mla_cache_fill(
        _ptr(c_kv), _ptr(k_rope), dtype_code(c_kv.dtype), _ptr(cu_seqlens), B, int(max_len),
        _ptr(block_table), block_table.shape[1], ctypes.byref(kv), float(rope_theta),
        _ptr(dev_status), _stream(stream)))


def mla_cache_append(c_new, k_rope_new, pos, block_table, kv: KVCache, rope_theta=10000.0,
                     dev_status=None, stream=None):
    """Append one token per sequence at position pos[b] (see mla72.h)."""
    B = c_new.shape[0]
    _check("mla_cache_append", lib().mla_cache_append(
        _ptr(c_new), _ptr(k_rope_new), dtype_code(c_new.dtype), _ptr(pos), B, _ptr(block_table),
        block_table.shape[1], ctypes.byref(kv), float(rope_theta), _ptr(dev_status),
        _stream(stream)))


def mla_linear_workspace_bytes(M: int, K: int, N: int) -> int:
    return int(lib().mla_linear_workspace_bytes(M, K, N))


def mla_linear(x, w, y, workspace=None, stream=None):
    """y[m, n] = sum_k x[m, k] w[n, k] (see mla72.h); x [M, K], w [N, K], y [M, N]."""
    M, K = x.shape
    N = w.shape[0]
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("mla_linear", lib().mla_linear(
        _ptr(x), _ptr(w), _ptr(y), M, K, N, dtype_code(y.dtype), _ptr(workspace), ws,
        _stream(stream)))
    return y


def mla_fold_uv_into_o(w_uv, w_o, w_fold, stream=None):
    """w_fold [d_model, h * d_c] <- W_O merged with W_UV (see mla72.h)."""
    h, d_v, d_c = w_uv.shape
    d_model = w_o.shape[0]
    _check("mla_fold_uv_into_o", lib().mla_fold_uv_into_o(
        _ptr(w_uv), _ptr(w_o), _ptr(w_fold), h, d_c, d_v, d_model, _stream(stream)))
    return w_fold


def mla_prefill_query(q_nope, q_rope, cu_seqlens, max_len, q, rope_theta=10000.0, stream=None):
    """q [T, h, 192] <- [q_nope, RoPE(q_rope) at each token's position] (see mla72.h)."""
    B = cu_seqlens.shape[0] - 1
    h = q_nope.shape[1]
    _check("mla_prefill_query", lib().mla_prefill_query(
        _ptr(q_nope), _ptr(q_rope), _ptr(cu_seqlens), B, int(max_len), h, float(rope_theta),
        _ptr(q), _stream(stream)))
    return q


def mla_prefill_fwd(q, k_nope, k_rope, v, cu_seqlens, max_len, out, lse=None, *,
                    softmax_scale=0.0, dev_status=None, stream=None):
    """Causal prefill attention in the MHA form; out [T, h, 128] (see mla72.h)."""
    B = cu_seqlens.shape[0] - 1
    T, h, _ = q.shape
    _check("mla_prefill_fwd", lib().mla_prefill_fwd(
        _ptr(q), _ptr(k_nope), _ptr(k_rope), _ptr(v), _ptr(cu_seqlens), B, int(max_len), T, h,
        float(softmax_scale), _ptr(out), dtype_code(out.dtype), _ptr(lse), _ptr(dev_status),
        _stream(stream)))
    return out


def mla_paged_gather(kv: KVCache, block_table, cu_seqlens, max_len, latent_out=None,
                     rope_out=None, dev_status=None, stream=None):
    """Bit-exact logical rows out of the pool (see mla72.h)."""
    B = cu_seqlens.shape[0] - 1
    _check("mla_paged_gather", lib().mla_paged_gather(
        ctypes.byref(kv), _ptr(block_table), block_table.shape[1], _ptr(cu_seqlens), B,
        int(max_len), _ptr(latent_out), _ptr(rope_out), _ptr(dev_status), _stream(stream)))
