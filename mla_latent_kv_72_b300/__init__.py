"""B300 (sm_103a) MLA absorbed decode over a latent KV cache.

Python binding of the C ABI declared in ``include/mla72.h``: argument
marshalling only (torch tensors -> device pointers, the current CUDA stream).
Every step of the decode runs in the CUDA kernels of ``libmla72.so``; there
is no CPU path.  Importing this package does not load the library; the first
call does, and fails loudly if the library is missing.
"""
from .binding import (  # noqa: F401
    MLA_BF16,
    MLA_F32,
    MLA_FP8E4M3,
    MLA_MAX_PARTS,
    MLA_MAX_Q_LEN,
    MLAError,
    KVCache,
    dtype_code,
    lib,
    library_path,
    mla_absorb_q,
    mla_cache_bytes_per_token,
    mla_cache_append,
    mla_cache_fill,
    mla_combine,
    mla_combine_out_proj,
    mla_decode_fwd,
    mla_decode_fwd_multi,
    mla_decode_num_partials,
    mla_decode_attend_noalloc,
    default_num_parts,
    mla_out_proj,
    mla_linear,
    mla_linear_workspace_bytes,
    mla_fold_uv_into_o,
    mla_paged_gather,
    mla_prefill_fwd,
    mla_prefill_query,
    mla_status_string,
    mla_version,
    EXPORTED_SYMBOLS,
)
