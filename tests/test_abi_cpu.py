"""The C-ABI library builds for sm_103a, loads, exports what include/mla72.h
declares, and rejects bad arguments on the host before launching anything.
No test here needs a GPU: every call below fails its host-side checks."""
import ctypes
import os
import re

import pytest

import mla_latent_kv_72_b300 as M
from mla_latent_kv_72_b300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla72.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return M.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert set(_declared_functions()) == set(M.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_binding_constants_match_the_header():
    from mla_latent_kv_72_b300 import binding
    defines = dict(re.findall(r"#define (MLA_[A-Z0-9_]+) (\d+)u?", open(HEADER).read()))
    assert defines
    for name, value in defines.items():
        assert getattr(binding, name) == int(value), name


def test_library_is_built_for_sm103a(lib):
    assert "arch=compute_103a,code=sm_103a" in " ".join(B.ARCH)
    assert os.path.getsize(M.library_path()) > 0


def test_status_strings_and_version(lib):
    assert M.mla_version() == 100
    assert M.mla_status_string(0) == "ok"
    for st in range(-6, 0):
        assert M.mla_status_string(st) != "unknown status"
    assert M.mla_status_string(-99) == "unknown status"


def test_cache_bytes_per_token(lib):
    assert M.mla_cache_bytes_per_token(M.MLA_BF16, M.MLA_BF16, 512, 64, 64) == 1152.0
    assert M.mla_cache_bytes_per_token(M.MLA_F32, M.MLA_F32, 512, 64, 64) == 2304.0
    assert M.mla_cache_bytes_per_token(M.MLA_FP8E4M3, M.MLA_BF16, 512, 64, 64) == 640.0625
    assert M.mla_cache_bytes_per_token(M.MLA_BF16, M.MLA_FP8E4M3, 512, 64, 64) < 0
    assert M.mla_cache_bytes_per_token(M.MLA_BF16, M.MLA_BF16, 0, 64, 64) < 0


# Fake device addresses: never dereferenced, because every call below fails
# a host check first.  (Aligned ones pass the alignment check.)
A = 1 << 20          # 16-byte aligned
A2 = (1 << 20) + 32
MIS = (1 << 20) + 8  # not 16-byte aligned


def _kv(latent=A, rope=A + 1024, scale=None, lstride=576, rstride=576, ldt=M.MLA_BF16,
        rdt=M.MLA_BF16, nblk=8, bs=64, d_c=512, d_r=64):
    return M.KVCache(latent, rope, scale, lstride, rstride, ldt, rdt, nblk, bs, d_c, d_r)


def test_absorb_q_host_checks(lib):
    f = lib.mla_absorb_q
    ok = dict(B=2, h=4, dn=128, dc=512, dr=64, dt=M.MLA_BF16)
    args = lambda **k: [k.get("qn", A), A, A, A, k.get("qc", A2), k.get("B", 2), k.get("h", 4),
                        k.get("dn", 128), k.get("dc", 512), k.get("dr", 64),
                        k.get("dt", M.MLA_BF16), k.get("theta", 10000.0), None]
    assert f(*args(qn=None)) == -1
    assert f(*args(B=0)) == -1
    assert f(*args(h=-3)) == -1
    assert f(*args(theta=0.0)) == -1
    assert f(*args(dt=M.MLA_FP8E4M3)) == -3
    assert f(*args(dc=500)) == -4
    assert f(*args(dr=63)) == -4
    assert f(*args(qc=MIS)) == -2


def test_decode_fwd_host_checks(lib):
    f = lib.mla_decode_fwd

    def call(q=A, qdt=M.MLA_BF16, kv=None, table=A, maxb=4, lens=A, B=2, h=128, ns=2, o=A,
             lse=A, flags=0):
        kv = _kv() if kv is None else kv
        return f(q, qdt, ctypes.byref(kv), table, maxb, lens, B, h, ns, 0.0, o, lse, None, flags,
                 None)

    assert call(q=None) == -1
    assert call(table=None) == -1
    assert call(B=0) == -1
    assert call(ns=0) == -1
    assert call(maxb=0) == -1
    assert call(flags=7) == -1
    assert call(ns=1025) == -4
    assert call(kv=_kv(nblk=0)) == -1
    assert call(kv=_kv(d_c=500)) == -4
    assert call(kv=_kv(latent=MIS)) == -2
    assert call(kv=_kv(lstride=577)) == -2            # 1154-byte rows
    assert call(kv=_kv(lstride=100)) == -4            # stride below d_c
    assert call(kv=_kv(ldt=M.MLA_FP8E4M3, scale=None, rdt=M.MLA_BF16, lstride=512, rstride=64)) == -1
    assert call(kv=_kv(ldt=M.MLA_FP8E4M3, scale=A, rdt=M.MLA_F32, lstride=512, rstride=64)) == -3
    assert call(kv=_kv(ldt=M.MLA_BF16, rdt=M.MLA_F32)) == -3
    assert call(qdt=M.MLA_F32) == -3                   # f32 query over a bf16 cache
    assert call(qdt=M.MLA_FP8E4M3) == -3
    assert call(q=MIS) == -2


def test_decode_num_partials(lib):
    assert lib.mla_decode_num_partials(64, 74) == 137
    assert lib.mla_decode_num_partials(1, 1) == 1
    assert lib.mla_decode_num_partials(0, 4) == -1
    assert lib.mla_decode_num_partials(4, 0) == -1
    assert lib.mla_decode_num_partials(4, 1025) == -1


def test_combine_and_out_proj_host_checks(lib):
    c = lib.mla_combine

    def call(op=A, seq=A, bs=64, maxb=4, B=2, h=4, d_c=512, parts=2, o=A, odt=M.MLA_F32):
        return c(op, A, seq, bs, maxb, B, h, d_c, parts, o, odt, None, None)

    assert call(op=None) == -1
    assert call(seq=None) == -1
    assert call(parts=0) == -1
    assert call(bs=0) == -1
    assert call(maxb=0) == -1
    assert call(d_c=510) == -4
    assert call(parts=2000) == -4
    assert call(odt=M.MLA_FP8E4M3) == -3
    assert call(o=MIS) == -2
    o = lib.mla_out_proj
    assert o(None, A, A, 2, 4, 512, 128, 1, 0, None) == -1
    assert o(A, A, A, 2, 4, 512, 0, 1, 0, None) == -1
    assert o(A, A, A, 2, 4, 500, 128, 1, 0, None) == -4
    assert o(A, A, A, 2, 4, 512, 128, 2, 0, None) == -3
    assert o(A, A, MIS, 2, 4, 512, 128, 1, 0, None) == -2


def test_cache_fill_and_gather_host_checks(lib):
    f = lib.mla_cache_fill
    kv = _kv()
    assert f(None, A, 1, A, 2, 100, A, 4, ctypes.byref(kv), 10000.0, None, None) == -1
    assert f(A, A, 1, A, 0, 100, A, 4, ctypes.byref(kv), 10000.0, None, None) == -1
    assert f(A, A, 1, A, 2, 100, A, 4, ctypes.byref(kv), -1.0, None, None) == -1
    assert f(A, A, 0, A, 2, 100, A, 4, ctypes.byref(kv), 10000.0, None, None) == -3
    kv8 = _kv(ldt=M.MLA_FP8E4M3, scale=A, lstride=512, rstride=64)
    assert f(A, A, 0, A, 2, 100, A, 4, ctypes.byref(kv8), 10000.0, None, None) == -3
    g = lib.mla_paged_gather
    assert g(ctypes.byref(kv), None, 4, A, 2, 100, A, A, None, None) == -1
    assert g(ctypes.byref(kv), A, 4, A, 2, -1, A, A, None, None) == -1
    assert g(ctypes.byref(_kv(rope=MIS)), A, 4, A, 2, 100, A, A, None, None) == -2


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from mla_latent_kv_72_b300 import binding
    monkeypatch.setattr(binding, "_LIB", None)
    monkeypatch.setattr(binding, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        binding.lib()


def test_decode_multi_token_host_checks(lib):
    f = lib.mla_decode_fwd_multi

    def call(q_len=2, h=128, kv=None):
        kv = _kv() if kv is None else kv
        return f(A, M.MLA_BF16, ctypes.byref(kv), A, 4, A, 2, q_len, h, 2, 0.0, A, A, None, 0,
                 None)

    assert call(q_len=0) == -1
    assert call(q_len=M.MLA_MAX_Q_LEN + 1) == -4
    assert call(q_len=8, h=1024) == -4                 # q_len * h > 4096 query rows
    assert call(kv=_kv(nblk=0)) == -1


def test_cache_append_host_checks(lib):
    f = lib.mla_cache_append
    kv = _kv()

    def call(c=A, kr=A, sdt=M.MLA_BF16, pos=A, B=2, table=A, maxb=4, kv=kv, theta=10000.0):
        return f(c, kr, sdt, pos, B, table, maxb, ctypes.byref(kv), theta, None, None)

    assert call(c=None) == -1
    assert call(pos=None) == -1
    assert call(B=0) == -1
    assert call(maxb=0) == -1
    assert call(theta=0.0) == -1
    assert call(kv=_kv(nblk=0)) == -1
    assert call(sdt=M.MLA_FP8E4M3) == -3
    assert call(sdt=M.MLA_F32) == -3                   # f32 rows into a bf16 cache
    kv8 = _kv(ldt=M.MLA_FP8E4M3, scale=A, lstride=512, rstride=64)
    assert call(sdt=M.MLA_F32, kv=kv8) == -3           # FP8 latent takes bf16 rows
    assert call(c=MIS) == -2


def test_linear_and_fold_host_checks(lib):
    ws = lib.mla_linear_workspace_bytes
    # 7168-long contraction at 64 rows: eight 896-long splits of float32 partials
    assert ws(64, 7168, 1536) == 8 * 64 * 1536 * 4
    assert ws(64, 128, 128) == 0                       # one split: no workspace
    assert ws(64, 100, 128) == 0 and ws(0, 128, 128) == 0
    f = lib.mla_linear
    assert f(None, A, A, 64, 128, 128, M.MLA_BF16, None, 0, None) == -1
    assert f(A, A, A, 0, 128, 128, M.MLA_BF16, None, 0, None) == -1
    assert f(A, A, A, 64, 128, 128, M.MLA_FP8E4M3, None, 0, None) == -3
    assert f(A, A, A, 64, 100, 128, M.MLA_BF16, None, 0, None) == -4
    assert f(A, A, A, 64, 128, 100, M.MLA_BF16, None, 0, None) == -4
    assert f(A, MIS, A, 64, 128, 128, M.MLA_BF16, None, 0, None) == -2
    need = 8 * 64 * 1536 * 4
    assert f(A, A, A, 64, 7168, 1536, M.MLA_BF16, None, 0, None) == -1
    assert f(A, A, A, 64, 7168, 1536, M.MLA_BF16, A, need - 1, None) == -1
    assert f(A, A, A, 64, 7168, 1536, M.MLA_BF16, MIS, need, None) == -2
    g = lib.mla_fold_uv_into_o
    assert g(None, A, A, 4, 512, 128, 1024, None) == -1
    assert g(A, A, A, 0, 512, 128, 1024, None) == -1
    assert g(A, A, A, 4, 256, 128, 1024, None) == -4
    assert g(A, A, MIS, 4, 512, 128, 1024, None) == -2


def test_prefill_host_checks(lib):
    q = lib.mla_prefill_query
    assert q(None, A, A, 2, 100, 4, 10000.0, A, None) == -1
    assert q(A, A, A, 0, 100, 4, 10000.0, A, None) == -1
    assert q(A, A, A, 2, 100, 4, 0.0, A, None) == -1
    assert q(A, MIS, A, 2, 100, 4, 10000.0, A, None) == -2
    assert q(A, A, A, 2, 0, 4, 10000.0, A, None) == 0  # no rows: nothing to launch
    f = lib.mla_prefill_fwd

    def call(qp=A, kn=A, kr=A, v=A, cu=A, B=2, max_len=100, T=150, h=4, out=A,
             odt=M.MLA_BF16):
        return f(qp, kn, kr, v, cu, B, max_len, T, h, 0.0, out, odt, None, None, None)

    assert call(qp=None) == -1
    assert call(cu=None) == -1
    assert call(B=0) == -1
    assert call(T=0) == -1
    assert call(odt=M.MLA_FP8E4M3) == -3
    assert call(h=70000) == -4
    assert call(kr=MIS) == -2


def test_combine_out_proj_host_checks(lib):
    f = lib.mla_combine_out_proj

    def call(op=A, seq=A, B=2, h=4, d_c=512, parts=2, w=A, d_v=128, out=A, odt=M.MLA_BF16,
             olat=None, oldt=M.MLA_BF16):
        return f(op, A, seq, 64, 4, B, h, d_c, parts, w, d_v, out, odt, olat, oldt, None, None,
                 None)

    assert call(op=None) == -1
    assert call(w=None) == -1
    assert call(B=0) == -1
    assert call(parts=0) == -1
    assert call(odt=M.MLA_FP8E4M3) == -3
    assert call(olat=A, oldt=M.MLA_FP8E4M3) == -3
    assert call(d_c=256) == -4
    assert call(d_v=64) == -4
    assert call(parts=2000) == -4
    assert call(w=MIS) == -2
    assert call(olat=MIS) == -2
