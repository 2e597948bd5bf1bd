"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerance: max|err| / max|ref| <= 1e-4 for the float32 workload and <= 2e-2
for bf16 / FP8 workloads, on the output after W_UV and on the latent output.
The log-sum-exp is compared with an absolute bound of the same size: an
error d in lse is a relative error of about d in the softmax denominator.
Paged gathers are bit-exact.
"""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle as O

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="session", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_72_b300 import build
    build.build()


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), "non-finite values in the GPU result"
    return float(np.abs(got - ref).max() / np.abs(ref).max())


def oracle_for(w, batch, heads=None):
    inp = O.workload_inputs_f64(w)
    seqs = [O.sequence_view(w, b, int(inp["lens"][b])) for b in batch]
    idx = list(batch)
    return O.decode_reference(inp["q_nope"][idx], inp["q_rope"][idx], inp["q_pos"][idx],
                              inp["w_uk"], inp["w_uv"], seqs, heads=heads)


def make(w, **kw):
    from mla_latent_kv_72_b300.workload import DeviceWorkload
    return DeviceWorkload(w, **kw)


def abs_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), "non-finite values in the GPU result"
    return float(np.abs(got - np.asarray(ref, dtype=np.float64)).max())


def check_against(ref, dw, batch, heads, tol):
    hs = list(range(dw.w.h)) if heads is None else list(heads)
    out = dw.out.float().cpu().numpy()[np.ix_(list(batch), hs)]
    o_lat = dw.o_lat.float().cpu().numpy()[np.ix_(list(batch), hs)]
    lse = dw.lse.float().cpu().numpy()[np.ix_(list(batch), hs)]
    e_out = rel_err(out, ref["out"])
    e_lat = rel_err(o_lat, ref["o_lat"])
    e_lse = abs_err(lse, ref["lse"])
    assert e_out <= tol, ("out", e_out)
    assert e_lat <= tol, ("o_lat", e_lat)
    assert e_lse <= tol, ("lse", e_lse)
    return e_out, e_lat, e_lse


def compare(w, dw, batch, heads, tol):
    return check_against(oracle_for(w, batch, heads), dw, batch, heads, tol)


# ----------------------------------------------------------------------------
# whole workloads, small enough for the oracle to check every output
# ----------------------------------------------------------------------------

SMALL_CASES = {
    "tiny_fp32_full": mi.workload(1),
    "small_bf16_ragged": mi.scaled(mi.workload(2), B=3, L=1000),
    "v3_bf16_two_seqs": mi.scaled(mi.workload(3), B=2, L=700),
    "paged_bf16_ragged": mi.scaled(mi.workload(4), B=6, L_range=(1, 700)),
    "fp8_bf16_long": mi.scaled(mi.workload(5), B=2, L=2500),
}


@pytest.mark.parametrize("flags", [0, 1], ids=["auto", "simt"])
@pytest.mark.parametrize("name", list(SMALL_CASES))
def test_small_workloads_match_oracle(name, flags):
    w = SMALL_CASES[name]
    dw = make(w)
    dw.step(flags=flags)
    torch.cuda.synchronize()
    assert dw.check_status() == 0
    tol = TOL["f32" if w.dtype == "f32" else "bf16"]
    compare(w, dw, range(w.B), None, tol)


@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 129])
def test_edge_lengths(L):
    w = mi.scaled(mi.workload(3), B=2, h=16, L=L)
    for ns in (1, 3):
        dw = make(w, num_parts=ns)
        dw.step()
        torch.cuda.synchronize()
        compare(w, dw, range(w.B), None, TOL["bf16"])


def test_fp32_tolerance_is_tight():
    # the float32 workload must sit well inside 1e-4
    w = mi.workload(1)
    dw = make(w)
    dw.step()
    torch.cuda.synchronize()
    e = compare(w, dw, range(w.B), None, TOL["f32"])
    assert max(e) < 1e-5


# ----------------------------------------------------------------------------
# part partition, split-KV and paging invariants
# ----------------------------------------------------------------------------

def expected_slots(lens, block_size, num_parts):
    """Partial slots p + b written under the part partition (its definition in
    include/mla72.h, restated here on the host)."""
    nb = [(int(L) + block_size - 1) // block_size for L in lens]
    T = sum(nb)
    P = min(num_parts, T)
    bounds = [p * T // P for p in range(P + 1)]
    slots = set()
    start = 0
    for b, n in enumerate(nb):
        for g in range(start, start + n):
            p = max(q for q in range(P) if bounds[q] <= g)
            slots.add(p + b)
        start += n
    return slots


# Two part counts split the key range at different blocks, so the online
# softmax runs against different running maxima and each P is rounded to bf16
# relative to a different maximum (up to 2^-9 of each term) before the P.C
# MMA.  Merged in float32, the two latent outputs may differ by that
# rounding, 2^-9 of max|o_lat|; their log-sum-exps (sums of float32 P, not
# rounded) by float32 rounding.  Stored in bf16 they may further differ by one
# output ulp, up to 2^-7 of max|o_lat|.
PART_TOL_F32 = 2.0 ** -9
PART_TOL_BF16 = 2.0 ** -7 + 2.0 ** -9
LSE_TOL_F32 = 1e-5


def _combine_f32(dw):
    from mla_latent_kv_72_b300 import binding as C
    o = torch.empty(dw.o_lat.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(dw.lse.shape, dtype=torch.float32, device="cuda")
    C.mla_combine(dw.o_part, dw.lse_part, dw.seq_lens, dw.w.block_size,
                  dw.block_table.shape[1], dw.num_parts, o, lse)
    torch.cuda.synchronize()
    return o.cpu().numpy(), lse.cpu().numpy()


# (B, L, num_parts): the last case gives every sequence 74 chunks (296 parts
# over 4 sequences of 128 blocks), the split-KV depth of the long-context use
@pytest.mark.parametrize("B,L,num_parts", [(2, 3000, 1), (2, 3000, 2), (2, 3000, 7),
                                           (2, 3000, 64), (2, 3000, 148), (4, 8192, 296)])
def test_part_count_invariance(B, L, num_parts):
    w = mi.scaled(mi.workload(3), B=B, h=128, L=L)
    dw1 = make(w, num_parts=1)
    dw1.step()
    dw = make(w, num_parts=num_parts)
    dw.step()
    torch.cuda.synchronize()
    ref = dw1.o_lat.float().cpu().numpy()
    o = dw.o_lat.float().cpu().numpy()
    assert np.abs(o - ref).max() / np.abs(ref).max() <= PART_TOL_BF16
    o1, l1 = _combine_f32(dw1)
    on, ln = _combine_f32(dw)
    assert np.abs(on - o1).max() / np.abs(o1).max() <= PART_TOL_F32
    assert abs_err(ln, l1) <= LSE_TOL_F32
    compare(w, dw, range(w.B), None, TOL["bf16"])


@pytest.mark.parametrize("flags", [0, 1], ids=["auto", "simt"])
def test_partial_slots_follow_the_partition(flags):
    # variable lengths, more parts than some sequences have blocks, and more
    # parts than the whole stream (16 sequences, 200 parts)
    w = mi.scaled(mi.workload(4), B=16, h=16, L_range=(1, 400))
    for num_parts in (5, 37, 200):
        dw = make(w, num_parts=num_parts)
        dw.o_part.fill_(float("nan"))
        dw.lse_part.fill_(float("nan"))
        dw.step(flags=flags)
        torch.cuda.synchronize()
        assert dw.check_status() == 0
        want = expected_slots(dw.lens_np, w.block_size, num_parts)
        written = ~torch.isnan(dw.lse_part[:, 0]).cpu().numpy()
        assert set(np.nonzero(written)[0].tolist()) == want
        compare(w, dw, range(w.B), None, TOL["bf16"])


def test_paged_permutation_is_bit_exact():
    base = mi.scaled(mi.workload(4), B=4, L_range=(100, 900))
    contig = mi.scaled(base, layout="contiguous")
    a = make(base, num_parts=3)
    b = make(contig, num_parts=3)
    assert not np.array_equal(a.table_np, b.table_np)
    for dw in (a, b):
        dw.step()
    torch.cuda.synchronize()
    assert torch.equal(a.o_part.view(torch.int32), b.o_part.view(torch.int32))
    assert torch.equal(a.out.view(torch.int32), b.out.view(torch.int32))


def test_bad_block_is_reported_not_dereferenced():
    w = mi.scaled(mi.workload(3), B=2, h=16, L=200)
    dw = make(w, num_parts=1)
    dw.block_table[1, 1] = dw.num_blocks + 1000
    dw.step()
    torch.cuda.synchronize()
    from mla_latent_kv_72_b300 import binding
    assert dw.check_status() == 1          # MLA_DEV_BAD_BLOCK
    dw.status.zero_()
    dw.step(flags=binding.MLA_DECODE_FORCE_SIMT)
    torch.cuda.synchronize()
    assert dw.check_status() == 1


# ----------------------------------------------------------------------------
# the cache writer and the gather
# ----------------------------------------------------------------------------

def _gather(dw):
    from mla_latent_kv_72_b300 import binding as C
    w = dw.w
    T = int(dw.lens_np.sum())
    cu = np.zeros(w.B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(dw.lens_np)
    ldt = torch.uint8 if w.latent_dtype == "fp8e4m3" else (torch.float32 if w.dtype == "f32" else torch.bfloat16)
    lat = torch.empty((T, w.d_c), dtype=ldt, device="cuda")
    rope = torch.empty((T, w.d_r), dtype=torch.float32 if w.dtype == "f32" else torch.bfloat16,
                       device="cuda")
    C.mla_paged_gather(dw.kv, dw.block_table, torch.from_numpy(cu).cuda(), dw.max_len, lat, rope,
                       dev_status=dw.status)
    torch.cuda.synchronize()
    return lat.cpu(), rope.float().cpu().numpy(), cu


@pytest.mark.parametrize("idx", [1, 4, 5])
def test_cache_fill_and_gather(idx):
    w = mi.scaled(mi.workload(idx), B=3, L=None, L_range=(1, 300)) if idx == 4 else \
        mi.scaled(mi.workload(idx), B=2, L=200)
    dw = make(w)
    lat, rope, cu = _gather(dw)
    assert dw.check_status() == 0
    src_dt = mi.latent_source_dtype(w)
    for b in range(w.B):
        L = int(dw.lens_np[b])
        c_src, kr_src = mi.sequence(w, b, L)
        got = lat[cu[b]:cu[b + 1]]
        if w.latent_dtype == "fp8e4m3":
            c32 = mi.storage_to_f64(c_src, src_dt).astype(np.float32)
            codes, scales, _ = O.quantized_latent_f64(c32, w.block_size)
            np.testing.assert_array_equal(got.numpy(), codes)          # bit-exact codes
            sc = dw.scale.cpu().numpy()[dw.table_np[b, : len(scales)]]
            np.testing.assert_array_equal(sc, scales)
        elif w.dtype == "bf16":
            np.testing.assert_array_equal(got.view(torch.int16).numpy().view(np.uint16), c_src)
        else:
            np.testing.assert_array_equal(got.numpy(), c_src)
        # rotated key against the float64 rotation of the same pre-image
        kr_ref = O.rope(mi.storage_to_f64(kr_src, w.dtype), np.arange(L))
        ulp = 2.0 ** -7 if w.dtype == "bf16" else 2.0 ** -20
        assert np.all(np.abs(rope[cu[b]:cu[b + 1]] - kr_ref) <= ulp * np.abs(kr_ref) + 1e-6)


def test_absorb_q_matches_oracle():
    for idx in (1, 3):
        w = mi.scaled(mi.workload(idx), B=5) if idx == 3 else mi.workload(idx)
        dw = make(w)
        dw.absorb()
        torch.cuda.synchronize()
        inp = O.workload_inputs_f64(w)
        ref = O.absorb_query(inp["q_nope"], inp["q_rope"], inp["q_pos"], inp["w_uk"])
        got = dw.q_cat.float().cpu().numpy()
        tol = 1e-5 if w.dtype == "f32" else 1e-2
        assert rel_err(got[..., :512], ref[..., :512]) < tol
        assert rel_err(got[..., 512:], ref[..., 512:]) < tol


def test_out_proj_matches_oracle():
    w = mi.scaled(mi.workload(3), B=5)
    dw = make(w)
    g = torch.Generator(device="cpu").manual_seed(0)
    o_lat = torch.randn((w.B, w.h, w.d_c), generator=g).to(torch.bfloat16)
    dw.o_lat.copy_(o_lat)
    dw.project()
    torch.cuda.synchronize()
    inp = O.workload_inputs_f64(w)
    ref = O.output_projection(o_lat.double().numpy(), inp["w_uv"])
    assert rel_err(dw.out.float().cpu().numpy(), ref) < 1e-3


# ----------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times
# ----------------------------------------------------------------------------
#
# The checker is the oracle's absorbed form (decode_absorbed), which the CPU
# pins tie to the non-absorbed definition at 1e-12; it is cheap enough to
# check every (sequence, head) output of the full workloads.

def absorbed_oracle(w, batch, heads=None):
    inp = O.workload_inputs_f64(w)
    seqs = [O.sequence_view(w, b, int(inp["lens"][b])) for b in batch]
    idx = list(batch)
    return O.decode_absorbed(inp["q_nope"][idx], inp["q_rope"][idx], inp["q_pos"][idx],
                             inp["w_uk"], inp["w_uv"], seqs, heads=heads)


def check_full(w, dw, heads=None, chunk=8):
    for b0 in range(0, w.B, chunk):
        batch = range(b0, min(w.B, b0 + chunk))
        check_against(absorbed_oracle(w, batch, heads), dw, batch, heads, TOL["bf16"])


# (workload, heads checked, num_parts): every output of workloads 2, 3 and 5;
# every sequence of workload 4 at 8 heads spread over the 128; workload 5 also
# with 256 parts, 64 or more key chunks per sequence
FULL_CASES = {
    "w2": (2, None, None),
    "w3": (3, None, None),
    "w4_8heads": (4, [0, 17, 38, 63, 64, 90, 111, 127], None),
    "w5": (5, None, None),
    "w5_256parts": (5, None, 256),
}


@pytest.mark.parametrize("case", list(FULL_CASES))
def test_full_size_every_output(case):
    idx, heads, parts = FULL_CASES[case]
    w = mi.workload(idx)
    dw = make(w, num_parts=parts)
    dw.step()
    torch.cuda.synchronize()
    assert dw.check_status() == 0
    assert torch.isfinite(dw.out).all()
    check_full(w, dw, heads)


# ----------------------------------------------------------------------------
# interface conventions and device-side error reporting
# ----------------------------------------------------------------------------

def test_sixteen_byte_aligned_buffers_give_the_same_bits():
    # q_cat and o_part 16-byte but not 32-byte aligned: the decode takes its
    # 16-byte access path, which must give the same bits as the 32-byte one
    from mla_latent_kv_72_b300 import binding as C
    w = mi.scaled(mi.workload(3), B=3, L=700)
    dw = make(w, num_parts=5)
    dw.absorb()
    dw.attend()
    torch.cuda.synchronize()
    q_big = torch.empty(dw.q_cat.numel() + 16, dtype=dw.q_cat.dtype, device="cuda")
    q_off = q_big[8:8 + dw.q_cat.numel()].view(dw.q_cat.shape)       # +16 bytes
    q_off.copy_(dw.q_cat)
    o_big = torch.empty(dw.o_part.numel() + 8, dtype=torch.float32, device="cuda")
    o_off = o_big[4:4 + dw.o_part.numel()].view(dw.o_part.shape)     # +16 bytes
    lse_off = torch.empty_like(dw.lse_part)
    assert q_off.data_ptr() % 32 == 16 and o_off.data_ptr() % 32 == 16
    o_off.fill_(float("nan"))
    C.mla_decode_fwd(q_off, dw.kv, dw.block_table, dw.seq_lens, dw.num_parts, o_off, lse_off,
                     dev_status=dw.status)
    torch.cuda.synchronize()
    assert dw.check_status() == 0
    slots = sorted(expected_slots(dw.lens_np, w.block_size, dw.num_parts))
    assert torch.equal(o_off[slots].view(torch.int32), dw.o_part[slots].view(torch.int32))
    assert torch.equal(lse_off[slots].view(torch.int32), dw.lse_part[slots].view(torch.int32))


def test_forced_wait_timeout_is_reported_and_the_device_stays_usable():
    # MLA_DECODE_TEST_WAIT_TIMEOUT makes the kernel's first MMA wait run on a
    # barrier that nothing signals, with a short limit: the status word must
    # read MLA_DEV_WAIT_TIMEOUT and the kernel must return (no hang, no trap)
    from mla_latent_kv_72_b300 import binding as C
    for idx in (3, 5):
        w = mi.scaled(mi.workload(idx), B=2, L=900)
        dw = make(w, num_parts=3)
        dw.absorb()
        torch.cuda.synchronize()
        C.mla_decode_fwd(dw.q_cat, dw.kv, dw.block_table, dw.seq_lens, dw.num_parts, dw.o_part,
                         dw.lse_part, dev_status=dw.status, flags=C.MLA_DECODE_TEST_WAIT_TIMEOUT)
        torch.cuda.synchronize()
        assert dw.check_status() == C.MLA_DEV_WAIT_TIMEOUT
        # the context is still good: a normal step afterwards is correct
        dw.status.zero_()
        dw.step()
        torch.cuda.synchronize()
        assert dw.check_status() == 0
        compare(w, dw, range(w.B), None, TOL["bf16"])
    # the SIMT kernel has no pipeline waits: the flag is refused there
    w = mi.workload(1)
    dw = make(w)
    with pytest.raises(C.MLAError):
        C.mla_decode_fwd(dw.q_cat, dw.kv, dw.block_table, dw.seq_lens, dw.num_parts, dw.o_part,
                         dw.lse_part, dev_status=dw.status,
                         flags=C.MLA_DECODE_TEST_WAIT_TIMEOUT)


@pytest.mark.parametrize("flags", [0, 1], ids=["auto", "simt"])
def test_length_beyond_the_table_is_clamped_and_reported(flags):
    # a length past max_blocks_per_seq * block_size is clamped to the table
    # and reported as MLA_DEV_BAD_LENGTH; the result equals the clamped length's
    from mla_latent_kv_72_b300 import binding as C
    w = mi.scaled(mi.workload(3), B=3, h=16, L=640)
    dw = make(w, num_parts=4)
    dw.step(flags=flags)
    torch.cuda.synchronize()
    ref_out = dw.out.clone()
    dw.seq_lens[1] = 640 + 64 * 5
    dw.status.zero_()
    dw.attend(flags=flags)
    torch.cuda.synchronize()
    assert dw.check_status() == C.MLA_DEV_BAD_LENGTH
    dw.seq_lens[1] = 640
    dw.combine()
    dw.project()
    torch.cuda.synchronize()
    assert torch.equal(dw.out.view(torch.int32), ref_out.view(torch.int32))


# ----------------------------------------------------------------------------
# the per-step cache append (one token per sequence per call)
# ----------------------------------------------------------------------------

APPEND_CASES = {
    "bf16_contiguous": mi.scaled(mi.workload(3), B=3, h=16, L=None, L_range=(70, 300),
                                 layout="contiguous"),
    "bf16_paged": mi.scaled(mi.workload(4), B=4, h=16, L_range=(70, 300)),
    "fp8": mi.scaled(mi.workload(5), B=3, h=16, L=None, L_range=(70, 300)),
}


@pytest.mark.parametrize("name", list(APPEND_CASES))
def test_cache_append_matches_oracle(name):
    # each sequence is filled to L - k rows (k crosses a block boundary) and
    # its last k rows are appended one token per call; the cache must then
    # hold the oracle's append result bit for bit (codes and scales for the
    # FP8 latent; the rotated keys equal the fill's), and the decode over it
    # must match the oracle
    w = APPEND_CASES[name]
    lens = mi.lengths(w)
    k = np.array([40, 65, 1, 64][: w.B])[: w.B]
    fill = np.maximum(lens - k, 0)
    dw = make(w, fill_lens=fill, num_parts=5)
    ref = make(w, num_parts=5)                  # the same rows, filled at once
    calls = dw.append_tail()
    assert calls == int((lens - fill).max())
    assert dw.check_status() == 0
    lat, rope, cu = _gather(dw)
    lat_f, rope_f, _ = _gather(ref)
    np.testing.assert_array_equal(rope, rope_f)                 # same rotation arithmetic
    src_dt = mi.latent_source_dtype(w)
    for b in range(w.B):
        L = int(lens[b])
        c_src, _ = mi.sequence(w, b, L)
        got = lat[cu[b]:cu[b + 1]]
        if w.latent_dtype == "fp8e4m3":
            c32 = mi.storage_to_f64(c_src, src_dt).astype(np.float32)
            codes, scales, _ = O.quantized_latent_appended(c32, w.block_size, int(fill[b]))
            np.testing.assert_array_equal(got.numpy(), codes)
            sc = dw.scale.cpu().numpy()[dw.table_np[b, : len(scales)]]
            np.testing.assert_array_equal(sc, scales)
        else:
            ref_rows = lat_f[cu[b]:cu[b + 1]]
            bits = torch.int16 if got.element_size() == 2 else torch.int32
            assert torch.equal(got.view(bits), ref_rows.view(bits))
    dw.step()
    torch.cuda.synchronize()
    assert dw.check_status() == 0
    inp = O.workload_inputs_f64(w)
    seqs = [O.sequence_view(w, b, int(lens[b]), n_fill=int(fill[b])) for b in range(w.B)]
    oref = O.decode_reference(inp["q_nope"], inp["q_rope"], inp["q_pos"], inp["w_uk"],
                              inp["w_uv"], seqs)
    check_against(oref, dw, range(w.B), None, TOL["bf16"])


def test_cache_append_reports_bad_positions():
    from mla_latent_kv_72_b300 import binding as C
    w = mi.scaled(mi.workload(3), B=2, h=16, L=100)
    dw = make(w)
    c = torch.zeros((2, 512), dtype=torch.bfloat16, device="cuda")
    kr = torch.zeros((2, 64), dtype=torch.bfloat16, device="cuda")
    before = dw.pool.clone()
    pos = torch.tensor([-1, 64 * dw.block_table.shape[1]], dtype=torch.int32, device="cuda")
    C.mla_cache_append(c, kr, pos, dw.block_table, dw.kv, dev_status=dw.status)
    torch.cuda.synchronize()
    assert dw.check_status() == C.MLA_DEV_BAD_LENGTH
    assert torch.equal(dw.pool.view(torch.int16), before.view(torch.int16))   # nothing written


# ----------------------------------------------------------------------------
# multi-token decode (q_len new tokens per sequence, causal among them)
# ----------------------------------------------------------------------------

MULTI_CASES = {
    # 64 rows (one CTA pair per part); lengths below q_len, at and around block edges
    "h16_q4_edges": (mi.scaled(mi.workload(3), B=9, h=16, L=None,
                               lens=(1, 2, 3, 63, 64, 65, 66, 67, 300)), 4),
    # 256 rows: two row groups per part
    "h128_q2": (mi.scaled(mi.workload(4), B=3, L_range=(60, 400)), 2),
    # FP8 latent, 384 rows: three row groups
    "fp8_h128_q3": (mi.scaled(mi.workload(5), B=2, L=None, lens=(130, 259)), 3),
}


def check_multi(w, q_len, dw, tol):
    inp = O.workload_inputs_f64(w)
    qn, qr = mi.queries_multi(w, q_len)
    seqs = [O.sequence_view(w, b, int(inp["lens"][b])) for b in range(w.B)]
    ref = O.decode_reference_multi(mi.storage_to_f64(qn, w.dtype), mi.storage_to_f64(qr, w.dtype),
                                   inp["w_uk"], inp["w_uv"], seqs)
    out = dw.out.float().cpu().numpy()
    o_lat = dw.o_lat.float().cpu().numpy()
    lse = dw.lse.float().cpu().numpy()
    # tokens that see no row: output 0 and lse -inf, as in the oracle
    empty = np.isneginf(ref["lse"])
    np.testing.assert_array_equal(np.isneginf(lse), empty)
    assert np.all(out[empty] == 0) and np.all(o_lat[empty] == 0)
    assert rel_err(out, ref["out"]) <= tol
    assert rel_err(o_lat, ref["o_lat"]) <= tol
    assert abs_err(lse[~empty], ref["lse"][~empty]) <= tol


@pytest.mark.parametrize("flags", [0, 1], ids=["auto", "simt"])
@pytest.mark.parametrize("name", list(MULTI_CASES))
def test_multi_token_decode_matches_oracle(name, flags):
    w, q_len = MULTI_CASES[name]
    dw = make(w, q_len=q_len, num_parts=7)
    dw.step(flags=flags)
    torch.cuda.synchronize()
    assert dw.check_status() == 0
    check_multi(w, q_len, dw, TOL["bf16"])


def test_multi_token_entry_with_one_token_equals_the_one_token_decode():
    from mla_latent_kv_72_b300 import binding as C
    w = mi.scaled(mi.workload(4), B=4, L_range=(1, 500))
    dw = make(w, num_parts=9)
    dw.absorb()
    dw.attend()
    torch.cuda.synchronize()
    o2 = torch.full_like(dw.o_part, float("nan"))
    l2 = torch.full_like(dw.lse_part, float("nan"))
    C.mla_decode_fwd_multi(dw.q_cat.unsqueeze(1), dw.kv, dw.block_table, dw.seq_lens,
                           dw.num_parts, o2, l2, dev_status=dw.status)
    torch.cuda.synchronize()
    slots = sorted(expected_slots(dw.lens_np, w.block_size, dw.num_parts))
    assert torch.equal(o2[slots].view(torch.int32), dw.o_part[slots].view(torch.int32))
    assert torch.equal(l2[slots].view(torch.int32), dw.lse_part[slots].view(torch.int32))


# ----------------------------------------------------------------------------
# linear layers, the W_UV / W_O fold and the step at the hidden-state boundary
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("M,K,N", [(64, 7168, 1536), (5, 512, 256), (300, 1024, 384),
                                   (64, 16384, 1024)])
def test_linear_matches_float64(M, K, N):
    from mla_latent_kv_72_b300 import binding as C
    g = torch.Generator(device="cpu").manual_seed(M * 7 + N)
    x = torch.randn((M, K), generator=g).to(torch.bfloat16)
    wt = (torch.randn((N, K), generator=g) / K ** 0.5).to(torch.bfloat16)
    ref = x.double() @ wt.double().T
    ws_bytes = C.mla_linear_workspace_bytes(M, K, N)
    ws = torch.empty(max(1, ws_bytes // 4), dtype=torch.float32, device="cuda")
    xg, wg = x.cuda(), wt.cuda()
    for dt, tol in ((torch.float32, 1e-5), (torch.bfloat16, 2.0 ** -8)):
        y = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        C.mla_linear(xg, wg, y, ws)
        torch.cuda.synchronize()
        assert rel_err(y.double().cpu().numpy(), ref.numpy()) <= tol
    # the same inputs give the same bits (fixed-order sum of the splits)
    y2 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    y3 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    C.mla_linear(xg, wg, y2, ws)
    C.mla_linear(xg, wg, y3, ws)
    torch.cuda.synchronize()
    assert torch.equal(y2.view(torch.int32), y3.view(torch.int32))


def test_fold_matches_oracle():
    from mla_latent_kv_72_b300 import binding as C
    w = mi.scaled(mi.workload(3), B=2, h=16)
    _, wuv = mi.weights(w)
    hid = mi.hidden_inputs(w, 1024, 256)
    from mla_latent_kv_72_b300.workload import storage_to_torch
    wuv_t = storage_to_torch(wuv, "bf16", "cuda")
    wo_t = storage_to_torch(hid["w_o"], "bf16", "cuda")
    fold = torch.empty((1024, 16 * 512), dtype=torch.bfloat16, device="cuda")
    C.mla_fold_uv_into_o(wuv_t, wo_t, fold)
    torch.cuda.synchronize()
    ref = O.fold_uv_into_o(mi.storage_to_f64(wuv, "bf16"), mi.storage_to_f64(hid["w_o"], "bf16"))
    assert rel_err(fold.float().cpu().numpy(), ref) <= 2.0 ** -8


@pytest.mark.parametrize("folded", [False, True], ids=["w_uv_then_w_o", "folded"])
def test_step_from_hidden_state_matches_oracle(folded):
    w = mi.scaled(mi.workload(4), B=5, h=16, L_range=(1, 600))
    d_model, d_cq = 1024, 256
    dw = make(w, num_parts=7)
    dw.enable_hidden(d_model, d_cq)
    y = dw.hidden_step(folded=folded)
    torch.cuda.synchronize()
    assert dw.check_status() == 0
    inp = O.workload_inputs_f64(w)
    hid = {k: mi.storage_to_f64(v, "bf16") for k, v in mi.hidden_inputs(w, d_model, d_cq).items()}
    seqs = [O.sequence_view(w, b, int(inp["lens"][b])) for b in range(w.B)]
    y_ref, _ = O.decode_from_hidden(hid["x"], hid["w_dq"], hid["w_uq"], hid["w_qr"], inp["w_uk"],
                                    inp["w_uv"], hid["w_o"], inp["q_pos"], seqs)
    assert rel_err(y.cpu().numpy(), y_ref) <= TOL["bf16"]


# ----------------------------------------------------------------------------
# prefill in the MHA form (causal, d_qk = 192, d_v = 128)
# ----------------------------------------------------------------------------

PREFILL_CASES = {
    # lengths around the 128-token tile: 1, 127, 128, 129, 300
    "h4_edges": mi.scaled(mi.workload(3), B=5, h=4, L=None, lens=(1, 127, 128, 129, 300)),
    "h16_ragged": mi.scaled(mi.workload(4), B=3, h=16, L_range=(200, 700)),
    # up to 17 key tiles per query tile: the K/V ring wraps many times, and
    # the last CTA of each sequence has only its first query tile
    "h2_long": mi.scaled(mi.workload(3), B=2, h=2, L=None, lens=(1500, 2100)),
    # mixed lengths with a one-token sequence between two long ones (most query
    # tiles of the grid are empty for it)
    "h32_mixed": mi.scaled(mi.workload(4), B=3, h=32, L=None, lens=(700, 1, 1300)),
}


@pytest.mark.parametrize("name", list(PREFILL_CASES))
def test_prefill_matches_oracle(name):
    from mla_latent_kv_72_b300.workload import DevicePrefill
    w = PREFILL_CASES[name]
    pf = DevicePrefill(w)
    pf.run()
    torch.cuda.synchronize()
    assert pf.dw.check_status() == 0
    out = pf.out.cpu().numpy()
    lse = pf.lse.cpu().numpy()
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    inp = O.workload_inputs_f64(w)
    qn, qr = mi.prefill_queries(w)
    qn = mi.storage_to_f64(qn, w.dtype)
    qr = mi.storage_to_f64(qr, w.dtype)
    cu = np.concatenate([[0], np.cumsum(pf.lens_np)])
    for b in range(w.B):
        L = int(pf.lens_np[b])
        c, kr = O.sequence_view(w, b, L)
        r = O.prefill_reference(qn[cu[b]:cu[b + 1]], qr[cu[b]:cu[b + 1]], inp["w_uk"],
                                inp["w_uv"], c, kr)
        assert rel_err(out[cu[b]:cu[b + 1]], r["out"]) <= TOL["bf16"], b
        assert abs_err(lse[cu[b]:cu[b + 1]], r["lse"]) <= TOL["bf16"], b


COMBINE_PROJ_CASES = {
    "v3_b3": (3, dict(B=3, L=900), None),
    # two batch tiles of 64 rows, the second ragged; few parts per sequence
    "v3_b70": (3, dict(B=70, h=16, L=700), 40),
    "paged_b5": (4, dict(B=5, h=16, L_range=(1, 2000)), 37),
    "fp8_b2_256parts": (5, dict(B=2, L=20000), 256),
}


def _same_bits(a, b):
    bits = torch.int16 if a.element_size() == 2 else torch.int32
    return a.shape == b.shape and torch.equal(a.view(bits), b.view(bits))


@pytest.mark.parametrize("case", list(COMBINE_PROJ_CASES))
def test_combine_out_proj_equals_the_pair(case):
    """mla_combine_out_proj: o_lat and lse bit for bit equal to mla_combine's,
    out equal to mla_out_proj's to float32 rounding, and to the oracle."""
    idx, kw, parts = COMBINE_PROJ_CASES[case]
    w = mi.scaled(mi.workload(idx), **kw)
    dw = make(w, num_parts=parts)
    dw.absorb()
    dw.attend()
    dw.combine()
    dw.project()
    torch.cuda.synchronize()
    ref = (dw.o_lat.clone(), dw.lse.clone(), dw.out.clone())
    for t in (dw.o_lat, dw.lse, dw.out):
        t.fill_(float("nan"))
    dw.combine_project()
    torch.cuda.synchronize()
    assert dw.check_status() == 0
    assert _same_bits(dw.o_lat, ref[0]) and _same_bits(dw.lse, ref[1])
    o, r = dw.out.float().cpu().numpy(), ref[2].float().cpu().numpy()
    assert np.all(np.isfinite(o))
    assert np.abs(o - r).max() <= 1e-5 * np.abs(r).max()
    compare(w, dw, range(min(w.B, 2)), [0, 7], TOL["bf16"])
