"""Pins for the float64 oracle: facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: numbers the
pages print, closed forms of RoPE, special cases of softmax attention, the
absorption identity between two different computations, and brute-force
scalar loops written independently of the oracle's matrix code.
"""
import json
import math
import os

import numpy as np
import pytest

import mla_inputs as mi
import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand_case(rng, B=2, h=3, d_c=16, d_r=8, d_nope=6, d_v=5, lens=(7, 3)):
    qn = rng.standard_normal((B, h, d_nope))
    qr = rng.standard_normal((B, h, d_r))
    wuk = rng.standard_normal((h, d_nope, d_c)) / math.sqrt(d_c)
    wuv = rng.standard_normal((h, d_v, d_c)) / math.sqrt(d_c)
    seqs = [(rng.standard_normal((L, d_c)), rng.standard_normal((L, d_r))) for L in lens]
    q_pos = np.array([L - 1 for L in lens])
    return qn, qr, q_pos, wuk, wuv, seqs


# ----------------------------------------------------------------------------
# cache arithmetic printed on the pages
# ----------------------------------------------------------------------------

def test_cache_arithmetic_matches_printed_values():
    g = _golden("cache_arithmetic.json")
    v3 = g["v3_geometry"]
    mla = O.cache_elements_per_token_layer("mla", d_c=v3["d_c"], d_r=v3["d_r"])
    mha = O.cache_elements_per_token_layer("mha", n_h=v3["n_h"], d_h=v3["d_h"])
    assert mla == v3["mla_elements_per_layer"]
    assert mla * v3["layers"] == v3["mla_elements_all_layers"]
    assert mla * v3["layers"] * v3["bytes_per_element"] == v3["mla_bytes_all_layers"]
    assert round(mla * v3["layers"] * 2 / 1024, 1) == v3["mla_kib_all_layers_1dp"]
    assert mha == v3["mha_elements_per_layer"]
    assert mha * v3["layers"] == v3["mha_elements_all_layers"]
    assert round(mha / mla, 1) == v3["mha_over_mla_ratio_1dp"]

    gq = g["gqa8_comparison"]
    gqa = O.cache_elements_per_token_layer("gqa", n_g=gq["n_g"], d_h=gq["d_h"])
    assert gqa == gq["gqa_elements_per_layer"]
    assert round(100 * (1 - mla / gqa), 1) == gq["mla_reduction_vs_gqa8_pct_1dp"]
    assert round(100 * (1 - mla / mha), 1) == gq["mla_reduction_vs_mha_pct_1dp"]

    qw = g["qwen72b_gqa"]
    gqa72 = O.cache_elements_per_token_layer("gqa", n_g=qw["n_g"], d_h=qw["d_h"]) * qw["layers"]
    assert gqa72 == qw["gqa_elements_all_layers"]
    assert gqa72 * 2 == qw["gqa_bytes_all_layers"]
    assert O.cache_elements_per_token_layer("mha", n_h=qw["n_h"], d_h=qw["d_h"]) * qw["layers"] \
        == qw["mha_elements_all_layers"]
    assert O.cache_elements_per_token_layer("mqa", d_h=qw["d_h"]) * qw["layers"] * 2 / 1024 \
        == qw["mqa_kib_all_layers"]


def test_cache_bytes_per_token_layouts():
    # bf16 packed row: (d_c + d_r) * 2 = 1152 bytes; MHA twin at h=128: 65,536 bytes
    assert O.mla_cache_bytes_per_token("bf16", "bf16", 512, 64, 64) == 1152
    assert O.cache_elements_per_token_layer("mha", n_h=128, d_h=128) * 2 == 65536
    assert O.mla_cache_bytes_per_token("f32", "f32", 512, 64, 64) == 2304
    # FP8 latent + bf16 rope + one float32 scale per 64-token block
    assert O.mla_cache_bytes_per_token("fp8e4m3", "bf16", 512, 64, 64) == 512 + 128 + 4 / 64


# ----------------------------------------------------------------------------
# RoPE closed forms (kexue.fm "Part 2": R_m R_n^T = R_{m-n})
# ----------------------------------------------------------------------------

def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).standard_normal((5, 64))
    np.testing.assert_array_equal(O.rope(x, 0.0), x)


def test_rope_two_dim_hand_case():
    # d = 2: omega_0 = theta^0 = 1, so (1, 0) at position p -> (cos p, sin p)
    for p in [0.0, 1.0, 2.5, 1000.0]:
        r = O.rope(np.array([1.0, 0.0]), p)
        assert r[0] == pytest.approx(math.cos(p), abs=1e-15)
        assert r[1] == pytest.approx(math.sin(p), abs=1e-15)
    # (0, 1) -> (-sin p, cos p)
    r = O.rope(np.array([0.0, 1.0]), 0.75)
    assert r[0] == pytest.approx(-math.sin(0.75), abs=1e-15)
    assert r[1] == pytest.approx(math.cos(0.75), abs=1e-15)


def test_rope_inverse_frequencies():
    f = O.rope_inv_freq(64, 10000.0)
    assert f[0] == 1.0
    assert f[1] == pytest.approx(10000.0 ** (-2 / 64), rel=1e-15)
    assert f[-1] == pytest.approx(10000.0 ** (-62 / 64), rel=1e-15)
    # pair i of a unit vector rotates with angular speed omega_i
    x = np.zeros(64)
    x[2 * 5] = 1.0
    r = O.rope(x, 3.0)
    assert r[10] == pytest.approx(math.cos(3.0 * f[5]), abs=1e-15)
    assert r[11] == pytest.approx(math.sin(3.0 * f[5]), abs=1e-15)


def test_rope_preserves_norm():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((10, 64))
    pos = rng.integers(0, 131072, size=10)
    r = O.rope(x, pos)
    np.testing.assert_allclose(np.linalg.norm(r, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rope_relative_position_property():
    # R_m R_n^T = R_{m-n}  <=>  <R_m x, R_n y> = <R_{m-n} x, y>
    rng = np.random.default_rng(3)
    for m, n in [(5, 2), (100, 3), (8191, 0), (17, 40)]:
        Rm = O.rope_matrix(64, m)
        Rn = O.rope_matrix(64, n)
        Rmn = O.rope_matrix(64, m - n)
        np.testing.assert_allclose(Rm @ Rn.T, Rmn, atol=1e-12)
        x, y = rng.standard_normal(64), rng.standard_normal(64)
        assert O.rope(x, m) @ O.rope(y, n) == pytest.approx(O.rope(x, m - n) @ y, abs=1e-11)


# ----------------------------------------------------------------------------
# absorption identity (kexue.fm "Part 1"; iotdigitaltwinplm.com: the two
# paths are algebraically identical and make a unit test)
# ----------------------------------------------------------------------------

def test_absorbed_equals_non_absorbed():
    rng = np.random.default_rng(4)
    qn, qr, q_pos, wuk, wuv, seqs = _rand_case(rng, B=3, h=4, lens=(9, 1, 17))
    ref = O.decode_reference(qn, qr, q_pos, wuk, wuv, seqs)
    ab = O.decode_absorbed(qn, qr, q_pos, wuk, wuv, seqs)
    for k in ("out", "o_lat", "lse"):
        err = np.abs(ref[k] - ab[k]).max() / np.abs(ref[k]).max()
        assert err < 1e-12, (k, err)


def test_absorbed_equals_non_absorbed_full_dims():
    w = mi.scaled(mi.workload(3), B=2, h=4, L=130)
    inp = O.workload_inputs_f64(w)
    seqs = [O.sequence_view(w, b, int(inp["lens"][b])) for b in range(w.B)]
    args = (inp["q_nope"], inp["q_rope"], inp["q_pos"], inp["w_uk"], inp["w_uv"], seqs)
    ref = O.decode_reference(*args)
    ab = O.decode_absorbed(*args)
    for k in ("out", "o_lat", "lse"):
        assert np.abs(ref[k] - ab[k]).max() / np.abs(ref[k]).max() < 1e-12
    # the absorbed query is 576-d, the value is the 512-d latent (kexue.fm eq. mla-mqa)
    assert ab["q_cat"].shape == (2, 4, 576)
    assert ab["o_lat"].shape == (2, 4, 512)


def test_merged_weight_matrix_equals_sequential_absorption():
    # x (W_q W_k^T) c^T == (x W_q)(c W_k)^T for the content part
    rng = np.random.default_rng(5)
    d, d_k, d_c = 12, 6, 10
    x = rng.standard_normal(d)
    wq = rng.standard_normal((d, d_k))
    wk = rng.standard_normal((d_c, d_k))
    c = rng.standard_normal(d_c)
    assert x @ (wq @ wk.T) @ c == pytest.approx((x @ wq) @ (c @ wk), rel=1e-12)


# ----------------------------------------------------------------------------
# softmax attention special cases
# ----------------------------------------------------------------------------

def test_position_shift_invariance():
    rng = np.random.default_rng(6)
    qn, qr, q_pos, wuk, wuv, seqs = _rand_case(rng, B=2, h=3, lens=(11, 5))
    base = O.decode_reference(qn, qr, q_pos, wuk, wuv, seqs)
    for delta in (1, 37, 100000):
        k_pos = [np.arange(c.shape[0]) + delta for c, _ in seqs]
        sh = O.decode_reference(qn, qr, q_pos + delta, wuk, wuv, seqs, k_pos=k_pos)
        np.testing.assert_allclose(sh["out"], base["out"], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(sh["lse"], base["lse"], rtol=1e-9, atol=1e-9)


def test_single_cached_token():
    rng = np.random.default_rng(7)
    qn, qr, q_pos, wuk, wuv, seqs = _rand_case(rng, B=1, h=3, lens=(1,))
    r = O.decode_reference(qn, qr, q_pos, wuk, wuv, seqs)
    c0, kr0 = seqs[0][0][0], seqs[0][1][0]
    for s in range(3):
        np.testing.assert_allclose(r["out"][0, s], wuv[s] @ c0, rtol=1e-13)
        np.testing.assert_allclose(r["o_lat"][0, s], c0, rtol=1e-13)
        # lse of one term is the scaled score itself; both at position 0 => no rotation
        z = (qn[0, s] @ (wuk[s] @ c0) + qr[0, s] @ kr0) / math.sqrt(6 + 8)
        assert r["lse"][0, s] == pytest.approx(z, rel=1e-12)


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(8)
    qn, qr, q_pos, wuk, wuv, seqs = _rand_case(rng, B=1, h=2, lens=(6,))
    qn[:] = 0.0
    qr[:] = 0.0
    r = O.decode_reference(qn, qr, q_pos, wuk, wuv, seqs)
    c = seqs[0][0]
    for s in range(2):
        np.testing.assert_allclose(r["out"][0, s], (c @ wuv[s].T).mean(axis=0), rtol=1e-12)
        np.testing.assert_allclose(r["o_lat"][0, s], c.mean(axis=0), rtol=1e-12)
        assert r["lse"][0, s] == pytest.approx(math.log(6), rel=1e-13)


def test_dominant_token_selects_its_value():
    # d_nope > L, so the content keys have full row rank and a query can be
    # solved for that gives score 200 to one token and 0 to the others
    rng = np.random.default_rng(9)
    qn, qr, q_pos, wuk, wuv, seqs = _rand_case(rng, B=1, h=1, d_nope=12, lens=(8,))
    qr[:] = 0.0
    c = seqs[0][0]
    target = 5
    k_c = c @ wuk[0].T
    want = np.zeros(8)
    want[target] = 200.0
    qn[0, 0] = np.linalg.lstsq(k_c, want, rcond=None)[0]
    r = O.decode_reference(qn, qr, q_pos, wuk, wuv, seqs)
    np.testing.assert_allclose(r["out"][0, 0], wuv[0] @ c[target], rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(r["o_lat"][0, 0], c[target], rtol=1e-9, atol=1e-12)


def test_softmax_shift_invariance_and_lse():
    z = np.array([0.3, -1.2, 4.0, 2.2])
    p1, l1 = O.softmax_with_lse(z)
    p2, l2 = O.softmax_with_lse(z + 1000.0)
    np.testing.assert_allclose(p1, p2, rtol=1e-12)
    assert l2 - l1 == pytest.approx(1000.0, rel=1e-12)
    assert l1 == pytest.approx(math.log(sum(math.exp(v) for v in z)), rel=1e-14)


def test_merge_of_partials_equals_full_attention():
    rng = np.random.default_rng(10)
    qn, qr, q_pos, wuk, wuv, seqs = _rand_case(rng, B=1, h=3, lens=(23,))
    full = O.decode_reference(qn, qr, q_pos, wuk, wuv, seqs)
    c, kr = seqs[0]
    parts, lses = [], []
    for lo, hi in [(0, 7), (7, 7), (7, 20), (20, 23)]:     # includes an empty range
        if hi == lo:
            parts.append(np.zeros((1, 3, c.shape[1])))
            lses.append(np.full((1, 3), -np.inf))
            continue
        r = O.decode_reference(qn, qr, q_pos, wuk, wuv, [(c[lo:hi], kr[lo:hi])],
                               k_pos=[np.arange(lo, hi)])
        parts.append(r["o_lat"])
        lses.append(r["lse"])
    o, lse = O.merge_partials(parts, lses)
    np.testing.assert_allclose(o, full["o_lat"], rtol=1e-12)
    np.testing.assert_allclose(lse, full["lse"], rtol=1e-12)
    # every range empty -> lse -inf, output 0, no NaN
    o0, l0 = O.merge_partials(np.zeros((2, 1, 4)), np.full((2, 1), -np.inf))
    assert np.all(o0 == 0) and np.all(np.isneginf(l0))


# ----------------------------------------------------------------------------
# brute force with scalar loops at tiny dims
# ----------------------------------------------------------------------------

def _brute_force(qn, qr, q_pos, wuk, wuv, seqs, theta=10000.0):
    B, h, d_nope = len(qn), len(qn[0]), len(qn[0][0])
    d_r = len(qr[0][0])
    d_v, d_c = len(wuv[0]), len(wuv[0][0])
    out = [[[0.0] * d_v for _ in range(h)] for _ in range(B)]
    for b in range(B):
        c, kr = seqs[b]
        L = len(c)
        for s in range(h):
            # rotate q_r by hand, pair by pair
            qrot = [0.0] * d_r
            for i in range(d_r // 2):
                ang = q_pos[b] * theta ** (-2.0 * i / d_r)
                a, bb = qr[b][s][2 * i], qr[b][s][2 * i + 1]
                qrot[2 * i] = a * math.cos(ang) - bb * math.sin(ang)
                qrot[2 * i + 1] = a * math.sin(ang) + bb * math.cos(ang)
            scores = []
            for t in range(L):
                acc = 0.0
                for d in range(d_nope):
                    kd = 0.0
                    for cc in range(d_c):
                        kd += c[t][cc] * wuk[s][d][cc]
                    acc += qn[b][s][d] * kd
                for i in range(d_r // 2):
                    ang = t * theta ** (-2.0 * i / d_r)
                    a, bb = kr[t][2 * i], kr[t][2 * i + 1]
                    acc += qrot[2 * i] * (a * math.cos(ang) - bb * math.sin(ang))
                    acc += qrot[2 * i + 1] * (a * math.sin(ang) + bb * math.cos(ang))
                scores.append(acc / math.sqrt(d_nope + d_r))
            mx = max(scores)
            ws = [math.exp(z - mx) for z in scores]
            tot = sum(ws)
            for v in range(d_v):
                num = 0.0
                for t in range(L):
                    vt = 0.0
                    for cc in range(d_c):
                        vt += c[t][cc] * wuv[s][v][cc]
                    num += ws[t] * vt
                out[b][s][v] = num / tot
    return np.array(out)


def test_bruteforce_tiny_dims():
    rng = np.random.default_rng(11)
    for lens in [(3, 5), (1, 4), (5, 2)]:
        qn, qr, q_pos, wuk, wuv, seqs = _rand_case(rng, B=2, h=2, d_c=8, d_r=4, d_nope=4,
                                                   d_v=4, lens=lens)
        ref = O.decode_reference(qn, qr, q_pos, wuk, wuv, seqs)["out"]
        bf = _brute_force(qn.tolist(), qr.tolist(), q_pos.tolist(), wuk.tolist(), wuv.tolist(),
                          [(c.tolist(), k.tolist()) for c, k in seqs])
        np.testing.assert_allclose(ref, bf, rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------------------
# FP8 e4m3 storage
# ----------------------------------------------------------------------------

def test_e4m3_decode_table_pins():
    g = _golden("e4m3_codes.json")
    t = O.e4m3_value_table()
    for e in g["decode"]:
        assert t[e["code"]] == e["value"], e
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    finite = t[~np.isnan(t)]
    assert finite.max() == 448.0 and finite.min() == -448.0


def test_e4m3_encode_pins():
    g = _golden("e4m3_codes.json")
    for e in g["encode_round_nearest_even_saturating"]:
        assert int(O.e4m3_encode(e["value"])) == e["code"], e


def test_e4m3_round_trip_and_nearest():
    t = O.e4m3_value_table()
    codes = np.array([c for c in range(256) if not np.isnan(t[c])], dtype=np.uint8)
    np.testing.assert_array_equal(O.e4m3_encode(t[codes]), codes)
    # nearest: no finite code is strictly closer than the chosen one
    v = np.random.default_rng(12).standard_normal(2000) * 50
    enc = O.e4m3_decode(O.e4m3_encode(v))
    finite = t[~np.isnan(t)]
    best = np.min(np.abs(finite[None, :] - np.clip(v, -448, 448)[:, None]), axis=1)
    np.testing.assert_allclose(np.abs(enc - np.clip(v, -448, 448)), best, rtol=0, atol=0)


def test_fp8_block_quantisation_bounds():
    rng = np.random.default_rng(13)
    x = rng.standard_normal((64, 512)).astype(np.float32)
    codes, scale = O.fp8_quantize_block(x)
    amax = np.abs(x).max()
    assert scale == np.float32(amax / np.float32(448.0))
    # the largest magnitude maps to the largest code
    assert (codes & 0x7F).max() == 0x7E
    deq = O.fp8_dequantize(codes, scale)
    err = np.abs(deq - x.astype(np.float64))
    # normals: half an ulp of a 3-bit mantissa; subnormals: half the spacing 2^-9
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * float(scale)) * (1 + 1e-6) + 1e-6 * float(scale)
    assert np.all(err <= bound)
    z, s0 = O.fp8_quantize_block(np.zeros((4, 8), np.float32))
    assert s0 == 1.0 and np.all(z == 0)


# ----------------------------------------------------------------------------
# paged layout and the input generator
# ----------------------------------------------------------------------------

def test_paged_gather_equals_contiguous_rows():
    w = mi.scaled(mi.workload(4), B=5, h=2, L=None, L_range=(1, 300))
    lens = mi.lengths(w)
    table, nblk = mi.block_table(w, lens)
    assert sorted(table[table >= 0].tolist()) == list(range(nblk))
    pool = np.full((nblk, w.block_size, 3), np.nan)
    rows = []
    for b in range(w.B):
        r = np.random.default_rng(b).standard_normal((int(lens[b]), 3))
        rows.append(r)
        for t in range(int(lens[b])):
            pool[table[b, t // 64], t % 64] = r[t]
    for b in range(w.B):
        g = O.paged_gather(pool, table[b], int(lens[b]), w.block_size)
        np.testing.assert_array_equal(g, rows[b])
        assert not np.isnan(g).any()


def test_generator_is_deterministic_and_per_sequence():
    w = mi.scaled(mi.workload(3), B=3, h=2, L=70)
    a = mi.sequence(w, 1, 70)
    b = mi.sequence(w, 1, 70)
    np.testing.assert_array_equal(a[0], b[0])
    # a shorter request is a prefix of the same stream only per call shape; the
    # draw of sequence 1 does not depend on sequence 0
    c = mi.sequence(w, 0, 70)
    assert not np.array_equal(a[0], c[0])
    q1 = mi.queries(w)
    q2 = mi.queries(w)
    np.testing.assert_array_equal(q1[0], q2[0])


def test_bf16_rounding_matches_library():
    ml = pytest.importorskip("ml_dtypes")
    x = np.random.default_rng(14).standard_normal(100000).astype(np.float32) * 10
    x[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]      # ties
    ours = mi.f32_to_bf16_bits(x)
    lib = x.astype(ml.bfloat16).view(np.uint16)
    np.testing.assert_array_equal(ours, lib)
    np.testing.assert_array_equal(mi.bf16_bits_to_f32(ours), x.astype(ml.bfloat16).astype(np.float32))


def test_variable_lengths_within_range():
    w = mi.workload(4)
    lens = mi.lengths(w)
    assert lens.shape == (128,)
    assert lens.min() >= 1024 and lens.max() <= 32768
    table, nblk = mi.block_table(w, lens)
    assert nblk == int(((lens + 63) // 64).sum())


# ----------------------------------------------------------------------------
# the oracle's per-step helpers that the GPU tests use as checkers
# ----------------------------------------------------------------------------

def test_absorb_query_equals_scalar_loops():
    # kexue.fm "Part 1": q k^T = x (W_q W_k^T) c^T, so the absorbed latent query
    # of head s is q_nope^(s) W_UK^(s): q_abs[c] = sum_d q_nope[d] w_uk[s, d, c].
    # The RoPE part is the interleaved 2x2 rotation of each pair by q_pos * omega_i,
    # written out with math.cos / math.sin (d_nope != d_c, B != h, so a swapped
    # index or a mis-broadcast position changes the result or fails on shape)
    rng = np.random.default_rng(21)
    B, h, d_nope, d_c, d_r = 3, 2, 5, 7, 6
    qn = rng.standard_normal((B, h, d_nope))
    qr = rng.standard_normal((B, h, d_r))
    wuk = rng.standard_normal((h, d_nope, d_c))
    q_pos = np.array([0, 5, 1234])
    got = O.absorb_query(qn, qr, q_pos, wuk)
    assert got.shape == (B, h, d_c + d_r)
    theta = 10000.0
    for b in range(B):
        for s in range(h):
            for c in range(d_c):
                acc = 0.0
                for d in range(d_nope):
                    acc += qn[b, s, d] * wuk[s, d, c]
                assert abs(got[b, s, c] - acc) <= 1e-12 * (1 + abs(acc))
            for i in range(d_r // 2):
                ang = float(q_pos[b]) * theta ** (-2.0 * i / d_r)
                a, bb = qr[b, s, 2 * i], qr[b, s, 2 * i + 1]
                want0 = a * math.cos(ang) - bb * math.sin(ang)
                want1 = a * math.sin(ang) + bb * math.cos(ang)
                assert abs(got[b, s, d_c + 2 * i] - want0) <= 1e-12
                assert abs(got[b, s, d_c + 2 * i + 1] - want1) <= 1e-12


def test_absorb_query_scores_equal_per_head_keys():
    # the absorbed query dotted with raw latents equals the non-absorbed score
    # q_nope . (c W_UK^(s)T), and its RoPE part dotted with the rotated key
    # equals RoPE(q_r, t) . RoPE(k_r, i) (kexue.fm "Part 1" and "Part 2")
    rng = np.random.default_rng(22)
    B, h, d_nope, d_c, d_r, L = 2, 3, 6, 10, 4, 9
    qn = rng.standard_normal((B, h, d_nope))
    qr = rng.standard_normal((B, h, d_r))
    wuk = rng.standard_normal((h, d_nope, d_c))
    q_pos = np.array([8, 3])
    c = rng.standard_normal((L, d_c))
    kr = rng.standard_normal((L, d_r))
    q_cat = O.absorb_query(qn, qr, q_pos, wuk)
    for b in range(B):
        for s in range(h):
            k_c = c @ wuk[s].T                       # per-head content keys [L, d_nope]
            np.testing.assert_allclose(q_cat[b, s, :d_c] @ c.T, k_c @ qn[b, s],
                                       rtol=1e-12, atol=1e-12)
            rel = q_cat[b, s, d_c:] @ O.rope(kr, np.arange(L)).T
            want = [np.dot(O.rope_matrix(d_r, q_pos[b]).T @ qr[b, s],
                           O.rope_matrix(d_r, i).T @ kr[i]) for i in range(L)]
            np.testing.assert_allclose(rel, want, rtol=1e-12, atol=1e-12)


def test_output_projection_equals_per_head_values():
    # o_lat W_UV^(s)T must equal the output the non-absorbed reference forms from
    # per-head values v_i = c_i W_UV^(s)T (kexue.fm "Part 1": W_v moves to the
    # output side), and a scalar loop at tiny dims
    rng = np.random.default_rng(23)
    qn, qr, q_pos, wuk, wuv, seqs = _rand_case(rng, B=2, h=3, d_c=12, d_r=4, d_nope=5, d_v=7,
                                               lens=(6, 11))
    ref = O.decode_reference(qn, qr, q_pos, wuk, wuv, seqs)
    np.testing.assert_allclose(O.output_projection(ref["o_lat"], wuv), ref["out"],
                               rtol=1e-12, atol=1e-14)
    o = rng.standard_normal((2, 3, 12))
    got = O.output_projection(o, wuv)
    for b in range(2):
        for s in range(3):
            for v in range(7):
                acc = sum(o[b, s, c] * wuv[s, v, c] for c in range(12))
                assert abs(got[b, s, v] - acc) <= 1e-12


def test_quantized_latent_blocks_follow_the_rows():
    # L = 130 rows: blocks [0, 64), [64, 128), [128, 130), each with its own
    # magnitude, so an off-by-one block boundary changes some block's amax
    rng = np.random.default_rng(24)
    d_c = 32
    x = rng.standard_normal((130, d_c)).astype(np.float32)
    x[:64] *= np.float32(0.5)
    x[64:128] *= np.float32(3.0)
    x[128:] *= np.float32(40.0)
    x[5, 3] = np.float32(9.0)           # block 0's amax sits inside the block
    x[127, 0] = np.float32(-30.0)       # block 1's amax is its last row
    x[128, 1] = np.float32(500.0)       # block 2's amax is its first row
    codes, scales, deq = O.quantized_latent_f64(x, 64)
    assert codes.shape == x.shape and scales.shape == (3,)
    bounds = [(0, 64), (64, 128), (128, 130)]
    want_amax = [9.0, 30.0, 500.0]
    for j, (r0, r1) in enumerate(bounds):
        blk = x[r0:r1]
        assert float(np.abs(blk).max()) == want_amax[j]
        assert scales[j] == np.float32(np.float32(want_amax[j]) / np.float32(448.0))
        # every code of the block decodes to within half an e4m3 step of x / scale
        q = (blk / scales[j]).astype(np.float64)
        vals = O.e4m3_decode(codes[r0:r1])
        assert np.all(np.abs(vals - q) <= np.maximum(np.abs(q) * 2.0 ** -4, 2.0 ** -10) + 1e-12)
        np.testing.assert_array_equal(deq[r0:r1], vals * np.float64(scales[j]))
    # the block's largest magnitude maps to the largest code, 448
    assert O.e4m3_decode(codes[5, 3]) == 448.0
    assert O.e4m3_decode(codes[127, 0]) == -448.0
    assert O.e4m3_decode(codes[128, 1]) == 448.0


# ----------------------------------------------------------------------------
# FP8 append (one token into a partly filled block)
# ----------------------------------------------------------------------------

def test_fp8_append_to_empty_block_is_block_quantisation():
    x = np.random.default_rng(31).standard_normal(64).astype(np.float32)
    codes, sc = O.fp8_append_row(np.zeros((0, 64), np.uint8), np.float32(1.0), x)
    ref_codes, ref_sc = O.fp8_quantize_block(x[None, :])
    np.testing.assert_array_equal(codes, ref_codes)
    assert sc == ref_sc


def test_fp8_append_hand_examples():
    # block row [1, -2]: scale 2/448, codes 224 and -448
    blk, s = O.fp8_quantize_block(np.array([[1.0, -2.0]], np.float32))
    assert s == np.float32(2.0 / 448.0)
    np.testing.assert_array_equal(O.e4m3_decode(blk), [[224.0, -448.0]])
    # a smaller row keeps the scale and the earlier codes: 0.5 / (2/448) = 112
    b2, s2 = O.fp8_append_row(blk, s, np.array([0.5, 0.0], np.float32))
    assert s2 == s
    np.testing.assert_array_equal(b2[0], blk[0])
    np.testing.assert_array_equal(O.e4m3_decode(b2[1]), [112.0, 0.0])
    # a row with amax 4 > 448 s = 2 grows the scale to 4/448: the earlier row
    # re-quantises exactly to 112 and -224, the new one to 448 and 56
    b3, s3 = O.fp8_append_row(blk, s, np.array([4.0, 0.5], np.float32))
    assert s3 == np.float32(np.float32(4.0) / np.float32(448.0))
    np.testing.assert_array_equal(O.e4m3_decode(b3), [[112.0, -224.0], [448.0, 56.0]])
    # double rounding: row [3, 1] has codes 448 and e4m3(149.33) = 144; growing
    # to 10/448 re-quantises 144 * (3/448) / (10/448) = 43.2 to 44
    b4, s4 = O.fp8_quantize_block(np.array([[3.0, 1.0]], np.float32))
    np.testing.assert_array_equal(O.e4m3_decode(b4), [[448.0, 144.0]])
    b5, _ = O.fp8_append_row(b4, s4, np.array([10.0, 0.0], np.float32))
    # 448 * (3/448) / (10/448) = 134.4 -> 128 (e4m3 steps of 16 there)
    np.testing.assert_array_equal(O.e4m3_decode(b5[0]), [128.0, 44.0])


def test_fp8_append_scale_matches_whole_block_quantisation():
    # appending a block's rows one by one ends with the scale of quantising
    # the block at once (amax of all rows / 448), whatever the row order
    rng = np.random.default_rng(32)
    x = rng.standard_normal((64, 48)).astype(np.float32)
    x[17] *= np.float32(9.0)
    blk, sc = np.zeros((0, 48), np.uint8), np.float32(1.0)
    growths = 0
    for r in range(64):
        prev = sc
        blk, sc = O.fp8_append_row(blk, sc, x[r])
        growths += int(r > 0 and sc != prev)
    assert growths >= 1
    _, ref_sc = O.fp8_quantize_block(x)
    assert sc == ref_sc
    # rows appended after the largest one keep exactly the block quantiser's codes
    ref_codes, _ = O.fp8_quantize_block(x)
    np.testing.assert_array_equal(blk[17:], ref_codes[17:])
    # a row is rounded once when appended and once more at each later growth
    # of the scale: each rounding moves it by at most half an e4m3 step at the
    # (final, coarsest) scale
    deq = O.fp8_dequantize(blk, sc)
    n_round = growths + 1
    bound = (n_round * np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * float(sc)) * 1.1
             + 1e-6 * float(sc))
    assert np.all(np.abs(deq - x) <= bound)


def test_quantized_latent_appended_reduces_to_the_fill():
    rng = np.random.default_rng(33)
    x = rng.standard_normal((150, 16)).astype(np.float32)
    full = O.quantized_latent_f64(x, 64)
    app = O.quantized_latent_appended(x, 64, 150)
    for a, b in zip(full, app):
        np.testing.assert_array_equal(a, b)
    # filled to 100 rows, then 50 appended: blocks 0 (full) is untouched
    codes, scales, _ = O.quantized_latent_appended(x, 64, 100)
    np.testing.assert_array_equal(codes[:64], full[0][:64])
    assert scales[0] == full[1][0]
    # block 1 = rows 64..99 quantised together, then rows 100..127 appended
    blk, sc = O.fp8_quantize_block(x[64:100])
    for r in range(100, 128):
        blk, sc = O.fp8_append_row(blk, sc, x[r])
    np.testing.assert_array_equal(codes[64:128], blk)
    assert scales[1] == sc


# ----------------------------------------------------------------------------
# multi-token decode (q_len new tokens, causal among them)
# ----------------------------------------------------------------------------

def _brute_force_multi(qn, qr, wuk, wuv, seqs, theta=10000.0):
    # scalar loops with an explicit causal mask: token j of sequence b is at
    # position L - q_len + j and sees the rows at positions <= its own
    B, q_len, h, d_nope = qn.shape
    d_r = qr.shape[3]
    d_v, d_c = wuv.shape[1], wuk.shape[2]
    sc = 1.0 / math.sqrt(d_nope + d_r)
    out = np.zeros((B, q_len, h, d_v))
    for b in range(B):
        c, kr = seqs[b]
        L = len(c)
        for j in range(q_len):
            pos = L - q_len + j
            for s in range(h):
                z = []
                for i in range(L):
                    if i > pos:
                        continue
                    dot = 0.0
                    for d in range(d_nope):
                        kd = sum(c[i][cc] * wuk[s][d][cc] for cc in range(d_c))
                        dot += qn[b][j][s][d] * kd
                    for p2 in range(d_r // 2):
                        a_q = pos * theta ** (-2.0 * p2 / d_r)
                        a_k = i * theta ** (-2.0 * p2 / d_r)
                        q0, q1 = qr[b][j][s][2 * p2], qr[b][j][s][2 * p2 + 1]
                        k0, k1 = kr[i][2 * p2], kr[i][2 * p2 + 1]
                        rq = (q0 * math.cos(a_q) - q1 * math.sin(a_q), q0 * math.sin(a_q) + q1 * math.cos(a_q))
                        rk = (k0 * math.cos(a_k) - k1 * math.sin(a_k), k0 * math.sin(a_k) + k1 * math.cos(a_k))
                        dot += rq[0] * rk[0] + rq[1] * rk[1]
                    z.append((i, dot * sc))
                if not z:
                    continue
                mz = max(v for _, v in z)
                ws = [(i, math.exp(v - mz)) for i, v in z]
                tot = sum(wv for _, wv in ws)
                for v in range(d_v):
                    out[b, j, s, v] = sum(wv * sum(c[i][cc] * wuv[s][v][cc] for cc in range(d_c))
                                          for i, wv in ws) / tot
    return out


def test_multi_token_decode_bruteforce_and_mask():
    rng = np.random.default_rng(41)
    B, q_len, h, d_c, d_r, d_nope, d_v = 2, 3, 2, 6, 4, 3, 4
    qn = rng.standard_normal((B, q_len, h, d_nope))
    qr = rng.standard_normal((B, q_len, h, d_r))
    wuk = rng.standard_normal((h, d_nope, d_c)) / math.sqrt(d_c)
    wuv = rng.standard_normal((h, d_v, d_c)) / math.sqrt(d_c)
    seqs = [(rng.standard_normal((L, d_c)), rng.standard_normal((L, d_r))) for L in (5, 2)]
    ref = O.decode_reference_multi(qn, qr, wuk, wuv, seqs)
    bf = _brute_force_multi(qn, qr, wuk, wuv, seqs)
    np.testing.assert_allclose(ref["out"], bf, rtol=1e-12, atol=1e-14)
    # sequence 1 has L = 2 < q_len: its first token sees nothing
    assert np.all(ref["out"][1, 0] == 0) and np.all(np.isneginf(ref["lse"][1, 0]))
    assert np.all(np.isfinite(ref["lse"][1, 1:]))


def test_multi_token_decode_is_causal_and_reduces_to_one_token():
    rng = np.random.default_rng(42)
    qn, qr, _, wuk, wuv, seqs = _rand_case(rng, B=2, h=3, lens=(9, 7))
    # q_len = 1 is the one-token decode at the last position
    one = O.decode_reference_multi(qn[:, None], qr[:, None], wuk, wuv, seqs)
    ref = O.decode_reference(qn, qr, [8, 6], wuk, wuv, seqs)
    np.testing.assert_allclose(one["out"][:, 0], ref["out"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(one["lse"][:, 0], ref["lse"], rtol=1e-13)
    # token j never sees the rows after its own position: changing them only
    # changes the later tokens
    q4n = rng.standard_normal((2, 4, 3, qn.shape[2]))
    q4r = rng.standard_normal((2, 4, 3, qr.shape[2]))
    a = O.decode_reference_multi(q4n, q4r, wuk, wuv, seqs)
    seqs2 = [(c.copy(), k.copy()) for c, k in seqs]
    seqs2[0][0][-1] += 5.0         # the last row (position 8: token 3 only)
    seqs2[1][1][-2] -= 3.0         # position 5 of L = 7: tokens 2 and 3
    b = O.decode_reference_multi(q4n, q4r, wuk, wuv, seqs2)
    np.testing.assert_array_equal(a["out"][0, :3], b["out"][0, :3])
    assert not np.allclose(a["out"][0, 3], b["out"][0, 3])
    np.testing.assert_array_equal(a["out"][1, :2], b["out"][1, :2])
    assert not np.allclose(a["out"][1, 2:], b["out"][1, 2:])


# ----------------------------------------------------------------------------
# the hidden-state boundary: query compression and the output projection
# ----------------------------------------------------------------------------

def test_query_from_hidden_scalar_loops():
    rng = np.random.default_rng(51)
    B, d_model, d_cq, h, d_nope, d_r = 2, 7, 5, 3, 2, 4
    x = rng.standard_normal((B, d_model))
    wdq = rng.standard_normal((d_cq, d_model))
    wuq = rng.standard_normal((h * d_nope, d_cq))
    wqr = rng.standard_normal((h * d_r, d_cq))
    qn, qr = O.query_from_hidden(x, wdq, wuq, wqr, h)
    assert qn.shape == (B, h, d_nope) and qr.shape == (B, h, d_r)
    for b in range(B):
        c = [sum(x[b, i] * wdq[j, i] for i in range(d_model)) for j in range(d_cq)]
        for s in range(h):
            for d in range(d_nope):
                want = sum(c[j] * wuq[s * d_nope + d, j] for j in range(d_cq))
                assert abs(qn[b, s, d] - want) <= 1e-12
            for d in range(d_r):
                want = sum(c[j] * wqr[s * d_r + d, j] for j in range(d_cq))
                assert abs(qr[b, s, d] - want) <= 1e-12


def test_folded_output_projection_equals_the_pair():
    # associativity: (o_lat W_UV^(s)T) W_O^T == o_lat W_fold^T, and a scalar
    # loop over the fold's definition
    rng = np.random.default_rng(52)
    B, h, d_c, d_v, d_model = 3, 4, 6, 5, 7
    o_lat = rng.standard_normal((B, h, d_c))
    wuv = rng.standard_normal((h, d_v, d_c))
    wo = rng.standard_normal((d_model, h * d_v))
    fold = O.fold_uv_into_o(wuv, wo)
    y_pair = O.output_to_hidden(O.output_projection(o_lat, wuv), wo)
    y_fold = o_lat.reshape(B, -1) @ fold.T
    np.testing.assert_allclose(y_fold, y_pair, rtol=1e-12, atol=1e-12)
    for n in range(d_model):
        for s in range(h):
            for c in range(d_c):
                want = sum(wo[n, s * d_v + v] * wuv[s, v, c] for v in range(d_v))
                assert abs(fold[n, s * d_c + c] - want) <= 1e-12
    # output_to_hidden concatenates heads in order
    out = rng.standard_normal((B, h, d_v))
    y = O.output_to_hidden(out, wo)
    for b in range(B):
        for n in range(d_model):
            want = sum(out[b, s, v] * wo[n, s * d_v + v] for s in range(h) for v in range(d_v))
            assert abs(y[b, n] - want) <= 1e-12


def test_decode_from_hidden_composes_the_steps():
    rng = np.random.default_rng(53)
    B, h, d_c, d_r, d_nope, d_v, d_model, d_cq = 2, 3, 8, 4, 3, 5, 9, 6
    x = rng.standard_normal((B, d_model))
    wdq = rng.standard_normal((d_cq, d_model)) / 3
    wuq = rng.standard_normal((h * d_nope, d_cq)) / 3
    wqr = rng.standard_normal((h * d_r, d_cq)) / 3
    wuk = rng.standard_normal((h, d_nope, d_c)) / 3
    wuv = rng.standard_normal((h, d_v, d_c)) / 3
    wo = rng.standard_normal((d_model, h * d_v)) / 3
    seqs = [(rng.standard_normal((L, d_c)), rng.standard_normal((L, d_r))) for L in (6, 4)]
    y, r = O.decode_from_hidden(x, wdq, wuq, wqr, wuk, wuv, wo, [5, 3], seqs)
    qn, qr = O.query_from_hidden(x, wdq, wuq, wqr, h)
    bf = _brute_force(qn.tolist(), qr.tolist(), [5, 3], wuk.tolist(), wuv.tolist(),
                      [(c.tolist(), k.tolist()) for c, k in seqs])
    np.testing.assert_allclose(r["out"], bf, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(y, bf.reshape(B, -1) @ wo.T, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------
# prefill in the MHA form
# ----------------------------------------------------------------------------

def test_prefill_rows_equal_the_decode_of_their_prefix():
    # row t of the causal prefill is the one-token decode of token t over the
    # rows 0..t (the MHA form of the prefill and the decode form agree)
    rng = np.random.default_rng(61)
    T, h, d_c, d_r, d_nope, d_v = 9, 3, 8, 4, 5, 6
    qn = rng.standard_normal((T, h, d_nope))
    qr = rng.standard_normal((T, h, d_r))
    wuk = rng.standard_normal((h, d_nope, d_c)) / 3
    wuv = rng.standard_normal((h, d_v, d_c)) / 3
    c = rng.standard_normal((T, d_c))
    kr = rng.standard_normal((T, d_r))
    ref = O.prefill_reference(qn, qr, wuk, wuv, c, kr)
    for t in range(T):
        d = O.decode_reference(qn[t][None], qr[t][None], [t], wuk, wuv, [(c[:t + 1], kr[:t + 1])])
        np.testing.assert_allclose(ref["out"][t], d["out"][0], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(ref["lse"][t], d["lse"][0], rtol=1e-12)
    # the first row sees only itself: its output is v_0 exactly
    np.testing.assert_allclose(ref["out"][0], (c[0] @ wuv.transpose(0, 2, 1)).reshape(h, d_v),
                               rtol=1e-12, atol=1e-14)
