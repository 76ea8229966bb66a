"""Pins of the oracle's storage-format code against library routines and closed forms.

Formats: bf16 (top half of fp32), e4m3 per the OCP 8-bit floating point
specification, MXFP8 per OCP MX v1.0 (32-element groups, UE8M0 scale), which
the DeepSeek-V4.1 pages name for the checkpoint and the indexer cache
(recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview, "Mixed MXFP4/MXFP8 checkpoint";
miles.radixark.com "DeepSeek-V4.1 Flash", §1, "32-wide ue8m0 block scale").
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, 20000, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # no inf/NaN
    ref = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(O.bf16_to_f64(bits), ref)


def test_bf16_round_matches_torch_rne():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(50000) * np.exp(rng.uniform(-20, 20, 50000))).astype(np.float32)
    # exact ties: low 16 bits 0x8000 with even and odd kept parts
    u = rng.integers(0, 1 << 31, 2000, dtype=np.uint64).astype(np.uint32)
    ties = ((u & np.uint32(0x7F7F0000)) | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties, -ties, np.float32([0.0, -0.0, 1.0, 3.0e38])])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(O.f32_to_bf16_rne(x), ref)


def test_e4m3_table_exhaustive_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(O.E4M3_TABLE), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(O.E4M3_TABLE[~nan], ref[~nan])


def test_e4m3_closed_forms():
    # Largest normal, smallest normal, largest/smallest subnormal, one, minus two.
    assert O.e4m3_value(0x7E) == 448.0
    assert O.e4m3_value(0x08) == 2.0 ** -6
    assert O.e4m3_value(0x07) == 0.875 * 2.0 ** -6
    assert O.e4m3_value(0x01) == 2.0 ** -9
    assert O.e4m3_value(0x38) == 1.0
    assert O.e4m3_value(0xC0) == -2.0
    assert O.e4m3_value(0x80) == 0.0 and math.copysign(1, O.e4m3_value(0x80)) < 0


def test_e4m3_encode_vs_torch_in_range():
    vals = O.E4M3_TABLE[np.isfinite(O.E4M3_TABLE)]
    pos = np.unique(np.abs(vals))
    mids = (pos[1:] + pos[:-1]) / 2  # exact ties between neighbours
    rng = np.random.default_rng(3)
    rand = rng.uniform(-448, 448, 20000) * np.exp(rng.uniform(-12, 0, 20000))
    x = np.concatenate([vals, mids, -mids, rand]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode(x.astype(np.float64))
    # +-0 may differ only in sign for values that round to zero
    same = (got == ref) | (((got & 0x7F) == 0) & ((ref & 0x7F) == 0))
    assert same.all()


def test_e4m3_encode_saturates():
    x = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, -1e6])
    got = O.e4m3_encode(x)
    assert list(got) == [0x7E] * 6 + [0xFE]


def test_ue8m0_closed_forms():
    assert O.ue8m0_scale(np.array([127]))[0] == 1.0
    assert O.ue8m0_scale(np.array([0]))[0] == 2.0 ** -127
    assert O.ue8m0_scale(np.array([254]))[0] == 2.0 ** 127
    with pytest.raises(ValueError):
        O.ue8m0_scale(np.array([255]))


def test_mxfp8_decode_vs_torch():
    rng = np.random.default_rng(4)
    codes = rng.integers(0, 256, (64, 128), dtype=np.uint32).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x11
    scales = rng.integers(100, 150, (64, 4), dtype=np.uint32).astype(np.uint8)
    f = torch.from_numpy(codes).view(torch.float8_e4m3fn).double()
    s = torch.pow(2.0, torch.from_numpy(scales.astype(np.float64)) - 127.0)
    ref = (f.view(64, 4, 32) * s[..., None]).reshape(64, 128).numpy()
    assert np.array_equal(O.mxfp8_decode(codes, scales), ref)


def test_mxfp8_decode_rejects_nan():
    c = np.zeros((1, 32), np.uint8)
    c[0, 5] = 0x7F
    with pytest.raises(ValueError):
        O.mxfp8_decode(c, np.full((1, 1), 127, np.uint8))


def test_mxfp8_encode_scale_rule():
    # X = floor(log2(amax)) - 8: amax 1.0 -> -8; 0.75 -> -9; 2^-20 * 1.5 -> -28; 300 -> 0.
    for amax, X in [(1.0, -8), (0.75, -9), (1.5 * 2.0 ** -20, -28), (300.0, 0), (511.0, 0),
                    (512.0, 1)]:
        v = np.zeros((1, 32), np.float32)
        v[0, 7] = amax
        v[0, 3] = -amax / 3
        _, s = O.mxfp8_encode(v)
        assert int(s[0, 0]) - 127 == X, (amax, s)
    z = np.zeros((2, 64), np.float32)
    c, s = O.mxfp8_encode(z)
    assert (c == 0).all() and (s == 127).all()


def test_mxfp8_round_trip_of_representable_groups():
    rng = np.random.default_rng(5)
    fin = np.where(np.isfinite(O.E4M3_TABLE) & (np.abs(O.E4M3_TABLE) > 0))[0]
    big = np.where((np.abs(O.E4M3_TABLE) >= 256) & np.isfinite(O.E4M3_TABLE))[0]
    for X in [-20, -9, 0, 5]:
        codes = rng.choice(fin, (16, 32)).astype(np.uint8)
        codes[:, 0] = rng.choice(big, 16)  # amax in [256, 448] fixes the scale at X
        v = (O.E4M3_TABLE[codes] * 2.0 ** X).astype(np.float32)
        c2, s2 = O.mxfp8_encode(v)
        assert (s2.astype(int) - 127 == X).all()
        assert np.array_equal(O.mxfp8_decode(c2, s2), v.astype(np.float64))


def test_mxfp8_encode_error_bound_and_torch_elements():
    rng = np.random.default_rng(6)
    v = (rng.standard_normal((200, 128)) / np.sqrt(128)).astype(np.float32)
    c, s = O.mxfp8_encode(v)
    dec = O.mxfp8_decode(c, s)
    X = s.astype(np.int64) - 127
    # Element rounding of v / 2^X agrees with torch's float -> e4m3 rounding (values < 512).
    scaled = (v.reshape(200, 4, 32) * np.ldexp(1.0, -X)[..., None]).reshape(200, 128)
    sat = np.abs(scaled) > 448
    ref = torch.from_numpy(scaled.astype(np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()
    assert np.array_equal(c[~sat], ref[~sat])
    assert ((c[sat] & 0x7F) == 0x7E).all()
    # Relative error of a normal, unsaturated e4m3 element is at most 2^-4; a
    # saturated one (v / 2^X in (448, 512)) lands on 448 * 2^X.
    nz = (np.abs(scaled) >= 2.0 ** -6) & ~sat
    rel = np.abs(dec - v)[nz] / np.abs(v)[nz]
    assert rel.max() <= 2.0 ** -4 + 1e-12
    assert np.array_equal(np.abs(dec[sat]), (448.0 * np.ldexp(1.0, X))[:, :, None].repeat(
        32, -1).reshape(200, 128)[sat])


def test_pool_mean_order_golden():
    g = json.load(open(os.path.join(GOLDEN, "pool_fp32_order.json")))
    m = np.array(g["members"], np.float32)[:, None]
    assert O.pool_mean_f32(m)[0] == g["mean_in_order"]
    assert O.pool_mean_f32(m[::-1])[0] == g["mean_reversed"]


def test_pool_identical_members_give_the_member():
    rng = np.random.default_rng(7)
    k = rng.standard_normal(128).astype(np.float32)
    kb = O.bf16_to_f64(O.f32_to_bf16_rne(k))
    d, s = O.pool_keys(np.tile(kb, (8, 1)), 8, "bf16")
    assert np.array_equal(O.bf16_to_f64(d[0]), kb)
    c, sc = O.mxfp8_encode(k[None, :])
    km = O.mxfp8_decode(c, sc)[0]
    d, s = O.pool_keys(np.tile(km, (8, 1)), 8, "mxfp8")
    assert np.array_equal(d[0], c[0]) and np.array_equal(s[0], sc[0])


def test_pool_keys_brute_force_partial_blocks():
    rng = np.random.default_rng(8)
    n = 21  # blocks of 8, 8 and 5
    kv = O.bf16_to_f64(O.f32_to_bf16_rne(rng.standard_normal((n, 32)).astype(np.float32)))
    d, _ = O.pool_keys(kv, n, "fp32")
    assert d.shape == (3, 32)
    for b, c in [(0, 8), (1, 8), (2, 5)]:
        for j in range(32):
            acc = np.float32(kv[8 * b, j])
            for t in range(1, c):
                acc = np.float32(acc + np.float32(kv[8 * b + t, j]))
            assert d[b, j] == np.float32(acc / np.float32(c))
    db, _ = O.pool_keys(kv, n, "bf16")
    assert np.array_equal(db, O.f32_to_bf16_rne(d))
    dm, sm = O.pool_keys(kv, n, "mxfp8")
    c2, s2 = O.mxfp8_encode(d)
    assert np.array_equal(dm, c2) and np.array_equal(sm, s2)


# ---------------------------------------------------------------------------
# MXFP4 (OCP MX v1.0: e2m1 elements, 32-element groups, UE8M0 scale), the
# indexer-cache format the pages name (recipes.vllm.ai "DeepSeek-V4.1-Flash":
# indexer_kv_dtype mxfp4; sglang page: FP4 indexer cache). torch has no CPU
# conversion for float4_e2m1fn_x2, so the pins are the format's closed forms
# and a brute-force nearest-value search.
# ---------------------------------------------------------------------------


def test_e2m1_table_closed_forms():
    # the eight magnitudes of E2M1: subnormal 0.5, normals 1..6, then negatives
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(O.E2M1_TABLE[:8]) == mags
    assert list(O.E2M1_TABLE[8:]) == [-m for m in mags]
    assert math.copysign(1.0, O.E2M1_TABLE[8]) < 0


def _nearest_e2m1(y):
    """Brute force: the code of the representable magnitude nearest min(|y|, 6);
    on a tie the one with mantissa bit 0 (neighbouring codes differ in it)."""
    mags = O.E2M1_TABLE[:8]
    d = np.abs(mags - min(abs(y), 6.0))
    best = np.flatnonzero(d == d.min())
    c = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
    return c | (8 if np.signbit(y) else 0)


def test_e2m1_encode_vs_brute_force():
    rng = np.random.default_rng(40)
    mags = O.E2M1_TABLE[:8]
    mids = (mags[1:] + mags[:-1]) / 2  # exact ties: 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5
    ys = np.concatenate([mags, mids, mids + 1e-9, mids - 1e-9, rng.uniform(0, 8, 3000),
                         [6.5, 7.0, 7.5, 8.0, 100.0, 1e30]])
    ys = np.concatenate([ys, -ys])
    want = np.array([_nearest_e2m1(y) for y in ys], np.uint8)
    assert np.array_equal(O.e2m1_encode(ys), want)
    # the ties named: each goes to the even mantissa
    assert list(O.E2M1_TABLE[O.e2m1_encode(mids)]) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_mxfp4_pack_order_and_round_trip():
    codes = (np.arange(64) % 16).astype(np.uint8).reshape(2, 32)
    p = O.mxfp4_pack(codes)
    assert p.shape == (2, 16)
    assert p[0, 0] == codes[0, 0] | (codes[0, 1] << 4) and p[1, 15] == codes[1, 30] | (
        codes[1, 31] << 4)
    assert np.array_equal(O.mxfp4_unpack(p), codes)


def test_mxfp4_encode_scale_rule():
    # X = floor(log2(amax)) - 2: amax 1.0 -> -2; 0.75 -> -3; 6 -> 0; 7.9 -> 0; 8 -> 1;
    # 1.5 * 2^-30 -> -32
    for amax, X in [(1.0, -2), (0.75, -3), (6.0, 0), (7.9, 0), (8.0, 1),
                    (1.5 * 2.0 ** -30, -32)]:
        v = np.zeros((1, 32), np.float32)
        v[0, 11] = amax
        v[0, 2] = -amax / 3
        _, s = O.mxfp4_encode(v)
        assert int(s[0, 0]) - 127 == X, (amax, s)
    d, s = O.mxfp4_encode(np.zeros((2, 64), np.float32))
    assert (d == 0).all() and (s == 127).all()


def test_mxfp4_round_trip_of_representable_groups():
    rng = np.random.default_rng(41)
    for X in (-20, -3, 0, 7):
        codes = rng.integers(0, 16, (16, 32)).astype(np.uint8)
        codes[:, 0] = rng.choice([6, 7, 14, 15], 16)  # |amax| in {4, 6}: scale stays X
        v = O.E2M1_TABLE[codes] * 2.0 ** X
        d, s = O.mxfp4_encode(v.astype(np.float32))
        assert (s.astype(int) - 127 == X).all()
        assert np.array_equal(O.mxfp4_decode(d, s), v)
        assert np.array_equal(d, O.mxfp4_pack(codes))  # the same codes, -0 included


def test_mxfp4_encode_error_bound():
    rng = np.random.default_rng(42)
    v = (rng.standard_normal((200, 128)) / np.sqrt(128)).astype(np.float32)
    d, s = O.mxfp4_encode(v)
    dec = O.mxfp4_decode(d, s)
    X = np.repeat(s.astype(np.int64) - 127, 32, axis=-1)
    scaled = np.abs(v.astype(np.float64)) * np.ldexp(1.0, -X)
    assert scaled.max() < 8.0  # the group's largest element lands in [4, 8)
    # half the local spacing of the grid (0.25 below 2, 0.5 below 4, 1 up to 6),
    # and saturation above 6: |error| <= 2^X * max(0.25, |v / 2^X| / 4)
    bound = np.ldexp(1.0, X) * np.maximum(0.25, scaled / 4)
    assert (np.abs(dec - v) <= bound + 1e-300).all()
    # no sign flips: a decoded value is zero or has the input's sign
    assert ((dec == 0) | (np.sign(dec) == np.sign(v))).all()


def test_pool_keys_in_mxfp4():
    rng = np.random.default_rng(43)
    k = rng.standard_normal((1, 128)).astype(np.float32)
    d, s = O.mxfp4_encode(k)
    km = O.mxfp4_decode(d, s)[0]
    # identical members pool to the member's own codes and scales
    pd, ps = O.pool_keys(np.tile(km, (8, 1)), 8, "mxfp4")
    assert np.array_equal(pd[0], d[0]) and np.array_equal(ps[0], s[0])
    # otherwise the pooled key is the fp32 mean, then the MXFP4 conversion
    kv = O.bf16_to_f64(O.f32_to_bf16_rne(rng.standard_normal((21, 64)).astype(np.float32)))
    mean, _ = O.pool_keys(kv, 21, "fp32")
    dm, sm = O.pool_keys(kv, 21, "mxfp4")
    c2, s2 = O.mxfp4_encode(mean)
    assert np.array_equal(dm, c2) and np.array_equal(sm, s2)
    assert np.array_equal(O.decode_keys("mxfp4", dm, sm), O.mxfp4_decode(c2, s2))
