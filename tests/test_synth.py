"""The seeded input generator: determinism, distributions and layout."""
import numpy as np

import oracle as O
import synth


def test_deterministic_and_counter_based():
    a = synth.normal_bf16(3, 1, 0, 1000, 1.0)
    b = synth.normal_bf16(3, 1, 0, 1000, 1.0)
    assert np.array_equal(a, b)
    # element i depends only on its counter: a window of the stream matches
    c = synth.normal_bf16(3, 1, 333, 100, 1.0)
    assert np.array_equal(a[333:433], c)
    assert not np.array_equal(a, synth.normal_bf16(4, 1, 0, 1000, 1.0))
    assert not np.array_equal(a, synth.normal_bf16(3, 2, 0, 1000, 1.0))


def test_distributions():
    z = synth.normal_f32(0, 9, 0, 400000, 1.0).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    assert abs((np.abs(z) < 1).mean() - 0.6827) < 0.005
    u = synth.uniform_f32(0, 9, 0, 200000).astype(np.float64)
    assert u.min() >= 0 and u.max() < 1 and abs(u.mean() - 0.5) < 0.005
    assert np.array_equal(u * 2 ** 24, np.floor(u * 2 ** 24))


def test_mxfp8_generator_is_close_to_its_normals():
    codes, scales = synth.normal_mxfp8(1, 5, 0, 300, 128, 1 / np.sqrt(128))
    ref = synth.normal_f32(1, 5, 0, 300 * 128, 1 / np.sqrt(128)).reshape(300, 128)
    dec = O.mxfp8_decode(codes, scales)
    big = np.abs(ref) > 1e-3
    assert (np.abs(dec - ref)[big] / np.abs(ref)[big]).max() < 0.13
    # the generator's encoding is the OCP MX conversion
    c2, s2 = O.mxfp8_encode(ref)
    assert np.array_equal(codes, c2) and np.array_equal(scales, s2)


def test_decode_inputs_layout():
    inp = synth.decode_inputs([100, 37], 2, "mxfp8", seed=3)
    assert inp.q.shape == (2, 64, 512) and inp.q_idx.shape == (2, 16, 128)
    assert list(inp.n_latents) == [50, 18] and list(inp.swa_len) == [100, 37]
    assert inp.cap == 56 and inp.keys.scales.shape == (2, 56, 4)
    assert (inp.latents[1, 18:] == 0x7F80).all()      # poisoned tail
    assert (inp.swa[1, 37:] == 0).all()
    lat = O.bf16_to_f64(inp.latents[0, :50])
    assert abs(lat.std() * np.sqrt(512) - 1) < 0.02


def test_mxfp4_generator_is_the_ocp_conversion_of_its_normals():
    packed, scales = synth.normal_mxfp4(1, 5, 0, 300, 128, 1 / np.sqrt(128))
    assert packed.shape == (300, 64) and scales.shape == (300, 4)
    ref = synth.normal_f32(1, 5, 0, 300 * 128, 1 / np.sqrt(128)).reshape(300, 128)
    # two independent statements of the OCP MX conversion: the generator's C and
    # the oracle's numpy
    c2, s2 = O.mxfp4_encode(ref)
    assert np.array_equal(packed, c2) and np.array_equal(scales, s2)
    # the same values as the MXFP8 generator, so the two formats share one scale
    # grid: X(fp4) = X(fp8) + 6
    _, s8 = synth.normal_mxfp8(1, 5, 0, 300, 128, 1 / np.sqrt(128))
    assert np.array_equal(scales.astype(int), s8.astype(int) + 6)


def test_decode_inputs_with_mxfp4_keys():
    inp = synth.decode_inputs([100, 37], 2, "mxfp4", seed=3)
    assert inp.keys.data.shape == (2, 56, 64) and inp.keys.scales.shape == (2, 56, 4)
    assert (inp.keys.data[1, 18:] == 0x77).all() and (inp.keys.scales[1, 18:] == 254).all()
    k = O.decode_keys("mxfp4", inp.keys.data[0, :50], inp.keys.scales[0, :50])
    assert abs(k.std() * np.sqrt(128) - 1) < 0.1
    pf = synth.prefill_inputs(20, 100, 2, "mxfp4", seed=4)
    assert pf.keys.data.shape == (64, 64) and pf.keys.fmt == "mxfp4"


def test_fp8_cache_codes_match_the_oracle_encoder():
    """synth's fp8 cache rows (its own C conversion) are the oracle's E4M3
    encoding of the same fp32 normals divided by the cache scale."""
    v = synth.normal_f32(5, 3, 100, 200000, 1 / np.sqrt(512))
    for kv_scale in (2.0 ** -6, 2.0 ** -3, 1.0):
        c = synth.normal_e4m3(5, 3, 100, 200000, 1 / np.sqrt(512), kv_scale)
        assert np.array_equal(c, O.e4m3_encode(v.astype(np.float64) / kv_scale))
    inp = synth.decode_inputs([300, 20], 1, "mxfp8", seed=6, kv_fmt="fp8")
    assert inp.latents.dtype == np.uint8 and inp.swa.dtype == np.uint8
    assert (inp.latents[1, 20:] == 0x7E).all()  # the poisoned tail: 448
