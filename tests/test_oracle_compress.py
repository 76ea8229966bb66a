"""Pins of the oracle's compressed-latent rule (compress_latent): one position
is its own latent, equal gate logits give the group mean, a dominant logit
gives its position's vector, shifting every logit by a constant changes
nothing, and two positions weigh as the logistic function of their logit
difference (closed forms, not the oracle's formula retyped)."""
import math

import numpy as np

import oracle as O


def bf16(x):
    return O.f32_to_bf16_rne(np.asarray(x, np.float32))


def test_ratio_one_is_the_identity():
    rng = np.random.default_rng(1)
    kv = bf16(rng.normal(size=(1, 512)))
    for g in (-3.0, 0.0, 7.5):
        assert np.array_equal(O.compress_latent(kv, [g]), kv[0])


def test_equal_logits_give_the_mean():
    rng = np.random.default_rng(2)
    for r in (2, 4):
        kv = bf16(rng.normal(size=(r, 512)))
        want = bf16((O.bf16_to_f64(kv).sum(axis=0) / r).astype(np.float32))
        assert np.array_equal(O.compress_latent(kv, [0.75] * r), want)


def test_a_dominant_logit_selects_its_position():
    rng = np.random.default_rng(3)
    kv = bf16(rng.normal(size=(2, 512)))
    assert np.array_equal(O.compress_latent(kv, [80.0, 0.0]), kv[0])
    assert np.array_equal(O.compress_latent(kv, [0.0, 80.0]), kv[1])


def test_shift_invariance_and_the_logistic_weight():
    rng = np.random.default_rng(4)
    kv = bf16(rng.normal(size=(2, 64)))
    a = O.compress_latent(kv, [0.3, -1.2])
    assert np.array_equal(a, O.compress_latent(kv, [10.3, 8.8]))
    p = 1.0 / (1.0 + math.exp(-1.5))            # weight of position 0
    want = p * O.bf16_to_f64(kv[0]) + (1 - p) * O.bf16_to_f64(kv[1])
    got = O.bf16_to_f64(a)
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-30)
