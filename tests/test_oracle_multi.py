"""Pins of the multi-query decode reading: sequence b's n_q queries are the
prefill chunk of n_q queries after T_b - n_q tokens (synth.multi_as_prefill),
and the last of them is the plain decode query of that sequence (position
T_b - 1, window of the last 128 positions), computed by the oracle's decode
path on a batch built independently from the same bytes."""
import dataclasses

import numpy as np
import pytest

import oracle as O
import synth


@pytest.mark.parametrize("T,n_q,ratio,fmt", [([700, 131], 5, 2, "bf16"),
                                             ([333, 9], 3, 1, "mxfp8"),
                                             ([260], 16, 1, "mxfp4")])
def test_last_query_of_a_sequence_is_its_decode_query(T, n_q, ratio, fmt):
    m = synth.multi_inputs(T, n_q, ratio, fmt, seed=4, q_scale=4.0)
    cfg = O.StepConfig(k_blocks=8, k_tokens=40, ratio=ratio, sm_scale=2.0)
    # the same sequences as a decode batch (same caches), each query taken as
    # the last query of its sequence, with the last min(T, 128) window rows
    dec = synth.decode_inputs(T, ratio, fmt, seed=4)
    swa = np.zeros_like(dec.swa)
    swl = np.minimum(m.T, m.window).astype(np.int32)
    for b in range(m.B):
        swa[b, :swl[b]] = m.swa[b, m.swa.shape[1] - swl[b]:]
    dec = dataclasses.replace(dec, q=m.q[:, -1].copy(), q_idx=m.q_idx[:, -1].copy(),
                              w=m.w[:, -1].copy(), swa=swa, swa_len=swl)
    for b in range(m.B):
        view = synth.multi_as_prefill(m, b)
        kv, pooled, _ = O.prefill_caches(cfg, view)
        last = O.prefill_query(cfg, view, n_q - 1, kv, pooled)
        assert np.array_equal(dec.keys.data[b, :int(m.n_latents[b])],
                              m.keys.data[b, :int(m.n_latents[b])])
        r = O.decode_sequence(cfg, dec, b)
        assert np.array_equal(r["token_ids"], last["token_ids"])
        assert np.allclose(r["out"], last["out"], rtol=0, atol=1e-12)
        assert np.allclose(r["lse"], last["lse"], rtol=0, atol=1e-12)


def test_queries_see_their_own_causal_prefix():
    """Query i sees floor((T - n_q + i + 1) / ratio) latents and positions up to
    T - n_q + i in its window: an earlier query's selection never contains a
    later latent."""
    m = synth.multi_inputs([403], 6, 2, "bf16", seed=5)
    cfg = O.StepConfig(k_blocks=100, k_tokens=512, ratio=2)
    view = synth.multi_as_prefill(m, 0)
    kv, pooled, _ = O.prefill_caches(cfg, view)
    for i in range(6):
        r = O.prefill_query(cfg, view, i, kv, pooled, with_attention=False)
        n_vis = (403 - 6 + i + 1) // 2
        ids = r["token_ids"][r["token_ids"] >= 0]
        assert len(ids) == min(512, n_vis) and ids.max() == n_vis - 1
