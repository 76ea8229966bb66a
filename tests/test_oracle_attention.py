"""Pins of the oracle's attention stage and of the whole decode/prefill step.

Attention: all 64 query heads attend to one 512-wide latent per position used
as both key and value (miles.radixark.com "DeepSeek-V4.1 Flash", §1
"Architecture"), over the selected latents and the 128-position window
(recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview, "Two-tier sparse attention"),
under one softmax.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth


def sdpa(q, kv, tau):
    qt = torch.from_numpy(q)[None, None]          # [1, 1, H, D]
    kt = torch.from_numpy(kv)[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, kt, scale=tau)
    return o[0, 0].numpy()


def test_attend_matches_torch_sdpa():
    rng = np.random.default_rng(20)
    q, kv = rng.standard_normal((64, 512)), rng.standard_normal((640, 512))
    for tau in (1 / np.sqrt(512), 1.0, 0.05):
        o, lse = O.attend(q, kv, tau)
        assert np.allclose(o, sdpa(q, kv, tau), rtol=1e-10, atol=1e-12)
        z = tau * q @ kv.T
        assert np.allclose(lse, np.log(np.exp(z - z.max(1, keepdims=True)).sum(1))
                           + z.max(1), rtol=1e-12)


def test_attend_special_cases():
    rng = np.random.default_rng(21)
    q, kv = rng.standard_normal((4, 32)), rng.standard_normal((9, 32))
    # tau = 0: the plain mean of the rows, lse = log(rows)
    o, lse = O.attend(q, kv, 0.0)
    assert np.allclose(o, np.tile(kv.mean(0), (4, 1)))
    assert np.allclose(lse, np.log(9.0))
    # one row: that row
    o, _ = O.attend(q, kv[:1], 0.3)
    assert np.allclose(o, np.tile(kv[0], (4, 1)))
    # a large tau and one key planted along q: that key
    kv2 = rng.standard_normal((50, 32)) * 0.01
    kv2[17] = q[2] / np.linalg.norm(q[2])
    o, _ = O.attend(q[2:3], kv2, 1e4)
    assert np.allclose(o[0], kv2[17], atol=1e-9)
    # probabilities: non-negative rows summing to 1
    p = O.attention_probs(q, kv, 0.7)
    assert (p >= 0).all() and np.abs(p.sum(1) - 1).max() < 1e-12
    # row order does not matter
    perm = rng.permutation(9)
    assert np.allclose(O.attend(q, kv, 0.7)[0], O.attend(q, kv[perm], 0.7)[0], rtol=1e-13)


def _cfg(**kw):
    return O.StepConfig(**kw)


def test_decode_all_selected_equals_dense_attention():
    # k_tokens >= L: every latent is selected, so the step is dense attention
    # over all latents followed by the window, under one softmax.
    inp = synth.decode_inputs([600], 2, "bf16", seed=7)      # L = 300 latents
    cfg = _cfg(ratio=2, k_tokens=512)
    r = O.decode_sequence(cfg, inp, 0)
    assert list(r["token_ids"][:300]) == list(range(300))
    kv = np.concatenate([O.bf16_to_f64(inp.latents[0, :300]),
                         O.bf16_to_f64(inp.swa[0, :128])])
    q = O.bf16_to_f64(inp.q[0])
    assert np.allclose(r["out"], sdpa(q, kv, 1 / np.sqrt(512)), rtol=1e-10, atol=1e-13)


def test_decode_short_sequence_window_and_latents():
    # T = 5 at ratio 2: 2 latents (positions 0-3), window holds positions 0..4.
    inp = synth.decode_inputs([5], 2, "bf16", seed=8)
    assert inp.n_latents[0] == 2 and inp.swa_len[0] == 5
    r = O.decode_sequence(_cfg(ratio=2), inp, 0)
    assert list(r["token_ids"][:2]) == [0, 1] and (r["token_ids"][2:] == -1).all()
    kv = np.concatenate([O.bf16_to_f64(inp.latents[0, :2]), O.bf16_to_f64(inp.swa[0, :5])])
    assert np.allclose(r["out"], sdpa(O.bf16_to_f64(inp.q[0]), kv, 1 / np.sqrt(512)),
                       rtol=1e-10, atol=1e-13)


def test_decode_one_token_ratio_two_has_no_latent():
    inp = synth.decode_inputs([1], 2, "bf16", seed=9)
    r = O.decode_sequence(_cfg(ratio=2), inp, 0)
    assert (r["token_ids"] == -1).all()
    # one window row: the output is that row
    assert np.allclose(r["out"], np.tile(O.bf16_to_f64(inp.swa[0, 0]), (64, 1)))


def test_prefill_window_rows_closed_form():
    # row r of the prefill window buffer holds position ctx - 127 + r
    assert O.prefill_window_rows(1000, 0, 128) == (0, 128)
    assert O.prefill_window_rows(1000, 5, 128) == (5, 133)
    assert O.prefill_window_rows(10, 0, 128) == (117, 128)      # positions 0..10
    assert O.prefill_visible(1000, 0, 2) == 500 and O.prefill_visible(1000, 1, 2) == 501
    assert O.prefill_visible(1001, 0, 2) == 501


@pytest.mark.parametrize("fmt,ratio", [("bf16", 2), ("mxfp8", 1), ("bf16", 1)])
def test_prefill_last_query_equals_decode(fmt, ratio):
    ctx, n_q = 333, 20
    cfg = _cfg(ratio=ratio, k_blocks=6, k_tokens=40)
    pf = synth.prefill_inputs(n_q, ctx, ratio, fmt, seed=11)
    kv, pooled, _ = O.prefill_caches(cfg, pf)
    T = ctx + n_q
    L = T // ratio
    # the same sequence as a decode batch of one
    dec = synth.decode_inputs([T], ratio, fmt, seed=11)
    dec.q[0], dec.q_idx[0], dec.w[0] = pf.q[-1], pf.q_idx[-1], pf.w[-1]
    dec.latents[0, :L] = pf.latents[:L]
    dec.keys.data[0, :L] = pf.keys.data[:L]
    if fmt == "mxfp8":
        dec.keys.scales[0, :L] = pf.keys.scales[:L]
    lo, hi = O.prefill_window_rows(ctx, n_q - 1, 128)
    dec.swa[0, : hi - lo] = pf.swa[lo:hi]
    rp = O.prefill_query(cfg, pf, n_q - 1, kv, pooled)
    rd = O.decode_sequence(cfg, dec, 0)
    assert np.array_equal(rp["block_ids"], rd["block_ids"])
    assert np.array_equal(rp["token_ids"], rd["token_ids"])
    assert np.array_equal(rp["out"], rd["out"])


@pytest.mark.parametrize("fmt,ratio", [("bf16", 2), ("mxfp8", 1)])
def test_every_prefill_query_equals_decode_of_its_prefix(fmt, ratio):
    """Query i of a chunk sits at position ctx + i: it must see exactly what a
    one-query decode of the sequence's first ctx + i + 1 tokens sees (visible
    latents, the partly visible last block, the window ending at itself).
    The chunk crosses block boundaries and keeps the block stage active."""
    ctx, n_q = 150, 12
    cfg = _cfg(ratio=ratio, k_blocks=6, k_tokens=24)
    pf = synth.prefill_inputs(n_q, ctx, ratio, fmt, seed=13)
    kv, pooled, _ = O.prefill_caches(cfg, pf)
    seen_partial = set()
    for i in range(n_q):
        T = ctx + i + 1
        L = T // ratio
        dec = synth.decode_inputs([T], ratio, fmt, seed=14)
        dec.q[0], dec.q_idx[0], dec.w[0] = pf.q[i], pf.q_idx[i], pf.w[i]
        dec.latents[0, :L] = pf.latents[:L]
        dec.keys.data[0, :L] = pf.keys.data[:L]
        if fmt == "mxfp8":
            dec.keys.scales[0, :L] = pf.keys.scales[:L]
        lo, hi = O.prefill_window_rows(ctx, i, 128)
        assert hi - lo == int(dec.swa_len[0]) == min(128, T)
        dec.swa[0, : hi - lo] = pf.swa[lo:hi]
        rp = O.prefill_query(cfg, pf, i, kv, pooled)
        rd = O.decode_sequence(cfg, dec, 0)
        assert int(dec.n_latents[0]) == O.prefill_visible(ctx, i, ratio) == L
        assert np.array_equal(rp["block_ids"], rd["block_ids"]), i
        assert np.array_equal(rp["token_ids"], rd["token_ids"]), i
        assert np.array_equal(rp["out"], rd["out"]) and np.array_equal(rp["lse"], rd["lse"]), i
        seen_partial.add(L % 8 != 0)
    assert seen_partial == {True, False}  # both a complete and a partial last block occur


def test_prefill_partial_block_is_mean_of_visible_members():
    ctx, n_q, ratio = 100, 12, 1
    cfg = _cfg(ratio=ratio, k_blocks=3, k_tokens=16)
    pf = synth.prefill_inputs(n_q, ctx, ratio, "bf16", seed=12)
    kv, pooled, _ = O.prefill_caches(cfg, pf)
    for i in range(n_q):
        n_vis = O.prefill_visible(ctx, i, ratio)
        # recompute this query's block keys independently by decoding its own pool
        pd, _ = O.pool_keys(kv[:n_vis], n_vis, "bf16")
        r = O.select_query(cfg, pf.q_idx[i], pf.w[i], kv, O.bf16_to_f64(pd), n_vis)
        rp = O.prefill_query(cfg, pf, i, kv, pooled, with_attention=False)
        assert np.array_equal(r["block_ids"], rp["block_ids"])
        assert np.array_equal(r["token_ids"], rp["token_ids"])
        assert (rp["token_ids"][rp["token_ids"] >= 0] < n_vis).all()


def test_fp8_cache_rows_are_e4m3_values_times_one_scale():
    """An fp8 cache row stands for E4M3(code) x kv_scale. Every E4M3 value is
    exactly a bf16 value (3 mantissa bits of 7), so attending over fp8 rows
    must equal attending over the bf16 bit patterns of the same values, scaled
    once: a wrong code table, a scale applied twice or to the query, or window
    rows left unscaled all break it. The scale is a power of two here, so the
    bf16 patterns of the scaled values are exact too."""
    rng = np.random.default_rng(81)
    codes = rng.integers(0, 256, (300, 512), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C                # no NaN codes
    win = rng.integers(0, 256, (40, 512), dtype=np.uint8)
    win[(win & 0x7F) == 0x7F] = 0x41
    q = synth.normal_bf16(81, 1, 0, 64 * 512, 1 / np.sqrt(512)).reshape(64, 512)
    ids = np.array([5, 17, 299, -1, 0, 100], np.int64)
    cfg = O.StepConfig(k_blocks=16, k_tokens=6)
    for scale in (1.0, 2.0 ** -6, 8.0):
        o8, l8 = O.attend_query(cfg, q, codes, ids, win, "fp8", scale)
        vals = O.E4M3_TABLE[codes] * scale
        wvals = O.E4M3_TABLE[win] * scale
        bits = O.f32_to_bf16_rne(vals.astype(np.float32))
        wbits = O.f32_to_bf16_rne(wvals.astype(np.float32))
        assert np.array_equal(O.bf16_to_f64(bits), vals)  # exact in bf16
        ob, lb = O.attend_query(cfg, q, bits, ids, wbits)
        assert np.array_equal(o8, ob) and np.array_equal(l8, lb)
    # a decode step over an fp8 cache attends over those values
    inp = synth.decode_inputs([900, 33], 1, "bf16", seed=82, kv_fmt="fp8")
    r = O.decode_sequence(O.StepConfig(k_blocks=16, k_tokens=64), inp, 0)
    ids = r["token_ids_used"]
    kv = np.concatenate([O.E4M3_TABLE[inp.latents[0][ids[ids >= 0]]],
                         O.E4M3_TABLE[inp.swa[0][:int(inp.swa_len[0])]]]) * inp.kv_scale
    o, lse = O.attend(O.bf16_to_f64(inp.q[0]), kv, O.StepConfig().tau)
    assert np.array_equal(r["out"], o) and np.array_equal(r["lse"], lse)
