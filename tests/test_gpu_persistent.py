"""GPU parity of the unsplit attention over more queries than SMs: persistent
CTAs run several queries each through one pipeline (index lists, Q and ring
tiles of the next query loading while the current one finishes), with queries
that have no rows at all between others."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
import two_tier_sparse_gb300 as dsa
from parity import DecodeOnDevice, check_out, dev, host_u16
from test_gpu_parity import oracle_cfg, run_prefill

pytestmark = pytest.mark.gpu


def test_unsplit_decode_attention_with_empty_queries():
    """400 sequences (2-3 per CTA), ratio 2: every seventh has one token (no
    latent) and no window row, so it has no rows; the others are ragged, some
    with fewer selected ids than k. Every query is checked."""
    rng = np.random.default_rng(91)
    B = 400
    T = [int(t) for t in rng.integers(2, 1400, size=B)]
    for b in range(0, B, 7):
        T[b] = 1
    inp = synth.decode_inputs(T, 2, "bf16", seed=92, q_scale=8.0)
    for b in range(0, B, 7):
        inp.swa_len[b] = 0
    cfg = dsa.config(ratio=2, sm_scale=1.0)
    d = DecodeOnDevice(inp, cfg)
    ids = np.full((B, cfg.k_tokens), -1, np.int32)
    for b in range(B):
        n = int(inp.n_latents[b])
        take = min(n, int(rng.integers(1, cfg.k_tokens + 1)))
        if take > 0:
            ids[b, :take] = np.sort(rng.choice(n, take, replace=False))
    out = torch.empty((B, 64, 512), dtype=torch.int16, device="cuda")
    lse = torch.empty((B, 64), dtype=torch.float32, device="cuda")
    dsa.sparse_attn_decode(cfg, d.q, d.latents, d.n_lat, dev(ids), d.swa, d.swa_len, out, d.ws,
                           lse=lse)
    code, info = d.status()
    assert code == 0, hex(info)
    got, got_lse = host_u16(out), lse.cpu().numpy()
    oc = oracle_cfg(cfg)
    for b in range(B):
        sw = int(inp.swa_len[b])
        if (ids[b] < 0).all() and sw == 0:
            assert (got[b] == 0).all() and np.isneginf(got_lse[b]).all(), f"seq {b}"
            continue
        o, l = O.attend_query(oc, inp.q[b], inp.latents[b], ids[b], inp.swa[b][:sw])
        check_out(got[b], got_lse[b], o, l, f"seq {b}")


def test_unsplit_prefill_chunk_many_queries():
    """A 400-query chunk after 5 tokens at ratio 1: the first queries see one or
    two latents and a short window, the rest grow; 2-3 queries a CTA."""
    pf = synth.prefill_inputs(400, 5, 1, "bf16", seed=93, q_scale=8.0)
    cfg = dsa.config(k_blocks=12, k_tokens=40, ratio=1, sm_scale=1.0)
    out, lse, tok = run_prefill(pf, cfg)
    oc = oracle_cfg(cfg)
    kv, pooled, _ = O.prefill_caches(oc, pf)
    for i in range(pf.n_q):
        r = O.prefill_query(oc, pf, i, kv, pooled, token_ids=tok[i])
        check_out(out[i], lse[i], r["out"], r["lse"], f"q{i}")


def test_unsplit_decode_step_is_deterministic_across_replays():
    """The persistent kernel's result does not depend on which CTA ran a query
    after which: two runs of a 300-sequence step give the same bits."""
    T = [int(t) for t in np.random.default_rng(94).integers(600, 3000, size=300)]
    inp = synth.decode_inputs(T, 1, "mxfp8", seed=95)
    cfg = dsa.config(ratio=1)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    outs = []
    for _ in range(2):
        out = torch.empty((inp.B, 64, 512), dtype=torch.int16, device="cuda")
        dsa.decode_step(cfg, d.q, d.q_idx, d.w, d.keys, d.pooled, d.latents, d.n_lat, d.cap,
                        d.swa, d.swa_len, out, d.ws)
        outs.append(host_u16(out))
    assert d.status()[0] == 0
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "bf16"])
def test_scan_query_switches_in_every_cta(fmt):
    """600 short sequences (1-2 tiles of each stage per query): every scan CTA's
    tile range spans several queries, so each math set keeps building the next
    query's index vectors while the previous query's tiles are still in
    flight. Both tiers run (k_blocks 16, k_tokens 40); every sequence is
    checked against the oracle."""
    from test_gpu_parity import check_step, run_step
    rng = np.random.default_rng(96)
    T = [int(t) for t in rng.integers(100, 1200, size=600)]
    inp = synth.decode_inputs(T, 1, fmt, seed=97, q_scale=8.0)
    cfg = dsa.config(k_blocks=16, k_tokens=40, ratio=1, sm_scale=1.0)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    outs = run_step(d, cfg)
    code, info = d.status()
    assert code == 0, hex(info)
    check_step(inp, cfg, outs, range(inp.B))
