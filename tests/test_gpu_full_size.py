"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (dsa_decode_step with the pool tail update, dsa_sparse_attn_prefill).

The oracle recomputes sampled sequences (decode) or sampled queries (prefill)
one by one; every sequence or query is also checked for properties that hold at
any size: ids strictly ascending, within the visible range, -1 padding only at
the end, a finite output and a clean device status.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import synth
import two_tier_sparse_gb300 as dsa
from parity import DecodeOnDevice, check_ids, check_out, host_u16
from test_gpu_parity import block_near_tie, check_step, oracle_cfg, run_prefill, run_step

pytestmark = pytest.mark.gpu


def check_all_sequences(inp, cfg, outs):
    """Size-independent properties for every sequence of a decode batch."""
    out, lse, bids, tok = (x.cpu().numpy() for x in outs)
    for b in range(inp.B):
        n_vis = int(inp.n_latents[b])
        nb = (n_vis + 7) // 8
        for ids, hi, k, label in ((bids[b], nb, cfg.k_blocks, "blocks"),
                                  (tok[b], n_vis, cfg.k_tokens, "tokens")):
            v = ids[ids >= 0]
            assert len(v) == min(k, hi if label == "blocks" else min(n_vis, 8 * min(nb, cfg.k_blocks))), \
                f"{label} {b}: {len(v)} ids"
            assert (np.diff(v) > 0).all() and v.min() >= 0 and v.max() < hi, f"{label} {b}"
            assert (ids[len(v):] == -1).all(), f"{label} {b}: padding"
        assert np.isfinite(lse[b]).all(), f"lse {b}"
    assert np.isfinite(O.bf16_to_f64(out.view(np.uint16))).all()


@pytest.mark.parametrize("workload,sample", [
    ("decode_b1_t4096_r2_bf16", [0]),
    ("decode_b64_t131072_r1_mxfp8", [0, 9, 18, 27, 37, 45, 54, 63]),
    ("decode_b8_t1048576_r1_mxfp8", [0, 3, 5, 7]),
    ("decode_b64_t131072_r1_mxfp4", [0, 21, 42, 63]),
    ("decode_b64_t131072_r1_mxfp8_fp8kv", [0, 31, 63]),
])
def test_decode_workload_full_size(workload, sample):
    spec = synth.WORKLOADS[workload]
    inp = synth.workload_inputs(workload)
    fp8 = spec.get("kv_fmt", "bf16") == "fp8"
    cfg = dsa.config(ratio=spec["ratio"], kv_fmt=dsa.KV_FP8_E4M3 if fp8 else dsa.KV_BF16,
                     kv_scale=inp.kv_scale)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    outs = run_step(d, cfg, update_pool=True)
    code, info = d.status()
    assert code == 0, hex(info)
    check_all_sequences(inp, cfg, outs)
    check_step(inp, cfg, outs, sample)


def test_prefill_workload_full_size():
    """4096 causal queries after a 65536-token context at ratio 2 (bf16 keys)."""
    spec = synth.WORKLOADS["prefill_q4096_ctx65536_r2_bf16"]
    pf = synth.prefill_inputs(spec["n_q"], spec["ctx"], spec["ratio"], spec["key_fmt"],
                              spec["seed"])
    cfg = dsa.config(ratio=spec["ratio"])
    out, lse, tok = run_prefill(pf, cfg)
    n_q = pf.n_q
    # every query: ids ascending within its visible latents, output finite
    for i in range(n_q):
        n_vis = O.prefill_visible(pf.ctx, i, pf.ratio)
        v = tok[i][tok[i] >= 0]
        assert len(v) == min(cfg.k_tokens, n_vis), f"q{i}: {len(v)} ids"
        assert (np.diff(v) > 0).all() and v.min() >= 0 and v.max() < n_vis, f"q{i}"
    assert np.isfinite(lse).all()
    assert np.isfinite(O.bf16_to_f64(out)).all()
    # sampled queries against the oracle
    oc = oracle_cfg(cfg)
    kv, pooled, _ = O.prefill_caches(oc, pf)
    # queries whose last block is complete (0, 2047, 4095) and partly visible
    # (1, 3, 13, 1000, 2999, 4093: 1, 2, 7, 4, 4 and 7 of its 8 members)
    for i in (0, 1, 3, 13, 1000, 2047, 2999, 4093, 4095):
        r = O.prefill_query(oc, pf, i, kv, pooled, with_attention=False)
        pos = {int(t): s for t, s in zip(r["cand"], r["token_scores"])}
        if not block_near_tie(r["block_scores"], cfg.k_blocks):
            check_ids(tok[i], r["token_ids"], lambda j: pos[j], cfg.k_tokens, f"q{i}")
        r2 = O.prefill_query(oc, pf, i, kv, pooled, token_ids=tok[i])
        check_out(out[i], lse[i], r2["out"], r2["lse"], f"q{i}")
