"""Multi-query decode on the GPU (dsa_decode_multi): every query of every
sequence against the oracle's prefill-chunk reading of it, over both tiers,
all key formats, ratios 1 and 2, 1 to 16 queries a sequence, ragged and
short sequences."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
import two_tier_sparse_gb300 as dsa
from parity import check_ids, check_out, dev, host_u16, pooled_buffer
from test_gpu_parity import block_near_tie, oracle_cfg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    from two_tier_sparse_gb300 import build
    build.build()
    dsa.load()
    torch.cuda.set_device(cuda_device)


def run_multi(m, cfg):
    B, n_q, cap = m.B, m.n_q, m.cap
    fmt = m.keys.fmt
    keys = dsa.Keys(fmt, dev(m.keys.data), None if m.keys.scales is None else dev(m.keys.scales))
    n_lat = dev(m.n_latents)
    pooled = pooled_buffer(fmt, B, cap // 8)
    ws = dsa.workspace(cfg, B * n_q, cap)
    dsa.pool_index_keys(cfg, keys, n_lat, cap, pooled, ws)
    out = torch.empty((B, n_q, 64, 512), dtype=torch.int16, device="cuda")
    lse = torch.empty((B, n_q, 64), dtype=torch.float32, device="cuda")
    tok = torch.empty((B, n_q, cfg.k_tokens), dtype=torch.int32, device="cuda")
    dsa.decode_multi(cfg, dev(m.T.astype(np.int32)), dev(m.q), dev(m.q_idx), dev(m.w), keys,
                     pooled, dev(m.latents), cap, dev(m.swa), out, ws, lse=lse, token_ids=tok)
    status = dsa.read_device_status(ws)
    return host_u16(out), lse.cpu().numpy(), tok.cpu().numpy(), status


def check_multi(m, cfg, out, lse, tok, seqs, skip=()):
    oc = oracle_cfg(cfg)
    for b in seqs:
        view = synth.multi_as_prefill(m, b)
        kv, pooled, _ = O.prefill_caches(oc, view)
        for i in range(m.n_q):
            if (b, i) in skip:
                continue
            r = O.prefill_query(oc, view, i, kv, pooled, with_attention=False)
            pos = {int(t): s for t, s in zip(r["cand"], r["token_scores"])}
            if not block_near_tie(r["block_scores"], cfg.k_blocks):
                check_ids(tok[b, i], r["token_ids"], lambda j: pos[j], cfg.k_tokens, f"{b}/{i}")
            r2 = O.prefill_query(oc, view, i, kv, pooled, token_ids=tok[b, i])
            check_out(out[b, i], lse[b, i], r2["out"], r2["lse"], f"{b}/{i}")


@pytest.mark.parametrize("fmt,ratio,n_q,T,k_blocks", [
    ("bf16", 2, 5, [4096, 999, 130, 5], 64),      # both tiers; T = n_q
    ("mxfp8", 1, 5, [20000, 3001, 64, 7], 128),
    ("mxfp4", 1, 3, [9000, 700, 9], 96),
    ("mxfp8", 1, 16, [5000, 300], 256),
    ("bf16", 1, 1, [3000, 100], 64),              # one query: the decode position
    ("mxfp8", 2, 5, [70000, 40001], 2048),        # 4375 blocks: the block stage at full k
])
def test_multi_query_decode(fmt, ratio, n_q, T, k_blocks):
    m = synth.multi_inputs(T, n_q, ratio, fmt, seed=80, q_scale=8.0)
    cfg = dsa.config(k_blocks=k_blocks, ratio=ratio, sm_scale=8.0)
    out, lse, tok, (code, info) = run_multi(m, cfg)
    assert code == 0, hex(info)
    check_multi(m, cfg, out, lse, tok, range(m.B))


def test_multi_query_sequence_shorter_than_its_queries():
    """A sequence of 3 tokens with 5 queries: its first two queries have no
    position (reported as a device check, no rows); the rest are checked."""
    m = synth.multi_inputs([900, 3], 5, 1, "bf16", seed=81, q_scale=8.0)
    cfg = dsa.config(k_blocks=32, sm_scale=8.0)
    out, lse, tok, (code, info) = run_multi(m, cfg)
    assert code == 6 and (info >> 24) == 4, hex(info)
    assert np.isneginf(lse[1, :2]).all() and (out[1, :2] == 0).all()
    m_ok = synth.multi_inputs([900, 3], 5, 1, "bf16", seed=81, q_scale=8.0)
    check_multi(m_ok, cfg, out, lse, tok, [0])
