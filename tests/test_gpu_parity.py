"""GPU parity: every call of the C ABI against the CPU oracle on the same seeded inputs.

Sizes span several 128-row tiles with ragged tails, partial blocks, sequences
shorter than the window, empty selections, and the maximum k_blocks/k_tokens.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
import two_tier_sparse_gb300 as dsa
from parity import (DecodeOnDevice, check_ids, check_out, check_scores, dev, host_u16,
                    pooled_buffer)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    from two_tier_sparse_gb300 import build
    build.build()
    dsa.load()
    torch.cuda.set_device(cuda_device)


def oracle_cfg(cfg):
    return O.StepConfig(k_blocks=cfg.k_blocks, k_tokens=cfg.k_tokens, window=cfg.window,
                        ratio=cfg.ratio, sm_scale=cfg.sm_scale if cfg.sm_scale > 0 else None)


# ---------------------------------------------------------------------------
# S0: pooled keys, bit-exact
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "mxfp4"])
def test_pool_bit_exact(fmt):
    inp = synth.decode_inputs([1003, 77, 8, 1, 2051], 1, fmt, seed=21)
    cfg = dsa.config(ratio=1)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    assert d.status()[0] == 0
    pdat = d.pooled.data.cpu().numpy()
    psc = None if d.pooled.scales is None else d.pooled.scales.cpu().numpy()
    for b in range(inp.B):
        n = int(inp.n_latents[b])
        kv = O.decode_keys(fmt, inp.keys.data[b][:n],
                           None if inp.keys.scales is None else inp.keys.scales[b][:n])
        want, want_s = O.pool_keys(kv, n, fmt)
        nb = want.shape[0]
        got = pdat[b, :nb].view(np.uint16) if fmt == "bf16" else pdat[b, :nb]
        assert np.array_equal(got, want), f"seq {b}"
        if fmt != "bf16":
            assert np.array_equal(psc[b, :nb], want_s), f"seq {b} scales"


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_pool_tail_only_writes_the_last_block(fmt):
    inp = synth.decode_inputs([1003, 64], 1, fmt, seed=22)
    d = DecodeOnDevice(inp, dsa.config())
    d.pooled.data.fill_(0x55)
    d.pool(tail_only=True)
    got = d.pooled.data.cpu().numpy()
    for b, n in enumerate(inp.n_latents):
        last = (int(n) - 1) // 8
        kv = O.decode_keys(fmt, inp.keys.data[b][:n], inp.keys.scales[b][:n])
        want, _ = O.pool_keys(kv, int(n), fmt)
        assert np.array_equal(got[b, last], want[last])
        assert (got[b, :last] == 0x55).all()


# ---------------------------------------------------------------------------
# S1 + S2: candidate-block stage
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("fmt,k_blocks", [("bf16", 64), ("mxfp8", 64), ("mxfp8", 4096),
                                          ("bf16", 1), ("mxfp4", 64), ("mxfp4", 4096)])
def test_index_blocks(fmt, k_blocks):
    T = [5000, 3001, 700, 9]
    inp = synth.decode_inputs(T, 1, fmt, seed=23)
    cfg = dsa.config(k_blocks=k_blocks, ratio=1)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    nbc = d.cap // 8
    bids = torch.empty((inp.B, k_blocks), dtype=torch.int32, device="cuda")
    bsc = torch.empty((inp.B, nbc), dtype=torch.float32, device="cuda")
    dsa.index_blocks(cfg, d.q_idx, d.w, d.pooled, d.n_lat, d.cap, bids, d.ws, block_scores=bsc)
    assert d.status()[0] == 0
    bids, bsc = bids.cpu().numpy(), bsc.cpu().numpy()
    oc = oracle_cfg(cfg)
    for b in range(inp.B):
        r = O.decode_sequence(oc, inp, b, with_attention=False)
        nb = len(r["block_scores"])
        check_scores(bsc[b, :nb], r["block_scores"], f"block scores {b}")
        assert np.isneginf(bsc[b, nb:]).all()
        check_ids(bids[b], r["block_ids"], lambda i: r["block_scores"][i], k_blocks, f"blocks {b}")


# ---------------------------------------------------------------------------
# S3 + S4: token stage (over the GPU's block set, and over every block)
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("fmt,ratio", [("bf16", 2), ("mxfp8", 1), ("mxfp4", 1), ("mxfp4", 2)])
def test_topk_over_gpu_blocks(fmt, ratio):
    T = [12000, 4099, 2000]
    inp = synth.decode_inputs(T, ratio, fmt, seed=24)
    cfg = dsa.config(k_blocks=96, k_tokens=512, ratio=ratio)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    bids = torch.empty((inp.B, 96), dtype=torch.int32, device="cuda")
    dsa.index_blocks(cfg, d.q_idx, d.w, d.pooled, d.n_lat, d.cap, bids, d.ws)
    tok = torch.empty((inp.B, 512), dtype=torch.int32, device="cuda")
    tsc = torch.empty((inp.B, 96 * 8), dtype=torch.float32, device="cuda")
    dsa.topk(cfg, d.q_idx, d.w, d.keys, bids, d.n_lat, d.cap, tok, d.ws, token_scores=tsc)
    assert d.status()[0] == 0
    bids_h, tok_h, tsc_h = bids.cpu().numpy(), tok.cpu().numpy(), tsc.cpu().numpy()
    oc = oracle_cfg(cfg)
    for b in range(inp.B):
        r = O.decode_sequence(oc, inp, b, with_attention=False, block_ids=bids_h[b])
        # candidate i is latent 8 * bids[i // 8] + i % 8
        ref = np.full(96 * 8, -np.inf)
        pos = {int(t): s for t, s in zip(r["cand"], r["token_scores"])}
        for i in range(96 * 8):
            blk = bids_h[b, i // 8]
            t = blk * 8 + i % 8
            if blk >= 0 and t in pos:
                ref[i] = pos[t]
        check_scores(tsc_h[b], ref, f"token scores {b}")
        check_ids(tok_h[b], r["token_ids"], lambda i: pos[i], 512, f"tokens {b}")


@pytest.mark.parametrize("fmt,T", [("bf16", [4096, 1000, 513, 30]),
                                   ("mxfp8", [4096, 1000, 513, 30]),
                                   ("mxfp4", [4096, 1000, 513, 31]),
                                   ("bf16", [90000, 70001, 3])])  # > 32768 latents: two passes
def test_topk_all_blocks(fmt, T):
    inp = synth.decode_inputs(T, 2, fmt, seed=25)
    cfg = dsa.config(k_tokens=512, ratio=2)
    d = DecodeOnDevice(inp, cfg)
    tok = torch.empty((inp.B, 512), dtype=torch.int32, device="cuda")
    dsa.topk(cfg, d.q_idx, d.w, d.keys, None, d.n_lat, d.cap, tok, d.ws)
    assert d.status()[0] == 0
    tok_h = tok.cpu().numpy()
    oc = oracle_cfg(cfg)
    for b in range(inp.B):
        # without block ids every visible latent is a candidate: the oracle's
        # token stage over all blocks
        nb = (int(inp.n_latents[b]) + 7) // 8
        r = O.decode_sequence(oc, inp, b, with_attention=False, block_ids=np.arange(nb))
        pos = {int(t): s for t, s in zip(r["cand"], r["token_scores"])}
        check_ids(tok_h[b], r["token_ids"], lambda i: pos[i], 512, f"tokens {b}")


# ---------------------------------------------------------------------------
# S5 - S7: attention given ids
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("T,ratio,q_scale,sm_scale", [
    ([4096, 1000, 300, 100, 5], 2, 1.0, 0.0),     # default scale (near-uniform softmax)
    ([4096, 1000, 300, 100, 5], 2, 8.0, 1.0),     # sharpened: logit std about 0.35
    ([4096, 1000, 300, 100, 5], 2, 8.0, 8.0),     # sharper: logit std about 2.8
    ([70000, 1], 1, 8.0, 1.0),                    # 512 selected of many; a 1-token sequence
    ([2], 2, 1.0, 0.0),                           # one latent, two window rows
])
def test_attention_given_oracle_ids(T, ratio, q_scale, sm_scale):
    inp = synth.decode_inputs(T, ratio, "bf16", seed=26, q_scale=q_scale)
    cfg = dsa.config(ratio=ratio, sm_scale=sm_scale)
    oc = oracle_cfg(cfg)
    d = DecodeOnDevice(inp, cfg)
    refs = [O.decode_sequence(oc, inp, b) for b in range(inp.B)]
    ids = np.stack([r["token_ids"] for r in refs]).astype(np.int32)
    out = torch.empty((inp.B, 64, 512), dtype=torch.int16, device="cuda")
    lse = torch.empty((inp.B, 64), dtype=torch.float32, device="cuda")
    dsa.sparse_attn_decode(cfg, d.q, d.latents, d.n_lat, dev(ids), d.swa, d.swa_len, out, d.ws,
                           lse=lse)
    assert d.status()[0] == 0
    out_h, lse_h = host_u16(out), lse.cpu().numpy()
    for b, r in enumerate(refs):
        check_out(out_h[b], lse_h[b], r["out"], r["lse"], f"seq {b}")


def test_attention_no_rows_and_bad_ids():
    # T = 1 at ratio 2: no latent; with swa_len forced to 0 the query has no rows.
    inp = synth.decode_inputs([1, 300], 2, "bf16", seed=27)
    inp.swa_len[0] = 0
    cfg = dsa.config(ratio=2)
    d = DecodeOnDevice(inp, cfg)
    ids = np.full((2, 512), -1, np.int32)
    ids[1, :3] = [0, 5, 149]
    out = torch.empty((2, 64, 512), dtype=torch.int16, device="cuda")
    lse = torch.empty((2, 64), dtype=torch.float32, device="cuda")
    dsa.sparse_attn_decode(cfg, d.q, d.latents, d.n_lat, dev(ids), d.swa, d.swa_len, out, d.ws,
                           lse=lse)
    assert d.status()[0] == 0
    assert (out[0] == 0).all() and torch.isneginf(lse[0]).all()
    r = O.decode_sequence(O.StepConfig(ratio=2), inp, 1, token_ids=ids[1])
    check_out(host_u16(out)[1], lse.cpu().numpy()[1], r["out"], r["lse"])
    # an id past the sequence's latents is flagged and skipped
    ids[1, 3] = 150
    dsa.sparse_attn_decode(cfg, d.q, d.latents, d.n_lat, dev(ids), d.swa, d.swa_len, out, d.ws,
                           lse=lse)
    code, info = d.status()
    assert code == 6 and (info >> 24) == 4 and (info & 0xFFFFFF) == 150
    check_out(host_u16(out)[1], lse.cpu().numpy()[1], r["out"], r["lse"])
    assert d.status()[0] == 0  # reading clears it


# ---------------------------------------------------------------------------
# The whole decode step
# ---------------------------------------------------------------------------


def run_step(d, cfg, update_pool=False):
    inp = d.inp
    B = inp.B
    out = torch.empty((B, 64, 512), dtype=torch.int16, device="cuda")
    lse = torch.empty((B, 64), dtype=torch.float32, device="cuda")
    bids = torch.empty((B, cfg.k_blocks), dtype=torch.int32, device="cuda")
    tok = torch.empty((B, cfg.k_tokens), dtype=torch.int32, device="cuda")
    dsa.decode_step(cfg, d.q, d.q_idx, d.w, d.keys, d.pooled, d.latents, d.n_lat, d.cap, d.swa,
                    d.swa_len, out, d.ws, lse=lse, block_ids=bids, token_ids=tok,
                    update_pool=update_pool)
    return out, lse, bids, tok


def check_step(inp, cfg, outs, seqs):
    out, lse, bids, tok = (x.cpu().numpy() for x in outs)
    out = out.view(np.uint16)
    oc = oracle_cfg(cfg)
    for b in seqs:
        r = O.decode_sequence(oc, inp, b, with_attention=False)
        check_ids(bids[b], r["block_ids"], lambda i: r["block_scores"][i], cfg.k_blocks,
                  f"blocks {b}")
        r2 = O.decode_sequence(oc, inp, b, block_ids=bids[b], token_ids=tok[b])
        pos = {int(t): s for t, s in zip(r2["cand"], r2["token_scores"])}
        check_ids(tok[b], r2["token_ids"], lambda i: pos[i], cfg.k_tokens, f"tokens {b}")
        check_out(out[b], lse[b], r2["out"], r2["lse"], f"out {b}")


@pytest.mark.parametrize("T,ratio,fmt,k_blocks,q_scale,sm", [
    ([4096], 2, "bf16", 2048, 1.0, 0.0),                       # decode, 4096 tokens, batch 1
    ([20000, 9001, 777, 64, 3], 1, "mxfp8", 128, 8.0, 1.0),     # both tiers, ragged, sharpened
    ([20000, 9001, 777], 2, "bf16", 200, 1.0, 0.0),
    ([20000, 9001, 777, 64, 3], 1, "mxfp4", 128, 8.0, 8.0),     # MXFP4 keys, sharpened
    ([30001, 5003], 2, "mxfp4", 300, 1.0, 0.0),
])
def test_decode_step(T, ratio, fmt, k_blocks, q_scale, sm):
    inp = synth.decode_inputs(T, ratio, fmt, seed=28, q_scale=q_scale)
    cfg = dsa.config(k_blocks=k_blocks, ratio=ratio, sm_scale=sm)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    outs = run_step(d, cfg)
    assert d.status()[0] == 0
    check_step(inp, cfg, outs, range(inp.B))


@pytest.mark.parametrize("fmt,k_blocks", [("mxfp8", 256), ("bf16", 256), ("mxfp8", 4096),
                                          ("mxfp4", 256)])
def test_decode_step_is_deterministic_and_updates_the_pool(fmt, k_blocks):
    """The step's pooling of each sequence's newest block restores it bit for
    bit (codes and MXFP8 scales), with a block stage (k_blocks 256) and
    without one (k_blocks 4096)."""
    inp = synth.decode_inputs([30000, 17], 1, fmt, seed=29)
    cfg = dsa.config(k_blocks=k_blocks)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    ref_pool = d.pooled.data.clone()
    ref_scales = None if d.pooled.scales is None else d.pooled.scales.clone()
    # clobber each sequence's newest block, then let the step rebuild it
    for b, n in enumerate(inp.n_latents):
        d.pooled.data[b, (int(n) - 1) // 8] = 0
        if d.pooled.scales is not None:
            d.pooled.scales[b, (int(n) - 1) // 8] = 0
    a = run_step(d, cfg, update_pool=True)
    assert torch.equal(d.pooled.data, ref_pool)
    if ref_scales is not None:
        assert torch.equal(d.pooled.scales, ref_scales)
    b_ = run_step(d, cfg, update_pool=True)
    for x, y in zip(a, b_):
        assert torch.equal(x, y)
    assert d.status()[0] == 0


@pytest.mark.parametrize("fmt,B,t_max,k_blocks", [
    ("mxfp8", 40, 40000, 256),   # 40 tiles a sequence: a CTA holds at most one last block
    ("mxfp4", 300, 1000, 16),    # one tile a sequence: some CTAs hold two last blocks
    ("bf16", 300, 1000, 16),
])
def test_decode_step_tail_update_many_sequences(fmt, B, t_max, k_blocks):
    """The step's tail update over many sequences, right before a block scan
    whose CTAs each cover one or several sequences' last blocks. Every
    sequence's newest block key is clobbered; after the step the block keys
    equal those the pooling kernel writes for the whole cache, bit for bit,
    for ragged lengths (multiples of 8, a single token, the longest), and the
    step's outputs agree with the oracle on a sample."""
    rng = np.random.default_rng(3000 + B)
    T = [int(t) for t in rng.integers(1, t_max, B)]
    T[0], T[1], T[2] = t_max, 8 * (t_max // 16), 1
    inp = synth.decode_inputs(T, 1, fmt, seed=70 + B)
    cfg = dsa.config(k_blocks=k_blocks, k_tokens=64)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    ref_pool = d.pooled.data.clone()
    ref_scales = None if d.pooled.scales is None else d.pooled.scales.clone()
    for b, n in enumerate(inp.n_latents):
        d.pooled.data[b, (int(n) - 1) // 8] = 0
        if d.pooled.scales is not None:
            d.pooled.scales[b, (int(n) - 1) // 8] = 0
    outs = run_step(d, cfg, update_pool=True)
    assert d.status()[0] == 0
    assert torch.equal(d.pooled.data, ref_pool)
    if ref_scales is not None:
        assert torch.equal(d.pooled.scales, ref_scales)
    check_step(inp, cfg, outs, [0, 1, 2, B // 2, B - 1])


@pytest.mark.parametrize("fmt,k_blocks", [("mxfp8", 256), ("bf16", 2048)])
def test_decode_step_replays_from_a_cuda_graph(fmt, k_blocks):
    """The whole step captured once in a CUDA graph, programmatic launch edges
    included, replays to the same bits as direct launches. A replay after new
    queries are copied into the same buffers follows them, and it agrees with
    the oracle."""
    import dataclasses
    inp = synth.decode_inputs([30000, 9001, 17], 1, fmt, seed=33)
    cfg = dsa.config(k_blocks=k_blocks)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    B = inp.B
    outs = (torch.empty((B, 64, 512), dtype=torch.int16, device="cuda"),
            torch.empty((B, 64), dtype=torch.float32, device="cuda"),
            torch.empty((B, cfg.k_blocks), dtype=torch.int32, device="cuda"),
            torch.empty((B, cfg.k_tokens), dtype=torch.int32, device="cuda"))

    def step():
        dsa.decode_step(cfg, d.q, d.q_idx, d.w, d.keys, d.pooled, d.latents, d.n_lat, d.cap,
                        d.swa, d.swa_len, outs[0], d.ws, lse=outs[1], block_ids=outs[2],
                        token_ids=outs[3], update_pool=True)

    step()  # first use sets the kernels' shared-memory attributes, outside the capture
    torch.cuda.synchronize()
    direct = [x.clone() for x in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for x in outs:
        x.fill_(-1)
    g.replay()
    torch.cuda.synchronize()
    assert d.status()[0] == 0
    for x, y in zip(outs, direct):
        assert torch.equal(x, y)
    # new queries in the same buffers: the replay reads them
    inp2 = synth.decode_inputs([30000, 9001, 17], 1, fmt, seed=34)
    d.q.copy_(dev(inp2.q))
    d.q_idx.copy_(dev(inp2.q_idx))
    d.w.copy_(dev(inp2.w))
    g.replay()
    torch.cuda.synchronize()
    replayed = [x.clone() for x in outs]
    assert not torch.equal(replayed[0], direct[0])
    step()
    torch.cuda.synchronize()
    for x, y in zip(outs, replayed):
        assert torch.equal(x, y)
    assert d.status()[0] == 0
    check_step(dataclasses.replace(inp, q=inp2.q, q_idx=inp2.q_idx, w=inp2.w), cfg, replayed,
               [0, 2])


@pytest.mark.parametrize("q_scale,sm", [(1.0, 0.0), (8.0, 8.0)])
def test_decode_32_sequences_of_32768_tokens(q_scale, sm):
    """Decode, batch 32, 32768 tokens at ratio 2 (16384 latents, 2048 blocks, all
    kept), at the default softmax scale and sharpened (q x 8, tau = 8: logit std
    about 2.8, so each split's running maximum differs)."""
    inp = synth.workload_inputs("decode_b32_t32768_r2_bf16", q_scale=q_scale)
    cfg = dsa.config(ratio=2, sm_scale=sm)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    outs = run_step(d, cfg)
    assert d.status()[0] == 0
    check_step(inp, cfg, outs, range(inp.B))


def plant_dominant_row(inp, b, s, strength):
    """Make window row s of sequence b line up with head 0 of its query (row =
    strength x the query row's direction, rounded to bf16), so that one row,
    held by one CTA of a split, dominates that head's softmax."""
    qh = O.bf16_to_f64(inp.q[b, 0])
    v = qh / np.sqrt((qh ** 2).sum()) * strength
    inp.swa[b, s] = O.f32_to_bf16_rne(v.astype(np.float32))


@pytest.mark.parametrize("B", [19, 20, 32, 38, 39, 64, 76, 77, 128])
def test_decode_step_split_paths_sharpened(B):
    """The attention splits a query's rows over an S-CTA cluster while S x B
    fits the SMs (152 on a GB300: S = 8 up to 19 queries, 4 up to 38, 2 up to
    76) and runs one CTA a query beyond. With a sharpened softmax (q x 8,
    tau = 8: logit std about 2.8) the CTAs of a cluster see different running
    maxima, so a wrong max or sum rescale in the on-chip merge shows; in every
    fourth sequence one window row is made to dominate head 0. Both selection
    tiers run (k_blocks 96 of up to 500 blocks) on ragged sequences; every
    sequence is checked against the oracle."""
    rng = np.random.default_rng(1000 + B)
    T = [int(t) for t in rng.integers(900, 4000, B)]
    T[0], T[-1] = 4000, 70          # the longest, and one shorter than the window
    fmt = "mxfp8" if B % 2 else "bf16"
    inp = synth.decode_inputs(T, 1, fmt, seed=50 + B, q_scale=8.0)
    for b in range(0, B, 4):
        plant_dominant_row(inp, b, int(rng.integers(0, inp.swa_len[b])), 0.6)
    cfg = dsa.config(k_blocks=96, ratio=1, sm_scale=8.0)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    outs = run_step(d, cfg)
    assert d.status()[0] == 0
    check_step(inp, cfg, outs, range(B))


@pytest.mark.parametrize("B,fmt", [(5, "mxfp8"), (30, "bf16"), (64, "mxfp4"), (100, "mxfp8")])
def test_decode_step_fp8_kv_cache(B, fmt):
    """An fp8 KV cache (latents and window rows as E4M3 codes times one
    scale): the attention converts the rows to f16 as they land and takes Q to
    f16 with a power-of-two scale per head. Split over 8, 4 and 2 CTAs a query
    (B = 5, 30, 64) and, with fp8, over 2 in two waves at B = 100; sharpened
    (q x 8, tau = 8) so the CTAs' running maxima differ, one window row made to
    dominate head 0 in every fourth sequence, ragged lengths and a sequence
    shorter than the window. Every sequence against the oracle."""
    rng = np.random.default_rng(4000 + B)
    T = [int(t) for t in rng.integers(900, 4000, B)]
    T[0], T[-1] = 4000, 70
    inp = synth.decode_inputs(T, 1, fmt, seed=90 + B, q_scale=8.0, kv_fmt="fp8",
                              kv_scale=2.0 ** -6)
    for b in range(0, B, 4):
        s_ = int(rng.integers(0, inp.swa_len[b]))
        qh = O.bf16_to_f64(inp.q[b, 0])
        v = qh / np.sqrt((qh ** 2).sum()) * 0.6 / inp.kv_scale
        inp.swa[b, s_] = O.e4m3_encode(v)
    cfg = dsa.config(k_blocks=96, ratio=1, sm_scale=8.0, kv_fmt=dsa.KV_FP8_E4M3,
                     kv_scale=inp.kv_scale)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    outs = run_step(d, cfg)
    assert d.status()[0] == 0
    check_step(inp, cfg, outs, range(B))


# ---------------------------------------------------------------------------
# Prefill
# ---------------------------------------------------------------------------


def block_near_tie(scores, k):
    """True when the block tier's k-th and (k+1)-th best oracle scores are a near-tie."""
    if len(scores) <= k:
        return False
    srt = np.sort(scores)[::-1]
    return abs(srt[k - 1] - srt[k]) <= 1e-5 * abs(srt[k - 1])


def run_prefill(pf, cfg):
    n_q = pf.n_q
    fmt = pf.keys.fmt
    n_lat = (pf.ctx + n_q) // pf.ratio
    keys = dsa.Keys(fmt, dev(pf.keys.data), None if pf.keys.scales is None else dev(pf.keys.scales))
    # pooled keys of complete blocks, built on the GPU (the pool call over one sequence)
    nbf = n_lat // 8
    pooled = pooled_buffer(fmt, 1, max(nbf, 1))
    ws = dsa.workspace(cfg, n_q, n_lat)
    keys1 = dsa.Keys(fmt, keys.data[None], None if keys.scales is None else keys.scales[None])
    n1 = torch.tensor([nbf * 8], dtype=torch.int32, device="cuda")
    dsa.pool_index_keys(cfg, keys1, n1, nbf * 8, pooled, ws)
    pooled2 = dsa.Keys(fmt, pooled.data[0], None if pooled.scales is None else pooled.scales[0])
    out = torch.empty((n_q, 64, 512), dtype=torch.int16, device="cuda")
    lse = torch.empty((n_q, 64), dtype=torch.float32, device="cuda")
    tok = torch.empty((n_q, cfg.k_tokens), dtype=torch.int32, device="cuda")
    dsa.sparse_attn_prefill(cfg, pf.ctx, dev(pf.q), dev(pf.q_idx), dev(pf.w), dev(pf.latents),
                            keys, pooled2, dev(pf.swa), out, ws, lse=lse, token_ids=tok)
    code, info = dsa.read_device_status(ws)
    assert code == 0, hex(info)
    return host_u16(out), lse.cpu().numpy(), tok.cpu().numpy()


@pytest.mark.parametrize("fmt,ratio,ctx,n_q", [("bf16", 2, 333, 50), ("mxfp8", 1, 1000, 37),
                                               ("bf16", 1, 5, 130), ("mxfp4", 2, 333, 50),
                                               ("mxfp4", 1, 1001, 37)])
def test_prefill(fmt, ratio, ctx, n_q):
    pf = synth.prefill_inputs(n_q, ctx, ratio, fmt, seed=30, q_scale=8.0)
    cfg = dsa.config(k_blocks=12, k_tokens=40, ratio=ratio, sm_scale=1.0)
    out, lse, tok = run_prefill(pf, cfg)
    oc = oracle_cfg(cfg)
    kv, pooled, _ = O.prefill_caches(oc, pf)
    for i in range(n_q):
        r = O.prefill_query(oc, pf, i, kv, pooled, with_attention=False)
        pos = {int(t): s for t, s in zip(r["cand"], r["token_scores"])}
        if not block_near_tie(r["block_scores"], cfg.k_blocks):
            check_ids(tok[i], r["token_ids"], lambda j: pos[j], cfg.k_tokens, f"q{i}")
        r2 = O.prefill_query(oc, pf, i, kv, pooled, token_ids=tok[i])
        check_out(out[i], lse[i], r2["out"], r2["lse"], f"q{i}")


@pytest.mark.parametrize("fmt", ["bf16", "mxfp8", "mxfp4"])
def test_scan_many_short_queries(fmt):
    """One or two tiles per query, so the scan pipeline switches query on
    almost every tile (the per-query operand slots are rebuilt constantly)."""
    rng = np.random.default_rng(41)
    T = [int(t) for t in rng.integers(1, 300, 200)]
    inp = synth.decode_inputs(T, 1, fmt, seed=41)
    cfg = dsa.config(k_blocks=4, k_tokens=24)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    bids = torch.empty((inp.B, 4), dtype=torch.int32, device="cuda")
    bsc = torch.empty((inp.B, d.cap // 8), dtype=torch.float32, device="cuda")
    dsa.index_blocks(cfg, d.q_idx, d.w, d.pooled, d.n_lat, d.cap, bids, d.ws, block_scores=bsc)
    tok = torch.empty((inp.B, 24), dtype=torch.int32, device="cuda")
    dsa.topk(cfg, d.q_idx, d.w, d.keys, None, d.n_lat, d.cap, tok, d.ws)
    assert d.status()[0] == 0
    bids, bsc, tok = bids.cpu().numpy(), bsc.cpu().numpy(), tok.cpu().numpy()
    oc = oracle_cfg(cfg)
    for b in range(inp.B):
        r = O.decode_sequence(oc, inp, b, with_attention=False)
        nb = len(r["block_scores"])
        check_scores(bsc[b, :nb], r["block_scores"], f"block scores {b}")
        check_ids(bids[b], r["block_ids"], lambda i: r["block_scores"][i], 4, f"blocks {b}")
        single = O.select_query(O.StepConfig(k_blocks=1 << 20, k_tokens=24), inp.q_idx[b],
                                inp.w[b], O.decode_keys(fmt, inp.keys.data[b][:T[b]],
                                None if inp.keys.scales is None else inp.keys.scales[b][:T[b]]),
                                np.zeros(((T[b] + 7) // 8, 128)), T[b])
        pos = {int(t): s for t, s in zip(single["cand"], single["token_scores"])}
        check_ids(tok[b], single["token_ids"], lambda i: pos[i], 24, f"tokens {b}")


@pytest.mark.parametrize("fmt,k_blocks", [("bf16", 64), ("mxfp8", 64), ("bf16", 4096)])
def test_select_all_scores_tied(fmt, k_blocks):
    """Weights 0 make every score 0: both tiers must keep the lowest indices
    (the tie rule), whatever path the selection takes for heavy ties. With
    4096 of 5000 blocks most candidates are kept and the shorter sequence
    keeps all of its blocks, padded with -1."""
    inp = synth.decode_inputs([40000, 30001], 1, fmt, seed=42)
    inp.w[:] = 0.0
    cfg = dsa.config(k_blocks=k_blocks, k_tokens=100)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    bids = torch.empty((inp.B, k_blocks), dtype=torch.int32, device="cuda")
    dsa.index_blocks(cfg, d.q_idx, d.w, d.pooled, d.n_lat, d.cap, bids, d.ws)
    tok = torch.empty((inp.B, 100), dtype=torch.int32, device="cuda")
    dsa.topk(cfg, d.q_idx, d.w, d.keys, bids, d.n_lat, d.cap, tok, d.ws)
    tok_all = torch.empty((inp.B, 100), dtype=torch.int32, device="cuda")
    dsa.topk(cfg, d.q_idx, d.w, d.keys, None, d.n_lat, d.cap, tok_all, d.ws)
    assert d.status()[0] == 0
    for b in range(inp.B):
        nb = (int(inp.n_latents[b]) + 7) // 8
        m = min(k_blocks, nb)
        assert bids[b].tolist() == list(range(m)) + [-1] * (k_blocks - m)
        assert tok[b].tolist() == list(range(100))
        assert tok_all[b].tolist() == list(range(100))


def top_k_of(scores, k):
    """Ids of the k best finite scores (score desc, index asc), ascending, -1 padded."""
    scores = np.asarray(scores)
    idx = np.flatnonzero(np.isfinite(scores))
    order = np.lexsort((idx, -scores[idx].astype(np.float64)))
    sel = np.sort(idx[order[:k]])
    return np.concatenate([sel, np.full(k - len(sel), -1)]).astype(np.int64)


def scale_key_row(inp, b, t, log2_factor):
    """Multiply index key t of sequence b by 2**log2_factor, exactly."""
    if inp.keys.fmt == "bf16":
        row = inp.keys.data[b, t]
        nz = (row & 0x7FFF) != 0
        row[nz] = row[nz] + np.uint16(log2_factor << 7)
    else:
        inp.keys.scales[b, t] += np.uint8(log2_factor)


@pytest.mark.parametrize("T,fmt,k_blocks,outliers", [
    ([60000, 33000, 20000], "bf16", 2048, False),
    ([60000, 33000, 20000], "mxfp8", 4096, False),
    ([60000, 33000, 20000], "bf16", 2048, True),
    ([60000, 33000, 20000], "mxfp8", 600, True),
    ([300000, 270001, 5000], "mxfp8", 2048, False),  # 37500 blocks: two-pass selection
    ([300000, 270001, 5000], "bf16", 64, True),
    ([60000, 33000, 20000], "mxfp4", 2048, True),
])
def test_select_thousands_of_candidates(T, fmt, k_blocks, outliers):
    """Block sets of 600-37500 and token sets of 4800-32768 candidates (above
    32768 a query's block selection runs in two passes, chunk by chunk, then
    over the chunks' winners). With outliers a
    few keys are 4096x larger, so nearly every other score falls in the lowest
    few of the value-space bins and the selection must refine by key bits.
    The ids are checked against the oracle and, exactly, against the scores the
    GPU returned (top-k of those by score desc, index asc)."""
    inp = synth.decode_inputs(T, 1, fmt, seed=26)
    if outliers:
        for t in (803, 32001, 56000):
            scale_key_row(inp, 0, t, 12)
        scale_key_row(inp, 1, 9, 12)
    cfg = dsa.config(k_blocks=k_blocks, k_tokens=512, ratio=1)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    nbc = d.cap // 8
    bids = torch.empty((inp.B, k_blocks), dtype=torch.int32, device="cuda")
    bsc = torch.empty((inp.B, nbc), dtype=torch.float32, device="cuda")
    dsa.index_blocks(cfg, d.q_idx, d.w, d.pooled, d.n_lat, d.cap, bids, d.ws, block_scores=bsc)
    tok = torch.empty((inp.B, 512), dtype=torch.int32, device="cuda")
    tsc = torch.empty((inp.B, k_blocks * 8), dtype=torch.float32, device="cuda")
    dsa.topk(cfg, d.q_idx, d.w, d.keys, bids, d.n_lat, d.cap, tok, d.ws, token_scores=tsc)
    assert d.status()[0] == 0
    bids_h, bsc_h = bids.cpu().numpy(), bsc.cpu().numpy()
    tok_h, tsc_h = tok.cpu().numpy(), tsc.cpu().numpy()
    oc = oracle_cfg(cfg)
    for b in range(inp.B):
        assert np.array_equal(bids_h[b], top_k_of(bsc_h[b], k_blocks)), f"blocks {b} vs own scores"
        cand = top_k_of(tsc_h[b], 512)
        want = np.where(cand >= 0, 8 * bids_h[b][np.maximum(cand, 0) // 8] + cand % 8, -1)
        assert np.array_equal(tok_h[b], want), f"tokens {b} vs own scores"
        r = O.decode_sequence(oc, inp, b, with_attention=False)
        nb = len(r["block_scores"])
        check_scores(bsc_h[b, :nb], r["block_scores"], f"block scores {b}")
        check_ids(bids_h[b], r["block_ids"], lambda i: r["block_scores"][i], k_blocks,
                  f"blocks {b}")
        r = O.decode_sequence(oc, inp, b, with_attention=False, block_ids=bids_h[b])
        pos = {int(t): s for t, s in zip(r["cand"], r["token_scores"])}
        check_ids(tok_h[b], r["token_ids"], lambda i: pos[i], 512, f"tokens {b}")


@pytest.mark.parametrize("B,t_max", [(3, 9000), (30, 9000), (50, 9000), (100, 9000),
                                     (100, 5000), (100, 6000)])
def test_select_cluster_paths(B, t_max):
    """A query's candidates are split over a cluster of 4 or 2 CTAs while the
    B clusters fit the SMs at once (one CTA a query beyond), each CTA holding a
    contiguous share; the CTAs merge their key ranges, histograms, members of
    the threshold bin and output offsets. Token selection over every latent of
    ragged sequences of 200-9000 latents (a share of 4096 candidates a CTA
    leaves the fourth CTA of a 9000-latent query with none), with: every score
    tied in some sequences (w = 0: the lowest ids win across the CTAs),
    outlier keys in others (the value-space bins degenerate and the radix
    levels run), and a sequence with fewer latents than k (-1 padding). The ids
    must equal the top-k of the scores the GPU returned (score desc, index
    asc), and two sequences' scores are checked against the oracle. At 100
    queries one CTA takes a query; 5000 and 6000 candidates run the 5- and
    6-slot variants."""
    rng = np.random.default_rng(2000 + B + t_max)
    T = [int(t) for t in rng.integers(300, t_max, B)]
    T[0], T[-1] = t_max, 200
    inp = synth.decode_inputs(T, 1, "mxfp8", seed=60 + B)
    for b in range(1, B, 5):
        inp.w[b] = 0.0
    for b in range(2, B, 5):
        for t in rng.integers(0, T[b], 3):
            scale_key_row(inp, b, int(t), 12)
    cfg = dsa.config(k_tokens=512, ratio=1)
    d = DecodeOnDevice(inp, cfg)
    n_cand = (d.cap + 7) // 8 * 8
    tok = torch.empty((B, 512), dtype=torch.int32, device="cuda")
    tsc = torch.empty((B, n_cand), dtype=torch.float32, device="cuda")
    dsa.topk(cfg, d.q_idx, d.w, d.keys, None, d.n_lat, d.cap, tok, d.ws, token_scores=tsc)
    assert d.status()[0] == 0
    tok_h, tsc_h = tok.cpu().numpy(), tsc.cpu().numpy()
    for b in range(B):
        assert np.isneginf(tsc_h[b, T[b]:]).all(), f"scores past the sequence {b}"
        assert np.array_equal(tok_h[b], top_k_of(tsc_h[b], 512)), f"tokens {b} vs own scores"
        if inp.w[b].max() == 0.0:
            assert tok_h[b].tolist() == list(range(min(512, T[b]))) + [-1] * max(0, 512 - T[b])
    assert tok_h[B - 1].tolist() == list(range(200)) + [-1] * 312
    oc = oracle_cfg(cfg)
    for b in (0, 2):
        single = O.select_query(O.StepConfig(k_blocks=1 << 20, k_tokens=512), inp.q_idx[b],
                                inp.w[b], O.decode_keys("mxfp8", inp.keys.data[b][:T[b]],
                                                        inp.keys.scales[b][:T[b]]),
                                np.zeros(((T[b] + 7) // 8, 128)), T[b])
        check_scores(tsc_h[b, :T[b]], single["token_scores"], f"token scores {b}")
        pos = {int(t): s for t, s in zip(single["cand"], single["token_scores"])}
        check_ids(tok_h[b], single["token_ids"], lambda i: pos[i], 512, f"tokens {b}")


# ---------------------------------------------------------------------------
# Failure report: a bounded device wait that runs out
# ---------------------------------------------------------------------------


def test_bounded_wait_reports_a_timeout_and_the_device_stays_usable():
    """A wait that nothing satisfies gives up after its limit (~1 ms here) and
    records DSA_ERR_TIMEOUT (site 6); the status is read and cleared on the
    host and the next step runs normally."""
    inp = synth.decode_inputs([300, 40], 1, "bf16", seed=31)
    cfg = dsa.config(k_blocks=16, k_tokens=64)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    dsa.selftest_timeout(d.ws)
    code, info = d.status()
    assert code == 7, (code, hex(info))
    assert info >> 24 == 6
    assert d.status()[0] == 0  # read and cleared
    outs = run_step(d, cfg, update_pool=True)
    assert d.status()[0] == 0
    assert np.isfinite(outs[1].cpu().numpy()).all()
    check_step(inp, cfg, outs, [0, 1])

