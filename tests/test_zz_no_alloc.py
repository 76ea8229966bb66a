"""dsa_topk_noalloc, the token stage for callers that cannot allocate device
memory (its candidate scores live in a scratch array the library defines
statically), gives the same token ids as dsa_topk with a caller workspace, on
two calls in a row (the shared scratch keeps the previous call's contents).

This file is collected last on purpose, so that a run stopping at the first
failure has run every other test first; it also passes alone in a fresh
process."""
import ctypes

import numpy as np
import pytest
import torch

import synth
import two_tier_sparse_gb300 as dsa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    from two_tier_sparse_gb300 import build
    build.build()
    dsa.load()
    torch.cuda.set_device(cuda_device)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("fmt,ratio,T,k_blocks,gathered", [
    ("mxfp8", 1, [20000, 9001, 777, 5], 96, True),
    ("bf16", 2, [4096, 1000, 30], 2048, False),
    # more than 32768 candidates without a workspace: the selection without the
    # two-pass scratch (keys cached in shared memory up to 40960, global passes
    # beyond), against dsa_topk's two-pass selection
    ("bf16", 1, [36000, 33001], 4096, False),
    ("mxfp8", 1, [50000, 12345], 4096, False),
])
def test_noalloc_topk_matches_topk(fmt, ratio, T, k_blocks, gathered):
    inp = synth.decode_inputs(T, ratio, fmt, seed=40)
    cfg = dsa.config(k_blocks=k_blocks, ratio=ratio)
    B, cap = inp.B, inp.cap
    keys = dsa.Keys(fmt, _dev(inp.keys.data),
                    None if inp.keys.scales is None else _dev(inp.keys.scales))
    q_idx, w, n_lat = _dev(inp.q_idx), _dev(inp.w), _dev(inp.n_latents)
    ws = dsa.workspace(cfg, B, cap)
    bids = None
    if gathered:
        nbc = cap // 8
        shape = (B, nbc, 128)
        pdat = torch.zeros(shape, dtype=torch.int16 if fmt == "bf16" else torch.uint8,
                           device="cuda")
        psc = None if fmt == "bf16" else torch.zeros((B, nbc, 4), dtype=torch.uint8,
                                                     device="cuda")
        pooled = dsa.Keys(fmt, pdat, psc)
        dsa.pool_index_keys(cfg, keys, n_lat, cap, pooled, ws)
        bids = torch.empty((B, k_blocks), dtype=torch.int32, device="cuda")
        dsa.index_blocks(cfg, q_idx, w, pooled, n_lat, cap, bids, ws)
    ref = torch.empty((B, cfg.k_tokens), dtype=torch.int32, device="cuda")
    dsa.topk(cfg, q_idx, w, keys, bids, n_lat, cap, ref, ws)
    assert dsa.read_device_status(ws)[0] == 0
    for _ in range(2):
        got = torch.full((B, cfg.k_tokens), -7, dtype=torch.int32, device="cuda")
        dsa.topk_noalloc(cfg, q_idx, w, keys, bids, n_lat, cap, got)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)


def _gathered_case(fmt, T, k_blocks, seed):
    """Inputs, block ids and dsa_topk's token ids for a token stage over the
    block stage's choice (both computed with a caller workspace)."""
    inp = synth.decode_inputs(T, 1, fmt, seed=seed)
    cfg = dsa.config(k_blocks=k_blocks)
    B, cap = inp.B, inp.cap
    keys = dsa.Keys(fmt, _dev(inp.keys.data),
                    None if inp.keys.scales is None else _dev(inp.keys.scales))
    q_idx, w, n_lat = _dev(inp.q_idx), _dev(inp.w), _dev(inp.n_latents)
    ws = dsa.workspace(cfg, B, cap)
    nbc = cap // 8
    pdat = torch.zeros((B, nbc, 128), dtype=torch.int16 if fmt == "bf16" else torch.uint8,
                       device="cuda")
    psc = None if fmt == "bf16" else torch.zeros((B, nbc, 4), dtype=torch.uint8, device="cuda")
    pooled = dsa.Keys(fmt, pdat, psc)
    dsa.pool_index_keys(cfg, keys, n_lat, cap, pooled, ws)
    bids = torch.empty((B, k_blocks), dtype=torch.int32, device="cuda")
    dsa.index_blocks(cfg, q_idx, w, pooled, n_lat, cap, bids, ws)
    ref = torch.empty((B, cfg.k_tokens), dtype=torch.int32, device="cuda")
    dsa.topk(cfg, q_idx, w, keys, bids, n_lat, cap, ref, ws)
    assert dsa.read_device_status(ws)[0] == 0
    return dict(cfg=cfg, q_idx=q_idx, w=w, keys=keys, bids=bids, n_lat=n_lat, cap=cap, ref=ref)


def test_noalloc_smaller_call_after_a_larger_one():
    """The scratch keeps the previous call's scores. A large call (four long
    sequences) followed by a smaller one with other inputs, whose short
    sequences leave most of their block lists as -1 padding, must give exactly
    dsa_topk's ids for the smaller inputs: nothing the second call reads may
    come from the first."""
    big = _gathered_case("mxfp8", [40000, 39001, 38000, 30000], 256, seed=61)
    small = _gathered_case("mxfp8", [900, 333, 64], 256, seed=62)
    for c in (big, small):
        got = torch.full_like(c["ref"], -7)
        dsa.topk_noalloc(c["cfg"], c["q_idx"], c["w"], c["keys"], c["bids"], c["n_lat"],
                         c["cap"], got)
        torch.cuda.synchronize()
        assert torch.equal(got, c["ref"])
    assert (small["bids"].cpu().numpy() == -1).sum() > 256  # most of the list is padding


def test_noalloc_topk_rejects_requests_beyond_its_scratch():
    cfg = dsa.config(k_blocks=2048)
    lib = dsa.load()
    # 129 queries x 16384 candidates > 2^21 scores: refused before any launch.
    keys = dsa._Keys(0, 16, None, 1 << 20)
    code = lib.dsa_topk_noalloc(ctypes.byref(cfg), 16, 16, ctypes.byref(keys), 16, 16, 129,
                                1 << 20, 16, None)
    assert dsa.STATUS[code] == "DSA_ERR_WORKSPACE"
