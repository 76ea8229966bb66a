"""Paged caches (a block table per sequence over shared page pools) on the GPU:
the whole decode step and the attention alone give, bit for bit, what they give
on the same logical caches laid out contiguously, and agree with the oracle; a
page-table entry outside the pool is reported as a device check, never read."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
import two_tier_sparse_gb300 as dsa
from parity import DecodeOnDevice, check_out, dev, host_u16
from test_gpu_parity import check_step, oracle_cfg, run_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    from two_tier_sparse_gb300 import build
    build.build()
    dsa.load()
    torch.cuda.set_device(cuda_device)


class PagedOnDevice:
    """The batch of a DecodeOnDevice with its index keys, block keys and latents
    in shuffled page pools behind one page table (spare pages poisoned)."""

    def __init__(self, inp, cfg, page_rows, seed):
        self.inp, self.cfg, self.page_rows = inp, cfg, page_rows
        B, cap = inp.B, inp.cap
        fmt = inp.keys.fmt
        kpool, table = synth.paginate(inp.keys.data, page_rows, seed)
        lpool, t2 = synth.paginate(inp.latents, page_rows, seed)
        assert np.array_equal(table, t2)
        spool = None
        if inp.keys.scales is not None:
            spool, t3 = synth.paginate(inp.keys.scales, page_rows, seed)
            assert np.array_equal(table, t3)
        self.table_h = table
        self.n_pages = kpool.shape[0] // page_rows
        self.pages = dsa.Pages(dev(table), page_rows, self.n_pages)
        self.keys = dsa.Keys(fmt, dev(kpool), None if spool is None else dev(spool), self.pages)
        prow = self.n_pages * page_rows // 8
        if fmt == "bf16":
            pd = torch.zeros((prow, 128), dtype=torch.int16, device="cuda")
            ps = None
        else:
            pd = torch.zeros((prow, 64 if fmt == "mxfp4" else 128), dtype=torch.uint8,
                             device="cuda")
            ps = torch.zeros((prow, 4), dtype=torch.uint8, device="cuda")
        self.pooled = dsa.Keys(fmt, pd, ps, self.pages)
        self.latents = dev(lpool)
        self.q, self.q_idx, self.w = dev(inp.q), dev(inp.q_idx), dev(inp.w)
        self.swa, self.swa_len, self.n_lat = dev(inp.swa), dev(inp.swa_len), dev(inp.n_latents)
        self.cap = cap
        self.ws = dsa.workspace(cfg, B, cap)

    def pool(self):
        dsa.pool_index_keys(self.cfg, self.keys, self.n_lat, self.cap, self.pooled, self.ws)

    def step(self, update_pool=False):
        B, cfg = self.inp.B, self.cfg
        out = torch.empty((B, 64, 512), dtype=torch.int16, device="cuda")
        lse = torch.empty((B, 64), dtype=torch.float32, device="cuda")
        bids = torch.empty((B, cfg.k_blocks), dtype=torch.int32, device="cuda")
        tok = torch.empty((B, cfg.k_tokens), dtype=torch.int32, device="cuda")
        dsa.decode_step(cfg, self.q, self.q_idx, self.w, self.keys, self.pooled, self.latents,
                        self.n_lat, self.cap, self.swa, self.swa_len, out, self.ws, lse=lse,
                        block_ids=bids, token_ids=tok, update_pool=update_pool)
        return out, lse, bids, tok

    def pooled_logical(self, b, nb):
        """Block keys of sequence b read back through the table (codes, scales)."""
        R = self.page_rows // 8
        data = self.pooled.data.cpu().numpy()
        sc = None if self.pooled.scales is None else self.pooled.scales.cpu().numpy()
        got = O.gather_paged(data, self.table_h[b], R, nb)
        return got, (None if sc is None else O.gather_paged(sc, self.table_h[b], R, nb))


@pytest.mark.parametrize("fmt,ratio,page_rows,k_blocks", [
    ("mxfp8", 1, 64, 128),     # both tiers, 8 block keys a page
    ("bf16", 2, 128, 200),
    ("mxfp4", 1, 64, 96),
    ("mxfp8", 1, 256, 4096),   # no block stage: the token stage over paged latents
])
def test_paged_decode_step_equals_contiguous(fmt, ratio, page_rows, k_blocks):
    T = [20000, 9001, 777, 64, 3]
    inp = synth.decode_inputs(T, ratio, fmt, seed=70, q_scale=8.0)
    cfg = dsa.config(k_blocks=k_blocks, ratio=ratio, sm_scale=8.0)
    d = DecodeOnDevice(inp, cfg)
    d.pool()
    want = run_step(d, cfg, update_pool=True)
    assert d.status()[0] == 0
    p = PagedOnDevice(inp, cfg, page_rows, seed=71)
    p.pool()
    got = p.step(update_pool=True)
    code, info = dsa.read_device_status(p.ws)
    assert code == 0, hex(info)
    for x, y, name in zip(got, want, ("out", "lse", "block ids", "token ids")):
        assert torch.equal(x, y), name
    pd = d.pooled.data.cpu().numpy()
    psc = None if d.pooled.scales is None else d.pooled.scales.cpu().numpy()
    for b in range(inp.B):
        nb = (int(inp.n_latents[b]) + 7) // 8
        g, gs = p.pooled_logical(b, nb)
        assert np.array_equal(g, pd[b, :nb]), f"block keys {b}"
        if gs is not None:
            assert np.array_equal(gs, psc[b, :nb]), f"block scales {b}"
    check_step(inp, cfg, got, [0, 2, 4])


@pytest.mark.parametrize("kv_fmt", ["bf16", "fp8"])
def test_paged_attention_equals_contiguous(kv_fmt):
    """Attention over a paged latent pool gives the bits of the contiguous
    cache, with bf16 rows and with an fp8 cache (E4M3 codes, one scale)."""
    inp = synth.decode_inputs([5000, 3001, 70], 1, "bf16", seed=72, q_scale=8.0, kv_fmt=kv_fmt)
    cfg = dsa.config(sm_scale=8.0, kv_fmt=dsa.KV_FP8_E4M3 if kv_fmt == "fp8" else dsa.KV_BF16,
                     kv_scale=inp.kv_scale)
    oc = oracle_cfg(cfg)
    refs = [O.decode_sequence(oc, inp, b) for b in range(inp.B)]
    ids = dev(np.stack([r["token_ids"] for r in refs]).astype(np.int32))
    d = DecodeOnDevice(inp, cfg)
    p = PagedOnDevice(inp, cfg, 64, seed=73)
    outs = []
    for paged in (False, True):
        out = torch.empty((inp.B, 64, 512), dtype=torch.int16, device="cuda")
        lse = torch.empty((inp.B, 64), dtype=torch.float32, device="cuda")
        if paged:
            dsa.sparse_attn_decode_paged(cfg, p.q, p.latents, p.pages, p.n_lat, ids, p.swa,
                                         p.swa_len, out, p.ws, lse=lse)
            assert dsa.read_device_status(p.ws)[0] == 0
        else:
            dsa.sparse_attn_decode(cfg, d.q, d.latents, d.n_lat, ids, d.swa, d.swa_len, out,
                                   d.ws, lse=lse)
            assert d.status()[0] == 0
        outs.append((out, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    out_h, lse_h = host_u16(outs[1][0]), outs[1][1].cpu().numpy()
    for b, r in enumerate(refs):
        check_out(out_h[b], lse_h[b], r["out"], r["lse"], f"seq {b}")


def test_page_entry_outside_the_pool_is_reported():
    """Sequence 1's first page points past the pool: the step records a device
    check (its rows are skipped, never read), and sequence 0 is unaffected."""
    inp = synth.decode_inputs([6000, 5000], 1, "mxfp8", seed=74)
    cfg = dsa.config(k_blocks=64)
    p = PagedOnDevice(inp, cfg, 64, seed=75)
    p.pool()
    good = p.step()
    assert dsa.read_device_status(p.ws)[0] == 0
    p.pages.table[1, 0] = p.n_pages + 5
    bad = p.step()
    code, info = dsa.read_device_status(p.ws)
    assert code == 6 and (info >> 24) in (2, 4), hex(info)   # scan or attention
    for x, y in zip(good, bad):
        assert torch.equal(x[0], y[0])
    assert np.isfinite(bad[1].cpu().numpy()[1]).all()
