"""The cache append at the compression step (dsa_compress_append) on the GPU:
the new latent equals the oracle's softmax-gated pooling of its positions
(within one bf16 ulp: the kernel sums in fp32, the oracle in fp64), the new
index key is written as given, the block key of its block is re-pooled bit for
bit, and sequences that complete no latent are left as they were; contiguous
and paged caches."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
import two_tier_sparse_gb300 as dsa
from parity import dev, pooled_buffer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    from two_tier_sparse_gb300 import build
    build.build()
    dsa.load()
    torch.cuda.set_device(cuda_device)


def new_key_rows(fmt, B, seed):
    if fmt == "bf16":
        return synth.normal_bf16(seed, 9, 0, B * 128, 1 / np.sqrt(128)).reshape(B, 128), None
    if fmt == "mxfp8":
        return synth.normal_mxfp8(seed, 9, 0, B, 128, 1 / np.sqrt(128))
    return synth.normal_mxfp4(seed, 9, 0, B, 128, 1 / np.sqrt(128))


@pytest.mark.parametrize("fmt,ratio,page_rows", [("bf16", 2, 0), ("mxfp8", 1, 0),
                                                 ("mxfp4", 2, 0), ("mxfp8", 2, 64)])
def test_compress_append(fmt, ratio, page_rows):
    T = np.array([4096, 1001, 64, 2, 17, 0], np.int64)  # tokens after this step
    B = len(T)
    inp = synth.decode_inputs(T, ratio, fmt, seed=90)
    cap = inp.cap
    kv = synth.normal_bf16(91, 4, 0, B * ratio * 512, 1 / np.sqrt(512)).reshape(B, ratio, 512)
    gate = (synth.uniform_f32(91, 3, 0, B * ratio) * 8 - 4).reshape(B, ratio)
    nk, ns = new_key_rows(fmt, B, 92)
    cfg = dsa.config(ratio=ratio)
    n_lat = dev(inp.n_latents)
    if page_rows:
        kpool, table = synth.paginate(inp.keys.data, page_rows, 93)
        lpool, _ = synth.paginate(inp.latents, page_rows, 93)
        spool, _ = synth.paginate(inp.keys.scales, page_rows, 93)
        n_pages = kpool.shape[0] // page_rows
        pages = dsa.Pages(dev(table), page_rows, n_pages)
        keys = dsa.Keys(fmt, dev(kpool), dev(spool), pages)
        latents = dev(lpool)
        prow = n_pages * page_rows // 8
        pooled = dsa.Keys(fmt, torch.zeros((prow, 128), dtype=torch.uint8, device="cuda"),
                          torch.zeros((prow, 4), dtype=torch.uint8, device="cuda"), pages)

        def logical(t, b, rows, per_page):
            return O.gather_paged(t.cpu().numpy(), table[b], per_page, rows)
    else:
        keys = dsa.Keys(fmt, dev(inp.keys.data),
                        None if inp.keys.scales is None else dev(inp.keys.scales))
        latents = dev(inp.latents)
        pooled = pooled_buffer(fmt, B, cap // 8)

        def logical(t, b, rows, per_page):
            return t.cpu().numpy()[b, :rows]
    ws = dsa.workspace(cfg, B, cap)
    dsa.pool_index_keys(cfg, keys, n_lat, cap, pooled, ws)
    lat0 = latents.clone()
    new_keys = dsa.Keys(fmt, dev(nk), None if ns is None else dev(ns))
    dsa.compress_append(cfg, dev(T.astype(np.int32)), dev(kv), dev(gate), new_keys, latents,
                        keys, pooled, cap, ws)
    code, info = dsa.read_device_status(ws)
    assert code == 0, hex(info)
    pr = page_rows // 8
    for b in range(B):
        n = int(inp.n_latents[b])
        got_lat = logical(latents, b, max(n, 1), page_rows)
        was_lat = logical(lat0, b, max(n, 1), page_rows)
        if T[b] == 0 or T[b] % ratio:
            assert np.array_equal(got_lat, was_lat), f"seq {b} changed"
            continue
        j = n - 1
        want = O.compress_latent(kv[b], gate[b])
        g, w = O.bf16_to_f64(got_lat[j].view(np.uint16)), O.bf16_to_f64(want)
        assert np.all(np.abs(g - w) <= 2.0 ** -8 * np.abs(w) + 1e-30), f"seq {b} latent"
        assert np.array_equal(got_lat[:j], was_lat[:j]), f"seq {b} earlier rows"
        kd = logical(keys.data, b, n, page_rows)
        assert np.array_equal(kd[j].view(np.uint8), np.ascontiguousarray(nk[b]).view(np.uint8))
        ksc = None
        if ns is not None:
            ksc = logical(keys.scales, b, n, page_rows)
            assert np.array_equal(ksc[j], ns[b])
        # the block holding j, re-pooled from the updated keys
        kv_vals = O.decode_keys(fmt, kd, ksc)
        want_p, want_s = O.pool_keys(kv_vals, n, fmt)
        nb = want_p.shape[0]
        got_p = logical(pooled.data, b, nb, pr)
        got_p = got_p.view(np.uint16) if fmt == "bf16" else got_p
        assert np.array_equal(got_p[nb - 1], want_p[nb - 1]), f"seq {b} block key"
        if want_s is not None:
            assert np.array_equal(logical(pooled.scales, b, nb, pr)[nb - 1], want_s[nb - 1])
