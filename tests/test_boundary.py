"""The C-ABI library loads and exports every call include/dsa.h declares; host-side
argument checks answer without touching a GPU (no compute call runs here)."""
import ctypes
import os
import re

import pytest
import torch

import two_tier_sparse_gb300 as dsa
from two_tier_sparse_gb300 import build as dsa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def lib():
    dsa_build.build()
    return dsa.load()


def declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared()
    for n in ("dsa_index_blocks", "dsa_topk", "dsa_sparse_attn_decode",
              "dsa_sparse_attn_prefill"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared():
        assert hasattr(lib, name), name
    assert set(declared()) == set(dsa.EXPORTS)


def test_default_config_and_status_strings(lib):
    c = dsa.config()
    assert (c.n_heads, c.latent_dim, c.n_idx_heads, c.idx_dim, c.block) == (64, 512, 16, 128, 8)
    assert (c.k_blocks, c.k_tokens, c.window, c.ratio) == (2048, 512, 128, 1)
    for code, name in dsa.STATUS.items():
        assert lib.dsa_status_string(code).decode() == name
    assert lib.dsa_status_string(99).decode() == "DSA_ERR_UNKNOWN"


def test_workspace_size(lib):
    c = dsa.config()
    small = dsa.workspace_size(c, 1, 2048)
    big = dsa.workspace_size(c, 64, 131072)
    assert 0 < small < big
    # block scores (64 x 16384 fp32) and token scores (64 x 131072 fp32) at least
    assert big >= 64 * 16384 * 4 + 64 * 131072 * 4
    with pytest.raises(dsa.DsaError):
        dsa.workspace_size(c, -1, 10)


def _call_topk(lib, cfg, **over):
    args = dict(q=16, w=16, keys=dsa._Keys(0, 16, None, 100), block_ids=None, n=16, B=2,
                max_latents=100, tok=16, ts=None, ws=256, ws_bytes=1 << 30)
    args.update(over)
    keys = args["keys"]
    return lib.dsa_topk(ctypes.byref(cfg), args["q"], args["w"],
                        ctypes.byref(keys) if keys is not None else None, args["block_ids"],
                        args["n"], args["B"], args["max_latents"], args["tok"], args["ts"],
                        args["ws"], args["ws_bytes"], None)


def test_argument_errors_are_found_on_the_host(lib):
    # Pointers below are never dereferenced: every case fails validation first.
    cfg = dsa.config()
    assert _call_topk(lib, cfg, q=None) == 1                       # null pointer
    assert _call_topk(lib, cfg, q=18) == 2                         # misaligned
    assert _call_topk(lib, cfg, keys=dsa._Keys(1, 16, None, 100)) == 1  # MXFP8 without scales
    assert _call_topk(lib, cfg, keys=dsa._Keys(7, 16, None, 100)) == 1  # bad format
    assert _call_topk(lib, cfg, keys=dsa._Keys(3, 16, 16, 100)) == 1    # bad format
    assert _call_topk(lib, cfg, keys=dsa._Keys(2, 16, None, 100)) == 1  # MXFP4 without scales
    assert _call_topk(lib, cfg, keys=dsa._Keys(2, 16, 18, 100)) == 2    # scales misaligned
    assert _call_topk(lib, cfg, keys=dsa._Keys(2, 16, 16, 101)) == 1    # MXFP4: odd row stride
    assert _call_topk(lib, cfg, keys=dsa._Keys(0, 16, None, 50)) == 1   # stride < max_latents
    assert _call_topk(lib, cfg, ws_bytes=10) == 4                  # workspace too small
    assert _call_topk(lib, cfg, ws=None) == 4
    assert _call_topk(lib, cfg, ws=272) == 2                       # workspace not 256-aligned
    assert _call_topk(lib, cfg, B=-1) == 1
    bad = dsa.config()
    bad.n_heads = 32
    assert _call_topk(lib, bad) == 3                               # unsupported dims
    bad = dsa.config(k_tokens=513)
    assert _call_topk(lib, bad) == 1
    bad = dsa.config(window=0)
    assert _call_topk(lib, bad) == 1
    assert lib.dsa_read_device_status(None, None, None) == 1


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(dsa, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(dsa, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        dsa.load()


# The cases below pass fake device addresses (A is 256-byte aligned, A + 2 is
# not). None is dereferenced: each case stops in the host-side checks, and the
# zero-size calls return before any launch.
A = 1 << 12


def _k(fmt=0, data=A, scales=None, stride=100):
    return dsa._Keys(fmt, data, scales, stride)


def _ref(x):
    return ctypes.byref(x) if x is not None else None


def test_index_blocks_argument_errors(lib):
    cfg = dsa.config()

    def call(q=A, w=A, pooled=_k(stride=13), n=A, B=2, L=100, ids=A, sc=None, ws=A,
             wsb=1 << 30, c=cfg):
        return lib.dsa_index_blocks(ctypes.byref(c), q, w, _ref(pooled), n, B, L, ids, sc, ws,
                                    wsb, None)
    assert call(q=None) == 1
    assert call(ids=None) == 1
    assert call(n=None) == 1
    assert call(w=A + 4) == 2
    assert call(sc=A + 8) == 2
    assert call(pooled=None) == 1
    assert call(pooled=_k(stride=12)) == 1             # fewer rows than ceil(100 / 8) blocks
    assert call(pooled=_k(data=A + 2, stride=13)) == 2
    assert call(pooled=_k(fmt=1, scales=A + 2, stride=13)) == 2  # scales need 4-byte alignment
    assert call(ws=None) == 4
    assert call(wsb=16) == 4
    assert call(ws=A + 16) == 2                        # workspace not 256-byte aligned
    assert call(B=-1) == 1
    assert call(L=-1) == 1
    assert call(L=(1 << 30) + 1) == 1
    assert call(B=0) == 0                              # nothing to do, nothing launched


def test_attention_argument_errors(lib):
    cfg = dsa.config()

    def call(q=A, lat=A, stride=100, n=A, tok=A, swa=A, swl=A, B=2, out=A, lse=None, ws=A,
             wsb=1 << 30, c=cfg):
        return lib.dsa_sparse_attn_decode(ctypes.byref(c), q, lat, stride, n, tok, swa, swl, B,
                                          out, lse, ws, wsb, None)
    for bad in ("q", "lat", "n", "tok", "swa", "swl", "out"):
        assert call(**{bad: None}) == 1, bad
    assert call(stride=-1) == 1
    assert call(B=-1) == 1
    assert call(out=A + 2) == 2
    assert call(lse=A + 4) == 2
    assert call(ws=None) == 4
    assert call(ws=A + 16) == 2
    assert call(c=dsa.config(window=129)) == 1
    assert call(c=dsa.config(sm_scale=float("nan"))) == 1
    assert call(c=dsa.config(sm_scale=float("inf"))) == 1
    bad = dsa.config()
    bad.latent_dim = 256
    assert call(c=bad) == 3
    # the KV cache format: bf16 or E4M3 with a finite positive scale
    assert call(c=dsa.config(kv_fmt=2)) == 1
    assert call(c=dsa.config(kv_fmt=dsa.KV_FP8_E4M3, kv_scale=0.0)) == 1
    assert call(c=dsa.config(kv_fmt=dsa.KV_FP8_E4M3, kv_scale=float("inf"))) == 1
    assert call(c=dsa.config(kv_fmt=dsa.KV_FP8_E4M3, kv_scale=float("nan"))) == 1
    assert call(B=0) == 0
    assert call(B=0, c=dsa.config(kv_fmt=dsa.KV_FP8_E4M3, kv_scale=0.5)) == 0


def test_decode_step_argument_errors(lib):
    cfg = dsa.config()

    def call(q=A, qi=A, w=A, keys=_k(), pooled=_k(stride=13), lat=A, stride=100, n=A, L=100,
             swa=A, swl=A, B=2, bids=None, tok=None, out=A, lse=None, ws=A, wsb=1 << 30, c=cfg):
        return lib.dsa_decode_step(ctypes.byref(c), q, qi, w, _ref(keys), _ref(pooled), 1, lat,
                                   stride, n, L, swa, swl, B, bids, tok, out, lse, ws, wsb, None)
    assert call(pooled=None) == 1
    assert call(keys=None) == 1
    assert call(stride=99) == 1                        # latent rows per sequence < max_latents
    assert call(keys=_k(stride=99)) == 1               # key rows per sequence < max_latents
    assert call(pooled=_k(stride=12)) == 1
    assert call(keys=_k(fmt=1, scales=A), pooled=_k(stride=13)) == 1  # formats differ
    assert call(qi=None) == 1
    assert call(qi=A + 2) == 2
    assert call(tok=A + 8) == 2
    assert call(bids=A + 8) == 2
    assert call(ws=None) == 4
    assert call(wsb=1024) == 4
    assert call(B=-1) == 1
    assert call(B=0) == 0


def test_prefill_argument_errors(lib):
    cfg = dsa.config(ratio=2)

    def call(nq=16, ctx=100, q=A, qi=A, w=A, lat=A, keys=_k(), pooled=_k(), swa=A, out=A,
             lse=None, tok=None, ws=A, wsb=1 << 30, c=cfg):
        return lib.dsa_sparse_attn_prefill(ctypes.byref(c), nq, ctx, q, qi, w, lat, _ref(keys),
                                           _ref(pooled), swa, out, lse, tok, ws, wsb, None)
    assert call(nq=-1) == 1
    assert call(ctx=-1) == 1
    assert call(ctx=1 << 32) == 1                      # more latents than the library supports
    for bad in ("q", "qi", "w", "lat", "swa", "out"):
        assert call(**{bad: None}) == 1, bad
    assert call(out=A + 2) == 2
    assert call(tok=A + 4) == 2
    assert call(keys=None) == 1
    assert call(pooled=_k(fmt=1, scales=A)) == 1       # formats differ
    assert call(ws=None) == 4
    assert call(wsb=4096) == 4
    assert call(nq=0) == 0
    # an fp8 KV cache is a decode-only format
    assert call(c=dsa.config(ratio=2, kv_fmt=dsa.KV_FP8_E4M3, kv_scale=1.0)) == 3


def test_pool_argument_errors(lib):
    cfg = dsa.config()

    def call(keys=_k(), n=A, B=2, L=100, pooled=_k(stride=13), ws=A, wsb=1 << 30, c=cfg):
        return lib.dsa_pool_index_keys(ctypes.byref(c), _ref(keys), n, B, L, 0, _ref(pooled), ws,
                                       wsb, None)
    assert call(pooled=None) == 1
    assert call(keys=_k(fmt=1, scales=None)) == 1      # MXFP8 without scales
    assert call(pooled=_k(stride=12)) == 1
    assert call(n=None) == 1
    assert call(keys=_k(fmt=1, scales=A), pooled=_k(stride=13)) == 1
    assert call(ws=None) == 4
    assert call(B=-1) == 1
    assert call(B=0) == 0


def test_topk_noalloc_capacity_and_errors(lib):
    cfg = dsa.config()

    # The default request (129 queries) is beyond the scratch: a case that got
    # past the argument checks would stop at the capacity check, never launch.
    def call(q=A, w=A, keys=_k(stride=1 << 20), bids=A, n=A, B=129, L=1 << 20, tok=A, c=cfg):
        return lib.dsa_topk_noalloc(ctypes.byref(c), q, w, _ref(keys), bids, n, B, L, tok, None)
    # 2^21 fp32 candidate scores: 128 queries of 2048 x 8 candidates fit, 129 do not
    assert call(B=129) == 4
    assert call(bids=None, B=3) == 4                   # 3 x 2^20 latents without a block stage
    assert call(tok=None) == 1
    assert call(bids=A + 4) == 2
    assert call(keys=_k(stride=10)) == 1
    assert call(B=0) == 0


def test_paged_cache_argument_errors(lib):
    cfg = dsa.config()

    def pages(table=A, rows=64, per_seq=2, n=10):
        return dsa._Pages(table, rows, per_seq, n)

    def call_topk(pg, L=100):
        keys = dsa._Keys(0, A, None, 0, ctypes.pointer(pg) if pg is not None else None)
        return lib.dsa_topk(ctypes.byref(cfg), A, A, ctypes.byref(keys), None, A, 2, L, A, None,
                            A, 16, None)   # workspace too small: nothing may launch
    assert call_topk(pages()) == 4                     # valid pages, then the workspace check
    assert call_topk(pages(rows=32)) == 1              # pages of a multiple of 64 tokens
    assert call_topk(pages(rows=0)) == 1
    assert call_topk(pages(table=None)) == 1
    assert call_topk(pages(table=A + 2)) == 2
    assert call_topk(pages(per_seq=1), L=100) == 1     # 64 tokens a sequence < 100
    assert call_topk(pages(n=0)) == 1
    assert call_topk(pages(n=1 << 26)) == 1            # more than 2^31 rows in the pool
    pg = pages()
    # prefill reads one contiguous sequence
    keys = dsa._Keys(0, A, None, 0, ctypes.pointer(pg))
    assert lib.dsa_sparse_attn_prefill(ctypes.byref(dsa.config(ratio=2)), 16, 100, A, A, A, A,
                                       ctypes.byref(keys), ctypes.byref(keys), A, A, None, None,
                                       A, 1 << 30, None) == 1
    # the step's keys and block keys: both paged by the same table, or neither
    flat = dsa._Keys(0, A, None, 13, None)
    assert lib.dsa_decode_step(ctypes.byref(cfg), A, A, A, ctypes.byref(keys), ctypes.byref(flat),
                               1, A, 0, A, 100, A, A, 2, None, None, A, None, A, 16,
                               None) == 1
    assert lib.dsa_sparse_attn_decode_paged(ctypes.byref(cfg), A, A, None, A, A, A, A, 2, A,
                                            None, A, 1 << 30, None) == 1
    assert lib.dsa_sparse_attn_decode_paged(ctypes.byref(cfg), A, A, ctypes.byref(pages(rows=100)),
                                            A, A, A, A, 2, A, None, A, 1 << 30, None) == 1


def test_compress_append_argument_errors(lib):
    def call(c=dsa.config(ratio=2), B=2, n=A, kv=A, g=A, new=_k(stride=1), lat=A, stride=100,
             keys=_k(), pooled=_k(stride=13), L=100, ws=A, wsb=16):
        return lib.dsa_compress_append(ctypes.byref(c), B, n, kv, g, _ref(new), lat, stride,
                                       _ref(keys), _ref(pooled), L, ws, wsb, None)
    assert call() == 4                                  # valid, then the (tiny) workspace
    assert call(c=dsa.config(ratio=33)) == 3            # groups of more than 32 positions
    assert call(n=None) == 1 and call(kv=None) == 1 and call(g=None) == 1
    assert call(new=None) == 1 and call(keys=None) == 1 and call(pooled=None) == 1
    assert call(kv=A + 8) == 2
    assert call(g=A + 2) == 2
    assert call(stride=99) == 1                         # latent rows a sequence < capacity
    assert call(new=_k(fmt=1, scales=A, stride=1)) == 1  # formats differ
    assert call(B=-1) == 1
    # the append writes bf16 latents
    assert call(c=dsa.config(ratio=2, kv_fmt=dsa.KV_FP8_E4M3, kv_scale=1.0)) == 3


def test_hooks_and_self_test_argument_errors(lib):
    n_kinds = len(dsa.KERNEL_KINDS)
    assert lib.dsa_profile_events(-1, None, None, 0) == 1
    assert lib.dsa_profile_events(n_kinds, None, None, 0) == 1
    assert lib.dsa_profile_events(0, None, None, -1) == 1
    assert lib.dsa_profile_events(0, None, None, 2) == 1  # events needed when n > 0
    assert lib.dsa_profile_events(0, None, None, 0) == 0  # switched off
    assert lib.dsa_launch_counts(None, 0) == 1
    counts = (ctypes.c_uint64 * n_kinds)()
    assert lib.dsa_launch_counts(counts, 1) == 0
    assert lib.dsa_selftest_timeout(None, 1 << 20, None) == 1
    assert lib.dsa_selftest_timeout(A, 8, None) == 1     # smaller than the status word
    size = ctypes.c_size_t(0)
    assert lib.dsa_workspace_size(ctypes.byref(dsa.config()), 1, 10, None) == 1
    assert lib.dsa_workspace_size(None, 1, 10, ctypes.byref(size)) == 1


C_CALLER = r"""
#include <stdio.h>
#include <string.h>
#include "dsa.h"
int main(void) {
  dsa_config_t c;
  size_t bytes = 0;
  dsa_default_config(&c);
  if (c.n_heads != 64 || c.latent_dim != 512 || c.k_blocks != 2048 || c.k_tokens != 512) return 1;
  if (dsa_workspace_size(&c, 4, 4096, &bytes) != DSA_OK || bytes == 0) return 2;
  if (dsa_workspace_size(&c, -1, 4096, &bytes) != DSA_ERR_INVALID_ARG) return 3;
  if (strcmp(dsa_status_string(DSA_ERR_TIMEOUT), "DSA_ERR_TIMEOUT") != 0) return 4;
  printf("%zu\n", bytes);
  return 0;
}
"""


def test_header_is_plain_c_and_links_from_c(lib, tmp_path):
    """The boundary is a C ABI: the header compiles as strict C99 and a C program
    links against the library and calls it (host-only calls, no GPU)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(dsa.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), str(src), "-L", libdir, "-ldsa",
                    f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stderr)
    c = dsa.config()
    assert int(out.stdout) == dsa.workspace_size(c, 4, 4096)
