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
