"""Two-tier sparse attention (DeepSeek-V4.1) on one GB300: Python binding.

A thin ctypes layer over libdsa.so (include/dsa.h). It marshals torch tensors
(device pointers) and the current CUDA stream into the C calls and turns
status codes into exceptions; every step of the computation runs in the
library's CUDA kernels. There is no fallback: if libdsa.so is missing, every
call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsa.so")

FMT_BF16 = 0
FMT_MXFP8 = 1
FMT_MXFP4 = 2
_FMT = {"bf16": FMT_BF16, "mxfp8": FMT_MXFP8, "mxfp4": FMT_MXFP4}

STATUS = {
    0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_MISALIGNED", 3: "DSA_ERR_UNSUPPORTED",
    4: "DSA_ERR_WORKSPACE", 5: "DSA_ERR_CUDA", 6: "DSA_ERR_DEVICE_CHECK", 7: "DSA_ERR_TIMEOUT",
}

EXPORTS = ("dsa_default_config", "dsa_status_string", "dsa_workspace_size",
           "dsa_pool_index_keys", "dsa_index_blocks", "dsa_topk", "dsa_sparse_attn_decode",
           "dsa_decode_step", "dsa_sparse_attn_prefill", "dsa_read_device_status",
           "dsa_profile_events", "dsa_launch_counts", "dsa_topk_noalloc",
           "dsa_selftest_timeout", "dsa_sparse_attn_decode_paged", "dsa_decode_multi",
           "dsa_compress_append")

TOPK_NOALLOC_MAX_SCORES = 1 << 21

KERNEL_KINDS = ("pool", "scan", "select", "attn", "other")


class DsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


class Config(ctypes.Structure):
    """dsa_config_t."""
    _fields_ = [("n_heads", ctypes.c_int), ("latent_dim", ctypes.c_int),
                ("n_idx_heads", ctypes.c_int), ("idx_dim", ctypes.c_int),
                ("block", ctypes.c_int), ("k_blocks", ctypes.c_int), ("k_tokens", ctypes.c_int),
                ("window", ctypes.c_int), ("ratio", ctypes.c_int), ("sm_scale", ctypes.c_float),
                ("kv_fmt", ctypes.c_int), ("kv_scale", ctypes.c_float)]


KV_BF16, KV_FP8_E4M3 = 0, 1


class _Pages(ctypes.Structure):
    """dsa_pages_t."""
    _fields_ = [("page_table", ctypes.c_void_p), ("page_rows", ctypes.c_int32),
                ("pages_per_seq", ctypes.c_int32), ("n_pages", ctypes.c_int64)]


class _Keys(ctypes.Structure):
    """dsa_keys_t / dsa_keys_out_t (same layout)."""
    _fields_ = [("fmt", ctypes.c_int), ("data", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("seq_stride_rows", ctypes.c_int64), ("pages", ctypes.POINTER(_Pages))]


_lib = None


def load() -> ctypes.CDLL:
    """Loads libdsa.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m two_tier_sparse_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        cp = ctypes.POINTER(Config)
        kp = ctypes.POINTER(_Keys)
        lib.dsa_default_config.argtypes = [cp]
        lib.dsa_default_config.restype = None
        lib.dsa_status_string.argtypes = [i32]
        lib.dsa_status_string.restype = ctypes.c_char_p
        lib.dsa_workspace_size.argtypes = [cp, i32, i64, ctypes.POINTER(sz)]
        lib.dsa_pool_index_keys.argtypes = [cp, kp, vp, i32, i64, i32, kp, vp, sz, vp]
        lib.dsa_index_blocks.argtypes = [cp, vp, vp, kp, vp, i32, i64, vp, vp, vp, sz, vp]
        lib.dsa_topk.argtypes = [cp, vp, vp, kp, vp, vp, i32, i64, vp, vp, vp, sz, vp]
        lib.dsa_sparse_attn_decode.argtypes = [cp, vp, vp, i64, vp, vp, vp, vp, i32, vp, vp, vp,
                                               sz, vp]
        lib.dsa_decode_step.argtypes = [cp, vp, vp, vp, kp, kp, i32, vp, i64, vp, i64, vp, vp, i32,
                                        vp, vp, vp, vp, vp, sz, vp]
        lib.dsa_sparse_attn_prefill.argtypes = [cp, i32, i64, vp, vp, vp, vp, kp, kp, vp, vp, vp,
                                                vp, vp, sz, vp]
        lib.dsa_read_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.dsa_profile_events.argtypes = [i32, ctypes.POINTER(vp), ctypes.POINTER(vp), i32]
        lib.dsa_launch_counts.argtypes = [ctypes.POINTER(ctypes.c_uint64), i32]
        lib.dsa_topk_noalloc.argtypes = [cp, vp, vp, kp, vp, vp, i32, i64, vp, vp]
        lib.dsa_selftest_timeout.argtypes = [vp, sz, vp]
        lib.dsa_sparse_attn_decode_paged.argtypes = [cp, vp, vp, ctypes.POINTER(_Pages), vp, vp,
                                                     vp, vp, i32, vp, vp, vp, sz, vp]
        lib.dsa_decode_multi.argtypes = [cp, i32, vp, vp, vp, vp, kp, kp, vp, i64, i64, vp, i32,
                                         vp, vp, vp, vp, sz, vp]
        lib.dsa_compress_append.argtypes = [cp, i32, vp, vp, vp, kp, vp, i64, kp, kp, i64, vp,
                                            sz, vp]
        for f in EXPORTS:
            if f not in ("dsa_default_config", "dsa_status_string"):
                getattr(lib, f).restype = ctypes.c_int
        _lib = lib
    return _lib


def _check(code: int, where: str) -> None:
    if code != 0:
        raise DsaError(code, where)


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def config(k_blocks=2048, k_tokens=512, window=128, ratio=1, sm_scale=0.0, kv_fmt=KV_BF16,
           kv_scale=1.0) -> Config:
    """kv_fmt: KV_BF16, or KV_FP8_E4M3 (latents and window rows as E4M3 codes
    standing for code * kv_scale; decode attention and the decode step only)."""
    c = Config()
    load().dsa_default_config(ctypes.byref(c))
    c.k_blocks, c.k_tokens, c.window, c.ratio = k_blocks, k_tokens, window, ratio
    c.sm_scale = sm_scale
    c.kv_fmt, c.kv_scale = kv_fmt, kv_scale
    return c


class Pages:
    """A page table (dsa_pages_t) over pools of n_pages pages of page_rows tokens:
    table is a device int32 tensor [B, pages_per_seq]."""

    def __init__(self, table: torch.Tensor, page_rows: int, n_pages: int):
        assert table.dtype == torch.int32 and table.dim() == 2
        self.table = table
        self.c = _Pages(table.data_ptr(), page_rows, table.shape[1], n_pages)


@dataclass
class Keys:
    """A key cache on the device: data [B, rows, 128] (bf16 as 16-bit words, or
    uint8 e4m3 codes) or [B, rows, 64] (uint8, two e2m1 codes a byte) and, for
    MXFP8 and MXFP4, scales uint8 [B, rows, 4]."""
    fmt: str
    data: torch.Tensor
    scales: Optional[torch.Tensor] = None
    pages: Optional[Pages] = None  # paged pool (data rows = n_pages x rows per page)

    def c(self) -> _Keys:
        stride = self.data.shape[-2] if self.data.dim() >= 3 else 0
        pages = ctypes.pointer(self.pages.c) if self.pages is not None else None
        return _Keys(_FMT[self.fmt], self.data.data_ptr(),
                     self.scales.data_ptr() if self.scales is not None else None, stride,
                     pages)


def workspace_size(cfg: Config, n_queries: int, max_latents: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().dsa_workspace_size(ctypes.byref(cfg), n_queries, max_latents, ctypes.byref(n)),
           "dsa_workspace_size")
    return int(n.value)


def workspace(cfg: Config, n_queries: int, max_latents: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace (the status word must start at zero)."""
    return torch.zeros(workspace_size(cfg, n_queries, max_latents), dtype=torch.uint8,
                       device=device)


def pool_index_keys(cfg, keys: Keys, n_latents, max_latents, pooled: Keys, ws, tail_only=False,
                    stream=None):
    B = n_latents.shape[0]
    _check(load().dsa_pool_index_keys(ctypes.byref(cfg), ctypes.byref(keys.c()), _p(n_latents), B,
                                      max_latents, int(tail_only), ctypes.byref(pooled.c()),
                                      _p(ws), ws.numel(), _stream(stream)), "dsa_pool_index_keys")


def index_blocks(cfg, q_idx, w, pooled: Keys, n_latents, max_latents, block_ids, ws,
                 block_scores=None, stream=None):
    B = q_idx.shape[0]
    _check(load().dsa_index_blocks(ctypes.byref(cfg), _p(q_idx), _p(w), ctypes.byref(pooled.c()),
                                   _p(n_latents), B, max_latents, _p(block_ids), _p(block_scores),
                                   _p(ws), ws.numel(), _stream(stream)), "dsa_index_blocks")


def topk(cfg, q_idx, w, keys: Keys, block_ids, n_latents, max_latents, token_ids, ws,
         token_scores=None, stream=None):
    B = q_idx.shape[0]
    _check(load().dsa_topk(ctypes.byref(cfg), _p(q_idx), _p(w), ctypes.byref(keys.c()),
                           _p(block_ids), _p(n_latents), B, max_latents, _p(token_ids),
                           _p(token_scores), _p(ws), ws.numel(), _stream(stream)), "dsa_topk")


def topk_noalloc(cfg, q_idx, w, keys: Keys, block_ids, n_latents, max_latents, token_ids,
                 stream=None):
    """dsa_topk without a workspace: for callers that cannot allocate device
    memory. Candidate scores go to a scratch array the library defines
    statically (at most TOPK_NOALLOC_MAX_SCORES values for the whole batch);
    calls that may overlap on the GPU share it and must be serialised."""
    B = q_idx.shape[0]
    _check(load().dsa_topk_noalloc(ctypes.byref(cfg), _p(q_idx), _p(w), ctypes.byref(keys.c()),
                                   _p(block_ids), _p(n_latents), B, max_latents, _p(token_ids),
                                   _stream(stream)), "dsa_topk_noalloc")


def sparse_attn_decode(cfg, q, latents, n_latents, token_ids, swa, swa_len, out, ws, lse=None,
                       stream=None):
    B = q.shape[0]
    _check(load().dsa_sparse_attn_decode(ctypes.byref(cfg), _p(q), _p(latents), latents.shape[1],
                                         _p(n_latents), _p(token_ids), _p(swa), _p(swa_len), B,
                                         _p(out), _p(lse), _p(ws), ws.numel(), _stream(stream)),
           "dsa_sparse_attn_decode")


def sparse_attn_decode_paged(cfg, q, latents, pages: Pages, n_latents, token_ids, swa, swa_len,
                             out, ws, lse=None, stream=None):
    """dsa_sparse_attn_decode over a paged latent pool (latents [n_pages * page_rows, 512])."""
    B = q.shape[0]
    _check(load().dsa_sparse_attn_decode_paged(ctypes.byref(cfg), _p(q), _p(latents),
                                               ctypes.byref(pages.c), _p(n_latents),
                                               _p(token_ids), _p(swa), _p(swa_len), B, _p(out),
                                               _p(lse), _p(ws), ws.numel(), _stream(stream)),
           "dsa_sparse_attn_decode_paged")


def decode_step(cfg, q, q_idx, w, keys: Keys, pooled: Keys, latents, n_latents, max_latents, swa,
                swa_len, out, ws, lse=None, block_ids=None, token_ids=None, update_pool=False,
                stream=None):
    B = q.shape[0]
    lat_stride = latents.shape[1] if keys.pages is None else 0
    _check(load().dsa_decode_step(ctypes.byref(cfg), _p(q), _p(q_idx), _p(w),
                                  ctypes.byref(keys.c()), ctypes.byref(pooled.c()),
                                  int(update_pool), _p(latents), lat_stride, _p(n_latents),
                                  max_latents, _p(swa), _p(swa_len), B, _p(block_ids),
                                  _p(token_ids), _p(out), _p(lse), _p(ws), ws.numel(),
                                  _stream(stream)), "dsa_decode_step")


def decode_multi(cfg, n_tokens, q, q_idx, w, keys: Keys, pooled: Keys, latents, max_latents, swa,
                 out, ws, lse=None, token_ids=None, stream=None):
    """Multi-query decode: q [B, n_q, 64, 512], each sequence's n_q queries at its
    last n_q positions (n_tokens [B] device int32)."""
    B, n_q = q.shape[0], q.shape[1]
    _check(load().dsa_decode_multi(ctypes.byref(cfg), n_q, _p(n_tokens), _p(q), _p(q_idx), _p(w),
                                   ctypes.byref(keys.c()), ctypes.byref(pooled.c()), _p(latents),
                                   latents.shape[1], max_latents, _p(swa), B, _p(out), _p(lse),
                                   _p(token_ids), _p(ws), ws.numel(), _stream(stream)),
           "dsa_decode_multi")


def compress_append(cfg, n_tokens, kv, gate, new_keys: Keys, latents, keys: Keys, pooled: Keys,
                    max_latents, ws, stream=None):
    """The cache append at the compression step: kv bf16 [B, ratio, 512], gate
    fp32 [B, ratio], new_keys one index-key row per sequence."""
    B = n_tokens.shape[0]
    lat_stride = latents.shape[1] if keys.pages is None else 0
    _check(load().dsa_compress_append(ctypes.byref(cfg), B, _p(n_tokens), _p(kv), _p(gate),
                                      ctypes.byref(new_keys.c()), _p(latents), lat_stride,
                                      ctypes.byref(keys.c()), ctypes.byref(pooled.c()),
                                      max_latents, _p(ws), ws.numel(), _stream(stream)),
           "dsa_compress_append")


def sparse_attn_prefill(cfg, ctx_len, q, q_idx, w, latents, keys: Keys, pooled: Keys, swa, out,
                        ws, lse=None, token_ids=None, stream=None):
    n_q = q.shape[0]
    _check(load().dsa_sparse_attn_prefill(ctypes.byref(cfg), n_q, ctx_len, _p(q), _p(q_idx),
                                          _p(w), _p(latents), ctypes.byref(keys.c()),
                                          ctypes.byref(pooled.c()), _p(swa), _p(out), _p(lse),
                                          _p(token_ids), _p(ws), ws.numel(), _stream(stream)),
           "dsa_sparse_attn_prefill")


def read_device_status(ws, stream=None):
    """(status code, info word); synchronises the stream and clears the status."""
    info = ctypes.c_uint32(0)
    code = load().dsa_read_device_status(_p(ws), _stream(stream), ctypes.byref(info))
    return int(code), int(info.value)


def selftest_timeout(ws, stream=None) -> None:
    """Launches the failure-report self-test: a wait that nothing satisfies
    runs out (about 1 ms) and records DSA_ERR_TIMEOUT in ws's status word (read
    it with read_device_status)."""
    _check(load().dsa_selftest_timeout(_p(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "dsa_selftest_timeout")


def profile_events(kind: str, starts, ends) -> None:
    """Brackets each later launch of kernel `kind` with the given torch.cuda.Events
    (recorded round-robin); pass empty lists to switch off."""
    n = len(starts)
    assert len(ends) == n
    for e in list(starts) + list(ends):
        if e.cuda_event == 0:
            e.record()  # torch creates its event lazily
    arr_s = (ctypes.c_void_p * max(n, 1))(*[ctypes.c_void_p(e.cuda_event) for e in starts])
    arr_e = (ctypes.c_void_p * max(n, 1))(*[ctypes.c_void_p(e.cuda_event) for e in ends])
    _profile_keepalive[kind] = (arr_s, arr_e, list(starts), list(ends))
    _check(load().dsa_profile_events(KERNEL_KINDS.index(kind), arr_s, arr_e, n),
           "dsa_profile_events")


_profile_keepalive: dict = {}


def launch_counts(reset: bool = False) -> dict:
    arr = (ctypes.c_uint64 * len(KERNEL_KINDS))()
    _check(load().dsa_launch_counts(arr, int(reset)), "dsa_launch_counts")
    return {k: int(arr[i]) for i, k in enumerate(KERNEL_KINDS)}


def default_tau() -> float:
    return 1.0 / math.sqrt(512.0)
