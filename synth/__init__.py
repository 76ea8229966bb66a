"""Seeded synthetic workloads for the two-tier sparse-attention step.

This module holds none of the attention method's arithmetic: it only produces
input bytes (bf16 values as uint16 bit patterns, MXFP8 codes and UE8M0
scales, fp32 head weights) from a counter-based SplitMix64 stream, through the
small C library built from ``gen.c`` beside this file. The CUDA path and the
CPU oracle are both fed these bytes; neither computes them.

Distributions follow the workloads of the two-tier sparse-attention step of
DeepSeek-V4.1 (recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview, bullet
"Two-tier sparse attention"; miles.radixark.com "DeepSeek-V4.1 Flash", §1
Architecture): values N(0,1)/sqrt(d) with d = 512 for query heads, latents and
window rows and d = 128 for index queries and index keys; head weights U(0,1).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None

# Dimensions of the step (miles.radixark.com "DeepSeek-V4.1 Flash", §1:
# 64 query heads, one 512-wide latent; index heads and width of the indexer).
N_HEADS = 64
LATENT_DIM = 512
N_IDX_HEADS = 16
IDX_DIM = 128
WINDOW = 128

# Stream tags, one per tensor.
TAG_Q, TAG_QIDX, TAG_W, TAG_LAT, TAG_KEYS, TAG_SWA = 1, 2, 3, 4, 5, 6

BF16_POS_INF = np.uint16(0x7F80)


def build(force: bool = False) -> str:
    """Compile libsynth.so from gen.c with gcc (OpenMP) if it is missing or stale."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.synth_normal_bf16.argtypes = [u64, u64, i64, i64, dbl, vp]
        lib.synth_normal_f32.argtypes = [u64, u64, i64, i64, dbl, vp]
        lib.synth_normal_e4m3.argtypes = [u64, u64, i64, i64, dbl, dbl, vp]
        lib.synth_uniform_f32.argtypes = [u64, u64, i64, i64, vp]
        lib.synth_normal_mxfp8.argtypes = [u64, u64, i64, i64, ctypes.c_int, dbl, vp, vp]
        lib.synth_normal_mxfp4.argtypes = [u64, u64, i64, i64, ctypes.c_int, dbl, vp, vp]
        lib.synth_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


def num_threads() -> int:
    return int(_load().synth_num_threads())


def normal_bf16(seed: int, tag: int, offset: int, n: int, scale: float, out=None) -> np.ndarray:
    """bf16 bit patterns of scale * N(0,1), counters offset .. offset + n - 1."""
    out = np.empty(n, np.uint16) if out is None else out
    if n:
        _load().synth_normal_bf16(seed, tag, offset, n, scale, _ptr(out))
    return out


def normal_f32(seed: int, tag: int, offset: int, n: int, scale: float) -> np.ndarray:
    out = np.empty(n, np.float32)
    if n:
        _load().synth_normal_f32(seed, tag, offset, n, scale, _ptr(out))
    return out


def normal_e4m3(seed: int, tag: int, offset: int, n: int, scale: float, kv_scale: float,
                out=None) -> np.ndarray:
    """E4M3 codes (round to nearest even) of fp32(scale * N(0,1)) / kv_scale,
    the counters of normal_f32: an fp8 cache with one power-of-two scale."""
    out = np.empty(n, np.uint8) if out is None else out
    if n:
        _load().synth_normal_e4m3(seed, tag, offset, n, scale, kv_scale, _ptr(out))
    return out


def uniform_f32(seed: int, tag: int, offset: int, n: int) -> np.ndarray:
    """U[0,1) on a 2^-24 grid (exact in fp32)."""
    out = np.empty(n, np.float32)
    if n:
        _load().synth_uniform_f32(seed, tag, offset, n, _ptr(out))
    return out


def normal_mxfp8(seed: int, tag: int, row_offset: int, rows: int, dim: int, scale: float,
                 codes=None, scales=None):
    """MXFP8 rows of scale * N(0,1): (codes uint8 [rows, dim], scales uint8 [rows, dim/32])."""
    assert dim % 32 == 0
    codes = np.empty((rows, dim), np.uint8) if codes is None else codes
    scales = np.empty((rows, dim // 32), np.uint8) if scales is None else scales
    if rows:
        _load().synth_normal_mxfp8(seed, tag, row_offset, rows, dim, scale, _ptr(codes),
                                   _ptr(scales))
    return codes, scales


def normal_mxfp4(seed: int, tag: int, row_offset: int, rows: int, dim: int, scale: float,
                 packed=None, scales=None):
    """MXFP4 rows of scale * N(0,1): (packed e2m1 codes uint8 [rows, dim/2], element 2i
    in the low nibble; scales uint8 [rows, dim/32]). The values are those of
    normal_mxfp8 with the same arguments."""
    assert dim % 32 == 0
    packed = np.empty((rows, dim // 2), np.uint8) if packed is None else packed
    scales = np.empty((rows, dim // 32), np.uint8) if scales is None else scales
    if rows:
        _load().synth_normal_mxfp4(seed, tag, row_offset, rows, dim, scale, _ptr(packed),
                                   _ptr(scales))
    return packed, scales


def _seq_offset(b: int) -> int:
    # Counter space of sequence b: elements (b << 40) + row * dim + j.
    return b << 40


@dataclass
class Keys:
    """Index keys (or pooled keys) in one of the two storage formats.

    fmt "bf16": data uint16 [..., rows, 128], scales None.
    fmt "mxfp8": data uint8 e4m3 codes [..., rows, 128], scales uint8 UE8M0 [..., rows, 4].
    fmt "mxfp4": data uint8 packed e2m1 codes [..., rows, 64] (element 2i in the low
    nibble), scales uint8 UE8M0 [..., rows, 4].
    """
    fmt: str
    data: np.ndarray
    scales: Optional[np.ndarray] = None


@dataclass
class DecodeInputs:
    """One decode step for B sequences; sequence b has T[b] tokens.

    The query sits at position T[b] - 1. Latents visible: n_latents[b] =
    T[b] // ratio (rows beyond it, up to the allocated capacity, are never part
    of the sequence). Window slot s holds position T[b] - swa_len[b] + s.
    """
    T: np.ndarray              # int64 [B]
    ratio: int
    q: np.ndarray              # uint16 bf16 [B, 64, 512]
    q_idx: np.ndarray          # uint16 bf16 [B, 16, 128]
    w: np.ndarray              # float32 [B, 16]
    latents: np.ndarray        # uint16 bf16 [B, cap, 512]
    keys: Keys                 # [B, cap, 128]
    swa: np.ndarray            # uint16 bf16 [B, window, 512]
    n_latents: np.ndarray      # int32 [B]
    swa_len: np.ndarray        # int32 [B]
    window: int = WINDOW
    meta: dict = field(default_factory=dict)
    # "fp8": latents and window rows are E4M3 codes (uint8 [.., 512]) standing
    # for code * kv_scale
    kv_fmt: str = "bf16"
    kv_scale: float = 1.0

    @property
    def B(self) -> int:
        return int(self.T.shape[0])

    @property
    def cap(self) -> int:
        return int(self.latents.shape[1])


def decode_inputs(T, ratio: int, key_fmt: str, seed: int, window: int = WINDOW,
                  q_scale: float = 1.0, cap: Optional[int] = None,
                  poison_tail: bool = True, kv_fmt: str = "bf16",
                  kv_scale: float = 2.0 ** -6) -> DecodeInputs:
    """Build the synthetic decode workload.

    T: tokens per sequence (list). cap: latent rows allocated per sequence
    (default: max latents rounded up to a multiple of 8). q_scale multiplies
    the N(0,1)/sqrt(512) query (the "sharpened" variants use 8).
    poison_tail fills rows past each sequence's end with +inf (bf16) or the
    largest MXFP8 or MXFP4 value, so a kernel that reads them gives a visibly wrong result.
    kv_fmt "fp8": latents and window rows are the E4M3 codes of the same
    N(0,1)/sqrt(512) values divided by kv_scale (rows past the end: 448).
    """
    T = np.asarray(T, np.int64).reshape(-1)
    B = int(T.shape[0])
    n_lat = (T // ratio).astype(np.int32)
    if cap is None:
        cap = int(-(-int(n_lat.max(initial=0)) // 8) * 8) if B else 0
        cap = max(cap, 8)
    s512 = 1.0 / np.sqrt(512.0)
    s128 = 1.0 / np.sqrt(128.0)
    q = np.empty((B, N_HEADS, LATENT_DIM), np.uint16)
    q_idx = np.empty((B, N_IDX_HEADS, IDX_DIM), np.uint16)
    w = np.empty((B, N_IDX_HEADS), np.float32)
    if kv_fmt not in ("bf16", "fp8"):
        raise ValueError(kv_fmt)
    fp8 = kv_fmt == "fp8"
    lat = np.empty((B, cap, LATENT_DIM), np.uint8 if fp8 else np.uint16)
    swa = np.zeros((B, window, LATENT_DIM), np.uint8 if fp8 else np.uint16)
    swa_len = np.minimum(T, window).astype(np.int32)
    if key_fmt == "bf16":
        kdata = np.empty((B, cap, IDX_DIM), np.uint16)
        kscales = None
    elif key_fmt == "mxfp8":
        kdata = np.empty((B, cap, IDX_DIM), np.uint8)
        kscales = np.empty((B, cap, IDX_DIM // 32), np.uint8)
    elif key_fmt == "mxfp4":
        kdata = np.empty((B, cap, IDX_DIM // 2), np.uint8)
        kscales = np.empty((B, cap, IDX_DIM // 32), np.uint8)
    else:
        raise ValueError(key_fmt)
    for b in range(B):
        off = _seq_offset(b)
        normal_bf16(seed, TAG_Q, off, N_HEADS * LATENT_DIM, s512 * q_scale, out=q[b].reshape(-1))
        normal_bf16(seed, TAG_QIDX, off, N_IDX_HEADS * IDX_DIM, s128, out=q_idx[b].reshape(-1))
        w[b] = uniform_f32(seed, TAG_W, off, N_IDX_HEADS)
        n_sw = int(swa_len[b])
        if fp8:
            normal_e4m3(seed, TAG_LAT, off, cap * LATENT_DIM, s512, kv_scale,
                        out=lat[b].reshape(-1))
            if n_sw:
                normal_e4m3(seed, TAG_SWA, off, n_sw * LATENT_DIM, s512, kv_scale,
                            out=swa[b, :n_sw].reshape(-1))
        else:
            normal_bf16(seed, TAG_LAT, off, cap * LATENT_DIM, s512, out=lat[b].reshape(-1))
            if n_sw:
                normal_bf16(seed, TAG_SWA, off, n_sw * LATENT_DIM, s512,
                            out=swa[b, :n_sw].reshape(-1))
        if key_fmt == "bf16":
            normal_bf16(seed, TAG_KEYS, off, cap * IDX_DIM, s128, out=kdata[b].reshape(-1))
        elif key_fmt == "mxfp8":
            normal_mxfp8(seed, TAG_KEYS, b << 31, cap, IDX_DIM, s128, codes=kdata[b],
                         scales=kscales[b])
        else:
            normal_mxfp4(seed, TAG_KEYS, b << 31, cap, IDX_DIM, s128, packed=kdata[b],
                         scales=kscales[b])
        if poison_tail:
            n = int(n_lat[b])
            lat[b, n:] = BF16_POS_INF if kv_fmt == "bf16" else 0x7E
            if key_fmt == "bf16":
                kdata[b, n:] = BF16_POS_INF
            elif key_fmt == "mxfp8":
                kdata[b, n:] = 0x7E
                kscales[b, n:] = 254
            else:
                kdata[b, n:] = 0x77  # 6, 6
                kscales[b, n:] = 254
    return DecodeInputs(T=T, ratio=ratio, q=q, q_idx=q_idx, w=w, latents=lat,
                        keys=Keys(key_fmt, kdata, kscales), swa=swa, n_latents=n_lat,
                        swa_len=swa_len, window=window, kv_fmt=kv_fmt, kv_scale=kv_scale)


@dataclass
class MultiInputs:
    """A multi-query decode batch: sequence b holds T[b] tokens and its n_q
    queries sit at positions T[b] - n_q + i. Caches are those of a DecodeInputs
    batch; q, q_idx and w gain a query axis, and window row r of sequence b
    holds position T[b] - n_q - window + 1 + r (zero rows before position 0)."""
    T: np.ndarray
    n_q: int
    ratio: int
    q: np.ndarray          # uint16 bf16 [B, n_q, 64, 512]
    q_idx: np.ndarray      # uint16 bf16 [B, n_q, 16, 128]
    w: np.ndarray          # float32 [B, n_q, 16]
    latents: np.ndarray    # uint16 bf16 [B, cap, 512]
    keys: Keys             # [B, cap, ...]
    swa: np.ndarray        # uint16 bf16 [B, window + n_q - 1, 512]
    n_latents: np.ndarray  # int32 [B] = T // ratio
    window: int = WINDOW

    @property
    def B(self) -> int:
        return int(self.T.shape[0])

    @property
    def cap(self) -> int:
        return int(self.latents.shape[1])


def multi_inputs(T, n_q: int, ratio: int, key_fmt: str, seed: int, window: int = WINDOW,
                 q_scale: float = 1.0) -> MultiInputs:
    """A multi-query decode batch over the caches decode_inputs builds for the
    same T (its own query, index-query, weight and window streams)."""
    base = decode_inputs(T, ratio, key_fmt, seed, window=window, q_scale=q_scale)
    B = base.B
    s512 = 1.0 / np.sqrt(512.0)
    s128 = 1.0 / np.sqrt(128.0)
    q = np.empty((B, n_q, N_HEADS, LATENT_DIM), np.uint16)
    q_idx = np.empty((B, n_q, N_IDX_HEADS, IDX_DIM), np.uint16)
    w = np.empty((B, n_q, N_IDX_HEADS), np.float32)
    n_sw = window + n_q - 1
    swa = np.empty((B, n_sw, LATENT_DIM), np.uint16)
    for b in range(B):
        off = _seq_offset(b) + (1 << 39)  # apart from decode_inputs' streams
        normal_bf16(seed, TAG_Q, off, n_q * N_HEADS * LATENT_DIM, s512 * q_scale,
                    out=q[b].reshape(-1))
        normal_bf16(seed, TAG_QIDX, off, n_q * N_IDX_HEADS * IDX_DIM, s128,
                    out=q_idx[b].reshape(-1))
        w[b] = uniform_f32(seed, TAG_W, off, n_q * N_IDX_HEADS).reshape(n_q, N_IDX_HEADS)
        normal_bf16(seed, TAG_SWA, off, n_sw * LATENT_DIM, s512, out=swa[b].reshape(-1))
        first_pos = int(base.T[b]) - n_q - window + 1
        if first_pos < 0:
            swa[b, :min(n_sw, -first_pos)] = 0
    return MultiInputs(T=base.T, n_q=n_q, ratio=ratio, q=q, q_idx=q_idx, w=w,
                       latents=base.latents, keys=base.keys, swa=swa, n_latents=base.n_latents,
                       window=window)


def multi_as_prefill(inp: MultiInputs, b: int) -> "PrefillInputs":
    """Sequence b of a multi-query batch seen as a prefill chunk: n_q queries
    appended after T[b] - n_q tokens, with the same bytes (no copy of values)."""
    n_lat = int(inp.n_latents[b])
    keys = Keys(inp.keys.fmt, inp.keys.data[b], None if inp.keys.scales is None
                else inp.keys.scales[b])
    return PrefillInputs(ctx=int(inp.T[b]) - inp.n_q, ratio=inp.ratio, q=inp.q[b],
                         q_idx=inp.q_idx[b], w=inp.w[b], latents=inp.latents[b],
                         keys=keys, swa=inp.swa[b], window=inp.window)


@dataclass
class PrefillInputs:
    """A prefill chunk of n_q queries appended after ctx tokens of one sequence.

    Query i sits at position ctx + i. Latent j stands for positions
    [j * ratio, (j + 1) * ratio). Window row r holds position ctx - window + 1 + r
    (rows for negative positions exist but are never read).
    """
    ctx: int
    ratio: int
    q: np.ndarray          # uint16 bf16 [n_q, 64, 512]
    q_idx: np.ndarray      # uint16 bf16 [n_q, 16, 128]
    w: np.ndarray          # float32 [n_q, 16]
    latents: np.ndarray    # uint16 bf16 [n_lat, 512]
    keys: Keys             # [n_lat, 128]
    swa: np.ndarray        # uint16 bf16 [n_q + window - 1, 512]
    window: int = WINDOW

    @property
    def n_q(self) -> int:
        return int(self.q.shape[0])


def prefill_inputs(n_q: int, ctx: int, ratio: int, key_fmt: str, seed: int,
                   window: int = WINDOW, q_scale: float = 1.0) -> PrefillInputs:
    n_lat = (ctx + n_q) // ratio
    n_lat_cap = -(-n_lat // 8) * 8
    s512 = 1.0 / np.sqrt(512.0)
    s128 = 1.0 / np.sqrt(128.0)
    q = normal_bf16(seed, TAG_Q, 0, n_q * N_HEADS * LATENT_DIM, s512 * q_scale)
    q_idx = normal_bf16(seed, TAG_QIDX, 0, n_q * N_IDX_HEADS * IDX_DIM, s128)
    w = uniform_f32(seed, TAG_W, 0, n_q * N_IDX_HEADS)
    lat = normal_bf16(seed, TAG_LAT, 0, n_lat_cap * LATENT_DIM, s512)
    n_sw = n_q + window - 1
    swa = normal_bf16(seed, TAG_SWA, 0, n_sw * LATENT_DIM, s512)
    if key_fmt == "bf16":
        keys = Keys("bf16", normal_bf16(seed, TAG_KEYS, 0, n_lat_cap * IDX_DIM, s128)
                    .reshape(n_lat_cap, IDX_DIM))
    elif key_fmt == "mxfp8":
        c, s = normal_mxfp8(seed, TAG_KEYS, 0, n_lat_cap, IDX_DIM, s128)
        keys = Keys("mxfp8", c, s)
    elif key_fmt == "mxfp4":
        c, s = normal_mxfp4(seed, TAG_KEYS, 0, n_lat_cap, IDX_DIM, s128)
        keys = Keys("mxfp4", c, s)
    else:
        raise ValueError(key_fmt)
    return PrefillInputs(ctx=ctx, ratio=ratio,
                         q=q.reshape(n_q, N_HEADS, LATENT_DIM),
                         q_idx=q_idx.reshape(n_q, N_IDX_HEADS, IDX_DIM),
                         w=w.reshape(n_q, N_IDX_HEADS),
                         latents=lat.reshape(n_lat_cap, LATENT_DIM)[:n_lat_cap],
                         keys=keys, swa=swa.reshape(n_sw, LATENT_DIM), window=window)


def paginate(arr: np.ndarray, page_rows: int, seed: int, spare_pages: int = 3,
             poison: int = 0xFF):
    """Lays a per-sequence cache arr [B, cap, ...] out as a pool of pages, the
    way a serving engine's block table does: sequence b's logical page p (rows
    [p * page_rows, (p + 1) * page_rows)) goes to physical page table[b, p] of
    pool [n_pages * page_rows, ...]. Physical pages are a seeded permutation of
    B * pages_per_seq + spare_pages pages; the spare ones and the rows past cap
    are filled with the byte `poison`. Returns (pool, table int32 [B, pages_per_seq]).
    Holds no arithmetic of the method: only where bytes go."""
    arr = np.asarray(arr)
    B, cap = arr.shape[0], arr.shape[1]
    pps = max(1, -(-cap // page_rows))
    n_pages = B * pps + spare_pages
    rng = np.random.default_rng(seed)
    perm = rng.permutation(n_pages)
    table = perm[:B * pps].reshape(B, pps).astype(np.int32)
    pool = np.empty((n_pages * page_rows,) + arr.shape[2:], arr.dtype)
    pool.view(np.uint8)[...] = poison
    for b in range(B):
        for p in range(pps):
            lo, hi = p * page_rows, min(cap, (p + 1) * page_rows)
            dst = int(table[b, p]) * page_rows
            pool[dst:dst + hi - lo] = arr[b, lo:hi]
    return pool, table


# The workloads, named by what they are (tokens per sequence, batch,
# compression ratio, index-key format) with their seeds.
WORKLOADS = {
    "decode_b1_t4096_r2_bf16": dict(kind="decode", B=1, T=4096, ratio=2, key_fmt="bf16", seed=0),
    "decode_b32_t32768_r2_bf16": dict(kind="decode", B=32, T=32768, ratio=2, key_fmt="bf16",
                                      seed=1),
    "decode_b64_t131072_r1_mxfp8": dict(kind="decode", B=64, T=131072, ratio=1,
                                        key_fmt="mxfp8", seed=2),
    "prefill_q4096_ctx65536_r2_bf16": dict(kind="prefill", n_q=4096, ctx=65536, ratio=2,
                                           key_fmt="bf16", seed=3),
    "decode_b8_t1048576_r1_mxfp8": dict(kind="decode", B=8, T=1048576, ratio=1,
                                        key_fmt="mxfp8", seed=4),
    # The 64 x 131072 decode with the MXFP4 index cache the serving pages name
    # (recipes.vllm.ai "DeepSeek-V4.1-Flash", indexer_kv_dtype mxfp4).
    "decode_b64_t131072_r1_mxfp4": dict(kind="decode", B=64, T=131072, ratio=1,
                                        key_fmt="mxfp4", seed=2),
    # The same batch with every cache in shuffled pages of 64 tokens behind a
    # block table (the paged layout serving engines use).
    "decode_b64_t131072_r1_mxfp8_paged64": dict(kind="decode", B=64, T=131072, ratio=1,
                                                key_fmt="mxfp8", seed=2, page_rows=64),
    # The same batch with an fp8 KV cache (latents and window rows as E4M3
    # codes with one scale; recipes.vllm.ai "DeepSeek-V4.1-Flash", serving
    # configurations, --kv-cache-dtype fp8).
    "decode_b64_t131072_r1_mxfp8_fp8kv": dict(kind="decode", B=64, T=131072, ratio=1,
                                              key_fmt="mxfp8", seed=2, kv_fmt="fp8"),
    # Multi-query decode: the 64 x 131072 batch with 5 queries a sequence (a
    # DSpark block of draft tokens verified in one pass).
    "decode_mq5_b64_t131072_r1_mxfp8": dict(kind="multi", B=64, n_q=5, T=131072, ratio=1,
                                            key_fmt="mxfp8", seed=2),
}


def workload_inputs(name: str, **kw):
    spec = dict(WORKLOADS[name])
    kind = spec.pop("kind")
    spec.pop("page_rows", None)  # the layout, not the values
    spec.update(kw)
    if kind == "decode":
        B, T = spec.pop("B"), spec.pop("T")
        return decode_inputs([T] * B, **spec)
    if kind == "multi":
        B, T, n_q = spec.pop("B"), spec.pop("T"), spec.pop("n_q")
        return multi_inputs([T] * B, n_q, **spec)
    return prefill_inputs(**spec)
