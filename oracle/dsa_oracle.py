"""CPU oracle for the two-tier sparse-attention step (test infrastructure only).

This module is the plain, slow, obviously correct statement of what the step
computes. Only the tests, the smoke check and the benchmark's CPU-baseline leg
use it; the library never imports it and it imports nothing from the library.
Floating point runs in float64 except where the method itself fixes a storage
format (bf16, fp32, e4m3/UE8M0, e2m1/UE8M0); library matmuls serve as plain dot
products. The MXFP4 index-key format (e2m1 codes) is stated here ahead of the
library, which does not take it yet.

The method (DeepSeek-V4.1, two-tier sparse attention):
  * recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview, bullet "Two-tier sparse
    attention": every layer attends over a 128-token sliding window; layers with
    a compression ratio add compressed KV latents; an indexer side attention
    scores the latents and keeps the best 512 per query, after a candidate stage
    that keeps 2048 blocks of 8; ratios are 1 and 2.
  * miles.radixark.com "DeepSeek-V4.1 Flash", §1 Model Introduction,
    "Architecture" and "Sparse retrieval": one 512-wide latent per position
    serves as key and value for all 64 query heads (no value projection); a
    top-512 candidate set per retrieving layer; a coarser candidate-block pass.
  * Same page, §1: fp8 weights use a 32-wide UE8M0 block scale; the vLLM page's
    Overview bullet "Mixed MXFP4/MXFP8 checkpoint" names MXFP8 with UE8M0 scales.
  * The vLLM page's serving configurations set indexer_kv_dtype to mxfp4, and the
    sglang page lists an FP4 indexer cache: MXFP4 per OCP MX v1.0.
  * The pages leave the indexer formula open; this build fixes it as
    score = sum_h w_h * ReLU(q_h . k), the block key as the mean of the block's
    8 index keys and ties as "lower index first".

Readings taken where the pages are silent (each listed with its reason in the
design notes): softmax scale tau defaults to 1/sqrt(512); the window includes
the query's own position; latents and window rows are concatenated without
de-duplication (two different stores); a latent is visible only once all of
its positions are; a partial last block is the mean of its visible members;
pooled keys are stored in the index-key format; the block stage keeps every
block when there are at most k_blocks of them; fewer candidates than k keeps
them all and pads with -1; ids are reported in ascending order; the top-k
decisions rank on the score rounded to fp32 (the precision the kernels use),
with -0 equal to +0 and ties to the lower index.

Parity pins: every function here is pinned by tests in tests/test_oracle_*.py
against library routines, closed forms, brute force or invariants.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np

# ---------------------------------------------------------------------------
# Configuration of the step
# ---------------------------------------------------------------------------


@dataclass(frozen=True)
class StepConfig:
    """Dimensions of the step (miles.radixark.com "DeepSeek-V4.1 Flash", §1;
    recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview, "Two-tier sparse attention")."""
    n_heads: int = 64
    latent_dim: int = 512
    n_idx_heads: int = 16
    idx_dim: int = 128
    block: int = 8
    k_blocks: int = 2048
    k_tokens: int = 512
    window: int = 128
    ratio: int = 1
    sm_scale: Optional[float] = None  # None: 1/sqrt(latent_dim)

    @property
    def tau(self) -> float:
        return 1.0 / math.sqrt(self.latent_dim) if self.sm_scale is None else self.sm_scale


# ---------------------------------------------------------------------------
# Storage formats
# ---------------------------------------------------------------------------


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) to float64, exactly: bf16 is the top half of fp32."""
    u32 = np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """fp32 values to bf16 bit patterns, round to nearest, ties to even (no NaN input)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    keep = u >> np.uint64(16)
    rest = u & np.uint64(0xFFFF)
    up = (rest > 0x8000) | ((rest == 0x8000) & ((keep & np.uint64(1)) == 1))
    return (keep + up.astype(np.uint64)).astype(np.uint16)


def e4m3_value(code: int) -> float:
    """Value of an e4m3 code (OCP 8-bit floating point spec, E4M3: bias 7, no
    infinities, S.1111.111 is NaN, largest normal 448, subnormals m * 2^-9)."""
    s = -1.0 if code & 0x80 else 1.0
    E = (code >> 3) & 0xF
    m = code & 0x7
    if E == 0xF and m == 0x7:
        return math.nan
    if E == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (E - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], np.float64)


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """float64 values to e4m3 codes: round to nearest, ties to even, saturating
    finite values to +-448 (the OCP MX conversion's element rounding)."""
    y = np.asarray(y, np.float64)
    sign = np.where(np.signbit(y), 0x80, 0).astype(np.uint8)
    a = np.abs(y)
    code = np.zeros(y.shape, np.int64)
    sub = a < 2.0 ** -6
    code[sub] = np.rint(a[sub] * 2.0 ** 9).astype(np.int64)        # 0..8 (8 = 2^-6)
    nrm = ~sub
    if np.any(nrm):
        an = a[nrm]
        _, e = np.frexp(an)
        E = e.astype(np.int64) - 1
        m = np.rint((an / np.ldexp(1.0, E) - 1.0) * 8.0).astype(np.int64)
        carry = m == 8
        E[carry] += 1
        m[carry] = 0
        c = ((E + 7) << 3) | m
        c = np.where(E > 8, 0x7E, np.minimum(c, 0x7E))
        code[nrm] = c
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def ue8m0_scale(byte: np.ndarray) -> np.ndarray:
    """UE8M0 scale byte e -> 2^(e - 127) (byte 255 is NaN and rejected)."""
    b = np.asarray(byte, np.int64)
    if np.any(b == 255):
        raise ValueError("UE8M0 scale 0xFF (NaN) in input")
    return np.ldexp(1.0, b - 127)


def mxfp8_decode(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """MXFP8 rows [..., d] with scales [..., d/32] to float64, exactly:
    v = e4m3(code) * 2^(scale - 127) (OCP MX v1.0, 32-element blocks)."""
    codes = np.asarray(codes, np.uint8)
    if np.any((codes & 0x7F) == 0x7F):
        raise ValueError("e4m3 NaN code in input")
    v = E4M3_TABLE[codes]
    sc = ue8m0_scale(scales)
    shp = v.shape
    v = v.reshape(shp[:-1] + (shp[-1] // 32, 32)) * sc[..., None]
    return v.reshape(shp)


def mxfp8_encode(v32: np.ndarray):
    """fp32 rows [..., d] to MXFP8 (OCP MX v1.0): per 32-element group
    X = floor(log2(amax)) - 8 (8 = emax of e4m3), clamped to [-127, 127],
    X = 0 for an all-zero group; codes = e4m3(v / 2^X), scale byte X + 127."""
    v = np.asarray(v32, np.float32).astype(np.float64)
    shp = v.shape
    g = v.reshape(shp[:-1] + (shp[-1] // 32, 32))
    amax = np.max(np.abs(g), axis=-1)
    _, e = np.frexp(amax)
    X = np.where(amax > 0, e.astype(np.int64) - 1 - 8, 0)
    X = np.clip(X, -127, 127)
    codes = e4m3_encode(g * np.ldexp(1.0, -X)[..., None]).reshape(shp)
    return codes, (X + 127).astype(np.uint8)


def e2m1_value(code: int) -> float:
    """Value of a 4-bit e2m1 code (OCP MX v1.0, FP4 E2M1: 1 sign, 2 exponent
    bits with bias 1, 1 mantissa bit; no infinities or NaN; largest normal 6,
    subnormals m * 0.5)."""
    s = -1.0 if code & 0x8 else 1.0
    E = (code >> 1) & 0x3
    m = code & 0x1
    if E == 0:
        return s * m * 0.5
    return s * (1.0 + m / 2.0) * 2.0 ** (E - 1)


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], np.float64)


def e2m1_encode(y: np.ndarray) -> np.ndarray:
    """float64 values to e2m1 codes (0..15): round to nearest, ties to the even
    mantissa, finite values beyond 6 saturating to +-6 (the element rounding of
    the OCP MX conversion)."""
    y = np.asarray(y, np.float64)
    sign = np.where(np.signbit(y), 0x8, 0).astype(np.int64)
    a = np.abs(y)
    code = np.zeros(y.shape, np.int64)
    sub = a < 1.0
    code[sub] = np.rint(a[sub] * 2.0).astype(np.int64)             # 0, 1, or 2 (= 1.0)
    nrm = ~sub
    if np.any(nrm):
        an = a[nrm]
        _, e = np.frexp(an)
        E = e.astype(np.int64) - 1                                  # 2^E <= a < 2^(E+1)
        m = np.rint((an / np.ldexp(1.0, E) - 1.0) * 2.0).astype(np.int64)
        carry = m == 2
        E[carry] += 1
        m[carry] = 0
        c = ((E + 1) << 1) | m
        code[nrm] = np.where(E > 2, 0x7, np.minimum(c, 0x7))
    return (code | sign).astype(np.uint8)


def mxfp4_pack(codes: np.ndarray) -> np.ndarray:
    """e2m1 codes [..., d] to bytes [..., d/2]: element 2i in the low nibble,
    element 2i + 1 in the high one (this library's storage order)."""
    c = np.asarray(codes, np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def mxfp4_unpack(packed: np.ndarray) -> np.ndarray:
    """Bytes [..., d/2] to e2m1 codes [..., d] (inverse of mxfp4_pack)."""
    p = np.asarray(packed, np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def mxfp4_decode(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """MXFP4 rows (packed bytes [..., d/2], scales [..., d/32]) to float64,
    exactly: v = e2m1(code) * 2^(scale - 127) (OCP MX v1.0, 32-element blocks).
    The pages name the format for the indexer cache: recipes.vllm.ai
    "DeepSeek-V4.1-Flash" sets indexer_kv_dtype to mxfp4; the sglang page lists
    an FP4 indexer cache."""
    v = E2M1_TABLE[mxfp4_unpack(packed)]
    sc = ue8m0_scale(scales)
    shp = v.shape
    v = v.reshape(shp[:-1] + (shp[-1] // 32, 32)) * sc[..., None]
    return v.reshape(shp)


def mxfp4_encode(v32: np.ndarray):
    """fp32 rows [..., d] to MXFP4 (OCP MX v1.0): per 32-element group
    X = floor(log2(amax)) - 2 (2 = emax of e2m1), clamped to [-127, 127],
    X = 0 for an all-zero group; codes = e2m1(v / 2^X), packed two a byte;
    scale byte X + 127."""
    v = np.asarray(v32, np.float32).astype(np.float64)
    shp = v.shape
    g = v.reshape(shp[:-1] + (shp[-1] // 32, 32))
    amax = np.max(np.abs(g), axis=-1)
    _, e = np.frexp(amax)
    X = np.where(amax > 0, e.astype(np.int64) - 1 - 2, 0)
    X = np.clip(X, -127, 127)
    codes = e2m1_encode(g * np.ldexp(1.0, -X)[..., None]).reshape(shp)
    return mxfp4_pack(codes), (X + 127).astype(np.uint8)


def decode_keys(fmt: str, data: np.ndarray, scales: Optional[np.ndarray] = None) -> np.ndarray:
    """Index keys (or pooled keys) in their storage format to float64."""
    if fmt == "bf16":
        return bf16_to_f64(data)
    if fmt == "mxfp8":
        return mxfp8_decode(data, scales)
    if fmt == "mxfp4":
        return mxfp4_decode(data, scales)
    if fmt == "fp32":
        return np.asarray(data, np.float32).astype(np.float64)
    raise ValueError(fmt)


# ---------------------------------------------------------------------------
# S0: block-pooled index keys
# ---------------------------------------------------------------------------


def pool_mean_f32(members: np.ndarray) -> np.ndarray:
    """Mean of a block's visible member keys [c, d] (c >= 1): fp32 sum taken in
    member order, then divided by c in fp32 (block key = mean of the block's
    index keys; recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview, candidate stage
    of "blocks of 8")."""
    m = np.asarray(members, np.float32)
    acc = m[0].copy()
    for j in range(1, m.shape[0]):
        acc = (acc + m[j]).astype(np.float32)
    return (acc / np.float32(m.shape[0])).astype(np.float32)


def pool_keys(key_vals: np.ndarray, n_vis: int, fmt: str, block: int = 8):
    """Block keys of the first n_vis keys [n, d] (values exactly representable
    in fp32), stored in `fmt`. Returns (data, scales) for ceil(n_vis/block)
    blocks; the last block averages only its visible members."""
    kv = np.asarray(key_vals, np.float64)
    nb = -(-n_vis // block)
    d = kv.shape[-1]
    mean = np.empty((nb, d), np.float32)
    full = n_vis // block
    if full:
        x = kv[: full * block].astype(np.float32).reshape(full, block, d)
        acc = x[:, 0].copy()
        for j in range(1, block):
            acc = (acc + x[:, j]).astype(np.float32)
        mean[:full] = (acc / np.float32(block)).astype(np.float32)
    if nb > full:
        mean[full] = pool_mean_f32(kv[full * block: n_vis])
    return store_f32(mean, fmt)


def store_f32(v32: np.ndarray, fmt: str):
    """fp32 values to a storage format: (data, scales)."""
    if fmt == "bf16":
        return f32_to_bf16_rne(v32), None
    if fmt == "mxfp8":
        return mxfp8_encode(v32)
    if fmt == "mxfp4":
        return mxfp4_encode(v32)
    if fmt == "fp32":
        return np.asarray(v32, np.float32).copy(), None
    raise ValueError(fmt)


# ---------------------------------------------------------------------------
# Cache append: the compressed latent of a group of `ratio` positions
# ---------------------------------------------------------------------------


def compress_latent(kv_bits: np.ndarray, gate: np.ndarray) -> np.ndarray:
    """The latent of one group of positions, pooled by a softmax gate
    (recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview, "Two-tier sparse
    attention": compressed KV latents "pooled by a learned softmax gate"; ratio
    1 or 2 positions a latent). kv_bits: bf16 [ratio, D] (the group's per-position
    KV vectors, in position order); gate: the group's ratio gate logits (the
    learned projection that makes them is not on the pages, so they are given).
    latent = RN_bf16(sum_i softmax(gate)_i * kv_i), computed in float64."""
    g = np.asarray(gate, np.float32).astype(np.float64)
    e = np.exp(g - g.max())
    wts = e / e.sum()
    v = wts @ bf16_to_f64(kv_bits)
    return f32_to_bf16_rne(v.astype(np.float32))


# ---------------------------------------------------------------------------
# S1 / S3: indexer scores;  S2 / S4: top-k selection
# ---------------------------------------------------------------------------


def index_scores(q_idx: np.ndarray, w: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """score(k) = sum_h w_h * max(0, q_h . k) in float64, for keys [n, d],
    index query [H, d] and head weights [H]."""
    dots = np.asarray(keys, np.float64) @ np.asarray(q_idx, np.float64).T   # [n, H]
    return np.maximum(dots, 0.0) @ np.asarray(w, np.float64)


def rank_key(scores: np.ndarray) -> np.ndarray:
    """The value the top-k decisions compare: the score rounded to fp32, -0 as +0."""
    return np.asarray(scores, np.float64).astype(np.float32) + np.float32(0.0)


def topk_ids(scores: np.ndarray, ids: np.ndarray, k: int) -> np.ndarray:
    """Keep the k best candidates by (score desc, id asc); return their ids in
    ascending order, padded with -1 to length k when there are fewer."""
    ids = np.asarray(ids, np.int64)
    out = np.full(k, -1, np.int64)
    if ids.size == 0 or k == 0:
        return out
    order = np.lexsort((ids, -rank_key(scores).astype(np.float64)))
    keep = np.sort(ids[order[:k]])
    out[: keep.size] = keep
    return out


# ---------------------------------------------------------------------------
# S5 - S7: attention over gathered latents and the window, one softmax
# ---------------------------------------------------------------------------


def attend(q: np.ndarray, kv: np.ndarray, tau: float):
    """All heads of q [H, D] attend to rows kv [m, D], used as key and value:
    z = tau * q . v, p = softmax over the m rows, o = sum_j p_j v_j.
    Returns (o [H, D] float64, lse [H] float64 = log sum_j exp z_j)."""
    q = np.asarray(q, np.float64)
    kv = np.asarray(kv, np.float64)
    if kv.shape[0] == 0:
        return np.zeros_like(q), np.full(q.shape[0], -np.inf)
    z = tau * (q @ kv.T)                      # [H, m]
    m = np.max(z, axis=1, keepdims=True)
    e = np.exp(z - m)
    s = np.sum(e, axis=1, keepdims=True)
    p = e / s
    return p @ kv, (m + np.log(s))[:, 0]


def attention_probs(q: np.ndarray, kv: np.ndarray, tau: float) -> np.ndarray:
    z = tau * (np.asarray(q, np.float64) @ np.asarray(kv, np.float64).T)
    e = np.exp(z - np.max(z, axis=1, keepdims=True))
    return e / np.sum(e, axis=1, keepdims=True)


# ---------------------------------------------------------------------------
# One query: both selection tiers and the attention
# ---------------------------------------------------------------------------


def block_members(b: int, n_vis: int, block: int = 8) -> np.ndarray:
    return np.arange(b * block, min((b + 1) * block, n_vis), dtype=np.int64)


def select_query(cfg: StepConfig, q_idx_bits, w, key_vals: np.ndarray, pooled_vals: np.ndarray,
                 n_vis: int, block_ids: Optional[np.ndarray] = None) -> dict:
    """Both selection tiers for one query that sees n_vis latents.

    key_vals: decoded index keys [>= n_vis, d]; pooled_vals: decoded block keys
    [>= ceil(n_vis/8), d]. If block_ids is given it replaces the query's own
    block choice (used to re-check the token tier against another block set).
    """
    qi = bf16_to_f64(q_idx_bits)
    wf = np.asarray(w, np.float32).astype(np.float64)
    nb = -(-n_vis // cfg.block)
    bscores = index_scores(qi, wf, pooled_vals[:nb])
    all_blocks = np.arange(nb, dtype=np.int64)
    if block_ids is None:
        if nb <= cfg.k_blocks:
            block_ids = np.full(cfg.k_blocks, -1, np.int64)
            block_ids[:nb] = all_blocks
        else:
            block_ids = topk_ids(bscores, all_blocks, cfg.k_blocks)
    kept = np.asarray(block_ids, np.int64)
    kept = kept[kept >= 0]
    if kept.size:
        cand = np.concatenate([block_members(int(b), n_vis, cfg.block) for b in kept])
    else:
        cand = np.zeros(0, np.int64)
    tscores = index_scores(qi, wf, key_vals[cand]) if cand.size else np.zeros(0)
    token_ids = topk_ids(tscores, cand, cfg.k_tokens)
    return dict(block_scores=bscores, block_ids=np.asarray(block_ids, np.int64),
                cand=cand, token_scores=tscores, token_ids=token_ids)


def latent_values(rows: np.ndarray, kv_fmt: str = "bf16", kv_scale: float = 1.0) -> np.ndarray:
    """Latent or window rows as values. bf16: the bit patterns; fp8: E4M3 codes
    (OCP 8-bit floating point, the e4m3_value table above) times one scale for
    the whole cache -- the plainest reading of an "fp8" KV cache dtype
    (recipes.vllm.ai "DeepSeek-V4.1-Flash", serving configurations,
    --kv-cache-dtype fp8), which names no scale granularity."""
    if kv_fmt == "bf16":
        return bf16_to_f64(rows)
    if kv_fmt == "fp8":
        return E4M3_TABLE[np.asarray(rows, np.uint8)] * float(kv_scale)
    raise ValueError(kv_fmt)


def attend_query(cfg: StepConfig, q_bits, latents_bits: np.ndarray, token_ids: np.ndarray,
                 window_bits: np.ndarray, kv_fmt: str = "bf16", kv_scale: float = 1.0):
    """Attention of one query over its selected latents ++ its window rows
    (both in the cache format kv_fmt, see latent_values)."""
    ids = np.asarray(token_ids, np.int64)
    ids = ids[ids >= 0]
    kv = np.concatenate([latent_values(latents_bits[ids], kv_fmt, kv_scale),
                         latent_values(window_bits, kv_fmt, kv_scale)], axis=0)
    return attend(bf16_to_f64(q_bits), kv, cfg.tau)


# ---------------------------------------------------------------------------
# Decode: B sequences, the query at position T - 1
# ---------------------------------------------------------------------------


def gather_paged(pool: np.ndarray, page_table_row: np.ndarray, page_rows: int,
                 n_rows: int) -> np.ndarray:
    """Logical rows 0 .. n_rows - 1 of one sequence of a paged cache: row r is row
    r mod page_rows of physical page page_table_row[r // page_rows] of the pool
    [n_pages * page_rows, ...] (the block-table layout serving engines keep KV
    caches in; miles.radixark.com "DeepSeek-V4.1 Flash", §4.1, names a paged
    indexer). The step computes on these rows exactly as on a contiguous
    sequence."""
    r = np.arange(n_rows, dtype=np.int64)
    page = np.asarray(page_table_row, np.int64)[r // page_rows]
    return np.asarray(pool)[page * page_rows + r % page_rows]


def decoded_key_cache(keys_fmt: str, data: np.ndarray, scales) -> np.ndarray:
    return decode_keys(keys_fmt, data, scales)


def pooled_cache(cfg: StepConfig, key_vals: np.ndarray, n_vis: int, fmt: str):
    """S0 for one sequence: block keys of its n_vis latents, stored in fmt."""
    return pool_keys(key_vals, n_vis, fmt, cfg.block)


def decode_sequence(cfg: StepConfig, inp, b: int, with_attention: bool = True,
                    block_ids: Optional[np.ndarray] = None,
                    token_ids: Optional[np.ndarray] = None) -> dict:
    """The whole step for sequence b of a decode batch (synth.DecodeInputs layout).

    block_ids / token_ids, when given, replace the query's own choices of that
    tier (so later tiers can be checked against another implementation's
    choices)."""
    n_vis = int(inp.n_latents[b])
    kf = inp.keys.fmt
    kv = decode_keys(kf, inp.keys.data[b][:n_vis],
                     None if inp.keys.scales is None else inp.keys.scales[b][:n_vis])
    pdata, pscales = pooled_cache(cfg, kv, n_vis, kf)
    pv = decode_keys(kf, pdata, pscales)
    r = select_query(cfg, inp.q_idx[b], inp.w[b], kv, pv, n_vis, block_ids=block_ids)
    r["pooled"] = (pdata, pscales)
    if token_ids is not None:
        r["token_ids_used"] = np.asarray(token_ids, np.int64)
    else:
        r["token_ids_used"] = r["token_ids"]
    if with_attention:
        sw = int(inp.swa_len[b])
        o, lse = attend_query(cfg, inp.q[b], inp.latents[b], r["token_ids_used"],
                              inp.swa[b][:sw], getattr(inp, "kv_fmt", "bf16"),
                              getattr(inp, "kv_scale", 1.0))
        r["out"], r["lse"] = o, lse
    return r


# ---------------------------------------------------------------------------
# Prefill: n_q queries after ctx tokens, each with its own causal selection
# ---------------------------------------------------------------------------


def prefill_visible(ctx: int, i: int, ratio: int) -> int:
    """Latents visible to query i (position P = ctx + i): floor((P + 1) / ratio)."""
    return (ctx + i + 1) // ratio


def prefill_window_rows(ctx: int, i: int, window: int):
    """Rows of the prefill window buffer (row r = position ctx - window + 1 + r)
    holding positions max(0, P - window + 1) .. P for P = ctx + i."""
    P = ctx + i
    first = max(0, P - window + 1)
    base = ctx - window + 1
    return first - base, P - base + 1


def prefill_query(cfg: StepConfig, inp, i: int, key_vals: np.ndarray,
                  pooled_full: np.ndarray, with_attention: bool = True,
                  block_ids: Optional[np.ndarray] = None,
                  token_ids: Optional[np.ndarray] = None) -> dict:
    """The whole step for prefill query i.

    key_vals: decoded index keys of the chunk; pooled_full: decoded block keys
    of every complete block (pool_keys over all latents). A block that is only
    partly visible to this query is pooled here over its visible members."""
    n_vis = prefill_visible(inp.ctx, i, cfg.ratio)
    nb = -(-n_vis // cfg.block)
    pv = np.zeros((nb, key_vals.shape[-1]), np.float64)
    full = n_vis // cfg.block
    pv[:full] = pooled_full[:full]
    if n_vis % cfg.block:
        lastb = nb - 1
        mean = pool_mean_f32(key_vals[lastb * cfg.block: n_vis])
        d, s = store_f32(mean[None, :], inp.keys.fmt)
        pv[lastb] = decode_keys(inp.keys.fmt, d, s)[0]
    r = select_query(cfg, inp.q_idx[i], inp.w[i], key_vals, pv, n_vis, block_ids=block_ids)
    r["token_ids_used"] = r["token_ids"] if token_ids is None else np.asarray(token_ids)
    if with_attention:
        lo, hi = prefill_window_rows(inp.ctx, i, cfg.window)
        o, lse = attend_query(cfg, inp.q[i], inp.latents, r["token_ids_used"], inp.swa[lo:hi])
        r["out"], r["lse"] = o, lse
    return r


def prefill_caches(cfg: StepConfig, inp):
    """Decoded index keys and decoded complete-block keys of a prefill chunk."""
    n_lat = prefill_visible(inp.ctx, inp.n_q - 1, cfg.ratio)
    kv = decode_keys(inp.keys.fmt, inp.keys.data[:n_lat],
                     None if inp.keys.scales is None else inp.keys.scales[:n_lat])
    full = n_lat // cfg.block
    pdata, pscales = pool_keys(kv, full * cfg.block, inp.keys.fmt, cfg.block)
    return kv, decode_keys(inp.keys.fmt, pdata, pscales), (pdata, pscales)
