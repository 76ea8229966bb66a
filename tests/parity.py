"""Helpers of the GPU parity tests: moving synthetic inputs to the device, running
the library through its C ABI, and comparing with the oracle.

Tolerances (the bar the step is held to):
  * ids: bit-exact, except that an id may differ where the oracle's k-th best
    score has a neighbour within 1e-5 relative (a near-tie);
  * pooled keys: bit-exact;
  * fp32 scores: within 1e-3 relative of the oracle's float64 scores;
  * bf16 outputs: max-abs error <= 2e-2, and (since the default-scale softmax
    is almost uniform, so an all-zero output would pass a max-abs bar) a
    relative RMS error <= 1e-2 and LSE within 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import two_tier_sparse_gb300 as dsa

NEAR_TIE = 1e-5
SCORE_RTOL = 1e-3
OUT_MAX_ABS = 2e-2
OUT_REL_RMS = 1e-2
LSE_ABS = 1e-3


def dev(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def pooled_buffer(fmt, B, blocks, device="cuda"):
    """Zeroed block-key cache [B, blocks, ...] in `fmt`. MXFP4 caches are read in
    pairs of rows, so their per-sequence row count is even."""
    if fmt == "bf16":
        return dsa.Keys(fmt, torch.zeros((B, blocks, 128), dtype=torch.int16, device=device))
    if fmt == "mxfp4":
        blocks += blocks & 1
    width = 64 if fmt == "mxfp4" else 128
    return dsa.Keys(fmt, torch.zeros((B, blocks, width), dtype=torch.uint8, device=device),
                    torch.zeros((B, blocks, 4), dtype=torch.uint8, device=device))


class DecodeOnDevice:
    """A DecodeInputs batch resident on the GPU, with its pooled-key buffers."""

    def __init__(self, inp, cfg, device="cuda"):
        self.inp = inp
        self.cfg = cfg
        B, cap = inp.B, inp.cap
        self.cap = cap
        self.q = dev(inp.q, device)
        self.q_idx = dev(inp.q_idx, device)
        self.w = dev(inp.w, device)
        self.latents = dev(inp.latents, device)
        self.swa = dev(inp.swa, device)
        self.n_lat = dev(inp.n_latents, device)
        self.swa_len = dev(inp.swa_len, device)
        fmt = inp.keys.fmt
        self.keys = dsa.Keys(fmt, dev(inp.keys.data, device),
                             None if inp.keys.scales is None else dev(inp.keys.scales, device))
        self.pooled = pooled_buffer(fmt, B, cap // 8, device)
        self.ws = dsa.workspace(cfg, B, cap, device)
        self.device = device

    def pool(self, tail_only=False):
        dsa.pool_index_keys(self.cfg, self.keys, self.n_lat, self.cap, self.pooled, self.ws,
                            tail_only=tail_only)

    def status(self):
        return dsa.read_device_status(self.ws)


def check_ids(gpu_ids, oracle_ids, score_of, k, label=""):
    """gpu_ids/oracle_ids: id arrays (ascending, -1 padded). score_of: id -> oracle
    float64 score. The two sets may differ only in ids whose score is within
    NEAR_TIE relative of the k-th best oracle score. Returns #near-tie swaps."""
    g = np.asarray(gpu_ids)
    o = np.asarray(oracle_ids)
    gv, ov = g[g >= 0], o[o >= 0]
    assert len(gv) == len(ov), f"{label}: {len(gv)} ids vs oracle {len(ov)}"
    assert (np.diff(gv) > 0).all(), f"{label}: ids not strictly ascending"
    assert (g[len(gv):] == -1).all(), f"{label}: padding is not -1"
    diff = set(gv.tolist()) ^ set(ov.tolist())
    if not diff:
        return 0
    kth = min(score_of(int(i)) for i in ov)
    bad = [i for i in diff if abs(score_of(int(i)) - kth) > NEAR_TIE * abs(kth)]
    assert not bad, f"{label}: ids differ beyond near-ties: {sorted(bad)[:8]} (kth={kth})"
    return len(diff) // 2


def check_scores(gpu, ref, label=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(gpu), fin), f"{label}: -inf pattern differs"
    err = np.abs(gpu[fin] - ref[fin])
    tol = SCORE_RTOL * np.maximum(np.abs(ref[fin]), 1e-30)
    # a score near zero from cancellation gets an absolute floor of 1e-3 of the row's scale
    scale = np.abs(ref[fin]).max() if fin.any() else 1.0
    ok = (err <= tol) | (err <= SCORE_RTOL * 1e-3 * scale)
    assert ok.all(), f"{label}: score error {err[~ok].max()} at {np.where(~ok)[0][:5]}"


def check_out(gpu_bits, lse_gpu, ref_out, ref_lse, label=""):
    got = O.bf16_to_f64(gpu_bits)
    err = np.abs(got - ref_out)
    assert err.max() <= OUT_MAX_ABS, f"{label}: max abs {err.max()}"
    den = np.sqrt((ref_out ** 2).mean())
    rel = np.sqrt((err ** 2).mean()) / max(den, 1e-30)
    assert rel <= OUT_REL_RMS, f"{label}: rel rms {rel}"
    if lse_gpu is not None:
        lerr = np.abs(np.asarray(lse_gpu, np.float64) - ref_lse)
        assert lerr.max() <= LSE_ABS, f"{label}: lse err {lerr.max()}"
