"""Pins of the oracle's indexer scores and both selection tiers.

Indexer and candidate stage: recipes.vllm.ai "DeepSeek-V4.1-Flash", Overview,
bullet "Two-tier sparse attention" (keep the best 512 latents per query after a
candidate stage of 2048 blocks of 8); miles.radixark.com "DeepSeek-V4.1 Flash",
§1 "Sparse retrieval" (top-512 candidate set, coarser candidate-block pass).
Formula fixed by this build: score = sum_h w_h * ReLU(q_h . k); block key =
mean of the block's keys; ties to the lower index.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_scores(q, w, keys):
    out = []
    for k in keys:
        s = 0.0
        for h in range(len(q)):
            d = 0.0
            for j in range(len(k)):
                d += float(q[h][j]) * float(k[j])
            s += float(w[h]) * (d if d > 0 else 0.0)
        out.append(s)
    return np.array(out)


def test_scores_golden():
    g = json.load(open(os.path.join(GOLDEN, "indexer_tiny.json")))
    s = O.index_scores(np.array(g["q"]), np.array(g["w"]), np.array(g["keys"]))
    assert np.array_equal(s, np.array(g["scores"]))
    for k, ids in g["topk"].items():
        assert list(O.topk_ids(s, np.arange(4), int(k))) == ids


def test_scores_brute_force():
    rng = np.random.default_rng(10)
    q, w, keys = rng.standard_normal((3, 5)), rng.uniform(0, 1, 3), rng.standard_normal((7, 5))
    assert np.allclose(O.index_scores(q, w, keys), brute_scores(q, w, keys), rtol=1e-13,
                       atol=1e-15)


def test_scores_special_cases():
    rng = np.random.default_rng(11)
    q, keys = rng.standard_normal((1, 6)), rng.standard_normal((9, 6))
    # one head with weight 1: plain ReLU of the dot product
    assert np.allclose(O.index_scores(q, np.ones(1), keys), np.maximum(keys @ q[0], 0.0))
    # weights 0: every score is 0, so the selection is the lowest indices
    q16 = rng.standard_normal((16, 6))
    s = O.index_scores(q16, np.zeros(16), keys)
    assert (s == 0).all()
    assert list(O.topk_ids(s, np.arange(9), 4)) == [0, 1, 2, 3]
    # scaling every weight by 2 doubles the scores and keeps the selection
    w = rng.uniform(0, 1, 16)
    s1, s2 = O.index_scores(q16, w, keys), O.index_scores(q16, 2 * w, keys)
    assert np.array_equal(2 * s1, s2)
    assert np.array_equal(O.topk_ids(s1, np.arange(9), 5), O.topk_ids(s2, np.arange(9), 5))


def _beats(a, b):
    """Candidate a = (score, id) ranks before b."""
    return a[0] > b[0] or (a[0] == b[0] and a[1] < b[1])


@pytest.mark.parametrize("n", range(0, 10))
def test_topk_exhaustive_subsets(n):
    rng = np.random.default_rng(100 + n)
    # few distinct values so ties are common
    scores = rng.integers(0, 3, n).astype(np.float64)
    ids = rng.permutation(50)[:n]
    cands = [(float(O.rank_key(scores)[i]), int(ids[i])) for i in range(n)]
    for k in range(0, n + 2):
        got = O.topk_ids(scores, ids, k)
        kk = min(k, n)
        winners = []
        for sub in itertools.combinations(range(n), kk):
            rest = [c for i, c in enumerate(cands) if i not in sub]
            if all(_beats(cands[i], r) for i in sub for r in rest):
                winners.append(sorted(cands[i][1] for i in sub))
        assert len(winners) == 1
        assert list(got[:kk]) == winners[0]
        assert (got[kk:] == -1).all() and len(got) == k


def test_topk_invariants_large():
    rng = np.random.default_rng(12)
    s = rng.standard_normal(5000)
    ids = np.arange(5000)
    got = O.topk_ids(s, ids, 512)
    assert (np.diff(got) > 0).all()
    sel = np.zeros(5000, bool)
    sel[got] = True
    assert s[sel].min() >= s[~sel].max()


def test_topk_all_equal_and_fp32_ties():
    assert list(O.topk_ids(np.ones(10), np.arange(10), 4)) == [0, 1, 2, 3]
    # two fp64 scores that round to the same fp32 value tie; the lower id wins
    a = 1.0
    b = 1.0 + 2.0 ** -30
    assert np.float32(a) == np.float32(b)
    assert list(O.topk_ids(np.array([a, b]), np.array([7, 3]), 1)) == [3]
    # -0 equals +0
    assert list(O.topk_ids(np.array([0.0, -0.0]), np.array([5, 2]), 1)) == [2]


# --- two tiers ---------------------------------------------------------------


def _tiny_keys(rng, n, d=128):
    return O.bf16_to_f64(O.f32_to_bf16_rne(
        (rng.standard_normal((n, d)) / np.sqrt(d)).astype(np.float32)))


def _query(rng):
    qi = O.f32_to_bf16_rne((rng.standard_normal((16, 128)) / np.sqrt(128)).astype(np.float32))
    w = rng.uniform(0, 1, 16).astype(np.float32)
    return qi, w


def brute_two_tier(qi_bits, w, kv, n_vis, k_blocks, k_tokens, block=8):
    """Two tiers by plain loops: block means (fp32, member order), scores,
    sort by (score desc, id asc), candidates, token scores, sort, ascending ids."""
    q = O.bf16_to_f64(qi_bits)
    nb = -(-n_vis // block)
    bkeys = []
    for b in range(nb):
        mem = kv[b * block: min((b + 1) * block, n_vis)].astype(np.float32)
        acc = mem[0].copy()
        for m in mem[1:]:
            acc = (acc + m).astype(np.float32)
        mean = (acc / np.float32(len(mem))).astype(np.float32)
        bkeys.append(O.bf16_to_f64(O.f32_to_bf16_rne(mean)))
    bs = brute_scores(q, w, bkeys)
    border = sorted(range(nb), key=lambda b: (-np.float32(bs[b]), b))
    kept = sorted(border[:k_blocks]) if nb > k_blocks else list(range(nb))
    cand = [t for b in kept for t in range(b * block, min((b + 1) * block, n_vis))]
    ts = brute_scores(q, w, kv[cand])
    torder = sorted(range(len(cand)), key=lambda i: (-np.float32(ts[i]), cand[i]))
    ids = sorted(cand[i] for i in torder[:k_tokens])
    return kept, ids + [-1] * (k_tokens - len(ids))


@pytest.mark.parametrize("n_vis,k_blocks,k_tokens", [(61, 3, 10), (64, 8, 17), (9, 1, 20),
                                                     (40, 16, 7), (1, 4, 4)])
def test_two_tier_brute_force(n_vis, k_blocks, k_tokens):
    rng = np.random.default_rng(n_vis * 31 + k_blocks)
    kv = _tiny_keys(rng, n_vis)
    qi, w = _query(rng)
    cfg = O.StepConfig(k_blocks=k_blocks, k_tokens=k_tokens)
    pd, _ = O.pool_keys(kv, n_vis, "bf16")
    r = O.select_query(cfg, qi, w, kv, O.bf16_to_f64(pd), n_vis)
    kept, ids = brute_two_tier(qi, w, kv, n_vis, k_blocks, k_tokens)
    got_blocks = [int(b) for b in r["block_ids"] if b >= 0]
    assert got_blocks == kept
    assert list(r["token_ids"]) == ids


def test_block_stage_identity_when_few_blocks():
    rng = np.random.default_rng(13)
    n_vis = 2048
    kv = _tiny_keys(rng, n_vis)
    qi, w = _query(rng)
    cfg = O.StepConfig(k_blocks=2048, k_tokens=512)
    pd, _ = O.pool_keys(kv, n_vis, "bf16")
    r = O.select_query(cfg, qi, w, kv, O.bf16_to_f64(pd), n_vis)
    assert list(r["block_ids"][:256]) == list(range(256))
    assert (r["block_ids"][256:] == -1).all()
    # ... and then the token tier is single-tier top-512 over every latent
    single = O.topk_ids(O.index_scores(O.bf16_to_f64(qi), w, kv), np.arange(n_vis), 512)
    assert np.array_equal(r["token_ids"], single)


def test_block_permutation_permutes_ids():
    rng = np.random.default_rng(14)
    n_vis, nb = 96, 12
    kv = _tiny_keys(rng, n_vis)
    qi, w = _query(rng)
    cfg = O.StepConfig(k_blocks=5, k_tokens=20)
    perm = rng.permutation(nb)                  # new block j holds old block perm[j]
    kvp = kv.reshape(nb, 8, -1)[perm].reshape(n_vis, -1)
    res = []
    for k in (kv, kvp):
        pd, _ = O.pool_keys(k, n_vis, "bf16")
        res.append(O.select_query(cfg, qi, w, k, O.bf16_to_f64(pd), n_vis))
    inv = np.argsort(perm)                      # old block b sits at inv[b]
    mapped = sorted(int(inv[t // 8] * 8 + t % 8) for t in res[0]["token_ids"])
    assert mapped == list(res[1]["token_ids"])
