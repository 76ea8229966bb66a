"""The bench's flop accounting for a prefill chunk, against counts made by hand, and its CPU legs."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_algorithmic_prefill_flops_small_chunk():
    # 3 queries at positions 20, 21, 22, ratio 1: 21..23 visible latents in 3 blocks;
    # k_blocks 2 keeps 2 blocks = 16 tokens; k_tokens 4, window 5 -> 9 attention rows.
    # Per query: scores 2*16*128 flop per key over 3 blocks + 16 tokens, and
    # QK^T + PV 2*2*64*512 flop per row.
    per_query = 2 * 16 * 128 * (3 + 16) + 2 * 2 * 64 * 512 * 9
    assert bench.prefill_flops(3, 20, 1, k_blocks=2, k_tokens=4, window=5) == 3 * per_query


def test_executed_prefill_flops_small_chunk():
    # 23 latents: 2 complete blocks (one 128-row block tile) and 24 latent columns
    # (one token tile) for the single group of 16 queries; each MMA tile is
    # 2*128*256*128 flop. Attention rows 42, 44, 46 round up to one 64-row
    # tile each, at 2*128*512 (QK^T, M=128) + 2*512*64 (PV) flop per row.
    scans = 2 * (2 * 128 * 256 * 128)
    attn = 3 * 64 * (2 * 128 * 512 + 2 * 512 * 64)
    assert bench.prefill_executed_flops(3, 20, 1) == scans + attn


def test_executed_covers_algorithmic_at_the_prefill_workload():
    a = bench.prefill_flops(4096, 65536, 2)
    e = bench.prefill_executed_flops(4096, 65536, 2)
    assert 689e9 < a < 690e9
    assert a < e < 2 * a


def test_prefill_cpu_leg_runs_on_a_spread_sample():
    qps, t, threads, sample = bench.cpu_oracle_prefill_rate("prefill_q4096_ctx65536_r2_bf16", 3)
    assert qps > 0 and t > 0 and threads >= 1
    assert sample.startswith("3 of the chunk's 4096 queries")


def test_profile_summaries_name_commands_the_bench_accepts():
    """Every summary under profiles/ gives the command that made it; each bench
    command there parses with the bench's own arguments and names a workload
    that exists."""
    import glob
    import re
    import shlex

    import synth
    cmds = set()
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        text = open(path).read()
        found = re.findall(r"python bench\.py[^`|\n]*", text)
        assert found or "ncu" not in text, f"{path} names no bench command"
        cmds.update(c.strip() for c in found)
    assert cmds
    for c in cmds:
        argv = shlex.split(c)[2:]
        old = sys.argv
        sys.argv = ["bench.py"] + argv
        try:
            args = bench.parse()
        finally:
            sys.argv = old
        assert args.workload in synth.WORKLOADS, c
