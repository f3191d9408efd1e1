"""bench.py host logic without a GPU: max-over-ranks timing with two gloo ranks, and the
reference arm's JSON line (the fp64 oracle on a bounded sample)."""
import json
import os
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    got = bench.max_over_ranks(1.5 + rank)  # rank 1 is the slowest
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 2.5, 1: 2.5}


def test_max_over_ranks_without_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25) == 3.25


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["higher_is_better"] is True


def test_bench_pair_counts_match_oracle():
    """bench.py counts the algorithmic work (allowed pairs) without the oracle; the counts agree
    with the oracle's brute-force count for every mask kind."""
    import bench
    import oracle
    from attention_attn_fwd_bwd_gb300 import inputs

    for N in (1, 100, 517, 1024):
        assert bench.allowed_pairs(N, "full") == oracle.allowed_pairs(N, oracle.Variant(mask=0))
        assert bench.allowed_pairs(N, "causal") == oracle.allowed_pairs(N, oracle.Variant(mask=1))
        for W in (1, 7, 300):
            for c in (False, True):
                assert bench.allowed_pairs(N, "window", causal=c, window=W) == oracle.allowed_pairs(
                    N, oracle.Variant(mask=2, window=W, causal=c))
        for blk in (64, 128):
            rp, ci = inputs.bigbird_csr(-(-N // blk), seed=3, n_random=2)
            for c in (False, True):
                assert bench.allowed_pairs(N, "block_sparse", causal=c, row_ptr=rp, col_idx=ci,
                                           blk=blk) == oracle.allowed_pairs(
                    N, oracle.Variant(mask=3, bs_block=blk, bs_row_ptr=rp, bs_col_idx=ci, causal=c))
