"""CPU tests of bench.py's host logic: the FLOP count, the max-over-ranks
reduction of the multi-process path (gloo, world size 2) and the oracle arm's
JSON line."""

import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from varlen_flashattention_backward_gb300 import workloads as wl  # noqa: E402


@pytest.mark.parametrize("cid", [10, 11, 12])
def test_feature_workload_pairs_match_the_oracle_window(cid):
    """The FLOP count of the feature workloads (outer split, bottom-right
    causal, explicit mask) against a brute-force count over the oracle's
    window and mask of every sequence."""
    import numpy as np
    import oracle
    w = wl.workload(cid)
    am = wl.make_atten_mask(w)
    want = 0
    for b, (lq, lk) in enumerate(zip(w.lens, w.lens_kv)):
        pre, nxt = oracle.mode_window(w.sparse_mode, w.pre_tokens, w.next_tokens, lq, lk)
        qs = w.q_start[b] if w.q_start else 0
        ks = w.kv_start[b] if w.kv_start else 0
        ok = oracle.window_allowed(lq, lk, pre, nxt, q_start=qs, kv_start=ks)
        if am is not None and w.sparse_mode in (0, 1, 4):
            ok &= am[:lq, :lk] == 0
        want += int(ok.sum())
    assert bench.workload_pairs(w, am) == want


def test_flop_count_matches_closed_forms():
    # causal: L (L + 1) / 2 pairs per head
    w2 = wl.workload(2)
    pairs = sum(L * (L + 1) // 2 for L in w2.lens)
    assert bench.allowed_pairs(w2.lens, w2.lens_kv, w2.pre_tokens, w2.next_tokens) == pairs
    assert bench.workload_flops(w2) == 10 * 128 * 16 * pairs == 59097743360
    # no mask: Lq * Lk
    w1 = wl.workload(1)
    assert bench.allowed_pairs(w1.lens, w1.lens_kv, w1.pre_tokens, w1.next_tokens) == 37 ** 2 + 64 ** 2
    # band pre=4096, next=0 on 16384 rows: sum_i min(i, 4096) + 1
    w5 = wl.workload(5)
    per_seq = sum(min(i, 4096) + 1 for i in range(16384))
    assert bench.allowed_pairs(w5.lens, w5.lens_kv, w5.pre_tokens, w5.next_tokens) == 4 * per_seq


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, _ = bench.dist_env()
    got = bench.max_over_ranks(10.0 + 5.0 * r, w)
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = 29500 + (os.getpid() % 2000)
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "1", "--steps", "1", "--warmup", "3", "--ref-budget", "0.2"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0
