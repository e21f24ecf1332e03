"""The benchmark's host-side pieces that need no GPU: the oracle worker
pool behind the CPU baseline (forked before any CUDA call, one worker per
core) times the same items as the one-core loop."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from linear_attention_speculative_recoverssm_gb300 import synth  # noqa: E402


def test_oracle_pool_covers_the_workload():
    case = synth.make("tiny-b2-h2-q2")
    before = case["state"].copy()
    pool = bench.OraclePool(case, workers=2)
    try:
        rate, done, wall = pool.rate(30.0)
    finally:
        pool.close()
    live = int((case["state_slots"] > case["null_slot"]).sum()) * case["H"]
    assert done == live          # every live item, split over the workers
    assert rate > 0 and wall > 0
    assert (case["state"] == before).all()  # the parent's workload is untouched
