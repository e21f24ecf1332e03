"""Parity of the CUDA replay / verify kernels with the FP64 oracle.

Element by element on the same seeded inputs: outputs (rel-L2 <= 2e-3, per
item too), states (max|dS| <= 1e-4 max|S|), corrections (same bound),
key / gate records and every untouched page / record row bit-exact, the
status word clean.  Sizes span several items per CTA with a ragged tail;
the full-size workloads are compared on sampled items.
"""
import numpy as np
import pytest

from linear_attention_speculative_recoverssm_gb300 import synth
from oracle import kda_oracle as ko

import kda_testutil as tu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from linear_attention_speculative_recoverssm_gb300 import _build, _lib
    assert torch.cuda.is_available()
    _build.build()
    _lib.load()


def _run_and_compare(case, *, replay=True, boundary=False, split=1):
    before = tu.copy_case(case)
    d = tu.device_case(case)
    ref = tu.copy_case(case)
    tu.oracle_step(ref, replay=replay, boundary=boundary)
    tu.gpu_step(case, d, replay=replay, boundary=boundary, split=split)
    tu.compare_step(ref, d, before)
    return d, ref


# --------------------------------------------------------------------------
# the tiny case: every pending combination, a null slot, a missing record row
# --------------------------------------------------------------------------

@pytest.mark.parametrize("split", [1, 2, 4])
@pytest.mark.parametrize("n0", [0, 1, 2])
@pytest.mark.parametrize("n1", [0, 1, 2])
def test_tiny_every_pending_pair(n0, n1, split):
    case = synth.make("tiny-b2-h2-q2")
    case["pending"][case["record_rows"][0]] = n0
    case["pending"][case["record_rows"][1]] = n1
    _run_and_compare(case, split=split)


@pytest.mark.parametrize("split", [1, 2, 4])
def test_tiny_null_slot_and_missing_record(split):
    case = synth.make("tiny-b2-h2-q2")
    case["pending"][:] = 2
    case["state_slots"][0] = 0          # inert request: zeros, nothing else
    _run_and_compare(case, split=split)
    case = synth.make("tiny-b2-h2-q2")
    case["pending"][:] = 2
    case["record_rows"][1] = -1         # no record row: no replay, no records
    _run_and_compare(case, split=split)


# --------------------------------------------------------------------------
# several items per CTA, ragged tail, every window size
# --------------------------------------------------------------------------

@pytest.mark.parametrize("Q", [1, 2, 3, 4, 5, 6, 7, 8])
def test_replay_verify_every_window(Q):
    case = synth.replay_verify_case(B=40, H=8, Q=Q, slots=64, seed=100 + Q,
                                    padding_frac=0.1, no_record_frac=0.1)
    _run_and_compare(case, split=1)


@pytest.mark.parametrize("Q", [1, 2, 5, 8])
@pytest.mark.parametrize("split", [2, 4])
def test_replay_verify_cluster_split(Q, split):
    case = synth.replay_verify_case(B=6, H=4, Q=Q, slots=16, seed=200 + Q,
                                    padding_frac=0.2, no_record_frac=0.2)
    _run_and_compare(case, split=split)


def test_record_capacity_larger_than_window():
    # records hold RQ = 8 tokens, this window verifies Q = 3
    case = synth.replay_verify_case(B=20, H=4, Q=3, RQ=8, slots=32, seed=7)
    _run_and_compare(case, split=1)


@pytest.mark.parametrize("Q", [3, 8])
@pytest.mark.parametrize("split", [1, 2, 4])
def test_boundary_states(Q, split):
    case = synth.replay_verify_case(B=24, H=4, Q=Q, slots=64, seed=300 + Q,
                                    boundary_frac=0.5, padding_frac=0.1)
    case["pending"][:] = np.random.default_rng(Q).integers(0, Q + 1, case["pending"].shape)
    _run_and_compare(case, boundary=True, split=split)


# --------------------------------------------------------------------------
# the stock verify (checkpoint never written), FP32 and BF16 pools
# --------------------------------------------------------------------------

@pytest.mark.parametrize("Q", [1, 4, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_verify_only(Q, dtype):
    case = synth.replay_verify_case(B=30, H=6, Q=Q, slots=40, seed=400 + Q, state_dtype=dtype,
                                    padding_frac=0.1, no_record_frac=0.1)
    before = tu.copy_case(case)
    d = tu.device_case(case)
    ref = tu.copy_case(case)
    tu.oracle_step(ref, replay=False)
    tu.gpu_step(case, d, replay=False)
    np.testing.assert_array_equal(tu.to_numpy(d["state"]), before["state"])
    tu.compare_step(ref, d, before)


def test_verify_without_record_rows_uses_row_b():
    import torch
    from linear_attention_speculative_recoverssm_gb300 import kda_verify
    case = synth.replay_verify_case(B=12, H=2, Q=4, slots=20, seed=9)
    case["record_rows"] = np.arange(12, dtype=np.int32)
    ref = tu.copy_case(case)
    tu.oracle_step(ref, replay=False)
    d = tu.device_case(case)
    kda_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"], d["dt_bias"],
               d["state"], d["state_slots"], d["corr"], d["key_gate"], d["out"], Q=4,
               lower_bound=case["lower_bound"], q_scale=case["q_scale"], record_rows=None)
    torch.cuda.synchronize()
    tu.compare_step(ref, d, case)


# --------------------------------------------------------------------------
# protocol invariants on the GPU
# --------------------------------------------------------------------------

def test_fused_equals_commit_then_verify():
    import torch
    from linear_attention_speculative_recoverssm_gb300 import (KDA_STATE_F32, kda_commit,
                                                               layer_tables)
    case = synth.replay_verify_case(B=32, H=4, Q=4, slots=48, seed=11, no_record_frac=0.1)
    fused = tu.device_case(case)
    tu.gpu_step(case, fused, replay=True)
    split = tu.device_case(case)
    rows = split["record_rows"]
    lens = torch.where(rows >= 0, split["pending"][rows.clamp(min=0).long()],
                       torch.zeros_like(rows)).to(torch.int32)
    tabs = layer_tables([split["state"]], [split["corr"]], [split["key_gate"]], "cuda")
    kda_commit(*tabs, split["A_log"], split["dt_bias"], split["state_slots"], lens,
               split["state_slots"], state_dtype=KDA_STATE_F32, lower_bound=case["lower_bound"],
               L=1, H=case["H"], B=case["B"], Q=case["RQ"], n_slots=case["state"].shape[0],
               n_rows=case["corr"].shape[0], record_rows=split["record_rows"])
    tu.gpu_step(case, split, replay=False)
    torch.cuda.synchronize()
    tu.assert_state_close(tu.to_numpy(split["state"]), tu.to_numpy(fused["state"]))
    tu.assert_out_close(tu.to_numpy(split["out"]), tu.to_numpy(fused["out"]), Q=4)
    tu.assert_corr_close(tu.to_numpy(split["corr"]), tu.to_numpy(fused["corr"]))
    np.testing.assert_array_equal(tu.to_numpy(split["key_gate"]), tu.to_numpy(fused["key_gate"]))


def test_multi_step_decode_loop():
    """verify -> sample -> defer -> replay+verify -> ... over several steps,
    against the oracle running the same protocol."""
    import torch
    from linear_attention_speculative_recoverssm_gb300 import kda_defer_commit
    case = synth.replay_verify_case(B=16, H=4, Q=4, slots=24, seed=12, no_record_frac=0.1)
    case["pending"][:] = 0
    ref = tu.copy_case(case)
    d = tu.device_case(case)
    rng = np.random.default_rng(5)
    for step in range(4):
        fresh = synth.replay_verify_case(B=16, H=4, Q=4, slots=24, seed=1000 + step)
        for key in ("q", "k", "v", "raw_g", "raw_beta"):
            ref[key] = fresh[key]
            d[key] = tu.to_torch(fresh[key], "cuda")
        tu.oracle_step(ref, replay=True)
        tu.gpu_step(ref, d, replay=True)
        torch.cuda.synchronize()
        tu.assert_out_close(tu.to_numpy(d["out"]), ref["out"], Q=4, what=f"step {step} out")
        tu.assert_state_close(tu.to_numpy(d["state"]), ref["state"], what=f"step {step} state")
        accepted = rng.integers(0, 5, size=16).astype(np.int32)
        lens_ref = accepted.copy()
        ko.defer_commit(state_slots=ref["state_slots"], commit_lens=lens_ref,
                        record_rows=ref["record_rows"], pending=ref["pending"], B=16)
        lens = tu.to_torch(accepted, "cuda")
        kda_defer_commit(d["state_slots"], lens, d["record_rows"], d["pending"])
        torch.cuda.synchronize()
        np.testing.assert_array_equal(tu.to_numpy(d["pending"]), ref["pending"])
        np.testing.assert_array_equal(tu.to_numpy(lens), lens_ref)
        # keep the device state in lockstep with the oracle's rounding
        d["state"].copy_(tu.to_torch(ref["state"], "cuda"))
        d["corr"].copy_(tu.to_torch(ref["corr"], "cuda"))


def test_out_of_range_indices_are_reported_not_faulted():
    import torch
    case = synth.replay_verify_case(B=8, H=2, Q=2, slots=12, seed=13)
    n_slots = case["state"].shape[0]
    case["state_slots"][3] = n_slots + 5         # outside the pool
    case["record_rows"][5] = case["corr"].shape[0] + 2  # outside the records
    d = tu.device_case(case)
    tu.gpu_step(case, d, replay=True)
    torch.cuda.synchronize()
    from linear_attention_speculative_recoverssm_gb300 import KDA_ERR_ARG
    assert int(tu.to_numpy(d["status"])[0]) == KDA_ERR_ARG
    out = tu.to_numpy(d["out"]).reshape(8, 2, 2, 128)
    assert not out[3].any()  # treated as inert


def test_device_wait_that_runs_out_reports_timeout_and_context_survives():
    """A bounded device wait on a barrier nothing completes gives up and
    reports KDA_ERR_TIMEOUT; afterwards the same context still computes a
    step that matches the oracle."""
    import time
    import torch
    from linear_attention_speculative_recoverssm_gb300 import (KDA_ERR_TIMEOUT,
                                                               kda_selftest_wait_timeout)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    kda_selftest_wait_timeout(status)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) == KDA_ERR_TIMEOUT
    assert 0.5 < waited < 30.0  # the wait limit, not an instant return or a hang
    case = synth.replay_verify_case(B=4, H=2, Q=3, slots=8, seed=31)
    _run_and_compare(case, split=1)


def test_empty_batch_is_a_noop():
    import torch
    from linear_attention_speculative_recoverssm_gb300 import kda_replay_verify
    case = synth.replay_verify_case(B=4, H=2, Q=2, slots=8, seed=14)
    d = tu.device_case(case)
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    assert kda_replay_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"],
                             d["dt_bias"], d["state"], empty, empty, d["pending"], d["corr"],
                             d["key_gate"], d["out"], Q=2, lower_bound=-5.0,
                             q_scale=0.088) == 0


# --------------------------------------------------------------------------
# the full-size workloads, in the launch configuration the benchmark times,
# on sampled items
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["replay-verify-f32-h32-b128-q4", "replay-verify-f32-h64-b512-q8"])
def test_full_size_sampled(name):
    import torch
    case = synth.make(name)
    B, H, Q = case["B"], case["H"], case["Q"]
    rng = np.random.default_rng(99)
    items = np.sort(rng.choice(B * H, size=192, replace=False))
    d = tu.device_case(case)
    tu.gpu_step(case, d, replay=True, split=1)
    torch.cuda.synchronize()
    assert int(tu.to_numpy(d["status"])[0]) == 0
    # oracle on the sampled items only (host arrays still hold the inputs)
    before_pages = {}
    for i in items:
        b, h = divmod(int(i), H)
        s = int(case["state_slots"][b])
        if s > 0:
            before_pages[(s, h)] = case["state"][s, h].copy()
    out = np.zeros(case["v"].shape, dtype=np.uint16)
    ko.replay_verify(q=case["q"], k=case["k"], v=case["v"], raw_g=case["raw_g"],
                     raw_beta=case["raw_beta"], A_log=case["A_log"], dt_bias=case["dt_bias"],
                     lower_bound=case["lower_bound"], q_scale=case["q_scale"],
                     state=case["state"], state_slots=case["state_slots"],
                     record_rows=case["record_rows"], corr=case["corr"],
                     key_gate=case["key_gate"], out=out, B=B, H=H, Q=Q,
                     pending=case["pending"], items=items)
    got_out = tu.to_numpy(d["out"]).reshape(B, Q, H, 128)
    ref_out = out.reshape(B, Q, H, 128)
    for i in items:
        b, h = divmod(int(i), H)
        tu.assert_out_close(got_out[b, :, h], ref_out[b, :, h], what=f"item {i}")
        s = int(case["state_slots"][b])
        if s > 0:
            tu.assert_state_close(tu.to_numpy(d["state"][s, h]), case["state"][s, h],
                                  what=f"item {i} state")
            r = int(case["record_rows"][b])
            if r >= 0:
                tu.assert_corr_close(tu.to_numpy(d["corr"][r, h, :Q]), case["corr"][r, h, :Q],
                                     what=f"item {i} corr")
                np.testing.assert_array_equal(tu.to_numpy(d["key_gate"][r, h, :Q]),
                                              case["key_gate"][r, h, :Q])
        else:
            assert not got_out[b, :, h].any()


# --------------------------------------------------------------------------
# degenerate and extreme cases
# --------------------------------------------------------------------------

def test_every_request_inert():
    """A batch whose every slot is the null slot: zero outputs, nothing else
    written (pool, records and pending bit-identical)."""
    case = synth.replay_verify_case(B=12, H=3, Q=4, slots=16, seed=41)
    case["state_slots"][:] = case["null_slot"]
    d, _ = _run_and_compare(case, split=1)
    assert not tu.to_numpy(d["out"]).any()


@pytest.mark.parametrize("fill", ["zero", "max"])
def test_pending_all_zero_or_all_full(fill):
    """Every request with nothing to replay (the checkpoint must stay
    bit-identical) or with the full record capacity pending."""
    case = synth.replay_verify_case(B=24, H=4, Q=8, slots=32, seed=43 if fill == "zero" else 44)
    case["pending"][:] = 0 if fill == "zero" else case["RQ"]
    _run_and_compare(case, split=1)


@pytest.mark.parametrize("B,H,Q", [(3, 4, 2), (1, 1, 8), (7, 3, 5)])
def test_fewer_items_than_sms_whole_items(B, H, Q):
    """Persistent CTAs with fewer items than SMs (one item per CTA, the rest
    idle), odd head counts, a single head."""
    case = synth.replay_verify_case(B=B, H=H, Q=Q, slots=B + 4, seed=50 + B * 10 + H)
    _run_and_compare(case, split=1)


@pytest.mark.parametrize("H", [128, 100])
def test_many_heads(H):
    """Many heads on few requests: the item index is split into request and
    head by a multiply and shifts (H = 100 is not a power of two), and the
    pages of one slot span H * 64 KB."""
    case = synth.replay_verify_case(B=3, H=H, Q=8, slots=7, seed=70 + H, padding_frac=0.0,
                                    no_record_frac=0.0)
    _run_and_compare(case, split=1)


@pytest.mark.parametrize("lower_bound", [-10.0, 0.0])
def test_gate_bound_extremes(lower_bound):
    """At the largest supported |lower_bound| the decay products over the
    window span e^-80 (1/Gamma stays finite in FP32); at 0 there is no decay
    (the plain delta rule)."""
    case = synth.replay_verify_case(B=16, H=4, Q=8, slots=24, seed=61)
    case["lower_bound"] = lower_bound
    _run_and_compare(case, split=1)


def test_mostly_inert_back_to_back():
    """Half the requests inert, twenty launches back to back.  Each main warp
    waits for an inert item's stage phase before counting its read of the
    stage, so the read counts of two items sharing a stage never mix (a
    mixed count would issue a page twice or never: a device fault or a
    timeout).  Nothing is pending, so every launch computes the same step."""
    import torch
    case = synth.replay_verify_case(B=192, H=16, Q=8, slots=200, seed=61, padding_frac=0.5)
    case["pending"][:] = 0
    before = tu.copy_case(case)
    ref = tu.copy_case(case)
    tu.oracle_step(ref, replay=True)
    d = tu.device_case(case)
    for _ in range(20):
        tu.gpu_step(case, d, replay=True, split=1)
    torch.cuda.synchronize()
    tu.compare_step(ref, d, before)


# --------------------------------------------------------------------------
# the latency sweep's own shapes: H = 32, B in {1, 4, 16}, q in {1, 2, 4, 8},
# split in {1, 2, 4} and the automatic choice, every item against the oracle
# --------------------------------------------------------------------------

_LATENCY_REF = {}


def _latency_ref(B, Q):
    """The oracle's result for one latency-sweep shape (computed once and
    shared by its four launch shapes)."""
    if (B, Q) not in _LATENCY_REF:
        case = synth.latency_case(B=B, Q=Q)
        ref = tu.copy_case(case)
        tu.oracle_step(ref, replay=True)
        _LATENCY_REF[(B, Q)] = (case, ref)
    return _LATENCY_REF[(B, Q)]


@pytest.mark.parametrize("split", [1, 2, 4, 0])
@pytest.mark.parametrize("Q", [1, 2, 4, 8])
@pytest.mark.parametrize("B", [1, 4, 16])
def test_latency_sweep_shapes(B, Q, split):
    case, ref = _latency_ref(B, Q)
    assert case["H"] == 32 and case["Q"] == Q and case["B"] == B
    before = tu.copy_case(case)
    d = tu.device_case(case)
    tu.gpu_step(case, d, replay=True, split=split)
    tu.compare_step(ref, d, before)


# --------------------------------------------------------------------------
# numerically extreme gates
# --------------------------------------------------------------------------

@pytest.mark.parametrize("split", [1, 2, 4])
def test_boundary_states_at_the_gate_bound(split):
    """lower_bound = -10 with boundary states: the boundary state is the
    partial replay sum divided by prod_{m<=s<n} d_s, which reaches e^70 over
    seven decays while S_0 D_n falls to ~1e-36; every request replays a full
    record (n = Q = 8), with boundaries after 1..7 tokens."""
    case = synth.replay_verify_case(B=24, H=4, Q=8, slots=64, seed=330 + split,
                                    boundary_frac=0.5, padding_frac=0.1)
    case["lower_bound"] = -10.0
    case["pending"][:] = 8
    # saturate the recorded gates towards the strongest decay
    kg = case["key_gate"]
    kg[..., 128:] = synth.to_bf16_bits(np.full(kg[..., 128:].shape, 30.0, np.float32))
    _run_and_compare(case, boundary=True, split=split)


@pytest.mark.parametrize("split", [1, 4])
def test_saturating_gates_and_beta(split):
    """Raw gates and raw betas with |exp(A_log) (raw_g + dt_bias)| and
    |raw_beta| around 100: the kernels' sigmoid 1 / (1 + e^-z) overflows its
    exponential to +inf (giving 0) or underflows it to 0 (giving 1)."""
    case = synth.replay_verify_case(B=16, H=4, Q=8, slots=24, seed=340 + split)
    rng = np.random.default_rng(341)
    a = np.exp(case["A_log"].astype(np.float64))[None, :, None]
    sign = np.where(rng.random(case["raw_g"].shape) < 0.5, -1.0, 1.0)
    g = sign * rng.uniform(90.0, 110.0, size=case["raw_g"].shape) / a
    case["raw_g"] = synth.to_bf16_bits(g.astype(np.float32))
    kg = case["key_gate"]
    sign = np.where(rng.random(kg[..., 128:].shape) < 0.5, -1.0, 1.0)
    g = sign * rng.uniform(90.0, 110.0, size=kg[..., 128:].shape) / a[:, :, None]
    kg[..., 128:] = synth.to_bf16_bits(g.astype(np.float32))
    sign = np.where(rng.random(case["raw_beta"].shape) < 0.5, -1.0, 1.0)
    case["raw_beta"] = synth.to_bf16_bits(
        (sign * rng.uniform(90.0, 110.0, size=case["raw_beta"].shape)).astype(np.float32))
    _run_and_compare(case, split=split)
