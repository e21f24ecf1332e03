"""Windows of different lengths (query_start_loc) on the GPU against the
FP64 oracle: per request a window of q_b = 0..Q tokens packed one request
after another, the last one ending at the activations' end (so the tensor
copies of the final windows run past it).  Outputs (rel-L2 <= 2e-3 overall
and per (request, head) window), states, corrections and key / gate records
are compared; every record row past a window, every untouched page, is
checked bit-exact."""
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


def _oracle(case, qsl, replay):
    out = np.zeros(case["v"].shape, dtype=np.uint16)
    ko.replay_verify(q=case["q"], k=case["k"], v=case["v"], raw_g=case["raw_g"],
                     raw_beta=case["raw_beta"], A_log=case["A_log"], dt_bias=case["dt_bias"],
                     lower_bound=case["lower_bound"], q_scale=case["q_scale"],
                     state=case["state"], state_slots=case["state_slots"],
                     record_rows=case["record_rows"], corr=case["corr"],
                     key_gate=case["key_gate"], out=out, B=case["B"], H=case["H"], Q=case["Q"],
                     pending=case["pending"] if replay else None, query_start_loc=qsl)
    case["out"] = out


def _gpu(case, d, qsl, replay, split):
    from linear_attention_speculative_recoverssm_gb300 import kda_replay_verify, kda_verify
    common = dict(Q=case["Q"], lower_bound=case["lower_bound"], q_scale=case["q_scale"],
                  status=d["status"], query_start_loc=qsl)
    if replay:
        kda_replay_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"],
                          d["dt_bias"], d["state"], d["state_slots"], d["record_rows"],
                          d["pending"], d["corr"], d["key_gate"], d["out"], split=split,
                          **common)
    else:
        kda_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"], d["dt_bias"],
                   d["state"], d["state_slots"], d["corr"], d["key_gate"], d["out"],
                   record_rows=d["record_rows"], **common)


def _compare(ref, d, before, qsl, status=0):
    got_out = tu.to_numpy(d["out"])
    tu.assert_out_close(got_out, ref["out"])
    H = ref["H"]
    for b in range(ref["B"]):
        rows = slice(int(qsl[b]), int(qsl[b + 1]))
        for h in range(H):
            tu.assert_out_close(got_out[rows, h], ref["out"][rows, h], what=f"request {b} head {h}")
    got_state = tu.to_numpy(d["state"])
    changed = np.any(ref["state"] != before["state"], axis=(2, 3))
    np.testing.assert_array_equal(got_state[~changed], before["state"][~changed])
    if changed.any():
        if ref["state"].dtype == np.uint16:
            tu.assert_bf16_state_close(got_state[changed], ref["state"][changed])
        else:
            tu.assert_state_close(got_state[changed], ref["state"][changed])
    got_corr = tu.to_numpy(d["corr"])
    tu.assert_corr_close(got_corr, ref["corr"])
    kept = ref["corr"] == before["corr"]
    np.testing.assert_array_equal(got_corr[kept], before["corr"][kept],
                                  err_msg="records past the windows")
    np.testing.assert_array_equal(tu.to_numpy(d["key_gate"]), ref["key_gate"])
    assert int(tu.to_numpy(d["status"])[0]) == status


@pytest.mark.parametrize("Q,B,H,split,replay,state_dtype", [
    (8, 40, 3, 1, True, "f32"),
    (3, 33, 4, 1, True, "f32"),
    (1, 20, 2, 1, True, "f32"),
    (5, 6, 2, 2, True, "f32"),
    (8, 3, 3, 4, True, "f32"),
    (4, 30, 2, 1, False, "f32"),
    (8, 17, 4, 1, False, "bf16"),
])
def test_varlen_matches_oracle(Q, B, H, split, replay, state_dtype):
    import torch
    case = synth.varlen_case(B=B, H=H, Q=Q, slots=2 * B + 4, seed=300 + 10 * Q + B,
                             padding_frac=0.1, no_record_frac=0.1, state_dtype=state_dtype)
    q_lens = case["q_lens"]
    assert (q_lens == 0).any() or Q == 1 or B < 8
    before = tu.copy_case(case)
    ref = tu.copy_case(case)
    qsl = case["query_start_loc"]
    _oracle(ref, qsl, replay)
    d = tu.device_case(case)
    _gpu(case, d, tu.to_torch(qsl, "cuda"), replay, split)
    torch.cuda.synchronize()
    _compare(ref, d, before, qsl)


def test_varlen_invalid_windows_are_reported_and_skipped():
    import torch
    from linear_attention_speculative_recoverssm_gb300 import KDA_ERR_ARG
    case = synth.varlen_case(B=12, H=2, Q=4, slots=30, seed=77, q_min=1)
    qsl = case["query_start_loc"].copy()
    qsl[3] = qsl[4] - 5                  # request 3: five tokens in a 4-token window
    qsl[12] = case["q"].shape[0] + 2     # request 11: past the activations
    before = tu.copy_case(case)
    ref = tu.copy_case(case)
    _oracle(ref, qsl, True)
    d = tu.device_case(case)
    _gpu(case, d, tu.to_torch(qsl, "cuda"), True, 1)
    torch.cuda.synchronize()
    for b in (3, 11):
        slot, rec = int(case["state_slots"][b]), int(case["record_rows"][b])
        np.testing.assert_array_equal(tu.to_numpy(d["state"][slot]), before["state"][slot])
        if rec >= 0:
            np.testing.assert_array_equal(tu.to_numpy(d["corr"][rec]), before["corr"][rec])
    # outputs: compare the valid requests' windows only (moving request 3's
    # start also moves request 2's end)
    n_tok = case["q"].shape[0]
    got_out = tu.to_numpy(d["out"])
    for b in range(12):
        if not (0 <= qsl[b] <= qsl[b + 1] <= n_tok and qsl[b + 1] - qsl[b] <= 4):
            assert b in (2, 3, 11)
            continue
        rows = slice(int(qsl[b]), int(qsl[b + 1]))
        tu.assert_out_close(got_out[rows], ref["out"][rows], what=f"request {b}")
    assert int(tu.to_numpy(d["status"])[0]) == KDA_ERR_ARG


def test_varlen_full_size_sampled():
    """The varlen benchmark workload (H=64, B=512, windows of 1..8 tokens) in
    the benchmark's launch configuration, on sampled items."""
    import torch
    case = synth.make("replay-verify-varlen-f32-h64-b512-q8")
    B, H = case["B"], case["H"]
    qsl = case["query_start_loc"]
    rng = np.random.default_rng(98)
    items = np.sort(rng.choice(B * H, size=160, replace=False))
    d = tu.device_case(case)
    _gpu(case, d, tu.to_torch(qsl, "cuda"), True, 0)
    torch.cuda.synchronize()
    assert int(tu.to_numpy(d["status"])[0]) == 0
    out = np.zeros(case["v"].shape, dtype=np.uint16)
    ko.replay_verify(q=case["q"], k=case["k"], v=case["v"], raw_g=case["raw_g"],
                     raw_beta=case["raw_beta"], A_log=case["A_log"], dt_bias=case["dt_bias"],
                     lower_bound=case["lower_bound"], q_scale=case["q_scale"],
                     state=case["state"], state_slots=case["state_slots"],
                     record_rows=case["record_rows"], corr=case["corr"],
                     key_gate=case["key_gate"], out=out, B=B, H=H, Q=case["Q"],
                     pending=case["pending"], items=items, query_start_loc=qsl)
    got_out = tu.to_numpy(d["out"])
    for i in items:
        b, h = divmod(int(i), H)
        rows = slice(int(qsl[b]), int(qsl[b + 1]))
        tu.assert_out_close(got_out[rows, h], out[rows, h], what=f"item {i}")
        s = int(case["state_slots"][b])
        if s > 0:
            tu.assert_state_close(tu.to_numpy(d["state"][s, h]), case["state"][s, h],
                                  what=f"item {i} state")
            r = int(case["record_rows"][b])
            qb = int(case["q_lens"][b])
            if r >= 0:
                tu.assert_corr_close(tu.to_numpy(d["corr"][r, h, :qb]), case["corr"][r, h, :qb])
                np.testing.assert_array_equal(tu.to_numpy(d["key_gate"][r, h, :qb]),
                                              case["key_gate"][r, h, :qb])


def test_varlen_mostly_inert_back_to_back():
    """Windows from query_start_loc, half the requests inert, twenty launches
    back to back (nothing pending: every launch computes the same step)."""
    import torch
    case = synth.varlen_case(B=192, H=16, Q=8, slots=200, seed=63, padding_frac=0.5)
    case["pending"][:] = 0
    qsl = case["query_start_loc"]
    before = tu.copy_case(case)
    ref = tu.copy_case(case)
    _oracle(ref, qsl, True)
    d = tu.device_case(case)
    dq = tu.to_torch(qsl, "cuda")
    for _ in range(20):
        _gpu(case, d, dq, True, 1)
    torch.cuda.synchronize()
    _compare(ref, d, before, qsl)
