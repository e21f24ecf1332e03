"""kda_layer_step_noalloc, the layer step for callers that cannot allocate.

A serving runtime that reserves all device memory in its own pool, or a
plugin whose host framework owns every device allocation, cannot call
cudaMalloc on the decode path, so it cannot hand kda_layer_step a workspace.
kda_layer_step_noalloc puts the step's operands in the library's own fixed
device array instead.  These tests call it through the C ABI and check it
against kda_layer_step (workspace from the caller) on identical copies of a
layer workload, on two calls in a row (the second starting from what the
first left in the pools, records and windows), within the tolerances the
other GPU tests use; that a call beyond the array is refused with
KDA_ERR_SCRATCH; and that a call takes no device memory.

This file is collected last, so that a run stopping at its first failure
has run every other test before these.
"""
import numpy as np
import pytest

from linear_attention_speculative_recoverssm_gb300 import synth

import kda_testutil as tu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from linear_attention_speculative_recoverssm_gb300 import _build, _lib
    assert torch.cuda.is_available()
    _build.build()
    _lib.load()


LAYER_KEYS = ("x", "conv_weight", "conv_bias", "conv_state", "f_a", "f_b", "gate", "norm_weight",
              "raw_beta", "A_log", "dt_bias", "state", "state_slots", "record_rows", "pending",
              "corr", "key_gate")


def _device(case):
    import torch
    d = {key: tu.to_torch(case[key], "cuda") for key in LAYER_KEYS}
    d["out"] = torch.zeros((case["B"] * case["Q"], case["H"] * 128), dtype=torch.bfloat16,
                           device="cuda")
    d["status"] = torch.zeros(1, dtype=torch.int32, device="cuda")
    return d


def _args(d):
    return (d["x"], d["conv_weight"], d["conv_bias"], d["conv_state"], d["f_a"], d["f_b"],
            d["raw_beta"], d["A_log"], d["dt_bias"], d["state"], d["state_slots"],
            d["record_rows"], d["pending"], d["corr"], d["key_gate"], d["gate"],
            d["norm_weight"], d["out"])


def _with_workspace(case, d, workspace):
    from linear_attention_speculative_recoverssm_gb300 import kda_layer_step
    kda_layer_step(*_args(d), workspace, Q=case["Q"], lower_bound=case["lower_bound"],
                   q_scale=case["q_scale"], eps=case["eps"], status=d["status"])


def _without_workspace(case, d):
    from linear_attention_speculative_recoverssm_gb300 import kda_layer_step_noalloc
    kda_layer_step_noalloc(*_args(d), Q=case["Q"], lower_bound=case["lower_bound"],
                           q_scale=case["q_scale"], eps=case["eps"], status=d["status"])


def _same_results(got, want, Q):
    """The no-alloc call's results against the workspace call's, within the
    parity tolerances: outputs rel-L2 <= 2e-3 overall and per item, states
    and corrections max|d| <= 1e-4 max, records and windows bit-exact."""
    T, D = want["out"].shape
    tu.assert_out_close(tu.to_numpy(got["out"]).reshape(T, D // 128, 128),
                        tu.to_numpy(want["out"]).reshape(T, D // 128, 128), Q=Q)
    tu.assert_state_close(tu.to_numpy(got["state"]), tu.to_numpy(want["state"]))
    tu.assert_corr_close(tu.to_numpy(got["corr"]), tu.to_numpy(want["corr"]))
    np.testing.assert_array_equal(tu.to_numpy(got["key_gate"]), tu.to_numpy(want["key_gate"]))
    np.testing.assert_array_equal(tu.to_numpy(got["conv_state"]),
                                  tu.to_numpy(want["conv_state"]))
    assert int(tu.to_numpy(got["status"])[0]) == 0
    assert int(tu.to_numpy(want["status"])[0]) == 0


@pytest.mark.parametrize("Q", [8, 3])
def test_noalloc_matches_the_workspace_entry_point_on_two_calls(Q):
    import torch
    from linear_attention_speculative_recoverssm_gb300 import kda_layer_step_workspace_bytes
    case = synth.layer_case(B=12, H=3, Q=Q, slots=32, seed=900 + Q, padding_frac=0.15,
                            no_record_frac=0.1)
    want, got = _device(case), _device(case)
    workspace = torch.empty(kda_layer_step_workspace_bytes(12, 3, Q), dtype=torch.uint8,
                            device="cuda")
    for call in range(2):
        _with_workspace(case, want, workspace)
        _without_workspace(case, got)
        torch.cuda.synchronize()
        _same_results(got, want, Q)
        assert tu.to_numpy(got["out"]).any(), f"call {call}: no outputs"


def test_noalloc_takes_no_device_memory():
    """After a first call on this device (which may load the library's code
    and its array), further calls leave the device's free memory as it was."""
    import torch
    case = synth.layer_case(B=8, H=2, Q=4, slots=16, seed=931)
    d = _device(case)
    _without_workspace(case, d)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _without_workspace(case, d)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert int(tu.to_numpy(d["status"])[0]) == 0


def test_noalloc_refuses_calls_beyond_its_scratch():
    """B * Q * H above 16384 (token, head) rows needs more than the fixed
    array: KDA_ERR_SCRATCH, before anything is read or launched (the tensors
    below are never touched)."""
    import torch
    from linear_attention_speculative_recoverssm_gb300 import (KDA_ERR_SCRATCH,
                                                               KDA_LAYER_STEP_NOALLOC_MAX_BYTES,
                                                               kda_layer_step_noalloc,
                                                               kda_layer_step_workspace_bytes)
    B, H, Q = 17, 128, 8
    assert kda_layer_step_workspace_bytes(B, H, Q) > KDA_LAYER_STEP_NOALLOC_MAX_BYTES
    assert kda_layer_step_workspace_bytes(16, H, Q) == KDA_LAYER_STEP_NOALLOC_MAX_BYTES
    bf = torch.zeros((1, 1, 16), dtype=torch.bfloat16, device="cuda")
    f32 = torch.zeros((1, 1, 16), dtype=torch.float32, device="cuda")
    i32 = torch.zeros(B, dtype=torch.int32, device="cuda")
    a_log = torch.zeros(H, dtype=torch.float32, device="cuda")
    rc = kda_layer_step_noalloc(bf, bf, None, bf, bf, bf, bf, a_log, f32, f32, i32, i32, i32,
                                f32, bf, bf, f32, bf, Q=Q, lower_bound=-5.0, q_scale=0.088,
                                eps=1e-6, raise_on_error=False)
    assert rc == KDA_ERR_SCRATCH
