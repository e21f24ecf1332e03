"""The multi-layer replay + verify (one launch over L layers with per-layer
pool, correction and key/gate bases) against L single-layer oracle calls.

Each layer l is compared element by element with the FP64 oracle run on
layer l's operands alone: outputs (rel-L2 <= 2e-3 overall and per item),
touched pages (max|dS| <= 1e-4 max|S|), corrections, key / gate records,
and every untouched page and record row bit-exact; the status word clean.
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


def _device(case):
    import torch
    dev = "cuda"
    d = {key: tu.to_torch(case[key], dev) for key in synth.LAYER_STACKED + synth.SHARED_INDEX}
    d["pools"] = [tu.to_torch(c["state"], dev) for c in case["layers"]]
    d["corrs"] = [tu.to_torch(c["corr"], dev) for c in case["layers"]]
    d["kgs"] = [tu.to_torch(c["key_gate"], dev) for c in case["layers"]]
    d["out"] = torch.zeros(case["q"].shape, dtype=torch.bfloat16, device=dev)
    d["status"] = torch.zeros(1, dtype=torch.int32, device=dev)
    return d


def _run(case, d):
    import torch
    from linear_attention_speculative_recoverssm_gb300 import kda_replay_verify_layers
    kda_replay_verify_layers(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"],
                             d["dt_bias"], d["pools"], d["state_slots"], d["record_rows"],
                             d["pending"], d["corrs"], d["kgs"], d["out"], Q=case["Q"],
                             lower_bound=case["lower_bound"], q_scale=case["q_scale"],
                             status=d["status"])
    torch.cuda.synchronize()


def _compare_layers(case, d):
    for l, layer in enumerate(case["layers"]):
        before = tu.copy_case(layer)
        ref = tu.copy_case(layer)
        tu.oracle_step(ref, replay=True)
        view = dict(state=d["pools"][l], out=d["out"][l], corr=d["corrs"][l],
                    key_gate=d["kgs"][l], status=d["status"])
        tu.compare_step(ref, view, before)


@pytest.mark.parametrize("L,Q", [(3, 1), (3, 4), (2, 8), (5, 3)])
def test_layers_match_single_layer_oracle(L, Q):
    case = synth.layers_case(L=L, B=20, H=4, Q=Q, slots=32, seed=800 + 10 * L + Q,
                             padding_frac=0.1, no_record_frac=0.1)
    d = _device(case)
    _run(case, d)
    _compare_layers(case, d)


def test_layers_many_heads():
    """H = 128 on three requests over two layers: each layer's slot spans 128
    pages, and the (layer, request, head) index is split by the layer and
    head counts at a large head count."""
    case = synth.layers_case(L=2, B=3, H=128, Q=8, slots=8, seed=870)
    d = _device(case)
    _run(case, d)
    _compare_layers(case, d)


def test_layers_spread_key_norms():
    """Per-vector key norms spread over 1e-3 .. 1e2 in every layer."""
    case = synth.layers_case(L=3, B=16, H=4, Q=6, slots=24, seed=830, padding_frac=0.1,
                             key_norms="spread")
    d = _device(case)
    _run(case, d)
    _compare_layers(case, d)


def test_layers_with_record_capacity_above_the_window_and_separate_pools():
    """Record capacity 8 with a window of 3; each layer's pool, corrections
    and records are separate allocations (per-layer bases, not one stride)."""
    case = synth.layers_case(L=4, B=12, H=2, Q=3, RQ=8, slots=20, seed=840)
    d = _device(case)
    _run(case, d)
    _compare_layers(case, d)


def test_one_layer_equals_the_single_layer_call():
    """L = 1 through the multi-layer entry point gives bit for bit what
    kda_replay_verify (split 1) gives."""
    import torch
    case = synth.layers_case(L=1, B=24, H=4, Q=8, slots=32, seed=850, padding_frac=0.1)
    d = _device(case)
    _run(case, d)
    layer = case["layers"][0]
    single = tu.device_case(layer)
    tu.gpu_step(layer, single, replay=True, split=1)
    torch.cuda.synchronize()
    assert torch.equal(single["out"], d["out"][0])
    assert torch.equal(single["state"], d["pools"][0])
    assert torch.equal(single["corr"], d["corrs"][0])
    assert torch.equal(single["key_gate"], d["kgs"][0])


def test_layers_out_of_range_indices_reported():
    """A slot outside the pools and a record row outside the records are
    reported (KDA_ERR_ARG) in every layer and treated as inert / record-less,
    never faulted."""
    from linear_attention_speculative_recoverssm_gb300 import KDA_ERR_ARG
    case = synth.layers_case(L=2, B=8, H=2, Q=2, slots=12, seed=860)
    case["state_slots"][3] = 12 + 5
    case["record_rows"][5] = case["layers"][0]["corr"].shape[0] + 2
    d = _device(case)
    _run(case, d)
    assert int(tu.to_numpy(d["status"])[0]) == KDA_ERR_ARG
    out = tu.to_numpy(d["out"]).reshape(2, 8, 2, 2, 128)
    assert not out[:, 3].any()
