"""The model layer around the step on the GPU against the FP64 oracle.

The convolution + SiLU, the gate projection and the gated norm round their
FP32 sums once to BF16, the oracle its FP64 sums: a value near a rounding
boundary may land one BF16 step apart, so those outputs are compared within
one BF16 unit in the last place of the oracle's value (plus 1e-6 of the
largest magnitude, for sums that cancel to far below their terms), and
rel-L2 <= 2e-3 overall.  The convolution windows are copies: bit-exact.  The
whole layer (prologue, step, epilogue) is compared stage by stage: the step
and the norm are checked on the GPU's own BF16 intermediates, so a rounding
step apart in one stage does not carry into the next.
"""
import numpy as np
import pytest

from linear_attention_speculative_recoverssm_gb300 import synth
from oracle import kda_oracle as ko

import kda_testutil as tu

pytestmark = pytest.mark.gpu

SENTINEL = 0x7FC1  # a NaN pattern: outputs of skipped items must keep it


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from linear_attention_speculative_recoverssm_gb300 import _build, _lib
    assert torch.cuda.is_available()
    _build.build()
    _lib.load()


def assert_bf16_close(got_bits, ref_bits, what):
    got = ko.bf16_to_f64(got_bits)
    ref = ko.bf16_to_f64(ref_bits)
    bound = tu.bf16_ulp(ref) + 1e-6 * np.abs(ref).max()
    excess = np.abs(got - ref) - bound
    assert excess.max() <= 0, f"{what}: exceeds one BF16 step by {excess.max():.3e}"
    assert tu.rel_l2(got, ref) <= tu.OUT_REL_L2, what


def _device_layer(case):
    import torch
    d = {key: tu.to_torch(case[key], "cuda") for key in
         ("x", "conv_weight", "conv_state", "f_a", "f_b", "state_slots", "record_rows",
          "pending", "gate", "norm_weight")}
    d["conv_bias"] = None if case["conv_bias"] is None else tu.to_torch(case["conv_bias"], "cuda")
    shape = (case["B"] * case["Q"], case["H"], 128)
    for key in ("q", "k", "v", "raw_g"):
        d[key] = tu.to_torch(np.full(shape, SENTINEL, dtype=np.uint16), "cuda")
    d["status"] = torch.zeros(1, dtype=torch.int32, device="cuda")
    return d


def _gpu_prologue(case, d, pending=True):
    from linear_attention_speculative_recoverssm_gb300 import kda_layer_prologue
    kda_layer_prologue(d["x"], d["conv_weight"], d["conv_bias"], d["conv_state"], d["f_a"],
                       d["f_b"], d["state_slots"], d["record_rows"],
                       d["pending"] if pending else None, d["q"], d["k"], d["v"], d["raw_g"],
                       Q=case["Q"], status=d["status"])


def _oracle_prologue(case, pending=True, items=None):
    state = case["conv_state"].copy()
    out = ko.layer_prologue(x=case["x"], conv_weight=case["conv_weight"],
                            conv_bias=case["conv_bias"], conv_state=state, f_a=case["f_a"],
                            f_b=case["f_b"], state_slots=case["state_slots"],
                            record_rows=case["record_rows"],
                            pending=case["pending"] if pending else None, B=case["B"],
                            H=case["H"], Q=case["Q"], items=items)
    return out, state


def _compare_prologue(case, d, ref, ref_state, items=None):
    Q, H = case["Q"], case["H"]
    got = [tu.to_numpy(d[key]) for key in ("q", "k", "v", "raw_g")]
    live = case["state_slots"] > 0
    todo = items if items is not None else range(case["B"] * H)
    for name, g, r in zip(("q", "k", "v", "raw_g"), got, ref):
        sel_g, sel_r = [], []
        for i in todo:
            b, h = divmod(int(i), H)
            rows = slice(b * Q, (b + 1) * Q)
            if live[b]:
                sel_g.append(g[rows, h])
                sel_r.append(r[rows, h])
            else:
                assert np.all(g[rows, h] == SENTINEL), f"{name}: inert item {i} written"
        assert_bf16_close(np.concatenate(sel_g), np.concatenate(sel_r), name)
    got_state = tu.to_numpy(d["conv_state"])
    if items is None:
        np.testing.assert_array_equal(got_state, ref_state, err_msg="convolution windows")
    else:
        D = H * 128
        for i in todo:
            b, h = divmod(int(i), H)
            s = int(case["state_slots"][b])
            if s > 0:
                for part in range(3):
                    chans = slice(part * D + h * 128, part * D + (h + 1) * 128)
                    np.testing.assert_array_equal(got_state[s, chans], ref_state[s, chans])


@pytest.mark.parametrize("Q,bias,pending,RQ", [(8, True, True, 8), (4, False, True, 4),
                                               (1, True, True, 1), (5, True, False, 5),
                                               (3, False, False, 3), (4, True, True, 7)])
def test_layer_prologue(Q, bias, pending, RQ):
    """RQ > Q: the window is longer than the new one, whose tail is kept."""
    import torch
    case = synth.layer_case(B=14, H=3, Q=Q, slots=40, seed=80 + Q, bias=bias,
                            padding_frac=0.2, RQ=RQ)
    d = _device_layer(case)
    _gpu_prologue(case, d, pending)
    torch.cuda.synchronize()
    assert int(tu.to_numpy(d["status"])[0]) == 0
    ref, ref_state = _oracle_prologue(case, pending)
    _compare_prologue(case, d, ref, ref_state)


def test_layer_epilogue():
    import torch
    from linear_attention_speculative_recoverssm_gb300 import kda_layer_epilogue
    rng = np.random.default_rng(5)
    T, H = 37, 5
    o = synth.to_bf16_bits(rng.standard_normal((T, H, 128)).astype(np.float32))
    o[3, 2] = 0  # an all-zero row (an inert item's outputs)
    gate = synth.to_bf16_bits(rng.standard_normal((T, H * 128)).astype(np.float32))
    w = (1 + 0.1 * rng.standard_normal(128)).astype(np.float32)
    out = torch.zeros((T, H * 128), dtype=torch.bfloat16, device="cuda")
    kda_layer_epilogue(tu.to_torch(o, "cuda"), tu.to_torch(gate, "cuda"), tu.to_torch(w, "cuda"),
                       out, eps=1e-6)
    torch.cuda.synchronize()
    ref = ko.layer_epilogue(o=o, gate=gate, norm_weight=w, eps=1e-6)
    assert_bf16_close(tu.to_numpy(out), ref, "gated norm")
    assert not tu.to_numpy(out).reshape(T, H, 128)[3, 2].any()


@pytest.mark.parametrize("split", [1, 2, 4])
@pytest.mark.parametrize("Q", [4, 8])
def test_layer_whole_step(Q, split):
    """Prologue -> fused replay + verify -> epilogue, each stage against the
    oracle on the previous stage's GPU outputs; the step on every launch
    shape (split 1 is the persistent kernel the benchmark times).  The
    prologue's q, k come out of a convolution + SiLU, so their norms vary
    from token to token."""
    import torch
    from linear_attention_speculative_recoverssm_gb300 import kda_layer_epilogue, kda_replay_verify
    case = synth.layer_case(B=10, H=2, Q=Q, slots=24, seed=90 + Q, padding_frac=0.1,
                            no_record_frac=0.1)
    d = _device_layer(case)
    _gpu_prologue(case, d)
    # the step on the prologue's outputs
    step = tu.device_case(case)
    for key in ("q", "k", "v", "raw_g"):
        step[key] = d[key]
    kda_replay_verify(step["q"], step["k"], step["v"], step["raw_g"], step["raw_beta"],
                      step["A_log"], step["dt_bias"], step["state"], step["state_slots"],
                      step["record_rows"], step["pending"], step["corr"], step["key_gate"],
                      step["out"], Q=Q, lower_bound=case["lower_bound"], q_scale=case["q_scale"],
                      split=split, status=step["status"])
    out = torch.zeros((case["B"] * Q, case["H"] * 128), dtype=torch.bfloat16, device="cuda")
    kda_layer_epilogue(step["out"], tu.to_torch(case["gate"], "cuda"), d["norm_weight"], out,
                       eps=case["eps"])
    torch.cuda.synchronize()
    assert int(tu.to_numpy(d["status"])[0]) == 0
    assert int(tu.to_numpy(step["status"])[0]) == 0
    # stage 1: the prologue
    ref, ref_state = _oracle_prologue(case)
    _compare_prologue(case, d, ref, ref_state)
    # stage 2: the step on the GPU's q, k, v, raw gates (inert items' inputs
    # are never read; zero them for the oracle)
    before = tu.copy_case(case)
    stage = tu.copy_case(case)
    for key in ("q", "k", "v", "raw_g"):
        a = tu.to_numpy(d[key]).copy()
        a[a == SENTINEL] = 0
        stage[key] = a
    tu.oracle_step(stage, replay=True)
    tu.compare_step(stage, step, before)
    # stage 3: the gated norm of the GPU's step outputs
    ref_out = ko.layer_epilogue(o=tu.to_numpy(step["out"]), gate=case["gate"],
                                norm_weight=case["norm_weight"], eps=case["eps"])
    assert_bf16_close(tu.to_numpy(out), ref_out, "layer output")


def test_layer_prologue_full_size_sampled():
    """The layer workload at full size (H=64, B=512, Q=8) on sampled items."""
    import torch
    case = synth.make("layer-f32-h64-b512-q8")
    d = _device_layer(case)
    _gpu_prologue(case, d)
    torch.cuda.synchronize()
    assert int(tu.to_numpy(d["status"])[0]) == 0
    rng = np.random.default_rng(11)
    items = np.sort(rng.choice(case["B"] * case["H"], size=96, replace=False))
    ref, ref_state = _oracle_prologue(case, items=items)
    _compare_prologue(case, d, ref, ref_state, items=items)
