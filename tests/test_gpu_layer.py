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


def test_layer_prologue_many_heads():
    """H = 128 on four requests: one token tile, 128 head tiles over the
    gate projection's CTAs (one or two each), and 384 channel parts per
    request for the convolution."""
    import torch
    case = synth.layer_case(B=4, H=128, Q=8, slots=8, seed=960, padding_frac=0.0)
    d = _device_layer(case)
    _gpu_prologue(case, d)
    torch.cuda.synchronize()
    assert int(tu.to_numpy(d["status"])[0]) == 0
    ref, ref_state = _oracle_prologue(case)
    _compare_prologue(case, d, ref, ref_state)


@pytest.mark.parametrize("B,H", [(3700, 1), (2900, 3)])
def test_layer_prologue_many_token_tiles(B, H):
    """Few heads and long batches: the gate projection's persistent CTAs
    (on half the SMs) each walk three or more 128-token tiles, so a CTA
    reloads its resident f_a tile into a slot freed by an earlier tile's last
    MMA, and the last tile is ragged (B * 8 not a multiple of 128).  One
    request per (tile, head) is checked against the oracle, so every tile
    and head is covered; inert requests' rows must stay untouched."""
    import torch
    Q = 8
    case = synth.layer_case(B=B, H=H, Q=Q, slots=B + 64, seed=900 + H, padding_frac=0.1)
    assert (B * Q) % 128 != 0
    d = _device_layer(case)
    _gpu_prologue(case, d)
    torch.cuda.synchronize()
    assert int(tu.to_numpy(d["status"])[0]) == 0
    rng = np.random.default_rng(12 + H)
    per_tile = 128 // Q  # requests per token tile
    items = []
    for r0 in range(0, B, per_tile):
        for h in range(H):
            b = int(rng.integers(r0, min(B, r0 + per_tile)))
            items.append(b * H + h)
    items = np.array(items)
    ref, ref_state = _oracle_prologue(case, items=items)
    _compare_prologue(case, d, ref, ref_state, items=items)


# --------------------------------------------------------------------------
# the fused layer step: prologue into a workspace, then the step with the
# gated RMSNorm folded into its row solve
# --------------------------------------------------------------------------

def _fused_layer(case, d, step, out, workspace):
    from linear_attention_speculative_recoverssm_gb300 import kda_layer_step
    kda_layer_step(d["x"], d["conv_weight"], d["conv_bias"], d["conv_state"], d["f_a"], d["f_b"],
                   step["raw_beta"], step["A_log"], step["dt_bias"], step["state"],
                   step["state_slots"], step["record_rows"], step["pending"], step["corr"],
                   step["key_gate"], d["gate"], d["norm_weight"], out, workspace, Q=case["Q"],
                   lower_bound=case["lower_bound"], q_scale=case["q_scale"], eps=case["eps"],
                   status=step["status"])


def _check_fused_layer(case, d, step, out, workspace, items=None):
    """Stage by stage: the workspace's q, k, v, raw_g against the oracle's
    prologue (one BF16 step), the pool, records and windows against the
    oracle's step on the GPU's own q, k, v, raw_g, and the layer output
    against the oracle's gated norm of that step's outputs (rel-L2 <= 2e-3,
    overall and per (request, head) item)."""
    B, H, Q = case["B"], case["H"], case["Q"]
    T = B * Q
    ws = tu.to_numpy(workspace).reshape(4, T, H, 128)
    for i, key in enumerate(("q", "k", "v", "raw_g")):
        d[key] = tu.to_torch(ws[i], "cuda")
    ref, ref_state = _oracle_prologue(case, items=items)
    _compare_prologue(case, d, ref, ref_state, items=items)
    # (on sampled items the oracle may update the case's own arrays: the
    # whole-pool comparisons below need the copies only without sampling)
    before = tu.copy_case(case) if items is None else None
    stage = tu.copy_case(case) if items is None else dict(case)
    for i, key in enumerate(("q", "k", "v", "raw_g")):
        a = ws[i].copy()
        a[a == SENTINEL] = 0
        stage[key] = a
    o_ref = np.zeros((T, H, 128), dtype=np.uint16)
    ko.replay_verify(q=stage["q"], k=stage["k"], v=stage["v"], raw_g=stage["raw_g"],
                     raw_beta=stage["raw_beta"], A_log=stage["A_log"],
                     dt_bias=stage["dt_bias"], lower_bound=stage["lower_bound"],
                     q_scale=stage["q_scale"], state=stage["state"],
                     state_slots=stage["state_slots"], record_rows=stage["record_rows"],
                     corr=stage["corr"], key_gate=stage["key_gate"], out=o_ref, B=B, H=H, Q=Q,
                     pending=stage["pending"], items=items)
    ref_out = ko.layer_epilogue(o=o_ref, gate=case["gate"], norm_weight=case["norm_weight"],
                                eps=case["eps"]).reshape(T, H, 128)
    got_out = tu.to_numpy(out).reshape(T, H, 128)
    if items is None:
        tu.assert_out_close(got_out, ref_out, what="layer output", Q=Q)
        stage["out"] = o_ref
        # the step's state and records (its outputs were normed in place)
        view = dict(step, out=tu.to_torch(o_ref, "cuda"))
        tu.compare_step(stage, view, before)
    else:
        for i in items:
            b, h = divmod(int(i), H)
            rows = slice(b * Q, (b + 1) * Q)
            tu.assert_out_close(got_out[rows, h], ref_out[rows, h], what=f"item {i}")
            s = int(case["state_slots"][b])
            if s > 0:
                tu.assert_state_close(tu.to_numpy(step["state"][s, h]), stage["state"][s, h],
                                      what=f"item {i} state")
    assert int(tu.to_numpy(step["status"])[0]) == 0


@pytest.mark.parametrize("Q,bias,RQ", [(8, True, 8), (4, False, 4), (1, True, 1), (5, True, 7),
                                       (3, False, 3)])
def test_fused_layer_step(Q, bias, RQ):
    import torch
    from linear_attention_speculative_recoverssm_gb300 import kda_layer_step_workspace_bytes
    case = synth.layer_case(B=12, H=3, Q=Q, slots=32, seed=95 + Q, bias=bias, padding_frac=0.15,
                            no_record_frac=0.1, RQ=RQ)
    d = _device_layer(case)
    step = tu.device_case(case)
    B, H = case["B"], case["H"]
    nbytes = kda_layer_step_workspace_bytes(B, H, Q)
    assert nbytes == 4 * B * Q * H * 128 * 2
    workspace = tu.to_torch(np.full(nbytes // 2, SENTINEL, dtype=np.uint16), "cuda")
    out = torch.full((B * Q, H * 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    _fused_layer(case, d, step, out, workspace)
    torch.cuda.synchronize()
    _check_fused_layer(case, d, step, out, workspace)


def test_fused_layer_step_spread_key_norms_and_back_to_back():
    """Spread key norms in the step's records; three launches back to back
    (each reads the pool, records and windows the previous one wrote) against
    three oracle layer steps."""
    import torch
    case = synth.layer_case(B=16, H=4, Q=6, slots=40, seed=120, padding_frac=0.2,
                            key_norms="spread")
    d = _device_layer(case)
    step = tu.device_case(case)
    from linear_attention_speculative_recoverssm_gb300 import kda_layer_step_workspace_bytes
    nbytes = kda_layer_step_workspace_bytes(16, 4, 6)
    workspace = tu.to_torch(np.full(nbytes // 2, SENTINEL, dtype=np.uint16), "cuda")
    out = torch.zeros((16 * 6, 4 * 128), dtype=torch.bfloat16, device="cuda")
    for it in range(3):
        _fused_layer(case, d, step, out, workspace)
        torch.cuda.synchronize()
        _check_fused_layer(case, d, step, out, workspace)
        # the next launch starts from what this one left (the oracle's copy
        # of the pool, records and windows follows the GPU's)
        for key in ("state", "corr", "key_gate"):
            case[key] = tu.to_numpy(step[key]).copy()
        case["conv_state"] = tu.to_numpy(d["conv_state"]).copy()


def test_fused_layer_step_full_size_sampled():
    """The benchmark's layer workload (H=64, B=512, Q=8) on sampled items."""
    import torch
    from linear_attention_speculative_recoverssm_gb300 import kda_layer_step_workspace_bytes
    case = synth.make("layer-f32-h64-b512-q8")
    B, H, Q = case["B"], case["H"], case["Q"]
    d = _device_layer(case)
    step = tu.device_case(case)
    workspace = torch.full((kda_layer_step_workspace_bytes(B, H, Q) // 2,), SENTINEL,
                           dtype=torch.int16, device="cuda")
    out = torch.zeros((B * Q, H * 128), dtype=torch.bfloat16, device="cuda")
    _fused_layer(case, d, step, out, workspace)
    torch.cuda.synchronize()
    items = np.sort(np.random.default_rng(17).choice(B * H, size=96, replace=False))
    _check_fused_layer(case, d, step, out, workspace.view(torch.bfloat16), items=items)
