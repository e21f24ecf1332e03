"""Sentinel guard regions around every buffer the library writes.

Each pool, record array and output is allocated with a margin of sentinel
values on both sides of its leading dimension; the library gets the inner
view (same strides), runs twice back to back, and the margins must come back
bit-identical: a write past either end of any buffer shows here even where it
would land in other valid memory.
"""
import numpy as np
import pytest

from linear_attention_speculative_recoverssm_gb300 import synth

import kda_testutil as tu

pytestmark = pytest.mark.gpu

MARGIN = 2
SENT16 = 0x7FC1          # a NaN pattern in BF16
SENT32 = 0x7FC0BEEF      # a NaN pattern in FP32


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from linear_attention_speculative_recoverssm_gb300 import _build, _lib
    assert torch.cuda.is_available()
    _build.build()
    _lib.load()


def guarded(a):
    """(full, inner): a device tensor with MARGIN sentinel rows on both sides
    of dim 0, and the inner view holding ``a``."""
    import torch
    shape = (a.shape[0] + 2 * MARGIN,) + a.shape[1:]
    if a.dtype == np.uint16:
        full_np = np.full(shape, SENT16, dtype=np.uint16)
    else:
        full_np = np.full(shape, SENT32, dtype=np.uint32).view(a.dtype)
    full_np[MARGIN:-MARGIN] = a
    full = tu.to_torch(full_np, "cuda")
    return full, full[MARGIN:-MARGIN]


def assert_margins(full, what):
    got = tu.to_numpy(full)
    bits = got.view(np.uint16) if got.dtype == np.uint16 else got.view(np.uint32)
    sent = SENT16 if got.dtype == np.uint16 else SENT32
    assert np.all(bits[:MARGIN] == sent), f"{what}: written below the buffer"
    assert np.all(bits[-MARGIN:] == sent), f"{what}: written past the buffer"


@pytest.mark.parametrize("varlen,split", [(False, 1), (False, 2), (False, 4), (True, 1), (True, 4)])
def test_guard_regions_step(varlen, split):
    import torch
    from linear_attention_speculative_recoverssm_gb300 import kda_replay_verify
    B, H, Q = (40, 3, 8) if split == 1 else (6, 2, 8)
    kw = dict(B=B, H=H, Q=Q, slots=2 * B + 4, seed=120 + split, padding_frac=0.2,
              no_record_frac=0.1)
    case = synth.varlen_case(**kw) if varlen else synth.replay_verify_case(**kw)
    d = tu.device_case(case)
    fulls = {}
    for key in ("state", "corr", "key_gate"):
        fulls[key], d[key] = guarded(case[key])
    fulls["out"], d["out"] = guarded(np.zeros(case["v"].shape, dtype=np.uint16))
    qsl = tu.to_torch(case["query_start_loc"], "cuda") if varlen else None
    for _ in range(2):
        kda_replay_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"],
                          d["dt_bias"], d["state"], d["state_slots"], d["record_rows"],
                          d["pending"], d["corr"], d["key_gate"], d["out"], Q=Q,
                          lower_bound=case["lower_bound"], q_scale=case["q_scale"],
                          query_start_loc=qsl, split=split, status=d["status"])
    torch.cuda.synchronize()
    assert int(tu.to_numpy(d["status"])[0]) == 0
    for key, full in fulls.items():
        assert_margins(full, key)


def test_guard_regions_verify_bf16():
    import torch
    from linear_attention_speculative_recoverssm_gb300 import kda_verify
    case = synth.replay_verify_case(B=30, H=2, Q=5, slots=64, seed=131, state_dtype="bf16",
                                    padding_frac=0.2)
    d = tu.device_case(case)
    fulls = {}
    for key in ("state", "corr", "key_gate"):
        fulls[key], d[key] = guarded(case[key])
    fulls["out"], d["out"] = guarded(np.zeros(case["v"].shape, dtype=np.uint16))
    kda_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"], d["dt_bias"],
               d["state"], d["state_slots"], d["corr"], d["key_gate"], d["out"], Q=5,
               lower_bound=case["lower_bound"], q_scale=case["q_scale"],
               record_rows=d["record_rows"], status=d["status"])
    torch.cuda.synchronize()
    assert int(tu.to_numpy(d["status"])[0]) == 0
    for key, full in fulls.items():
        assert_margins(full, key)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_guard_regions_commit(dtype):
    import torch
    from linear_attention_speculative_recoverssm_gb300 import (KDA_STATE_BF16, KDA_STATE_F32,
                                                               kda_commit, layer_tables)
    c = synth.commit_case(L=2, B=48, H=8, Q=4, slots=160, seed=132, state_dtype=dtype)
    fulls, states, corrs, kgs = [], [], [], []
    for lay in c["layers"]:
        f, s = guarded(lay["state"])
        fulls.append(f)
        states.append(s)
        corrs.append(tu.to_torch(lay["corr"], "cuda"))
        kgs.append(tu.to_torch(lay["key_gate"], "cuda"))
    tabs = layer_tables(states, corrs, kgs, "cuda")
    t = lambda a: tu.to_torch(a, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        kda_commit(*tabs, t(c["A_log"]), t(c["dt_bias"]), t(c["sources"]), t(c["commit_lens"]),
                   t(c["destinations"]),
                   state_dtype=KDA_STATE_BF16 if dtype == "bf16" else KDA_STATE_F32,
                   lower_bound=c["lower_bound"], L=c["L"], H=c["H"], B=c["B"], Q=c["Q"],
                   n_slots=states[0].shape[0], n_rows=corrs[0].shape[0],
                   boundaries=t(c["boundaries"]), boundary_lens=t(c["boundary_lens"]),
                   status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for l, f in enumerate(fulls):
        assert_margins(f, f"layer {l} state")


def test_guard_regions_layer():
    import torch
    from linear_attention_speculative_recoverssm_gb300 import kda_layer_epilogue, kda_layer_prologue
    case = synth.layer_case(B=10, H=3, Q=6, slots=24, seed=133, padding_frac=0.2)
    d = {key: tu.to_torch(case[key], "cuda") for key in
         ("x", "conv_weight", "conv_bias", "f_a", "f_b", "state_slots", "record_rows",
          "pending", "gate", "norm_weight")}
    f_conv, d["conv_state"] = guarded(case["conv_state"])
    shape = (case["B"] * case["Q"], case["H"], 128)
    outs = [guarded(np.zeros(shape, dtype=np.uint16)) for _ in range(4)]
    f_out, out = guarded(np.zeros((shape[0], case["H"] * 128), dtype=np.uint16))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        kda_layer_prologue(d["x"], d["conv_weight"], d["conv_bias"], d["conv_state"], d["f_a"],
                           d["f_b"], d["state_slots"], d["record_rows"], d["pending"],
                           *(o[1] for o in outs), Q=case["Q"], status=status)
        kda_layer_epilogue(outs[0][1], d["gate"], d["norm_weight"], out, eps=case["eps"])
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_margins(f_conv, "convolution windows")
    for name, (f, _) in zip(("q", "k", "v", "raw_g"), outs):
        assert_margins(f, name)
    assert_margins(f_out, "layer output")
