"""Helpers shared by the GPU tests: moving generator cases between numpy
(the oracle's side) and torch device tensors (the library's side), running
both sides, and the comparison metrics with the stated tolerances."""
from __future__ import annotations

import numpy as np

from oracle import kda_oracle as ko

# Tolerances (the target's own, except the two marked as derived here):
OUT_REL_L2 = 2e-3          # BF16 outputs, rel-L2
STATE_REL_MAX = 1e-4       # FP32 states, max|dS| <= 1e-4 * max|S|
CORR_REL_MAX = 1e-4        # FP32 corrections (derived: same bound as the state)
# BF16 states (derived): the kernel rounds its FP32 result once, the oracle
# its FP64 result once; if the two pre-rounding values differ by d, the
# rounded ones differ by at most 1 BF16 ulp + d.  d is bounded by the FP32
# state tolerance, so |got - ref| <= ulp(ref) + 1e-4 * max|S| (an element that
# cancels to far below max|S| can differ by many of its own ulps).


def to_torch(a, device):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_numpy(t):
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


STEP_ARRAYS = ("q", "k", "v", "raw_g", "raw_beta", "A_log", "dt_bias", "state", "state_slots",
               "record_rows", "pending", "corr", "key_gate", "boundary_slots", "boundary_lens")


def device_case(case, device="cuda"):
    import torch
    d = {k: to_torch(case[k], device) for k in STEP_ARRAYS}
    d["out"] = torch.zeros(case["v"].shape, dtype=torch.bfloat16, device=device)
    d["status"] = torch.zeros(1, dtype=torch.int32, device=device)
    return d


def copy_case(case):
    return {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in case.items()}


def oracle_step(case, *, replay=True, boundary=False, items=None):
    """Runs the oracle in place on `case` (numpy) and returns its BF16 out."""
    out = np.zeros(case["v"].shape, dtype=np.uint16)
    ko.replay_verify(
        q=case["q"], k=case["k"], v=case["v"], raw_g=case["raw_g"], raw_beta=case["raw_beta"],
        A_log=case["A_log"], dt_bias=case["dt_bias"], lower_bound=case["lower_bound"],
        q_scale=case["q_scale"], state=case["state"], state_slots=case["state_slots"],
        record_rows=case["record_rows"], corr=case["corr"], key_gate=case["key_gate"], out=out,
        B=case["B"], H=case["H"], Q=case["Q"], null_slot=case["null_slot"],
        pending=case["pending"] if replay else None,
        boundary_slots=case["boundary_slots"] if boundary else None,
        boundary_lens=case["boundary_lens"] if boundary else None, items=items)
    case["out"] = out
    return out


def gpu_step(case, d, *, replay=True, boundary=False, split=1):
    from linear_attention_speculative_recoverssm_gb300 import kda_replay_verify, kda_verify
    common = dict(Q=case["Q"], lower_bound=case["lower_bound"], q_scale=case["q_scale"],
                  null_slot=case["null_slot"], status=d["status"])
    if replay:
        kda_replay_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"],
                          d["dt_bias"], d["state"], d["state_slots"], d["record_rows"],
                          d["pending"], d["corr"], d["key_gate"], d["out"],
                          boundary_slots=d["boundary_slots"] if boundary else None,
                          boundary_lens=d["boundary_lens"] if boundary else None,
                          split=split, **common)
    else:
        kda_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"], d["dt_bias"],
                   d["state"], d["state_slots"], d["corr"], d["key_gate"], d["out"],
                   record_rows=d["record_rows"], **common)


def rel_l2(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def assert_out_close(got_bits, ref_bits, what="out", Q=None):
    """rel-L2 <= 2e-3 over the whole output and over each (request, head)
    item's window when Q is given (so one bad item cannot hide); all-zero
    reference items (inert rows) must be exactly zero."""
    got = ko.bf16_to_f64(got_bits)
    ref = ko.bf16_to_f64(ref_bits)
    if not np.any(ref):
        np.testing.assert_array_equal(got_bits, ref_bits, err_msg=what)
        return
    err = rel_l2(got, ref)
    assert err <= OUT_REL_L2, f"{what}: rel-L2 {err:.3e} > {OUT_REL_L2}"
    if Q is not None:
        T, H, V = ref.shape
        g4 = got.reshape(T // Q, Q, H, V).transpose(0, 2, 1, 3).reshape(-1, Q * V)
        r4 = ref.reshape(T // Q, Q, H, V).transpose(0, 2, 1, 3).reshape(-1, Q * V)
        num = np.linalg.norm(g4 - r4, axis=1)
        den = np.linalg.norm(r4, axis=1)
        zero = den == 0
        assert np.all(num[zero] == 0), f"{what}: nonzero output on an inert item"
        worst = (num[~zero] / den[~zero]).max() if (~zero).any() else 0.0
        assert worst <= OUT_REL_L2, f"{what}: worst item rel-L2 {worst:.3e}"


def assert_state_close(got, ref, what="state"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    assert err <= STATE_REL_MAX * max(scale, 1e-30), \
        f"{what}: max|dS| {err:.3e} > {STATE_REL_MAX} * {scale:.3e}"


def assert_corr_close(got, ref, what="corr"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    assert err <= CORR_REL_MAX * max(scale, 1e-30), \
        f"{what}: max|du| {err:.3e} > {CORR_REL_MAX} * {scale:.3e}"


def bf16_ulp(x):
    """Spacing of BF16 numbers at |x| (8 significant bits)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(x > 0, x, 2.0 ** -126))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def assert_bf16_state_close(got_bits, ref_bits, what="bf16 state"):
    """|got - ref| <= ulp(ref) + 1e-4 max|ref| per element; rel-L2 <= 2e-3."""
    got = ko.bf16_to_f64(got_bits)
    ref = ko.bf16_to_f64(ref_bits)
    bound = bf16_ulp(ref) + STATE_REL_MAX * np.abs(ref).max()
    excess = np.abs(got - ref) - bound
    assert excess.max() <= 0, f"{what}: |d| exceeds ulp + 1e-4 max|S| by {excess.max():.3e}"
    err = rel_l2(got, ref)
    assert err <= OUT_REL_L2, f"{what}: rel-L2 {err:.3e}"


def compare_step(case_ref, d, case_before, *, items=None, check_all_slots=True):
    """Compares every output of one step: out, state pool (touched pages within
    tolerance, untouched pages bit-exact), corrections, key/gate records
    (bit-exact copies) and untouched record rows."""
    got_state = to_numpy(d["state"])
    got_out = to_numpy(d["out"])
    got_corr = to_numpy(d["corr"])
    got_kg = to_numpy(d["key_gate"])
    assert_out_close(got_out, case_ref["out"], Q=case_ref["Q"])
    np.testing.assert_array_equal(got_kg, case_ref["key_gate"], err_msg="key/gate records")
    assert_corr_close(got_corr, case_ref["corr"])
    kept = np.all(case_ref["corr"] == case_before["corr"], axis=(2, 3))
    np.testing.assert_array_equal(got_corr[kept], case_before["corr"][kept],
                                  err_msg="untouched correction records")
    changed = np.any(case_ref["state"] != case_before["state"], axis=(2, 3))
    if check_all_slots:
        np.testing.assert_array_equal(got_state[~changed], case_before["state"][~changed],
                                      err_msg="untouched state pages")
    if changed.any():
        assert_state_close(got_state[changed], case_ref["state"][changed])
    assert int(to_numpy(d["status"])[0]) == 0
