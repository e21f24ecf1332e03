"""Parity with per-vector key norms spread over 1e-3 .. 1e2.

The workloads draw q, k and the recorded keys as unit directions, which is
the right recipe to time but cannot tell a kernel that normalises each
vector by its own norm from one that skips a normalisation or takes another
token's or head's norm: with unit vectors every such norm is ~1.  These
tests draw the same cases with ``key_norms="spread"`` (every (token, head)
vector of q, k and of the recorded keys at its own norm, a tenth of them
near sqrt(1e-6), where the 1e-6 inside the root matters) and run them
through every kernel that normalises: the persistent step kernel (uniform
and query_start_loc windows), the cluster split, the verify-only path on
FP32 and BF16 pools, the standalone commit, and the deferred decode loop.
``tests/test_norm_discrimination.py`` shows on the CPU that these inputs
separate a correct normalisation from a skipped or mis-indexed one by far
more than the tolerances.
"""
import numpy as np
import pytest

from linear_attention_speculative_recoverssm_gb300 import synth
from oracle import kda_oracle as ko

import kda_testutil as tu

pytestmark = pytest.mark.gpu

SPREAD = dict(key_norms="spread")


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


@pytest.mark.parametrize("Q", [1, 3, 8])
def test_replay_verify_whole_items(Q):
    """The persistent kernel the benchmark times (split 1)."""
    case = synth.replay_verify_case(B=40, H=8, Q=Q, slots=64, seed=700 + Q, padding_frac=0.1,
                                    no_record_frac=0.1, **SPREAD)
    _run_and_compare(case, split=1)


@pytest.mark.parametrize("Q", [2, 8])
def test_replay_verify_whole_items_with_boundary(Q):
    case = synth.replay_verify_case(B=24, H=4, Q=Q, slots=64, seed=710 + Q, boundary_frac=0.5,
                                    padding_frac=0.1, **SPREAD)
    _run_and_compare(case, boundary=True, split=1)


@pytest.mark.parametrize("Q", [1, 5, 8])
@pytest.mark.parametrize("split", [2, 4])
def test_replay_verify_cluster_split(Q, split):
    case = synth.replay_verify_case(B=6, H=4, Q=Q, slots=16, seed=720 + Q, padding_frac=0.2,
                                    no_record_frac=0.2, **SPREAD)
    _run_and_compare(case, split=split)


@pytest.mark.parametrize("Q", [1, 4, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_verify_only(Q, dtype):
    case = synth.replay_verify_case(B=30, H=6, Q=Q, slots=40, seed=730 + Q, state_dtype=dtype,
                                    padding_frac=0.1, no_record_frac=0.1, **SPREAD)
    _run_and_compare(case, replay=False)


@pytest.mark.parametrize("split", [1, 2, 4])
@pytest.mark.parametrize("replay", [True, False])
def test_variable_windows(split, replay):
    """query_start_loc windows of 0..Q tokens (the VARLEN instances)."""
    if not replay and split != 1:
        pytest.skip("the verify-only path has no cluster split")
    case = synth.varlen_case(B=24, H=4, Q=8, slots=40, seed=740 + split, padding_frac=0.1,
                             **SPREAD)
    qsl = case["query_start_loc"]
    before = tu.copy_case(case)
    ref = tu.copy_case(case)
    out = np.zeros(case["v"].shape, dtype=np.uint16)
    ko.replay_verify(q=ref["q"], k=ref["k"], v=ref["v"], raw_g=ref["raw_g"],
                     raw_beta=ref["raw_beta"], A_log=ref["A_log"], dt_bias=ref["dt_bias"],
                     lower_bound=ref["lower_bound"], q_scale=ref["q_scale"], state=ref["state"],
                     state_slots=ref["state_slots"], record_rows=ref["record_rows"],
                     corr=ref["corr"], key_gate=ref["key_gate"], out=out, B=ref["B"],
                     H=ref["H"], Q=ref["Q"], pending=ref["pending"] if replay else None,
                     query_start_loc=qsl)
    d = tu.device_case(case)
    from linear_attention_speculative_recoverssm_gb300 import kda_replay_verify, kda_verify
    common = dict(Q=case["Q"], lower_bound=case["lower_bound"], q_scale=case["q_scale"],
                  status=d["status"], query_start_loc=tu.to_torch(qsl, "cuda"))
    if replay:
        kda_replay_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"],
                          d["dt_bias"], d["state"], d["state_slots"], d["record_rows"],
                          d["pending"], d["corr"], d["key_gate"], d["out"], split=split,
                          **common)
    else:
        kda_verify(d["q"], d["k"], d["v"], d["raw_g"], d["raw_beta"], d["A_log"], d["dt_bias"],
                   d["state"], d["state_slots"], d["corr"], d["key_gate"], d["out"],
                   record_rows=d["record_rows"], **common)
    import torch
    torch.cuda.synchronize()
    got = tu.to_numpy(d["out"])
    tu.assert_out_close(got, out)
    for b in range(case["B"]):
        rows = slice(int(qsl[b]), int(qsl[b + 1]))
        for h in range(case["H"]):
            tu.assert_out_close(got[rows, h], out[rows, h], what=f"request {b} head {h}")
    changed = np.any(ref["state"] != before["state"], axis=(2, 3))
    got_state = tu.to_numpy(d["state"])
    np.testing.assert_array_equal(got_state[~changed], before["state"][~changed])
    if changed.any():
        tu.assert_state_close(got_state[changed], ref["state"][changed])
    tu.assert_corr_close(tu.to_numpy(d["corr"]), ref["corr"])
    np.testing.assert_array_equal(tu.to_numpy(d["key_gate"]), ref["key_gate"])
    assert int(tu.to_numpy(d["status"])[0]) == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("Q", [4, 8])
def test_commit_align(dtype, Q):
    """The standalone commit replays recorded keys, each normalised by its
    own norm."""
    import torch
    from linear_attention_speculative_recoverssm_gb300 import (KDA_STATE_BF16, KDA_STATE_F32,
                                                               kda_commit, layer_tables)
    c = synth.commit_case(L=2, B=24, H=4, Q=Q, slots=96, seed=750 + Q, state_dtype=dtype,
                          boundary_frac=0.4, **SPREAD)
    dev = "cuda"
    states = [tu.to_torch(lay["state"], dev) for lay in c["layers"]]
    corrs = [tu.to_torch(lay["corr"], dev) for lay in c["layers"]]
    kgs = [tu.to_torch(lay["key_gate"], dev) for lay in c["layers"]]
    tabs = layer_tables(states, corrs, kgs, dev)
    t = lambda a: tu.to_torch(a, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kda_commit(*tabs, t(c["A_log"]), t(c["dt_bias"]), t(c["sources"]), t(c["commit_lens"]),
               t(c["destinations"]), state_dtype=KDA_STATE_BF16 if dtype == "bf16" else
               KDA_STATE_F32, lower_bound=c["lower_bound"], L=c["L"], H=c["H"], B=c["B"],
               Q=c["Q"], n_slots=states[0].shape[0], n_rows=corrs[0].shape[0],
               boundaries=t(c["boundaries"]), boundary_lens=t(c["boundary_lens"]), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_layers = [{k: v.copy() for k, v in lay.items()} for lay in c["layers"]]
    ko.commit(layers=ref_layers, A_log=c["A_log"], dt_bias=c["dt_bias"], sources=c["sources"],
              commit_lens=c["commit_lens"], destinations=c["destinations"],
              lower_bound=c["lower_bound"], Q=c["Q"], B=c["B"], H=c["H"],
              boundaries=c["boundaries"], boundary_lens=c["boundary_lens"])
    for l, (got_t, ref, orig) in enumerate(zip(states, ref_layers, c["layers"])):
        got = tu.to_numpy(got_t)
        changed = np.any(ref["state"] != orig["state"], axis=(2, 3))
        assert changed.any()
        np.testing.assert_array_equal(got[~changed], orig["state"][~changed])
        if dtype == "bf16":
            tu.assert_bf16_state_close(got[changed], ref["state"][changed], what=f"layer {l}")
        else:
            tu.assert_state_close(got[changed], ref["state"][changed], what=f"layer {l}")


@pytest.mark.parametrize("split", [1, 4])
def test_decode_loop(split):
    """The deferred protocol over 10 steps (fused replay + verify, defers,
    eager rows, flushes) against the FP64 stock recurrence, never
    resynchronised."""
    import torch
    from linear_attention_speculative_recoverssm_gb300 import DeferredRecoverSSM
    B, H, Q, steps = 8, 3, 6, 10
    case = synth.decode_loop_case(B=B, H=H, Q=Q, slots=2 * B + 4, steps=steps, seed=760 + split,
                                  padding_frac=0.15, eager_frac=0.2, **SPREAD)
    ref_outs, finals = ko.decode_stock(
        windows=case["windows"], window_of_step=case["window_of_step"],
        accepted=case["accepted"], A_log=case["A_log"], dt_bias=case["dt_bias"],
        lower_bound=case["lower_bound"], q_scale=case["q_scale"], state=case["state"],
        state_slots=case["state_slots"], B=B, H=H, Q=Q)
    d = tu.device_case(case)
    keys = ("q", "k", "v", "raw_g", "raw_beta")
    win = {key: tu.to_torch(case["windows"][key], "cuda") for key in keys}
    accepted = tu.to_torch(case["accepted"], "cuda")
    eager = tu.to_torch(case["eager"], "cuda")
    loop = DeferredRecoverSSM(d["state"], d["state_slots"], d["record_rows"], d["pending"],
                              d["corr"], d["key_gate"], d["A_log"], d["dt_bias"], Q=Q,
                              lower_bound=case["lower_bound"], q_scale=case["q_scale"],
                              split=split, status=d["status"])
    for s in range(steps):
        w = int(case["window_of_step"][s])
        out = torch.zeros_like(d["out"])
        loop.verify(*(win[key][w] for key in keys), out)
        loop.accept(accepted[s].clone(), eager[s])
        if (s + 1) % 4 == 0 or s == steps - 1:
            loop.flush()
        torch.cuda.synchronize()
        tu.assert_out_close(tu.to_numpy(out), ko.f64_to_bf16(ref_outs[s]), what=f"step {s}",
                            Q=Q)
    assert int(tu.to_numpy(d["status"])[0]) == 0
    pool = tu.to_numpy(d["state"])
    for (b, h), S in finals.items():
        tu.assert_state_close(pool[case["state_slots"][b], h], S, what=f"item {(b, h)}")
