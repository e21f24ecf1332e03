"""Pins of the FP64 oracle to things other than itself (no GPU needed).

Each test checks the oracle against what the pages or the mathematics fix:
a hand-derived worked example, alternative formulations the pages state
(closed-form replay, chunked WY verify), special cases that reduce to a
textbook routine, and invariants (n = 0 leaves the checkpoint, deferred then
flushed equals eager).  Shapes with K != V are used where a transposed
operand would otherwise go unnoticed.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import kda_oracle as ko
from linear_attention_speculative_recoverssm_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(x):
    """Exactly representable FP32 values -> BF16 bits (test helper)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not exactly representable in BF16"
    return (b >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# conversions
# ---------------------------------------------------------------------------

def test_bf16_rounding_known_patterns():
    cases = {
        1.0: 0x3F80, -2.0: 0xC000, 0.0: 0x0000,
        1.0 + 2.0 ** -8: 0x3F80,            # tie -> even (down)
        1.0 + 3 * 2.0 ** -8: 0x3F82,        # tie -> even (up)
        1.0 + 2.0 ** -8 + 2.0 ** -30: 0x3F81,  # just above the tie
        2.0 ** -130: 0x0008,                 # subnormal
        3.4e38: 0x7F80,                      # rounds past the largest -> inf
    }
    for value, bits in cases.items():
        assert int(ko.f64_to_bf16(np.array([value]))[0]) == bits, value


def test_bf16_rounding_matches_torch_on_fp32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ko.f64_to_bf16(x.astype(np.float64)), ref)
    back = ko.bf16_to_f64(ref)
    np.testing.assert_array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


# ---------------------------------------------------------------------------
# per-channel operands
# ---------------------------------------------------------------------------

def test_decay_special_values():
    # sigmoid(0) = 1/2: d = exp(lb / 2); A_log = 0 -> exp(A_log) = 1
    d = ko.decay(np.zeros(3), 0.0, np.zeros(3), -5.0)
    np.testing.assert_allclose(d, math.exp(-2.5), rtol=1e-15)
    # lower bound 0: no decay at all
    np.testing.assert_array_equal(ko.decay(np.array([-3.0, 0.0, 7.0]), 1.3, np.ones(3), 0.0), 1.0)
    # saturated gate: sigmoid -> 1, d -> exp(lb); very negative: d -> 1
    np.testing.assert_allclose(ko.decay(np.array([80.0]), 0.0, np.zeros(1), -5.0), math.exp(-5.0), rtol=1e-15)
    np.testing.assert_allclose(ko.decay(np.array([-80.0]), 0.0, np.zeros(1), -5.0), 1.0, rtol=1e-15)
    # exp(A_log) multiplies (raw_g + dt_bias): A_log = ln 2, raw_g = 1, dt = -0.5 -> sigmoid(1)
    d = ko.decay(np.array([1.0]), math.log(2.0), np.array([-0.5]), -1.0)
    np.testing.assert_allclose(d, math.exp(-1.0 / (1.0 + math.exp(-1.0))), rtol=1e-14)


def test_l2norm_closed_form():
    x = np.array([[3.0, 4.0], [0.0, 0.0], [1e-4, 0.0]])
    y = ko.l2norm(x)
    np.testing.assert_allclose(y[0], np.array([3.0, 4.0]) / math.sqrt(25.0 + 1e-6), rtol=1e-15)
    np.testing.assert_array_equal(y[1], 0.0)
    np.testing.assert_allclose(y[2, 0], 1e-4 / math.sqrt(1e-8 + 1e-6), rtol=1e-14)


# ---------------------------------------------------------------------------
# the hand-derived worked example (K = V = 2)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case_index", [0, 1])
def test_hand_worked_example(case_index):
    g = json.load(open(os.path.join(GOLDEN, "kda_hand_k2.json")))
    c = g["cases"][case_index]
    Q = len(c["q"])
    K = V = 2
    rec = c["records"]
    state = np.zeros((2, 1, V, K), dtype=np.float32)
    state[1, 0] = np.array(c["S0"], dtype=np.float32)
    corr = np.zeros((1, 1, 2, V), dtype=np.float32)
    key_gate = np.zeros((1, 1, 2, 2 * K), dtype=np.uint16)
    if rec is not None:
        corr[0, 0] = np.array(rec["u"], dtype=np.float32)
        key_gate[0, 0, :, :K] = _bits(rec["k"])
        key_gate[0, 0, :, K:] = _bits(rec["raw_g"])
    out = np.zeros((Q, 1, V), dtype=np.uint16)
    out64 = np.zeros((Q, 1, V))
    ko.replay_verify(
        q=_bits(c["q"]).reshape(Q, 1, K), k=_bits(c["k"]).reshape(Q, 1, K),
        v=_bits(c["v"]).reshape(Q, 1, V), raw_g=_bits(c["raw_g"]).reshape(Q, 1, K),
        raw_beta=_bits(c["raw_beta"]).reshape(Q, 1),
        A_log=np.array(g["A_log"], dtype=np.float32),
        dt_bias=np.array(g["dt_bias"], dtype=np.float32),
        lower_bound=g["lower_bound"], q_scale=g["q_scale"], state=state,
        state_slots=np.array([1], dtype=np.int32), record_rows=np.array([0], dtype=np.int32),
        pending=np.array([c["pending"]], dtype=np.int32), corr=corr, key_gate=key_gate,
        out=out, out_f64=out64, B=1, H=1, Q=Q)
    np.testing.assert_allclose(out64[:, 0, :], np.array(c["expect_o"]), atol=1e-5, rtol=1e-5)
    np.testing.assert_allclose(corr[0, 0, :Q], np.array(c["expect_u"]), atol=1e-5, rtol=1e-5)
    np.testing.assert_allclose(state[1, 0], np.array(c["expect_state_after"]), atol=1e-5, rtol=1e-5)
    # records now hold the verified window's key and raw gate, copied bit-exactly
    np.testing.assert_array_equal(key_gate[0, 0, :Q, :K], _bits(c["k"]))
    np.testing.assert_array_equal(key_gate[0, 0, :Q, K:], _bits(c["raw_g"]))


# ---------------------------------------------------------------------------
# alternative formulations stated on the pages
# ---------------------------------------------------------------------------

def _toy(rng, K, V, n, Q):
    S0 = rng.standard_normal((V, K))
    u = rng.standard_normal((n, V)) * 0.5
    kr = rng.standard_normal((n, K))
    gr = rng.standard_normal((n, K))
    q = rng.standard_normal((Q, K))
    k = rng.standard_normal((Q, K))
    v = rng.standard_normal((Q, V))
    g = rng.standard_normal((Q, K))
    rb = rng.standard_normal(Q)
    a_log = rng.uniform(0, 2.5)
    dt = rng.standard_normal(K) * 0.1
    return S0, u, kr, gr, q, k, v, g, rb, a_log, dt


@pytest.mark.parametrize("K,V", [(2, 3), (5, 4), (128, 128)])
def test_closed_form_replay_equals_sequential(K, V):
    rng = np.random.default_rng(K * 31 + V)
    for n in range(0, 9):
        S0, u, kr, gr, *_, a_log, dt = _toy(rng, K, V, n, 1)
        seq, _ = ko.replay_item(S0, u, kr, gr, n, a_log, dt, -5.0)
        closed = ko.replay_closed_form(S0, u, kr, gr, n, a_log, dt, -5.0)
        np.testing.assert_allclose(closed, seq, rtol=1e-12, atol=1e-12 * np.abs(seq).max())


@pytest.mark.parametrize("K,V", [(2, 3), (6, 4), (128, 128)])
def test_chunked_verify_equals_stock_recurrence(K, V):
    rng = np.random.default_rng(K * 17 + V)
    for Q in range(1, 9):
        S0, _, _, _, q, k, v, g, rb, a_log, dt = _toy(rng, K, V, 0, Q)
        u1, o1 = ko.verify_item(S0, q, k, v, g, rb, a_log, dt, -5.0, K ** -0.5)
        u2, o2 = ko.verify_chunked(S0, q, k, v, g, rb, a_log, dt, -5.0, K ** -0.5)
        np.testing.assert_allclose(u2, u1, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(o2, o1, rtol=1e-11, atol=1e-12)


def test_boundary_state_is_prefix_replay():
    rng = np.random.default_rng(3)
    S0, u, kr, gr, *_, a_log, dt = _toy(rng, 4, 3, 6, 1)
    S_n, _ = ko.replay_item(S0, u, kr, gr, 6, a_log, dt, -5.0)
    for m in range(1, 9):
        _, S_m = ko.replay_item(S0, u, kr, gr, 6, a_log, dt, -5.0, m=m)
        ref = ko.replay_closed_form(S0, u, kr, gr, min(m, 6), a_log, dt, -5.0)
        np.testing.assert_allclose(S_m, ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S_m, S_n, rtol=1e-12)


# ---------------------------------------------------------------------------
# special cases reducing to textbook routines
# ---------------------------------------------------------------------------

def test_beta_zero_is_a_plain_decayed_gemv():
    # beta = 0 (raw_beta = -inf) and no decay (lower_bound = 0): u = 0 and
    # o_t = S qn_t, one matrix-vector product with the normalised query.
    rng = np.random.default_rng(11)
    K, V, Q = 5, 3, 4
    S0, _, _, _, q, k, v, g, _, a_log, dt = _toy(rng, K, V, 0, Q)
    rb = np.full(Q, -np.inf)
    u, o = ko.verify_item(S0, q, k, v, g, rb, a_log, dt, 0.0, 0.7)
    np.testing.assert_array_equal(u, 0.0)
    qn = q / np.sqrt(np.linalg.norm(q, axis=1, keepdims=True) ** 2 + 1e-6)
    np.testing.assert_allclose(o, 0.7 * qn @ S0.T, rtol=1e-13)


def test_delta_rule_with_unit_step_writes_v_at_k():
    # lower_bound = 0 and beta = 1 reduce each token to the delta rule with a
    # unit step: afterwards S kn_t = v_t (up to the 1e-6 in the norm).  With
    # q_t = k_t and q_scale = 1 the output is therefore v_t.
    rng = np.random.default_rng(5)
    K, V, Q = 7, 3, 6
    S0, _, _, _, _, k, v, g, _, a_log, dt = _toy(rng, K, V, 0, Q)
    u, o = ko.verify_item(S0, k, k, v, g, np.full(Q, np.inf), a_log, dt, 0.0, 1.0)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-5 * np.abs(v).max())
    # and the correction is exactly the residual against the current state
    S = S0.copy()
    kn = k / np.sqrt((k * k).sum(1, keepdims=True) + 1e-6)
    for t in range(Q):
        np.testing.assert_allclose(u[t], v[t] - S @ kn[t], rtol=1e-12, atol=1e-12)
        S = S + np.outer(u[t], kn[t])


def test_zero_state_single_token():
    # S = 0, one token: u = beta v, o = beta v (kn . qn)
    K, V = 4, 3
    q = np.array([[1.0, 2.0, 0.0, -1.0]])
    k = np.array([[0.5, -1.0, 2.0, 0.0]])
    v = np.array([[1.0, -2.0, 3.0]])
    u, o = ko.verify_item(np.zeros((V, K)), q, k, v, np.zeros((1, K)), np.array([0.0]),
                          0.0, np.zeros(K), -5.0, 0.25)
    kn = k[0] / math.sqrt(k[0] @ k[0] + 1e-6)
    qn = q[0] / math.sqrt(q[0] @ q[0] + 1e-6) * 0.25
    np.testing.assert_allclose(u[0], 0.5 * v[0], rtol=1e-15)
    np.testing.assert_allclose(o[0], 0.5 * v[0] * (kn @ qn), rtol=1e-14)


def test_q_scale_is_linear_and_inputs_are_normalised():
    rng = np.random.default_rng(9)
    K, V, Q = 8, 5, 3
    S0, _, _, _, q, k, v, g, rb, a_log, dt = _toy(rng, K, V, 0, Q)
    u1, o1 = ko.verify_item(S0, q, k, v, g, rb, a_log, dt, -5.0, 1.0)
    u2, o2 = ko.verify_item(S0, q, k, v, g, rb, a_log, dt, -5.0, 3.0)
    np.testing.assert_allclose(o2, 3.0 * o1, rtol=1e-13)
    np.testing.assert_allclose(u2, u1, rtol=1e-14)
    # scaling the raw q or k by a constant changes nothing (normalised inputs)
    u3, o3 = ko.verify_item(S0, 4.0 * q, 2.0 * k, v, g, rb, a_log, dt, -5.0, 1.0)
    np.testing.assert_allclose(o3, o1, rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(u3, u1, rtol=1e-5, atol=1e-7)


# ---------------------------------------------------------------------------
# invariants of the protocol
# ---------------------------------------------------------------------------

def _case(**kw):
    base = dict(B=6, H=3, Q=3, slots=16, seed=21, K=8, V=6)
    base.update(kw)
    return synth.replay_verify_case(**base)


def _run(case, pending=True, **kw):
    c = {key: (val.copy() if isinstance(val, np.ndarray) else val) for key, val in case.items()}
    B, H, Q = c["B"], c["H"], c["Q"]
    out = np.zeros(c["v"].shape, dtype=np.uint16)
    ko.replay_verify(q=c["q"], k=c["k"], v=c["v"], raw_g=c["raw_g"], raw_beta=c["raw_beta"],
                     A_log=c["A_log"], dt_bias=c["dt_bias"], lower_bound=c["lower_bound"],
                     q_scale=c["q_scale"], state=c["state"], state_slots=c["state_slots"],
                     record_rows=c["record_rows"], corr=c["corr"], key_gate=c["key_gate"],
                     out=out, B=B, H=H, Q=Q, pending=c["pending"] if pending else None, **kw)
    c["out"] = out
    return c


def test_n_zero_leaves_the_checkpoint_bit_identical():
    case = _case()
    case["pending"][:] = 0
    after = _run(case)
    np.testing.assert_array_equal(after["state"], case["state"])
    # and the stock verify (no pending) never writes it
    after = _run(_case(), pending=False)
    np.testing.assert_array_equal(after["state"], _case()["state"])
    # align: with n = 0 the boundary slot is not written either; with n > 0 it
    # receives S_min(m, n)
    case = _case(boundary_frac=0.5)
    crossing = case["boundary_slots"] > 0
    assert crossing.any()
    case["pending"][:] = 0
    after = _run(case, boundary_slots=case["boundary_slots"], boundary_lens=case["boundary_lens"])
    np.testing.assert_array_equal(after["state"], case["state"])
    case["pending"][:] = case["RQ"]
    after = _run(case, boundary_slots=case["boundary_slots"], boundary_lens=case["boundary_lens"])
    for b in np.flatnonzero(crossing & (case["record_rows"] >= 0)):
        for h in range(case["H"]):
            rec, m = case["record_rows"][b], min(case["boundary_lens"][b], case["RQ"])
            K = case["q"].shape[-1]
            ref = ko.replay_closed_form(
                case["state"][case["state_slots"][b], h].astype(np.float64),
                case["corr"][rec, h, :m].astype(np.float64),
                ko.bf16_to_f64(case["key_gate"][rec, h, :m, :K]),
                ko.bf16_to_f64(case["key_gate"][rec, h, :m, K:]), m,
                float(case["A_log"][h]), case["dt_bias"][h].astype(np.float64), case["lower_bound"])
            np.testing.assert_allclose(after["state"][case["boundary_slots"][b], h], ref,
                                       rtol=1e-6, atol=1e-7)


def test_pending_is_clamped():
    case = _case(Q=3)
    rows = case["record_rows"]
    live = rows >= 0
    case["pending"][rows[live]] = case["RQ"]
    a = _run(case)
    case["pending"][rows[live]] = case["RQ"] + 5
    b = _run(case)
    np.testing.assert_array_equal(a["state"], b["state"])
    np.testing.assert_array_equal(a["out"], b["out"])
    case["pending"][:] = -4
    c = _run(case)
    np.testing.assert_array_equal(c["state"], case["state"])


def test_inert_and_recordless_rows():
    case = _case(B=8, padding_frac=0.25, no_record_frac=0.25)
    after = _run(case)
    slots, rows = case["state_slots"], case["record_rows"]
    Q = case["Q"]
    for b in range(case["B"]):
        tok = slice(b * Q, (b + 1) * Q)
        if slots[b] <= 0:
            np.testing.assert_array_equal(after["out"][tok], 0)
        if rows[b] < 0 and slots[b] > 0:
            # no record row: no replay, checkpoint untouched
            np.testing.assert_array_equal(after["state"][slots[b]], case["state"][slots[b]])
    # record rows not referenced by a live request are never written
    used = set(int(r) for b, r in enumerate(rows) if r >= 0 and slots[b] > 0)
    for r in range(case["corr"].shape[0]):
        if r not in used:
            np.testing.assert_array_equal(after["corr"][r], case["corr"][r])
            np.testing.assert_array_equal(after["key_gate"][r], case["key_gate"][r])


def test_fused_step_equals_commit_then_verify():
    # One step of replay + verify == the commit of the pending tokens
    # (in place, FP32) followed by the stock verify of the new window.
    case = _case(B=5, H=2, Q=4, K=16, V=12)
    fused = _run(case)
    split = {key: (val.copy() if isinstance(val, np.ndarray) else val) for key, val in case.items()}
    rows = split["record_rows"]
    lens = np.array([split["pending"][r] if r >= 0 else 0 for r in rows], dtype=np.int32)
    layer = dict(state=split["state"], corr=split["corr"], key_gate=split["key_gate"])
    ko.commit(layers=[layer], A_log=split["A_log"][None], dt_bias=split["dt_bias"][None],
              sources=split["state_slots"], commit_lens=np.minimum(lens, split["RQ"]),
              destinations=split["state_slots"], lower_bound=split["lower_bound"],
              Q=split["RQ"], B=split["B"], H=split["H"], record_rows=rows)
    verified = _run(split, pending=False)
    np.testing.assert_allclose(verified["state"], fused["state"], rtol=0, atol=1e-6)
    np.testing.assert_allclose(ko.bf16_to_f64(verified["out"]), ko.bf16_to_f64(fused["out"]),
                               rtol=1e-2, atol=1e-2)
    np.testing.assert_allclose(verified["corr"], fused["corr"], rtol=1e-5, atol=1e-5)
    np.testing.assert_array_equal(verified["key_gate"], fused["key_gate"])


def test_deferred_then_flushed_equals_eager_commit():
    # Step 1 verifies (records written, checkpoint kept); sampling accepts a_b
    # tokens.  Eager: commit a_b now.  Deferred: defer (pending <- a_b), then
    # the flush plan and the same commit in place.  The states must agree
    # bit-exactly, the integer arrays too.
    case = _case(B=6, H=2, Q=4, K=8, V=8, no_record_frac=0.2, padding_frac=0.2)
    step1 = _run(case, pending=False)
    rng = np.random.default_rng(2)
    B, Q = case["B"], case["Q"]
    accepted = rng.integers(0, Q + 1, size=B).astype(np.int32)
    slots, rows = case["state_slots"], case["record_rows"]

    eager_state = step1["state"].copy()
    eager_lens = np.where((rows >= 0) & (slots > 0), accepted, 0).astype(np.int32)
    ko.commit(layers=[dict(state=eager_state, corr=step1["corr"], key_gate=step1["key_gate"])],
              A_log=case["A_log"][None], dt_bias=case["dt_bias"][None], sources=slots,
              commit_lens=eager_lens, destinations=slots, lower_bound=case["lower_bound"],
              Q=Q, B=B, H=case["H"], record_rows=rows)

    pending = np.full(case["pending"].shape, 77, dtype=np.int32)
    lens = accepted.copy()
    ko.defer_commit(state_slots=slots, commit_lens=lens, record_rows=rows, pending=pending, B=B)
    live = (rows >= 0) & (slots > 0)
    np.testing.assert_array_equal(lens[live], 0)
    np.testing.assert_array_equal(pending[rows[live]], accepted[live])
    plan = dict(commit_lens=np.zeros(B, np.int32), final_slots=np.zeros(B, np.int32),
                boundary_slots=np.ones(B, np.int32), boundary_lens=np.ones(B, np.int32))
    ko.flush_plan(state_slots=slots, record_rows=rows, pending=pending, B=B, Q=Q, **plan)
    np.testing.assert_array_equal(plan["commit_lens"], eager_lens)
    np.testing.assert_array_equal(plan["final_slots"], slots)
    deferred_state = step1["state"].copy()
    ko.commit(layers=[dict(state=deferred_state, corr=step1["corr"], key_gate=step1["key_gate"])],
              A_log=case["A_log"][None], dt_bias=case["dt_bias"][None], sources=slots,
              commit_lens=plan["commit_lens"], destinations=plan["final_slots"],
              boundaries=plan["boundary_slots"], boundary_lens=plan["boundary_lens"],
              lower_bound=case["lower_bound"], Q=Q, B=B, H=case["H"], record_rows=rows)
    np.testing.assert_array_equal(deferred_state, eager_state)
    # ... and the fused step from the deferred checkpoint replays the same
    nxt = dict(step1)
    nxt["state"] = step1["state"].copy()
    nxt["pending"] = pending
    fused = _run(nxt)
    for b in range(B):
        if live[b] and accepted[b] > 0:
            np.testing.assert_allclose(fused["state"][slots[b]], eager_state[slots[b]],
                                       rtol=0, atol=1e-6)


def test_commit_skips_dead_rows_and_writes_boundary():
    c = synth.commit_case(L=2, B=12, H=2, Q=4, slots=40, seed=5, K=8, V=8,
                          state_dtype="f32", boundary_frac=0.5)
    layers = [{k: v.copy() for k, v in lay.items()} for lay in c["layers"]]
    ko.commit(layers=layers, A_log=c["A_log"], dt_bias=c["dt_bias"], sources=c["sources"],
              commit_lens=c["commit_lens"], destinations=c["destinations"],
              boundaries=c["boundaries"], boundary_lens=c["boundary_lens"],
              lower_bound=c["lower_bound"], Q=c["Q"], B=c["B"], H=c["H"])
    written = set()
    for b in range(c["B"]):
        n, src, dst = c["commit_lens"][b], c["sources"][b], c["destinations"][b]
        if n > 0 and src > 0 and dst > 0:
            written.add(int(dst))
            if c["boundary_lens"][b] > 0 and c["boundaries"][b] > 0:
                written.add(int(c["boundaries"][b]))
                for l, lay in enumerate(layers):
                    for h in range(c["H"]):
                        m = min(int(c["boundary_lens"][b]), int(n))
                        src_page = c["layers"][l]["state"][src, h].astype(np.float64)
                        ref = ko.replay_closed_form(
                            src_page, c["layers"][l]["corr"][b, h, :m].astype(np.float64),
                            ko.bf16_to_f64(c["layers"][l]["key_gate"][b, h, :m, :8]),
                            ko.bf16_to_f64(c["layers"][l]["key_gate"][b, h, :m, 8:]), m,
                            float(c["A_log"][l, h]), c["dt_bias"][l, h].astype(np.float64),
                            c["lower_bound"])
                        np.testing.assert_allclose(lay["state"][c["boundaries"][b], h], ref,
                                                   rtol=1e-6, atol=1e-7)
    for l, lay in enumerate(layers):
        for s in range(lay["state"].shape[0]):
            if s not in written:
                np.testing.assert_array_equal(lay["state"][s], c["layers"][l]["state"][s])


# ---------------------------------------------------------------------------
# bookkeeping, against the hand-worked fixture
# ---------------------------------------------------------------------------

def test_bookkeeping_hand_worked():
    g = json.load(open(os.path.join(GOLDEN, "bookkeeping_hand.json")))
    d = g["defer"]
    for eager, key in ((np.array(d["eager"], np.uint8), "expect_eager"), (None, "expect_no_eager")):
        pending = np.array(d["pending"], np.int32)
        lens = np.array(d["commit_lens"], np.int32)
        ko.defer_commit(state_slots=np.array(d["state_slots"], np.int32), commit_lens=lens,
                        record_rows=np.array(d["record_rows"], np.int32), pending=pending,
                        B=len(lens), eager=eager)
        np.testing.assert_array_equal(pending, d[key]["pending"])
        np.testing.assert_array_equal(lens, d[key]["commit_lens"])
    f = g["flush"]
    B = len(f["state_slots"])
    plan = {k: np.full(B, 99, np.int32) for k in f["expect"]}
    ko.flush_plan(state_slots=np.array(f["state_slots"], np.int32),
                  record_rows=np.array(f["record_rows"], np.int32),
                  pending=np.array(f["pending"], np.int32), B=B, Q=f["Q"], **plan)
    for k, v in f["expect"].items():
        np.testing.assert_array_equal(plan[k], v)


# ---------------------------------------------------------------------------
# several decode steps: the stock recurrence and the deferred protocol
# ---------------------------------------------------------------------------

_WINDOW_KEYS = ("q", "k", "v", "raw_g", "raw_beta")


def _decode_case(**kw):
    base = dict(B=6, H=2, Q=3, slots=16, steps=7, seed=31, K=8, V=6)
    base.update(kw)
    return synth.decode_loop_case(**base)


def _stock(case, **kw):
    return ko.decode_stock(windows=case["windows"], window_of_step=case["window_of_step"],
                           accepted=case["accepted"], A_log=case["A_log"],
                           dt_bias=case["dt_bias"], lower_bound=case["lower_bound"],
                           q_scale=case["q_scale"], state=case["state"],
                           state_slots=case["state_slots"], B=case["B"], H=case["H"],
                           Q=case["Q"], **kw)


def _oracle_protocol(case, flush_every):
    """The deferred protocol run by the oracle's own step functions: a fused
    step (or the stock verify right after a flush), then defer with the eager
    rows committed at once, and a flush every ``flush_every`` steps and at the
    end.  Returns (FP64 outputs per step, the final pool)."""
    c = {key: (val.copy() if isinstance(val, np.ndarray) else val) for key, val in case.items()}
    B, H, Q = c["B"], c["H"], c["Q"]
    slots, rows = c["state_slots"], c["record_rows"]
    layer = dict(state=c["state"], corr=c["corr"], key_gate=c["key_gate"])
    common = dict(A_log=c["A_log"][None], dt_bias=c["dt_bias"][None],
                  lower_bound=c["lower_bound"], Q=c["RQ"], B=B, H=H, record_rows=rows)
    outs, flushed = [], False
    steps = c["accepted"].shape[0]
    for s in range(steps):
        win = {key: c["windows"][key][c["window_of_step"][s]] for key in _WINDOW_KEYS}
        out = np.zeros(win["v"].shape, dtype=np.uint16)
        out64 = np.zeros(win["v"].shape)
        ko.replay_verify(**win, A_log=c["A_log"], dt_bias=c["dt_bias"],
                         lower_bound=c["lower_bound"], q_scale=c["q_scale"], state=c["state"],
                         state_slots=slots, record_rows=rows, corr=c["corr"],
                         key_gate=c["key_gate"], out=out, B=B, H=H, Q=Q,
                         pending=None if flushed else c["pending"], out_f64=out64)
        outs.append(out64)
        lens = c["accepted"][s].copy()
        eager = c["eager"][s]
        ko.defer_commit(state_slots=slots, commit_lens=lens, record_rows=rows,
                        pending=c["pending"], B=B, eager=eager)
        if eager.any():
            ko.commit(layers=[layer], sources=slots, commit_lens=lens, destinations=slots,
                      **common)
        flushed = False
        if (s + 1) % flush_every == 0 or s == steps - 1:
            plan = dict(commit_lens=np.zeros(B, np.int32), final_slots=np.zeros(B, np.int32),
                        boundary_slots=np.zeros(B, np.int32),
                        boundary_lens=np.zeros(B, np.int32))
            ko.flush_plan(state_slots=slots, record_rows=rows, pending=c["pending"], B=B, Q=Q,
                          **plan)
            ko.commit(layers=[layer], sources=slots, commit_lens=plan["commit_lens"],
                      destinations=plan["final_slots"], boundaries=plan["boundary_slots"],
                      boundary_lens=plan["boundary_lens"], **common)
            flushed = True
    return outs, c["state"]


@pytest.mark.parametrize("flush_every,eager_frac", [(3, 0.3), (100, 0.0), (1, 0.5)])
def test_deferred_protocol_equals_stock_recurrence(flush_every, eager_frac):
    # Records, pending replays, eager commits and flushes are a schedule of
    # the stock recurrence: outputs and final checkpoints agree with it up to
    # the FP32 roundings of records and checkpoints.
    case = _decode_case(padding_frac=0.2, eager_frac=eager_frac)
    assert case["accepted"].any() and (case["accepted"] < case["Q"]).any()
    outs, pool = _oracle_protocol(case, flush_every)
    ref_outs, finals = _stock(case)
    for s, o in enumerate(outs):
        scale = np.abs(ref_outs[s]).max()
        assert np.abs(o - ref_outs[s]).max() <= 1e-5 * scale, f"step {s}"
    live = [(b, h) for b in range(case["B"]) for h in range(case["H"])
            if case["state_slots"][b] > 0]
    assert set(finals) == set(live)
    for (b, h), S in finals.items():
        got = pool[case["state_slots"][b], h].astype(np.float64)
        assert np.abs(got - S).max() <= 1e-5 * np.abs(S).max(), (b, h)
    for b in range(case["B"]):
        if case["state_slots"][b] <= 0:
            assert not any(o[b * case["Q"]:(b + 1) * case["Q"]].any() for o in ref_outs)


def test_decode_stock_nothing_accepted_keeps_the_checkpoint():
    # No token accepted: the state never moves, so every step's outputs are
    # the one-window verify from the initial page.
    case = _decode_case()
    case["accepted"][:] = 0
    ref_outs, finals = _stock(case)
    for (b, h), S in finals.items():
        np.testing.assert_array_equal(S, case["state"][case["state_slots"][b], h])
    for s in range(case["steps"]):
        step = dict(case)
        for key in _WINDOW_KEYS:
            step[key] = case["windows"][key][case["window_of_step"][s]]
        step["state"] = case["state"].copy()
        out64 = np.zeros(ref_outs[s].shape)
        _run(step, pending=False, out_f64=out64)
        np.testing.assert_allclose(ref_outs[s], out64, rtol=0, atol=1e-12)


def test_decode_stock_without_decay_or_writes_is_a_fixed_gemv():
    # lower_bound = 0 gives d = 1 and beta = sigmoid(-inf) = 0 gives u = 0:
    # the state is S_0 forever and o_t = S_0 qn_t at every step.
    case = _decode_case(B=3, H=2, Q=2, K=6, V=5)
    case["lower_bound"] = 0.0
    case["windows"]["raw_beta"][:] = 0xFF80  # BF16 -inf
    ref_outs, finals = _stock(case)
    K = case["windows"]["q"].shape[-1]
    for (b, h), S in finals.items():
        S0 = case["state"][case["state_slots"][b], h].astype(np.float64)
        np.testing.assert_array_equal(S, S0)
        for s in range(case["steps"]):
            w = case["window_of_step"][s]
            for t in range(case["Q"]):
                q = ko.bf16_to_f64(case["windows"]["q"][w, b * case["Q"] + t, h])
                qn = q / math.sqrt(float(q @ q) + 1e-6) * case["q_scale"]
                np.testing.assert_allclose(ref_outs[s][b * case["Q"] + t, h], S0 @ qn,
                                           rtol=1e-13, atol=1e-15)
    assert K == 6


def test_decode_stock_full_acceptance_is_one_long_recurrence():
    # Accepting every token of every window makes the steps one sequential
    # recurrence over the concatenated windows: step s's outputs are the
    # long verify's outputs at positions s*Q .. s*Q + Q - 1.
    case = _decode_case(B=1, H=1, Q=3, steps=5)
    case["accepted"][:] = case["Q"]
    ref_outs, finals = _stock(case)
    Q, steps = case["Q"], case["steps"]
    seq = {key: np.concatenate([case["windows"][key][case["window_of_step"][s]]
                                for s in range(steps)])[:, 0] for key in _WINDOW_KEYS}
    S0 = case["state"][case["state_slots"][0], 0]
    _, o = ko.verify_item(S0, *(ko.bf16_to_f64(seq[key]) for key in _WINDOW_KEYS),
                          float(case["A_log"][0]), case["dt_bias"][0].astype(np.float64),
                          case["lower_bound"], case["q_scale"])
    for s in range(steps):
        np.testing.assert_allclose(ref_outs[s][:, 0], o[s * Q:(s + 1) * Q], rtol=1e-12,
                                   atol=1e-14)


# ---------------------------------------------------------------------------
# windows of different lengths (query_start_loc)
# ---------------------------------------------------------------------------

def test_full_windows_through_query_start_loc_equal_the_uniform_step():
    case = _case(padding_frac=0.2, no_record_frac=0.2)
    B, Q = case["B"], case["Q"]
    uni = _run(case)
    var = _run(case, query_start_loc=np.arange(B + 1, dtype=np.int32) * Q)
    for key in ("out", "state", "corr", "key_gate"):
        np.testing.assert_array_equal(var[key], uni[key], err_msg=key)


def test_short_windows_are_prefixes_of_the_full_window():
    # The recurrence is causal: a request's first q_b outputs and corrections
    # do not depend on its later tokens, so verifying only the packed first
    # q_b tokens gives the full window's first q_b results; records past q_b
    # are left as they were, and the replay does not depend on the window.
    case = _case(B=7, H=2, Q=4, padding_frac=0.15, no_record_frac=0.15)
    B, Q, K = case["B"], case["Q"], case["k"].shape[-1]
    q_lens = np.array([0, 4, 1, 3, 2, 0, 4], dtype=np.int32)
    uni = _run(case)
    packed = synth.pack_windows(case, q_lens)
    vcase = dict(case)
    vcase.update(packed)
    qsl = packed["query_start_loc"]
    assert qsl[-1] == q_lens.sum() == vcase["q"].shape[0]
    var = _run(vcase, query_start_loc=qsl)
    np.testing.assert_array_equal(var["state"], uni["state"])
    for b in range(B):
        qb = int(q_lens[b])
        np.testing.assert_array_equal(var["out"][qsl[b]:qsl[b + 1]],
                                      uni["out"][b * Q:b * Q + qb], err_msg=f"request {b}")
        rec = int(case["record_rows"][b])
        if rec < 0:
            continue
        if case["state_slots"][b] > 0:
            np.testing.assert_array_equal(var["corr"][rec, :, :qb], uni["corr"][rec, :, :qb])
            np.testing.assert_array_equal(var["key_gate"][rec, :, :qb],
                                          uni["key_gate"][rec, :, :qb])
        np.testing.assert_array_equal(var["corr"][rec, :, qb:], case["corr"][rec, :, qb:])
        np.testing.assert_array_equal(var["key_gate"][rec, :, qb:],
                                      case["key_gate"][rec, :, qb:])
    assert K == 8


def test_invalid_window_leaves_the_request_untouched():
    case = _case(B=4, H=2, Q=3)
    case["pending"][:] = 2
    B, Q = case["B"], case["Q"]
    q_lens = np.array([2, 3, 1, 3], dtype=np.int32)
    packed = synth.pack_windows(case, q_lens)
    vcase = dict(case)
    vcase.update(packed)
    qsl = packed["query_start_loc"].copy()
    qsl[1] = qsl[2] - (Q + 1)  # request 1: a window longer than Q
    qsl[4] = vcase["q"].shape[0] + 1  # request 3: past the activations
    var = _run(vcase, query_start_loc=qsl)
    for b in (1, 3):
        slot, rec = int(case["state_slots"][b]), int(case["record_rows"][b])
        assert slot > 0 and rec >= 0
        np.testing.assert_array_equal(var["state"][slot], case["state"][slot])
        np.testing.assert_array_equal(var["corr"][rec], case["corr"][rec])
        np.testing.assert_array_equal(var["key_gate"][rec], case["key_gate"][rec])
    # the valid requests are still served (their checkpoints replayed)
    for b in (0, 2):
        slot = int(case["state_slots"][b])
        assert not np.array_equal(var["state"][slot], case["state"][slot])


# ---------------------------------------------------------------------------
# the model layer: convolution and SiLU, gate projection, gated RMSNorm
# ---------------------------------------------------------------------------

def _layer(**kw):
    base = dict(B=3, H=2, Q=4, slots=8, seed=71)
    base.update(kw)
    return synth.layer_case(**base)


def _prologue(c, pending=True, conv_state=None):
    state = (c["conv_state"] if conv_state is None else conv_state).copy()
    out = ko.layer_prologue(x=c["x"], conv_weight=c["conv_weight"], conv_bias=c["conv_bias"],
                            conv_state=state, f_a=c["f_a"], f_b=c["f_b"],
                            state_slots=c["state_slots"], record_rows=c["record_rows"],
                            pending=c["pending"] if pending else None, B=c["B"], H=c["H"],
                            Q=c["Q"])
    return out, state


def _one_hot_taps(c, i):
    w = np.zeros(c["conv_weight"].shape, dtype=np.float32)
    w[:, i, :] = 1.0
    c["conv_weight"] = _bits(w)
    c["conv_bias"] = None


@pytest.mark.parametrize("n", [0, 1, 3])
def test_conv_taps_and_window_roll(n):
    # With only tap 0 (the oldest) the output at t is SiLU of s[t], the
    # sequence s = window[n-1 .. n+1] (from 0 when n = 0) followed by x; with
    # only tap 3 (the current token) it is SiLU of x_t.  So the tap-0 layer
    # on x equals the tap-3 layer on the sequence written out as inputs.
    c = _layer()
    c["pending"][:] = n
    B, H, Q, D = c["B"], c["H"], c["Q"], c["H"] * 128
    _one_hot_taps(c, 0)
    (q0, k0, v0, _), _ = _prologue(c)
    shifted = dict(c)
    _one_hot_taps(shifted, 3)
    x2 = c["x"].copy()
    off = n - 1 if n > 0 else 0
    for b in range(B):
        slot = int(c["state_slots"][b])
        if slot <= 0:
            continue
        window = c["conv_state"][slot]                       # [3D, RQ + 2]
        seq = np.concatenate([window[:, off:off + 3], c["x"][b * Q:(b + 1) * Q].T], axis=1)
        x2[b * Q:(b + 1) * Q] = seq[:, :Q].T
    shifted["x"] = x2
    (q3, k3, v3, _), _ = _prologue(shifted)
    for a, b_ in ((q0, q3), (k0, k3), (v0, v3)):
        np.testing.assert_array_equal(a, b_)
    assert D == 256


def test_silu_is_odd_up_to_the_identity():
    # silu(z) - silu(-z) = z: negating x flips every current-tap output by
    # the input itself (within the BF16 rounding of both outputs).
    c = _layer(bias=False)
    _one_hot_taps(c, 3)
    (q, k, v, _), _ = _prologue(c)
    neg = dict(c)
    neg["x"] = c["x"] ^ np.uint16(0x8000)  # exact negation of BF16 bits
    (qn, kn, vn, _), _ = _prologue(neg)
    B, H, Q, D = c["B"], c["H"], c["Q"], c["H"] * 128
    xs = ko.bf16_to_f64(c["x"]).reshape(B * Q, 3, H, 128)
    live = np.repeat(c["state_slots"] > 0, Q)
    for part, (a, b_) in enumerate(((q, qn), (k, kn), (v, vn))):
        diff = ko.bf16_to_f64(a) - ko.bf16_to_f64(b_)
        ref = xs[:, part]
        err = np.abs(diff - ref)[live]
        bound = 2 * 2.0 ** -8 * np.abs(ref)[live] + 1e-30
        assert np.all(err <= bound + 2 * 2.0 ** -8 * np.abs(diff)[live])


def test_conv_bias_indexed_by_part_head_and_channel():
    # With every convolution weight zero the output is SiLU of the bias
    # alone.  The bias of (part p, head h, channel c) is the exact BF16 value
    # 2^(4 + p + 3 h) * (1 + c / 128): distinct for every (p, h, c), and at
    # least 16, where silu(b) = b / (1 + e^-b) lies within 1.2e-7 b of b, far
    # inside half a BF16 step (2^-9 b), so the output must be the bias bits
    # exactly -- with no appeal to the oracle's SiLU.  A bias indexed without
    # the part offset, by head only, or by channel only, gives other values.
    c = _layer()
    H, D = c["H"], c["H"] * 128
    c["conv_weight"] = np.zeros_like(c["conv_weight"])
    bias = np.zeros(3 * D, dtype=np.float32)
    for part in range(3):
        for h in range(H):
            ch = np.arange(128)
            bias[part * D + h * 128 + ch] = 2.0 ** (4 + part + 3 * h) * (1.0 + ch / 128.0)
    c["conv_bias"] = _bits(bias)
    assert len(np.unique(c["conv_bias"])) == 3 * D
    for pending in (True, False):
        (q, k, v, _), _ = _prologue(c, pending=pending)
        B, Q = c["B"], c["Q"]
        for b in range(B):
            rows = slice(b * Q, (b + 1) * Q)
            if c["state_slots"][b] <= 0:
                continue
            for part, out in enumerate((q, k, v)):
                want = c["conv_bias"][part * D:(part + 1) * D].reshape(H, 128)
                np.testing.assert_array_equal(out[rows], np.broadcast_to(want, (Q, H, 128)))


def test_new_window_is_taps_then_inputs():
    c = _layer()
    c["pending"][:] = 2
    _, state = _prologue(c)
    Q, RQ = c["Q"], c["RQ"]
    for b in range(c["B"]):
        slot = int(c["state_slots"][b])
        if slot <= 0:
            continue
        old = c["conv_state"][slot]
        np.testing.assert_array_equal(state[slot][:, 0], old[:, 2])   # window[n-1+1], n = 2
        np.testing.assert_array_equal(state[slot][:, 1], old[:, 3])
        np.testing.assert_array_equal(state[slot][:, 2:2 + Q], c["x"][b * Q:(b + 1) * Q].T)
        np.testing.assert_array_equal(state[slot][:, 2 + Q:], old[:, 2 + Q:])
    assert RQ == Q


def test_gate_projection_with_unit_rows_copies_the_activations():
    # Row f of head h's f_b block is the unit vector at column (f + 1 + h) mod
    # 128, so raw_g[t, h, f] = f_a[t, (f + 1 + h) mod 128] exactly: a
    # transposed product or a head mix-up picks other columns.
    c = _layer()
    fb = np.zeros((c["H"] * 128, 128), dtype=np.float32)
    f = np.arange(128)
    for h in range(c["H"]):
        fb[h * 128 + f, (f + 1 + h) % 128] = 1.0
    c["f_b"] = _bits(fb)
    (_, _, _, g), _ = _prologue(c)
    Q = c["Q"]
    for b in range(c["B"]):
        if c["state_slots"][b] <= 0:
            assert not g[b * Q:(b + 1) * Q].any()
            continue
        for h in range(c["H"]):
            np.testing.assert_array_equal(g[b * Q:(b + 1) * Q, h],
                                          c["f_a"][b * Q:(b + 1) * Q][:, (f + 1 + h) % 128])


def test_gated_norm_closed_form_and_scale_invariance():
    T, H = 3, 2
    w = np.linspace(0.5, 1.5, 128).astype(np.float32)
    c0 = 0.75
    o = np.full((T, H, 128), c0, dtype=np.float32)
    gate0 = np.zeros((T, H * 128), dtype=np.float32)
    out = ko.layer_epilogue(o=_bits(o), gate=_bits(gate0), norm_weight=w, eps=1e-6)
    expect = c0 / math.sqrt(c0 * c0 + 1e-6) * w.astype(np.float64) * 0.5
    np.testing.assert_array_equal(out.reshape(T, H, 128), np.broadcast_to(ko.f64_to_bf16(expect),
                                                                         (T, H, 128)))
    rng = np.random.default_rng(3)
    o = _bits(np.ldexp(np.round(rng.standard_normal((T, H, 128)) * 64), -6).astype(np.float32))
    gate = _bits(np.round(rng.standard_normal((T, H * 128)) * 8).astype(np.float32) / 8)
    a = ko.layer_epilogue(o=o, gate=gate, norm_weight=w, eps=0.0)
    doubled = _bits(ko.bf16_to_f64(o).astype(np.float32) * 2)
    b = ko.layer_epilogue(o=doubled, gate=gate, norm_weight=w, eps=0.0)
    np.testing.assert_array_equal(a, b)
    minus_inf = np.full(gate.shape, 0xFF80, dtype=np.uint16)
    z = ko.layer_epilogue(o=o, gate=minus_inf, norm_weight=w, eps=1e-6)
    assert not np.any(ko.bf16_to_f64(z))


def test_decode_stock_uniform_windows_through_query_start_loc():
    case = _decode_case(padding_frac=0.2)
    B, Q, steps = case["B"], case["Q"], case["steps"]
    qsl = np.tile(np.arange(B + 1, dtype=np.int32) * Q, (steps, 1))
    a_outs, a_fin = _stock(case)
    b_outs, b_fin = _stock(case, query_start_loc=qsl)
    np.testing.assert_array_equal(a_outs, b_outs)
    assert a_fin.keys() == b_fin.keys()
    for key in a_fin:
        np.testing.assert_array_equal(a_fin[key], b_fin[key])
