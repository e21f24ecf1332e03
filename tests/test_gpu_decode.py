"""Several speculative decode steps on the GPU against the FP64 stock
recurrence.

The library runs the deferred protocol (fused replay + verify, defer, eager
commits, flushes, the stock verify after a flush) through the C ABI, with no
resynchronisation to the oracle between steps; the oracle runs the plain
recurrence (verify each window from the state, then advance the state by
the accepted tokens).  Every step's outputs are compared (rel-L2 <= 2e-3 on
BF16), and after the last flush every live checkpoint (max|dS| <=
1e-4 max|S|); the accumulated drift is printed.
"""
import numpy as np
import pytest

from linear_attention_speculative_recoverssm_gb300 import synth
from oracle import kda_oracle as ko

import kda_testutil as tu

pytestmark = pytest.mark.gpu

WINDOW_KEYS = ("q", "k", "v", "raw_g", "raw_beta")


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    from linear_attention_speculative_recoverssm_gb300 import _build, _lib
    assert torch.cuda.is_available()
    _build.build()
    _lib.load()


def _loop(case, d, split=0):
    from linear_attention_speculative_recoverssm_gb300 import DeferredRecoverSSM
    return DeferredRecoverSSM(d["state"], d["state_slots"], d["record_rows"], d["pending"],
                              d["corr"], d["key_gate"], d["A_log"], d["dt_bias"], Q=case["Q"],
                              lower_bound=case["lower_bound"], q_scale=case["q_scale"],
                              split=split, status=d["status"])


def _stock(case, items=None):
    return ko.decode_stock(windows=case["windows"], window_of_step=case["window_of_step"],
                           accepted=case["accepted"], A_log=case["A_log"],
                           dt_bias=case["dt_bias"], lower_bound=case["lower_bound"],
                           q_scale=case["q_scale"], state=case["state"],
                           state_slots=case["state_slots"], B=case["B"], H=case["H"],
                           Q=case["Q"], items=items)


def _drift(got_pool, case, finals):
    worst = 0.0
    for (b, h), S in finals.items():
        got = got_pool[case["state_slots"][b], h].astype(np.float64)
        worst = max(worst, float(np.abs(got - S).max() / np.abs(S).max()))
    return worst


@pytest.mark.parametrize("B,H,Q,steps,flush_every,eager_frac,split", [
    (16, 4, 4, 12, 5, 0.2, 0),
    (8, 2, 8, 24, 8, 0.0, 2),
    (5, 3, 1, 10, 4, 0.3, 0),
    (7, 2, 6, 9, 100, 0.1, 4),
])
def test_decode_loop_matches_stock_recurrence(B, H, Q, steps, flush_every, eager_frac, split):
    import torch
    case = synth.decode_loop_case(B=B, H=H, Q=Q, slots=2 * B + 4, steps=steps,
                                  seed=40 + B + Q, padding_frac=0.15, eager_frac=eager_frac)
    ref_outs, finals = _stock(case)
    d = tu.device_case(case)
    win = {key: tu.to_torch(case["windows"][key], "cuda") for key in WINDOW_KEYS}
    accepted = tu.to_torch(case["accepted"], "cuda")
    eager = tu.to_torch(case["eager"], "cuda")
    loop = _loop(case, d, split)
    for s in range(steps):
        w = int(case["window_of_step"][s])
        out = torch.zeros_like(d["out"])
        loop.verify(*(win[key][w] for key in WINDOW_KEYS), out)
        loop.accept(accepted[s].clone(), eager[s] if eager_frac > 0 else None)
        if (s + 1) % flush_every == 0 or s == steps - 1:
            loop.flush()
        torch.cuda.synchronize()
        tu.assert_out_close(tu.to_numpy(out), ko.f64_to_bf16(ref_outs[s]), what=f"step {s}",
                            Q=Q)
    assert int(tu.to_numpy(d["status"])[0]) == 0
    pool = tu.to_numpy(d["state"])
    for (b, h), S in finals.items():
        tu.assert_state_close(pool[case["state_slots"][b], h], S, what=f"item {(b, h)}")
    # pages no request uses are untouched
    used = set(int(x) for x in case["state_slots"] if x > 0)
    for slot in range(pool.shape[0]):
        if slot not in used:
            np.testing.assert_array_equal(pool[slot], case["state"][slot])
    print(f"\ndecode drift B={B} H={H} Q={Q} steps={steps}: "
          f"max|dS|/max|S| = {_drift(pool, case, finals):.2e}")


def test_decode_loop_full_size_graph_sampled():
    """The benchmark's decode workload (H=64, B=512, Q=8; a flush every 8
    steps) captured in a CUDA graph as the benchmark runs it, replayed twice;
    outputs of the last step and the final checkpoints compared on sampled
    items against the stock recurrence over all 16 steps."""
    import torch
    case = synth.make("decode-loop-f32-h64-b512-q8")
    B, H, Q, steps = case["B"], case["H"], case["Q"], case["steps"]
    cycles = 2
    d = tu.device_case(case)
    win = {key: tu.to_torch(case["windows"][key], "cuda") for key in WINDOW_KEYS}
    accepted0 = tu.to_torch(case["accepted"], "cuda")
    accepted = accepted0.clone()
    outs = [torch.zeros_like(d["out"]) for _ in range(steps)]
    loop = _loop(case, d)
    stream = torch.cuda.Stream()
    loop.stream = stream
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        accepted.copy_(accepted0)
        loop.flushed = True  # a cycle starts after a flush (or with nothing pending)
        for s in range(steps):
            w = int(case["window_of_step"][s])
            loop.verify(*(win[key][w] for key in WINDOW_KEYS), outs[s])
            loop.accept(accepted[s])
        loop.flush()
    for _ in range(cycles):
        graph.replay()
    torch.cuda.synchronize()
    assert int(tu.to_numpy(d["status"])[0]) == 0
    # the stock recurrence over both cycles (step s of a cycle uses window
    # s mod 2 and the cycle's accepted counts) on sampled items
    rng = np.random.default_rng(7)
    items = np.sort(rng.choice(B * H, size=24, replace=False))
    long_case = dict(case)
    long_case["accepted"] = np.concatenate([case["accepted"]] * cycles)
    long_case["window_of_step"] = np.concatenate([case["window_of_step"]] * cycles)
    ref_outs, finals = _stock(long_case, items=items)
    got_out = tu.to_numpy(outs[-1]).reshape(B, Q, H, 128)
    ref_last = ko.f64_to_bf16(ref_outs[-1]).reshape(B, Q, H, 128)
    pool_rows = {}
    for i in items:
        b, h = divmod(int(i), H)
        tu.assert_out_close(got_out[b, :, h], ref_last[b, :, h], what=f"item {i}")
        slot = int(case["state_slots"][b])
        if slot > 0:
            pool_rows[(b, h)] = tu.to_numpy(d["state"][slot, h])
            tu.assert_state_close(pool_rows[(b, h)], finals[(b, h)], what=f"item {i} state")
        else:
            assert not got_out[b, :, h].any()
    worst = max(float(np.abs(pool_rows[key].astype(np.float64) - S).max() / np.abs(S).max())
                for key, S in finals.items())
    print(f"\ndecode drift full size, {cycles * steps} steps: max|dS|/max|S| = {worst:.2e}")


def _varlen_steps(case, seed):
    """Each step's window repacked to q_b ~ U{1..Q} tokens per request
    (query_start_loc [steps, B + 1]), padded with zero rows to B*Q; the
    accepted counts limited to q_b."""
    B, Q, steps = case["B"], case["Q"], case["steps"]
    rng = np.random.default_rng(seed)
    q_lens = rng.integers(1, Q + 1, size=(steps, B)).astype(np.int32)
    packed = {key: np.zeros((steps,) + case["windows"][key].shape[1:], dtype=np.uint16)
              for key in WINDOW_KEYS}
    qsl = np.zeros((steps, B + 1), dtype=np.int32)
    for s in range(steps):
        w = int(case["window_of_step"][s])
        step = {key: case["windows"][key][w] for key in WINDOW_KEYS}
        step.update(B=B, Q=Q)
        pk = synth.pack_windows(step, q_lens[s])
        qsl[s] = pk["query_start_loc"]
        for key in WINDOW_KEYS:
            packed[key][s, :pk[key].shape[0]] = pk[key]
    case = dict(case)
    case["windows"] = packed
    case["window_of_step"] = np.arange(steps)
    case["accepted"] = np.minimum(case["accepted"], q_lens)
    return case, qsl


def test_decode_loop_variable_windows():
    """The deferred loop with each step's windows of 1..Q tokens."""
    import torch
    B, H, Q, steps = 12, 3, 6, 9
    case = synth.decode_loop_case(B=B, H=H, Q=Q, slots=2 * B + 4, steps=steps, seed=77,
                                  padding_frac=0.15, eager_frac=0.2)
    case, qsl = _varlen_steps(case, 78)
    ref_outs, finals = ko.decode_stock(
        windows=case["windows"], window_of_step=case["window_of_step"],
        accepted=case["accepted"], A_log=case["A_log"], dt_bias=case["dt_bias"],
        lower_bound=case["lower_bound"], q_scale=case["q_scale"], state=case["state"],
        state_slots=case["state_slots"], B=B, H=H, Q=Q, query_start_loc=qsl)
    d = tu.device_case(case)
    win = {key: tu.to_torch(case["windows"][key], "cuda") for key in WINDOW_KEYS}
    dq = tu.to_torch(qsl, "cuda")
    accepted = tu.to_torch(case["accepted"], "cuda")
    eager = tu.to_torch(case["eager"], "cuda")
    loop = _loop(case, d)
    for s in range(steps):
        out = torch.zeros((B * Q, H, 128), dtype=torch.bfloat16, device="cuda")
        loop.verify(*(win[key][s] for key in WINDOW_KEYS), out, query_start_loc=dq[s])
        loop.accept(accepted[s].clone(), eager[s])
        if (s + 1) % 4 == 0 or s == steps - 1:
            loop.flush()
        torch.cuda.synchronize()
        got = tu.to_numpy(out)
        n_tok = int(qsl[s, -1])
        tu.assert_out_close(got[:n_tok], ko.f64_to_bf16(ref_outs[s][:n_tok]), what=f"step {s}")
        assert not got[n_tok:].any()  # rows past the windows are never written
    assert int(tu.to_numpy(d["status"])[0]) == 0
    pool = tu.to_numpy(d["state"])
    for (b, h), S in finals.items():
        tu.assert_state_close(pool[case["state_slots"][b], h], S, what=f"item {(b, h)}")
