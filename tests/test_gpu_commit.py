"""Parity of the CUDA commit and bookkeeping kernels with the oracle.

Commit: BF16 pools within 1 BF16 ulp of the oracle's single RNE rounding
(and rel-L2 <= 2e-3), FP32 pools within max|dS| <= 1e-4 max|S|; every page
the oracle leaves alone bit-exact.  Bookkeeping: bit-exact.
"""
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


def _commit_both(c, align=True, record_rows=None, items=None):
    import torch
    from linear_attention_speculative_recoverssm_gb300 import (KDA_STATE_BF16, KDA_STATE_F32,
                                                               kda_commit, layer_tables)
    dev = "cuda"
    states = [tu.to_torch(lay["state"], dev) for lay in c["layers"]]
    corrs = [tu.to_torch(lay["corr"], dev) for lay in c["layers"]]
    kgs = [tu.to_torch(lay["key_gate"], dev) for lay in c["layers"]]
    tabs = layer_tables(states, corrs, kgs, dev)
    t = lambda a: None if a is None else tu.to_torch(a, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    bf16 = c["layers"][0]["state"].dtype == np.uint16
    kda_commit(*tabs, t(c["A_log"]), t(c["dt_bias"]), t(c["sources"]), t(c["commit_lens"]),
               t(c["destinations"]), state_dtype=KDA_STATE_BF16 if bf16 else KDA_STATE_F32,
               lower_bound=c["lower_bound"], L=c["L"], H=c["H"], B=c["B"], Q=c["Q"],
               n_slots=c["layers"][0]["state"].shape[0], n_rows=c["layers"][0]["corr"].shape[0],
               boundaries=t(c["boundaries"]) if align else None,
               boundary_lens=t(c["boundary_lens"]) if align else None,
               record_rows=t(record_rows), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_layers = [{k: v.copy() for k, v in lay.items()} for lay in c["layers"]]
    ko.commit(layers=ref_layers, A_log=c["A_log"], dt_bias=c["dt_bias"], sources=c["sources"],
              commit_lens=c["commit_lens"], destinations=c["destinations"],
              lower_bound=c["lower_bound"], Q=c["Q"], B=c["B"], H=c["H"],
              boundaries=c["boundaries"] if align else None,
              boundary_lens=c["boundary_lens"] if align else None, record_rows=record_rows,
              items=items)
    return [tu.to_numpy(s) for s in states], ref_layers


def _compare_pools(got_states, ref_layers, orig_layers):
    for l, (got, ref, orig) in enumerate(zip(got_states, ref_layers, orig_layers)):
        changed = np.any(ref["state"] != orig["state"], axis=(2, 3))
        np.testing.assert_array_equal(got[~changed], orig["state"][~changed],
                                      err_msg=f"layer {l}: untouched pages")
        if changed.any():
            if got.dtype == np.uint16:
                tu.assert_bf16_state_close(got[changed], ref["state"][changed], what=f"layer {l}")
            else:
                tu.assert_state_close(got[changed], ref["state"][changed], what=f"layer {l}")


@pytest.mark.parametrize("Q", [1, 4, 8])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("align", [True, False])
def test_commit(Q, dtype, align):
    c = synth.commit_case(L=3, B=24, H=4, Q=Q, slots=96, seed=500 + Q, state_dtype=dtype,
                          boundary_frac=0.4 if align else 0.0)
    got, ref = _commit_both(c, align=align)
    _compare_pools(got, ref, c["layers"])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_commit_many_heads(dtype):
    """H = 128 on few requests and two layers: a layer's slot spans 128
    pages, and the (layer, request, head) items of one request cover most of
    the grid."""
    c = synth.commit_case(L=2, B=3, H=128, Q=4, slots=8, seed=530, state_dtype=dtype,
                          boundary_frac=0.4)
    got, ref = _commit_both(c, align=True)
    _compare_pools(got, ref, c["layers"])


def test_commit_with_record_rows():
    c = synth.commit_case(L=2, B=16, H=2, Q=4, slots=64, seed=17, state_dtype="f32")
    rows = np.random.default_rng(1).permutation(16).astype(np.int32)
    rows[3] = -1
    got, ref = _commit_both(c, align=True, record_rows=rows)
    _compare_pools(got, ref, c["layers"])


def test_commit_full_size_sampled():
    """The standalone-commit workload (L=4, H=32, B=64, Q=4, BF16, align), in
    the benchmark's launch configuration, checked on sampled items."""
    c = synth.make("commit-bf16-l4-h32-b64-q4-align")
    L, B, H = c["L"], c["B"], c["H"]
    items = np.sort(np.random.default_rng(3).choice(L * B * H, size=256, replace=False))
    got, ref = _commit_both(c, align=True, items=items)
    for i in items:
        l, b, h = int(i) // (B * H), (int(i) // H) % B, int(i) % H
        for slot in (c["destinations"][b], c["boundaries"][b]):
            if slot > 0:
                tu.assert_bf16_state_close(got[l][slot, h], ref[l]["state"][slot, h],
                                           what=f"item {i} slot {slot}")


def test_bookkeeping_bit_exact():
    import torch
    from linear_attention_speculative_recoverssm_gb300 import kda_defer_commit, kda_flush_plan
    rng = np.random.default_rng(21)
    B, rows = 300, 400
    slots = rng.integers(-1, 6, size=B).astype(np.int32)
    record_rows = rng.permutation(rows)[:B].astype(np.int32)
    record_rows[rng.random(B) < 0.15] = -1
    lens = rng.integers(0, 9, size=B).astype(np.int32)
    pending = rng.integers(-3, 12, size=rows).astype(np.int32)
    eager = (rng.random(B) < 0.3).astype(np.uint8)
    for use_eager in (True, False):
        p_ref, l_ref = pending.copy(), lens.copy()
        ko.defer_commit(state_slots=slots, commit_lens=l_ref, record_rows=record_rows,
                        pending=p_ref, B=B, eager=eager if use_eager else None)
        dp, dl = tu.to_torch(pending, "cuda"), tu.to_torch(lens, "cuda")
        kda_defer_commit(tu.to_torch(slots, "cuda"), dl, tu.to_torch(record_rows, "cuda"), dp,
                         eager=tu.to_torch(eager, "cuda") if use_eager else None)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(tu.to_numpy(dp), p_ref)
        np.testing.assert_array_equal(tu.to_numpy(dl), l_ref)
    for Q in (1, 4, 8):
        plan_ref = {k: np.full(B, 55, np.int32) for k in
                    ("commit_lens", "final_slots", "boundary_slots", "boundary_lens")}
        ko.flush_plan(state_slots=slots, record_rows=record_rows, pending=pending, B=B, Q=Q,
                      **plan_ref)
        plan = {k: torch.full((B,), 55, dtype=torch.int32, device="cuda") for k in plan_ref}
        kda_flush_plan(tu.to_torch(slots, "cuda"), tu.to_torch(record_rows, "cuda"),
                       tu.to_torch(pending, "cuda"), plan["commit_lens"], plan["final_slots"],
                       plan["boundary_slots"], plan["boundary_lens"], Q=Q)
        torch.cuda.synchronize()
        for k in plan_ref:
            np.testing.assert_array_equal(tu.to_numpy(plan[k]), plan_ref[k], err_msg=k)


def test_deferred_then_flushed_equals_eager_on_gpu():
    """verify (records) -> defer -> flush plan -> FP32 commit equals the eager
    FP32 commit of the accepted tokens (bit-exact: same kernel, same inputs)."""
    import torch
    from linear_attention_speculative_recoverssm_gb300 import (KDA_STATE_F32, kda_commit,
                                                               kda_defer_commit, kda_flush_plan,
                                                               layer_tables)
    case = synth.replay_verify_case(B=20, H=4, Q=4, slots=32, seed=23, no_record_frac=0.15,
                                    padding_frac=0.1)
    d = tu.device_case(case)
    tu.gpu_step(case, d, replay=False)  # verify: records written, checkpoint kept
    accepted = tu.to_torch(np.random.default_rng(4).integers(0, 5, 20).astype(np.int32), "cuda")
    B, H, Q = 20, 4, 4
    n_slots, n_rows = case["state"].shape[0], case["corr"].shape[0]

    def commit(state, lens, dst, bslots=None, blens=None):
        tabs = layer_tables([state], [d["corr"]], [d["key_gate"]], "cuda")
        kda_commit(*tabs, d["A_log"], d["dt_bias"], d["state_slots"], lens, dst,
                   state_dtype=KDA_STATE_F32, lower_bound=case["lower_bound"], L=1, H=H, B=B,
                   Q=Q, n_slots=n_slots, n_rows=n_rows, boundaries=bslots, boundary_lens=blens,
                   record_rows=d["record_rows"])

    eager_state = d["state"].clone()
    live = (d["record_rows"] >= 0) & (d["state_slots"] > 0)
    commit(eager_state, torch.where(live, accepted, 0).to(torch.int32), d["state_slots"])
    lens = accepted.clone()
    kda_defer_commit(d["state_slots"], lens, d["record_rows"], d["pending"])
    plan = [torch.zeros(B, dtype=torch.int32, device="cuda") for _ in range(4)]
    kda_flush_plan(d["state_slots"], d["record_rows"], d["pending"], *plan, Q=Q)
    deferred_state = d["state"].clone()
    commit(deferred_state, plan[0], plan[1], plan[2], plan[3])
    torch.cuda.synchronize()
    assert torch.equal(deferred_state, eager_state)


def test_commit_mostly_dead_back_to_back():
    """FP32 pools (two stages), half the requests with a null source and
    many zero lengths, twenty launches back to back: each main warp waits
    for a dead item's stage phase before counting its read, so the read
    counts of two items sharing a stage never mix.  Every destination is a
    fresh slot, so every launch writes the same pages."""
    import torch
    from linear_attention_speculative_recoverssm_gb300 import KDA_STATE_F32, kda_commit, layer_tables
    c = synth.commit_case(L=2, B=96, H=16, Q=8, slots=400, seed=62, state_dtype="f32",
                          null_frac=0.5, in_place_frac=0.0, boundary_frac=0.25)
    orig = [{k: v.copy() for k, v in lay.items()} for lay in c["layers"]]
    dev = "cuda"
    states = [tu.to_torch(lay["state"], dev) for lay in c["layers"]]
    corrs = [tu.to_torch(lay["corr"], dev) for lay in c["layers"]]
    kgs = [tu.to_torch(lay["key_gate"], dev) for lay in c["layers"]]
    tabs = layer_tables(states, corrs, kgs, dev)
    t = lambda a: tu.to_torch(a, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    args = [t(c[k]) for k in ("A_log", "dt_bias", "sources", "commit_lens", "destinations")]
    for _ in range(20):
        kda_commit(*tabs, *args, state_dtype=KDA_STATE_F32, lower_bound=c["lower_bound"],
                   L=c["L"], H=c["H"], B=c["B"], Q=c["Q"], n_slots=states[0].shape[0],
                   n_rows=corrs[0].shape[0], boundaries=t(c["boundaries"]),
                   boundary_lens=t(c["boundary_lens"]), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_layers = [{k: v.copy() for k, v in lay.items()} for lay in c["layers"]]
    ko.commit(layers=ref_layers, A_log=c["A_log"], dt_bias=c["dt_bias"], sources=c["sources"],
              commit_lens=c["commit_lens"], destinations=c["destinations"],
              lower_bound=c["lower_bound"], Q=c["Q"], B=c["B"], H=c["H"],
              boundaries=c["boundaries"], boundary_lens=c["boundary_lens"])
    _compare_pools([tu.to_numpy(s) for s in states], ref_layers, orig)


def test_commit_at_the_gate_bound_with_align():
    """lower_bound = -10, Q = 8, every request committing a full window with a
    boundary: the boundary state divides the partial replay sum by a product
    of up to seven decays of e^-10 each."""
    c = synth.commit_case(L=2, B=24, H=4, Q=8, slots=96, seed=520, state_dtype="f32",
                          boundary_frac=0.5)
    c["lower_bound"] = -10.0
    c["commit_lens"][:] = 8
    for lay in c["layers"]:
        lay["key_gate"][..., 128:] = synth.to_bf16_bits(
            np.full(lay["key_gate"][..., 128:].shape, 30.0, np.float32))
    got, ref = _commit_both(c, align=True)
    _compare_pools(got, ref, c["layers"])


def test_commit_undersized_layer_stride_is_reported_not_written():
    """A per-layer stride below one slot's extent (or negative) is caught by
    the kernel: KDA_ERR_ARG in the status word, that layer's items skipped
    (its pool bit-identical), the other layers committed as usual."""
    import torch
    from linear_attention_speculative_recoverssm_gb300 import (KDA_ERR_ARG, KDA_STATE_F32,
                                                               kda_commit, layer_tables)
    c = synth.commit_case(L=3, B=16, H=2, Q=4, slots=48, seed=521, state_dtype="f32")
    dev = "cuda"
    states = [tu.to_torch(lay["state"], dev) for lay in c["layers"]]
    corrs = [tu.to_torch(lay["corr"], dev) for lay in c["layers"]]
    kgs = [tu.to_torch(lay["key_gate"], dev) for lay in c["layers"]]
    t = lambda a: tu.to_torch(a, dev)
    for bad_table, bad_value in ((3, 2 * 128 * 128 - 4), (4, -2 * 4 * 128), (5, 16)):
        tabs = list(layer_tables(states, corrs, kgs, dev))
        tabs[bad_table][1] = bad_value  # layer 1: state / corr / key-gate stride
        pools = [s.clone() for s in states]
        tabs[0] = torch.tensor([p.data_ptr() for p in pools], dtype=torch.int64, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        kda_commit(*tabs, t(c["A_log"]), t(c["dt_bias"]), t(c["sources"]),
                   t(c["commit_lens"]), t(c["destinations"]), state_dtype=KDA_STATE_F32,
                   lower_bound=c["lower_bound"], L=3, H=2, B=16, Q=4, n_slots=48,
                   n_rows=corrs[0].shape[0], boundaries=t(c["boundaries"]),
                   boundary_lens=t(c["boundary_lens"]), status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == KDA_ERR_ARG
        np.testing.assert_array_equal(tu.to_numpy(pools[1]), c["layers"][1]["state"])
        ref_layers = [{k: v.copy() for k, v in lay.items()} for lay in c["layers"]]
        ko.commit(layers=ref_layers, A_log=c["A_log"], dt_bias=c["dt_bias"],
                  sources=c["sources"], commit_lens=c["commit_lens"],
                  destinations=c["destinations"], lower_bound=c["lower_bound"], Q=4, B=16, H=2,
                  boundaries=c["boundaries"], boundary_lens=c["boundary_lens"])
        for l in (0, 2):
            _compare_pools([tu.to_numpy(pools[l])], [ref_layers[l]], [c["layers"][l]])
