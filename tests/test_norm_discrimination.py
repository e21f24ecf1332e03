"""The spread-norm inputs separate a correct key normalisation from a wrong
one (CPU only).

The GPU tests in ``test_gpu_norms.py`` are only as strong as their inputs.
Here mistakes are planted in the oracle (never in the library): the
normalisation x * rsqrt(|x|^2 + 1e-6) replaced by the identity (a skipped
normalisation) or by the norm of the previously normalised vector (another
token's or head's norm).  On the spread-norm inputs each planted oracle
misses the true one by far more than the parity tolerances, so a kernel with
that mistake would fail; on the unit-norm workload recipe the skipped
normalisation stays inside the tolerances, which is why the spread inputs
exist.
"""
import numpy as np
import pytest

from linear_attention_speculative_recoverssm_gb300 import synth
from oracle import kda_oracle as ko

import kda_testutil as tu


def _step(case):
    c = tu.copy_case(case)
    out = tu.oracle_step(c, replay=True)
    return c, out


def _errors(ref_case, ref_out, got_case, got_out):
    """(output rel-L2, state max|dS| / max|S|) of a planted run."""
    out_err = tu.rel_l2(ko.bf16_to_f64(got_out), ko.bf16_to_f64(ref_out))
    ds = np.abs(got_case["state"].astype(np.float64) - ref_case["state"]).max()
    return out_err, ds / np.abs(ref_case["state"]).max()


def _planted(monkeypatch, kind):
    true_l2norm = ko.l2norm
    if kind == "skipped":
        monkeypatch.setattr(ko, "l2norm", lambda x: np.asarray(x, dtype=np.float64))
    else:
        last = {"norm": None}

        def stale(x):
            x = np.asarray(x, dtype=np.float64)
            norm = np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + ko.EPS)
            use = norm if last["norm"] is None else last["norm"]
            last["norm"] = norm
            return x / use
        monkeypatch.setattr(ko, "l2norm", stale)
    return true_l2norm


def _case(key_norms):
    c = synth.replay_verify_case(B=6, H=2, Q=4, slots=10, seed=3, key_norms=key_norms)
    c["pending"][:] = 3  # every live item replays recorded keys
    return c


def test_spread_inputs_have_the_stated_norms():
    c = _case("spread")
    kn = np.linalg.norm(ko.bf16_to_f64(c["k"]), axis=-1)
    rn = np.linalg.norm(ko.bf16_to_f64(c["key_gate"][..., :128]), axis=-1)
    qn = np.linalg.norm(ko.bf16_to_f64(c["q"]), axis=-1) * 128 ** 0.5
    for norms in (kn, rn, qn):
        assert norms.min() < 3e-3 and norms.max() > 10.0
        assert np.std(np.log10(norms)) > 0.8
    # the unit recipe: every norm 1 up to BF16 rounding
    u = _case("unit")
    assert np.allclose(np.linalg.norm(ko.bf16_to_f64(u["k"]), axis=-1), 1.0, atol=1e-2)
    # only the key tensors differ between the two recipes
    for key in ("v", "raw_g", "raw_beta", "state", "corr", "state_slots", "pending"):
        np.testing.assert_array_equal(u[key], c[key])


@pytest.mark.parametrize("kind", ["skipped", "stale"])
def test_planted_normalisation_mistakes_fail_on_spread_norms(monkeypatch, kind):
    case = _case("spread")
    ref_case, ref_out = _step(case)
    _planted(monkeypatch, kind)
    got_case, got_out = _step(case)
    out_err, state_err = _errors(ref_case, ref_out, got_case, got_out)
    # far outside rel-L2 2e-3 and 1e-4 max|S|
    assert out_err > 50 * tu.OUT_REL_L2, out_err
    assert state_err > 50 * tu.STATE_REL_MAX, state_err


def test_skipped_key_normalisation_hides_in_unit_norms(monkeypatch):
    """Why the spread recipe is needed: on unit vectors a kernel that left
    the current and recorded keys unnormalised would pass the output
    tolerance, and miss the state tolerance only by the BF16 rounding of the
    keys' norms (a few times 1e-4).  (In the unit recipe every key has norm 1
    and every q norm 128^-1/2, so the planted normalisation skips exactly
    the vectors of norm above 0.3.)"""
    case = _case("unit")
    ref_case, ref_out = _step(case)
    true_l2norm = ko.l2norm

    def keys_unnormalised(x):
        x = np.asarray(x, dtype=np.float64)
        return x if np.linalg.norm(x) > 0.3 else true_l2norm(x)
    monkeypatch.setattr(ko, "l2norm", keys_unnormalised)
    got_case, got_out = _step(case)
    out_err, state_err = _errors(ref_case, ref_out, got_case, got_out)
    assert out_err < tu.OUT_REL_L2
    assert state_err < 10 * tu.STATE_REL_MAX
    # the same planted mistake on the spread inputs fails by far
    case = _case("spread")
    monkeypatch.setattr(ko, "l2norm", true_l2norm)
    ref_case, ref_out = _step(case)
    monkeypatch.setattr(ko, "l2norm", keys_unnormalised)
    got_case, got_out = _step(case)
    out_err, state_err = _errors(ref_case, ref_out, got_case, got_out)
    assert out_err > 50 * tu.OUT_REL_L2 and state_err > 50 * tu.STATE_REL_MAX
