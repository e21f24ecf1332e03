"""Seeded synthetic inputs for the KDA RecoverSSM step.

This module draws random operands and index structure only; it holds none of
the method's arithmetic.  Both the CUDA path (tests, bench) and the CPU oracle
(tests) take their inputs from here, as numpy arrays:

* BF16 tensors are uint16 bit patterns (rounded to nearest even from FP32
  draws), FP32 tensors are float32, indices are int32.
* Activations are token-major: token ``b * Q + t`` of request ``b``.

Distributions (one recipe for every workload):

* state S_0 ~ N(0, 0.05^2) on the slots a request uses, zero elsewhere;
* q, k: a N(0, 1) draw per (token, head) scaled onto the unit sphere (a
  uniform random direction), q additionally multiplied by K^-1/2;
* v, raw_g, raw_beta ~ N(0, 1); A_log ~ U(0, 2.5) per head;
  dt_bias ~ N(0, 0.1^2) per (head, key channel); lower_bound = -5;
* records of the previous window: corrections u ~ N(0, 0.5^2) (FP32), keys
  drawn like k, raw gates ~ N(0, 1);
* test-only option ``key_norms="spread"``: q, k and the recorded keys keep
  their directions but take per-(token, head) norms spread over 1e-3 .. 1e2
  (``_KeyDraws``), so a kernel that skipped or mis-indexed a normalisation
  would be caught;
* slots: distinct live slots in 1..slots-1 (slot 0 is the null slot),
  record rows a random permutation, counts uniform on their ranges.
"""
from __future__ import annotations

import numpy as np

NULL_SLOT = 0
LOWER_BOUND = -5.0


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """FP32 draws -> BF16 bit patterns (round to nearest even; finite input)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    b = b + (((b >> 16) & 1) + 0x7FFF)
    return (b >> 16).astype(np.uint16)


def _normal(rng, shape, std=1.0):
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def _unit_directions(rng, shape):
    """Random directions on the unit sphere along the last axis."""
    x = rng.standard_normal(shape, dtype=np.float32)
    x /= np.linalg.norm(x, axis=-1, keepdims=True)
    return x


# Norms of the "spread" key draws: log10 |x| ~ U(-2, 2) per (token, head),
# and a tenth of the vectors near sqrt(1e-6) = 1e-3 (log10 |x| ~ U(-3.5,
# -2.5)), where the 1e-6 inside the normalisation's root is not negligible.
SPREAD_LOG10 = (-2.0, 2.0)
SPREAD_TINY_FRAC = 0.1
SPREAD_TINY_LOG10 = (-3.5, -2.5)


def _norm_factors(rng, lead_shape):
    """Per-vector norms for the "spread" key draws (see SPREAD_*)."""
    lg = rng.uniform(*SPREAD_LOG10, size=lead_shape)
    tiny = rng.random(lead_shape) < SPREAD_TINY_FRAC
    lg[tiny] = rng.uniform(*SPREAD_TINY_LOG10, size=int(tiny.sum()))
    return (10.0 ** lg).astype(np.float32)[..., None]


class _KeyDraws:
    """Directions for q, k and the recorded keys: unit vectors (the
    workloads' recipe), or with ``key_norms="spread"`` the same directions
    scaled to per-(token, head) norms spread over 1e-3 .. 1e2 (a test-only
    recipe: the kernels must normalise each vector by its own norm).  The
    norms come from a generator of their own, so every other draw of a case
    is the same either way."""

    def __init__(self, key_norms, seed):
        if key_norms not in ("unit", "spread"):
            raise ValueError(f"key_norms must be 'unit' or 'spread', not {key_norms!r}")
        self.spread = key_norms == "spread"
        self.rng = np.random.default_rng(seed + 2_147_483_629) if self.spread else None

    def __call__(self, rng, shape):
        x = _unit_directions(rng, shape)
        if self.spread:
            x *= _norm_factors(self.rng, shape[:-1])
        return x


def replay_verify_case(*, B, H, Q, slots, seed, RQ=None, rows=None, K=128,
                       V=128, pending_max=None, padding_frac=0.0,
                       no_record_frac=0.0, state_dtype="f32",
                       boundary_frac=0.0, key_norms="unit"):
    """Operands of one RecoverSSM verify step (replay + verify).

    Returns a dict with q, k, v, raw_g [B*Q, H, K|V], raw_beta [B*Q, H] (BF16
    bits); A_log [H], dt_bias [H, K] (FP32); state [slots, H, V, K] (FP32 or
    BF16 bits); state_slots [B]; record_rows [B]; pending [rows]; corr
    [rows, H, RQ, V] FP32; key_gate [rows, H, RQ, 2K] BF16 bits; boundary_slots
    and boundary_lens [B] (all null / 0 unless ``boundary_frac`` > 0); and the
    scalars lower_bound, q_scale, null_slot, B, H, Q, RQ.
    """
    RQ = Q if RQ is None else RQ
    rows = B if rows is None else rows
    pending_max = RQ if pending_max is None else pending_max
    assert rows >= B and Q <= RQ
    rng = np.random.default_rng(seed)
    keys = _KeyDraws(key_norms, seed)

    n_pad = int(round(padding_frac * B))
    order = rng.permutation(B)
    padding = np.zeros(B, dtype=bool)
    padding[order[:n_pad]] = True
    live_idx = np.flatnonzero(~padding)
    n_bnd = int(round(boundary_frac * len(live_idx)))
    need = len(live_idx) + n_bnd
    assert need <= slots - 1, "not enough distinct slots"
    chosen = rng.choice(np.arange(1, slots, dtype=np.int64), size=need,
                        replace=False)
    state_slots = np.full(B, NULL_SLOT, dtype=np.int32)
    state_slots[live_idx] = chosen[:len(live_idx)]

    record_rows = rng.permutation(rows)[:B].astype(np.int32)
    n_norec = int(round(no_record_frac * B))
    if n_norec:
        record_rows[rng.choice(live_idx, size=n_norec, replace=False)] = -1
    record_rows[padding] = -1
    pending = rng.integers(0, pending_max + 1, size=rows, dtype=np.int32)

    boundary_slots = np.full(B, NULL_SLOT, dtype=np.int32)
    boundary_lens = np.zeros(B, dtype=np.int32)
    if n_bnd:
        crossing = rng.choice(live_idx, size=n_bnd, replace=False)
        boundary_slots[crossing] = chosen[len(live_idx):]
        boundary_lens[crossing] = rng.integers(1, max(RQ, 2), size=n_bnd,
                                               dtype=np.int32)

    if state_dtype == "f32":
        state = np.zeros((slots, H, V, K), dtype=np.float32)
    else:
        state = np.zeros((slots, H, V, K), dtype=np.uint16)
    used = np.sort(state_slots[state_slots > NULL_SLOT])
    draw = _normal(rng, (len(used), H, V, K), 0.05)
    state[used] = draw if state_dtype == "f32" else to_bf16_bits(draw)
    del draw

    T = B * Q
    q = keys(rng, (T, H, K)) * np.float32(K ** -0.5)
    k = keys(rng, (T, H, K))
    case = dict(
        q=to_bf16_bits(q),
        k=to_bf16_bits(k),
        v=to_bf16_bits(_normal(rng, (T, H, V))),
        raw_g=to_bf16_bits(_normal(rng, (T, H, K))),
        raw_beta=to_bf16_bits(_normal(rng, (T, H))),
        A_log=rng.uniform(0.0, 2.5, size=H).astype(np.float32),
        dt_bias=_normal(rng, (H, K), 0.1),
        state=state,
        state_slots=state_slots,
        record_rows=record_rows,
        pending=pending,
        corr=_normal(rng, (rows, H, RQ, V), 0.5),
        key_gate=np.concatenate(
            [to_bf16_bits(keys(rng, (rows, H, RQ, K))),
             to_bf16_bits(_normal(rng, (rows, H, RQ, K)))], axis=-1),
        boundary_slots=boundary_slots,
        boundary_lens=boundary_lens,
        lower_bound=LOWER_BOUND,
        q_scale=float(K ** -0.5),
        null_slot=NULL_SLOT,
        B=B, H=H, Q=Q, RQ=RQ,
    )
    return case


LAYER_STACKED = ("q", "k", "v", "raw_g", "raw_beta", "A_log", "dt_bias")
SHARED_INDEX = ("state_slots", "record_rows", "pending")


def layers_case(*, L, B, H, Q, slots, seed, **kw):
    """Operands of one replay + verify step over L layers that share the
    requests' slots, record rows and pending counts (a request has the same
    slot and record row in every layer's pool).  ``layers`` holds L cases of
    ``replay_verify_case`` (layer l drawn with seed + 1000 l, its state
    drawn on layer 0's slots); the activations, A_log and dt_bias are also
    given stacked over the layers ([L, ...], the multi-layer call's layout)."""
    base = replay_verify_case(B=B, H=H, Q=Q, slots=slots, seed=seed, **kw)
    layers = [base]
    used = np.sort(base["state_slots"][base["state_slots"] > NULL_SLOT])
    for l in range(1, L):
        c = replay_verify_case(B=B, H=H, Q=Q, slots=slots, seed=seed + 1000 * l, **kw)
        rng = np.random.default_rng(seed + 1000 * l + 17)
        state = np.zeros_like(c["state"])
        draw = _normal(rng, (len(used),) + c["state"].shape[1:], 0.05)
        state[used] = draw if state.dtype == np.float32 else to_bf16_bits(draw)
        del draw
        c["state"] = state
        for key in SHARED_INDEX + ("boundary_slots", "boundary_lens"):
            c[key] = base[key]
        layers.append(c)
    case = {key: np.stack([c[key] for c in layers]) for key in LAYER_STACKED}
    for key in SHARED_INDEX:
        case[key] = base[key]
    case.update(layers=layers, L=L, B=B, H=H, Q=Q, RQ=base["RQ"],
                lower_bound=base["lower_bound"], q_scale=base["q_scale"],
                null_slot=base["null_slot"])
    return case


WINDOW_KEYS = ("q", "k", "v", "raw_g", "raw_beta")


def pack_windows(case, q_lens):
    """The first q_lens[b] tokens of each request's window, packed one
    request after another, and the query_start_loc [B + 1] (int32) that
    indexes them: request b's tokens are rows query_start_loc[b] ..
    query_start_loc[b + 1] - 1."""
    B, Q = case["B"], case["Q"]
    qsl = np.zeros(B + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    idx = np.concatenate([np.arange(b * Q, b * Q + int(q_lens[b]), dtype=np.int64)
                          for b in range(B)])
    packed = {key: np.ascontiguousarray(case[key][idx]) for key in WINDOW_KEYS}
    packed["query_start_loc"] = qsl
    return packed


def varlen_case(*, B, H, Q, slots, seed, q_min=0, **kw):
    """A replay + verify step whose requests verify windows of different
    lengths q_b ~ U{q_min..Q} (``q_lens`` [B]), packed as query_start_loc
    describes; everything else as ``replay_verify_case``."""
    case = replay_verify_case(B=B, H=H, Q=Q, slots=slots, seed=seed, **kw)
    rng = np.random.default_rng(seed + 104729)
    q_lens = rng.integers(q_min, Q + 1, size=B).astype(np.int32)
    case.update(pack_windows(case, q_lens))
    case["q_lens"] = q_lens
    return case


def layer_case(*, B, H, Q, slots, seed, bias=True, eps=1e-6, **kw):
    """Operands of the model layer around one step: the step's own operands
    (``replay_verify_case``; its q, k, v, raw_g are what the layer prologue
    produces) plus synthetic layer weights and inputs:

    * x [B*Q, 3*H*128] BF16 ~ N(0, 1): q | k | v channels before the
      convolution; conv_weight [3, 4, H*128] BF16 ~ N(0, 0.5^2) (tap 3 is
      the current token); conv_bias [3*H*128] BF16 ~ N(0, 0.1^2) or None;
      conv_state [slots, 3*H*128, RQ + 2] BF16 ~ N(0, 1) on the slots in use;
    * f_a [B*Q, 128] BF16 ~ N(0, 1), f_b [H*128, 128] BF16 ~ N(0, 1/128)
      (so the raw gates come out ~ N(0, 1));
    * gate [B*Q, H*128] BF16 ~ N(0, 1), norm_weight [128] FP32 ~ 1 + N(0,
      0.1^2), eps.
    """
    case = replay_verify_case(B=B, H=H, Q=Q, slots=slots, seed=seed, **kw)
    rng = np.random.default_rng(seed + 15485863)
    D = H * 128
    T = B * Q
    RQ = case["RQ"]
    conv_state = np.zeros((slots, 3 * D, RQ + 2), dtype=np.uint16)
    used = np.sort(case["state_slots"][case["state_slots"] > NULL_SLOT])
    for s_ in used:
        conv_state[s_] = to_bf16_bits(_normal(rng, (3 * D, RQ + 2)))
    case.update(
        x=to_bf16_bits(_normal(rng, (T, 3 * D))),
        conv_weight=to_bf16_bits(_normal(rng, (3, 4, D), 0.5)),
        conv_bias=to_bf16_bits(_normal(rng, (3 * D,), 0.1)) if bias else None,
        conv_state=conv_state,
        f_a=to_bf16_bits(_normal(rng, (T, 128))),
        f_b=to_bf16_bits(_normal(rng, (D, 128), 128 ** -0.5)),
        gate=to_bf16_bits(_normal(rng, (T, D))),
        norm_weight=(1.0 + _normal(rng, (128,), 0.1)).astype(np.float32),
        eps=eps,
    )
    return case


def decode_loop_case(*, B, H, Q, slots, steps, seed, windows=None, K=128, V=128,
                     padding_frac=0.0, accept_min=0, eager_frac=0.0, key_norms="unit"):
    """Operands of a multi-step speculative decode of one layer.

    The first step's operands are those of ``replay_verify_case`` with every
    live request owning a record row and nothing pending yet.  Added:

    * ``windows``: each step's q, k, v, raw_g [steps, B*Q, H, K|V] and
      raw_beta [steps, B*Q, H] (BF16 bits), drawn like the first window (step
      0 is the first window itself); with ``windows=W`` only W distinct
      windows are drawn and step s uses window s mod W;
    * ``accepted`` [steps, B] int32: how many of the step's Q tokens sampling
      accepts, uniform on accept_min..Q;
    * ``eager`` [steps, B] uint8: the rows committed at once instead of
      deferred, an ``eager_frac`` share of the requests per step.
    """
    case = replay_verify_case(B=B, H=H, Q=Q, slots=slots, seed=seed, K=K, V=V,
                              padding_frac=padding_frac, key_norms=key_norms)
    case["pending"][:] = 0
    rng = np.random.default_rng(seed + 7919)
    draw_keys = _KeyDraws(key_norms, seed + 7919)
    n_win = steps if windows is None else min(windows, steps)
    T = B * Q
    keys = ("q", "k", "v", "raw_g", "raw_beta")
    stacks = {key: np.empty((n_win,) + case[key].shape, dtype=np.uint16) for key in keys}
    for key in keys:
        stacks[key][0] = case[key]
    for w in range(1, n_win):
        q = draw_keys(rng, (T, H, K)) * np.float32(K ** -0.5)
        stacks["q"][w] = to_bf16_bits(q)
        stacks["k"][w] = to_bf16_bits(draw_keys(rng, (T, H, K)))
        stacks["v"][w] = to_bf16_bits(_normal(rng, (T, H, V)))
        stacks["raw_g"][w] = to_bf16_bits(_normal(rng, (T, H, K)))
        stacks["raw_beta"][w] = to_bf16_bits(_normal(rng, (T, H)))
    case["windows"] = stacks
    case["window_of_step"] = np.arange(steps, dtype=np.int64) % n_win
    case["accepted"] = rng.integers(accept_min, Q + 1, size=(steps, B), dtype=np.int32)
    case["eager"] = (rng.random((steps, B)) < eager_frac).astype(np.uint8)
    case["steps"] = steps
    return case


def commit_case(*, L, B, H, Q, slots, seed, K=128, V=128, state_dtype="bf16",
                null_frac=0.10, in_place_frac=0.5, boundary_frac=0.25, key_norms="unit"):
    """Operands of the standalone commit over L layers.

    Per layer: state [slots, H, V, K] (BF16 bits or FP32), corr [B, H, Q, V]
    FP32, key_gate [B, H, Q, 2K] BF16 bits (request b's records in row b).
    Shared across layers: sources, commit_lens, destinations, boundaries,
    boundary_lens [B] and A_log [L, H], dt_bias [L, H, K].  A ``null_frac``
    share of requests has source = destination = null; of the others,
    ``in_place_frac`` commit in place and the rest to a fresh slot; a
    ``boundary_frac`` share of all requests crosses a block boundary after
    m ~ U{1..Q-1} tokens into a fresh boundary slot.
    """
    rng = np.random.default_rng(seed)
    keys = _KeyDraws(key_norms, seed)
    order = rng.permutation(B)
    n_null = int(round(null_frac * B))
    null_rows = order[:n_null]
    live_idx = np.sort(order[n_null:])
    in_place = rng.random(len(live_idx)) < in_place_frac
    n_fresh = int((~in_place).sum())
    n_bnd = int(round(boundary_frac * B))
    need = len(live_idx) + n_fresh + n_bnd
    assert need <= slots - 1, "not enough distinct slots"
    chosen = rng.choice(np.arange(1, slots, dtype=np.int64), size=need,
                        replace=False)
    sources = np.full(B, NULL_SLOT, dtype=np.int32)
    destinations = np.full(B, NULL_SLOT, dtype=np.int32)
    sources[live_idx] = chosen[:len(live_idx)]
    dst = sources[live_idx].copy()
    dst[~in_place] = chosen[len(live_idx):len(live_idx) + n_fresh]
    destinations[live_idx] = dst
    commit_lens = rng.integers(0, Q + 1, size=B, dtype=np.int32)
    boundaries = np.full(B, NULL_SLOT, dtype=np.int32)
    boundary_lens = np.zeros(B, dtype=np.int32)
    if n_bnd:
        crossing = rng.choice(np.arange(B), size=n_bnd, replace=False)
        boundaries[crossing] = chosen[len(live_idx) + n_fresh:]
        boundary_lens[crossing] = rng.integers(1, max(Q, 2), size=n_bnd,
                                               dtype=np.int32)
    del null_rows

    layers = []
    used = np.sort(sources[sources > NULL_SLOT])
    for _ in range(L):
        if state_dtype == "bf16":
            state = np.zeros((slots, H, V, K), dtype=np.uint16)
            state[used] = to_bf16_bits(_normal(rng, (len(used), H, V, K), 0.05))
        else:
            state = np.zeros((slots, H, V, K), dtype=np.float32)
            state[used] = _normal(rng, (len(used), H, V, K), 0.05)
        corr = _normal(rng, (B, H, Q, V), 0.5)
        key_gate = np.concatenate(
            [to_bf16_bits(keys(rng, (B, H, Q, K))),
             to_bf16_bits(_normal(rng, (B, H, Q, K)))], axis=-1)
        layers.append(dict(state=state, corr=corr, key_gate=key_gate))
    return dict(
        layers=layers,
        A_log=rng.uniform(0.0, 2.5, size=(L, H)).astype(np.float32),
        dt_bias=_normal(rng, (L, H, K), 0.1),
        sources=sources, commit_lens=commit_lens, destinations=destinations,
        boundaries=boundaries, boundary_lens=boundary_lens,
        lower_bound=LOWER_BOUND, null_slot=NULL_SLOT, L=L, B=B, H=H, Q=Q,
    )


# The workloads of the five measured configurations and the measured next
# rows, by what they are.
WORKLOADS = {
    "tiny-b2-h2-q2": dict(kind="replay_verify", B=2, H=2, Q=2, slots=4,
                          seed=0),
    "commit-bf16-l4-h32-b64-q4-align": dict(kind="commit", L=4, H=32, B=64,
                                            Q=4, slots=256, seed=1),
    "replay-verify-f32-h32-b128-q4": dict(kind="replay_verify", B=128, H=32,
                                          Q=4, slots=512, seed=2,
                                          no_record_frac=0.05),
    "replay-verify-f32-h64-b512-q8": dict(kind="replay_verify", B=512, H=64,
                                          Q=8, slots=1024, seed=3,
                                          padding_frac=0.05),
    # the model layer around the large-batch step (convolution, gate
    # projection, the step, gated norm), synthetic weights
    "layer-f32-h64-b512-q8": dict(kind="layer", B=512, H=64, Q=8, slots=1024,
                                  seed=9, padding_frac=0.05),
    # the large-batch step with windows of 1..8 tokens per request
    "replay-verify-varlen-f32-h64-b512-q8": dict(kind="varlen", B=512, H=64, Q=8,
                                                 slots=1024, seed=8, q_min=1,
                                                 padding_frac=0.05),
    # eight decode steps of the large-batch shape (a flush after every
    # eighth, so the first step of each cycle is the stock verify); sampling
    # accepts 1..8 tokens per request and step; two distinct windows
    "decode-loop-f32-h64-b512-q8": dict(kind="decode_loop", B=512, H=64, Q=8,
                                        slots=1024, steps=8, seed=6, windows=2,
                                        padding_frac=0.05, accept_min=1),
    # the model layer at a quarter of the requests (profiler captures)
    "layer-f32-h64-b128-q8": dict(kind="layer", B=128, H=64, Q=8, slots=160,
                                  seed=10, padding_frac=0.05),
    # the large-batch shape at a quarter of the requests (the same kernel
    # instance, ~0.6 GB of state): small enough for a full profiler capture
    "replay-verify-f32-h64-b128-q8": dict(kind="replay_verify", B=128, H=64,
                                          Q=8, slots=160, seed=5,
                                          padding_frac=0.05),
}


def make(name, **overrides):
    """Build a named workload (see WORKLOADS), with optional overrides."""
    spec = dict(WORKLOADS[name])
    spec.update(overrides)
    kind = spec.pop("kind")
    if kind == "commit":
        return commit_case(**spec)
    if kind == "decode_loop":
        return decode_loop_case(**spec)
    if kind == "varlen":
        return varlen_case(**spec)
    if kind == "layer":
        return layer_case(**spec)
    return replay_verify_case(**spec)


def latency_case(*, B, Q, seed=4, H=32, slots=64):
    """The latency sweep's small batches: H=32, B in {1, 4, 16}, Q in
    {1, 2, 4, 8}, pending ~ U{0..Q}."""
    return replay_verify_case(B=B, H=H, Q=Q, slots=max(slots, B + 1),
                              seed=seed + 100 * B + Q)
