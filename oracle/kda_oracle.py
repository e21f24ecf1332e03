"""FP64 CPU oracle of the KDA RecoverSSM step (replay + verify + commit).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and ``--impl reference`` arm) may import
this module.  The library in ``linear_attention_speculative_recoverssm_gb300``
never imports it, and this module imports nothing from the library: the two
share no code.  Inputs come from the seeded generator, which holds none of the
method's arithmetic.

What it computes, and where the pages define it (page titles as printed):

* ``decay`` -- the per-key-channel gate decay
  d = exp(lower_bound * sigmoid(exp(A_log) * (raw_g + dt_bias))),
  page "...cutedsl.kda.fused", method ``KdaFused.decay``; the commit uses the
  same quantity in log form (page "...recoverssm.cutedsl.commit", kernel body,
  "thread c: key channel c's decays").
* ``l2norm`` -- x * rsqrt(sum x^2 + 1e-6): page "...cutedsl.kda.fused",
  kernel prologue (normalized q with the 1/sqrt(K) scale, and k), and the
  commit page (recorded keys).
* ``replay_verify`` -- per (request, head) item, the *stock sequential*
  recurrence S <- S diag(d_t); u_t = beta_t (v_t - S k_t); S <- S + u_t k_t^T;
  o_t = S q_t (page "...cutedsl.kda.fused", module docstring, step 2), first
  over the n pending recorded tokens (replay; u_t taken from the records
  instead of recomputed -- module docstring step 1), then over this step's q
  tokens (verify).  S_n is written back iff n > 0; the verify never writes
  the checkpoint (page "...recoverssm.kernels", ``kda_recoverssm_verify``).
  Records of the new window are written to the request's record row (module
  docstring step 3).  Inert rows (slot <= null) output zeros only (fused
  kernel, first branch).  Windows of different lengths are given by
  ``query_start_loc`` as the stock verify takes them (page
  "...recoverssm.kernels", ``kda_recoverssm_verify``).
* ``commit`` -- the standalone commit: the replay alone, source -> destination,
  plus the align-mode boundary state S_min(m, n) (page
  "...recoverssm.cutedsl.commit", module docstring and ``KdaCommit.kernel``).
* ``defer_commit`` / ``flush_plan`` -- the two bookkeeping steps, as integer
  code (page "...recoverssm.kernels", ``_defer_commit_kernel`` and
  ``_prepare_flush_plan_kernel``).
* ``layer_prologue`` / ``layer_epilogue`` -- the model layer around the
  step (page "...cutedsl.kda.fused", ``KdaFused.kernel``): the depthwise
  convolution of q, k, v over the window rolled by n - 1, SiLU, the gate
  projection f_b . f_a, the window rewritten; and the gated RMSNorm of the
  outputs.  BF16 at the stock points (convolution / SiLU outputs, raw
  gates, recurrence outputs, the window).
* ``decode_stock`` -- several decode steps of one layer by the stock
  recurrence alone (verify every window from the state, then advance the
  state by the accepted tokens, ``advance_item``): the result the deferred
  protocol (records, pending replays, eager commits, flushes) must equal
  (page "...cutedsl.kda.fused", module docstring).

Self-check formulations, used only by the oracle's own pin tests:

* ``replay_closed_form`` -- S_n = S_0 diag(D_n) + sum_{t<n} u_t (kn_t * P_t)^T
  (commit page docstring; fused page docstring step 1).
* ``verify_chunked`` -- the chunked (WY) verify from S_n with Gamma_t, P(s,t),
  the A / B pair products and the per-row forward substitution (fused page
  docstring step 2).

Precision: every arithmetic step is FP64 on inputs converted exactly from
BF16 / FP32.  Results are rounded once at the storage points the pages name:
outputs to BF16 (round to nearest even), corrections to FP32, the state to the
pool's dtype.

Readings where the pages leave a step open (each is listed in the design
notes as well):
* inputs q, k are always L2-normalised here (with the 1e-6 inside the sqrt)
  and q is then multiplied by ``q_scale``; records keep the key as input;
* pending counts are clamped to [0, RQ]; commit lengths to [0, Q];
* a slot is inert when ``slot <= null_slot``; a record row < 0 means none;
* under align, the boundary state is S_min(m, n) and is written only when
  the commit itself is live;
* a standalone commit whose record row is < 0 is not live.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


# --------------------------------------------------------------------------
# exact conversions at the storage points
# --------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) -> exact FP64 values."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """FP64 -> BF16 bit patterns, rounded once to nearest even.

    Written from the BF16 format (1 sign, 8 exponent, 7 fraction bits):
    a normal value m * 2^e with m in [0.5, 1) keeps 8 significant bits, so
    it rounds to rint(m * 2^8) * 2^(e - 8); below 2^-126 the spacing is the
    fixed subnormal quantum 2^-133.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    finite = np.isfinite(x)
    m, e = np.frexp(np.where(finite, x, 0.0))
    normal = e - 1 >= -126
    rounded_normal = np.ldexp(np.rint(m * 256.0), e - 8)
    rounded_sub = np.rint(np.where(finite, x, 0.0) * 2.0 ** 133) * 2.0 ** -133
    out[...] = np.where(normal, rounded_normal, rounded_sub)
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    out = np.where(np.abs(out) > bf16_max, np.copysign(np.inf, out), out)
    out = np.where(finite, out, x)
    bits = (out.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bits = np.where(np.isnan(x), np.uint16(0x7FC0), bits)
    return bits.astype(np.uint16)


def state_to_f64(page: np.ndarray) -> np.ndarray:
    """A state page (FP32 values or BF16 bit patterns) -> FP64."""
    if page.dtype == np.uint16:
        return bf16_to_f64(page)
    return page.astype(np.float64)


def f64_to_state(S: np.ndarray, dtype) -> np.ndarray:
    """FP64 state -> the pool dtype, rounded once (FP32 RNE or BF16 RNE)."""
    if np.dtype(dtype) == np.uint16:
        return f64_to_bf16(S)
    return S.astype(np.float32)


# --------------------------------------------------------------------------
# per-channel operands
# --------------------------------------------------------------------------

def sigmoid(z: np.ndarray) -> np.ndarray:
    """1 / (1 + e^-z) in FP64."""
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def decay(raw_g: np.ndarray, a_log: float, dt_bias: np.ndarray,
          lower_bound: float) -> np.ndarray:
    """Per-key-channel decay of one token (KdaFused.decay):
    exp(lower_bound * sigmoid(exp(A_log) * (raw_g + dt_bias)))."""
    return np.exp(lower_bound * sigmoid(np.exp(a_log) * (raw_g + dt_bias)))


def l2norm(x: np.ndarray) -> np.ndarray:
    """x * rsqrt(sum(x^2) + 1e-6) over the last axis."""
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + EPS)


# --------------------------------------------------------------------------
# one (request, head) item
# --------------------------------------------------------------------------

def replay_item(S0, u_rec, k_rec, g_rec, n, a_log, dt_bias, lower_bound,
                m=0):
    """Replay of the n recorded tokens by the stock recurrence.

    S <- S diag(d_t); S <- S + u_t kn_t^T for t < n, where d_t is the decay
    of the recorded raw gate, kn_t the normalised recorded key and u_t the
    recorded correction.  Returns (S_n, S_min(m, n)); the second is None when
    m <= 0.
    """
    S = np.array(S0, dtype=np.float64, copy=True)
    S_m = S.copy() if m > 0 and n == 0 else None
    for t in range(n):
        d = decay(g_rec[t], a_log, dt_bias, lower_bound)
        kn = l2norm(k_rec[t])
        S = S * d[None, :]
        S = S + np.outer(u_rec[t], kn)
        if t + 1 == min(m, n):
            S_m = S.copy()
    return S, S_m


def verify_item(S, q, k, v, raw_g, raw_beta, a_log, dt_bias, lower_bound,
                q_scale):
    """Stock sequential verify of one window from state S (not modified).

    For t < Q: S <- S diag(d_t); u_t = beta_t (v_t - S kn_t);
    S <- S + u_t kn_t^T; o_t = S qn_t, with kn_t = l2norm(k_t),
    qn_t = l2norm(q_t) * q_scale and beta_t = sigmoid(raw_beta_t).
    Returns (u [Q, V], o [Q, V]) in FP64.
    """
    S = np.array(S, dtype=np.float64, copy=True)
    Q = q.shape[0]
    V = S.shape[0]
    u = np.zeros((Q, V))
    o = np.zeros((Q, V))
    for t in range(Q):
        d = decay(raw_g[t], a_log, dt_bias, lower_bound)
        kn = l2norm(k[t])
        qn = l2norm(q[t]) * q_scale
        beta = sigmoid(raw_beta[t])
        S = S * d[None, :]
        u[t] = beta * (v[t] - S @ kn)
        S = S + np.outer(u[t], kn)
        o[t] = S @ qn
    return u, o


def advance_item(S, k, v, raw_g, raw_beta, a, a_log, dt_bias, lower_bound):
    """The state after the first ``a`` tokens of a window by the stock
    recurrence, S <- S diag(d_t); u_t = beta_t (v_t - S kn_t);
    S <- S + u_t kn_t^T: the checkpoint that committing ``a`` accepted tokens
    yields.  Returns a new FP64 array; S is not modified."""
    S = np.array(S, dtype=np.float64, copy=True)
    for t in range(a):
        d = decay(raw_g[t], a_log, dt_bias, lower_bound)
        kn = l2norm(k[t])
        beta = sigmoid(raw_beta[t])
        S = S * d[None, :]
        u = beta * (v[t] - S @ kn)
        S = S + np.outer(u, kn)
    return S


# --------------------------------------------------------------------------
# batched steps (in place on the given numpy arrays)
# --------------------------------------------------------------------------

def _items(B, H, items):
    if items is None:
        return [(b, h) for b in range(B) for h in range(H)]
    return [(int(i) // H, int(i) % H) for i in items]


def replay_verify(*, q, k, v, raw_g, raw_beta, A_log, dt_bias, lower_bound,
                  q_scale, state, state_slots, record_rows, corr, key_gate,
                  out, B, H, Q, null_slot=0, pending=None,
                  boundary_slots=None, boundary_lens=None, items=None,
                  out_f64=None, query_start_loc=None):
    """The RecoverSSM step for every (request, head) item, in place.

    Shapes: q, k, raw_g [B*Q, H, K] and v [B*Q, H, V] (BF16 bits);
    raw_beta [B*Q, H]; A_log [H]; dt_bias [H, K]; state [slots, H, V, K]
    (FP32 or BF16 bits); state_slots [B]; record_rows [B] or None (row b);
    pending [rows] or None (None: the stock verify -- no replay, the
    checkpoint is never written); corr [rows, H, RQ, V] FP32;
    key_gate [rows, H, RQ, 2K] BF16 bits ([..., :K] key, [..., K:] raw
    gate); out [B*Q, H, V] BF16 bits.  ``items`` restricts the work to the
    listed flat item ids b*H + h.  Returns nothing; writes state (iff n > 0
    and pending given), the boundary slot (align), records and outputs.

    With ``query_start_loc`` ([B + 1], the stock wrapper's argument on page
    "...recoverssm.kernels"), the activations hold the packed windows:
    request b's window is tokens query_start_loc[b] .. query_start_loc[b+1]
    - 1, its length q_b <= Q; only those q_b tokens are verified, and only
    their outputs and records are written.  A window outside the activations
    or longer than Q leaves the request untouched.  The replay does not
    depend on the window.
    """
    K = q.shape[-1]
    RQ = corr.shape[2]
    n_tok = q.shape[0]
    for b, h in _items(B, H, items):
        if query_start_loc is None:
            t0, qb = b * Q, Q
        else:
            t0 = int(query_start_loc[b])
            qb = int(query_start_loc[b + 1]) - t0
            if t0 < 0 or qb < 0 or qb > Q or t0 + qb > n_tok:
                continue
        tok = slice(t0, t0 + qb)
        slot = int(state_slots[b])
        if slot <= null_slot:
            out[tok, h, :] = 0
            if out_f64 is not None:
                out_f64[tok, h, :] = 0.0
            continue
        rec = int(record_rows[b]) if record_rows is not None else b
        n = 0
        if pending is not None and rec >= 0:
            n = min(max(int(pending[rec]), 0), RQ)
        a_log = float(A_log[h])
        bias = dt_bias[h].astype(np.float64)
        S0 = state_to_f64(state[slot, h])
        if n > 0:
            u_rec = corr[rec, h, :n].astype(np.float64)
            k_rec = bf16_to_f64(key_gate[rec, h, :n, :K])
            g_rec = bf16_to_f64(key_gate[rec, h, :n, K:])
        else:
            u_rec = k_rec = g_rec = None
        m = 0
        bslot = null_slot
        if boundary_slots is not None:
            m = int(boundary_lens[b])
            bslot = int(boundary_slots[b])
        S_n, S_m = replay_item(S0, u_rec, k_rec, g_rec, n, a_log, bias,
                               lower_bound, m)
        u, o = verify_item(
            S_n, bf16_to_f64(q[tok, h]), bf16_to_f64(k[tok, h]),
            bf16_to_f64(v[tok, h]), bf16_to_f64(raw_g[tok, h]),
            bf16_to_f64(raw_beta[tok, h]), a_log, bias, lower_bound, q_scale)
        # every old record was read above; now the new ones are written
        if n > 0:
            state[slot, h] = f64_to_state(S_n, state.dtype)
            if m > 0 and bslot > null_slot:
                state[bslot, h] = f64_to_state(S_m, state.dtype)
        out[tok, h, :] = f64_to_bf16(o)
        if out_f64 is not None:
            out_f64[tok, h, :] = o
        if rec >= 0:
            corr[rec, h, :qb] = u.astype(np.float32)
            key_gate[rec, h, :qb, :K] = k[tok, h]
            key_gate[rec, h, :qb, K:] = raw_g[tok, h]


def commit(*, layers, A_log, dt_bias, sources, commit_lens, destinations,
           lower_bound, Q, B, H, null_slot=0, boundaries=None,
           boundary_lens=None, record_rows=None, items=None):
    """Standalone commit over L layers, in place.

    ``layers`` is a list of dicts with ``state`` [slots, H, V, K] (FP32 or
    BF16 bits), ``corr`` [rows, H, Q, V] FP32 and ``key_gate``
    [rows, H, Q, 2K] BF16 bits.  A_log [L, H], dt_bias [L, H, K].  Per
    (layer, request, head) with live = n > 0, source > null, destination >
    null (and a record row >= 0): destination <- S_n of the source replayed
    from the request's records; under align (``boundaries`` given) and
    m > 0, boundary > null, the boundary slot <- S_min(m, n).  ``items``:
    flat ids (l*B + b)*H + h.
    """
    L = len(layers)
    if items is None:
        todo = [(l, b, h) for l in range(L) for b in range(B) for h in range(H)]
    else:
        todo = [(int(i) // (B * H), (int(i) // H) % B, int(i) % H) for i in items]
    for l, b, h in todo:
        lay = layers[l]
        K = lay["state"].shape[-1]
        n = int(commit_lens[b])
        src = int(sources[b])
        dst = int(destinations[b])
        rec = int(record_rows[b]) if record_rows is not None else b
        live = n > 0 and src > null_slot and dst > null_slot and rec >= 0
        if not live:
            continue
        n = min(n, Q)
        m, bslot = 0, null_slot
        if boundaries is not None:
            m = min(int(boundary_lens[b]), Q)
            bslot = int(boundaries[b])
        S0 = state_to_f64(lay["state"][src, h])
        u_rec = lay["corr"][rec, h, :n].astype(np.float64)
        k_rec = bf16_to_f64(lay["key_gate"][rec, h, :n, :K])
        g_rec = bf16_to_f64(lay["key_gate"][rec, h, :n, K:])
        S_n, S_m = replay_item(S0, u_rec, k_rec, g_rec, n, float(A_log[l, h]),
                               dt_bias[l, h].astype(np.float64), lower_bound, m)
        lay["state"][dst, h] = f64_to_state(S_n, lay["state"].dtype)
        if m > 0 and bslot > null_slot:
            lay["state"][bslot, h] = f64_to_state(S_m, lay["state"].dtype)


def defer_commit(*, state_slots, commit_lens, record_rows, pending, B,
                 null_slot=0, eager=None):
    """After sampling (``_defer_commit_kernel``), per request b: rows with no
    record slot or no state slot change nothing; an eager row zeroes its
    pending count and keeps its commit length; any other row moves its commit
    length into pending[record_rows[b]] and zeroes the commit length."""
    for b in range(B):
        rec = int(record_rows[b])
        slot = int(state_slots[b])
        if rec < 0 or slot <= null_slot:
            continue
        if eager is not None and int(eager[b]) != 0:
            pending[rec] = 0
        else:
            pending[rec] = commit_lens[b]
            commit_lens[b] = 0


def flush_plan(*, state_slots, record_rows, pending, commit_lens, final_slots,
               boundary_slots, boundary_lens, B, Q, null_slot=0):
    """The in-place flush plan (``_prepare_flush_plan_kernel``), per request
    b: length = pending[record_rows[b]] (0 without a record row) clamped to
    [0, Q]; commit length = length if the slot is live and length > 0, else 0;
    the final slot is the source; no boundary."""
    for b in range(B):
        slot = int(state_slots[b])
        rec = int(record_rows[b])
        length = int(pending[rec]) if rec >= 0 else 0
        length = min(max(length, 0), Q)
        valid = slot > null_slot and length > 0
        commit_lens[b] = length if valid else 0
        final_slots[b] = slot
        boundary_slots[b] = null_slot
        boundary_lens[b] = 0


def decode_stock(*, windows, window_of_step, accepted, A_log, dt_bias,
                 lower_bound, q_scale, state, state_slots, B, H, Q,
                 null_slot=0, items=None, query_start_loc=None):
    """Speculative decoding of one layer over several steps by the stock
    recurrence alone, with no records, deferral or flush: per live item an
    FP64 state starts from its pool page; at every step the window is
    verified from the state (outputs), then the state advances by the
    window's first accepted tokens (page "...cutedsl.kda.fused", module
    docstring: what the deferred RecoverSSM must reproduce; the accepted count
    is what sampling records as the pending replay).

    windows: q, k, v, raw_g [W, B*Q, H, K|V] and raw_beta [W, B*Q, H] (BF16
    bits), step s using window ``window_of_step[s]``; accepted [steps, B],
    clamped to [0, q_b].  With ``query_start_loc`` [steps, B + 1] the
    windows are packed: step s's request b has the q_b tokens
    query_start_loc[s, b] .. query_start_loc[s, b+1] - 1.  Returns (outs,
    finals): outs [steps, T, H, V] FP64 (zero on inert rows) and finals, a
    dict (b, h) -> the FP64 state after the last step.
    """
    steps = accepted.shape[0]
    V = state.shape[2]
    T = windows["q"].shape[1]
    outs = np.zeros((steps, T, H, V))
    finals = {}
    for b, h in _items(B, H, items):
        slot = int(state_slots[b])
        if slot <= null_slot:
            continue
        a_log = float(A_log[h])
        bias = dt_bias[h].astype(np.float64)
        S = state_to_f64(state[slot, h])
        for s in range(steps):
            if query_start_loc is None:
                tok, qb = slice(b * Q, (b + 1) * Q), Q
            else:
                t0, t1 = int(query_start_loc[s, b]), int(query_start_loc[s, b + 1])
                tok, qb = slice(t0, t1), t1 - t0
            w = int(window_of_step[s])
            q, k, v, g, beta = (bf16_to_f64(windows[key][w, tok, h])
                                for key in ("q", "k", "v", "raw_g", "raw_beta"))
            _, outs[s, tok, h] = verify_item(S, q, k, v, g, beta, a_log, bias,
                                             lower_bound, q_scale)
            a = min(max(int(accepted[s, b]), 0), qb)
            S = advance_item(S, k, v, g, beta, a, a_log, bias, lower_bound)
        finals[(b, h)] = S
    return outs, finals


# --------------------------------------------------------------------------
# the model layer around the step: convolution, gate projection, gated norm
# --------------------------------------------------------------------------

def silu(z: np.ndarray) -> np.ndarray:
    """The convolution's SiLU, z / (1 + e^-z), in FP64."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def conv_window_taps(window, n):
    """The three history values before this window's first token.  The
    stored window is [tap 1, tap 2, x_0 .. x_{RQ-1}] of the previous verify;
    after n accepted tokens the history starts at n - 1 (0 when none is
    pending) (page "...cutedsl.kda.fused", the convolution operands)."""
    off = n - 1 if n > 0 else 0
    return window[off:off + 3]


def layer_prologue(*, x, conv_weight, conv_bias, conv_state, f_a, f_b,
                   state_slots, record_rows, pending, B, H, Q, null_slot=0,
                   items=None):
    """The layer's prologue for every live (request, head) item (page
    "...cutedsl.kda.fused", ``KdaFused.kernel``: convolution operands,
    convolution and SiLU, gate projection; the convolution window written
    last).

    x [B*Q, 3*H*128] BF16 bits (q | k | v channels before the convolution);
    conv_weight [3, 4, H*128] BF16 bits (tap i = 3 is the current token);
    conv_bias [3*H*128] BF16 bits or None; conv_state [slots, 3*H*128, RQ+2]
    BF16 bits, rewritten in place to [tap 2, tap 3, x_0 .. x_{Q-1}] (entries
    past 2 + Q kept); f_a [B*Q, 128], f_b [H*128, 128] BF16 bits; pending
    None for the stock verify (no replay).  For channel ch of part p (0 q,
    1 k, 2 v) and token t: acc = bias + sum_i w[p, i, ch] * s[t + i] over the
    sequence s = taps + x, then BF16(silu(acc)); raw_g[t, f] =
    BF16(sum_j f_b[h*128 + f, j] * f_a[t, j]).  Returns q, k, v, raw_g
    [B*Q, H, 128] BF16 bits (zero on inert items, which are skipped).
    """
    RQ = conv_state.shape[2] - 2
    D = H * 128
    q = np.zeros((B * Q, H, 128), dtype=np.uint16)
    k = np.zeros_like(q)
    v = np.zeros_like(q)
    g = np.zeros_like(q)
    outs = (q, k, v)
    fa = bf16_to_f64(f_a)
    fb = bf16_to_f64(f_b)
    w = bf16_to_f64(conv_weight)
    bias = None if conv_bias is None else bf16_to_f64(conv_bias)
    for b, h in _items(B, H, items):
        slot = int(state_slots[b])
        if slot <= null_slot:
            continue
        rec = int(record_rows[b]) if record_rows is not None else b
        n = 0
        if pending is not None and rec >= 0:
            n = min(max(int(pending[rec]), 0), RQ)
        tok = slice(b * Q, (b + 1) * Q)
        for part in range(3):
            chans = part * D + h * 128 + np.arange(128)
            window = bf16_to_f64(conv_state[slot, chans])       # [128, RQ+2]
            taps = np.stack([conv_window_taps(window[c], n) for c in range(128)])
            xs = bf16_to_f64(x[tok][:, chans]).T                 # [128, Q]
            seq = np.concatenate([taps, xs], axis=1)             # [128, 3 + Q]
            for t in range(Q):
                acc = np.zeros(128) if bias is None else bias[chans].copy()
                for i in range(4):
                    acc = acc + w[part, i, h * 128:(h + 1) * 128] * seq[:, t + i]
                outs[part][b * Q + t, h] = f64_to_bf16(silu(acc))
            new = conv_state[slot, chans].copy()
            new[:, 0] = f64_to_bf16(taps[:, 1])
            new[:, 1] = f64_to_bf16(taps[:, 2])
            new[:, 2:2 + Q] = x[tok][:, chans].T
            conv_state[slot, chans] = new
        proj = fb[h * 128:(h + 1) * 128] @ fa[tok].T             # [128 features, Q]
        g[tok, h] = f64_to_bf16(proj.T)
    return q, k, v, g


def layer_epilogue(*, o, gate, norm_weight, eps):
    """The gated RMSNorm of the step's outputs (page "...cutedsl.kda.fused",
    kernel end): per (token, head), over its 128 value rows,
    out = BF16(o * rsqrt(mean(o^2) + eps) * norm_weight * sigmoid(gate)).
    o [T, H, 128] BF16 bits (the recurrence outputs, BF16 at the stock
    point); gate [T, H*128] BF16 bits; norm_weight [128] FP32.  Returns
    [T, H*128] BF16 bits."""
    T, H, V = o.shape
    of = bf16_to_f64(o)
    rstd = 1.0 / np.sqrt(np.mean(of * of, axis=-1, keepdims=True) + eps)
    gf = bf16_to_f64(gate).reshape(T, H, V)
    res = of * rstd * norm_weight.astype(np.float64)[None, None, :] * sigmoid(gf)
    return f64_to_bf16(res).reshape(T, H * V)


# --------------------------------------------------------------------------
# alternative formulations (self-checks of the oracle only)
# --------------------------------------------------------------------------

def replay_closed_form(S0, u_rec, k_rec, g_rec, n, a_log, dt_bias,
                       lower_bound):
    """S_n = S_0 diag(D_n) + sum_{t<n} u_t (kn_t * P_t)^T with
    D_n = prod_{s<n} d_s and P_t = prod_{t<s<n} d_s."""
    S0 = np.asarray(S0, dtype=np.float64)
    K = S0.shape[1]
    d = [decay(g_rec[t], a_log, dt_bias, lower_bound) for t in range(n)]
    D = np.ones(K)
    for t in range(n):
        D = D * d[t]
    S = S0 * D[None, :]
    for t in range(n):
        P = np.ones(K)
        for s in range(t + 1, n):
            P = P * d[s]
        S = S + np.outer(u_rec[t], l2norm(k_rec[t]) * P)
    return S


def verify_chunked(S, q, k, v, raw_g, raw_beta, a_log, dt_bias, lower_bound,
                   q_scale):
    """The chunked (WY) verify from S_n: with Gamma_t = prod_{r<=t} d_r and
    P(s, t) = prod_{s<r<=t} d_r,
    w_t = S (Gamma_t * kn_t), y_t = S (Gamma_t * qn_t),
    A_ts = kn_s . (P(s,t) * kn_t) (s < t), B_ts = kn_s . (P(s,t) * qn_t)
    (s <= t), u_t = beta_t (v_t - w_t - sum_{s<t} A_ts u_s),
    o_t = y_t + sum_{s<=t} B_ts u_s.  S is only read."""
    S = np.asarray(S, dtype=np.float64)
    Q = q.shape[0]
    K = S.shape[1]
    d = np.stack([decay(raw_g[t], a_log, dt_bias, lower_bound) for t in range(Q)])
    kn = l2norm(k)
    qn = l2norm(q) * q_scale
    beta = sigmoid(raw_beta)
    gamma = np.cumprod(d, axis=0)
    w = np.stack([S @ (gamma[t] * kn[t]) for t in range(Q)])
    y = np.stack([S @ (gamma[t] * qn[t]) for t in range(Q)])

    def P(s, t):
        p = np.ones(K)
        for r in range(s + 1, t + 1):
            p = p * d[r]
        return p

    u = np.zeros((Q, S.shape[0]))
    o = np.zeros((Q, S.shape[0]))
    for t in range(Q):
        acc = v[t] - w[t]
        for s in range(t):
            acc = acc - (kn[s] @ (P(s, t) * kn[t])) * u[s]
        u[t] = beta[t] * acc
    for t in range(Q):
        o[t] = y[t].copy()
        for s in range(t + 1):
            o[t] = o[t] + (kn[s] @ (P(s, t) * qn[t])) * u[s]
    return u, o
