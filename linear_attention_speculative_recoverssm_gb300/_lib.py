"""ctypes binding of libkda_recoverssm.so (argument marshalling only).

Every function here takes torch tensors on the GPU, reads their data
pointers, sizes and strides, and calls the C entry point of the same name on
the current CUDA stream (or the given one).  All compute runs in the
library's kernels; there is no fallback: if the library is missing, import
fails with an error that says how to build it.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkda_recoverssm.so")

# status codes (include/kda_recoverssm.h)
KDA_OK = 0
KDA_ERR_ARG = -1
KDA_ERR_ALIGN = -2
KDA_ERR_UNSUPPORTED = -3
KDA_ERR_CUDA = -4
KDA_ERR_TIMEOUT = -5
KDA_ERR_SCRATCH = -6
KDA_LAYER_STEP_NOALLOC_MAX_BYTES = 16 * 1024 * 1024
KDA_STATE_F32 = 0
KDA_STATE_BF16 = 1

EXPORTS = ("kda_abi_version", "kda_error_string", "kda_check_status", "kda_verify",
           "kda_replay_verify", "kda_replay_verify_layers",
           "kda_commit", "kda_defer_commit", "kda_flush_plan", "kda_selftest_wait_timeout",
           "kda_layer_prologue", "kda_layer_epilogue", "kda_layer_step_workspace_bytes",
           "kda_layer_step", "kda_layer_step_noalloc")

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float

_SIGS = {
    "kda_abi_version": ([], _I),
    "kda_error_string": ([_I], ctypes.c_char_p),
    "kda_check_status": ([_P, _P], _I),
    "kda_verify": ([_P] * 7 + [_F, _F, _P, _I, _I64, _I, _P, _P, _I, _P, _P, _P, _I64, _I64,
                               _I, _I, _P, _I, _I, _I, _I, _P, _P], _I),
    "kda_replay_verify": ([_P] * 7 + [_F, _F, _P, _I64, _I, _P, _P, _I, _P, _P, _P, _P, _I64,
                                      _I64, _I, _I, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P],
                          _I),
    "kda_replay_verify_layers": ([_P] * 7 + [_F, _F, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I,
                                             _I, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "kda_commit": ([_P] * 14 + [_I, _F, _I, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "kda_defer_commit": ([_P] * 5 + [_I, _I, _I, _P, _P], _I),
    "kda_flush_plan": ([_P] * 7 + [_I, _I, _I, _I, _P, _P], _I),
    "kda_selftest_wait_timeout": ([_P, _P], _I),
    "kda_layer_prologue": ([_P] * 4 + [_I64] + [_P] * 5 + [_I, _I, _I] + [_P] * 4
                           + [_I, _I, _I, _I, _P, _P], _I),
    "kda_layer_epilogue": ([_P, _P, _P, _F, _P, _I, _I, _P], _I),
    "kda_layer_step_workspace_bytes": ([_I, _I, _I], _I64),
    "kda_layer_step_noalloc": ([_P] * 4 + [_I64] + [_P] * 5 + [_F, _F, _P, _I64, _I, _P, _P, _P,
                                                           _P, _P, _I64, _I64, _I, _I, _P, _P, _F,
                                                           _P, _I, _I, _I, _I, _P, _P], _I),
    "kda_layer_step": ([_P] * 4 + [_I64] + [_P] * 5 + [_F, _F, _P, _I64, _I, _P, _P, _P, _P, _P,
                                                   _I64, _I64, _I, _I, _P, _P, _F, _P, _P, _I64,
                                                   _I, _I, _I, _I, _P, _P], _I),
}

_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library once; raise ImportError if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(
            f"{p} is missing: build it with `python -m "
            "linear_attention_speculative_recoverssm_gb300._build` "
            "(or __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _lib = lib
    return lib


class KdaError(RuntimeError):
    def __init__(self, fn, code):
        msg = load().kda_error_string(code).decode()
        super().__init__(f"{fn} returned {code} ({msg})")
        self.code = code


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, code, raise_on_error):
    if code != KDA_OK and raise_on_error:
        raise KdaError(fn, code)
    return code


def _expect(t, dtype, name):
    if t is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _check_step_dtypes(q, k, v, raw_g, raw_beta, A_log, dt_bias, state_slots, record_rows,
                       corr, key_gate, out):
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("raw_g", raw_g), ("raw_beta", raw_beta),
                    ("key_gate", key_gate), ("out", out)):
        _expect(t, torch.bfloat16, name)
    for name, t in (("A_log", A_log), ("dt_bias", dt_bias), ("corr", corr)):
        _expect(t, torch.float32, name)
    for name, t in (("state_slots", state_slots), ("record_rows", record_rows)):
        _expect(t, torch.int32, name)


def kda_check_status(status, *, stream=None):
    """The code held by the device status word ``status`` (int32 tensor),
    read back after the work already enqueued on the stream (this call waits
    for that stream)."""
    import torch
    _expect(status, torch.int32, "status")
    return load().kda_check_status(_ptr(status), _stream(stream))


def kda_verify(q, k, v, raw_g, raw_beta, A_log, dt_bias, state_pool, state_slots, corr,
               key_gate, out, *, Q, lower_bound, q_scale, record_rows=None,
               query_start_loc=None, null_slot=0, status=None, stream=None,
               raise_on_error=True):
    """Stock verify of one window (state read only).  Shapes as in
    include/kda_recoverssm.h; state_pool is float32 or bfloat16; the
    activations' first dimension is the token count (B*Q without
    query_start_loc)."""
    import torch
    _check_step_dtypes(q, k, v, raw_g, raw_beta, A_log, dt_bias, state_slots, record_rows,
                       corr, key_gate, out)
    _expect(query_start_loc, torch.int32, "query_start_loc")
    dtype = KDA_STATE_F32 if state_pool.dtype == torch.float32 else KDA_STATE_BF16
    if state_pool.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("state_pool must be float32 or bfloat16")
    B = state_slots.shape[0]
    H = q.shape[1]
    rc = load().kda_verify(
        _ptr(q), _ptr(k), _ptr(v), _ptr(raw_g), _ptr(raw_beta), _ptr(A_log), _ptr(dt_bias),
        lower_bound, q_scale, _ptr(state_pool), dtype, state_pool.stride(0),
        state_pool.shape[0], _ptr(state_slots), _ptr(query_start_loc), q.shape[0],
        _ptr(record_rows), _ptr(corr), _ptr(key_gate), corr.stride(0), key_gate.stride(0),
        corr.shape[0], corr.shape[2], _ptr(out), B, H, Q, null_slot, _ptr(status),
        _stream(stream))
    return _check("kda_verify", rc, raise_on_error)


def kda_replay_verify(q, k, v, raw_g, raw_beta, A_log, dt_bias, state_pool, state_slots,
                      record_rows, pending, corr, key_gate, out, *, Q, lower_bound, q_scale,
                      boundary_slots=None, boundary_lens=None, query_start_loc=None,
                      null_slot=0, split=0, status=None, stream=None, raise_on_error=True):
    """Fused replay + verify (FP32 state pool, written in place)."""
    import torch
    _check_step_dtypes(q, k, v, raw_g, raw_beta, A_log, dt_bias, state_slots, record_rows,
                       corr, key_gate, out)
    _expect(query_start_loc, torch.int32, "query_start_loc")
    _expect(state_pool, torch.float32, "state_pool")
    _expect(pending, torch.int32, "pending")
    B = state_slots.shape[0]
    H = q.shape[1]
    rc = load().kda_replay_verify(
        _ptr(q), _ptr(k), _ptr(v), _ptr(raw_g), _ptr(raw_beta), _ptr(A_log), _ptr(dt_bias),
        lower_bound, q_scale, _ptr(state_pool), state_pool.stride(0), state_pool.shape[0],
        _ptr(state_slots), _ptr(query_start_loc), q.shape[0], _ptr(record_rows), _ptr(pending),
        _ptr(corr), _ptr(key_gate), corr.stride(0), key_gate.stride(0), corr.shape[0],
        corr.shape[2], _ptr(boundary_slots), _ptr(boundary_lens), _ptr(out), B, H, Q,
        null_slot, split, _ptr(status), _stream(stream))
    return _check("kda_replay_verify", rc, raise_on_error)


def kda_replay_verify_layers(q, k, v, raw_g, raw_beta, A_log, dt_bias, state_pools, state_slots,
                             record_rows, pending, corrs, key_gates, out, *, Q, lower_bound,
                             q_scale, null_slot=0, status=None, stream=None,
                             raise_on_error=True):
    """Fused replay + verify over L layers in one launch: q, k, v, raw_g, out
    [L, B*Q, H, 128] and raw_beta [L, B*Q, H] layer-stacked; A_log [L, H],
    dt_bias [L, H, 128]; state_pools, corrs, key_gates lists of the L
    layers' FP32 pools, FP32 corrections and BF16 key/gate records (their
    addresses and strides are passed as host arrays); the index arrays are
    shared by the layers."""
    import torch
    L = len(state_pools)
    if not (len(corrs) == len(key_gates) == L):
        raise ValueError("state_pools, corrs and key_gates must list the same layers")
    for t in state_pools:
        _expect(t, torch.float32, "state_pools[l]")
    for t in corrs:
        _expect(t, torch.float32, "corrs[l]")
    if any(t.shape[2] != corrs[0].shape[2] for t in list(corrs) + list(key_gates)):
        raise ValueError("every layer's records must hold the same number of tokens")
    for t in key_gates:
        _expect(t, torch.bfloat16, "key_gates[l]")
    _check_step_dtypes(q, k, v, raw_g, raw_beta, A_log, dt_bias, state_slots, record_rows,
                       corrs[0], key_gates[0], out)
    _expect(pending, torch.int32, "pending")
    ptrs = lambda ts: (ctypes.c_void_p * L)(*[t.data_ptr() for t in ts])
    strides = lambda ts: (ctypes.c_int64 * L)(*[t.stride(0) for t in ts])
    B = state_slots.shape[0]
    H = q.shape[2]
    rc = load().kda_replay_verify_layers(
        _ptr(q), _ptr(k), _ptr(v), _ptr(raw_g), _ptr(raw_beta), _ptr(A_log), _ptr(dt_bias),
        lower_bound, q_scale, ptrs(state_pools), strides(state_pools),
        min(t.shape[0] for t in state_pools), _ptr(state_slots), _ptr(record_rows),
        _ptr(pending), ptrs(corrs), ptrs(key_gates), strides(corrs), strides(key_gates),
        min(min(t.shape[0] for t in corrs), min(t.shape[0] for t in key_gates)),
        corrs[0].shape[2], _ptr(out), L,
        B, H, Q, null_slot, _ptr(status), _stream(stream))
    return _check("kda_replay_verify_layers", rc, raise_on_error)


def kda_commit(state_ptrs, corr_ptrs, kg_ptrs, state_strides, corr_strides, kg_strides, A_log,
               dt_bias, sources, commit_lens, destinations, *, state_dtype, lower_bound, L, H,
               B, Q, n_slots, n_rows, boundaries=None, boundary_lens=None, record_rows=None,
               null_slot=0, status=None, stream=None, raise_on_error=True):
    """Standalone commit over L layers; the six tables are device int64
    tensors of [L] addresses / strides (see layer_tables)."""
    rc = load().kda_commit(
        _ptr(state_ptrs), _ptr(corr_ptrs), _ptr(kg_ptrs), _ptr(state_strides),
        _ptr(corr_strides), _ptr(kg_strides), _ptr(A_log), _ptr(dt_bias), _ptr(sources),
        _ptr(commit_lens), _ptr(destinations), _ptr(boundaries), _ptr(boundary_lens),
        _ptr(record_rows), state_dtype, lower_bound, null_slot, L, H, B, Q, n_slots, n_rows,
        _ptr(status), _stream(stream))
    return _check("kda_commit", rc, raise_on_error)


def layer_tables(states, corrs, key_gates, device):
    """The per-layer address and stride tables kda_commit reads, as device
    int64 tensors: (state_ptrs, corr_ptrs, kg_ptrs, state_strides,
    corr_strides, kg_strides)."""
    import torch
    mk = lambda xs: torch.tensor(xs, dtype=torch.int64, device=device)
    return (mk([s.data_ptr() for s in states]), mk([c.data_ptr() for c in corrs]),
            mk([g.data_ptr() for g in key_gates]), mk([s.stride(0) for s in states]),
            mk([c.stride(0) for c in corrs]), mk([g.stride(0) for g in key_gates]))


def kda_defer_commit(state_slots, commit_lens, record_rows, pending, *, eager=None, null_slot=0,
                     status=None, stream=None, raise_on_error=True):
    rc = load().kda_defer_commit(
        _ptr(state_slots), _ptr(commit_lens), _ptr(record_rows), _ptr(pending), _ptr(eager),
        state_slots.shape[0], null_slot, pending.shape[0], _ptr(status), _stream(stream))
    return _check("kda_defer_commit", rc, raise_on_error)


def kda_flush_plan(state_slots, record_rows, pending, commit_lens, final_slots, boundary_slots,
                   boundary_lens, *, Q, null_slot=0, status=None, stream=None,
                   raise_on_error=True):
    rc = load().kda_flush_plan(
        _ptr(state_slots), _ptr(record_rows), _ptr(pending), _ptr(commit_lens),
        _ptr(final_slots), _ptr(boundary_slots), _ptr(boundary_lens), state_slots.shape[0], Q,
        null_slot, pending.shape[0], _ptr(status), _stream(stream))
    return _check("kda_flush_plan", rc, raise_on_error)


def kda_selftest_wait_timeout(status, *, stream=None, raise_on_error=True):
    """Failure-detection self-test: a device wait that runs out writes
    KDA_ERR_TIMEOUT to ``status`` (device int32)."""
    rc = load().kda_selftest_wait_timeout(_ptr(status), _stream(stream))
    return _check("kda_selftest_wait_timeout", rc, raise_on_error)


def kda_layer_prologue(x, conv_weight, conv_bias, conv_state, f_a, f_b, state_slots,
                       record_rows, pending, q, k, v, raw_g, *, Q, rq=None, null_slot=0,
                       status=None, stream=None, raise_on_error=True):
    """The layer's convolution + SiLU, gate projection and window rewrite
    (shapes as in include/kda_recoverssm.h; conv_state [slots, 3*H*128,
    rq + 2])."""
    import torch
    for name, t in (("x", x), ("conv_weight", conv_weight), ("conv_bias", conv_bias),
                    ("conv_state", conv_state), ("f_a", f_a), ("f_b", f_b), ("q", q), ("k", k),
                    ("v", v), ("raw_g", raw_g)):
        _expect(t, torch.bfloat16, name)
    for name, t in (("state_slots", state_slots), ("record_rows", record_rows),
                    ("pending", pending)):
        _expect(t, torch.int32, name)
    rq = conv_state.shape[2] - 2 if rq is None else rq
    rc = load().kda_layer_prologue(
        _ptr(x), _ptr(conv_weight), _ptr(conv_bias), _ptr(conv_state), conv_state.stride(0),
        _ptr(f_a), _ptr(f_b), _ptr(state_slots), _ptr(record_rows), _ptr(pending),
        conv_state.shape[0], 0 if pending is None else pending.shape[0], rq, _ptr(q), _ptr(k),
        _ptr(v), _ptr(raw_g), state_slots.shape[0], q.shape[1], Q, null_slot, _ptr(status),
        _stream(stream))
    return _check("kda_layer_prologue", rc, raise_on_error)


def kda_layer_epilogue(o, gate, norm_weight, out, *, eps, stream=None, raise_on_error=True):
    """The gated RMSNorm of the step's outputs o [T, H, 128] into out
    [T, H*128]."""
    import torch
    _expect(o, torch.bfloat16, "o")
    _expect(gate, torch.bfloat16, "gate")
    _expect(out, torch.bfloat16, "out")
    _expect(norm_weight, torch.float32, "norm_weight")
    rc = load().kda_layer_epilogue(_ptr(o), _ptr(gate), _ptr(norm_weight), eps, _ptr(out),
                                   o.shape[0], o.shape[1], _stream(stream))
    return _check("kda_layer_epilogue", rc, raise_on_error)


def kda_layer_step_workspace_bytes(B, H, Q):
    """Bytes of workspace kda_layer_step needs (the step's q, k, v, raw_g)."""
    return load().kda_layer_step_workspace_bytes(B, H, Q)


def kda_layer_step(x, conv_weight, conv_bias, conv_state, f_a, f_b, raw_beta, A_log, dt_bias,
                   state_pool, state_slots, record_rows, pending, corr, key_gate, gate,
                   norm_weight, out, workspace, *, Q, lower_bound, q_scale, eps, rq=None,
                   null_slot=0, status=None, stream=None, raise_on_error=True):
    """One model-layer step (convolution + SiLU, gate projection, fused
    replay + verify with the gated RMSNorm folded in): out [B*Q, H*128]
    BF16.  ``workspace`` is a device tensor of at least
    kda_layer_step_workspace_bytes(B, H, Q) bytes; afterwards it holds the
    step's q, k, v, raw_g ([B*Q, H, 128] BF16 each, in that order)."""
    import torch
    for name, t in (("x", x), ("conv_weight", conv_weight), ("conv_bias", conv_bias),
                    ("conv_state", conv_state), ("f_a", f_a), ("f_b", f_b),
                    ("raw_beta", raw_beta), ("key_gate", key_gate), ("gate", gate),
                    ("out", out)):
        _expect(t, torch.bfloat16, name)
    for name, t in (("A_log", A_log), ("dt_bias", dt_bias), ("state_pool", state_pool),
                    ("corr", corr), ("norm_weight", norm_weight)):
        _expect(t, torch.float32, name)
    for name, t in (("state_slots", state_slots), ("record_rows", record_rows),
                    ("pending", pending)):
        _expect(t, torch.int32, name)
    rq = corr.shape[2] if rq is None else rq
    B = state_slots.shape[0]
    H = A_log.shape[0]
    nbytes = workspace.numel() * workspace.element_size()
    rc = load().kda_layer_step(
        _ptr(x), _ptr(conv_weight), _ptr(conv_bias), _ptr(conv_state), conv_state.stride(0),
        _ptr(f_a), _ptr(f_b), _ptr(raw_beta), _ptr(A_log), _ptr(dt_bias), lower_bound, q_scale,
        _ptr(state_pool), state_pool.stride(0), state_pool.shape[0], _ptr(state_slots),
        _ptr(record_rows), _ptr(pending), _ptr(corr), _ptr(key_gate), corr.stride(0),
        key_gate.stride(0), corr.shape[0], rq, _ptr(gate), _ptr(norm_weight), eps, _ptr(out),
        _ptr(workspace), nbytes, B, H, Q, null_slot, _ptr(status), _stream(stream))
    return _check("kda_layer_step", rc, raise_on_error)


def kda_layer_step_noalloc(x, conv_weight, conv_bias, conv_state, f_a, f_b, raw_beta, A_log,
                           dt_bias, state_pool, state_slots, record_rows, pending, corr,
                           key_gate, gate, norm_weight, out, *, Q, lower_bound, q_scale, eps,
                           rq=None, null_slot=0, status=None, stream=None,
                           raise_on_error=True):
    """kda_layer_step without a workspace, for callers that cannot allocate
    device memory on the decode path: the step's operands go to the
    library's own fixed array (KDA_LAYER_STEP_NOALLOC_MAX_BYTES per GPU), so
    nothing is allocated.  Calls larger than that raise KDA_ERR_SCRATCH;
    calls that overlap on the GPU share the array and must be ordered."""
    import torch
    for name, t in (("x", x), ("conv_weight", conv_weight), ("conv_bias", conv_bias),
                    ("conv_state", conv_state), ("f_a", f_a), ("f_b", f_b),
                    ("raw_beta", raw_beta), ("key_gate", key_gate), ("gate", gate),
                    ("out", out)):
        _expect(t, torch.bfloat16, name)
    for name, t in (("A_log", A_log), ("dt_bias", dt_bias), ("state_pool", state_pool),
                    ("corr", corr), ("norm_weight", norm_weight)):
        _expect(t, torch.float32, name)
    for name, t in (("state_slots", state_slots), ("record_rows", record_rows),
                    ("pending", pending)):
        _expect(t, torch.int32, name)
    rq = corr.shape[2] if rq is None else rq
    B = state_slots.shape[0]
    H = A_log.shape[0]
    rc = load().kda_layer_step_noalloc(
        _ptr(x), _ptr(conv_weight), _ptr(conv_bias), _ptr(conv_state), conv_state.stride(0),
        _ptr(f_a), _ptr(f_b), _ptr(raw_beta), _ptr(A_log), _ptr(dt_bias), lower_bound, q_scale,
        _ptr(state_pool), state_pool.stride(0), state_pool.shape[0], _ptr(state_slots),
        _ptr(record_rows), _ptr(pending), _ptr(corr), _ptr(key_gate), corr.stride(0),
        key_gate.stride(0), corr.shape[0], rq, _ptr(gate), _ptr(norm_weight), eps, _ptr(out),
        B, H, Q, null_slot, _ptr(status), _stream(stream))
    return _check("kda_layer_step_noalloc", rc, raise_on_error)
