"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, and its host-side argument checks reject bad calls before
anything is launched (so these calls are safe on any machine)."""
import ctypes
import os
import re

import pytest

from linear_attention_speculative_recoverssm_gb300 import _build, _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return _lib.load()


def _declared():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            names += re.findall(r"^(?:int|int64_t|const char \*)\s*(kda_\w+)\s*\(", text, re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert set(_lib.EXPORTS) <= set(declared)
    for name in declared:
        assert hasattr(lib, name), name


def test_version_and_error_strings(lib):
    assert lib.kda_abi_version() == 2
    assert lib.kda_error_string(0) == b"ok"
    assert lib.kda_error_string(-2).startswith(b"pointer")
    assert lib.kda_error_string(123) == b"unknown status"


A = 0x10000  # a 16-byte aligned stand-in address: never dereferenced below


def _verify_args(**over):
    args = dict(q=A, k=A, v=A, g=A, beta=A, A_log=A, dt_bias=A, lb=-5.0, qs=0.088,
                state=A, dtype=0, slot_stride=2 * 128 * 128, n_slots=4, slots=A, qsl=None,
                n_tokens=4, rows=A,
                corr=A, kg=A, crs=2 * 2 * 128, krs=2 * 2 * 256, n_rows=2, rq=2, out=A,
                B=2, H=2, Q=2, null=0, status=None, stream=None)
    args.update(over)
    return list(args.values())


@pytest.mark.parametrize("over,code", [
    (dict(Q=0), _lib.KDA_ERR_ARG), (dict(Q=9), _lib.KDA_ERR_ARG),
    (dict(rq=1), _lib.KDA_ERR_ARG), (dict(H=0), _lib.KDA_ERR_ARG),
    (dict(B=-1), _lib.KDA_ERR_ARG), (dict(q=None), _lib.KDA_ERR_ARG),
    (dict(state=None), _lib.KDA_ERR_ARG), (dict(slot_stride=100), _lib.KDA_ERR_ARG),
    (dict(q=A + 2), _lib.KDA_ERR_ALIGN), (dict(state=A + 4), _lib.KDA_ERR_ALIGN),
    (dict(slot_stride=2 * 128 * 128 + 1), _lib.KDA_ERR_ALIGN),
    (dict(dtype=7), _lib.KDA_ERR_UNSUPPORTED),
    (dict(lb=-20.0), _lib.KDA_ERR_UNSUPPORTED), (dict(lb=float("nan")), _lib.KDA_ERR_UNSUPPORTED),
    (dict(B=0, n_tokens=0), _lib.KDA_OK),
    # the token count: B*Q without query_start_loc, at most B*Q with it
    (dict(n_tokens=3), _lib.KDA_ERR_ARG), (dict(qsl=A, n_tokens=5), _lib.KDA_ERR_ARG),
    (dict(qsl=A, n_tokens=-1), _lib.KDA_ERR_ARG), (dict(qsl=A, n_tokens=0), _lib.KDA_OK),
])
def test_verify_host_checks(lib, over, code):
    assert lib.kda_verify(*_verify_args(**over)) == code


def test_replay_verify_host_checks(lib):
    base = dict(q=A, k=A, v=A, g=A, beta=A, A_log=A, dt_bias=A, lb=-5.0, qs=0.088, state=A,
                slot_stride=2 * 128 * 128, n_slots=4, slots=A, qsl=None, n_tokens=4, rows=A,
                pending=A, corr=A,
                kg=A, crs=2 * 2 * 128, krs=2 * 2 * 256, n_rows=2, rq=2, bslots=None,
                blens=None, out=A, B=2, H=2, Q=2, null=0, split=1, status=None, stream=None)

    def call(**over):
        a = dict(base)
        a.update(over)
        return lib.kda_replay_verify(*a.values())

    assert call(split=3) == _lib.KDA_ERR_ARG
    assert call(pending=None) == _lib.KDA_ERR_ARG
    assert call(rows=None) == _lib.KDA_ERR_ARG
    assert call(bslots=A) == _lib.KDA_ERR_ARG  # boundary lengths missing
    assert call(corr=A + 8) == _lib.KDA_ERR_ALIGN
    assert call(B=0, n_tokens=0) == _lib.KDA_OK
    assert call(n_tokens=5) == _lib.KDA_ERR_ARG
    assert call(qsl=A, n_tokens=9) == _lib.KDA_ERR_ARG
    assert call(qsl=A, n_tokens=0) == _lib.KDA_OK  # zero tokens: nothing to do


def test_replay_verify_layers_host_checks(lib):
    # host arrays of per-layer addresses / strides (values only read, never
    # dereferenced: every call below is refused before a launch)
    def arr(vals, t=ctypes.c_void_p):
        return (t * len(vals))(*vals)

    def call(L=2, **over):
        a = dict(q=A, k=A, v=A, g=A, beta=A, A_log=A, dt_bias=A, lb=-5.0, qs=0.088,
                 pools=arr([A] * L), sstr=arr([2 * 128 * 128] * L, ctypes.c_int64), n_slots=4,
                 slots=A, rows=A, pending=A, corrs=arr([A] * L), kgs=arr([A] * L),
                 cstr=arr([2 * 2 * 128] * L, ctypes.c_int64),
                 kstr=arr([2 * 2 * 256] * L, ctypes.c_int64), n_rows=2, rq=2, out=A, L=L, B=2,
                 H=2, Q=2, null=0, status=None, stream=None)
        a.update(over)
        return lib.kda_replay_verify_layers(*a.values())

    assert call(L=0) == _lib.KDA_ERR_ARG
    assert call(L=65) == _lib.KDA_ERR_ARG
    assert call(pools=None) == _lib.KDA_ERR_ARG
    assert call(pools=arr([A, None])) == _lib.KDA_ERR_ARG
    assert call(sstr=arr([2 * 128 * 128, 100], ctypes.c_int64)) == _lib.KDA_ERR_ARG
    assert call(cstr=arr([2 * 2 * 128, -512], ctypes.c_int64)) == _lib.KDA_ERR_ARG
    assert call(kgs=arr([A, A + 8])) == _lib.KDA_ERR_ALIGN
    assert call(sstr=arr([2 * 128 * 128, 2 * 128 * 128 + 1], ctypes.c_int64)) == \
        _lib.KDA_ERR_ALIGN
    assert call(pending=None) == _lib.KDA_ERR_ARG
    assert call(lb=-11.0) == _lib.KDA_ERR_UNSUPPORTED
    assert call(Q=9) == _lib.KDA_ERR_ARG
    assert call(B=0) == _lib.KDA_OK


def test_commit_and_bookkeeping_host_checks(lib):
    P = [A] * 14
    assert lib.kda_commit(*P, 5, -5.0, 0, 1, 2, 2, 2, 4, 2, None, None) == _lib.KDA_ERR_UNSUPPORTED
    assert lib.kda_commit(*P, 1, -5.0, 0, 1, 2, 2, 0, 4, 2, None, None) == _lib.KDA_ERR_ARG
    P2 = list(P)
    P2[12] = None  # boundaries given without lengths
    assert lib.kda_commit(*P2, 1, -5.0, 0, 1, 2, 2, 2, 4, 2, None, None) == _lib.KDA_ERR_ARG
    assert lib.kda_commit(*P, 1, -5.0, 0, 1, 2, 0, 2, 4, 2, None, None) == _lib.KDA_OK
    # the gate bound: the boundary state divides by a product of decays
    assert lib.kda_commit(*P, 1, -11.0, 0, 1, 2, 2, 2, 4, 2, None, None) == \
        _lib.KDA_ERR_UNSUPPORTED
    assert lib.kda_commit(*P, 0, float("nan"), 0, 1, 2, 2, 2, 4, 2, None, None) == \
        _lib.KDA_ERR_UNSUPPORTED
    assert lib.kda_defer_commit(A, A, None, A, None, 2, 0, 2, None, None) == _lib.KDA_ERR_ARG
    assert lib.kda_defer_commit(A, A, A, A, None, 0, 0, 2, None, None) == _lib.KDA_OK
    assert lib.kda_flush_plan(A, A, A, A, A, A, A, 2, 9, 0, 2, None, None) == _lib.KDA_ERR_ARG
    assert lib.kda_flush_plan(A, A, A, A, A, A, A, 0, 4, 0, 2, None, None) == _lib.KDA_OK


def test_check_status_rejects_null(lib):
    assert lib.kda_check_status(None, None) == _lib.KDA_ERR_ARG


def test_layer_host_checks(lib):
    # kda_layer_prologue(x, w, bias, conv_state, stride, f_a, f_b, slots, rows, pending,
    #                    n_slots, n_rows, rq, q, k, v, g, B, H, Q, null, status, stream)
    def pro(**over):
        a = dict(x=A, w=A, bias=None, cs=A, stride=3 * 2 * 128 * 6, fa=A, fb=A, slots=A,
                 rows=None, pending=None, n_slots=4, n_rows=2, rq=4, q=A, k=A, v=A, g=A, B=2,
                 H=2, Q=4, null=0, status=None, stream=None)
        a.update(over)
        return lib.kda_layer_prologue(*a.values())
    assert pro(Q=0) == _lib.KDA_ERR_ARG
    assert pro(Q=5) == _lib.KDA_ERR_ARG            # Q > rq
    assert pro(stride=100) == _lib.KDA_ERR_ARG     # window smaller than 3 * D * (rq + 2)
    assert pro(x=None) == _lib.KDA_ERR_ARG
    assert pro(fb=A + 2) == _lib.KDA_ERR_ALIGN
    assert pro(g=A + 8) == _lib.KDA_ERR_ALIGN       # raw gates: 16-byte stores
    assert pro(B=0) == _lib.KDA_OK
    # kda_layer_epilogue(o, gate, w, eps, out, n_tokens, H, stream)
    assert lib.kda_layer_epilogue(A, A, A, -1.0, A, 4, 2, None) == _lib.KDA_ERR_ARG
    assert lib.kda_layer_epilogue(A, A, A + 4, 1e-6, A, 4, 2, None) == _lib.KDA_ERR_ALIGN
    assert lib.kda_layer_epilogue(A, A, A, 1e-6, A, 0, 2, None) == _lib.KDA_OK
    assert lib.kda_layer_epilogue(None, A, A, 1e-6, A, 4, 2, None) == _lib.KDA_ERR_ARG


def test_missing_library_raises():
    """The binding has no fallback: without the built library it raises."""
    with pytest.raises(ImportError):
        _lib.load(os.path.join(ROOT, "no_such_dir", "libkda_recoverssm.so"))


def test_wrong_dtypes_are_rejected_before_any_call(lib):
    """dtype checks run on the host before the C ABI is reached (CPU tensors:
    nothing is launched)."""
    import torch
    from linear_attention_speculative_recoverssm_gb300 import kda_layer_epilogue
    o = torch.zeros((2, 1, 128), dtype=torch.float32)
    gate = torch.zeros((2, 128), dtype=torch.bfloat16)
    w = torch.ones(128, dtype=torch.float32)
    out = torch.zeros((2, 128), dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        kda_layer_epilogue(o, gate, w, out, eps=1e-6)


def test_product_path_never_imports_the_oracle():
    """The package (the product path) and its CUDA sources never reach the
    oracle: parity would prove nothing if they did."""
    pkg = os.path.join(ROOT, "linear_attention_speculative_recoverssm_gb300")
    pattern = re.compile(r"^\s*(from\s+oracle\b|import\s+oracle\b|from\s+\.\.?oracle)|"
                         r"#include\s+[<\"].*oracle", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not pattern.search(text), os.path.join(dirpath, f)


def test_head_divisor_method():
    """The step kernels divide item indices by the head count with a multiply
    and two shifts (Granlund and Montgomery's round-up method for an
    invariant divisor): m = floor(2^32 (2^l - H) / H) + 1 with l =
    ceil(log2 H), n / H = (t + ((n - t) >> 1)) >> (l - 1), t = mulhi(m, n)
    (H = 1: m = 1, both shifts 0).  The method, checked here against exact
    division for every head count up to 1024 and the 32-bit edge cases."""
    import random
    rng = random.Random(3)
    for H in list(range(1, 1025)) + [4095, 4096, 65535]:
        l = (H - 1).bit_length()
        m = ((1 << 32) * ((1 << l) - H)) // H + 1
        assert 0 < m < (1 << 32)
        sh1, sh2 = (1, l - 1) if l > 0 else (0, 0)
        for n in [0, 1, H - 1, H, H + 1, 2 ** 31 - 1, 2 ** 32 - 1] + \
                [rng.randrange(2 ** 32) for _ in range(40)]:
            t = (m * n) >> 32
            assert (t + ((n - t) >> sh1)) >> sh2 == n // H, (H, n)
