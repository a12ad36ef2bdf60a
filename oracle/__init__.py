"""Python access to the CPU oracle (oracle.c) for tests, smoke and the CPU baseline.

TEST INFRASTRUCTURE ONLY: only tests/, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package.  The product library
(top_reduction_gb300) never imports it.  It takes numpy arrays; bf16/f16
tensors are passed as their raw 16-bit patterns (numpy uint16).

Each function is a thin ctypes wrapper: all arithmetic happens in oracle.c,
which cites the passages it follows.
"""
import ctypes
import os

import numpy as np

from . import build as _build

BF16, F16, F32, F64 = 0, 1, 2, 3

ERR_ARG, ERR_BAD_CU, ERR_OVERFLOW, ERR_SEL_RANGE, ERR_NOMEM = 1, 2, 3, 4, 5

# planted mistakes, used only by the pin-strength tests
MUT_NONE = 0
MUT_SELECT_SHIFT = 1
MUT_PROJECT_DROP_TERM = 2
MUT_PROJECT_TRANSPOSE = 3
MUT_LSE_DROP_TERM = 4
MUT_LOGPROB_SIGN = 5
MUT_TIE_ID_DESC = 6
MUT_TOPK_SKIP_FIRST = 7
MUT_DECODE_LAST_ONLY = 8
MUT_PHILOX_9_ROUNDS = 9
MUT_GUMBEL_SIGN = 10
MUT_MASK_IGNORED = 11
MUT_TEMP_TIMES = 12

_lib = None


class OracleError(ValueError):
    def __init__(self, code, what):
        super().__init__("%s: oracle error %d" % (what, code))
        self.code = code


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.oracle_select_rows.argtypes = [P, i32, i32, P, i32, P, P, P]
        lib.oracle_select_rows.restype = ctypes.c_int
        lib.oracle_project.argtypes = [P, i64, P, i32, i32, P, ctypes.c_int, i32, P,
                                       ctypes.c_int, P]
        lib.oracle_project.restype = ctypes.c_int
        lib.oracle_logprobs.argtypes = [P, ctypes.c_int, i32, i32, i64, P, P, i32, P, P, P,
                                        P, ctypes.c_int, P]
        lib.oracle_logprobs.restype = ctypes.c_int
        lib.oracle_set_mutation.argtypes = [ctypes.c_int]
        lib.oracle_get_mutation.restype = ctypes.c_int
        lib.oracle_cores.restype = ctypes.c_int
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_sample_uniform.argtypes = [ctypes.c_uint64, i64, i32]
        lib.oracle_sample_uniform.restype = ctypes.c_double
        lib.oracle_sample.argtypes = [P, i32, i32, P, P, i32, ctypes.c_uint64, P, P, P, P]
        lib.oracle_sample.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def cores() -> int:
    """Online host cores (what threads=0 uses)."""
    return _load().oracle_cores()


class mutation:
    """Context manager that plants one deliberate mistake in the oracle."""

    def __init__(self, m):
        self.m = m

    def __enter__(self):
        _load().oracle_set_mutation(self.m)
        return self

    def __exit__(self, *exc):
        _load().oracle_set_mutation(MUT_NONE)
        return False


def select_rows(cu_seqlens, num_decode, all_rows_mask=None, max_out=None):
    """Row selection.  Returns (row_idx int32[n_sel], logits_cu_seqlens int32[S+1])."""
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    S = cu.shape[0] - 1
    if max_out is None:
        max_out = int(cu[-1]) if S >= 0 else 0
    mask = None
    if all_rows_mask is not None:
        mask = np.ascontiguousarray(all_rows_mask, dtype=np.uint8)
        assert mask.shape[0] == S
    row_idx = np.zeros(max(max_out, 1), dtype=np.int32)
    lcu = np.zeros(S + 1, dtype=np.int32)
    n = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_select_rows(_ptr(cu), S, int(num_decode), _ptr(mask), int(max_out),
                                    _ptr(row_idx), _ptr(lcu), _ptr(n))
    if rc:
        raise OracleError(rc, "select_rows")
    return row_idx[: int(n[0])].copy(), lcu


def project(hidden_bits, W_bits, row_idx=None, w_layout=0, threads=0, return_threads=False):
    """f64 head projection z = A @ W over bf16 inputs given as uint16 bit patterns.

    hidden_bits: uint16 [T, H] (rows may be strided); W_bits: uint16 [V, H]
    (w_layout 0, the lm_head.weight layout) or [H, V] (w_layout 1).
    """
    hidden = np.asarray(hidden_bits)
    assert hidden.dtype == np.uint16 and hidden.ndim == 2 and hidden.strides[1] == 2
    W = np.ascontiguousarray(W_bits, dtype=np.uint16)
    T, H = hidden.shape
    if w_layout == 0:
        V = W.shape[0]
        assert W.shape[1] == H
    else:
        V = W.shape[1]
        assert W.shape[0] == H
    ri = None
    if row_idx is not None:
        ri = np.ascontiguousarray(row_idx, dtype=np.int32)
        if ri.size and (ri.min() < 0 or ri.max() >= T):
            raise OracleError(ERR_ARG, "project: row index out of range")
        rows = ri.shape[0]
    else:
        rows = T
    z = np.empty((rows, V), dtype=np.float64)
    used = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_project(_ptr(hidden), hidden.strides[0] // 2, _ptr(ri), rows, H,
                                _ptr(W), int(w_layout), V, _ptr(z), int(threads), _ptr(used))
    if rc:
        raise OracleError(rc, "project")
    return (z, int(used[0])) if return_threads else z


_DT = {np.dtype(np.float64): F64, np.dtype(np.float32): F32}


def logprobs(x, dtype=None, sel=None, row_k=None, k_max=0, threads=0, return_threads=False):
    """Full-vocabulary f64 log-softmax + full sort.

    x: [rows, V] array; float64/float32 directly, or uint16 bit patterns with
    dtype=BF16 / F16.  Returns a dict with lse, sel_logprob (if sel given),
    topk_ids, topk_logprobs (float64 / int32 arrays).
    """
    x = np.asarray(x)
    if dtype is None:
        dtype = _DT[x.dtype]
    assert x.ndim == 2
    if x.strides[1] != x.itemsize or x.strides[0] < x.shape[1] * x.itemsize:
        x = np.array(x, order="C", copy=True)
    rows, V = x.shape
    stride = x.strides[0] // x.itemsize if rows > 1 else V
    lse = np.empty(rows, dtype=np.float64)
    sel_a = sel_lp = None
    if sel is not None:
        sel_a = np.ascontiguousarray(sel, dtype=np.int32)
        sel_lp = np.empty(rows, dtype=np.float64)
    rk = None if row_k is None else np.ascontiguousarray(row_k, dtype=np.int32)
    ids = np.empty((rows, max(k_max, 1)), dtype=np.int32)
    lps = np.empty((rows, max(k_max, 1)), dtype=np.float64)
    used = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_logprobs(_ptr(x), int(dtype), rows, V, stride, _ptr(sel_a), _ptr(rk),
                                 int(k_max), _ptr(lse), _ptr(sel_lp), _ptr(ids), _ptr(lps),
                                 int(threads), _ptr(used))
    if rc:
        raise OracleError(rc, "logprobs")
    out = {"lse": lse, "topk_ids": ids[:, :k_max], "topk_logprobs": lps[:, :k_max]}
    if sel is not None:
        out["sel_logprob"] = sel_lp
    if return_threads:
        out["threads"] = int(used[0])
    return out


def philox4x32_10(counter, key):
    """Philox4x32 with 10 rounds (Salmon et al., SC 2011): 4 uint32 counter words and
    2 key words to 4 uint32 output words."""
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    assert c.shape == (4,) and k.shape == (2,)
    out = np.empty(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def sample_uniform(seed, offset, token):
    """The uniform in (0, 1) that Gumbel-max sampling draws for `token` of a row."""
    return float(_load().oracle_sample_uniform(int(seed) & (2 ** 64 - 1), int(offset), int(token)))


def sample(z, temperature=None, mask=None, seed=0, offsets=None):
    """Gumbel-max sampling over f64 logits z [rows, V]: ids, best scores and runner-up scores.

    temperature: [rows] float32 or None (1.0); T <= 0 is greedy.  mask: uint32
    [rows, ceil(V/32)] allowed-token bits or None.  offsets: int64 [rows] or None
    (= row index), the per-row counter offset.  Ties go to the smaller id; -1 when
    no token is allowed.
    """
    z = np.ascontiguousarray(z, dtype=np.float64)
    rows, V = z.shape
    t = None if temperature is None else np.ascontiguousarray(temperature, dtype=np.float32)
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint32)
    words = (V + 31) // 32 if m is None else m.shape[1]
    off = None if offsets is None else np.ascontiguousarray(offsets, dtype=np.int64)
    ids = np.empty(rows, dtype=np.int32)
    best = np.empty(rows, dtype=np.float64)
    second = np.empty(rows, dtype=np.float64)
    rc = _load().oracle_sample(_ptr(z), rows, V, _ptr(t), _ptr(m), int(words), int(seed) & (2 ** 64 - 1),
                               _ptr(off), _ptr(ids), _ptr(best), _ptr(second))
    if rc:
        raise OracleError(rc, "sample")
    return ids, best, second
