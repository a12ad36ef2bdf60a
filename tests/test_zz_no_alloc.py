"""lmh_logprobs_from_logits_static: the logits reduction for callers that cannot allocate.

Some callers have no device memory to give a workspace. Examples: an engine
whose free HBM all went to its KV-cache pool, plain C code without the
framework's allocator, or a loop where cudaMalloc would synchronise the
device.  For them the library keeps the partials in its own fixed 8 MiB
device array.  These tests call that entry point through the C ABI (ctypes)
and check that its results match the regular entry point on the same inputs,
within the tolerance of the other from-logits tests: ids bit-exact, values
within 1e-5.  They do so on two calls in a row with different inputs,
because the array keeps the previous call's contents.

This file is collected last, so a run that stops at the first failure has
run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

TOL = 1e-5


def _entry(lib):
    f = lib.lmh_logprobs_from_logits_static
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f.argtypes = [P, ctypes.c_int, i32, i32, i64, P, P, i32, P, P, P, P, P, P]
    f.restype = ctypes.c_int
    return f


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_static(lmh, x, sel, k_max):
    """One call of the workspace-free entry point; outputs start as garbage on purpose.

    k_max = K_FULL (-1) asks for every id's logprob: topk_logprobs is [rows, V], no ids.
    """
    rows, V = x.shape
    dev = x.device
    full = k_max == lmh.K_FULL
    out = {"lse": torch.full((rows,), float("nan"), device=dev),
           "sel_logprob": torch.full((rows,), float("nan"), device=dev),
           "topk_ids": None if full else torch.full((rows, k_max), -7, dtype=torch.int32, device=dev),
           "topk_logprobs": torch.full((rows, V if full else k_max), float("nan"), device=dev)}
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = _entry(lmh.load())(_ptr(x), lmh.BF16, rows, V, x.stride(0), _ptr(sel), None, k_max, _ptr(out["lse"]),
                            _ptr(out["sel_logprob"]), _ptr(out["topk_ids"]), _ptr(out["topk_logprobs"]),
                            _ptr(st), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lmh.status_string(rc)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out


def _same(got, ref, what):
    if got["topk_ids"] is not None:
        assert torch.equal(got["topk_ids"], ref["topk_ids"]), what
    for key in ("lse", "sel_logprob", "topk_logprobs"):
        diff = (got[key] - ref[key]).abs().max().item()
        assert diff <= TOL, (what, key, diff)


def test_static_matches_workspace_entry_point_on_two_calls(lmh):
    for dist, seed, k in (("normal", 11, 20), ("ties", 12, 128)):
        c = workloads.logits_chunk(dist, seed=seed, rows=64, V=50000)
        x, sel = c["logits"].cuda(), c["sel"].cuda()
        ref = lmh.logprobs_from_logits(x, sel=sel, k_max=k)
        got = call_static(lmh, x, sel, k)
        _same(got, ref, dist)


def test_static_plain_load_path_and_full_vocabulary(lmh):
    """Rows whose stride is not a multiple of 16 bytes take the plain-load stream and the
    select kernel; k_max = K_FULL returns every id's logprob.  Two calls in a row."""
    c = workloads.logits_chunk("normal", seed=13, rows=40, V=30000)
    padded = torch.full((40, 30001), -1.0, dtype=torch.bfloat16)
    padded[:, :30000] = c["logits"]
    x = padded.cuda()[:, :30000]  # row stride 30001 elements: odd
    sel = c["sel"].cuda()
    for k in (20, lmh.K_FULL):
        ref = lmh.logprobs_from_logits(x, sel=sel, k_max=k)
        got = call_static(lmh, x, sel, k)
        _same(got, ref, "odd stride, k %d" % k)


def test_static_documented_size_fits(lmh):
    """The 256 x 248320 prompt-scoring chunk at k_max 128 fits the array (about 4.5 MB)."""
    c = workloads.logits_chunk("gumbel", seed=14)
    x, sel = c["logits"].cuda(), c["sel"].cuda()
    ref = lmh.logprobs_from_logits(x, sel=sel, k_max=128)
    got = call_static(lmh, x, sel, 128)
    _same(got, ref, "256 x 248320")


def test_static_rejects_requests_beyond_its_scratch(lmh):
    """Sizes whose partials exceed the fixed array are refused before any launch."""
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")  # never read: the call is rejected first
    dummy = torch.zeros(16, dtype=torch.float32, device="cuda")
    ids = torch.zeros(16, dtype=torch.int32, device="cuda")
    rc = _entry(lmh.load())(_ptr(x), lmh.BF16, 65536, 248320, 248320, None, None, 128, _ptr(dummy), None,
                            _ptr(ids), _ptr(dummy), None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    from top_reduction_gb300 import lmh as L
    assert rc == L.ERR_WORKSPACE_TOO_SMALL
