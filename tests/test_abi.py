"""The C-ABI library builds, loads and exports every symbol include/lmh.h declares.

CPU only: nothing here launches a kernel.  Host-side logic (argument checks
that return before touching a device, the host row-count helper) is
exercised directly.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    from top_reduction_gb300 import _build, lmh
    _build.build()
    return lmh.load()


def declared_functions():
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, h)).read(), flags=re.S)
            names |= set(re.findall(r"\b(lmh_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("lmh_select_rows", "lmh_project_logprobs", "lmh_logprobs_from_logits",
                 "lmh_workspace_bytes", "lmh_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    from top_reduction_gb300 import lmh
    names = declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(lmh.EXPORTS) <= set(names)
    assert lib.lmh_version() == 1


def test_status_strings(lib):
    from top_reduction_gb300 import lmh
    assert lmh.status_string(0) == "LMH_OK"
    assert lmh.status_string(3) == "LMH_ERR_WORKSPACE_TOO_SMALL"
    assert lmh.status_string(99) == "LMH_ERR_UNKNOWN"


def test_count_selected_rows_matches_oracle(lib):
    """Host helper vs the oracle's selection on random batches (host logic, no device)."""
    from top_reduction_gb300 import lmh
    rng = np.random.default_rng(11)
    for _ in range(200):
        S = int(rng.integers(0, 30))
        nd = int(rng.integers(0, S + 1))
        lens = rng.integers(1, 7, size=S)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        mask = (rng.random(S) < 0.3).astype(np.uint8)
        ri, _ = oracle.select_rows(cu, nd, mask)
        assert lmh.count_selected_rows(cu, nd, mask) == len(ri)
    for bad, nd in (([1, 2], 0), ([0, 3, 2], 0), ([0, 2, 2], 0)):
        with pytest.raises(ValueError):
            lmh.count_selected_rows(np.array(bad, dtype=np.int32), nd)


def _call_project(lib, **kw):
    args = dict(hidden=0x1000, stride=64, num_tokens=8, row_idx=None, rows=8, H=64, W=0x2000, layout=0,
                V=4096, sel=None, row_k=None, k_max=5, lse=0x3000, sel_lp=None, ids=0x4000, lps=0x5000,
                logits_out=None, ws=0x10000, ws_bytes=1 << 30, status=None)
    args.update(kw)
    P = ctypes.c_void_p
    return lib.lmh_project_logprobs(
        P(args["hidden"]) if args["hidden"] else None, args["stride"], args["num_tokens"], args["row_idx"],
        args["rows"], args["H"], P(args["W"]) if args["W"] else None, args["layout"], args["V"], args["sel"],
        args["row_k"], args["k_max"], P(args["lse"]) if args["lse"] else None,
        P(args["sel_lp"]) if args["sel_lp"] else None, P(args["ids"]) if args["ids"] else None,
        P(args["lps"]) if args["lps"] else None, args["logits_out"], P(args["ws"]), args["ws_bytes"],
        args["status"], None)


def test_project_argument_checks_return_before_launch(lib):
    """Bad arguments give an error status; none of these reach a device."""
    from top_reduction_gb300 import lmh as E
    assert _call_project(lib, rows=-1) == E.ERR_INVALID_ARG
    assert _call_project(lib, H=0) == E.ERR_INVALID_ARG
    assert _call_project(lib, V=0) == E.ERR_INVALID_ARG
    assert _call_project(lib, k_max=-2) == E.ERR_UNSUPPORTED
    assert _call_project(lib, k_max=-1, lps=None) == E.ERR_INVALID_ARG  # full-vocabulary output needs the buffer
    assert _call_project(lib, k_max=-1, lps=0x5004) == E.ERR_INVALID_ARG  # ... 16-byte aligned
    assert _call_project(lib, k_max=129) == E.ERR_UNSUPPORTED
    assert _call_project(lib, k_max=5, V=4) == E.ERR_INVALID_ARG     # k > vocab
    assert _call_project(lib, hidden=0) == E.ERR_INVALID_ARG
    assert _call_project(lib, W=0) == E.ERR_INVALID_ARG
    assert _call_project(lib, lse=0) == E.ERR_INVALID_ARG
    assert _call_project(lib, ids=0) == E.ERR_INVALID_ARG
    assert _call_project(lib, sel=ctypes.c_void_p(0x6000)) == E.ERR_INVALID_ARG  # sel without sel_logprob
    assert _call_project(lib, stride=32) == E.ERR_INVALID_ARG        # stride < H
    assert _call_project(lib, rows=9) == E.ERR_INVALID_ARG           # rows > num_tokens, no row_idx
    assert _call_project(lib, layout=1, V=4100) == E.ERR_UNSUPPORTED  # [H x V] storage needs V % 8 == 0
    assert _call_project(lib, layout=2) == E.ERR_INVALID_ARG
    assert _call_project(lib, layout=7) == E.ERR_INVALID_ARG
    assert _call_project(lib, H=60, stride=60) == E.ERR_UNSUPPORTED  # H % 8
    assert _call_project(lib, W=0x2002) == E.ERR_UNSUPPORTED         # misaligned W
    assert _call_project(lib, rows=0) == E.OK                        # empty batch: nothing to do


def test_from_logits_argument_checks(lib):
    from top_reduction_gb300 import lmh
    P = ctypes.c_void_p

    def call(logits=0x1000, dtype=0, rows=4, V=256, stride=256, k_max=5, lse=0x2000, ids=0x3000,
             lps=0x4000):
        return lib.lmh_logprobs_from_logits(P(logits) if logits else None, dtype, rows, V, stride, None,
                                            None, k_max, P(lse) if lse else None, None,
                                            P(ids) if ids else None, P(lps) if lps else None,
                                            P(0x10000), 1 << 30, None, None)

    assert call(rows=-1) == lmh.ERR_INVALID_ARG
    assert call(stride=100) == lmh.ERR_INVALID_ARG
    assert call(dtype=9) == lmh.ERR_INVALID_ARG
    assert call(logits=0) == lmh.ERR_INVALID_ARG
    assert call(k_max=200) == lmh.ERR_UNSUPPORTED
    assert call(k_max=300, V=256) == lmh.ERR_UNSUPPORTED
    assert call(logits=0x1001) == lmh.ERR_UNSUPPORTED                # not element aligned
    assert call(logits=0x1002, dtype=2) == lmh.ERR_UNSUPPORTED       # fp32 on a 2-byte boundary
    assert call(rows=0) == lmh.OK


def test_select_rows_argument_checks(lib):
    from top_reduction_gb300 import lmh
    P = ctypes.c_void_p
    assert lib.lmh_select_rows(None, 1, 0, None, 4, P(0x10), P(0x20), None, None) == lmh.ERR_INVALID_ARG
    assert lib.lmh_select_rows(P(0x10), -1, 0, None, 4, P(0x10), P(0x20), None, None) == lmh.ERR_INVALID_ARG
    assert lib.lmh_select_rows(P(0x10), 2, 3, None, 4, P(0x10), P(0x20), None, None) == lmh.ERR_INVALID_ARG
    assert lib.lmh_select_rows(P(0x10), 2, 0, None, 4, None, P(0x20), None, None) == lmh.ERR_INVALID_ARG


def test_product_path_has_no_fallback():
    """The binding raises when the library is missing instead of computing anything itself."""
    from top_reduction_gb300 import lmh
    src = open(lmh.__file__).read()
    assert "oracle" not in src and "import numpy" not in src
    saved, lmh._lib = lmh._lib, None
    real = lmh.LIB_PATH
    try:
        lmh.LIB_PATH = real + ".missing"
        with pytest.raises(ImportError):
            lmh.load()
    finally:
        lmh.LIB_PATH = real
        lmh._lib = saved


def test_head_transform_and_probe_argument_checks(lib):
    """The scaled projection and the probe reject bad transforms before any launch."""
    from top_reduction_gb300 import lmh as E
    P = ctypes.c_void_p
    for bad in (0.0, -0.5, float("inf"), float("nan")):
        st = lib.lmh_project_logprobs_scaled(
            P(0x1000), 64, 8, None, 8, 64, P(0x2000), 0, 4096, None, None, 5, P(0x3000), None, P(0x4000),
            P(0x5000), None, P(0x10000), 1 << 30, None, bad, None)
        assert st == E.ERR_INVALID_ARG, bad
    probe = dict(ref=P(0x8000), tol=0.0, count=P(0x9000), scale=1.0)

    def call(**kw):
        a = dict(probe, **kw)
        return lib.lmh_probe_selective(P(0x1000), 64, 8, None, 8, 64, P(0x2000), 4096, a["scale"], a["ref"],
                                       a["tol"], a["count"], P(0x10000), 1 << 30, None, None)
    assert call(ref=None) == E.ERR_INVALID_ARG
    assert call(count=None) == E.ERR_INVALID_ARG
    assert call(tol=-1.0) == E.ERR_INVALID_ARG
    assert call(tol=float("nan")) == E.ERR_INVALID_ARG
    assert call(scale=0.0) == E.ERR_INVALID_ARG
