"""Thin ctypes binding of liblmh (include/lmh.h).

Argument marshalling only: tensors are passed as device pointers and the
current torch CUDA stream as the launch stream; outputs and the workspace are
allocated with torch (the caching allocator), and every step of the path runs
in the library's CUDA kernels.  There is no fallback: if liblmh.so is missing
or no CUDA device is present, the calls raise.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblmh.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE_TOO_SMALL, ERR_CUDA, ERR_TIMEOUT = range(6)
BF16, F16, F32 = 0, 1, 2
W_VH, W_HV = 0, 1
PATH_PROJECT, PATH_FROM_LOGITS, PATH_PROBE = 0, 1, 2
K_MAX = 128
K_FULL = -1  # k_max for the full-vocabulary output: topk_logprobs is [rows, V] in id order

DS_BAD_CU_SEQLENS = 0x1
DS_SEL_OUT_OF_RANGE = 0x2
DS_ROWS_OVERFLOW = 0x4
DS_ROW_IDX_OUT_OF_RANGE = 0x8
DS_TIMEOUT = 0x10
DS_NO_ALLOWED_TOKEN = 0x20


class Sampling(ctypes.Structure):
    """struct lmh_sampling (include/lmh.h)."""
    _fields_ = [("temperature", ctypes.c_void_p), ("allowed_mask", ctypes.c_void_p), ("mask_words", ctypes.c_int32),
                ("seed", ctypes.c_uint64), ("offsets", ctypes.c_void_p), ("sampled_ids", ctypes.c_void_p),
                ("sampled_logprob", ctypes.c_void_p)]

EXPORTS = ("lmh_select_rows", "lmh_count_selected_rows", "lmh_workspace_bytes",
           "lmh_project_logprobs", "lmh_project_logprobs_scaled", "lmh_project_logprobs_sample",
           "lmh_probe_selective",
           "lmh_logprobs_from_logits", "lmh_status_string",
           "lmh_version", "lmh_trace_enable", "lmh_trace_read", "lmh_trace_reset", "lmh_debug_set_wait_limit",
           "lmh_record_bytes", "lmh_project_partials", "lmh_merge_workspace_bytes", "lmh_merge_records")

_lib = None


class LMHError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s failed: %s" % (what, status_string(status)))


def load():
    """Load liblmh.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("liblmh.so is not built (%s); run __graft_entry__.build() or "
                          "python top_reduction_gb300/_build.py" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.lmh_select_rows.argtypes = [P, i32, i32, P, i32, P, P, P, P]
    lib.lmh_select_rows.restype = ctypes.c_int
    lib.lmh_count_selected_rows.argtypes = [P, i32, i32, P]
    lib.lmh_count_selected_rows.restype = i32
    lib.lmh_workspace_bytes.argtypes = [i32, i32, i32, i32, ctypes.c_int]
    lib.lmh_workspace_bytes.restype = u64
    lib.lmh_project_logprobs.argtypes = [P, i64, i32, P, i32, i32, P, ctypes.c_int, i32, P, P, i32,
                                         P, P, P, P, P, P, u64, P, P]
    lib.lmh_project_logprobs.restype = ctypes.c_int
    lib.lmh_project_logprobs_scaled.argtypes = [P, i64, i32, P, i32, i32, P, ctypes.c_int, i32, P, P, i32,
                                                P, P, P, P, P, P, u64, P, ctypes.c_float, P]
    lib.lmh_project_logprobs_scaled.restype = ctypes.c_int
    lib.lmh_project_logprobs_sample.argtypes = [P, i64, i32, P, i32, i32, P, ctypes.c_int, i32, P, P, i32,
                                                P, P, P, P, P, P, u64, P, ctypes.c_float,
                                                ctypes.POINTER(Sampling), P]
    lib.lmh_project_logprobs_sample.restype = ctypes.c_int
    lib.lmh_probe_selective.argtypes = [P, i64, i32, P, i32, i32, P, i32, ctypes.c_float, P, ctypes.c_float, P,
                                        P, u64, P, P]
    lib.lmh_probe_selective.restype = ctypes.c_int
    lib.lmh_logprobs_from_logits.argtypes = [P, ctypes.c_int, i32, i32, i64, P, P, i32, P, P, P, P,
                                             P, u64, P, P]
    lib.lmh_logprobs_from_logits.restype = ctypes.c_int
    lib.lmh_status_string.argtypes = [ctypes.c_int]
    lib.lmh_status_string.restype = ctypes.c_char_p
    lib.lmh_version.restype = i32
    lib.lmh_trace_enable.argtypes = [i32]
    lib.lmh_trace_enable.restype = ctypes.c_int
    lib.lmh_trace_read.argtypes = [ctypes.c_char_p, ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_double)]
    lib.lmh_trace_read.restype = ctypes.c_int
    lib.lmh_trace_reset.restype = None
    lib.lmh_debug_set_wait_limit.argtypes = [ctypes.c_uint64]
    lib.lmh_debug_set_wait_limit.restype = ctypes.c_int
    lib.lmh_record_bytes.argtypes = [i32]
    lib.lmh_record_bytes.restype = u64
    lib.lmh_project_partials.argtypes = [P, i64, i32, P, i32, i32, P, ctypes.c_int, i32, i32, i32, P, P, i32,
                                         P, P, u64, P, P]
    lib.lmh_project_partials.restype = ctypes.c_int
    lib.lmh_merge_workspace_bytes.argtypes = [i32, i32, i32]
    lib.lmh_merge_workspace_bytes.restype = u64
    lib.lmh_merge_records.argtypes = [P, i32, i32, i32, P, P, i32, P, P, P, P, P, u64, P, P]
    lib.lmh_merge_records.restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status):
    return load().lmh_status_string(int(status)).decode()


def _check(status, what):
    if status != OK:
        raise LMHError(status, what)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev_i32(t, device, n=None, name="array"):
    if t is None:
        return None
    t = torch.as_tensor(t, dtype=torch.int32, device=device).contiguous()
    if n is not None and t.numel() != n:
        raise ValueError("%s must have %d entries" % (name, n))
    return t


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def count_selected_rows(cu_seqlens_host, num_decode, all_rows_mask_host=None):
    """Rows lmh_select_rows will select, from host copies (no device sync)."""
    cu = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).cpu().contiguous()
    mask = None
    if all_rows_mask_host is not None:
        mask = torch.as_tensor(all_rows_mask_host, dtype=torch.uint8).cpu().contiguous()
    n = load().lmh_count_selected_rows(ctypes.c_void_p(cu.data_ptr()), cu.numel() - 1, int(num_decode),
                                       None if mask is None else ctypes.c_void_p(mask.data_ptr()))
    if n < 0:
        raise ValueError("invalid packed batch (cu_seqlens / num_decode)")
    return int(n)


def select_rows(cu_seqlens, num_decode, all_rows_mask=None, max_out_rows=None, dev_status=None,
                stream=None):
    """Device row selection.  Returns (row_idx int32[max_out_rows], logits_cu_seqlens int32[S+1]).

    Pass max_out_rows (e.g. from count_selected_rows on a host copy) to avoid
    the device synchronisation needed to read cu_seqlens[-1].
    """
    cu = cu_seqlens
    assert cu.is_cuda and cu.dtype == torch.int32 and cu.is_contiguous()
    S = cu.numel() - 1
    if max_out_rows is None:
        max_out_rows = int(cu[-1].item()) if cu.numel() else 0
    row_idx = torch.empty(max(int(max_out_rows), 1), dtype=torch.int32, device=cu.device)
    lcu = torch.empty(S + 1, dtype=torch.int32, device=cu.device)
    mask = None
    if all_rows_mask is not None:
        mask = torch.as_tensor(all_rows_mask, dtype=torch.uint8, device=cu.device).contiguous()
    _check(load().lmh_select_rows(_p(cu), S, int(num_decode), _p(mask), int(max_out_rows), _p(row_idx),
                                  _p(lcu), _p(dev_status), _stream(stream)), "lmh_select_rows")
    return row_idx[:max_out_rows], lcu


def workspace_bytes(rows, hidden, vocab, k_max, path):
    n = load().lmh_workspace_bytes(int(rows), int(hidden), int(vocab), int(k_max), int(path))
    if n == 0:
        raise LMHError(ERR_INVALID_ARG, "lmh_workspace_bytes")
    return int(n)


def _outputs(rows, k_max, with_sel, device, V=None):
    out = {"lse": torch.empty(rows, dtype=torch.float32, device=device)}
    out["sel_logprob"] = torch.empty(rows, dtype=torch.float32, device=device) if with_sel else None
    if k_max == K_FULL:  # every id's logprob, in id order; no ids
        out["topk_ids"] = None
        out["topk_logprobs"] = torch.empty((rows, V), dtype=torch.float32, device=device)
        return out
    out["topk_ids"] = torch.empty((rows, k_max), dtype=torch.int32, device=device)
    out["topk_logprobs"] = torch.empty((rows, k_max), dtype=torch.float32, device=device)
    return out


def _workspace(workspace, nbytes, device):
    if workspace is None:
        return torch.empty(nbytes, dtype=torch.uint8, device=device)
    assert workspace.numel() * workspace.element_size() >= nbytes
    return workspace


def project_logprobs(hidden, W, row_idx=None, rows=None, sel=None, row_k=None, k_max=0,
                     logits_out=None, workspace=None, dev_status=None, out=None, stream=None, logit_scale=1.0,
                     sampling=None, w_layout=W_VH):
    """Selective head projection + per-row lse / selected logprob / top-k.

    hidden: bf16 [T, H] (rows may be strided); W: bf16 [V, H] (lm_head.weight), or
    [H, V] with w_layout=W_HV (V a multiple of 8);
    row_idx: int32 [rows] device tensor or None (rows 0..rows-1).
    logit_scale: head transform, every logit is logit_scale * (A . W)
    (lmh_project_logprobs_scaled); 1.0 is the plain projection.
    sampling: dict with optional temperature (fp32 [rows]), mask (int32/uint32 [rows, words]
    allowed-token bits), seed (int), offsets (int64 [rows]): device-side Gumbel-max sampling
    (lmh_project_logprobs_sample); adds sampled_ids and sampled_logprob to the result.
    Returns a dict with lse, sel_logprob (or None), topk_ids, topk_logprobs.
    """
    assert hidden.is_cuda and hidden.dtype == torch.bfloat16 and hidden.dim() == 2
    assert hidden.stride(1) == 1
    assert W.is_cuda and W.dtype == torch.bfloat16 and W.dim() == 2 and W.is_contiguous()
    T, H = hidden.shape
    assert w_layout in (W_VH, W_HV)
    V = W.shape[0] if w_layout == W_VH else W.shape[1]
    assert W.shape[1 if w_layout == W_VH else 0] == H
    dev = hidden.device
    if row_idx is not None:
        rows = row_idx.numel() if rows is None else rows
        assert row_idx.dtype == torch.int32 and row_idx.is_cuda
    elif rows is None:
        rows = T
    sel_t = _dev_i32(sel, dev, rows, "sel")
    rk_t = _dev_i32(row_k, dev, rows, "row_k")
    o = out if out is not None else _outputs(rows, k_max, sel_t is not None, dev, V)
    ws = _workspace(workspace, workspace_bytes(rows, H, V, k_max, PATH_PROJECT), dev)
    args = (_p(hidden), hidden.stride(0) if T > 1 else H, T, _p(row_idx), int(rows), H, _p(W), int(w_layout), V,
            _p(sel_t), _p(rk_t), int(k_max), _p(o["lse"]), _p(o["sel_logprob"]), _p(o["topk_ids"]),
            _p(o["topk_logprobs"]), _p(logits_out), _p(ws), ws.numel() * ws.element_size(), _p(dev_status))
    if sampling is not None:
        def dev(t, dtype):
            return None if t is None else torch.as_tensor(t, dtype=dtype, device=dev_).contiguous()
        dev_ = hidden.device
        temp = dev(sampling.get("temperature"), torch.float32)
        mask = sampling.get("mask")
        if mask is not None:
            mask = torch.as_tensor(mask, device=dev_).contiguous()
            assert mask.dim() == 2 and mask.shape[0] == rows and mask.element_size() == 4
        offs = dev(sampling.get("offsets"), torch.int64)
        o["sampled_ids"] = torch.empty(rows, dtype=torch.int32, device=dev_)
        o["sampled_logprob"] = torch.empty(rows, dtype=torch.float32, device=dev_)
        def addr(t):
            return None if t is None else t.data_ptr()
        sp = Sampling(addr(temp), addr(mask), 0 if mask is None else mask.shape[1],
                      int(sampling.get("seed", 0)) & (2 ** 64 - 1), addr(offs), addr(o["sampled_ids"]),
                      addr(o["sampled_logprob"]))
        _check(load().lmh_project_logprobs_sample(*args, float(logit_scale), ctypes.byref(sp), _stream(stream)),
               "lmh_project_logprobs_sample")
    elif logit_scale == 1.0:
        _check(load().lmh_project_logprobs(*args, _stream(stream)), "lmh_project_logprobs")
    else:
        _check(load().lmh_project_logprobs_scaled(*args, float(logit_scale), _stream(stream)),
               "lmh_project_logprobs_scaled")
    return o


def probe_selective(hidden, W, ref_logits, row_idx=None, rows=None, logit_scale=1.0, tolerance=0.0,
                    workspace=None, dev_status=None, stream=None):
    """Mismatching elements between this library's head output for the given rows and the
    model's own logits `ref_logits` (f32 [rows, V]); returns a device uint32 tensor [1]."""
    assert hidden.is_cuda and hidden.dtype == torch.bfloat16 and hidden.dim() == 2 and hidden.stride(1) == 1
    assert W.is_cuda and W.dtype == torch.bfloat16 and W.is_contiguous()
    T, H = hidden.shape
    V = W.shape[0]
    if row_idx is not None:
        rows = row_idx.numel() if rows is None else rows
    elif rows is None:
        rows = T
    assert ref_logits.is_cuda and ref_logits.dtype == torch.float32 and ref_logits.is_contiguous()
    assert tuple(ref_logits.shape) == (rows, V)
    dev = hidden.device
    count = torch.empty(1, dtype=torch.int32, device=dev)
    ws = _workspace(workspace, workspace_bytes(rows, H, V, 0, PATH_PROBE), dev)
    st = load().lmh_probe_selective(
        _p(hidden), hidden.stride(0) if T > 1 else H, T, _p(row_idx), int(rows), H, _p(W), V, float(logit_scale),
        _p(ref_logits), float(tolerance), _p(count), _p(ws), ws.numel() * ws.element_size(), _p(dev_status),
        _stream(stream))
    _check(st, "lmh_probe_selective")
    return count


_DTYPES = {torch.bfloat16: BF16, torch.float16: F16, torch.float32: F32}


def logprobs_from_logits(logits, sel=None, row_k=None, k_max=0, workspace=None, dev_status=None,
                         out=None, stream=None):
    """Per-row lse / selected logprob / top-k of given logits [rows, V] (bf16, f16 or f32)."""
    assert logits.is_cuda and logits.dim() == 2 and logits.stride(1) == 1
    rows, V = logits.shape
    dev = logits.device
    sel_t = _dev_i32(sel, dev, rows, "sel")
    rk_t = _dev_i32(row_k, dev, rows, "row_k")
    o = out if out is not None else _outputs(rows, k_max, sel_t is not None, dev, V)
    ws = _workspace(workspace, workspace_bytes(rows, 0, V, k_max, PATH_FROM_LOGITS), dev)
    stride = logits.stride(0) if rows > 1 else V
    st = load().lmh_logprobs_from_logits(
        _p(logits), _DTYPES[logits.dtype], rows, V, stride, _p(sel_t), _p(rk_t), int(k_max),
        _p(o["lse"]), _p(o["sel_logprob"]), _p(o["topk_ids"]), _p(o["topk_logprobs"]), _p(ws),
        ws.numel() * ws.element_size(), _p(dev_status), _stream(stream))
    _check(st, "lmh_logprobs_from_logits")
    return o


# ---------------------------------------------------------------------------
# kernel trace
# ---------------------------------------------------------------------------

TRACE_KERNELS = ("select_rows", "gather_rows", "head_logprobs", "logits_reduce", "merge_partials",
                 "logits_select", "full_logprobs")


def trace_enable(on=True):
    _check(load().lmh_trace_enable(1 if on else 0), "lmh_trace_enable")


def trace_reset():
    load().lmh_trace_reset()


def trace_read(kernel):
    """(launches, total_ms) of a kernel since the last reset (waits for its events)."""
    n = ctypes.c_int64(0)
    ms = ctypes.c_double(0.0)
    _check(load().lmh_trace_read(kernel.encode(), ctypes.byref(n), ctypes.byref(ms)), "lmh_trace_read")
    return int(n.value), float(ms.value)


def debug_set_wait_limit(limit_ns):
    """Test hook: the kernels' bounded waits give up after limit_ns (0: the 2 s default)."""
    _check(load().lmh_debug_set_wait_limit(int(limit_ns)), "lmh_debug_set_wait_limit")


# ---------------------------------------------------------------------------
# vocabulary-parallel head (several GPUs, each holding a share of the vocabulary)
# ---------------------------------------------------------------------------

def vocab_share(V, rank, world):
    """(v_begin, v_count): rank's share of token ids [0, V), whole 64-id blocks spread as
    evenly as possible (the last share takes the ragged tail).  Pure host arithmetic."""
    assert 0 <= rank < world and V >= 1
    nblk = (V + 63) // 64
    lo = (nblk * rank) // world
    hi = (nblk * (rank + 1)) // world
    begin, end = 64 * lo, min(V, 64 * hi)
    return begin, max(0, end - begin)


def record_bytes(k_max):
    """Bytes of one row's record (include/lmh.h: lmh_record_bytes)."""
    n = int(load().lmh_record_bytes(int(k_max)))
    if n == 0:
        raise LMHError(ERR_INVALID_ARG, "lmh_record_bytes")
    return n


def project_partials(hidden, W_share, v_begin, V, row_idx=None, rows=None, sel=None, row_k=None, k_max=0,
                     records=None, workspace=None, dev_status=None, stream=None):
    """One share of a vocabulary-parallel head (lmh_project_partials).

    W_share: bf16 [v_count, H], rows v_begin.. of lm_head.weight; sel holds global ids.
    Returns the uint8 [rows, record_bytes(k_max)] record buffer.
    """
    assert hidden.is_cuda and hidden.dtype == torch.bfloat16 and hidden.dim() == 2 and hidden.stride(1) == 1
    assert W_share.is_cuda and W_share.dtype == torch.bfloat16 and W_share.is_contiguous()
    T, H = hidden.shape
    v_count = W_share.shape[0]
    assert W_share.shape[1] == H
    dev = hidden.device
    if row_idx is not None:
        rows = row_idx.numel() if rows is None else rows
        assert row_idx.dtype == torch.int32 and row_idx.is_cuda
    elif rows is None:
        rows = T
    sel_t = _dev_i32(sel, dev, rows, "sel")
    rk_t = _dev_i32(row_k, dev, rows, "row_k")
    rb = record_bytes(k_max)
    if records is None:
        records = torch.empty((rows, rb), dtype=torch.uint8, device=dev)
    assert records.is_cuda and records.is_contiguous() and records.numel() >= rows * rb
    ws = _workspace(workspace, workspace_bytes(rows, H, v_count, k_max, PATH_PROJECT), dev)
    _check(load().lmh_project_partials(
        _p(hidden), hidden.stride(0) if T > 1 else H, T, _p(row_idx), int(rows), H, _p(W_share), W_VH,
        int(v_begin), int(v_count), int(V), _p(sel_t), _p(rk_t), int(k_max), _p(records), _p(ws),
        ws.numel() * ws.element_size(), _p(dev_status), _stream(stream)), "lmh_project_partials")
    return records


def merge_records(records, num_parts, rows, V, sel=None, row_k=None, k_max=0, workspace=None, dev_status=None,
                  out=None, stream=None):
    """Final results from the gathered records [num_parts, rows, record_bytes] (lmh_merge_records)."""
    assert records.is_cuda and records.is_contiguous()
    dev = records.device
    sel_t = _dev_i32(sel, dev, rows, "sel")
    rk_t = _dev_i32(row_k, dev, rows, "row_k")
    o = out if out is not None else _outputs(rows, k_max, sel_t is not None, dev, V)
    need = int(load().lmh_merge_workspace_bytes(int(rows), int(num_parts), int(k_max)))
    if need == 0:
        raise LMHError(ERR_INVALID_ARG, "lmh_merge_workspace_bytes")
    ws = _workspace(workspace, need, dev)
    _check(load().lmh_merge_records(
        _p(records), int(num_parts), int(rows), int(V), _p(sel_t), _p(rk_t), int(k_max), _p(o["lse"]),
        _p(o["sel_logprob"]), _p(o["topk_ids"]), _p(o["topk_logprobs"]), _p(ws), ws.numel() * ws.element_size(),
        _p(dev_status), _stream(stream)), "lmh_merge_records")
    return o


def gather_records(records, group=None):
    """All-gather of every rank's record buffer, in rank order: [world, *records.shape].

    The one exchange step of the vocabulary-parallel head (a collective of the
    caller's torch.distributed group: NCCL into device memory on GPUs, gloo on the
    host).  Pure plumbing: the records are opaque bytes here.
    """
    import torch.distributed as dist
    world = dist.get_world_size(group)
    out = torch.empty((world,) + tuple(records.shape), dtype=records.dtype, device=records.device)
    if dist.get_backend(group) == "nccl":
        dist.all_gather_into_tensor(out, records.contiguous(), group=group)
    else:
        dist.all_gather(list(out.unbind(0)), records.contiguous(), group=group)
    return out


def vocab_parallel_logprobs(hidden, W_share, v_begin, V, row_idx=None, rows=None, sel=None, row_k=None, k_max=0,
                            group=None, dev_status=None, stream=None):
    """The rows' O(k+1) results with the head split over the ranks of `group` by vocabulary:
    this rank's share (project_partials), one all-gather of the records, the merge."""
    rec = project_partials(hidden, W_share, v_begin, V, row_idx=row_idx, rows=rows, sel=sel, row_k=row_k,
                           k_max=k_max, dev_status=dev_status, stream=stream)
    allrec = gather_records(rec, group)
    n = rec.shape[0]
    return merge_records(allrec, allrec.shape[0], n, V, sel=sel, row_k=row_k, k_max=k_max, dev_status=dev_status,
                         stream=stream)
