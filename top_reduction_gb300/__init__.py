"""top_reduction_gb300 -- LM-head logprob path for one GB300 GPU (sm_103a).

The compute lives in liblmh.so (CUDA kernels behind the C ABI of
include/lmh.h); this package is its thin Python binding.
"""
from .lmh import (BF16, F16, F32, K_FULL, K_MAX, LMHError, PATH_FROM_LOGITS, PATH_PROBE, PATH_PROJECT, W_HV, W_VH,
                  count_selected_rows, gather_records, load, logprobs_from_logits, merge_records, probe_selective,
                  project_logprobs, project_partials, record_bytes, select_rows, status_string, trace_enable,
                  trace_read, trace_reset, vocab_parallel_logprobs, vocab_share, workspace_bytes)

__all__ = ["BF16", "F16", "F32", "K_FULL", "K_MAX", "LMHError", "PATH_FROM_LOGITS", "PATH_PROBE", "PATH_PROJECT",
           "W_HV", "W_VH",
           "count_selected_rows", "gather_records", "load", "logprobs_from_logits", "merge_records",
           "probe_selective", "project_logprobs", "project_partials", "record_bytes", "select_rows",
           "status_string", "trace_enable", "trace_read", "trace_reset", "vocab_parallel_logprobs", "vocab_share",
           "workspace_bytes"]
