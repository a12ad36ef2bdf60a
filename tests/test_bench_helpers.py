"""Host helpers of bench.py on the CPU: packed copy buffers and output shapes."""
import importlib.util
import os

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_packed_views_are_aligned_disjoint_and_round_trip():
    bench = _bench()
    src = {"hidden": torch.randn(3, 40).to(torch.bfloat16), "cu": torch.arange(5, dtype=torch.int32),
           "sel": torch.tensor([7, -1, 3], dtype=torch.int32)}
    buf, views = bench.packed(src, "cpu")
    spans = []
    for key, v in views.items():
        off = v.data_ptr() - buf.data_ptr()
        assert off % 256 == 0, key
        assert v.shape == src[key].shape and v.dtype == src[key].dtype
        spans.append((off, off + v.numel() * v.element_size()))
        v.copy_(src[key])
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))  # no overlap
    assert spans[-1][1] <= buf.numel()
    # a second buffer with the same layout receives everything in one copy
    buf2, views2 = bench.packed(views, "cpu")
    buf2.copy_(buf)
    for key in src:
        assert torch.equal(views2[key], src[key])


@pytest.mark.parametrize("k", [0, 5, -1])
def test_step_output_shapes(k):
    bench = _bench()
    o = bench.step_outputs(4, k, 100, True, "meta")
    assert o["lse"].shape == (4,) and o["sel_logprob"].shape == (4,)
    if k < 0:
        assert o["topk_ids"] is None and o["topk_logprobs"].shape == (4, 100)
    else:
        assert o["topk_ids"].shape == (4, k) and o["topk_logprobs"].shape == (4, k)
