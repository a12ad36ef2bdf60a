"""Row selection on the GPU (lmh_select_rows) vs the oracle: bit-exact."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "select_rows_examples.json")


def run(lmh, cu, nd, mask=None, max_out=None):
    cu_d = torch.as_tensor(np.asarray(cu, dtype=np.int32)).cuda()
    mask_d = None if mask is None else torch.as_tensor(np.asarray(mask, dtype=np.uint8)).cuda()
    if max_out is None:
        max_out = lmh.count_selected_rows(np.asarray(cu, dtype=np.int32), nd, mask)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ri, lcu = lmh.select_rows(cu_d, nd, mask_d, max_out_rows=max_out, dev_status=st)
    torch.cuda.synchronize()
    return ri.cpu().numpy(), lcu.cpu().numpy(), int(st.item())


def test_golden_examples(lmh):
    for c in json.load(open(GOLDEN))["cases"]:
        ri, lcu, st = run(lmh, c["cu_seqlens"], c["num_decode"], c["all_rows_mask"])
        assert st == 0, c["name"]
        assert ri.tolist() == c["row_idx"], c["name"]
        assert lcu.tolist() == c["logits_cu_seqlens"], c["name"]


@pytest.mark.parametrize("S", [1, 5, 37, 1023, 1024, 1025, 3000])
def test_random_batches(lmh, S):
    rng = np.random.default_rng(S)
    for trial in range(4):
        nd = int(rng.integers(0, S + 1))
        lens = rng.integers(1, 40, size=S)
        lens[:nd] = rng.integers(0, 4, size=nd)  # decode sequences may even be empty
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        mask = (rng.random(S) < 0.1).astype(np.uint8) if trial % 2 else None
        want_ri, want_lcu = oracle.select_rows(cu, nd, mask)
        ri, lcu, st = run(lmh, cu, nd, mask)
        assert st == 0
        assert np.array_equal(ri, want_ri)
        assert np.array_equal(lcu, want_lcu)


@pytest.mark.parametrize("make", [workloads.tiny_batch, workloads.prefill_batch,
                                  lambda: workloads.mixed_batch(with_weights=False)],
                         ids=["tiny_batch", "prefill_batch", "mixed_batch"])
def test_workload_batches(lmh, make):
    b = make()
    cu = b["cu_seqlens"].numpy()
    mask = None if b["all_rows_mask"] is None else b["all_rows_mask"].numpy()
    want_ri, want_lcu = oracle.select_rows(cu, b["num_decode"], mask)
    ri, lcu, st = run(lmh, cu, b["num_decode"], mask)
    assert st == 0 and len(ri) == b["n_sel"]
    assert np.array_equal(ri, want_ri) and np.array_equal(lcu, want_lcu)


def test_pure_decode_is_identity(lmh):
    cu = np.arange(33, dtype=np.int32)
    ri, lcu, st = run(lmh, cu, 32)
    assert st == 0 and ri.tolist() == list(range(32)) and np.array_equal(lcu, cu)


def test_empty_batch(lmh):
    ri, lcu, st = run(lmh, [0], 0, max_out=0)
    assert st == 0 and lcu.tolist() == [0]


@pytest.mark.parametrize("cu,nd", [([1, 2, 3], 0), ([0, 3, 2], 0), ([0, 2, 2], 0), ([0, 1, 1, 4], 1)])
def test_bad_cu_seqlens_sets_status(lmh, cu, nd):
    from top_reduction_gb300 import lmh as L
    with pytest.raises(oracle.OracleError):
        oracle.select_rows(cu, nd)
    _, _, st = run(lmh, cu, nd, max_out=8)
    assert st & L.DS_BAD_CU_SEQLENS


def test_overflow_sets_status_and_keeps_prefix(lmh):
    from top_reduction_gb300 import lmh as L
    cu = np.array([0, 4, 9, 20], dtype=np.int32)
    want, _ = oracle.select_rows(cu, 2)  # 4 + 5 decode rows + 1 prefill row
    ri, lcu, st = run(lmh, cu, 2, max_out=6)
    assert st & L.DS_ROWS_OVERFLOW
    assert np.array_equal(ri[:6], want[:6])
    assert lcu.tolist() == [0, 4, 9, 10]
