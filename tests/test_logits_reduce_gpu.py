"""lmh_logprobs_from_logits vs the oracle: ids bit-exact, values within 1e-5.

Full-size 256 x 248320 bf16 chunks in every distribution of the prompt-scoring
workload (normal, peaked, gumbel, ties, -inf) at K = 0, 1, 20, 128, plus
ragged vocabularies, fp32 / fp16 inputs, per-row K, strided rows, a row of
only -inf, and selected-token edge cases.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_from_logits, check_logprob_identity

pytestmark = pytest.mark.gpu

_ORACLE_DT = {torch.bfloat16: oracle.BF16, torch.float16: oracle.F16}


def oracle_ref(x, sel, k_max, row_k=None):
    if x.dtype in _ORACLE_DT:
        arr, dt = workloads.bits(x), _ORACLE_DT[x.dtype]
    else:
        arr, dt = x.contiguous().numpy(), None
    return oracle.logprobs(arr, dtype=dt, sel=None if sel is None else np.asarray(sel),
                           row_k=row_k, k_max=k_max)


def gpu_run(lmh, x_dev, sel, k_max, row_k=None):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = lmh.logprobs_from_logits(x_dev, sel=sel, row_k=row_k, k_max=k_max, dev_status=st)
    torch.cuda.synchronize()
    return o, int(st.item())


def _prefix(orc, k):
    return {"lse": orc["lse"], "sel_logprob": orc["sel_logprob"],
            "topk_ids": orc["topk_ids"][:, :k], "topk_logprobs": orc["topk_logprobs"][:, :k]}


@pytest.fixture(scope="module", params=workloads.DISTRIBUTIONS)
def chunk(request):
    c = workloads.logits_chunk(request.param)
    c["oracle"] = oracle_ref(c["logits"], c["sel"], 128)  # top-128; smaller K are its prefixes
    return c


@pytest.mark.parametrize("k", [0, 1, 20, 128])
def test_full_chunk(lmh, chunk, k):
    x = chunk["logits"].cuda()
    o, st = gpu_run(lmh, x, chunk["sel"], k)
    assert st == 0
    check_from_logits(o, _prefix(chunk["oracle"], k), k, what="%s K=%d" % (chunk["dist"], k))
    if k:
        check_logprob_identity(o, chunk["logits"], k)


def test_ragged_vocab_and_ties(lmh):
    for V in (4100, 65, 64, 130, 1000):
        c = workloads.logits_chunk("ties", rows=37, V=V, k_for_ties=20)
        k = min(128, V)
        o, st = gpu_run(lmh, c["logits"].cuda(), c["sel"], k)
        assert st == 0
        check_from_logits(o, oracle_ref(c["logits"], c["sel"], k), k, what="V=%d" % V)


def test_tiny_vocab_k_equals_v(lmh):
    x = torch.randn(5, 10).to(torch.bfloat16)
    x[1, 3] = x[1, 7]
    sel = torch.tensor([0, 3, 9, -1, 5], dtype=torch.int32)
    o, st = gpu_run(lmh, x.cuda(), sel, 10)
    assert st == 0
    check_from_logits(o, oracle_ref(x, sel, 10), 10, what="V=10")


def test_neginf_edge_rows(lmh):
    """A row of only -inf, rows with fewer finite logits than K, whole -inf blocks."""
    V = 248320
    x = workloads.logits_chunk("neginf", rows=6, V=V)["logits"]
    x[0] = float("-inf")                     # the degenerate row
    x[1] = float("-inf")
    x[1, [5, 100000, 248319]] = torch.tensor([1.0, 1.0, 2.0]).to(torch.bfloat16)  # 3 finite < K
    x[2, :V - 64] = float("-inf")            # only the last block finite
    sel = torch.tensor([3, 100000, V - 1, 0, -1, 7], dtype=torch.int32)
    o, st = gpu_run(lmh, x.cuda(), sel, 20)
    assert st == 0
    check_from_logits(o, oracle_ref(x, sel, 20), 20, what="neginf edges")
    assert torch.isneginf(o["lse"][0]) and torch.isnan(o["topk_logprobs"][0]).all()
    assert o["topk_ids"][0].tolist() == list(range(20))


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16])
def test_other_dtypes(lmh, dtype):
    g = torch.Generator().manual_seed(5)
    x = (torch.randn(64, 50000, generator=g) * 3).to(dtype)
    x[3, 100:140] = x[3, 7]                   # exact ties
    sel = torch.randint(0, 50000, (64,), generator=g, dtype=torch.int32)
    o, st = gpu_run(lmh, x.cuda(), sel, 128)
    assert st == 0
    check_from_logits(o, oracle_ref(x, sel, 128), 128, what=str(dtype))
    check_logprob_identity(o, x, 128)


def test_per_row_k(lmh):
    c = workloads.logits_chunk("normal", rows=64, V=151936)
    row_k = np.random.default_rng(3).integers(0, 21, size=64).astype(np.int32)
    row_k[0], row_k[1] = 0, 20
    o, st = gpu_run(lmh, c["logits"].cuda(), c["sel"], 20, row_k=torch.from_numpy(row_k))
    assert st == 0
    check_from_logits(o, oracle_ref(c["logits"], c["sel"], 20, row_k=row_k), 20, row_k=row_k, what="row_k")


def test_strided_rows(lmh):
    """Rows that are a view into a wider buffer (row stride > V)."""
    c = workloads.logits_chunk("gumbel", rows=16, V=4096 + 64)
    wide = torch.full((16, 4096 + 128), 99.0, dtype=torch.bfloat16)
    wide[:, :4096 + 64] = c["logits"]
    view = wide.cuda()[:, :4096 + 64]
    o, st = gpu_run(lmh, view, c["sel"], 20)
    assert st == 0
    check_from_logits(o, oracle_ref(c["logits"], c["sel"], 20), 20, what="strided")


def test_single_row_full_vocab(lmh):
    c = workloads.logits_chunk("peaked", rows=1)
    o, st = gpu_run(lmh, c["logits"].cuda(), c["sel"], 128)
    assert st == 0
    check_from_logits(o, oracle_ref(c["logits"], c["sel"], 128), 128, what="1 row")


def test_selected_token_edge_cases(lmh):
    from top_reduction_gb300 import lmh as L
    x = torch.randn(4, 3000).to(torch.bfloat16)
    sel = torch.tensor([-1, 0, 2999, 3000], dtype=torch.int32)
    o, st = gpu_run(lmh, x.cuda(), sel, 5)
    assert st & L.DS_SEL_OUT_OF_RANGE
    lp = o["sel_logprob"].cpu()
    assert torch.isnan(lp[0]) and torch.isnan(lp[3])
    orc = oracle_ref(x, torch.tensor([-1, 0, 2999, -1], dtype=torch.int32), 5)
    check_from_logits(o, {**orc, "sel_logprob": np.array([np.nan, orc["sel_logprob"][1],
                                                          orc["sel_logprob"][2], np.nan])}, 5)


def test_no_selected_tokens(lmh):
    x = torch.randn(3, 700).to(torch.bfloat16)
    o, st = gpu_run(lmh, x.cuda(), None, 3)
    assert st == 0 and o["sel_logprob"] is None
    check_from_logits(o, oracle_ref(x, None, 3), 3)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_layout_paths(lmh, dtype):
    """Row lengths and offsets on both sides of the 16-byte alignment the bulk-copy path needs.

    Rows whose start and length are multiples of 16 bytes are streamed through
    shared memory; the others are read with vector or element loads.  Partial
    last blocks, f32 blocks split over two threads and a start one element
    past the alignment are all covered.
    """
    g = torch.Generator().manual_seed(11)
    for V, offset in ((40, 0), (1000, 0), (1001, 0), (2056, 0), (3000, 1), (5000, 0)):
        wide = (torch.randn(9, V + 24, generator=g) * 2).to(dtype)
        wide[2, offset + 5:offset + 25] = wide[2, offset + 3]      # ties inside a block and across blocks
        x = wide[:, offset:offset + V]
        sel = torch.randint(-1, V, (9,), generator=g, dtype=torch.int32)
        k = min(20, V)
        o, st = gpu_run(lmh, wide.cuda()[:, offset:offset + V], sel, k)
        assert st == 0
        check_from_logits(o, oracle_ref(x.contiguous(), sel, k), k, what="%s V=%d offset=%d" % (dtype, V, offset))


def _oracle_full(x, lse):
    """Full-vocabulary logprobs from the oracle's lse: x - lse in f64 (x widened exactly)."""
    return x.float().double().numpy() - np.asarray(lse)[:, None]


def test_full_vocabulary_output(lmh, chunk):
    """k_max = LMH_K_FULL (openinfer issue #719, Acceptance criteria: the -1 full-vocabulary
    contract): every id's logprob in id order, within 1e-5 of x - lse."""
    if chunk["dist"] not in ("normal", "neginf"):
        pytest.skip("two distributions suffice for the elementwise output")
    from top_reduction_gb300 import lmh as L
    x = chunk["logits"]
    o, st = gpu_run(lmh, x.cuda(), chunk["sel"], L.K_FULL)
    assert st == 0 and o["topk_ids"] is None
    assert o["topk_logprobs"].shape == x.shape
    orc = chunk["oracle"]
    check_from_logits({"lse": o["lse"], "sel_logprob": o["sel_logprob"]},
                      {"lse": orc["lse"], "sel_logprob": orc["sel_logprob"]}, 0, what="full lse")
    got = o["topk_logprobs"].cpu().numpy()
    want = _oracle_full(x, orc["lse"])
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.max(np.abs(got[fin] - want[fin])) <= 1e-5


@pytest.mark.parametrize("dtype,V", [(torch.bfloat16, 4100), (torch.float32, 1001), (torch.float16, 3000)])
def test_full_vocabulary_ragged(lmh, dtype, V):
    from top_reduction_gb300 import lmh as L
    g = torch.Generator().manual_seed(V)
    x = (torch.randn(7, V, generator=g) * 3).to(dtype)
    sel = torch.randint(-1, V, (7,), generator=g, dtype=torch.int32)
    o, st = gpu_run(lmh, x.cuda(), sel, L.K_FULL)
    assert st == 0
    orc = oracle_ref(x, sel, 0)
    check_from_logits({"lse": o["lse"], "sel_logprob": o["sel_logprob"]},
                      {"lse": orc["lse"], "sel_logprob": orc["sel_logprob"]}, 0, what="full ragged")
    assert np.max(np.abs(o["topk_logprobs"].cpu().numpy() - _oracle_full(x, orc["lse"]))) <= 1e-5


def test_back_to_back_calls_overlap(lmh):
    """Calls enqueued back to back on one stream and one workspace, with no synchronisation
    between them: each stream kernel may start (and load its first chunks) while the previous
    call's select kernel still reads the workspace.  Every call still matches the oracle."""
    from top_reduction_gb300 import lmh as L
    V = 60000
    rows = (96, 64, 96, 80, 96)
    need = max(L.workspace_bytes(r, 0, V, 20, L.PATH_FROM_LOGITS) for r in rows)
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    chunks = [workloads.logits_chunk("normal", seed=60 + i, rows=r, V=V) for i, r in enumerate(rows)]
    dev = [(c["logits"].cuda(), c["sel"].cuda()) for c in chunks]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    outs = [lmh.logprobs_from_logits(x, sel=s, k_max=20, workspace=ws, dev_status=st) for x, s in dev]
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for i, (c, o) in enumerate(zip(chunks, outs)):
        check_from_logits(o, oracle_ref(c["logits"], c["sel"], 20), 20, what="call %d" % i)


def test_reused_workspace_schedules(lmh):
    """One workspace over several calls: its first call finds no valid chunk-counter base and
    hands out the chunks in a fixed order; the later calls draw them from the counter. Every
    call matches the oracle, on different inputs and row counts, and a workspace whose counter
    words hold leftovers of another use is still read correctly."""
    from top_reduction_gb300 import lmh as L
    V = 50000
    need = max(L.workspace_bytes(r, 0, V, 20, L.PATH_FROM_LOGITS) for r in (64, 48))
    ws = torch.full((need,), 0x5A, dtype=torch.uint8, device="cuda")  # leftovers, not zeros
    for i, rows in enumerate((64, 48, 64, 64)):
        c = workloads.logits_chunk("normal", seed=40 + i, rows=rows, V=V)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        o = lmh.logprobs_from_logits(c["logits"].cuda(), sel=c["sel"], k_max=20, workspace=ws, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        check_from_logits(o, oracle_ref(c["logits"], c["sel"], 20), 20, what="call %d" % i)
