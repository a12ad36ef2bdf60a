"""lmh_project_logprobs (row gather + tcgen05 head + fused reduction) vs the oracle.

Fused-head acceptance (tests/parity.py): logits, lse and logprobs within 2e-2
absolute of the f64 oracle; top-k ids bit-exact on the named workloads (no
certified near-tie swap allowed there), bit-exact or a certified near-tie on
the random shapes.
Workloads: the tiny packed batch, the decode batch (K 5 and 1), the
selective prefill batch, the mixed Llama-3-8B-shaped step and the full
16384-row projection arm (sampled rows), plus ragged shapes and invariants.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import TOL_FUSED, assert_close, check_fused

pytestmark = pytest.mark.gpu


def _bits(t):
    return workloads.bits(t)


def gpu_select(lmh, b):
    cu = b["cu_seqlens"].cuda()
    mask = None if b["all_rows_mask"] is None else b["all_rows_mask"].cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ri, _ = lmh.select_rows(cu, b["num_decode"], mask, max_out_rows=b["n_sel"], dev_status=st)
    return ri, st


def gpu_project(lmh, hidden_d, W_d, row_idx=None, rows=None, sel=None, row_k=None, k=5, materialize=False):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    n = rows if rows is not None else (row_idx.numel() if row_idx is not None else hidden_d.shape[0])
    logits = torch.empty((n, W_d.shape[0]), dtype=torch.float32, device="cuda") if materialize else None
    o = lmh.project_logprobs(hidden_d, W_d, row_idx=row_idx, rows=rows, sel=sel, row_k=row_k, k_max=k,
                             logits_out=logits, dev_status=st)
    torch.cuda.synchronize()
    return o, int(st.item()), logits


def oracle_rows(b, packed_rows, sel, k, row_k=None):
    """Oracle projection + reduction of the given packed rows."""
    rows = np.asarray(packed_rows, dtype=np.int32)
    z = oracle.project(_bits(b["hidden"]), _bits(b["W"]), row_idx=rows)
    orc = oracle.logprobs(z, sel=None if sel is None else np.asarray(sel), row_k=row_k, k_max=k)
    A = b["hidden"][torch.as_tensor(rows.astype(np.int64))].float().double().numpy()
    return z, orc, A


@pytest.fixture(scope="module")
def tiny():
    return workloads.tiny_batch()


@pytest.fixture(scope="module")
def decode():
    b = workloads.decode_batch()
    b["hidden_d"], b["W_d"] = b["hidden"].cuda(), b["W"].cuda()
    return b


@pytest.fixture(scope="module")
def prefill():
    b = workloads.prefill_batch()
    b["hidden_d"], b["W_d"] = b["hidden"].cuda(), b["W"].cuda()
    return b


def test_tiny_batch(lmh, tiny):
    b = tiny
    ri, st_sel = gpu_select(lmh, b)
    o, st, logits = gpu_project(lmh, b["hidden"].cuda(), b["W"].cuda(), row_idx=ri, sel=b["sel"], k=5,
                                materialize=True)
    assert st == 0 and int(st_sel.item()) == 0
    want_ri, _ = oracle.select_rows(b["cu_seqlens"].numpy(), b["num_decode"])
    assert np.array_equal(ri.cpu().numpy(), want_ri)
    z, orc, A = oracle_rows(b, want_ri, b["sel"], 5)
    assert_close(logits.cpu().numpy(), z, TOL_FUSED, "tiny logits")
    assert check_fused(o, orc, z, A, b["W"], 5, what="tiny") == 0


@pytest.mark.parametrize("k", [5, 1])
def test_decode_batch(lmh, decode, k):
    b = decode
    o, st, _ = gpu_project(lmh, b["hidden_d"], b["W_d"], sel=b["sel"], k=k)
    assert st == 0
    z, orc, A = oracle_rows(b, np.arange(32), b["sel"], k)
    assert check_fused(o, orc, z, A, b["W"], k, what="decode K=%d" % k) == 0


def test_prefill_selective(lmh, prefill):
    b = prefill
    ri, _ = gpu_select(lmh, b)
    o, st, _ = gpu_project(lmh, b["hidden_d"], b["W_d"], row_idx=ri, sel=b["sel"], k=20)
    assert st == 0
    assert ri.cpu().tolist() == [2048 * (j + 1) - 1 for j in range(8)]
    z, orc, A = oracle_rows(b, ri.cpu().numpy(), b["sel"], 20)
    assert check_fused(o, orc, z, A, b["W"], 20, what="prefill selective") == 0


def test_full_projection_arm_sampled(lmh, prefill):
    """All 16384 rows through the head (the 'before' arm), K=20; sampled rows vs the oracle."""
    b = prefill
    o, st, _ = gpu_project(lmh, b["hidden_d"], b["W_d"], sel=b["sel_all"], k=20)
    assert st == 0
    rng = np.random.default_rng(0)
    sample = np.unique(np.concatenate([[0, 127, 128, 2047, 16383], rng.choice(16384, 11, replace=False)]))
    z, orc, A = oracle_rows(b, sample, b["sel_all"][sample], 20)
    sub = {key: v[torch.as_tensor(sample)] for key, v in o.items() if v is not None}
    assert check_fused(sub, orc, z, A, b["W"], 20, what="full arm") == 0


def test_mixed_step_sampled(lmh):
    b = workloads.mixed_batch()
    hidden_d, W_d = b["hidden"].cuda(), b["W"].cuda()
    ri, st_sel = gpu_select(lmh, b)
    o, st, _ = gpu_project(lmh, hidden_d, W_d, row_idx=ri, sel=b["sel"], row_k=b["row_k"], k=20)
    assert st == 0 and int(st_sel.item()) == 0
    want_ri, _ = oracle.select_rows(b["cu_seqlens"].numpy(), b["num_decode"], b["all_rows_mask"].numpy())
    assert np.array_equal(ri.cpu().numpy(), want_ri)
    sample = np.array([0, 5, 31, 32, 63, 64, 65, 67, 68, 69, 500, 1000, 1090, 1091])
    rk = b["row_k"][sample].numpy()
    z, orc, A = oracle_rows(b, want_ri[sample], b["sel"][sample], 20, row_k=rk)
    sub = {key: v[torch.as_tensor(sample)] for key, v in o.items() if v is not None}
    assert check_fused(sub, orc, z, A, b["W"], 20, row_k=rk, what="mixed") == 0


@pytest.mark.parametrize("rows,H,V,k", [(200, 136, 4100, 20), (129, 64, 1000, 128), (3, 520, 70000, 0),
                                        (1, 8, 300, 7), (300, 1024, 20000, 33), (64, 256, 9000, 12),
                                        (130, 512, 12000, 30), (17, 64, 2000, 3), (16, 64, 40000, 128),
                                        # vocabulary ranges per row on 152 SMs: 128 (the warp-per-row
                                        # merge at 4 lists per lane), 129 (one CTA per row), 98 at K 32
                                        (40, 256, 32768, 20), (24, 128, 33000, 20), (50, 192, 25000, 32)])
def test_ragged_shapes(lmh, rows, H, V, k):
    g = torch.Generator().manual_seed(rows * 7 + H)
    T = rows + 5
    b = {"hidden": torch.randn(T, H, generator=g).to(torch.bfloat16),
         "W": (torch.randn(V, H, generator=g) / H ** 0.5).to(torch.bfloat16)}
    ri = torch.randperm(T, generator=g)[:rows].to(torch.int32)
    sel = torch.randint(-1, V, (rows,), generator=g, dtype=torch.int32)
    o, st, logits = gpu_project(lmh, b["hidden"].cuda(), b["W"].cuda(), row_idx=ri.cuda(), sel=sel, k=k,
                                materialize=True)
    assert st == 0
    z, orc, A = oracle_rows(b, ri.numpy(), sel, k)
    assert_close(logits.cpu().numpy(), z, TOL_FUSED, "ragged logits")
    check_fused(o, orc, z, A, b["W"], k, what="ragged %s" % ((rows, H, V, k),))


def test_fused_equals_reduction_of_its_own_logits(lmh, decode):
    """The fused epilogue reduces exactly the fp32 logits the same kernel writes out."""
    b = decode
    o, st, logits = gpu_project(lmh, b["hidden_d"], b["W_d"], sel=b["sel"], k=20, materialize=True)
    assert st == 0
    r = lmh.logprobs_from_logits(logits, sel=b["sel"], k_max=20)
    torch.cuda.synchronize()
    assert torch.equal(o["topk_ids"], r["topk_ids"])
    assert torch.allclose(o["lse"], r["lse"], rtol=1e-6, atol=0)
    assert torch.allclose(o["topk_logprobs"], r["topk_logprobs"], rtol=0, atol=1e-5)
    assert torch.allclose(o["sel_logprob"], r["sel_logprob"], rtol=0, atol=1e-5)


def test_selected_rows_equal_full_projection_sliced(lmh, tiny):
    """mlxcel PR #1969: the row sliced before the head equals the full forward's row."""
    b = tiny
    hidden_d, W_d = b["hidden"].cuda(), b["W"].cuda()
    ri, _ = gpu_select(lmh, b)
    _, _, sel_logits = gpu_project(lmh, hidden_d, W_d, row_idx=ri, k=0, materialize=True)
    _, _, full_logits = gpu_project(lmh, hidden_d, W_d, k=0, materialize=True)
    assert torch.equal(sel_logits, full_logits[ri.long()])
    shifted = torch.clamp(ri + 1, max=63)
    assert not torch.equal(sel_logits, full_logits[shifted.long()])


@pytest.mark.parametrize("rows,T,H,V", [(5, 64, 128, 4096), (37, 300, 512, 3000), (200, 260, 256, 2000),
                                         (129, 140, 64, 1000)])
def test_gather_paths_agree(lmh, rows, T, H, V):
    """The selected rows' logits are the full projection's rows, bit for bit, whether the row
    gather copies 16-byte vectors (aligned rows) or elements (a row stride that is not a
    multiple of 8 elements, which the head then reads from the gathered copy)."""
    g = torch.Generator().manual_seed(rows + T)
    hidden = torch.randn(T, H, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, H, generator=g) / H ** 0.5).to(torch.bfloat16).cuda()
    ri = torch.randperm(T, generator=g)[:rows].to(torch.int32).cuda()
    _, st0, full = gpu_project(lmh, hidden.cuda(), W, k=0, materialize=True)
    _, st1, by_vector = gpu_project(lmh, hidden.cuda(), W, row_idx=ri, k=0, materialize=True)
    padded = torch.zeros(T, H + 3, dtype=torch.bfloat16)
    padded[:, :H] = hidden
    odd = padded.cuda()[:, :H]  # row stride H + 3
    _, st2, by_element = gpu_project(lmh, odd, W, row_idx=ri, k=0, materialize=True)
    assert st0 == st1 == st2 == 0
    want = full[ri.long()]
    assert torch.equal(by_vector, want)
    assert torch.equal(by_element, want)


def test_row_idx_out_of_range_sets_status(lmh, tiny):
    from top_reduction_gb300 import lmh as L
    b = tiny
    ri = torch.tensor([0, 64, 5], dtype=torch.int32, device="cuda")  # 64 == num_tokens
    o, st, logits = gpu_project(lmh, b["hidden"].cuda(), b["W"].cuda(), row_idx=ri, k=3, materialize=True)
    assert st & L.DS_ROW_IDX_OUT_OF_RANGE
    assert torch.count_nonzero(logits[1]) == 0


@pytest.mark.parametrize("rows,H,V,k,gather", [(19400, 64, 512, 20, False), (10000, 128, 200, 128, True)])
def test_single_split_plans(lmh, rows, H, V, k, gather):
    """Plans with one vocabulary split: the head kernel writes lse, the selected
    logprob and the top-k itself (no merge launch).  152 row tiles of one split
    each, or a vocabulary of one column tile; per-row K includes 0 and ranks
    past a row's K; sampled rows vs the oracle."""
    g = torch.Generator().manual_seed(rows + V)
    T = rows + (7 if gather else 0)
    b = {"hidden": torch.randn(T, H, generator=g).to(torch.bfloat16),
         "W": (torch.randn(V, H, generator=g) / H ** 0.5).to(torch.bfloat16)}
    ri = torch.randperm(T, generator=g)[:rows].to(torch.int32) if gather else None
    sel = torch.randint(-1, V, (rows,), generator=g, dtype=torch.int32)
    row_k = torch.randint(0, k + 1, (rows,), generator=g, dtype=torch.int32)
    o, st, _ = gpu_project(lmh, b["hidden"].cuda(), b["W"].cuda(), row_idx=None if ri is None else ri.cuda(),
                           rows=rows, sel=sel, row_k=row_k, k=k)
    assert st == 0
    rng = np.random.default_rng(1)
    sample = np.unique(np.concatenate([[0, 1, 127, 128, rows - 1], rng.choice(rows, 120, replace=False)]))
    packed = sample if ri is None else ri.numpy()[sample]
    rk = row_k.numpy()[sample]
    z, orc, A = oracle_rows(b, packed, sel.numpy()[sample], k, row_k=rk)
    sub = {key: v[torch.as_tensor(sample)] for key, v in o.items() if v is not None}
    check_fused(sub, orc, z, A, b["W"], k, row_k=rk, what="one split %s" % ((rows, H, V, k),))


@pytest.mark.parametrize("scale", [0.0625, 1.0 / 8.0, 3.5])
def test_head_transform_logit_scale(lmh, scale):
    """Head transform (vllm-metal release, Summary: Cohere's logit_scale multiplies
    the logits, Granite's logits_scaling divides them): every logit is
    scale * (A . W) before the reduction, and in logits_out."""
    rows, H, V, k = 200, 136, 4100, 20
    g = torch.Generator().manual_seed(int(scale * 1000) + 11)
    T = rows + 5
    b = {"hidden": torch.randn(T, H, generator=g).to(torch.bfloat16),
         "W": (torch.randn(V, H, generator=g) / H ** 0.5 * 4).to(torch.bfloat16)}
    ri = torch.randperm(T, generator=g)[:rows].to(torch.int32)
    sel = torch.randint(-1, V, (rows,), generator=g, dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.empty((rows, V), dtype=torch.float32, device="cuda")
    o = lmh.project_logprobs(b["hidden"].cuda(), b["W"].cuda(), row_idx=ri.cuda(), sel=sel, k_max=k,
                             logits_out=logits, dev_status=st, logit_scale=scale)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows_np = ri.numpy()
    z = oracle.project(_bits(b["hidden"]), _bits(b["W"]), row_idx=rows_np) * scale
    orc = oracle.logprobs(z, sel=sel.numpy(), k_max=k)
    A = b["hidden"][ri.long()].float().double().numpy()
    assert_close(logits.cpu().numpy(), z, TOL_FUSED, "scaled logits")
    check_fused(o, orc, z, A, b["W"], k, what="logit_scale %g" % scale, scale=scale)


def test_probe_selective(lmh, tiny):
    """The load-time probe (vllm-metal release, Summary and Testing): the selective
    head reproduces the full projection's rows bit-exactly; a head transform that is
    not reproduced is rejected."""
    b = tiny
    hid, W = b["hidden"].cuda(), b["W"].cuda()
    T, V = hid.shape[0], W.shape[0]
    ri, _ = gpu_select(lmh, b)
    rows = ri.numel()
    full = torch.empty((T, V), dtype=torch.float32, device="cuda")
    lmh.project_logprobs(hid, W, k_max=0, logits_out=full)
    full_s = torch.empty((T, V), dtype=torch.float32, device="cuda")
    lmh.project_logprobs(hid, W, k_max=0, logits_out=full_s, logit_scale=0.0625)
    ref = full[ri.long()].contiguous()
    ref_s = full_s[ri.long()].contiguous()
    assert int(lmh.probe_selective(hid, W, ref, row_idx=ri).item()) == 0
    assert int(lmh.probe_selective(hid, W, ref_s, row_idx=ri, logit_scale=0.0625).item()) == 0
    bad = int(lmh.probe_selective(hid, W, ref, row_idx=ri, logit_scale=0.0625).item())
    assert bad > rows * V // 2       # a scaled head checked against unscaled logits: rejected
    assert int(lmh.probe_selective(hid, W, ref_s, row_idx=ri, tolerance=1e30).item()) == 0
    ref_one = ref.clone()
    ref_one[rows - 1, V - 1] += 1.0
    assert int(lmh.probe_selective(hid, W, ref_one, row_idx=ri).item()) == 1


@pytest.mark.parametrize("rows,H,V", [(129, 64, 1000), (8, 1024, 20000)])
def test_full_vocabulary_output(lmh, rows, H, V):
    """k_max = LMH_K_FULL on the head path: every id's logprob z - lse in id order
    (within 2e-2 of the oracle) and exactly fp32(logits_out) - lse."""
    from top_reduction_gb300 import lmh as L
    g = torch.Generator().manual_seed(rows + V)
    T = rows + 3
    b = {"hidden": torch.randn(T, H, generator=g).to(torch.bfloat16),
         "W": (torch.randn(V, H, generator=g) / H ** 0.5).to(torch.bfloat16)}
    ri = torch.randperm(T, generator=g)[:rows].to(torch.int32)
    sel = torch.randint(-1, V, (rows,), generator=g, dtype=torch.int32)
    o, st, logits = gpu_project(lmh, b["hidden"].cuda(), b["W"].cuda(), row_idx=ri.cuda(), sel=sel, k=L.K_FULL,
                                materialize=True)
    assert st == 0 and o["topk_ids"] is None
    z, orc, A = oracle_rows(b, ri.numpy(), sel, 0)
    assert_close(o["lse"].cpu().numpy(), orc["lse"], TOL_FUSED, "full lse")
    full = o["topk_logprobs"].cpu().numpy()
    assert_close(full, z - orc["lse"][:, None], TOL_FUSED, "full logprobs")
    exact = logits.cpu().numpy() - o["lse"].cpu().numpy()[:, None]
    assert np.array_equal(full, exact.astype(np.float32))
    o2, _, _ = gpu_project(lmh, b["hidden"].cuda(), b["W"].cuda(), row_idx=ri.cuda(), sel=sel, k=L.K_FULL)
    assert torch.equal(o2["topk_logprobs"], o["topk_logprobs"])   # same without logits_out


@pytest.mark.parametrize("rows,H,V,k", [(40, 128, 200, 20), (50, 256, 40000, 16), (32, 64, 70001, 5),
                                        (33, 192, 3000, 8), (9, 1024, 151936, 20), (2, 64, 513, 1),
                                        (20, 128, 5000, 25), (24, 2048, 20000, 20), (16, 2560, 9000, 16)])
def test_small_batch_column_split(lmh, rows, H, V, k):
    """Batches of at most 64 rows: with lists of 16 or 20 entries each tile's
    columns are split over the epilogue warps (4 copies of 32 rows, or 2 of 64)
    and the copies' lse, top-k and selected logit are folded per row; lighter
    lists on at most 32 rows take the deep-ring layout (4 KB A slices, 6
    stages; lists of 16-20 on hidden sizes of 2048 and more take it too).  Per-row K,
    selected ids in every block position, a one-split plan
    (V 200) and equal logits in different blocks (duplicated W rows) must all
    match the oracle."""
    g = torch.Generator().manual_seed(rows * 131 + V)
    T = rows + 3
    W = torch.randn(V, H, generator=g) / H ** 0.5
    dup = torch.randint(0, V, (V // 50 + 1,), generator=g)
    W[torch.randint(0, V, (dup.numel(),), generator=g)] = W[dup]  # equal logits at ids in different blocks
    b = {"hidden": torch.randn(T, H, generator=g).to(torch.bfloat16), "W": W.to(torch.bfloat16)}
    ri = torch.randperm(T, generator=g)[:rows].to(torch.int32)
    sel = torch.randint(-1, V, (rows,), generator=g, dtype=torch.int32)
    row_k = torch.randint(0, k + 1, (rows,), generator=g, dtype=torch.int32)
    o, st, logits = gpu_project(lmh, b["hidden"].cuda(), b["W"].cuda(), row_idx=ri.cuda(), sel=sel, row_k=row_k,
                                k=k, materialize=True)
    assert st == 0
    z, orc, A = oracle_rows(b, ri.numpy(), sel.numpy(), k, row_k=row_k.numpy())
    assert_close(logits.cpu().numpy(), z, TOL_FUSED, "column split logits")
    check_fused(o, orc, z, A, b["W"], k, row_k=row_k.numpy(), what="column split %s" % ((rows, H, V, k),))
    r = lmh.logprobs_from_logits(logits, sel=sel, row_k=row_k.cuda(), k_max=k)
    torch.cuda.synchronize()
    assert torch.equal(o["topk_ids"], r["topk_ids"])  # the same fp32 logits give the same ranking


def test_cuda_graph_capture_and_replay(lmh, tiny):
    """The whole step (row selection, gather, head, merge) can be captured in a CUDA
    graph: replays read the inputs' current contents and equal the eager call."""
    b = tiny
    hidden_d, W_d = b["hidden"].cuda(), b["W"].cuda()
    cu = b["cu_seqlens"].cuda()
    n = int(b["n_sel"])
    sel = b["sel"].cuda()
    ws = torch.empty(lmh.workspace_bytes(n, hidden_d.shape[1], W_d.shape[0], 5, lmh.PATH_PROJECT), dtype=torch.uint8,
                     device="cuda")

    def step():
        ri, _ = lmh.select_rows(cu, b["num_decode"], None, max_out_rows=n)
        return lmh.project_logprobs(hidden_d, W_d, row_idx=ri, sel=sel, k_max=5, workspace=ws)

    eager = step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap = step()
    g.replay()
    torch.cuda.synchronize()
    for key in ("lse", "sel_logprob", "topk_ids", "topk_logprobs"):
        assert torch.equal(cap[key], eager[key]), key
    hidden_d.mul_(-1.0)  # new inputs in the same buffers: the replay sees them
    g.replay()
    again = step()
    torch.cuda.synchronize()
    for key in ("lse", "topk_ids", "topk_logprobs"):
        assert torch.equal(cap[key], again[key]), key
    assert not torch.equal(cap["topk_ids"], eager["topk_ids"])


@pytest.mark.parametrize("rows,H,V,k,scale", [(32, 2560, 151936, 5, 1.0), (200, 136, 4104, 20, 1.0),
                                              (9, 1024, 20000, 20, 1.0), (129, 64, 1000, 128, 1.0),
                                              (40, 512, 33000, 8, 0.25)])
def test_w_stored_h_by_v(lmh, rows, H, V, k, scale):
    """W stored [H x V] (vocabulary contiguous, LMH_W_HV): the W slices enter the tensor
    cores vocabulary-major.  Parity with the oracle's [H x V] projection, and the same
    results as the [V x H] call on the transposed weight."""
    from top_reduction_gb300 import lmh as L
    g = torch.Generator().manual_seed(rows + H + V)
    T = rows + 3
    hidden = torch.randn(T, H, generator=g).to(torch.bfloat16)
    W_vh = (torch.randn(V, H, generator=g) * (2.0 / H ** 0.5)).to(torch.bfloat16)
    W_hv = W_vh.t().contiguous()
    ri = torch.randperm(T, generator=g)[:rows].to(torch.int32)
    sel = torch.randint(-1, V, (rows,), generator=g, dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = lmh.project_logprobs(hidden.cuda(), W_hv.cuda(), row_idx=ri.cuda(), sel=sel, k_max=k, dev_status=st,
                             logit_scale=scale, w_layout=L.W_HV)
    ref = lmh.project_logprobs(hidden.cuda(), W_vh.cuda(), row_idx=ri.cuda(), sel=sel, k_max=k, logit_scale=scale)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    z = oracle.project(_bits(hidden), _bits(W_hv), row_idx=ri.numpy(), w_layout=1) * scale
    orc = oracle.logprobs(z, sel=sel.numpy(), k_max=k)
    A = hidden[ri.long()].float().double().numpy()
    check_fused(o, orc, z, A, W_vh, k, what="W [H x V] %s" % ((rows, H, V, k),), scale=scale)
    for key in ("lse", "sel_logprob", "topk_ids", "topk_logprobs"):
        assert torch.equal(o[key], ref[key]), key
