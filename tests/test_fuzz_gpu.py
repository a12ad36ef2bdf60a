"""Seeded random configurations of the head path against the oracle.

Each case draws the batch size (1..300 rows, so every layout of the head kernel is hit: the
deep ring, the column split, plain row tiles and several row tiles), H (a multiple of 8),
V (ragged), K (0..40, per-row K on some cases), a logit scale and, on some cases,
sampling with a mask and mixed temperatures.  Everything must match the oracle as the
targeted tests require: lse and logprobs within 2e-2, ids exact or certified near-ties,
draws exact or certified near-ties.  A quarter of the head cases store W as [H x V]."""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL_FUSED, assert_close, check_fused
from test_sample_gpu import _bits, _mask, check_draws

pytestmark = pytest.mark.gpu

CASES = list(range(40))


@pytest.mark.parametrize("case", CASES)
def test_random_head_configurations(lmh, case):
    rng = np.random.default_rng(1000 + case)
    rows = int(rng.choice([1, 3, 8, 17, 32, 33, 64, 65, 128, 200, 300]))
    H = int(rng.choice([8, 64, 136, 512, 1024]))
    V = int(rng.integers(65, 20000))
    k = int(rng.choice([0, 1, 3, 5, 8, 16, 20, 25, 40]))
    scale = float(rng.choice([1.0, 1.0, 0.5, 2.5]))
    sampled = bool(rng.random() < 0.4)
    if sampled:
        scale = 1.0  # the draw's near-tie bound is stated for unscaled logits
    with_row_k = bool(rng.random() < 0.3) and k > 0
    hv = bool(rng.random() < 0.25)  # W stored [H x V]: V a multiple of 8
    if hv:
        V = max(8, V // 8 * 8)
        k = min(k, V)
    g = torch.Generator().manual_seed(case)
    T = rows + 4
    hidden = torch.randn(T, H, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, H, generator=g) * (2.0 / H ** 0.5)).to(torch.bfloat16)
    ri = torch.randperm(T, generator=g)[:rows].to(torch.int32)
    sel = torch.randint(-1, V, (rows,), generator=g, dtype=torch.int32)
    row_k = torch.randint(0, k + 1, (rows,), generator=g, dtype=torch.int32) if with_row_k else None
    sampling = None
    if sampled:
        temp = rng.choice(np.array([0.0, 0.6, 1.0, 1.7], dtype=np.float32), size=rows)
        mask = _mask(rows, V, rng, p_allow=0.5) if rng.random() < 0.5 else None
        offsets = rng.integers(0, 2 ** 40, size=rows, dtype=np.int64)
        sampling = {"temperature": temp, "seed": 77 + case, "offsets": offsets,
                    "mask": None if mask is None else mask.view(np.int32)}
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    from top_reduction_gb300 import lmh as L
    W_arg = W.t().contiguous() if hv else W
    o = lmh.project_logprobs(hidden.cuda(), W_arg.cuda(), row_idx=ri.cuda(), sel=sel,
                             row_k=None if row_k is None else row_k.cuda(), k_max=k, dev_status=st,
                             logit_scale=scale, sampling=sampling, w_layout=L.W_HV if hv else L.W_VH)
    torch.cuda.synchronize()
    status = int(st.item())
    assert status & ~L.DS_NO_ALLOWED_TOKEN == 0, status
    z = oracle.project(_bits(hidden), _bits(W), row_idx=ri.numpy()) * scale
    rk = None if row_k is None else row_k.numpy()
    orc = oracle.logprobs(z, sel=sel.numpy(), row_k=rk, k_max=k)
    A = hidden[ri.long()].float().double().numpy()
    what = "case %d %s" % (case, (rows, H, V, k, scale, sampled, with_row_k, hv))
    swaps = check_fused(o, orc, z, A, W, k, row_k=rk, what=what, scale=scale)
    print("%s: %d certified near-tie swaps" % (what, swaps))
    if sampled:
        check_draws(o["sampled_ids"].cpu().numpy(), o["sampled_logprob"].cpu().numpy(), z, orc["lse"],
                    sampling["temperature"], None if sampling["mask"] is None else sampling["mask"].view(np.uint32),
                    sampling["seed"], sampling["offsets"], A, W, what)


@pytest.mark.parametrize("case", list(range(24)))
def test_random_logits_configurations(lmh, case):
    """The standalone reduction on random shapes: rows 1..300, ragged V, bf16 / f16 / f32,
    padded row strides (aligned or not), K 0..130 with per-row K on some cases, peaked rows
    and exact ties.  ids bit-exact and values within 1e-5 of the oracle."""
    from test_logits_reduce_gpu import gpu_run, oracle_ref
    from parity import check_from_logits
    rng = np.random.default_rng(5000 + case)
    rows = int(rng.choice([1, 2, 7, 64, 256, 300]))
    V = int(rng.integers(2, 70000))
    k = int(min(V, rng.choice([0, 1, 5, 20, 64, 128])))
    dtype = [torch.bfloat16, torch.float16, torch.float32][int(rng.integers(0, 3))]
    pad = int(rng.choice([0, 0, 8, 3]))
    g = torch.Generator().manual_seed(case)
    x = (torch.randn(rows, V + pad, generator=g) * float(rng.choice([1.0, 4.0])))
    if rng.random() < 0.5:  # a peaked token and a group of exact ties in some rows
        r = int(rng.integers(0, rows))
        x[r, int(rng.integers(0, V))] += 15.0
        ids = torch.randint(0, V, (min(V, 6),), generator=g)
        x[r, ids] = 9.0
    x = x.to(dtype)
    x_dev = x.cuda()[:, :V]  # a strided view on the device when pad > 0
    x = x[:, :V].contiguous()
    sel = torch.randint(-1, V, (rows,), generator=g, dtype=torch.int32)
    row_k = torch.randint(0, k + 1, (rows,), generator=g, dtype=torch.int32) if (k > 0 and rng.random() < 0.3) else None
    o, st = gpu_run(lmh, x_dev, sel.cuda(), k, None if row_k is None else row_k.cuda())
    assert st == 0
    orc = oracle_ref(x, sel.numpy(), k, None if row_k is None else row_k.numpy())
    check_from_logits(o, orc, k, row_k=None if row_k is None else row_k.numpy(),
                      what="case %d %s" % (case, (rows, V, k, dtype, pad)))
