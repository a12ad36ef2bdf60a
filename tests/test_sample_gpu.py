"""lmh_project_logprobs_sample vs the oracle: Gumbel-max draws in the head epilogue.

The oracle draws from the same Philox4x32-10 noise in f64 (tests/test_oracle_pins.py pins
the generator and the sampler).  GPU and oracle must pick the same token, except where
the oracle's score of the GPU's token is within the fp32 rounding of the head (Higham's
bound on the dot product, over T) and of the noise of its own best score: a certified
near-tie.  Masks, greedy rows, a row with no allowed token, one-split plans and the
decode shape are covered; the top-k of the same call stays exact.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import TOL_FUSED, assert_close, check_fused, higham_delta

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def _case(rows, H, V, seed, w_scale=1.0):
    g = torch.Generator().manual_seed(seed)
    T = rows + 3
    hidden = torch.randn(T, H, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, H, generator=g) * (w_scale / H ** 0.5)).to(torch.bfloat16)
    ri = torch.randperm(T, generator=g)[:rows].to(torch.int32)
    return hidden, W, ri, g


def _mask(rows, V, rng, p_allow=0.3):
    words = (V + 31) // 32
    bits = rng.random((rows, words * 32)) < p_allow
    bits[:, V:] = False
    m = np.zeros((rows, words), dtype=np.uint32)
    for b in range(32):
        m |= (bits[:, b::32].astype(np.uint32) << np.uint32(b))
    return m


def check_draws(ids_g, lp_g, z, lse, temp, mask, seed, offsets, A, W, what):
    """GPU draws equal the oracle's, or are certified near-ties; logprobs within 2e-2."""
    ids_o, best, _ = oracle.sample(z, temperature=temp, mask=mask, seed=seed, offsets=offsets)
    rows = z.shape[0]
    certified = 0
    for i in range(rows):
        g, o = int(ids_g[i]), int(ids_o[i])
        if o < 0:
            assert g == -1 and math.isnan(lp_g[i]), (what, i)
            continue
        assert g >= 0, (what, i)
        if mask is not None:
            assert (mask[i, g // 32] >> np.uint32(g % 32)) & 1, (what, i, "masked token drawn")
        assert abs(lp_g[i] - (z[i, g] - lse[i])) <= TOL_FUSED, (what, i)
        if g == o:
            continue
        T = float(temp[i]) if temp is not None else 1.0
        off = int(offsets[i]) if offsets is not None else i
        Wc = W[[g, o]].float().double().numpy()
        dz = higham_delta(A[i], Wc)
        if T > 0:
            s_g = z[i, g] / T - math.log(-math.log(oracle.sample_uniform(seed, off, g)))
            bound = (dz.sum()) / T + 1e-5 * (1.0 + abs(best[i]))
        else:
            s_g = z[i, g]
            bound = dz.sum()
        gap = best[i] - s_g
        assert gap <= 2 * bound, "%s row %d: gpu %d vs oracle %d, gap %g > %g" % (what, i, g, o, gap, 2 * bound)
        certified += 1
    return certified


@pytest.mark.parametrize("rows,H,V,k", [(200, 136, 4100, 5), (129, 64, 1000, 0), (17, 64, 2000, 20),
                                        (50, 96, 30000, 8)])
def test_sampling_with_mask_and_temperatures(lmh, rows, H, V, k):
    hidden, W, ri, g = _case(rows, H, V, rows * 3 + V, w_scale=3.0)
    rng = np.random.default_rng(rows + V)
    temp = rng.choice(np.array([0.0, 0.7, 1.0, 1.5], dtype=np.float32), size=rows)
    mask = _mask(rows, V, rng)
    mask[1] = 0                                           # a row with no allowed token
    offsets = rng.integers(0, 2 ** 40, size=rows, dtype=np.int64)
    seed = 0x1234_5678_9ABC
    sel = torch.randint(-1, V, (rows,), generator=g, dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = lmh.project_logprobs(hidden.cuda(), W.cuda(), row_idx=ri.cuda(), sel=sel, k_max=k, dev_status=st,
                             sampling={"temperature": temp, "mask": mask.view(np.int32), "seed": seed,
                                       "offsets": offsets})
    torch.cuda.synchronize()
    from top_reduction_gb300 import lmh as L
    assert int(st.item()) == L.DS_NO_ALLOWED_TOKEN
    z = oracle.project(_bits(hidden), _bits(W), row_idx=ri.numpy())
    orc = oracle.logprobs(z, sel=sel.numpy(), k_max=k)
    A = hidden[ri.long()].float().double().numpy()
    check_fused(o, orc, z, A, W, k, what="sample+topk")
    check_draws(o["sampled_ids"].cpu().numpy(), o["sampled_logprob"].cpu().numpy(), z, orc["lse"], temp, mask,
                seed, offsets, A, W, "rows %d" % rows)


def test_sampling_decode_shape(lmh):
    """32 rows x 2560 x 151936 (the decode batch's head), T 1, no mask, default offsets."""
    rows, H, V = 32, 2560, 151936
    g = torch.Generator().manual_seed(77)
    hidden = torch.randn(rows, H, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, H, generator=g) * 0.02).to(torch.bfloat16)
    o = lmh.project_logprobs(hidden.cuda(), W.cuda(), k_max=5, sampling={"seed": 2024})
    torch.cuda.synchronize()
    z = oracle.project(_bits(hidden), _bits(W))
    orc = oracle.logprobs(z, k_max=5)
    A = hidden.float().double().numpy()
    check_fused(o, orc, z, A, W, 5, what="decode sample")
    check_draws(o["sampled_ids"].cpu().numpy(), o["sampled_logprob"].cpu().numpy(), z, orc["lse"], None, None,
                2024, None, A, W, "decode")


def test_greedy_equals_top1(lmh):
    """T <= 0 draws the argmax: the same token as the call's own top-1 (ties to the smaller id)."""
    hidden, W, ri, _ = _case(300, 128, 20000, 5)
    rows = 300
    o = lmh.project_logprobs(hidden.cuda(), W.cuda(), row_idx=ri.cuda(), k_max=1,
                             sampling={"temperature": np.zeros(rows, np.float32)})
    torch.cuda.synchronize()
    assert torch.equal(o["sampled_ids"], o["topk_ids"][:, 0])
    assert torch.equal(o["sampled_logprob"], o["topk_logprobs"][:, 0])


def test_sampling_one_split_plan(lmh):
    """A plan with one vocabulary range per row: the head kernel writes the draw itself."""
    rows, H, V = 10000, 128, 200
    hidden, W, ri, _ = _case(rows, H, V, 9)
    rng = np.random.default_rng(9)
    temp = rng.choice(np.array([0.0, 0.8, 1.2], dtype=np.float32), size=rows)
    offsets = np.arange(rows, dtype=np.int64) * 7 + 3
    o = lmh.project_logprobs(hidden.cuda(), W.cuda(), row_idx=ri.cuda(), k_max=0,
                             sampling={"temperature": temp, "seed": 99, "offsets": offsets})
    torch.cuda.synchronize()
    sample = np.unique(np.concatenate([[0, 1, rows - 1], rng.choice(rows, 300, replace=False)]))
    z = oracle.project(_bits(hidden), _bits(W), row_idx=ri.numpy()[sample])
    orc = oracle.logprobs(z, k_max=0)
    A = hidden[ri.long()[torch.as_tensor(sample)]].float().double().numpy()
    assert_close(o["lse"].cpu().numpy()[sample], orc["lse"], TOL_FUSED, "one split lse")
    check_draws(o["sampled_ids"].cpu().numpy()[sample], o["sampled_logprob"].cpu().numpy()[sample], z, orc["lse"],
                temp[sample], None, 99, offsets[sample], A, W, "one split")


@pytest.mark.parametrize("rows,H,V,k,w_scale", [(9, 256, 50000, 5, 3.0), (4096, 64, 32768, 0, 1.0),
                                                (4096, 64, 32768, 3, 6.0)])
def test_sampling_candidate_filter(lmh, rows, H, V, k, w_scale):
    """Plans where the head scores only candidate tokens (a raw-word test against the
    row's best score so far): at most 16 rows per warp, or 128 blocks per row and
    vocabulary range.  Draws vs the oracle on every row (small batch) or a sample."""
    hidden, W, ri, g = _case(rows, H, V, rows + V + 1, w_scale=w_scale)
    rng = np.random.default_rng(rows + H)
    temp = rng.choice(np.array([0.0, 0.5, 1.0, 2.0], dtype=np.float32), size=rows)
    mask = _mask(rows, V, rng, p_allow=0.6) if rows < 64 else None
    offsets = rng.integers(0, 2 ** 62, size=rows, dtype=np.int64)
    seed = 0xC0FFEE
    o = lmh.project_logprobs(hidden.cuda(), W.cuda(), row_idx=ri.cuda(), k_max=k,
                             sampling={"temperature": temp, "seed": seed, "offsets": offsets,
                                       "mask": None if mask is None else mask.view(np.int32)})
    torch.cuda.synchronize()
    sample = np.arange(rows) if rows < 64 else np.unique(np.concatenate([[0, rows - 1], rng.choice(rows, 160, replace=False)]))
    z = oracle.project(_bits(hidden), _bits(W), row_idx=ri.numpy()[sample])
    orc = oracle.logprobs(z, k_max=k)
    A = hidden[ri.long()[torch.as_tensor(sample)]].float().double().numpy()
    assert_close(o["lse"].cpu().numpy()[sample], orc["lse"], TOL_FUSED, "filter lse")
    check_draws(o["sampled_ids"].cpu().numpy()[sample], o["sampled_logprob"].cpu().numpy()[sample], z, orc["lse"],
                temp[sample], None if mask is None else mask[sample], seed, offsets[sample], A, W, "filter")


@pytest.mark.parametrize("rows", [64, 16])
def test_sampling_noise_tail_accuracy(lmh, rows):
    """Draws decided by the largest noises: per row two allowed tokens whose words are
    the row's two largest of 65536 (noise near 11, u within about 1e-4 of 1), with
    logits and temperature set so that their scores differ by 1e-3 -- above the
    certified near-tie band, so the GPU must pick the oracle's token.  A noise whose
    logarithm of u loses relative accuracy near u = 1 misses by more than that.  64 rows
    score every token; 16 rows take the candidate filter."""
    H, V = 64, 65536
    seed = 0x5EED_0001
    cand = np.arange(2 * rows, dtype=np.int64) * 1000003 + 17
    z0 = np.zeros((cand.size, V))
    ones = np.ones(cand.size, dtype=np.float32)
    a, g_a, _ = oracle.sample(z0, temperature=ones, seed=seed, offsets=cand)
    words = V // 32
    no_a = np.full((cand.size, words), 0xFFFFFFFF, dtype=np.uint32)
    no_a[np.arange(cand.size), a // 32] &= ~(np.uint32(1) << (a % 32).astype(np.uint32))
    b, g_b, _ = oracle.sample(z0, temperature=ones, seed=seed, offsets=cand, mask=no_a)
    keep = np.nonzero(g_a - g_b > 0.01)[0][:rows]  # offsets whose two largest words differ
    assert keep.size == rows
    offsets, a, b, g_a, g_b = cand[keep], a[keep], b[keep], g_a[keep], g_b[keep]
    assert np.all(g_a > 9.0) and np.all(g_b > 8.0)
    delta = np.where(np.arange(rows) % 2 == 0, 1e-3, -1e-3)  # b wins on even rows, a on odd rows
    temp = (1.0 / (g_a - g_b + delta)).astype(np.float32)
    gap = 1.0 / temp.astype(np.float64) + g_b - g_a  # score(b) - score(a) with the stored temperature
    assert np.all(np.abs(np.abs(gap) - 1e-3) < 1e-5)
    hidden = torch.zeros(rows, H)
    hidden[torch.arange(rows), torch.arange(rows) % H] = 1.0
    W = torch.zeros(V, H)
    W[torch.as_tensor(b), torch.arange(rows) % H] = 1.0  # z[i, b_i] = 1, every other logit 0
    hidden, W = hidden.to(torch.bfloat16), W.to(torch.bfloat16)
    mask = np.zeros((rows, words), dtype=np.uint32)
    for i in range(rows):
        for t in (a[i], b[i]):
            mask[i, t // 32] |= np.uint32(1) << np.uint32(t % 32)
    o = lmh.project_logprobs(hidden.cuda(), W.cuda(), k_max=0,
                             sampling={"temperature": temp, "mask": mask.view(np.int32), "seed": seed,
                                       "offsets": offsets})
    torch.cuda.synchronize()
    z = oracle.project(_bits(hidden), _bits(W))
    ids_o, _, _ = oracle.sample(z, temperature=temp, mask=mask, seed=seed, offsets=offsets)
    assert np.array_equal(ids_o, np.where(gap > 0, b, a))
    assert np.array_equal(o["sampled_ids"].cpu().numpy(), ids_o)
