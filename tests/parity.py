"""Comparison helpers for GPU-vs-oracle parity tests.

Acceptance (stated once, used by every parity test):
  * row selection, logits_cu_seqlens and top-k ids from given logits: bit-exact;
  * lse / logprobs from given bf16, f16 or f32 logits: within 1e-5 absolute
    (the logits widen exactly to fp32 and fp64, so ids and order are identical);
  * fused head (bf16 inputs, fp32 accumulation): logits, lse and logprobs
    within 2e-2 absolute; top-k ids bit-exact, except where the oracle's own
    values at the two swapped ids differ by no more than 2*delta, with
    delta = gamma_H * sum_h |A[h] * W[h][v]| and gamma_H = H*u/(1 - H*u),
    u = 2^-24 (the fp32 dot-product error bound, Higham, "Accuracy and
    Stability of Numerical Algorithms", section 3.1): such a swap is a
    certified near-tie and is counted, any other mismatch fails.  The named
    workloads (tiny, decode, selective prefill, mixed step, full arm) assert
    that the count is 0: their smallest adjacent top-k gaps are far above the
    fp32 accumulation error, so a correct kernel reproduces the ids exactly.
    With a head transform (logit scale s != 1) the kernel rounds s * z once
    more, so the window there also takes 2^-23 * |z| (one fp32 rounding of the
    product).
"""
import numpy as np

TOL_FROM_LOGITS = 1e-5
TOL_FUSED = 2e-2


def _close(a, b, atol):
    """Elementwise |a - b| <= atol, with -inf == -inf, +inf == +inf and NaN == NaN."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    same_nan = np.isnan(a) & np.isnan(b)
    same_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        ok = np.abs(a - b) <= atol
    return ok | same_nan | same_inf


def assert_close(a, b, atol, what):
    ok = _close(a, b, atol)
    if not ok.all():
        bad = np.argwhere(~ok)
        i = tuple(bad[0])
        raise AssertionError("%s: %d mismatches (> %g); first at %s: gpu %r oracle %r"
                             % (what, len(bad), atol, i, np.asarray(a)[i], np.asarray(b)[i]))


def row_k_of(k_max, rows, row_k=None):
    if row_k is None:
        return np.full(rows, k_max, dtype=np.int64)
    return np.clip(np.asarray(row_k, dtype=np.int64), 0, k_max)


def check_from_logits(gpu, orc, k_max, row_k=None, atol=TOL_FROM_LOGITS, what=""):
    """Bit-exact ids, values within atol; ranks >= k_i are (-1, -inf)."""
    assert_close(gpu["lse"].cpu().numpy(), orc["lse"], atol, what + " lse")
    if "sel_logprob" in orc:
        assert_close(gpu["sel_logprob"].cpu().numpy(), orc["sel_logprob"], atol, what + " sel_logprob")
    if k_max == 0:
        return
    ids_g = gpu["topk_ids"].cpu().numpy()
    lp_g = gpu["topk_logprobs"].cpu().numpy()
    ks = row_k_of(k_max, ids_g.shape[0], row_k)
    for i in range(ids_g.shape[0]):
        k = ks[i]
        if not np.array_equal(ids_g[i, :k], orc["topk_ids"][i, :k]):
            j = int(np.argmax(ids_g[i, :k] != orc["topk_ids"][i, :k]))
            raise AssertionError("%s row %d rank %d: gpu id %d oracle id %d" %
                                 (what, i, j, ids_g[i, j], orc["topk_ids"][i, j]))
        assert np.all(ids_g[i, k:] == -1), (what, i)
        assert np.all(np.isneginf(lp_g[i, k:])), (what, i)
        assert_close(lp_g[i, :k], orc["topk_logprobs"][i, :k], atol, "%s row %d logprobs" % (what, i))


def check_logprob_identity(gpu, logits, k_max, row_k=None):
    """Invariant: every returned logprob is fp32(x) - lse evaluated in fp32, bit for bit."""
    import torch
    x = logits.float().cpu()
    lse = gpu["lse"].cpu()
    ids = gpu["topk_ids"].cpu().long()
    lp = gpu["topk_logprobs"].cpu()
    ks = row_k_of(k_max, ids.shape[0], row_k)
    for i in range(ids.shape[0]):
        k = int(ks[i])
        if k == 0:
            continue
        want = x[i, ids[i, :k]] - lse[i]
        got = lp[i, :k]
        same = (want == got) | (torch.isnan(want) & torch.isnan(got))
        assert bool(same.all()), ("logprob != fp32(x) - lse", i)


def higham_delta(a_row_f64, W_f64_cols):
    """delta_v = gamma_H * sum_h |a_h * W[h][v]| for the given columns ([n, H] rows of W)."""
    H = a_row_f64.shape[0]
    u = 2.0 ** -24
    gamma = H * u / (1 - H * u)
    return gamma * np.abs(W_f64_cols * a_row_f64[None, :]).sum(axis=1)


def check_fused(gpu, orc, z_oracle, A_f64, W_bf16_vh, k_max, row_k=None, atol=TOL_FUSED, what="", scale=1.0):
    """Fused-head acceptance; returns the number of certified near-tie swaps.

    With a head transform, z_oracle holds the scaled logits scale * (A . W);
    the near-tie bound is then scale * delta plus the rounding of the product.
    """
    assert_close(gpu["lse"].cpu().numpy(), orc["lse"], atol, what + " lse")
    if "sel_logprob" in orc:
        assert_close(gpu["sel_logprob"].cpu().numpy(), orc["sel_logprob"], atol, what + " sel_logprob")
    if k_max == 0:
        return 0
    ids_g = gpu["topk_ids"].cpu().numpy()
    lp_g = gpu["topk_logprobs"].cpu().numpy()
    ks = row_k_of(k_max, ids_g.shape[0], row_k)
    certified = 0
    for i in range(ids_g.shape[0]):
        k = int(ks[i])
        g, o = ids_g[i, :k], orc["topk_ids"][i, :k]
        assert np.all(ids_g[i, k:] == -1), (what, i)
        assert len(set(g.tolist())) == k, (what, i, "duplicate ids")
        assert np.all((g >= 0) & (g < z_oracle.shape[1])), (what, i, "id out of range")
        assert_close(lp_g[i, :k], z_oracle[i, g] - orc["lse"][i], atol, "%s row %d logprobs" % (what, i))
        if np.array_equal(g, o):
            continue
        for r in np.nonzero(g != o)[0]:
            cols = np.array([g[r], o[r]])
            Wc = W_bf16_vh[cols].float().double().numpy()
            zmax = max(abs(z_oracle[i, g[r]]), abs(z_oracle[i, o[r]]))
            d = scale * higham_delta(A_f64[i], Wc).max()
            if scale != 1.0:  # the epilogue's product scale * z is rounded once more
                d += 2.0 ** -23 * zmax
            gap = abs(z_oracle[i, g[r]] - z_oracle[i, o[r]])
            if gap > 2 * d:
                raise AssertionError(
                    "%s row %d rank %d: gpu id %d (z=%r) vs oracle id %d (z=%r); gap %g > 2*delta %g"
                    % (what, i, r, g[r], z_oracle[i, g[r]], o[r], z_oracle[i, o[r]], gap, 2 * d))
            certified += 1
    return certified
