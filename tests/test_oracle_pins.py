"""Pins for the CPU oracle: it is checked against things other than itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
what the pages or the mathematics fix: hand-worked examples derived from the
pages' rules (tests/golden/), brute force by a different algorithm on tiny
inputs, library routines (torch f64 log_softmax / stable sort, numpy float16),
exact integer arithmetic, closed forms and invariants.  ``test_pins_catch``
plants one plausible mistake at a time in the oracle (its mutation hook) and
checks that at least one pin fails for each.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16)


def _bits(t):
    return workloads.bits(t)


# --------------------------------------------------------------------------
# row selection
# --------------------------------------------------------------------------

def pin_select_examples():
    """Hand-worked examples of the vllm-metal release's selection rule."""
    for c in _golden("select_rows_examples.json")["cases"]:
        ri, lcu = oracle.select_rows(c["cu_seqlens"], c["num_decode"], c["all_rows_mask"])
        assert ri.tolist() == c["row_idx"], c["name"]
        assert lcu.tolist() == c["logits_cu_seqlens"], c["name"]


def pin_select_properties():
    """Properties of the selection on random packed batches (written independently)."""
    rng = np.random.default_rng(7)
    for trial in range(50):
        S = int(rng.integers(1, 40))
        nd = int(rng.integers(0, S + 1))
        lens = rng.integers(1, 9, size=S)
        lens[:nd] = rng.integers(1, 4, size=nd)  # decode sequences: 1..3 rows
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        mask = (rng.random(S) < 0.2).astype(np.uint8)
        ri, lcu = oracle.select_rows(cu, nd, mask)
        taken = []
        for s in range(S):
            got = ri[lcu[s]:lcu[s + 1]].tolist()
            seg = list(range(int(cu[s]), int(cu[s + 1])))
            if s < nd or mask[s]:
                assert got == seg, (trial, s)
            else:
                assert got == [seg[-1]], (trial, s)
            taken += got
        assert taken == ri.tolist()
        assert all(a < b for a, b in zip(taken, taken[1:]))


def pin_select_rejects():
    """Invalid batches are rejected: bad cu[0], non-monotone, empty prefill segment."""
    for cu, nd in (([1, 2, 3], 0), ([0, 3, 2], 0), ([0, 2, 2], 0), ([0, 1, 1, 4], 1)):
        with pytest.raises(oracle.OracleError):
            oracle.select_rows(cu, nd)
    # an empty decode sequence is allowed: it contributes no row
    ri, lcu = oracle.select_rows([0, 0, 1, 5], 2)
    assert ri.tolist() == [0, 4] and lcu.tolist() == [0, 0, 1, 2]


# --------------------------------------------------------------------------
# projection
# --------------------------------------------------------------------------

def pin_project_exact_integers():
    """Small-integer bf16 inputs: the f64 sum is exact; compare with Python ints.

    Non-square shapes and a selected-row subset, so a transposed operand, a
    dropped term or a wrong row index changes the result.
    """
    rng = np.random.default_rng(1)
    T, H, V = 7, 37, 53
    A = rng.integers(-8, 9, size=(T, H))
    Wm = rng.integers(-8, 9, size=(H, V))  # the math [H x V] matrix
    rows = [6, 0, 3]
    hid = _bits(_bf16(A))
    w_vh = _bits(_bf16(Wm.T.copy()))
    w_hv = _bits(_bf16(Wm))
    want = [[sum(int(A[r, h]) * int(Wm[h, v]) for h in range(H)) for v in range(V)] for r in rows]
    for layout, w in ((0, w_vh), (1, w_hv)):
        z = oracle.project(hid, w, row_idx=np.array(rows), w_layout=layout)
        assert z.tolist() == want, layout


def pin_project_against_exact_sum():
    """Random bf16 inputs: each f64 dot product is within n*u of the exact sum."""
    rng = np.random.default_rng(2)
    T, H, V = 3, 64, 40
    hid_t = _bf16(rng.standard_normal((T, H)))
    w_t = _bf16(rng.standard_normal((V, H)) * 0.1)
    z = oracle.project(_bits(hid_t), _bits(w_t))
    A = hid_t.float().double().numpy()
    Wv = w_t.float().double().numpy()
    for i in range(T):
        for v in range(V):
            prods = [A[i, h] * Wv[v, h] for h in range(H)]  # exact in f64
            exact = math.fsum(prods)
            bound = H * 2.0 ** -53 * sum(abs(p) for p in prods) * 1.01 + 1e-300
            assert abs(z[i, v] - exact) <= bound, (i, v)


def pin_selected_equals_full_sliced():
    """mlxcel PR #1969: the row sliced before the head equals the full forward's row."""
    b = workloads.tiny_batch()
    ri, _ = oracle.select_rows(b["cu_seqlens"].numpy(), b["num_decode"])
    hid, w = _bits(b["hidden"]), _bits(b["W"])
    full = oracle.project(hid, w)
    sel = oracle.project(hid, w, row_idx=ri)
    assert np.array_equal(sel, full[ri])
    # the row rule itself: last row of each prefill segment, every decode row
    cu = b["cu_seqlens"].numpy()
    expect = list(range(int(cu[b["num_decode"]]))) + [int(c) - 1 for c in cu[b["num_decode"] + 1:]]
    assert ri.tolist() == expect
    # shifting the slice by one row must break the equality
    shifted = np.minimum(ri + 1, full.shape[0] - 1)
    assert not np.array_equal(oracle.project(hid, w, row_idx=shifted), full[ri])


# --------------------------------------------------------------------------
# log-softmax / top-K
# --------------------------------------------------------------------------

def _brute_topk(x, k):
    """Top-k by k repeated scans for the best remaining entry (lowest id on ties)."""
    taken, out = set(), []
    for _ in range(k):
        best = None
        for v in range(len(x)):
            if v in taken:
                continue
            if best is None or x[v] > x[best]:
                best = v
        taken.add(best)
        out.append(best)
    return out


def pin_brute_force_tiny():
    """V <= 16: lse by an unshifted exactly-rounded sum, top-K by repeated scans."""
    rng = np.random.default_rng(3)
    for trial in range(200):
        V = int(rng.integers(1, 17))
        vals = rng.choice([-2.0, -1.0, -0.5, 0.0, 0.5, 1.0, 1.5, 3.0], size=V)
        if trial % 3 == 0:
            vals = rng.standard_normal(V) * 3
        x = _bf16(vals).double().numpy()
        k = int(rng.integers(0, V + 1))
        sel = int(rng.integers(0, V))
        o = oracle.logprobs(x[None, :], sel=[sel], k_max=k)
        lse = math.log(math.fsum(math.exp(v) for v in x))
        assert abs(o["lse"][0] - lse) <= 1e-12 * max(1.0, abs(lse)), trial
        assert abs(o["sel_logprob"][0] - (x[sel] - lse)) <= 1e-12 * max(1.0, abs(lse))
        ids = _brute_topk(list(x), k)
        assert o["topk_ids"][0].tolist() == ids, (trial, x, k)
        for r, v in enumerate(ids):
            assert abs(o["topk_logprobs"][0, r] - (x[v] - lse)) <= 1e-12 * max(1.0, abs(lse))


def pin_torch_f64_crosscheck():
    """torch f64 log_softmax / logsumexp and a stable sort on bf16 rows (V 4100)."""
    for dist in ("normal", "ties", "neginf"):
        c = workloads.logits_chunk(dist, rows=6, V=4100, k_for_ties=20)
        xb = c["logits"]
        k = 128
        o = oracle.logprobs(_bits(xb), dtype=oracle.BF16, sel=c["sel"].numpy(), k_max=k)
        xd = xb.double()
        lse = torch.logsumexp(xd, dim=1)
        lsm = torch.log_softmax(xd, dim=1)
        assert torch.allclose(torch.from_numpy(o["lse"]), lse, rtol=0, atol=1e-12)
        # stable sort of -x keeps ascending id order among exact ties
        order = torch.sort(-xd, dim=1, stable=True).indices[:, :k]
        assert np.array_equal(o["topk_ids"], order.numpy().astype(np.int32)), dist
        want_lp = torch.gather(lsm, 1, order)
        assert torch.allclose(torch.from_numpy(o["topk_logprobs"]), want_lp, rtol=0, atol=1e-12)
        sel_lp = lsm[torch.arange(6), c["sel"].long()]
        assert torch.allclose(torch.from_numpy(o["sel_logprob"]), sel_lp, rtol=0, atol=1e-12)


def pin_invariants():
    """sum exp(logprob) = 1; top-K inside the K highest-max 64-blocks; logprob order = logit order."""
    rng = np.random.default_rng(4)
    for dist in ("normal", "peaked", "gumbel", "ties"):
        c = workloads.logits_chunk(dist, rows=4, V=4100)
        x = c["logits"].double().numpy()
        V = x.shape[1]
        full = oracle.logprobs(x, k_max=V)
        s = np.exp(full["topk_logprobs"]).sum(axis=1)
        assert np.all(np.abs(s - 1.0) <= 1e-9), dist
        for K in (1, 5, 20, 64):
            for r in range(x.shape[0]):
                ids = full["topk_ids"][r, :K]
                nb = (V + 63) // 64
                bmax = [x[r, 64 * b: 64 * b + 64].max() for b in range(nb)]
                ranked = sorted(range(nb), key=lambda b: (-bmax[b], b))[:K]
                assert set(int(i) // 64 for i in ids) <= set(ranked), (dist, K, r)
        for r in range(x.shape[0]):
            ids = full["topk_ids"][r]
            lps = full["topk_logprobs"][r]
            assert np.all(np.diff(lps) <= 0)
            xv = x[r, ids]
            assert np.all(np.diff(xv) <= 0)
            eq = np.diff(xv) == 0
            assert np.all(np.diff(ids)[eq] > 0), "exact ties must list by ascending id"
        _ = rng


def pin_closed_forms():
    """All-equal row, one finite entry, peaked row, whole row -inf, K=0."""
    V = 300
    for c in (0.0, 2.5, -7.0):
        o = oracle.logprobs(np.full((1, V), c), sel=[17], k_max=10)
        assert abs(o["lse"][0] - (c + math.log(V))) <= 1e-12 * max(1, abs(c) + 6)
        assert np.allclose(o["topk_logprobs"], -math.log(V), rtol=0, atol=1e-12)
        assert o["topk_ids"][0].tolist() == list(range(10))
        assert abs(o["sel_logprob"][0] + math.log(V)) <= 1e-12
    x = np.full((1, V), -np.inf)
    x[0, 123] = 1.25
    o = oracle.logprobs(x, sel=[123], k_max=4)
    assert o["lse"][0] == 1.25 and o["sel_logprob"][0] == 0.0
    assert o["topk_ids"][0].tolist() == [123, 0, 1, 2]
    assert o["topk_logprobs"][0, 0] == 0.0 and np.all(np.isneginf(o["topk_logprobs"][0, 1:]))
    c = workloads.logits_chunk("peaked", rows=8, V=4100)
    o = oracle.logprobs(_bits(c["logits"]), dtype=oracle.BF16, k_max=1)
    assert o["topk_ids"][:, 0].tolist() == c["peak_ids"].tolist()
    o = oracle.logprobs(_bits(workloads.all_neginf_row(V)), dtype=oracle.BF16, sel=[5], k_max=3)
    assert np.isneginf(o["lse"][0]) and np.isnan(o["sel_logprob"][0])
    assert o["topk_ids"][0].tolist() == [0, 1, 2] and np.all(np.isnan(o["topk_logprobs"]))
    o = oracle.logprobs(np.zeros((2, 8)), sel=[-1, 3], k_max=0)
    assert o["topk_ids"].shape == (2, 0)
    assert np.isnan(o["sel_logprob"][0]) and abs(o["sel_logprob"][1] + math.log(8)) < 1e-12


def pin_hand_example():
    """x = [2, 0, 2, -inf, 1] (bf16-exact), K = 4, worked by hand.

    Ties at 2 list ids 0 then 2 (ascending id, MTPLX PR #532 'Change');
    lse = 2 + log(2 + e^-2 + e^-1); the -inf entry ranks last.
    """
    x = np.array([[2.0, 0.0, 2.0, -np.inf, 1.0]])
    o = oracle.logprobs(x, sel=[3], k_max=5, row_k=[4])
    lse = 2.0 + math.log(2.0 + math.exp(-2.0) + math.exp(-1.0))
    assert abs(o["lse"][0] - lse) < 1e-14
    assert o["topk_ids"][0].tolist() == [0, 2, 4, 1, -1]
    want = [2.0 - lse, 2.0 - lse, 1.0 - lse, -lse]
    assert np.allclose(o["topk_logprobs"][0, :4], want, rtol=0, atol=1e-14)
    assert np.isneginf(o["topk_logprobs"][0, 4]) and np.isneginf(o["sel_logprob"][0])


def pin_fewer_finite_than_k():
    """k > #finite: the finite entries first, then -inf entries by ascending id."""
    x = np.full((1, 70), -np.inf)
    x[0, [65, 3, 40]] = [0.5, 0.5, 1.0]
    o = oracle.logprobs(x, k_max=6)
    assert o["topk_ids"][0].tolist() == [40, 3, 65, 0, 1, 2]
    assert np.all(np.isneginf(o["topk_logprobs"][0, 3:]))


def pin_dtype_conversions():
    """bf16 / f16 / f32 inputs are widened exactly (numpy float16 as the f16 reference)."""
    rng = np.random.default_rng(5)
    h = (rng.standard_normal((2, 300)) * 1000).astype(np.float16)
    h[0, :5] = [np.float16(6e-8), np.float16(-0.0), np.float16(65504), np.float16(-np.inf), 1]
    o16 = oracle.logprobs(h.view(np.uint16), dtype=oracle.F16, k_max=300)
    o64 = oracle.logprobs(h.astype(np.float64), k_max=300)
    assert np.array_equal(o16["topk_ids"], o64["topk_ids"])
    assert np.array_equal(o16["lse"], o64["lse"])
    f = rng.standard_normal((2, 300)).astype(np.float32)
    b = torch.from_numpy(f).to(torch.bfloat16)
    ob = oracle.logprobs(_bits(b), dtype=oracle.BF16, k_max=7)
    of = oracle.logprobs(b.float().numpy(), dtype=oracle.F32, k_max=7)
    assert np.array_equal(ob["topk_ids"], of["topk_ids"]) and np.array_equal(ob["lse"], of["lse"])


def pin_selected_id_range():
    """-1 means no selected token (NaN); any other id outside [0, V) is rejected."""
    o = oracle.logprobs(np.zeros((1, 4)), sel=[-1], k_max=0)
    assert np.isnan(o["sel_logprob"][0])
    for bad in (4, -2):
        with pytest.raises(oracle.OracleError):
            oracle.logprobs(np.zeros((1, 4)), sel=[bad], k_max=0)


def pin_page_sizes():
    """The pages' printed byte counts match the workloads' vocabularies and dtypes."""
    unit = {"MiB": 2 ** 20, "MB": 1e6, "KiB": 1024}
    for f in _golden("page_sizes.json")["facts"]:
        if "block" in f:
            assert f["vocab"] == f["block"] * f["blocks"]
            assert workloads.CHUNK_V == f["vocab"] and workloads.CHUNK_V % 64 == 0
            continue
        got = f["rows"] * f["vocab"] * f["elem_bytes"] / unit[f["unit"]]
        assert abs(got - f["value"]) <= f["rel_tol"] * f["value"], f["cite"]
    assert workloads.decode_batch.__defaults__ is not None


def pin_philox_kat():
    """Philox4x32-10 reproduces the generator's published known-answer vectors."""
    for vec in _golden("philox4x32_10_kat.json")["vectors"]:
        ctr = [int(w, 16) for w in vec["counter"]]
        key = [int(w, 16) for w in vec["key"]]
        want = [int(w, 16) for w in vec["output"]]
        assert oracle.philox4x32_10(ctr, key).tolist() == want, vec


def pin_sample_uniforms():
    """The sampling uniforms lie strictly inside (0, 1) on the 2^-24 grid (odd multiples,
    so exact in fp32), and differ across tokens, offsets and seeds."""
    us = [oracle.sample_uniform(7, 3, v) for v in range(400)]
    for u in us:
        assert 0.0 < u < 1.0
        m = u * 2 ** 24
        assert m == int(m) and int(m) % 2 == 1
    assert len(set(us)) == len(us)
    assert oracle.sample_uniform(7, 4, 0) != oracle.sample_uniform(7, 3, 0)
    assert oracle.sample_uniform(8, 3, 0) != oracle.sample_uniform(7, 3, 0)


def pin_gumbel_max_distribution():
    """argmax(z/T + Gumbel) draws token v with probability softmax(z/T)_v: the frequencies
    over 20000 row offsets pass a chi-square test (4 degrees of freedom) at T = 0.5, 1, 2."""
    z = np.array([0.2, -1.0, 1.5, 0.0, 0.7])
    n = 20000
    for T in (0.5, 1.0, 2.0):
        ids, _, _ = oracle.sample(np.tile(z, (n, 1)), temperature=np.full(n, T, np.float32), seed=12345,
                                  offsets=np.arange(n, dtype=np.int64))
        p = np.exp(z / T - np.max(z / T))
        p /= p.sum()
        counts = np.bincount(ids, minlength=len(z))
        chi2 = float(np.sum((counts - n * p) ** 2 / (n * p)))
        assert chi2 < 30.0, (T, chi2, counts, n * p)


def pin_sample_greedy_and_mask():
    """T <= 0 is argmax z with ties to the smaller id; disallowed tokens are never drawn;
    a row with no allowed token gives -1; a fixed (seed, offset) gives a fixed draw."""
    z = np.array([[0.5, 2.0, 2.0, -1.0], [3.0, 1.0, 0.0, -1.0], [0.0, 0.0, 0.0, 0.0]])
    ids, _, _ = oracle.sample(z, temperature=np.array([0.0, -1.0, 0.0], np.float32))
    assert ids.tolist() == [1, 0, 0]
    n, V = 3000, 40
    rng = np.random.default_rng(5)
    zz = rng.normal(size=(n, V))
    allowed = [3, 17, 33, 39]
    mask = np.zeros((n, 2), np.uint32)
    for v in allowed:
        mask[:, v // 32] |= np.uint32(1 << (v % 32))
    ids, _, _ = oracle.sample(zz, mask=mask, seed=9)
    assert set(ids.tolist()) <= set(allowed) and len(set(ids.tolist())) == len(allowed)
    ids_g, _, _ = oracle.sample(zz, temperature=np.zeros(n, np.float32), mask=mask)
    assert np.array_equal(ids_g, np.array(allowed)[np.argmax(zz[:, allowed], axis=1)])
    none, _, _ = oracle.sample(zz[:2], mask=np.zeros((2, 2), np.uint32))
    assert none.tolist() == [-1, -1]
    a, _, _ = oracle.sample(zz[:50], seed=1)
    b, _, _ = oracle.sample(zz[:50], seed=1)
    c, _, _ = oracle.sample(zz[:50], seed=2)
    assert np.array_equal(a, b) and not np.array_equal(a, c)


PINS = [pin_select_examples, pin_select_properties, pin_select_rejects,
        pin_project_exact_integers, pin_project_against_exact_sum,
        pin_selected_equals_full_sliced, pin_brute_force_tiny, pin_torch_f64_crosscheck,
        pin_invariants, pin_closed_forms, pin_hand_example, pin_fewer_finite_than_k,
        pin_dtype_conversions, pin_selected_id_range, pin_page_sizes,
        pin_philox_kat, pin_sample_uniforms, pin_gumbel_max_distribution, pin_sample_greedy_and_mask]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


MUTATIONS = {
    oracle.MUT_SELECT_SHIFT: "prefill row shifted by one",
    oracle.MUT_PROJECT_DROP_TERM: "projection drops its last term",
    oracle.MUT_PROJECT_TRANSPOSE: "projection reads W transposed",
    oracle.MUT_LSE_DROP_TERM: "exp-sum drops its last term",
    oracle.MUT_LOGPROB_SIGN: "logprob sign flipped",
    oracle.MUT_TIE_ID_DESC: "exact ties by descending id",
    oracle.MUT_TOPK_SKIP_FIRST: "top-K off by one rank",
    oracle.MUT_DECODE_LAST_ONLY: "multi-row decode keeps only its last row",
    oracle.MUT_PHILOX_9_ROUNDS: "Philox with 9 rounds",
    oracle.MUT_GUMBEL_SIGN: "Gumbel noise with the wrong sign",
    oracle.MUT_MASK_IGNORED: "grammar bitmask ignored",
    oracle.MUT_TEMP_TIMES: "logits multiplied by the temperature",
}


@pytest.mark.parametrize("mut", sorted(MUTATIONS), ids=lambda m: MUTATIONS[m])
def test_pins_catch(mut):
    """Each planted mistake makes at least one pin fail."""
    failed = []
    with oracle.mutation(mut):
        for pin in PINS:
            try:
                pin()
            except (AssertionError, oracle.OracleError, IndexError, ValueError):
                failed.append(pin.__name__)
    assert failed, "no pin caught: " + MUTATIONS[mut]
