"""Seeded synthetic inputs for the five workloads the library is tested and timed on.

Shared by the tests, the smoke check and the benchmark.  This module only
draws random numbers and lays out batches: it holds none of the method's
arithmetic (no projection, no softmax, no selection, no top-K).  Every tensor
is a torch CPU tensor; bf16 values come from an fp32 draw rounded to nearest
even (``Tensor.to(torch.bfloat16)``).

Workloads (shapes taken from the pages' own workloads):

* ``tiny_batch``      -- 2 decode rows + prefill segments of 5, 17, 40 rows
  (64 rows), H 128, V 4096, K 5.
* ``decode_batch``    -- 32 decode rows, H 2560, V 151936 (the head shape of
  the sm_89 measurement in openinfer issue #719), K 5 or 1.
* ``prefill_batch``   -- 8 packed 2048-token prompts, H 1024, V 151936 (the
  2048-row head of the vllm-metal release benchmark), K 20.
* ``logits_chunk``    -- one 256 x 248320 bf16 logits chunk (MTPLX PR #532:
  248,320 = 3,880 x 64), distributions normal / peaked / gumbel / ties /
  neginf.
* ``mixed_batch``     -- Llama-3-8B head shape (H 4096, V 128256): 64 decode
  rows, 4 prefill segments of 512, and one 1024-token segment whose every
  position is scored.

Seeds: workload index (tiny 0, decode 1, prefill 2, chunk 3, mixed 4) unless
given.
"""
import torch

TINY_CU = [0, 1, 2, 7, 24, 64]
CHUNK_ROWS, CHUNK_V = 256, 248320
DISTRIBUTIONS = ("normal", "peaked", "gumbel", "ties", "neginf")


def _gen(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _bf16_normal(shape, std, g):
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def _uniform_ids(n, V, g):
    return torch.randint(0, V, (n,), generator=g, dtype=torch.int32)


def tiny_batch(seed=0):
    """2 decode rows + prefill segments of lengths 5, 17, 40; H 128; V 4096; K 5.

    hidden ~ N(0,1) fp32 -> bf16; W ~ N(0, 1/128) (variance) stored as the
    [V x H] lm_head.weight; one selected token per sampled row, uniform.
    """
    g = _gen(seed)
    H, V = 128, 4096
    cu = torch.tensor(TINY_CU, dtype=torch.int32)
    hidden = _bf16_normal((64, H), 1.0, g)
    W = _bf16_normal((V, H), (1.0 / 128) ** 0.5, g)
    n_sel = 5
    sel = _uniform_ids(n_sel, V, g)
    return dict(name="tiny_batch", cu_seqlens=cu, num_decode=2, all_rows_mask=None,
                hidden=hidden, W=W, H=H, V=V, k=5, n_sel=n_sel, sel=sel, row_k=None)


def decode_batch(seed=1, k=5):
    """32 pure-decode rows, H 2560, V 151936, hidden ~ N(0,1), W ~ N(0, 0.02^2)."""
    g = _gen(seed)
    R, H, V = 32, 2560, 151936
    cu = torch.arange(R + 1, dtype=torch.int32)
    hidden = _bf16_normal((R, H), 1.0, g)
    W = _bf16_normal((V, H), 0.02, g)
    sel = _uniform_ids(R, V, g)
    return dict(name="decode_batch", cu_seqlens=cu, num_decode=R, all_rows_mask=None,
                hidden=hidden, W=W, H=H, V=V, k=k, n_sel=R, sel=sel, row_k=None)


def prefill_batch(seed=2):
    """8 packed prompts of 2048 tokens (16384 rows), H 1024, V 151936, K 20.

    The selective step samples the 8 last rows; ``sel_all`` gives one
    selected token per packed row for the full-projection arm.
    """
    g = _gen(seed)
    P, L, H, V = 8, 2048, 1024, 151936
    cu = torch.arange(0, P * L + 1, L, dtype=torch.int32)
    hidden = _bf16_normal((P * L, H), 1.0, g)
    W = _bf16_normal((V, H), 0.02, g)
    sel = _uniform_ids(P, V, g)
    sel_all = _uniform_ids(P * L, V, g)
    return dict(name="prefill_batch", cu_seqlens=cu, num_decode=0, all_rows_mask=None,
                hidden=hidden, W=W, H=H, V=V, k=20, n_sel=P, sel=sel, row_k=None,
                sel_all=sel_all)


def logits_chunk(dist="normal", seed=3, rows=CHUNK_ROWS, V=CHUNK_V, k_for_ties=20):
    """A [rows x V] bf16 logits chunk with one of DISTRIBUTIONS.

    normal  -- N(0,1).
    peaked  -- N(0,1) with +15 added at one uniform id per row.
    gumbel  -- -log(-log U), U ~ Uniform(0,1).
    ties    -- N(0,1) plus, per row, a group of 2..2*k_for_ties ids set to 6.0
               and a second group of 1..k_for_ties ids set to 5.5; half of each
               group lies inside one 64-block, half is spread over the row, so
               ties fall inside blocks, across blocks and on the K-th rank.
    neginf  -- N(0,1) with 10% of the entries of every row set to -inf, and
               in rows 0..7 whole 64-blocks (every 7th block) set to -inf.
    The row that is entirely -inf is a separate edge case (``all_neginf_row``).
    """
    assert dist in DISTRIBUTIONS
    g = _gen(seed + 100 * DISTRIBUTIONS.index(dist))
    if dist == "gumbel":
        u = torch.rand((rows, V), generator=g, dtype=torch.float32)
        u = u.clamp_(min=1e-30)
        x = -torch.log(-torch.log(u))
        x[torch.isinf(x)] = 0.0  # u == 1 exactly: keep finite
        x = x.to(torch.bfloat16)
    else:
        x = torch.randn((rows, V), generator=g, dtype=torch.float32).to(torch.bfloat16)
    extra = {}
    if dist == "peaked":
        ids = torch.randint(0, V, (rows,), generator=g)
        r = torch.arange(rows)
        x[r, ids] = (x[r, ids].float() + 15.0).to(torch.bfloat16)
        extra["peak_ids"] = ids
    elif dist == "ties":
        nblk = V // 64
        for r in range(rows):
            for val, gmax in ((6.0, 2 * k_for_ties), (5.5, k_for_ties)):
                gsize = int(torch.randint(1 if val == 5.5 else 2, gmax + 1, (1,), generator=g))
                inblk = gsize // 2
                b = int(torch.randint(0, max(nblk, 1), (1,), generator=g))
                offs = torch.randperm(64, generator=g)[:inblk] + 64 * b
                spread = torch.randint(0, V, (gsize - inblk,), generator=g)
                ids = torch.cat([offs, spread]).clamp_(max=V - 1)
                x[r, ids] = torch.tensor(val, dtype=torch.bfloat16)
            if r % 4 == 0:  # include the lowest ids in some groups
                x[r, 0] = torch.tensor(6.0, dtype=torch.bfloat16)
    elif dist == "neginf":
        mask = torch.rand((rows, V), generator=g) < 0.10
        x[mask] = float("-inf")
        nblk = (V + 63) // 64
        for r in range(min(8, rows)):
            for b in range(r % 7, nblk, 7):
                x[r, 64 * b: min(64 * b + 64, V)] = float("-inf")
    sel = _uniform_ids(rows, V, g)
    return dict(name="logits_chunk", dist=dist, logits=x, rows=rows, V=V, sel=sel, **extra)


def all_neginf_row(V=CHUNK_V):
    """One row of -inf logits (the degenerate edge case)."""
    return torch.full((1, V), float("-inf"), dtype=torch.bfloat16)


def mixed_batch(seed=4, with_weights=True):
    """Llama-3-8B head shape: H 4096, V 128256.

    64 decode rows, 4 prefill segments of 512 rows, and one 1024-row segment
    with all_rows_mask = 1 (prompt scoring of every position): 1092 selected
    rows.  Per-row K: decode rows 0..31 ask K=20, decode rows 32..63 K=0,
    the four prefill last rows K=0, the 1024 prompt positions K=20.
    Selected tokens: uniform for decode and prefill rows; for prompt position
    t it is the next prompt token (a uniform synthetic token sequence), and
    the segment's last position has none (-1).
    """
    g = _gen(seed)
    H, V = 4096, 128256
    n_dec, n_pre, L_pre, L_prompt = 64, 4, 512, 1024
    lens = [1] * n_dec + [L_pre] * n_pre + [L_prompt]
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int32), 0)
    T = int(cu[-1])
    mask = torch.zeros(len(lens), dtype=torch.uint8)
    mask[-1] = 1
    hidden = _bf16_normal((T, H), 1.0, g)
    W = _bf16_normal((V, H), 0.02, g) if with_weights else None
    n_sel = n_dec + n_pre + L_prompt
    row_k = torch.zeros(n_sel, dtype=torch.int32)
    row_k[:32] = 20
    row_k[n_dec + n_pre:] = 20
    sel = torch.empty(n_sel, dtype=torch.int32)
    sel[: n_dec + n_pre] = _uniform_ids(n_dec + n_pre, V, g)
    prompt_tokens = _uniform_ids(L_prompt, V, g)
    sel[n_dec + n_pre: -1] = prompt_tokens[1:]
    sel[-1] = -1
    return dict(name="mixed_batch", cu_seqlens=cu, num_decode=n_dec, all_rows_mask=mask,
                hidden=hidden, W=W, H=H, V=V, k=20, n_sel=n_sel, sel=sel, row_k=row_k)


def bits(t):
    """Raw 16-bit patterns of a bf16/f16 CPU tensor as a numpy uint16 array."""
    assert t.dtype in (torch.bfloat16, torch.float16)
    return t.contiguous().view(torch.int16).numpy().view("uint16")
