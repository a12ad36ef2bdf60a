"""Vocabulary-parallel head on one GPU: the shares run one after another.

A vocabulary-parallel head splits W by vocabulary over several GPUs; every
rank computes a record per row over its share (lmh_project_partials), the
ranks all-gather the records, and lmh_merge_records finishes the rows
(openinfer issue #719, "Suggested direction": an exact multi-stage
reduction; MTPLX PR #532, "Change": the row's top-k lies in the union of the
parts' top-k lists).  Here every share runs on this one GPU, in turn, into
its slice of one buffer laid out as the all-gather lays it out; nothing waits
on another share.  The merged result must equal the f64 oracle's (ids
bit-exact, values within the fused-head tolerance) and the unsharded call's
(ids identical: each logit is the same fp32 accumulation).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import TOL_FUSED, assert_close, check_fused

pytestmark = pytest.mark.gpu


def _case(rows, T, H, V, seed):
    g = torch.Generator().manual_seed(seed)
    hidden = torch.randn(T, H, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, H, generator=g) / H ** 0.5).to(torch.bfloat16)
    ri = torch.randperm(T, generator=g)[:rows].to(torch.int32)
    sel = torch.randint(-1, V, (rows,), generator=g, dtype=torch.int32)
    return hidden, W, ri, sel


def sharded(lmh, hidden_d, W_d, ri_d, sel, row_k, k, V, world):
    rows = ri_d.numel()
    rb = lmh.record_bytes(k)
    allrec = torch.empty((world, rows, rb), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for r in range(world):
        b, n = lmh.vocab_share(V, r, world)
        lmh.project_partials(hidden_d, W_d[b:b + n], b, V, row_idx=ri_d, sel=sel, row_k=row_k, k_max=k,
                             records=allrec[r], dev_status=st)
    o = lmh.merge_records(allrec, world, rows, V, sel=sel, row_k=row_k, k_max=k, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return o


@pytest.mark.parametrize("world,rows,H,V,k", [(2, 40, 512, 20000, 5), (3, 130, 256, 30001, 20),
                                              (4, 8, 1024, 151936, 20), (2, 17, 136, 4100, 128),
                                              (5, 300, 64, 9000, 1), (2, 33, 512, 12800, 0)])
def test_shares_match_oracle_and_unsharded(lmh, world, rows, H, V, k):
    hidden, W, ri, sel = _case(rows, rows + 7, H, V, seed=world * 100 + rows)
    row_k = None
    if k > 1:
        row_k = torch.randint(0, k + 1, (rows,), generator=torch.Generator().manual_seed(rows), dtype=torch.int32)
    hd, Wd, rid = hidden.cuda(), W.cuda(), ri.cuda()
    rk_d = None if row_k is None else row_k.cuda()
    o = sharded(lmh, hd, Wd, rid, sel, rk_d, k, V, world)
    ref = lmh.project_logprobs(hd, Wd, row_idx=rid, sel=sel, row_k=rk_d, k_max=k)
    torch.cuda.synchronize()
    if k > 0:
        assert torch.equal(o["topk_ids"], ref["topk_ids"])
    for key in ("lse", "sel_logprob", "topk_logprobs"):
        assert_close(o[key].cpu().numpy(), ref[key].cpu().numpy(), 1e-5, "sharded vs unsharded " + key)
    z = oracle.project(workloads.bits(hidden), workloads.bits(W), row_idx=ri.numpy())
    rk = None if row_k is None else row_k.numpy()
    orc = oracle.logprobs(z, sel=sel.numpy(), row_k=rk, k_max=k)
    A = hidden[ri.long()].float().double().numpy()
    assert check_fused(o, orc, z, A, W, k, row_k=rk, atol=TOL_FUSED, what="vocab-parallel %d" % world) == 0


def test_record_layout(lmh):
    """One share's record: m is the share's max logit, s its sum of exp(z - m), the
    selected logit only in the share that holds the token, keys best first with global ids."""
    hidden, W, ri, sel = _case(4, 10, 128, 1000, seed=3)
    sel = torch.tensor([5, 600, -1, 999], dtype=torch.int32)
    k, V = 3, 1000
    b, n = 512, 488
    rec = lmh.project_partials(hidden.cuda(), W.cuda()[b:b + n].contiguous(), b, V, row_idx=ri.cuda(), sel=sel,
                               k_max=k)
    torch.cuda.synchronize()
    raw = rec.cpu().numpy()
    head = raw[:, :16].copy().view(np.float32).reshape(4, 4)
    flags = raw[:, 12:16].copy().view(np.uint32).reshape(4)
    keys = raw[:, 16:16 + 8 * k].copy().view(np.uint64).reshape(4, k)
    z = oracle.project(workloads.bits(hidden), workloads.bits(W), row_idx=ri.numpy())[:, b:b + n]
    for i in range(4):
        assert abs(head[i, 0] - z[i].max()) <= TOL_FUSED
        assert abs(head[i, 1] - np.exp(z[i] - head[i, 0]).sum()) <= 1e-3 * head[i, 1]
        in_share = b <= int(sel[i]) < b + n
        assert flags[i] == (1 if in_share else 0)
        if in_share:
            assert abs(head[i, 2] - z[i, int(sel[i]) - b]) <= TOL_FUSED
        ids = (~keys[i].astype(np.uint64) & np.uint64(0xFFFFFFFF)).astype(np.int64)
        assert np.array_equal(ids, np.argsort(-z[i], kind="stable")[:k] + b)


def test_nccl_exchange_one_rank(lmh):
    """The exchange through NCCL on this GPU: a one-rank group, so the all-gather is the
    identity, but the records go through the real path (project_partials -> NCCL
    all_gather_into_tensor into device memory -> merge_records) and must equal the
    unsharded call."""
    import os
    import socket
    import torch.distributed as dist
    if dist.is_initialized():
        pytest.skip("a process group is already initialised")
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    dist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % port, rank=0, world_size=1,
                            device_id=torch.device("cuda", torch.cuda.current_device()))
    try:
        hidden, W, ri, sel = _case(24, 40, 256, 6000, seed=9)
        hd, Wd, rid = hidden.cuda(), W.cuda(), ri.cuda()
        b, n = lmh.vocab_share(6000, 0, 1)
        o = lmh.vocab_parallel_logprobs(hd, Wd[b:b + n], b, 6000, row_idx=rid, sel=sel, k_max=8)
        ref = lmh.project_logprobs(hd, Wd, row_idx=rid, sel=sel, k_max=8)
        torch.cuda.synchronize()
        assert torch.equal(o["topk_ids"], ref["topk_ids"])
        for key in ("lse", "sel_logprob", "topk_logprobs"):
            assert_close(o[key].cpu().numpy(), ref[key].cpu().numpy(), 1e-5, "nccl exchange " + key)
    finally:
        dist.destroy_process_group()
