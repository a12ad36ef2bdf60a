"""The bounded-wait timeout path of the kernels, made to run out on purpose.

Every wait of a kernel on another role of its own CTA (a shared-memory stage
filled by TMA, a tensor-memory accumulator, a chunk of logits) gives up after
the library's wait limit, sets LMH_DS_TIMEOUT in the device status, lets the
copies and tensor-core work it has in flight finish, frees its tensor memory
and returns (openinfer issue #719, "Acceptance criteria": defined error
behaviour instead of a hang).  The limit is 2 s, so no legitimate wait reaches
it; here the test hook lmh_debug_set_wait_limit shortens it to 1 ns, shorter
than the latency of any load, so the first wait that does not succeed at once
runs out.  Nothing faults or hangs: the drain waits keep the 2 s limit.  The
test then restores the default and checks that the next call on the same
context is correct.
"""
import pytest
import torch

import oracle
import workloads
from parity import TOL_FROM_LOGITS, TOL_FUSED, check_from_logits, check_fused

pytestmark = pytest.mark.gpu


def _head_case():
    g = torch.Generator().manual_seed(5)
    rows, H, V, T = 40, 512, 20000, 48
    hidden = torch.randn(T, H, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, H, generator=g) / H ** 0.5).to(torch.bfloat16)
    ri = torch.randperm(T, generator=g)[:rows].to(torch.int32)
    sel = torch.randint(0, V, (rows,), generator=g, dtype=torch.int32)
    return hidden, W, ri, sel


def test_head_wait_runs_out_then_recovers(lmh):
    from top_reduction_gb300 import lmh as L
    hidden, W, ri, sel = _head_case()
    hd, Wd, rid = hidden.cuda(), W.cuda(), ri.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        L.debug_set_wait_limit(1)
        lmh.project_logprobs(hd, Wd, row_idx=rid, sel=sel, k_max=5, dev_status=st)
        torch.cuda.synchronize()  # the call returned and the grid finished: no hang, no fault
    finally:
        L.debug_set_wait_limit(0)
    assert int(st.item()) & L.DS_TIMEOUT, "status %#x: no wait ran out" % int(st.item())

    st.zero_()
    o = lmh.project_logprobs(hd, Wd, row_idx=rid, sel=sel, k_max=5, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    z = oracle.project(workloads.bits(hidden), workloads.bits(W), row_idx=ri.numpy())
    orc = oracle.logprobs(z, sel=sel.numpy(), k_max=5)
    A = hidden[ri.long()].float().double().numpy()
    assert check_fused(o, orc, z, A, W, 5, atol=TOL_FUSED, what="after timeout") == 0


def test_logits_wait_runs_out_then_recovers(lmh):
    from top_reduction_gb300 import lmh as L
    c = workloads.logits_chunk("normal", seed=21, rows=64, V=50000)
    x, sel = c["logits"].cuda(), c["sel"].cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        L.debug_set_wait_limit(1)
        lmh.logprobs_from_logits(x, sel=sel, k_max=20, dev_status=st)
        torch.cuda.synchronize()
    finally:
        L.debug_set_wait_limit(0)
    assert int(st.item()) & L.DS_TIMEOUT, "status %#x: no wait ran out" % int(st.item())

    st.zero_()
    r = lmh.logprobs_from_logits(x, sel=sel, k_max=20, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.logprobs(workloads.bits(c["logits"]), dtype=oracle.BF16, sel=c["sel"].numpy(), k_max=20)
    check_from_logits(r, ref, 20, atol=TOL_FROM_LOGITS, what="after timeout")
