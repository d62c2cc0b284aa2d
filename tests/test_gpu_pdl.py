"""Programmatic dependent launch: every kernel of the library is launched
so that it may be scheduled while the grid before it in the stream is still
running, and waits for that grid before touching global memory.  These
chains make each launch read what the launch before it wrote (read after
write) or overwrite what it read (write after read); the results must be
those of plain stream order, bit for bit.
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

nts = pytest.importorskip("normalization_token_split_gb300")
DEV = "cuda:0"


def chain(X, g, beta):
    y1, _ = nts.qknorm_rms(X, g, N=4)                          # reads X
    y2, _ = nts.qknorm_rms(y1, g, N=2)                         # reads y1 at once
    m1 = nts.rmsnorm_mxcast(y2, None, B=32)                    # reads y2
    y3 = y2.clone()
    m2 = nts.mxnorm_cast(y3, None, B=16, fmt="nvfp4", p=2)     # reads y3 ...
    nts.qknorm_rms(y3, g, N=1, out=y3)                         # ... then y3 is overwritten
    y4, _, _ = nts.layernorm_split(y3, g, beta, N=4)           # reads the new y3
    y5, _ = nts.qknorm_rms_heads(y4, g[:128].contiguous(), head_dim=128)   # reads y4
    return [y1, y2, m1.codes, m1.scales, m2.codes, m2.scales, y3, y4, y5]


@pytest.mark.parametrize("T", [8, 300, 4096])
def test_chained_launches_match_plain_stream_order(T):
    X, g = workloads.qk_inputs(T, 4096, seed=990 + T, device=DEV)
    b = workloads.beta_vector(4096, seed=990, device=DEV)
    try:
        nts.set_pdl(False)
        want = chain(X, g, b)
        torch.cuda.synchronize()
        nts.set_pdl(True)
        for _ in range(4):
            got = chain(X, g, b)
            torch.cuda.synchronize()
            for w, o in zip(want, got):
                assert torch.equal(w, o)
        nts.check_status()
    finally:
        nts.set_pdl(True)


def test_chain_in_a_graph():
    X, g = workloads.qk_inputs(2048, 4096, seed=995, device=DEV)
    b = workloads.beta_vector(4096, seed=995, device=DEV)
    want = chain(X, g, b)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        got = chain(X, g, b)
    for _ in range(3):
        for t in got:
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for w, o in zip(want, got):
            assert torch.equal(w, o)
    nts.check_status()
