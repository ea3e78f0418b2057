"""The inversion and the backward captured in one CUDA graph (torch.cuda.graph) and replayed.

A caller that runs many small layers launches the whole backward as one graph instead of a
handful of kernel launches from the host.  Capture needs every launch on the caller's stream and
no host synchronisation inside; replay must re-read the inputs, so the graph
is checked on the inputs it was captured with and again after new inputs (another selection,
other activations) have been copied into the same buffers.  dK and dV involve no atomics and
must equal the eager result bit for bit; dQ's fp32 partial sums are added in a varying order
(within 5e-3 of max|dQ|, the pages' run-to-run figure).
"""
import math

import pytest
import torch

from block_sparse_video_tok_gb300 import workloads as wl
from tests.parity import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vsa():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from block_sparse_video_tok_gb300 import build
    build.build()
    from block_sparse_video_tok_gb300 import vsa as binding
    return binding


def _forward(vsa, case, dev):
    return vsa.vsa_fwd(dev["q"], dev["k"], dev["v"], dev["q2k_idx"], dev["q2k_num"], dev["vbs"],
                       case["sm_scale"])


def _eager(vsa, case, dev, o, lse):
    k2q_idx, k2q_num = vsa.vsa_invert_indices(dev["q2k_idx"], dev["q2k_num"], case["nb"])
    return vsa.vsa_bwd(dev["do"], dev["q"], dev["k"], dev["v"], o, lse, k2q_idx, k2q_num,
                       dev["vbs"], case["sm_scale"])


def _same(got, ref, label):
    dq, dk, dv = got
    rq, rk, rv = ref
    assert torch.equal(dk, rk), label + ": dk differs from the eager backward"
    assert torch.equal(dv, rv), label + ": dv differs from the eager backward"
    d = (dq.float() - rq.float()).abs().max().item()
    assert math.isfinite(d) and d <= 5e-3 * rq.float().abs().max().item(), (label, d)


@pytest.mark.parametrize("name", ["4k_25pct", "65k_12pct_zipf"])
def test_graph_replay_matches_eager(vsa, name):
    """4k: fewer items than 8 per SM (sorted work order, split items); 65k: 1024 kv tiles
    (sorted order), ragged blocks."""
    cases = [wl.make_config(name), wl.make_config(name, seed=1)]
    B, H, S, nb = (cases[0][n] for n in ("B", "H", "S", "nb"))
    devs = [to_device(c) for c in cases]
    fwds = [_forward(vsa, c, d) for c, d in zip(cases, devs)]
    refs = [[t.clone() for t in _eager(vsa, c, d, *f)] for c, d, f in zip(cases, devs, fwds)]
    torch.cuda.synchronize()

    # The graph's buffers, holding the first case.
    x = {n: t.clone() for n, t in devs[0].items()}
    o, lse = (t.clone() for t in fwds[0])
    k2q_idx = torch.empty((B, H, nb, nb), dtype=torch.int32, device="cuda")
    k2q_num = torch.empty((B, H, nb), dtype=torch.int32, device="cuda")
    ws = torch.empty(vsa.vsa_bwd_workspace_bytes(B, H, S), dtype=torch.uint8, device="cuda")
    out = [torch.empty_like(x["q"]) for _ in range(3)]
    sc = cases[0]["sm_scale"]

    def step():
        vsa.vsa_invert_indices(x["q2k_idx"], x["q2k_num"], nb, k2q_idx, k2q_num)
        vsa.vsa_bwd(x["do"], x["q"], x["k"], x["v"], o, lse, k2q_idx, k2q_num, x["vbs"], sc,
                    dq=out[0], dk=out[1], dv=out[2], workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # one eager run on a side stream before capture
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()

    for c, (dev, (o_c, lse_c), ref) in enumerate(zip(devs, fwds, refs)):
        for n, t in dev.items():
            x[n].copy_(t)
        o.copy_(o_c)
        lse.copy_(lse_c)
        for t in out:
            t.fill_(float("nan"))
        for rep in range(2):
            graph.replay()
            torch.cuda.synchronize()
            assert vsa.vsa_read_device_error(ws) == 0
            _same(out, ref, "%s case %d replay %d" % (name, c, rep))
