"""The C ABI inside CUDA graphs: a forward and its backward captured once on a side
stream and replayed give bit-identical results to the eager calls (launch-bound loops
are meant to run as graphs; every entry point is asynchronous on the given stream and
allocates nothing after the plan)."""
import numpy as np
import pytest
import torch

import gapped_varlen_attention_gb300 as gva
from gapped_varlen_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gva.build()


@pytest.mark.parametrize("causal_block", [0, 64])
def test_forward_and_backward_replay_in_a_graph(causal_block):
    rng = np.random.default_rng(701 + causal_block)
    g = W.random_geometry(rng, 5, 700, 900, 16, 4, 128, allow_empty=False)
    q, k, v = W.make_qkv(g, 701, device="cuda")
    do = torch.randn(q.shape, device="cuda").bfloat16()
    plan = gva.Plan.from_geometry(g, causal_block=causal_block)
    ws = torch.empty(max(16, gva.backward_workspace_bytes(plan)), dtype=torch.uint8, device="cuda")

    def run(o, l, dq, dk, dv):
        gva.forward(plan, q, k, v, o, l)
        gva.backward(plan, q, k, v, o, l, do, dq, dk, dv, workspace=ws)

    def buffers():
        o, l = W.make_outputs(g, 0.0, device="cuda")
        return [o, l, torch.zeros_like(q), torch.zeros_like(k), torch.zeros_like(v)]

    eager = buffers()
    run(*eager)
    torch.cuda.synchronize()
    gva.device_status(plan)

    graphed = buffers()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm the lazy module / attribute setup outside capture
        run(*graphed)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for t in graphed:
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(*graphed)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    gva.device_status(plan)
    for a, b in zip(eager, graphed):
        assert torch.equal(a, b)
