"""The library's calls record into a CUDA graph: no allocation, synchronisation
or host read on the path, tensor maps baked into the captured launches.  A
replay must reproduce the eager results bitwise (deterministic backward)."""

import pytest
import torch

import workloads as W
from tests._helpers import cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,dtype,det", [(64, "bf16", True), (128, "bf16", True), (256, "bf16", True),
                                         (128, "bf16", 2), (128, "fp32", True), (64, "fp32", True)])
def test_fwd_bwd_graph_replay_matches_eager(d, dtype, det):
    """Also the ordered single pass (its counters are reset by a memset node)
    and the float32 tensor-core path."""
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 700, 900, 4, 2, d, dtype, True, None, "graph")
    q, k, v, do = cuda(*W.make_inputs(p))
    kl = torch.tensor([900, 333], dtype=torch.int32, device="cuda")

    def step():
        o, lse = ea.forward(q, k, v, causal=True, kv_lens=kl)
        return (o, lse) + tuple(ea.backward(q, k, v, o, lse, do, causal=True, kv_lens=kl, deterministic=det))

    eager = step()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = step()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert ea.attn_device_status()[1] == 0
    for a, b in zip(eager, captured):
        assert torch.equal(a, b)


def test_decode_graph_replay_matches_eager():
    import exact_attention_34_gb300 as ea

    p = W.Problem(2, 1, 5000, 8, 2, 128, "bf16", False, (5000, 1200), "graphdec")
    q, k, v, _ = cuda(*W.make_inputs(p))
    kl = torch.tensor(p.kv_lens, dtype=torch.int32, device="cuda")
    eager = ea.decode(q, k, v, kv_lens=kl, num_splits=4)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ea.decode(q, k, v, kv_lens=kl, num_splits=4)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = ea.decode(q, k, v, kv_lens=kl, num_splits=4)
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, captured):
        assert torch.equal(a, b)
