"""The forward and backward launch nothing but kernels on the given stream, so
they can be captured in a CUDA graph (after one eager call on the device, which
sets the kernels' shared-memory attributes) and replayed: the replays give the
eager results bit for bit, also after the inputs are overwritten in place."""
import pytest
import torch

import tiled_attention_forward_gb300 as fattn

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float16, 64), (torch.float32, 64)])
def test_forward_graph_replay(dtype, D):
    B, H, N = 2, 3, 500
    g = torch.Generator().manual_seed(1)
    q, k, v = (torch.randn(B, H, N, D, generator=g).to(dtype).cuda() for _ in range(3))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    fattn.fwd(q, k, v, causal=True, out=o, lse=lse)  # eager first call on the device
    torch.cuda.synchronize()
    o_eager, lse_eager = o.clone(), lse.clone()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            fattn.fwd(q, k, v, causal=True, out=o, lse=lse, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    o.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_eager) and torch.equal(lse, lse_eager)
    # new inputs in the same buffers: the replay computes on them
    q2 = torch.randn(B, H, N, D, generator=g).to(dtype).cuda()
    q.copy_(q2)
    graph.replay()
    o_new, lse_new = fattn.fwd(q2, k, v, causal=True)
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    assert torch.equal(o, o_new) and torch.equal(lse, lse_new)


def test_backward_graph_replay():
    B, H, N, D = 1, 4, 400, 128
    g = torch.Generator().manual_seed(2)
    q, k, v, do = (torch.randn(B, H, N, D, generator=g).to(torch.bfloat16).cuda() for _ in range(4))
    o, lse = fattn.fwd(q, k, v, causal=False)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(fattn.bwd_workspace_bytes(B, H, N), dtype=torch.uint8, device="cuda")
    fattn.bwd(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, workspace=ws)  # eager first call
    torch.cuda.synchronize()
    ref = (dq.clone(), dk.clone(), dv.clone())
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            fattn.bwd(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv, workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for t in (dq, dk, dv):
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert fattn.get_device_status() == 0
    for a, b in zip((dq, dk, dv), ref):
        assert torch.equal(a, b)
