"""The hot path inside a CUDA graph: pstat_forward_backward and the fused
lm_head forward, captured once (after an eager call, which does the
per-context set-up) and replayed, give the same bits as eager calls -- also
after the inputs are overwritten in place between replays, as a training
loop that reuses its buffers would do."""
import pytest
import torch

pytestmark = pytest.mark.gpu
IGN = -100


def _bits(x):
    x = x.contiguous()
    return x.view(torch.int16 if x.element_size() == 2 else torch.int32)


@pytest.mark.parametrize("T,V", [(1, 151936), (64, 151936), (300, 10007)])
def test_single_pass_in_a_graph(cuda_lib, T, V):
    g = torch.Generator(device="cuda").manual_seed(T + V)
    z = (2.0 * torch.randn(T, V, generator=g, device="cuda")).to(torch.bfloat16)
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    w = torch.randn(T, generator=g, device="cuda")
    lp = torch.empty(T, device="cuda")
    ent = torch.empty(T, device="cuda")
    rs = torch.empty(T, 2, device="cuda")
    dl = torch.empty(T, V, dtype=torch.bfloat16, device="cuda")
    cuda_lib.forward_backward(z, y, w, IGN, out=(lp, ent, rs), dlogits=dl)  # set-up, eager
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cuda_lib.forward_backward(z, y, w, IGN, out=(lp, ent, rs), dlogits=dl)
    for step in range(2):
        if step:  # new inputs in the same buffers
            z.copy_((3.0 * torch.randn(T, V, generator=g, device="cuda")).to(torch.bfloat16))
            y.copy_(torch.randint(0, V, (T,), generator=g, device="cuda"))
        graph.replay()
        ref = cuda_lib.forward_backward(z, y, w, IGN)
        torch.cuda.synchronize()
        for a, b, name in zip((lp, ent, rs, dl), ref, ("logprob", "entropy", "rowstats",
                                                       "dlogits")):
            assert torch.equal(_bits(a), _bits(b)), (step, name)


def test_lmhead_forward_in_a_graph(cuda_lib):
    T, V, d = 200, 9000, 256
    g = torch.Generator(device="cuda").manual_seed(3)
    h = torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16)
    W = (0.05 * torch.randn(V, d, generator=g, device="cuda")).to(torch.bfloat16)
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    ws = torch.empty(cuda_lib.lmhead_workspace_size(T, V, d), dtype=torch.uint8, device="cuda")
    cuda_lib.lmhead_forward(h, W, y, IGN, workspace=ws)  # set-up, eager
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = cuda_lib.lmhead_forward(h, W, y, IGN, workspace=ws)
    h.copy_(torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16))
    graph.replay()
    ref = cuda_lib.lmhead_forward(h, W, y, IGN, workspace=ws)
    torch.cuda.synchronize()
    for a, b in zip(out, ref):
        assert torch.equal(_bits(a), _bits(b))
