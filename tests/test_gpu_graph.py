"""muon_step inside a CUDA graph: once a call with the same shapes and weight
pointers has run outside capture (it builds the plan and the weight tensor
maps, which allocates and synchronises), a step is a fixed sequence of kernel
launches on the caller's stream, so it can be captured once and replayed with
new gradients copied into the captured gradient buffers.  The replays must
give exactly the weights and momentum of the same steps run eagerly (the step
is deterministic)."""
import pytest
import torch

import pretraining_optimizer_step_b300 as mu
import workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["d2", "d12"])
def test_captured_step_replays_bit_exactly(name):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mu.muon_init(wait_timeout_s=2.0)
    try:
        p, g, m, shapes = workloads.make_stack(name, "cuda")
        steps = 3
        grads = [[workloads.make_grad(name, i, s, "cuda", 0, k) for i, s in enumerate(shapes)]
                 for k in range(steps)]
        p_e, g_e, m_e = [t.clone() for t in p], [t.clone() for t in g], [t.clone() for t in m]
        p_g, g_g, m_g = [t.clone() for t in p], [t.clone() for t in g], [t.clone() for t in m]

        # eager reference
        for k in range(steps):
            for dst, src in zip(g_e, grads[k]):
                dst.copy_(src)
            mu.muon_step(p_e, g_e, m_e)
        torch.cuda.synchronize()

        # warm-up outside capture on the graph's own buffers, then restore their state
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            mu.muon_step(p_g, g_g, m_g, stream=side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        for dst, src in zip(p_g + m_g, p + m):
            dst.copy_(src)
        torch.cuda.synchronize()

        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            mu.muon_step(p_g, g_g, m_g, stream=torch.cuda.current_stream())
        for k in range(steps):
            for dst, src in zip(g_g, grads[k]):
                dst.copy_(src)
            graph.replay()
        torch.cuda.synchronize()
        assert mu.muon_get_status(check=False) == mu.MUON_OK
        for i in range(len(shapes)):
            assert torch.equal(p_g[i], p_e[i]), i
            assert torch.equal(m_g[i], m_e[i]), i
        del graph
    finally:
        mu.muon_destroy()
