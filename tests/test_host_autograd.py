"""The 'visible + (graph - graph.detach())' form on the CPU: forward values from one
computation, gradients from another (vLLM blog "Finish RL training faster", section 3.1)."""
import torch

from bit_consistent_logprob_gb300 import visible_with_graph_gradient


def test_value_is_visible_and_gradient_is_the_graphs():
    torch.manual_seed(0)
    X = torch.randn(5, 8, dtype=torch.float64, requires_grad=True)
    W = torch.randn(11, 8, dtype=torch.float64, requires_grad=True)
    ids = torch.tensor([0, 3, 10, 7, 7])
    graph = torch.log_softmax(X @ W.T, dim=-1)[torch.arange(5), ids]
    visible = (graph + 1e-9).detach()  # e.g. the inference kernel's bits
    out = visible_with_graph_gradient(visible, graph)
    assert torch.equal(out.detach(), visible)
    g = torch.linspace(-1, 1, 5, dtype=torch.float64)
    (out * g).sum().backward(retain_graph=True)
    gx, gw = X.grad.clone(), W.grad.clone()
    X.grad = None
    W.grad = None
    (graph * g).sum().backward()
    assert torch.equal(gx, X.grad) and torch.equal(gw, W.grad)
