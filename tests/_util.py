"""Shared helpers of the test suite: the parity criteria and cached inputs."""
import functools

import torch

# Parity bar: bf16 outputs and gradients within 2e-2 * max|ref| + 2e-3 per
# tensor; fp32 LSE within 1e-4 relative (absolute below magnitude 1).
REL, ATOL, LSE_REL = 2e-2, 2e-3, 1e-4


def max_err(got, ref):
    got = got.detach().to("cpu", torch.float64)
    ref = ref.to(torch.float64)
    return (got - ref).abs().max().item(), REL * ref.abs().max().item() + ATOL


def assert_close(name, got, ref):
    assert got.shape == ref.shape, f"{name}: shape {tuple(got.shape)} vs {tuple(ref.shape)}"
    g = got.detach().to("cpu", torch.float64)
    assert torch.isfinite(g).all(), f"{name}: non-finite values"
    err, lim = max_err(g, ref)
    assert err <= lim, f"{name}: max err {err:.4e} > {lim:.4e}"


def assert_lse(name, got, ref):
    g = got.detach().to("cpu", torch.float64)
    r = ref.to(torch.float64)
    inf = torch.isinf(r)
    assert torch.equal(torch.isinf(g) & (g < 0), inf & (r < 0)), f"{name}: -inf pattern differs"
    fin = ~inf
    rel = ((g[fin] - r[fin]).abs() / r[fin].abs().clamp(min=1.0))
    if rel.numel():
        assert rel.max().item() <= LSE_REL, f"{name}: lse rel err {rel.max().item():.3e}"


@functools.lru_cache(maxsize=4)
def workload_inputs(name):
    from softmax_attention_backward_gb300 import workloads as W
    w = W.get_workload(name)
    return w, W.make_inputs(w)
