"""The host-buffer pipeline (copies and kernels on separate streams, two steps in
flight) gives every step the results of the plain calls on that step's inputs."""
import pytest
import torch

from exact_attention_26_gb300.inputs import normal_qkv
from exact_attention_26_gb300.pipeline import HostPipeline
from gpu_common import load_fa

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def fa():
    return load_fa()


@pytest.mark.parametrize("causal", [False, True])
def test_pipeline_matches_plain_calls(fa, causal):
    B, H, N, d = 1, 2, 300, 128
    steps = 5
    ins = [[t.pin_memory() for t in normal_qkv(B, H, N, d, seed=40 + i, with_do=True)] for i in range(steps)]
    outs = [[torch.empty((B, H, N, d), dtype=torch.bfloat16).pin_memory(),
             torch.empty((B, H, N), dtype=torch.float32).pin_memory()] +
            [torch.empty((B, H, N, d), dtype=torch.float32).pin_memory() for _ in range(3)]
            for _ in range(steps)]
    pipe = HostPipeline(B, H, N, d, causal=causal, device=DEV, depth=2)
    for i in range(steps):
        pipe.step(ins[i], outs[i])
    pipe.synchronize()
    for i in range(steps):
        q, k, v, do = (t.to(DEV) for t in ins[i])
        o, lse = fa.forward(q, k, v, causal=causal)
        dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal)
        torch.cuda.synchronize()
        got = outs[i]
        assert torch.equal(got[0], o.cpu()) and torch.equal(got[1], lse.cpu()), f"step {i} forward"
        assert torch.equal(got[3], dk.cpu()) and torch.equal(got[4], dv.cpu()), f"step {i} dK/dV"
        assert torch.allclose(got[2], dq.cpu(), rtol=1e-5, atol=1e-6), f"step {i} dQ"
    assert fa.fa_device_status(None) == 0
