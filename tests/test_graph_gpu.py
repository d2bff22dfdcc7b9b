"""The library's calls inside CUDA graphs: forward + backward, and decode, captured
once into a torch.cuda.CUDAGraph (static input and output tensors, the workspaces
allocated before capture) and replayed on new input values, against the same calls
made eagerly.  A call that synchronised, allocated device memory by itself or
launched outside the capture stream would fail the capture or the comparison.

Forward and decode are deterministic, so the replays must match bit for bit; the
backward's dQ sums partial products with asynchronous bulk adds whose order varies,
so dQ is compared to 1e-5 and dK, dV (one CTA each) bit for bit."""
import pytest
import torch

from exact_attention_26_gb300.inputs import decode_qkv, normal_qkv
from gpu_common import load_fa

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def test_forward_backward_step_replays_from_a_graph():
    fa = load_fa()
    B, H, N, d = 2, 4, 1000, 128
    first = [t.to(DEV) for t in normal_qkv(B, H, N, d, seed=41, with_do=True)]
    second = [t.to(DEV) for t in normal_qkv(B, H, N, d, seed=42, with_do=True)]
    q, k, v, do = (t.clone() for t in first)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    dq, dk, dv = (torch.empty(q.shape, dtype=torch.float32, device=DEV) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=DEV)

    def step():
        fa.forward(q, k, v, causal=True, out=o, lse=lse)
        fa.backward(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside the capture (kernel attributes, tensor maps)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for inputs in (second, first):
        for dst, src in zip((q, k, v, do), inputs):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        assert fa.fa_device_status(None) == 0
        got = [t.clone() for t in (o, lse, dq, dk, dv)]
        ro, rl = fa.forward(*inputs[:3], causal=True)
        rq, rk, rv = fa.backward(*inputs[:3], ro, rl, inputs[3], causal=True)
        torch.cuda.synchronize()
        assert torch.equal(got[0], ro) and torch.equal(got[1], rl)
        assert torch.allclose(got[2], rq, atol=1e-5, rtol=0)
        assert torch.equal(got[3], rk) and torch.equal(got[4], rv)


def test_decode_replays_from_a_graph():
    fa = load_fa()
    B, H, Nq, Nk, d = 2, 8, 1, 5000, 128
    q, k, v = decode_qkv(B, H, Nq, Nk, d, seed=43, device=DEV)
    q2 = decode_qkv(B, H, Nq, 1, d, seed=44, device=DEV)[0]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=DEV)
    ws = torch.empty(max(16, fa.fa_decode_workspace_bytes(B, H, H, Nq, Nk, d, 0)),
                     dtype=torch.uint8, device=DEV)
    qs = q.clone()

    def call():
        fa.decode(qs, k, v, out=o, lse=lse, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for qi in (q2, q):
        qs.copy_(qi)
        graph.replay()
        torch.cuda.synchronize()
        assert fa.fa_device_status(None) == 0
        ro, rl = fa.decode(qi, k, v)
        torch.cuda.synchronize()
        assert torch.equal(o, ro) and torch.equal(lse, rl)
