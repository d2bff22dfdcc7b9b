"""Host-buffer training steps with copies overlapped on separate streams.

Each step copies q, k, v, dO from pinned host memory to the device, runs the
forward and backward kernels, and copies o, lse, dq, dk, dv back to pinned host
memory.  Issued on one stream those three phases serialise; here each has its own
stream and the device buffers come in `depth` slots, so the copies of one step
overlap the kernels of the next (events order every slot's reuse).  Nothing here
computes: the copies are cudaMemcpyAsync calls and the kernels are the library's.
"""
from __future__ import annotations

import torch

from . import fa


class HostPipeline:
    """Forward + backward over host batches of one shape, `depth` batches in flight.

    q, k, v, dO host tensors: bf16 [B, H, N, d] (k, v may have Hkv heads), pinned for
    the copies to overlap.  Results land in the caller's pinned host tensors o (bf16),
    lse (fp32 [B, H, N]), dq, dk, dv (fp32) once the step's event has completed;
    `synchronize()` waits for every issued step."""

    def __init__(self, B, H, N, d, causal=False, scale=None, Hkv=None, device="cuda:0", depth=2):
        self.dev = torch.device(device)
        self.causal = causal
        self.scale = scale
        Hkv = H if Hkv is None else Hkv
        self.depth = depth
        qs, ks = (B, H, N, d), (B, Hkv, N, d)
        bf, f32 = torch.bfloat16, torch.float32
        with torch.cuda.device(self.dev):
            self.slots = []
            for _ in range(depth):
                self.slots.append({
                    "in": [torch.empty(s, dtype=bf, device=self.dev) for s in (qs, ks, ks, qs)],
                    "o": torch.empty(qs, dtype=bf, device=self.dev),
                    "lse": torch.empty((B, H, N), dtype=f32, device=self.dev),
                    "g": [torch.empty(s, dtype=f32, device=self.dev) for s in (qs, ks, ks)],
                    "ws": torch.empty(max(fa.fa_bwd_workspace_bytes(B, H, N, d), 16),
                                      dtype=torch.uint8, device=self.dev),
                    "h2d": torch.cuda.Event(), "done": torch.cuda.Event(), "d2h": torch.cuda.Event(),
                    "used": False,
                })
            self.s_h2d = torch.cuda.Stream(self.dev)
            self.s_run = torch.cuda.Stream(self.dev)
            self.s_d2h = torch.cuda.Stream(self.dev)
        self.n = 0

    def step(self, host_in, host_out):
        """Issue one step: host_in = (q, k, v, dO), host_out = (o, lse, dq, dk, dv).

        Returns (h2d, d2h) events.  The copies run asynchronously: do not overwrite
        the pinned host_in tensors until `h2d` has completed (their bytes are still
        being read), and read host_out only once `d2h` has completed."""
        sl = self.slots[self.n % self.depth]
        self.n += 1
        if sl["used"]:
            # the slot's inputs are free once its last kernels ran, its outputs once
            # they were copied out
            self.s_h2d.wait_event(sl["done"])
            self.s_run.wait_event(sl["d2h"])
        sl["used"] = True
        with torch.cuda.stream(self.s_h2d):
            for dst, src in zip(sl["in"], host_in):
                dst.copy_(src, non_blocking=True)
            sl["h2d"].record(self.s_h2d)
        self.s_run.wait_event(sl["h2d"])
        q, k, v, do = sl["in"]
        fa.forward(q, k, v, causal=self.causal, scale=self.scale, out=sl["o"], lse=sl["lse"],
                   stream=self.s_run)
        fa.backward(q, k, v, sl["o"], sl["lse"], do, causal=self.causal, scale=self.scale,
                    dq=sl["g"][0], dk=sl["g"][1], dv=sl["g"][2], workspace=sl["ws"],
                    stream=self.s_run)
        sl["done"].record(self.s_run)
        self.s_d2h.wait_event(sl["done"])
        with torch.cuda.stream(self.s_d2h):
            for dst, src in zip(host_out, [sl["o"], sl["lse"]] + sl["g"]):
                dst.copy_(src, non_blocking=True)
            sl["d2h"].record(self.s_d2h)
        return sl["h2d"], sl["d2h"]

    def synchronize(self):
        for s in (self.s_h2d, self.s_run, self.s_d2h):
            s.synchronize()
