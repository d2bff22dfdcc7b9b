"""Thin ctypes binding over libfa.so, with the C ABI's names.

Argument marshalling only: every step of the attention computation runs in the
library's CUDA kernels.  torch supplies device memory and the current stream.
There is no CPU path; a missing library or a non-CUDA tensor raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import os

import torch

from . import build as _build

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_MISALIGNED = 3
FA_ERR_CUDA = 4
FA_ERR_TIMEOUT = 5
FA_ERR_WORKSPACE = 6
FA_ERR_BAD_INDEX = 7

EXPORTED = ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_status_string", "fa_device_status",
            "fa_selftest_wait_timeout", "fa_decode", "fa_decode_num_splits",
            "fa_decode_uses_tensor_cores",
            "fa_decode_workspace_bytes", "fa_decode_paged", "fa_decode_paged_num_splits",
            "fa_decode_paged_workspace_bytes", "fa_fwd_gqa", "fa_bwd_gqa", "fa_fwd_varlen",
            "fa_bwd_varlen", "fa_quantize_fp8_workspace_bytes", "fa_quantize_fp8", "fa_fwd_fp8",
            "fa_probe_unit_rates", "fa_probe_read_bandwidth", "fa_fwd_ws", "fa_fwd_workspace_bytes",
            "fa_fwd_split_segments")

_vp = ctypes.c_void_p
_int = ctypes.c_int
_LIB = None


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fa_status_string(status)} (status {status})")


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libfa.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first (__graft_entry__.build())")
        lib = ctypes.CDLL(path)
        lib.fa_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _int,
                               ctypes.c_float, _vp]
        lib.fa_fwd.restype = _int
        lib.fa_bwd_workspace_bytes.argtypes = [_int, _int, _int, _int]
        lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _int, _int,
                               _int, _int, ctypes.c_float, _vp, ctypes.c_size_t, _vp]
        lib.fa_bwd.restype = _int
        lib.fa_status_string.argtypes = [_int]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_device_status.argtypes = [_vp]
        lib.fa_device_status.restype = _int
        lib.fa_fwd_gqa.argtypes = [_vp] * 5 + [_int] * 6 + [ctypes.c_float, _vp]
        lib.fa_fwd_gqa.restype = _int
        lib.fa_bwd_gqa.argtypes = [_vp] * 9 + [_int] * 6 + [ctypes.c_float, _vp, ctypes.c_size_t, _vp]
        lib.fa_bwd_gqa.restype = _int
        lib.fa_fwd_varlen.argtypes = [_vp] * 6 + [_int] * 7 + [ctypes.c_float, _vp]
        lib.fa_fwd_varlen.restype = _int
        lib.fa_bwd_varlen.argtypes = [_vp] * 10 + [_int] * 7 + [ctypes.c_float, _vp, ctypes.c_size_t,
                                                                 _vp]
        lib.fa_bwd_varlen.restype = _int
        lib.fa_quantize_fp8_workspace_bytes.argtypes = [_int] * 3
        lib.fa_quantize_fp8_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_quantize_fp8.argtypes = [_vp] * 3 + [_int] * 4 + [_vp, _int, _vp, ctypes.c_size_t, _vp]
        lib.fa_quantize_fp8.restype = _int
        lib.fa_fwd_fp8.argtypes = [_vp] * 8 + [_int] * 6 + [ctypes.c_float, _vp]
        lib.fa_fwd_fp8.restype = _int
        lib.fa_decode.argtypes = [_vp] * 5 + [_int] * 6 + [ctypes.c_float, _int, _vp,
                                                          ctypes.c_size_t, _vp]
        lib.fa_decode.restype = _int
        lib.fa_decode_num_splits.argtypes = [_int] * 7
        lib.fa_decode_num_splits.restype = _int
        lib.fa_decode_uses_tensor_cores.argtypes = [_int] * 5
        lib.fa_decode_uses_tensor_cores.restype = _int
        lib.fa_decode_workspace_bytes.argtypes = [_int] * 7
        lib.fa_decode_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_decode_paged.argtypes = [_vp] * 7 + [_int] * 8 + [ctypes.c_float, _int, _vp,
                                                                ctypes.c_size_t, _vp]
        lib.fa_decode_paged.restype = _int
        lib.fa_decode_paged_num_splits.argtypes = [_int] * 8
        lib.fa_decode_paged_num_splits.restype = _int
        lib.fa_decode_paged_workspace_bytes.argtypes = [_int] * 8
        lib.fa_decode_paged_workspace_bytes.restype = ctypes.c_size_t
        _LIB = lib
    return _LIB


# ------------------------------------------------------------ raw C-ABI calls

def fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, stream) -> int:
    return load().fa_fwd(q, k, v, o, lse, B, H, N, d, int(bool(causal)), scale, stream)


def fa_bwd_workspace_bytes(B, H, N, d) -> int:
    return load().fa_bwd_workspace_bytes(B, H, N, d)


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, causal, scale, workspace,
           workspace_bytes, stream) -> int:
    return load().fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, int(bool(causal)),
                         scale, workspace, workspace_bytes, stream)


def fa_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, causal, scale,
                   stream) -> int:
    """fa_bwd without a workspace: the library's fixed scratch array is used instead."""
    fn = load().fa_bwd_noalloc
    if fn.argtypes is None:
        fn.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _int,
                       ctypes.c_float, _vp]
        fn.restype = _int
    return fn(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, int(bool(causal)), scale, stream)


def fa_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    """Run the bounded-wait self test (a wait nothing satisfies, limited to limit_ns)."""
    fn = load().fa_selftest_wait_timeout
    if fn.argtypes is None:
        fn.argtypes = [ctypes.c_ulonglong, _vp]
        fn.restype = _int
    return fn(limit_ns, stream)


def fa_probe_unit_rates(rates, iters: int, stream=None) -> int:
    """Run the unit-rate probes; `rates` is a ctypes array of 3 doubles (host)."""
    fn = load().fa_probe_unit_rates
    if fn.argtypes is None:
        fn.argtypes = [ctypes.POINTER(ctypes.c_double), _int, _vp]
        fn.restype = _int
    return fn(rates, iters, stream)


def fa_probe_read_bandwidth(buf, nbytes: int, iters: int, stream, gbs) -> int:
    """Time streaming reads of nbytes at device pointer buf; `gbs` a ctypes double."""
    fn = load().fa_probe_read_bandwidth
    if fn.argtypes is None:
        fn.argtypes = [_vp, ctypes.c_size_t, _int, _vp, ctypes.POINTER(ctypes.c_double)]
        fn.restype = _int
    return fn(buf, nbytes, iters, stream, ctypes.byref(gbs))


def probe_read_bandwidth(t, iters: int = 5) -> float:
    """HBM read rate (GB/s) measured by reading the CUDA tensor `t` (contiguous, far
    larger than L2; its first multiple of 16 bytes is read, nothing is written)."""
    _check("t", t, t.dtype)
    nbytes = t.numel() * t.element_size() // 16 * 16
    gbs = ctypes.c_double(0.0)
    with torch.cuda.device(t.device):
        rc = fa_probe_read_bandwidth(t.data_ptr(), nbytes, int(iters), _stream(t, None), gbs)
    if rc != FA_OK:
        raise FaError(rc, "fa_probe_read_bandwidth")
    return gbs.value


def probe_unit_rates(iters: int = 2048, stream=None) -> dict:
    """Measured per-SM rates on the current device: dense bf16 MMA FLOPs per SM clock
    at M = 128 with N = 256 and N = 64, and MUFU ex2 results per SM clock."""
    rates = (ctypes.c_double * 3)()
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    rc = fa_probe_unit_rates(rates, int(iters), stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_probe_unit_rates")
    return {"mma_bf16_n256_flop_per_clk": rates[0], "mma_bf16_n64_flop_per_clk": rates[1],
            "ex2_per_clk": rates[2]}


def fa_fwd_workspace_bytes(B, H, N, d, causal, kv_chunk=0) -> int:
    fn = load().fa_fwd_workspace_bytes
    if fn.argtypes is None:
        fn.argtypes = [_int] * 6
        fn.restype = ctypes.c_size_t
    return fn(B, H, N, d, int(bool(causal)), kv_chunk)


def fa_fwd_split_segments(B, H, N, d, causal, num_sms, out=None, cap=0) -> int:
    """Raw call: fills `out` (ctypes int array of 7 * cap) and returns the count."""
    fn = load().fa_fwd_split_segments
    if fn.argtypes is None:
        fn.argtypes = [_int] * 6 + [_vp, _int]
        fn.restype = _int
    return fn(B, H, N, d, int(bool(causal)), num_sms, out, cap)


def fwd_split_segments(B, H, N, d, causal, num_sms):
    """The balanced cut of fa_fwd_ws (kv_chunk = 0) for num_sms SMs, as a list of
    (head, row block, first K/V tile, K/V tiles, part, parts, CTA) tuples ([]: no
    such cut).  Host only."""
    n = fa_fwd_split_segments(B, H, N, d, causal, num_sms)
    if n < 0:
        raise FaError(n, "fa_fwd_split_segments")
    if n == 0:
        return []
    buf = (ctypes.c_int * (7 * n))()
    fa_fwd_split_segments(B, H, N, d, causal, num_sms, ctypes.cast(buf, _vp), n)
    return [tuple(buf[7 * i:7 * i + 7]) for i in range(n)]


def fa_fwd_ws(q, k, v, o, lse, B, H, Hkv, N, d, causal, scale, kv_chunk, workspace,
              workspace_bytes, stream) -> int:
    fn = load().fa_fwd_ws
    if fn.argtypes is None:
        fn.argtypes = [_vp] * 5 + [_int] * 6 + [ctypes.c_float, _int, _vp, ctypes.c_size_t, _vp]
        fn.restype = _int
    return fn(q, k, v, o, lse, B, H, Hkv, N, d, int(bool(causal)), scale, kv_chunk, workspace,
              workspace_bytes, stream)


def fa_fwd_gqa(q, k, v, o, lse, B, H, Hkv, N, d, causal, scale, stream) -> int:
    return load().fa_fwd_gqa(q, k, v, o, lse, B, H, Hkv, N, d, int(bool(causal)), scale, stream)


def fa_bwd_gqa(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, d, causal, scale, workspace,
               workspace_bytes, stream) -> int:
    return load().fa_bwd_gqa(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, d, int(bool(causal)),
                             scale, workspace, workspace_bytes, stream)


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens, B, H, Hkv, total_tokens, max_seqlen, d, causal,
                  scale, stream) -> int:
    return load().fa_fwd_varlen(q, k, v, o, lse, cu_seqlens, B, H, Hkv, total_tokens, max_seqlen,
                                d, int(bool(causal)), scale, stream)


def fa_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens, B, H, Hkv, total_tokens,
                  max_seqlen, d, causal, scale, workspace, workspace_bytes, stream) -> int:
    return load().fa_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens, B, H, Hkv,
                                total_tokens, max_seqlen, d, int(bool(causal)), scale, workspace,
                                workspace_bytes, stream)


def fa_quantize_fp8_workspace_bytes(BH, N, d) -> int:
    return load().fa_quantize_fp8_workspace_bytes(BH, N, d)


def fa_quantize_fp8(x, codes, descale, BH, N, d, block_rows, signs, transpose, workspace,
                    workspace_bytes, stream) -> int:
    return load().fa_quantize_fp8(x, codes, descale, BH, N, d, block_rows, signs,
                                  int(bool(transpose)), workspace, workspace_bytes, stream)


def fa_fwd_fp8(q8, k8, vt8, q_descale, k_descale, v_descale, o, lse, B, H, Hkv, N, d, causal,
               scale, stream) -> int:
    return load().fa_fwd_fp8(q8, k8, vt8, q_descale, k_descale, v_descale, o, lse, B, H, Hkv, N,
                             d, int(bool(causal)), scale, stream)


def fa_decode(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, num_splits, workspace,
              workspace_bytes, stream) -> int:
    return load().fa_decode(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, num_splits, workspace,
                            workspace_bytes, stream)


def fa_decode_num_splits(B, H, Hkv, Nq, Nk, d, num_splits=0) -> int:
    return load().fa_decode_num_splits(B, H, Hkv, Nq, Nk, d, num_splits)


def fa_decode_uses_tensor_cores(H, Hkv, Nq, d, paged=0) -> int:
    return load().fa_decode_uses_tensor_cores(H, Hkv, Nq, d, int(paged))


def fa_decode_workspace_bytes(B, H, Hkv, Nq, Nk, d, num_splits=0) -> int:
    return load().fa_decode_workspace_bytes(B, H, Hkv, Nq, Nk, d, num_splits)


def fa_decode_paged(q, k_cache, v_cache, block_table, seq_lens, o, lse, B, H, Hkv, Nq, d,
                    page_size, max_pages, num_pages, scale, num_splits, workspace,
                    workspace_bytes, stream) -> int:
    return load().fa_decode_paged(q, k_cache, v_cache, block_table, seq_lens, o, lse, B, H, Hkv,
                                  Nq, d, page_size, max_pages, num_pages, scale, num_splits,
                                  workspace, workspace_bytes, stream)


def fa_decode_paged_num_splits(B, H, Hkv, Nq, d, page_size, max_pages, num_splits=0) -> int:
    return load().fa_decode_paged_num_splits(B, H, Hkv, Nq, d, page_size, max_pages, num_splits)


def fa_decode_paged_workspace_bytes(B, H, Hkv, Nq, d, page_size, max_pages, num_splits=0) -> int:
    return load().fa_decode_paged_workspace_bytes(B, H, Hkv, Nq, d, page_size, max_pages,
                                                  num_splits)


def fa_status_string(status: int) -> str:
    return load().fa_status_string(status).decode()


def fa_device_status(stream=None) -> int:
    return load().fa_device_status(stream)


# ------------------------------------------------------------ tensor wrappers

def _check(name, t, dtype, shape=None, dev=None):
    """Argument checks before any launch: a contiguous CUDA tensor of `dtype` (and
    `shape`) on device `dev` (a torch.device or an ordinal), the first tensor's device:
    the kernels dereference every pointer on that one GPU."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dev is not None and t.get_device() != (dev if isinstance(dev, int) else dev.index):
        raise ValueError(f"{name} is on {t.device}, the call's first tensor on {dev}")
    if t.dtype is not dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and t.shape != shape:
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


# The current stream's handle: torch's raw getter where it has one (a plain integer,
# no Stream object is built), else the public call.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(t, stream):
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(t.get_device())
        return torch.cuda.current_stream(t.device).cuda_stream
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


_SAME_DEVICE = contextlib.nullcontext()


def _device(index: int):
    """The device context for a call on GPU `index`: a no-op when it is already
    current (the common case), else torch.cuda.device(index)."""
    return _SAME_DEVICE if torch.cuda.current_device() == index else torch.cuda.device(index)


_SIZE_MEMO: dict = {}


def _memo(fn, *args):
    """fn(*args) for the workspace-size queries, remembered per argument tuple and
    current device (the answers depend only on them and the device's SM count)."""
    key = (fn, torch.cuda.current_device(), args)
    r = _SIZE_MEMO.get(key)
    if r is None:
        if len(_SIZE_MEMO) > 4096:
            _SIZE_MEMO.clear()
        r = _SIZE_MEMO[key] = fn(*args)
    return r


def _kv_heads(q, k, v):
    """Key/value head count of k, v [B, Hkv, N, d] next to q [B, H, N, d] (Hkv divides H)."""
    B, H, N, d = q.shape
    di = q.get_device()
    _check("k", k, torch.bfloat16, dev=di)
    if k.dim() != 4 or k.shape[0] != B or k.shape[2] != N or k.shape[3] != d or H % k.shape[1]:
        raise ValueError("k must be [B, Hkv, N, d] with Hkv dividing q's H")
    _check("v", v, torch.bfloat16, k.shape, dev=di)
    return k.shape[1]


def forward(q, k, v, causal=False, scale=None, out=None, lse=None, stream=None, kv_chunk=0,
            workspace=None):
    """O, L = attention(q, k, v); q bf16 CUDA [B,H,N,d], k/v [B,Hkv,N,d] (Hkv = H, or
    fewer heads shared by groups of query heads).  Returns (o, lse).

    When few long heads would leave SMs idle, the key ranges are cut over several
    CTAs and merged (fa_fwd_ws): kv_chunk = 0 lets the library decide, > 0 asks for
    chunks of about that many keys; the workspace that needs is allocated here
    unless given."""
    _check("q", q, torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    B, H, N, d = q.shape
    di = q.get_device()
    Hkv = _kv_heads(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    _check("out", out, torch.bfloat16, q.shape, dev=di)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check("lse", lse, torch.float32, (B, H, N), dev=di)
    with _device(di):
        need = _memo(fa_fwd_workspace_bytes, B, H, N, d, causal, int(kv_chunk))
        if need == 0:
            rc = fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            lse.data_ptr(), B, H, Hkv, N, d, causal, scale, _stream(q, stream))
            where = "fa_fwd_gqa"
        else:
            if workspace is None:
                workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            _check("workspace", workspace, torch.uint8, dev=q.device)
            rc = fa_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           lse.data_ptr(), B, H, Hkv, N, d, causal, scale, int(kv_chunk),
                           workspace.data_ptr(), workspace.numel(), _stream(q, stream))
            where = "fa_fwd_ws"
    if rc != FA_OK:
        raise FaError(rc, where)
    return out, lse


def backward(q, k, v, o, lse, do, causal=False, scale=None, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """dQ, dK, dV (fp32) of attention(q, k, v) given dO; o and lse from forward().
    With fewer key/value heads (k, v [B,Hkv,N,d]) dK, dV are [B,Hkv,N,d] sums over
    each head's query group."""
    _check("q", q, torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    B, H, N, d = q.shape
    Hkv = _kv_heads(q, k, v)
    for name, t in (("o", o), ("do", do)):
        _check(name, t, torch.bfloat16, q.shape, dev=q.device)
    _check("lse", lse, torch.float32, (B, H, N), dev=q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    grads = []
    for name, t, shape in (("dq", dq, q.shape), ("dk", dk, k.shape), ("dv", dv, k.shape)):
        if t is None:
            t = torch.empty(shape, dtype=torch.float32, device=q.device)
        _check(name, t, torch.float32, shape, dev=q.device)
        grads.append(t)
    need = fa_bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check("workspace", workspace, torch.uint8, dev=q.device)
    with torch.cuda.device(q.device):
        rc = fa_bwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        do.data_ptr(), grads[0].data_ptr(), grads[1].data_ptr(),
                        grads[2].data_ptr(), B, H, Hkv, N, d, causal, scale, workspace.data_ptr(),
                        workspace.numel(), _stream(q, stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_gqa")
    return tuple(grads)


def decode(q, k, v, scale=None, num_splits=0, out=None, lse=None, workspace=None, stream=None):
    """Decode attention: q bf16 CUDA [B,H,Nq,d] against the cache k, v [B,Hkv,Nk,d]
    (Hkv divides H; no mask), the key range split over CTAs and merged by LSE.
    Returns (o, lse)."""
    _check("q", q, torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, Nq, d]")
    B, H, Nq, d = q.shape
    di = q.get_device()
    _check("k", k, torch.bfloat16, dev=di)
    if k.dim() != 4 or k.shape[0] != B or k.shape[3] != d or H % k.shape[1]:
        raise ValueError("k must be [B, Hkv, Nk, d] with q's B and d, Hkv dividing H")
    Hkv, Nk = k.shape[1], k.shape[2]
    _check("v", v, torch.bfloat16, k.shape, dev=di)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    _check("out", out, torch.bfloat16, q.shape, dev=di)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    _check("lse", lse, torch.float32, (B, H, Nq), dev=di)
    with _device(di):
        need = _memo(fa_decode_workspace_bytes, B, H, Hkv, Nq, Nk, d, num_splits)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        if workspace is not None:
            _check("workspace", workspace, torch.uint8, dev=di)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_len = workspace.numel() if workspace is not None else 0
        rc = fa_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                       B, H, Hkv, Nq, Nk, d, scale, num_splits, ws_ptr, ws_len, _stream(q, stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_decode")
    return out, lse


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale=None, num_splits=0, out=None,
                 lse=None, workspace=None, stream=None):
    """Decode against a paged cache: q bf16 [B,H,Nq,d]; k_cache, v_cache bf16
    [num_pages, Hkv, page_size, d] (Hkv divides H); block_table int32 [B, max_pages];
    seq_lens int32 [B] (all CUDA).  Returns (o, lse)."""
    _check("q", q, torch.bfloat16)
    if q.dim() != 4:
        raise ValueError("q must be [B, H, Nq, d]")
    B, H, Nq, d = q.shape
    _check("k_cache", k_cache, torch.bfloat16, dev=q.device)
    if k_cache.dim() != 4 or H % k_cache.shape[1] or k_cache.shape[3] != d:
        raise ValueError("k_cache must be [num_pages, Hkv, page_size, d], Hkv dividing H")
    num_pages, Hkv, page_size, _ = k_cache.shape
    _check("v_cache", v_cache, torch.bfloat16, k_cache.shape, dev=q.device)
    _check("block_table", block_table, torch.int32, dev=q.device)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_pages]")
    max_pages = block_table.shape[1]
    _check("seq_lens", seq_lens, torch.int32, (B,), dev=q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    _check("out", out, torch.bfloat16, q.shape, dev=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    _check("lse", lse, torch.float32, (B, H, Nq), dev=q.device)
    with torch.cuda.device(q.device):
        need = fa_decode_paged_workspace_bytes(B, H, Hkv, Nq, d, page_size, max_pages, num_splits)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        if workspace is not None:
            _check("workspace", workspace, torch.uint8, dev=q.device)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_len = workspace.numel() if workspace is not None else 0
        rc = fa_decode_paged(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                             block_table.data_ptr(), seq_lens.data_ptr(), out.data_ptr(),
                             lse.data_ptr(), B, H, Hkv, Nq, d, page_size, max_pages, num_pages,
                             scale, num_splits, ws_ptr, ws_len, _stream(q, stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_decode_paged")
    return out, lse


def forward_varlen(q, k, v, cu_seqlens, max_seqlen, causal=False, scale=None, out=None, lse=None,
                   stream=None):
    """Packed variable-length forward: q bf16 CUDA [T,H,d], k/v [T,Hkv,d], cu_seqlens
    int32 CUDA [B+1] (sequence b = tokens cu[b]..cu[b+1]-1, each <= max_seqlen).
    Returns (o [T,H,d], lse [H,T])."""
    _check("q", q, torch.bfloat16)
    if q.dim() != 3:
        raise ValueError("q must be [T, H, d]")
    T, H, d = q.shape
    _check("k", k, torch.bfloat16, dev=q.device)
    if k.dim() != 3 or k.shape[0] != T or k.shape[2] != d or H % k.shape[1]:
        raise ValueError("k must be [T, Hkv, d] with Hkv dividing H")
    Hkv = k.shape[1]
    _check("v", v, torch.bfloat16, k.shape, dev=q.device)
    _check("cu_seqlens", cu_seqlens, torch.int32, dev=q.device)
    if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be [B + 1]")
    B = cu_seqlens.numel() - 1
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    _check("out", out, torch.bfloat16, q.shape, dev=q.device)
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    _check("lse", lse, torch.float32, (H, T), dev=q.device)
    with torch.cuda.device(q.device):
        rc = fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                           cu_seqlens.data_ptr(), B, H, Hkv, T, int(max_seqlen), d, causal, scale,
                           _stream(q, stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_varlen")
    return out, lse


def backward_varlen(q, k, v, o, lse, do, cu_seqlens, max_seqlen, causal=False, scale=None,
                    dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients of forward_varlen: q/o/do bf16 [T,H,d], k/v [T,Hkv,d], lse [H,T].
    Returns (dq [T,H,d], dk [T,Hkv,d], dv [T,Hkv,d]) fp32."""
    _check("q", q, torch.bfloat16)
    if q.dim() != 3:
        raise ValueError("q must be [T, H, d]")
    T, H, d = q.shape
    _check("k", k, torch.bfloat16, dev=q.device)
    if k.dim() != 3 or k.shape[0] != T or k.shape[2] != d or H % k.shape[1]:
        raise ValueError("k must be [T, Hkv, d] with Hkv dividing H")
    Hkv = k.shape[1]
    _check("v", v, torch.bfloat16, k.shape, dev=q.device)
    for name, t in (("o", o), ("do", do)):
        _check(name, t, torch.bfloat16, q.shape, dev=q.device)
    _check("lse", lse, torch.float32, (H, T), dev=q.device)
    _check("cu_seqlens", cu_seqlens, torch.int32, dev=q.device)
    B = cu_seqlens.numel() - 1
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    grads = []
    for name, t, shape in (("dq", dq, q.shape), ("dk", dk, k.shape), ("dv", dv, k.shape)):
        if t is None:
            t = torch.zeros(shape, dtype=torch.float32, device=q.device)
        _check(name, t, torch.float32, shape, dev=q.device)
        grads.append(t)
    need = fa_bwd_workspace_bytes(B, H, int(max_seqlen), d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check("workspace", workspace, torch.uint8, dev=q.device)
    with torch.cuda.device(q.device):
        rc = fa_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           do.data_ptr(), grads[0].data_ptr(), grads[1].data_ptr(),
                           grads[2].data_ptr(), cu_seqlens.data_ptr(), B, H, Hkv, T,
                           int(max_seqlen), d, causal, scale, workspace.data_ptr(),
                           workspace.numel(), _stream(q, stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_varlen")
    return tuple(grads)


def quantize_fp8(x, block_rows=128, signs=None, transpose=False, workspace=None, stream=None):
    """e4m3 block quantisation of x bf16 CUDA [..., N, d] (heads flattened).
    Returns (codes uint8 [..., N, d] or [..., d, Np], descale fp32 [..., n_blocks])."""
    _check("x", x, torch.bfloat16)
    if x.dim() < 2:
        raise ValueError("x must be [..., N, d]")
    *lead, N, d = x.shape
    BH = int(math.prod(lead)) if lead else 1
    Np = (N + 15) // 16 * 16
    codes = torch.empty((*lead, d, Np) if transpose else x.shape, dtype=torch.uint8, device=x.device)
    nb = 1 if block_rows == 0 else (N + block_rows - 1) // block_rows
    descale = torch.empty((*lead, nb), dtype=torch.float32, device=x.device)
    if signs is not None:
        _check("signs", signs, torch.float32, (d,), dev=x.device)
    need = fa_quantize_fp8_workspace_bytes(BH, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _check("workspace", workspace, torch.uint8, dev=x.device)
    with torch.cuda.device(x.device):
        rc = fa_quantize_fp8(x.data_ptr(), codes.data_ptr(), descale.data_ptr(), BH, N, d,
                             int(block_rows), None if signs is None else signs.data_ptr(),
                             transpose, workspace.data_ptr(), workspace.numel(), _stream(x, stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_quantize_fp8")
    return codes, descale


def forward_fp8(q8, k8, vt8, q_descale, k_descale, v_descale, causal=False, scale=None, out=None,
                lse=None, stream=None):
    """Attention on e4m3 inputs: q8 uint8 CUDA [B,H,N,d], k8 [B,Hkv,N,d], vt8 [B,Hkv,d,Np],
    q/k descales [B,H|Hkv,ceil(N/128)], v descale [B,Hkv,1].  Returns (o bf16, lse fp32)."""
    _check("q8", q8, torch.uint8)
    if q8.dim() != 4:
        raise ValueError("q8 must be [B, H, N, d]")
    B, H, N, d = q8.shape
    _check("k8", k8, torch.uint8, dev=q8.device)
    if k8.dim() != 4 or k8.shape[0] != B or k8.shape[2] != N or k8.shape[3] != d or H % k8.shape[1]:
        raise ValueError("k8 must be [B, Hkv, N, d] with Hkv dividing H")
    Hkv = k8.shape[1]
    Np = (N + 15) // 16 * 16
    _check("vt8", vt8, torch.uint8, (B, Hkv, d, Np), dev=q8.device)
    nb = (N + 127) // 128
    _check("q_descale", q_descale, torch.float32, (B, H, nb), dev=q8.device)
    _check("k_descale", k_descale, torch.float32, (B, Hkv, nb), dev=q8.device)
    _check("v_descale", v_descale, torch.float32, (B, Hkv, 1), dev=q8.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    _check("out", out, torch.bfloat16, (B, H, N, d), dev=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    _check("lse", lse, torch.float32, (B, H, N), dev=q8.device)
    with torch.cuda.device(q8.device):
        rc = fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), q_descale.data_ptr(),
                        k_descale.data_ptr(), v_descale.data_ptr(), out.data_ptr(), lse.data_ptr(),
                        B, H, Hkv, N, d, causal, scale, _stream(q8, stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_fp8")
    return out, lse
