"""The C ABI without a GPU: symbols, status strings and argument validation.

Every call here returns before anything touches CUDA, so it runs on the CPU.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fa():
    from exact_attention_26_gb300 import build as fb
    if fb.needs_build():
        fb.build()
    import exact_attention_26_gb300 as fa
    fa.load()
    return fa


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_status_string", "fa_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(fa):
    lib = ctypes.CDLL(fa.fa.lib_path())
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_status_strings(fa):
    for code in range(8):
        s = fa.fa_status_string(code)
        assert s and s != "unknown fa_status"
    assert fa.fa_status_string(99) == "unknown fa_status"


DUMMY = 0x10000  # 16-byte aligned, never dereferenced: validation fails first


def _fwd(fa, **kw):
    a = dict(q=DUMMY, k=DUMMY, v=DUMMY, o=DUMMY, lse=DUMMY, B=1, H=1, N=128, d=64, causal=0,
             scale=0.125, stream=None)
    a.update(kw)
    return fa.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["N"], a["d"],
                     a["causal"], a["scale"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(o=None), 1), (dict(lse=None), 1),
    (dict(B=0), 1), (dict(H=-1), 1), (dict(N=0), 1), (dict(B=65536, H=256, N=256), 1),
    (dict(d=80), 2), (dict(d=32), 2), (dict(d=0), 2),
    (dict(scale=0.0), 1), (dict(scale=-1.0), 1), (dict(scale=float("inf")), 1), (dict(scale=float("nan")), 1),
    (dict(q=DUMMY + 8), 3), (dict(lse=DUMMY + 4), 3), (dict(o=DUMMY + 2), 3),
])
def test_fwd_rejects_bad_arguments(fa, kw, code):
    assert _fwd(fa, **kw) == code


def _bwd(fa, **kw):
    a = dict(q=DUMMY, k=DUMMY, v=DUMMY, o=DUMMY, lse=DUMMY, do=DUMMY, dq=DUMMY, dk=DUMMY, dv=DUMMY,
             B=1, H=1, N=128, d=128, causal=1, scale=0.125, ws=DUMMY, ws_bytes=1 << 20, stream=None)
    a.update(kw)
    return fa.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"],
                     a["B"], a["H"], a["N"], a["d"], a["causal"], a["scale"], a["ws"], a["ws_bytes"],
                     a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(do=None), 1), (dict(dq=None), 1), (dict(dv=None), 1),
    (dict(N=0), 1), (dict(d=256), 2), (dict(d=80), 2), (dict(scale=0.0), 1),
    (dict(ws=None), 6), (dict(ws_bytes=16), 6),
    (dict(dk=DUMMY + 4), 3), (dict(ws=DUMMY + 8), 3),
])
def test_bwd_rejects_bad_arguments(fa, kw, code):
    assert _bwd(fa, **kw) == code


def test_workspace_size(fa):
    # delta and base-2 lse, fp32, rows padded to 128 per head, and a 16-byte work counter
    assert fa.fa_bwd_workspace_bytes(2, 16, 4096, 128) == 2 * 32 * 4096 * 4 + 16
    assert fa.fa_bwd_workspace_bytes(1, 1, 129, 64) == 2 * 256 * 4 + 16
    assert fa.fa_bwd_workspace_bytes(1, 1, 0, 64) == 0
    assert fa.fa_bwd_workspace_bytes(1, 1, 128, 256) == 0
    assert fa.fa_bwd_workspace_bytes(1, 2, 100, 96) == 2 * 2 * 128 * 4 + 16


def test_python_wrapper_rejects_cpu_tensors(fa):
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.forward(q, q, q)


def _on(t, index):
    """A CPU tensor that reports CUDA device `index`: enough for the wrappers'
    argument checks, which all run before anything is allocated or launched."""
    import torch

    class OnDevice(torch.Tensor):
        @property
        def device(self):
            return self._reported

        @property
        def is_cuda(self):
            return True

        def get_device(self):
            return self._reported.index

    s = t.as_subclass(OnDevice)
    s._reported = torch.device("cuda", index)
    return s


def test_python_wrapper_rejects_tensors_on_another_device(fa):
    import torch
    x = lambda i, shape=(1, 2, 8, 64), dt=torch.bfloat16: _on(torch.zeros(shape, dtype=dt), i)
    q = x(0)
    with pytest.raises(ValueError, match="k is on cuda:1"):
        fa.forward(q, x(1), x(0), out=x(0), lse=x(0, (1, 2, 8), torch.float32))
    with pytest.raises(ValueError, match="lse is on cuda:1"):
        fa.forward(q, x(0), x(0), out=x(0), lse=x(1, (1, 2, 8), torch.float32))
    lse0 = x(0, (1, 2, 8), torch.float32)
    with pytest.raises(ValueError, match="do is on cuda:1"):
        fa.backward(q, x(0), x(0), x(0), lse0, x(1))
    with pytest.raises(ValueError, match="dq is on cuda:1"):
        fa.backward(q, x(0), x(0), x(0), lse0, x(0), dq=x(1, dt=torch.float32))
    with pytest.raises(ValueError, match="v is on cuda:1"):
        fa.decode(x(0, (1, 2, 1, 64)), x(0), x(1))


def _dec(fa, **kw):
    a = dict(q=DUMMY, k=DUMMY, v=DUMMY, o=DUMMY, lse=DUMMY, B=1, H=2, Hkv=2, Nq=1, Nk=1000, d=128,
             scale=0.1, splits=0, ws=None, ws_bytes=0, stream=None)
    a.update(kw)
    return fa.fa_decode(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Hkv"], a["Nq"],
                        a["Nk"], a["d"], a["scale"], a["splits"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(o=None), 1), (dict(lse=None), 1),
    (dict(B=0), 1), (dict(H=0), 1), (dict(Nq=0), 1), (dict(Nq=65536), 1), (dict(Nk=0), 1),
    (dict(B=65536, H=256, Hkv=256, Nk=256), 1), (dict(d=80), 2), (dict(d=32), 2),
    (dict(Hkv=0), 1), (dict(Hkv=3), 1), (dict(Hkv=4), 1), (dict(H=4096, Hkv=1, Nq=17), 1),
    (dict(scale=0.0), 1), (dict(scale=float("nan")), 1), (dict(splits=-1), 1),
    (dict(q=DUMMY + 8), 3), (dict(k=DUMMY + 2), 3), (dict(lse=DUMMY + 4), 3),
])
def test_decode_rejects_bad_arguments(fa, kw, code):
    assert _dec(fa, **kw) == code


def test_decode_kernel_choice(fa):
    """Several rows per key/value head with d <= 128 and a contiguous cache: the
    tensor-core kernel; one row, d = 256 or a paged cache: the CUDA-core one."""
    assert fa.fa_decode_uses_tensor_cores(32, 32, 4, 128, 0) == 1
    assert fa.fa_decode_uses_tensor_cores(32, 8, 1, 64, 0) == 1
    assert fa.fa_decode_uses_tensor_cores(32, 32, 2, 96, 0) == 1
    assert fa.fa_decode_uses_tensor_cores(32, 32, 1, 128, 0) == 0
    assert fa.fa_decode_uses_tensor_cores(32, 32, 4, 256, 0) == 0
    assert fa.fa_decode_uses_tensor_cores(32, 32, 4, 128, 1) == 0
    assert fa.fa_decode_uses_tensor_cores(6, 4, 1, 128, 0) == -1
    assert fa.fa_decode_uses_tensor_cores(4, 4, 1, 80, 0) == -2


def test_decode_split_queries_reject_bad_sizes(fa):
    assert fa.fa_decode_num_splits(0, 1, 1, 1, 100, 128, 0) == -1
    assert fa.fa_decode_num_splits(1, 1, 1, 1, 100, 80, 0) == -2
    assert fa.fa_decode_num_splits(1, 1, 1, 1, 100, 128, -3) == -1
    assert fa.fa_decode_num_splits(1, 6, 4, 1, 100, 128, 0) == -1
    assert fa.fa_decode_workspace_bytes(1, 1, 1, 0, 100, 128, 0) == 0
    assert fa.fa_decode_workspace_bytes(1, 1, 1, 1, 100, 80, 2) == 0


def _pdec(fa, **kw):
    a = dict(q=DUMMY, kc=DUMMY, vc=DUMMY, bt=DUMMY, sl=DUMMY, o=DUMMY, lse=DUMMY, B=2, H=2, Hkv=1,
             Nq=1, d=128, ps=16, mp=8, np_=16, scale=0.1, splits=0, ws=None, ws_bytes=0, stream=None)
    a.update(kw)
    return fa.fa_decode_paged(a["q"], a["kc"], a["vc"], a["bt"], a["sl"], a["o"], a["lse"], a["B"],
                              a["H"], a["Hkv"], a["Nq"], a["d"], a["ps"], a["mp"], a["np_"],
                              a["scale"], a["splits"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(kc=None), 1), (dict(bt=None), 1), (dict(sl=None), 1), (dict(lse=None), 1),
    (dict(B=0), 1), (dict(Nq=0), 1), (dict(ps=0), 1), (dict(mp=0), 1), (dict(np_=0), 1),
    (dict(ps=1 << 16, mp=1 << 16), 1), (dict(d=80), 2), (dict(scale=-1.0), 1), (dict(splits=-2), 1),
    (dict(Hkv=3), 1), (dict(Hkv=0), 1),
    (dict(kc=DUMMY + 8), 3), (dict(bt=DUMMY + 2), 3), (dict(sl=DUMMY + 1), 3),
])
def test_decode_paged_rejects_bad_arguments(fa, kw, code):
    assert _pdec(fa, **kw) == code


def test_decode_paged_split_queries_reject_bad_sizes(fa):
    assert fa.fa_decode_paged_num_splits(1, 1, 1, 1, 128, 0, 4, 0) == -1
    assert fa.fa_decode_paged_num_splits(1, 1, 1, 1, 80, 16, 4, 0) == -2
    assert fa.fa_decode_paged_workspace_bytes(1, 1, 1, 1, 128, 16, 0, 2) == 0


@pytest.mark.parametrize("Hkv,code", [(0, 1), (3, 1), (5, 1), (-1, 1)])
def test_gqa_rejects_bad_head_counts(fa, Hkv, code):
    assert fa.fa.fa_fwd_gqa(DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, 1, 4, Hkv, 128, 64, 0, 0.1, None) == code
    assert fa.fa.fa_bwd_gqa(DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, 1, 4, Hkv, 128,
                            128, 1, 0.1, DUMMY, 1 << 20, None) == code


@pytest.mark.parametrize("kw,code", [
    (dict(cu=None), 1), (dict(q=None), 1), (dict(B=0), 1), (dict(T=0), 1), (dict(maxlen=0), 1),
    (dict(Hkv=3), 1), (dict(d=80), 2), (dict(scale=0.0), 1), (dict(cu=DUMMY + 2), 3), (dict(q=DUMMY + 8), 3),
])
def test_varlen_rejects_bad_arguments(fa, kw, code):
    a = dict(q=DUMMY, k=DUMMY, v=DUMMY, o=DUMMY, lse=DUMMY, cu=DUMMY, B=2, H=4, Hkv=2, T=100,
             maxlen=64, d=128, causal=1, scale=0.1)
    a.update(kw)
    assert fa.fa_fwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cu"], a["B"], a["H"], a["Hkv"],
                            a["T"], a["maxlen"], a["d"], a["causal"], a["scale"], None) == code


@pytest.mark.parametrize("kw,code", [
    (dict(cu=None), 1), (dict(dq=None), 1), (dict(T=0), 1), (dict(maxlen=0), 1), (dict(Hkv=3), 1),
    (dict(d=256), 2), (dict(ws=None), 6), (dict(ws_bytes=16), 6), (dict(cu=DUMMY + 1), 3),
])
def test_varlen_backward_rejects_bad_arguments(fa, kw, code):
    a = dict(cu=DUMMY, dq=DUMMY, T=100, maxlen=64, Hkv=2, d=128, ws=DUMMY, ws_bytes=1 << 20)
    a.update(kw)
    assert fa.fa.fa_bwd_varlen(DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, a["dq"], DUMMY, DUMMY, a["cu"], 2, 4,
                               a["Hkv"], a["T"], a["maxlen"], a["d"], 1, 0.1, a["ws"], a["ws_bytes"],
                               None) == code


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), 1), (dict(codes=None), 1), (dict(BH=0), 1), (dict(N=0), 1), (dict(d=96), 2),
    (dict(block_rows=100), 1), (dict(block_rows=-128), 1), (dict(ws=None), 6), (dict(ws_bytes=8), 6),
    (dict(x=DUMMY + 8), 3), (dict(signs=DUMMY + 4), 3), (dict(descale=DUMMY + 2), 3),
])
def test_quantize_fp8_rejects_bad_arguments(fa, kw, code):
    a = dict(x=DUMMY, codes=DUMMY, descale=DUMMY, BH=2, N=300, d=128, block_rows=128, signs=None,
             ws=DUMMY, ws_bytes=1 << 20)
    a.update(kw)
    assert fa.fa_quantize_fp8(a["x"], a["codes"], a["descale"], a["BH"], a["N"], a["d"], a["block_rows"],
                              a["signs"], 0, a["ws"], a["ws_bytes"], None) == code


def test_quantize_fp8_workspace_size(fa):
    assert fa.fa_quantize_fp8_workspace_bytes(2, 300, 128) == 32  # 2 heads x 3 chunks x 4 B, to 16
    assert fa.fa_quantize_fp8_workspace_bytes(1, 128, 64) == 16
    assert fa.fa_quantize_fp8_workspace_bytes(1, 128, 96) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(q8=None), 1), (dict(vd=None), 1), (dict(N=0), 1), (dict(d=64), 2), (dict(d=256), 2),
    (dict(Hkv=3), 1), (dict(scale=0.0), 1), (dict(q8=DUMMY + 8), 3), (dict(vt8=DUMMY + 4), 3),
    (dict(qd=DUMMY + 2), 3), (dict(lse=DUMMY + 4), 3),
])
def test_fwd_fp8_rejects_bad_arguments(fa, kw, code):
    a = dict(q8=DUMMY, k8=DUMMY, vt8=DUMMY, qd=DUMMY, kd=DUMMY, vd=DUMMY, o=DUMMY, lse=DUMMY, B=1,
             H=4, Hkv=2, N=256, d=128, scale=0.1)
    a.update(kw)
    assert fa.fa_fwd_fp8(a["q8"], a["k8"], a["vt8"], a["qd"], a["kd"], a["vd"], a["o"], a["lse"], a["B"],
                         a["H"], a["Hkv"], a["N"], a["d"], 1, a["scale"], None) == code


def test_fwd_ws_rejects_bad_arguments_before_touching_a_device(fa):
    a = [DUMMY] * 5
    ok = (1, 2, 2, 1000, 128, 1, 0.088)
    assert fa.fa_fwd_ws(*a, *ok, -1, None, 0, None) == 1                   # negative chunk
    assert fa.fa_fwd_ws(None, *a[1:], *ok, 0, None, 0, None) == 1          # null q
    assert fa.fa_fwd_ws(*a, 1, 2, 2, 1000, 80, 1, 0.088, 0, None, 0, None) == 2  # head dim
    assert fa.fa_fwd_ws(*a, 1, 2, 3, 1000, 128, 1, 0.088, 0, None, 0, None) == 1  # Hkv
    assert fa.fa_fwd_ws(*a, 1, 2, 2, 1000, 128, 1, 0.0, 0, None, 0, None) == 1    # scale
    assert fa.fa_fwd_ws(DUMMY + 8, *a[1:], *ok, 0, None, 0, None) == 3     # misaligned q
    assert fa.fa_fwd_workspace_bytes(1, 2, 1000, 80, 1, 0) == 0
    assert fa.fa_fwd_workspace_bytes(1, 2, 1000, 128, 1, -5) == 0


def test_read_probe_rejects_bad_arguments_before_touching_a_device(fa):
    import ctypes
    g = ctypes.c_double(0.0)
    ok_ptr, mib = 0x100000, 1 << 20
    assert fa.fa_probe_read_bandwidth(None, mib, 1, None, g) == 1
    assert fa.fa_probe_read_bandwidth(ok_ptr + 8, mib, 1, None, g) == 1   # not 16-byte aligned
    assert fa.fa_probe_read_bandwidth(ok_ptr, mib - 16, 1, None, g) == 1  # under 1 MiB
    assert fa.fa_probe_read_bandwidth(ok_ptr, mib + 8, 1, None, g) == 1   # not a multiple of 16
    assert fa.fa_probe_read_bandwidth(ok_ptr, mib, 0, None, g) == 1
    assert fa.fa_probe_read_bandwidth(ok_ptr, mib, 1001, None, g) == 1


def test_probe_rejects_bad_arguments_before_touching_a_device(fa):
    import ctypes
    rates = (ctypes.c_double * 3)()
    assert fa.fa_probe_unit_rates(rates, 15, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_probe_unit_rates(rates, (1 << 20) + 1, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_probe_unit_rates(None, 2048, None) == fa.FA_ERR_INVALID_ARG
