"""Forward with cut key ranges (fa_fwd_ws): the key range of each 128-row block is
split over several CTAs and the partial (O, L) merged by the log-sum-exp rule.

Small ragged shapes with forced chunk sizes cover every head dimension, both masks,
grouped-query heads, row blocks with one chunk next to row blocks with several, and
last chunks shorter than the rest; the batch-1 single-head long causal workload the
split exists for runs with the library's own choice and is checked on sampled rows
against the float64 oracle; the merged result agrees with the uncut kernel."""
import numpy as np
import pytest
import torch

from exact_attention_26_gb300.inputs import gqa_qkv, normal_qkv, sample_rows, to_f64
from gpu_common import L_ABS, assert_abs_close, assert_o_close, load_fa
from oracle import Oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def fa():
    return load_fa()


@pytest.fixture(scope="module")
def orc():
    return Oracle()


# (B, H, Hkv, N, d, kv_chunk in keys)
FORCED = [
    (1, 2, 2, 1000, 128, 256), (1, 1, 1, 777, 64, 128), (1, 2, 2, 700, 256, 128),
    (1, 1, 1, 1000, 96, 384), (1, 4, 2, 600, 128, 128), (2, 1, 1, 129, 128, 128),
    (1, 1, 1, 2048, 128, 640),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", FORCED, ids=lambda c: "x".join(map(str, c)))
def test_forced_chunks_match_the_oracle(fa, orc, case, causal):
    B, H, Hkv, N, d, chunk = case
    if Hkv == H:
        q, k, v = normal_qkv(B, H, N, d, seed=N + d + chunk)
    else:
        q, k, v = gqa_qkv(B, H, Hkv, N, d, seed=N + d)
    need = fa.fa_fwd_workspace_bytes(B, H, N, d, causal, chunk)
    assert need > 0, "a forced chunk shorter than the key range cuts it"
    o, lse = fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, kv_chunk=chunk)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    kr, vr = to_f64(k), to_f64(v)
    if Hkv != H:  # the oracle takes one key/value head per query head
        kr, vr = (np.repeat(x, H // Hkv, axis=1) for x in (kr, vr))
    ro, rl = orc.fwd(to_f64(q), kr, vr, causal=causal)
    assert_o_close(o.float().cpu().numpy(), ro, f"{case} causal={causal}")
    assert_abs_close(lse.cpu().numpy(), rl, L_ABS, f"{case} causal={causal} L")


def test_single_head_long_causal_workload(fa, orc):
    """B1 H1 N16384 d128 causal, the library's own choice (which cuts: one tile per
    CTA leaves the longest rows waiting); 256 seeded rows checked against the oracle."""
    B, H, N, d = 1, 1, 16384, 128
    assert fa.fa_fwd_workspace_bytes(B, H, N, d, True, 0) > 0
    q, k, v = normal_qkv(B, H, N, d, seed=0)
    o, lse = fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    rows = sample_rows(N, 256, seed=2).numpy()
    ro, rl = orc.fwd_rows(to_f64(q), to_f64(k), to_f64(v), rows, causal=True)
    assert_o_close(o.float().cpu().numpy()[:, :, rows], ro, "B1H1N16384 sample")
    assert_abs_close(lse.cpu().numpy()[:, :, rows], rl, L_ABS, "B1H1N16384 sample L")


# shapes the library cuts with its balanced plan (kv_chunk = 0): every head
# dimension, both masks, one and two heads, ragged N
AUTO = [(1, 2, 6000, 128, True), (1, 1, 8192, 64, True), (1, 2, 3000, 256, False),
        (1, 1, 8192, 96, False)]


@pytest.mark.parametrize("case", AUTO, ids=lambda c: "x".join(map(str, c)))
def test_balanced_cut_matches_the_oracle(fa, orc, case):
    B, H, N, d, causal = case
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    segs = fa.fwd_split_segments(B, H, N, d, causal, sms)
    assert segs and max(s[5] for s in segs) >= 2, "the library cuts this shape"
    q, k, v = normal_qkv(B, H, N, d, seed=N + d)
    o, lse = fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    # rows of every cut row block's first and last 128, plus seeded ones
    cut = sorted({s[1] for s in segs if s[5] >= 2})
    rows = np.unique(np.concatenate([sample_rows(N, 128, seed=3).numpy(),
                                     [cut[0] * 128, min(N, cut[-1] * 128 + 128) - 1, N - 1]]))
    ro, rl = orc.fwd_rows(to_f64(q), to_f64(k), to_f64(v), rows, causal=causal)
    assert_o_close(o.float().cpu().numpy()[:, :, rows], ro, f"{case}")
    assert_abs_close(lse.cpu().numpy()[:, :, rows], rl, L_ABS, f"{case} L")


def test_cut_and_uncut_agree(fa):
    """The same inputs through fa_fwd and through cut key ranges: O within the bf16
    rounding of either, L within fp32 rounding of the merge."""
    B, H, N, d = 1, 2, 3000, 128
    q, k, v = (t.to(DEV) for t in normal_qkv(B, H, N, d, seed=5))
    for causal in (False, True):
        o0 = torch.empty_like(q)
        l0 = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
        assert fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o0.data_ptr(), l0.data_ptr(),
                         B, H, N, d, causal, 1.0 / np.sqrt(d), None) == 0
        o1, l1 = fa.forward(q, k, v, causal=causal, kv_chunk=512)
        torch.cuda.synchronize()
        assert float((o1.float() - o0.float()).abs().max()) <= 2.0 ** -7 * max(
            1.0, float(o0.float().abs().max()))
        assert float((l1 - l0).abs().max()) <= 1e-4


def test_workspace_is_checked(fa):
    B, H, N, d = 1, 1, 1000, 128
    q, k, v = (t.to(DEV) for t in normal_qkv(B, H, N, d, seed=1))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    need = fa.fa_fwd_workspace_bytes(B, H, N, d, True, 256)
    ws = torch.empty(need + 512, dtype=torch.uint8, device=DEV)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, H, N,
            d, True, 1.0 / np.sqrt(d), 256)
    assert fa.fa_fwd_ws(*args, None, 0, None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_ws(*args, ws.data_ptr(), need - 1, None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_fwd_ws(*args, ws.data_ptr() + 16, need, None) == fa.FA_ERR_MISALIGNED
    assert fa.fa_fwd_ws(*args, ws.data_ptr(), need, None) == 0
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
