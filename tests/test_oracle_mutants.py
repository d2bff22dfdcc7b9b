"""Plant plausible mistakes in copies of the oracle and check that the pins catch them.

Each mutant replaces one exact snippet of ``oracle/oracle.c`` (a dropped term, a
wrong sign, an off-by-one mask, a transposed operand, a wrong log base), compiles
the copy with the oracle's own build script into a temporary directory, and runs
the pin battery on it.  A mutant that passes every pin would mean the pins leave
that part of the oracle unchecked.  Nothing here touches a GPU.
"""
import os

import pytest

import oracle_pins as pins
from oracle import Oracle
from oracle import build as obuild

MUTANTS = {
    "dropped_scale": ("s[j] = scale * acc;", "s[j] = acc;"),
    "mask_excludes_diagonal": ("return causal ? i + 1 : N;", "return causal ? (i > 0 ? i : 1) : N;"),
    "mask_one_past_diagonal": ("return causal ? i + 1 : N;", "return causal ? (i + 2 < N ? i + 2 : N) : N;"),
    "exp_sign_flipped": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "no_max_subtraction": ("s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
    "lse_log2": ("*lse_i = m + log(l);", "*lse_i = m + log2(l);"),
    "lse_missing_max": ("*lse_i = m + log(l);", "*lse_i = log(l);"),
    "no_normalisation": ("double p = s[j] / l;", "double p = s[j];"),
    "scores_transposed": ("double m = score_row(Q + i * d, K, n, d, scale, s, &l);",
                          "double m = score_row(K + i * d, Q, n, d, scale, s, &l);"),
    "bwd_ds_sign": ("double ds = s[j] * (dp[j] - Di);", "double ds = s[j] * (dp[j] + Di);"),
    "bwd_ds_missing_D": ("double ds = s[j] * (dp[j] - Di);", "double ds = s[j] * dp[j];"),
    "bwd_D_missing_P": ("Di += s[j] * dp[j];", "Di += dp[j];"),
    "bwd_dk_missing_scale": ("dkj[c] += jb->scale * ds * qi[c];", "dkj[c] += ds * qi[c];"),
    "bwd_dq_uses_q": ("dqi[c] += jb->scale * ds * kj[c];", "dqi[c] += jb->scale * ds * qi[c];"),
    "bwd_dv_uses_dp": ("dvj[c] += s[j] * doi[c];", "dvj[c] += dp[j] * doi[c];"),
    "bwd_p_unnormalised": ("s[j] = s[j] / l; /* P_ij */", "s[j] = s[j]; /* P_ij */"),
    "decode_kv_head_stride": ("size_t kv = (size_t)bh * (size_t)jb->N * (size_t)jb->d;",
                              "size_t kv = (size_t)bh * (size_t)jb->Nq * (size_t)jb->d;"),
    "decode_first_row_only": ("long bh = t / jb->Nq, i = t % jb->Nq;",
                              "long bh = t / jb->Nq, i = 0;"),
}

_FAST = {"check_blockwise_equivalence": lambda orc: pins.check_blockwise_equivalence(orc, big=False)}


def _caught(orc):
    failures = []
    for check in pins.ALL_CHECKS:
        fn = _FAST.get(check.__name__, check)
        try:
            fn(orc)
        except AssertionError as e:
            failures.append(f"{check.__name__}: {e}")
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    with open(obuild.SRC) as f:
        src = f.read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"snippet for {name} no longer matches oracle.c exactly once"
    path = tmp_path / "oracle_mutant.c"
    path.write_text(src.replace(old, new))
    lib = obuild.build(out=os.path.join(tmp_path, "libmutant.so"), src=str(path))
    failures = _caught(Oracle(lib))
    assert failures, f"mutant {name} passed every pin"
