"""fa_naive_fwd (standard attention with S and P through HBM, the baseline of "LLM Architecture
Refresh [3]", section 1) against the fp64 oracle, with the forward tolerances of gpu_util."""

import math

import pytest

import oracle
from gpu_util import assert_fwd_close, fa_mod
from online_softmax_09_gb300.inputs import make_qkv, to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N", [1, 7, 300, 1024])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_naive_matches_oracle(N, causal, d):
    fa = fa_mod()
    q, k, v, _ = make_qkv(2, 4, 2, N, d, seed=6000 + N + d)
    o, lse = fa.forward_naive(q.cuda(), k.cuda(), v.cuda(), causal)
    fa.check()
    O_ref, L_ref = oracle.attention_forward(to_f64(q), to_f64(k), to_f64(v), causal, 1 / math.sqrt(d))
    assert_fwd_close(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref, f"N={N}")
