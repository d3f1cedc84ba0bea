"""Failure detection on the GPU without a fault: a pipeline wait that can never complete gives
up after its bounded limit, the kernel returns, the host reads the timeout from the device
status word, and the same context keeps computing correct results."""

import math
import time

import pytest

import oracle
from gpu_util import assert_fwd_close, fa_mod
from online_softmax_09_gb300.inputs import make_qkv, to_f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_context_stays_usable():
    fa = fa_mod()
    fa.check()  # start from a clean status word
    t0 = time.monotonic()
    result = fa.selftest_wait_timeout()
    waited = time.monotonic() - t0
    assert result == 2  # the wait gave up and raised its abort flag
    assert 1.5 < waited < 30.0, waited  # the 2 s limit, not a hang
    with pytest.raises(fa.FAError) as err:
        fa.check()
    assert err.value.status == -5  # FA_ERR_TIMEOUT
    fa.check()  # reading the status cleared it
    q, k, v, _ = make_qkv(1, 2, 1, 300, 64, seed=71)
    o, lse = fa.forward(q.cuda(), k.cuda(), v.cuda(), True)
    fa.check()
    O_ref, L_ref = oracle.attention_forward(to_f64(q), to_f64(k), to_f64(v), True, 1 / math.sqrt(64))
    assert_fwd_close(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref, "after a timeout")
