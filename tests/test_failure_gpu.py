"""Failure detection on the GPU without a fault: a bounded pipeline wait that can never complete
times out, is reported by fa_sync_status, is cleared, and the context keeps computing correctly."""
import pytest
import torch

import exact_io_aware_08_gb300 as fa
from exact_io_aware_08_gb300 import inputs
from oracle import attention as A
from tests.gpu_common import assert_lse_close, assert_o_close, cuda, require_gpu

pytestmark = pytest.mark.gpu

TIMEOUT = 5


def test_unsatisfiable_wait_is_reported_and_context_survives():
    require_gpu()
    fa.fa_sync_status()                          # start from a clean status word
    fa.fa_selftest_wait_timeout(50_000)          # 50 ms bounded wait nobody satisfies
    with pytest.raises(fa.FaError) as e:
        fa.fa_sync_status()
    assert e.value.status == TIMEOUT
    assert "site 900" in str(e.value)
    fa.fa_sync_status()                          # reported once, then cleared
    # the context is intact: a normal forward still matches the oracle
    x = inputs.make_qkv(1, 2, 200, 200, 128, seed=5, with_do=False)
    o, lse = fa.forward(cuda(x["q"]), cuda(x["k"]), cuda(x["v"]), causal=True)
    fa.fa_sync_status()
    o_ref, lse_ref = A.forward(x["q"], x["k"], x["v"], 128 ** -0.5, True)
    assert_o_close(o, o_ref)
    assert_lse_close(lse, lse_ref)


def test_timeout_on_a_side_stream_is_seen_by_sync_status_of_that_stream():
    require_gpu()
    s = torch.cuda.Stream()
    fa.fa_selftest_wait_timeout(20_000, stream=s)
    with pytest.raises(fa.FaError) as e:
        fa.fa_sync_status(stream=s)
    assert e.value.status == TIMEOUT
    fa.fa_sync_status(stream=s)
