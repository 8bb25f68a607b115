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


def test_fa_log_writes_one_line_per_launch():
    """FA_LOG=1 makes every launch print its kernel and launch shape to stderr (host side)."""
    import os
    import subprocess
    import sys
    require_gpu()
    code = ("import torch, exact_io_aware_08_gb300 as fa\n"
            "q = torch.randn(1, 2, 300, 64, device='cuda').to(torch.bfloat16)\n"
            "o, lse = fa.forward(q, q, q, causal=True)\n"
            "torch.cuda.synchronize()\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       env={**os.environ, "FA_LOG": "1"}, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stderr.splitlines() if l.startswith("[fa] launch ")]
    assert len(lines) == 1 and "grid=" in lines[0] and "smem=" in lines[0], r.stderr[-2000:]
    r0 = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                        env={k: v for k, v in os.environ.items() if k != "FA_LOG"}, timeout=300)
    assert r0.returncode == 0 and "[fa] launch" not in r0.stderr
