"""Failure detection on the GPU without a fault: the bounded device wait the attention
kernel uses runs out on a barrier that nothing completes, records BSA_ERR_DEVICE_TIMEOUT
in the caller's status word and returns; the CTAs that wait with the library's 4 s limit
stop as soon as they see that status.  The context stays usable afterwards."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_long_kv_gb300 import build
    build.build()


def test_wait_runs_out_and_reports():
    import block_sparse_long_kv_gb300 as bsa
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    bsa.selftest_wait_timeout(st, 20_000_000, ctas=4)   # CTA 0 gives up after 20 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) == 6 and bsa.status_string(6) == "BSA_ERR_DEVICE_TIMEOUT"
    # the three CTAs with the 4 s limit stopped on seeing the status, long before their own limit
    assert dt < 1.0, dt


def test_context_usable_after_timeout():
    import block_sparse_long_kv_gb300 as bsa
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsa.selftest_wait_timeout(st, 5_000_000, ctas=1)
    torch.cuda.synchronize()
    assert int(st.item()) == 6
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 1023 * 1024 / 2
