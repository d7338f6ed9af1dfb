"""Failure detection without a GPU fault.

Every kernel of the library bounds its waits in time; a wait that runs out
records LDN_ERR_TIMEOUT in the device status word and the kernel returns
normally.  The GPU test makes such a wait run out on purpose (an mbarrier
that nothing arrives on, a 5 ms bound; the waiting kernel is in the test-only
diagnostic library, which has its own status word) and checks the status and
that the context, and the product library, are still usable afterwards.  Argument errors are covered on the CPU
(tests/test_abi_cpu.py)."""
import pytest

import gated_delta_rule_chunkwise_gb300 as ldn
from tests import _diag

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_delta_rule_chunkwise_gb300 import build
    build.build()
    ldn.load()


def test_bounded_wait_reports_timeout_and_context_survives():
    import torch
    from gated_delta_rule_chunkwise_gb300 import workloads as wl
    assert ldn.device_status() == ldn.LDN_OK              # clean slate
    assert _diag.status() == ldn.LDN_OK
    flag = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    st = _diag.load().ldn_diag_wait_timeout(5_000_000, flag.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == ldn.LDN_OK
    assert _diag.status() == ldn.LDN_ERR_TIMEOUT          # recorded ...
    assert int(flag.item()) == 0
    assert _diag.status() == ldn.LDN_OK                   # ... and cleared by the read
    # the context is intact: a real call still runs and reports ok
    w = wl.make_chunk("gdn_bf16_b4_t2048_h16_d128", B=1, T=70, H=1)
    t = w.torch_inputs("cuda")
    out, sf = ldn.chunk_fwd(t["q"], t["k"], t["v"], t["beta"], t["gate"], None, mode="gdn")
    assert ldn.device_status() == ldn.LDN_OK
    assert bool(torch.isfinite(out.float()).all())


def test_timeout_argument_validation():
    d = _diag.load()
    assert d.ldn_diag_wait_timeout(-1, 1 << 20, None) == ldn.LDN_ERR_INVALID_ARG
    assert d.ldn_diag_wait_timeout(3_000_000_000, 1 << 20, None) == ldn.LDN_ERR_INVALID_ARG
    assert d.ldn_diag_wait_timeout(1000, None, None) == ldn.LDN_ERR_INVALID_ARG
