"""Failure detection on the GPU without a fault: the bounded mbarrier wait the
GEMV kernels use is run against a barrier that nothing completes.  It must
give up after its limit (about 2 s), report it through a status word, and
leave the context usable: a GEMV launched afterwards gives the right result."""
import numpy as np
import pytest

import oracle
from int4_weight_only_w4_gb300 import synthetic as syn
from tests import w4_testutil as tu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def w4():
    from int4_weight_only_w4_gb300 import w4 as mod
    return mod


def test_bounded_wait_gives_up_and_context_stays_usable(w4):
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    w4.selftest_bounded_wait(status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    M, K, N = 2, 1024, 96
    p = syn.make_problem("after.wait", K, N, M, seed=31)
    qw, sc, zp, x = tu.to_device(p)
    y = w4.pack(qw, sc, zp, K, N).gemv_f32(x).cpu().numpy()
    ref = oracle.gemv_f64(p.qweight, p.scales, p.zeros, p.x, M, K, N)
    assert np.linalg.norm(y - ref) <= 1e-3 * np.linalg.norm(ref)
