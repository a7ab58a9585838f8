"""w4_gemv_ws_static -- the GEMV entry point that allocates nothing and keeps
its scratch in a static device array -- called through the C ABI and checked
against the existing entry points on the same inputs, over consecutive calls
that share that array.  Collected last on purpose (file name)."""
import ctypes

import numpy as np
import pytest

from int4_weight_only_w4_gb300 import synthetic as syn
from tests import w4_testutil as tu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def w4():
    from int4_weight_only_w4_gb300 import w4 as mod
    return mod


def _static_call(w4, packed, x, y, M):
    lib = ctypes.CDLL(w4.library_path())
    fn = lib.w4_gemv_ws_static
    fn.restype = ctypes.c_int
    P = ctypes.c_void_p
    fn.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
    stream = torch.cuda.current_stream().cuda_stream
    return fn(packed.qweight.data_ptr(), packed.scales.data_ptr(), packed.zeros.data_ptr(),
              x.data_ptr(), y.data_ptr(), M, packed.K, packed.N, stream)


def _problem(w4, name, K, N, M, seed):
    p = syn.make_problem(name, K, N, M, seed=seed)
    qw, sc, zp, x = tu.to_device(p)
    return w4.pack(qw, sc, zp, K, N), x


def _close(got, want):
    """The GEMV tolerances of the parity tests, output against output."""
    g = got.float().cpu().numpy().astype(np.float64)
    w = want.float().cpu().numpy().astype(np.float64)
    nw = np.linalg.norm(w)
    assert np.linalg.norm(g - w) <= tu.REL_L2 * nw
    assert np.abs(g - w).max() <= tu.MAX_ABS_FRAC * np.abs(w).max()


def test_static_scratch_matches_existing_entry_points(w4):
    # Two different products back to back (different row-block counts, so the
    # second call meets the first call's leftovers in the shared array), then
    # the first one again.
    cases = [("nz.a", 17408, 5120, 2, 1), ("nz.b", 3584, 4608, 1, 2)]
    probs = [_problem(w4, n, K, N, M, sd) for (n, K, N, M, sd) in cases]
    outs = []
    for (name, K, N, M, _), (packed, x) in zip(cases + cases[:1], probs + probs[:1]):
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        assert _static_call(w4, packed, x, y, M) == 0
        torch.cuda.synchronize()
        ws = w4.workspace(K, N)
        y_ws = packed.gemv(x, workspace=ws)
        y_cl = packed.gemv(x)
        torch.cuda.synchronize()
        # same kernel and split as w4_gemv_ws: identical bits
        assert torch.equal(y.view(torch.int16), y_ws.view(torch.int16)), name
        # against w4_gemv within the parity tolerance
        _close(y, y_cl)
        outs.append(y.clone())
    assert torch.equal(outs[0].view(torch.int16), outs[2].view(torch.int16))


def test_static_scratch_limit_refused_first(w4):
    # Enough rows that the row-block counters alone (4 bytes per 128 rows)
    # exceed the array, whatever the SM count; the size check runs before the
    # pointer checks, so NULL pointers never launch.
    rows = 128 * (w4.STATIC_SCRATCH_BYTES // 4 + 1)
    need = w4.gemv_workspace_bytes(128, rows)
    assert need > w4.STATIC_SCRATCH_BYTES
    lib = ctypes.CDLL(w4.library_path())
    fn = lib.w4_gemv_ws_static
    fn.restype = ctypes.c_int
    P = ctypes.c_void_p
    fn.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
    assert fn(None, None, None, None, None, 1, 128, rows, None) == w4.Status.SCRATCH_LIMIT
    # a product that fits, with a NULL pointer: refused as an argument error
    assert fn(None, None, None, None, None, 1, 3584, 3584, None) == w4.Status.INVALID_ARG
