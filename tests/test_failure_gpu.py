"""Failure detection on the GPU, with no fault: a bounded device wait on an
mbarrier that nothing completes runs out within its short limit, the kernel
sets MOE_DEVERR_TIMEOUT and returns, and the context stays usable (a decode
afterwards still matches the oracle).  Both forms of wait the kernels use are
driven to expiry: the sleeping polls of the decode kernels and the
device-time spin of the grouped and prompt-path kernels."""
import time

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle import formats as F  # noqa: E402
from quantized_routed_expert_route_gb300 import capi  # noqa: E402
from tests import cases  # noqa: E402
from tests import tolerance as tol  # noqa: E402


@pytest.mark.parametrize("mode,limit", [(0, 4), (0, 1), (1, 50), (1, 1)])
def test_bounded_wait_runs_out_and_reports(mode, limit):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    capi.moe_debug_wait_timeout(mode, limit, err.data_ptr(), stream)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(err.item()) == capi.MOE_DEVERR_TIMEOUT
    assert elapsed < 5.0, elapsed
    # the context is still usable: the tiny Q8_0 layer decodes within its bounds
    case = cases.make_case(256, 128, 8, 2, F.TYPE_Q8_0, F.TYPE_Q8_0, 1, seed=0, device="cuda:0")
    res = cases.run_gpu(case)
    ref, _, st = cases.oracle(case)
    beta, _, _ = tol.output_bounds(case.geom, st)
    tol.check_output(res["out"], ref, beta)
    assert res["err"] == 0
    assert np.isfinite(F.bf16_bits_to_f64(res["out"])).all()
