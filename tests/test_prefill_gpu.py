"""GPU checks of the prompt path's tensor-core machinery, through the C ABI.

The tcgen05 kind::f16 MMA on swizzled shared-memory tiles is checked against
a float64 matmul of the same fp16 operands: every product of two fp16 values
is exact in fp32, so the only error is the fp32 accumulation, bounded by
K * 2^-24 * sum|a*b| per element."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from quantized_routed_expert_route_gb300 import capi  # noqa: E402

DEV = "cuda"


@pytest.mark.parametrize("K,N", [(64, 16), (256, 256), (2048, 128), (768, 240)])
def test_tc_gemm_matches_f64(K, N):
    r = np.random.default_rng(K + N)
    a = r.standard_normal((128, K)).astype(np.float16)
    b = r.standard_normal((N, K)).astype(np.float16)
    ad = torch.from_numpy(a.view(np.int16)).to(DEV)
    bd = torch.from_numpy(b.view(np.int16)).to(DEV)
    d = torch.full((128, N), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    capi.moe_debug_tc_gemm(ad.data_ptr(), bd.data_ptr(), K, N, d.data_ptr(), err.data_ptr(),
                           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = d.cpu().numpy().astype(np.float64)
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    want = a64 @ b64.T
    bound = K * 2.0 ** -24 * (np.abs(a64) @ np.abs(b64).T) + 1e-30
    assert np.isfinite(got).all()
    assert (np.abs(got - want) <= bound).all(), float(np.max(np.abs(got - want) / bound))
