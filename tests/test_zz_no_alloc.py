"""moe_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (plugins whose host framework owns every device allocation,
serving paths where a cudaMalloc may synchronize the device).  It runs on the
library's fixed device workspace.  Through the C ABI this checks, on calls in
a row, that its outputs equal those of moe_decode with a caller workspace bit
for bit (the same kernels on the same inputs), including the grouped Q4_K
path whose tensor maps point into the fixed workspace; that one call is
within the oracle's derived bounds; and that moe_get_error with no workspace
reads the fixed workspace's error word.  This file is collected last so that
a failure here comes after every other test has run."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle import formats as F  # noqa: E402
from quantized_routed_expert_route_gb300 import capi  # noqa: E402
from quantized_routed_expert_route_gb300.layer import MoeLayer  # noqa: E402
from synth import banks as S  # noqa: E402
from tests import cases  # noqa: E402
from tests import tolerance as tol  # noqa: E402


def _layer(case):
    g = case.geom
    return MoeLayer(g.H, g.I, g.E, g.top_k, g.gate_up_type, g.down_type, case.gu_dev, case.dn_dev,
                    torch.from_numpy(case.sb).cuda(), borrow=True)


def _both(layer, x, ids, w, T, H, stream):
    ref = torch.empty((T, H), dtype=torch.int16, device="cuda")
    got = torch.full((T, H), -1, dtype=torch.int16, device="cuda")
    capi.moe_decode(layer.bank, x.data_ptr(), T, ids.data_ptr(), w.data_ptr(), ref.data_ptr(),
                    layer.ws.data_ptr(), layer.ws_bytes, stream)
    capi.moe_decode_noalloc(layer.bank, x.data_ptr(), T, ids.data_ptr(), w.data_ptr(), got.data_ptr(), stream)
    torch.cuda.synchronize()
    return got.cpu().numpy().view(np.uint16), ref.cpu().numpy().view(np.uint16)


def _no_device_error(stream):
    bits = capi.ctypes.c_int32(-1)
    st = capi.library().moe_get_error(None, 0, stream, capi.ctypes.byref(bits))
    assert st == capi.MOE_OK and bits.value == 0, (st, bits.value)


def test_noalloc_matches_moe_decode_on_calls_in_a_row():
    stream = torch.cuda.current_stream().cuda_stream
    # the Qwen3-30B-A3B-shaped NVFP4 layer: the fused kernel at T=1, the batched path at T=8
    case = cases.make_case(2048, 768, 128, 8, F.TYPE_NVFP4, F.TYPE_NVFP4, 1, seed=200)
    g = case.geom
    layer = _layer(case)
    for call, T in enumerate((1, 8)):
        assert capi.moe_workspace_bytes(layer.bank, T) <= capi.MOE_NOALLOC_WS_BYTES
        x = torch.from_numpy(S.hidden_bf16(300 + call, T, g.H).view(np.int16)).cuda()
        ids_np, w_np = S.softmax_topk_routing(400 + call, T, g.E, g.top_k)
        got, ref = _both(layer, x, torch.from_numpy(ids_np).cuda(), torch.from_numpy(w_np).cuda(), T, g.H, stream)
        assert np.array_equal(got, ref), f"call {call} (T={T}): outputs differ from moe_decode"
        _no_device_error(stream)
    # one call against the oracle: the case's own inputs (its routed experts hold converted rows)
    x = torch.from_numpy(case.x.view(np.int16)).cuda()
    got, ref = _both(layer, x, torch.from_numpy(case.ids).cuda(), torch.from_numpy(case.w).cuda(), 1, g.H, stream)
    assert np.array_equal(got, ref)
    want, _, st = cases.oracle(case)
    beta, _, _ = tol.output_bounds(g, st)
    tol.check_output(got, want, beta)
    layer.close()
    # the Laguna-shaped Q4_K layer at T=16: the grouped path, whose tensor maps
    # are encoded over the fixed workspace's device address
    case = cases.make_case(4096, 768, 256, 10, F.TYPE_Q4_K, F.TYPE_Q4_K, 16, seed=210, routing="zipf")
    g = case.geom
    layer = _layer(case)
    assert capi.moe_decode_kernel_count(layer.bank, 16) == 4
    assert capi.moe_workspace_bytes(layer.bank, 16) <= capi.MOE_NOALLOC_WS_BYTES
    x = torch.from_numpy(case.x.view(np.int16)).cuda()
    ids, w = torch.from_numpy(case.ids).cuda(), torch.from_numpy(case.w).cuda()
    for call in range(2):
        got, ref = _both(layer, x, ids, w, 16, g.H, stream)
        assert np.array_equal(got, ref), f"Laguna Q4_K call {call}: outputs differ from moe_decode"
    _no_device_error(stream)
    layer.close()


def test_noalloc_rejects_a_batch_beyond_its_workspace():
    # 32 experts, top-32, H = I = 2048 Q8_0 rows: one pass of 64 tokens holds
    # thousands of routes' intermediates, far more than the fixed workspace
    H = I = 2048
    E = K = 32
    rb = capi.moe_row_bytes(capi.MOE_Q8_0, H)
    g = capi.moe_layer_geom(H, I, E, K, capi.MOE_Q8_0, capi.MOE_Q8_0)
    gu = torch.zeros(E * 2 * I * rb + 16, dtype=torch.uint8, device="cuda")
    dn = torch.zeros(E * H * rb + 16, dtype=torch.uint8, device="cuda")
    bank = capi.moe_bank_create(g, gu.data_ptr(), E * 2 * I * rb, dn.data_ptr(), E * H * rb, 0,
                                capi.MOE_SRC_DEVICE_BORROW, 0)
    T = 64
    assert capi.moe_workspace_bytes(bank, T) > capi.MOE_NOALLOC_WS_BYTES
    x = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    ids = torch.arange(K, dtype=torch.int32, device="cuda").repeat(T, 1).contiguous()
    w = torch.ones((T, K), dtype=torch.float32, device="cuda")
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    st = capi.library().moe_decode_noalloc(bank, x.data_ptr(), T, ids.data_ptr(), w.data_ptr(), out.data_ptr(),
                                           None)
    assert st == capi.MOE_EINVAL
    assert "static workspace" in capi.library().moe_last_cuda_error().decode()
    capi.moe_bank_destroy(bank)
