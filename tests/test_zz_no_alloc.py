"""moe_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (plugins whose host framework owns every device allocation,
serving paths where a cudaMalloc may synchronize the device).  It runs on the library's
fixed device workspace; this checks, through the C ABI, that two calls in a
row give the same outputs as moe_decode with a caller workspace, within the
layer tolerance the other tests use.  This file is collected last so that a
failure here comes after every other test has run."""
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


def _close(a_bits, b_bits):
    a = F.bf16_bits_to_f64(a_bits)
    b = F.bf16_bits_to_f64(b_bits)
    scale = max(np.abs(b).max(), 1e-30)
    max_rel = np.abs(a - b).max() / scale
    rel_l2 = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    assert max_rel <= 2e-3 and rel_l2 <= 5e-4, (max_rel, rel_l2)


def test_noalloc_matches_moe_decode_on_two_calls():
    case = cases.make_case(2048, 768, 128, 8, F.TYPE_NVFP4, F.TYPE_NVFP4, 8, seed=200)
    g = case.geom
    layer = MoeLayer(g.H, g.I, g.E, g.top_k, g.gate_up_type, g.down_type, case.gu_dev, case.dn_dev,
                     torch.from_numpy(case.sb).cuda(), borrow=True)
    stream = torch.cuda.current_stream().cuda_stream
    for call, T in enumerate((1, 8)):
        x = torch.from_numpy(S.hidden_bf16(300 + call, T, g.H).view(np.int16)).cuda()
        ids_np, w_np = S.softmax_topk_routing(400 + call, T, g.E, g.top_k)
        ids = torch.from_numpy(ids_np).cuda()
        w = torch.from_numpy(w_np).cuda()
        ref = torch.empty((T, g.H), dtype=torch.int16, device="cuda")
        got = torch.full((T, g.H), -1, dtype=torch.int16, device="cuda")
        capi.moe_decode(layer.bank, x.data_ptr(), T, ids.data_ptr(), w.data_ptr(), ref.data_ptr(),
                        layer.ws.data_ptr(), layer.ws_bytes, stream)
        capi.moe_decode_noalloc(layer.bank, x.data_ptr(), T, ids.data_ptr(), w.data_ptr(), got.data_ptr(), stream)
        torch.cuda.synchronize()
        _close(got.cpu().numpy().view(np.uint16), ref.cpu().numpy().view(np.uint16))
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
