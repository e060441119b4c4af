"""GPU parity of the dense path: BF16 gate_up and down banks at batches the
fused small-batch kernel cannot hold, decoded by the tensor-core grouped
GEMMs (four launches per pass).  Same bounds as the other decode tests
(tests/tolerance.py); each case first asserts that the dense path is the
one that ran (its launch count)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle import formats as F  # noqa: E402
from quantized_routed_expert_route_gb300 import capi  # noqa: E402
from tests import cases  # noqa: E402
from tests.test_decode_gpu import _check_case  # noqa: E402

DENSE_LAUNCHES = 4
BF = F.TYPE_BF16


@pytest.mark.parametrize("T", [16, 64])
def test_laguna_bf16_zipf_batches(T):
    """H=4096 I=768 E=256 top-10, Zipf(1.1) routing: the BF16 layers of the
    47-layer stack at T=16 and T=64; the oracle checks a sample of tokens."""
    case = cases.make_case(4096, 768, 256, 10, BF, BF, T, seed=200 + T, routing="zipf")
    figs = _check_case(case, tokens=[0, 1, T - 1])
    assert figs["launches"] == DENSE_LAUNCHES
    assert figs["err_bits"] == 0


def test_ragged_tiles_every_token():
    """I = 320 (the last 128-row block of gate_up half full), 40 tokens over 24
    experts (token blocks of 1..16 columns), every token checked, with the
    stage exports (fp32 intermediate)."""
    case = cases.make_case(2048, 320, 24, 5, BF, BF, 40, seed=210)
    figs = _check_case(case)
    assert figs["launches"] == DENSE_LAUNCHES
    assert figs["err_bits"] == 0


def test_one_expert_over_two_token_blocks():
    """Every route on one expert (duplicates inside each token): 256 routed
    rows, two 128-token blocks per weight tile."""
    T, K = 64, 4
    ids = [[3] * K for _ in range(T)]
    case = cases.make_case(2048, 256, 8, K, BF, BF, T, seed=220, ids=ids)
    figs = _check_case(case, tokens=[0, 31, 32, 63])
    assert figs["launches"] == DENSE_LAUNCHES
    assert figs["err_bits"] == 0


def test_bad_ids_flag_and_contribute_zero():
    T, K = 48, 3
    r = np.random.default_rng(5)
    ids = r.integers(0, 16, size=(T, K)).astype(np.int32)
    ids[0, 1] = 99
    ids[7, 0] = -1
    ids[47, 2] = 16
    case = cases.make_case(2048, 256, 16, K, BF, BF, T, seed=230, ids=ids)
    figs = _check_case(case, tokens=[0, 7, 20, 47])
    assert figs["launches"] == DENSE_LAUNCHES
    assert figs["err_bits"] & capi.MOE_DEVERR_BAD_ID


def test_dense_graph_replay_equals_eager():
    case = cases.make_case(4096, 768, 64, 8, BF, BF, 32, seed=240)
    from quantized_routed_expert_route_gb300.layer import MoeLayer
    g = case.geom
    layer = MoeLayer(g.H, g.I, g.E, g.top_k, g.gate_up_type, g.down_type, case.gu_dev, case.dn_dev,
                     torch.from_numpy(case.sb).to("cuda"), borrow=True)
    assert capi.moe_decode_kernel_count(layer.bank, 32) == DENSE_LAUNCHES
    x = torch.from_numpy(case.x.view(np.int16)).to("cuda").view(torch.bfloat16)
    ids = torch.from_numpy(case.ids).to("cuda")
    w = torch.from_numpy(case.w).to("cuda")
    eager1 = layer.decode(x, ids, w).clone()
    eager2 = layer.decode(x, ids, w).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    out = torch.empty_like(eager1)
    with torch.cuda.stream(s):
        layer.decode(x, ids, w, out)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            layer.decode(x, ids, w, out)
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager1.view(torch.int16), eager2.view(torch.int16))
    assert torch.equal(out.view(torch.int16), eager1.view(torch.int16))
    assert layer.error_bits() == 0
    layer.close()


def test_more_tokens_than_one_pass():
    """150 tokens: three passes of the dense path through one workspace."""
    case = cases.make_case(2048, 256, 32, 4, BF, BF, 150, seed=250)
    figs = _check_case(case, tokens=[0, 63, 64, 127, 128, 149], check_stages=False)
    assert figs["launches"] == 3 * DENSE_LAUNCHES
    assert figs["err_bits"] == 0
