"""GPU parity of the batched path for Q4_K, Q4_0 and NVFP4 banks: batches the fused
small-batch kernel cannot hold, decoded by the grouped CUDA-core kernels
(route + quantize, gate_up + requantize, down, route sum: four launches per
pass).  Same bounds as the other decode tests (tests/tolerance.py),
including the bit-exact q8_1 blocks of x and the intermediate's q8_1 codes
(ambiguity-tolerant); each case first asserts that this path is the one that
ran (its launch count)."""
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

BATCHED_LAUNCHES = 4
Q4K = F.TYPE_Q4_K
NV4 = F.TYPE_NVFP4
Q40 = F.TYPE_Q4_0


@pytest.mark.parametrize("T", [16, 64])
def test_laguna_q4k_zipf_batches(T):
    """H=4096 I=768 E=256 top-10, Zipf(1.1) routing: the Q4_K layers of the
    47-layer stack at T=16 and T=64; the oracle checks a sample of tokens."""
    case = cases.make_case(4096, 768, 256, 10, Q4K, Q4K, T, seed=300 + T, routing="zipf")
    figs = _check_case(case, tokens=[0, 1, T - 1])
    assert figs["launches"] == BATCHED_LAUNCHES
    assert figs["err_bits"] == 0


@pytest.mark.parametrize("T", [8, 16])
def test_qwen3_30b_a3b_shaped_nvfp4_batches(T):
    """H=2048 I=768 E=128 top-8 NVFP4 with per-expert weight_scale_2, softmax
    routing, every token checked with the stage exports."""
    case = cases.make_case(2048, 768, 128, 8, NV4, NV4, T, seed=350 + T)
    figs = _check_case(case)
    assert figs["launches"] == BATCHED_LAUNCHES
    assert figs["err_bits"] == 0


@pytest.mark.parametrize("T", [8, 24])
def test_q4_0_32_experts_top8_batches(T):
    """H=2048 I=768 E=32 top-8 Q4_0, softmax routing, every token checked
    with the stage exports."""
    case = cases.make_case(2048, 768, 32, 8, Q40, Q40, T, seed=360 + T)
    figs = _check_case(case)
    assert figs["launches"] == BATCHED_LAUNCHES
    assert figs["err_bits"] == 0


@pytest.mark.parametrize("wtype", [Q4K, NV4, Q40])
def test_every_token_with_stages(wtype):
    """40 tokens over 24 experts (tiles of 1..8 tokens), every token checked
    with the stage exports."""
    case = cases.make_case(2048, 512, 24, 5, wtype, wtype, 40, seed=310 + wtype)
    figs = _check_case(case)
    assert figs["launches"] == BATCHED_LAUNCHES
    assert figs["err_bits"] == 0


@pytest.mark.parametrize("wtype", [Q4K, NV4, Q40])
def test_one_expert_over_many_token_blocks(wtype):
    """Every route on one expert (duplicates inside each token): 256 routed
    rows, thirty-two 8-token blocks per weight tile."""
    T, K = 64, 4
    ids = [[3] * K for _ in range(T)]
    case = cases.make_case(2048, 512, 8, K, wtype, wtype, T, seed=320 + wtype, ids=ids)
    figs = _check_case(case, tokens=[0, 31, 32, 63])
    assert figs["launches"] == BATCHED_LAUNCHES
    assert figs["err_bits"] == 0


@pytest.mark.parametrize("wtype", [Q4K, NV4, Q40])
def test_bad_ids_flag_and_contribute_zero(wtype):
    T, K = 48, 3
    r = np.random.default_rng(7)
    ids = r.integers(0, 16, size=(T, K)).astype(np.int32)
    ids[0, 1] = 99
    ids[7, 0] = -1
    ids[47, 2] = 16
    case = cases.make_case(2048, 512, 16, K, wtype, wtype, T, seed=330 + wtype, ids=ids)
    figs = _check_case(case, tokens=[0, 7, 20, 47])
    assert figs["launches"] == BATCHED_LAUNCHES
    assert figs["err_bits"] & capi.MOE_DEVERR_BAD_ID


def test_batched_graph_replay_equals_eager():
    case = cases.make_case(4096, 768, 64, 8, Q4K, Q4K, 32, seed=340)
    from quantized_routed_expert_route_gb300.layer import MoeLayer
    g = case.geom
    layer = MoeLayer(g.H, g.I, g.E, g.top_k, g.gate_up_type, g.down_type, case.gu_dev, case.dn_dev,
                     torch.from_numpy(case.sb).to("cuda"), borrow=True)
    assert capi.moe_decode_kernel_count(layer.bank, 32) == BATCHED_LAUNCHES
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
    """150 tokens: three passes of the batched path through one workspace
    (the tile counters and sorted planes are rebuilt every pass)."""
    case = cases.make_case(2048, 512, 32, 4, Q4K, Q4K, 150, seed=360)
    figs = _check_case(case, tokens=[0, 63, 64, 127, 128, 149], check_stages=False)
    assert figs["launches"] == 3 * BATCHED_LAUNCHES
    assert figs["err_bits"] == 0
