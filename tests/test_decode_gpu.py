"""GPU parity of the decode path against the oracle, through the C ABI.

Bit-exact: q8_1 codes and scales of the activation quantizer, per-block
integer dot products, the q8_1 blocks of x inside a decode pass.  Within
derived bounds (tests/tolerance.py): the fp32 intermediate, its q8_1 codes
(a code may differ only where the rounding is ambiguous) and the bf16 output
(bit-exact wherever its rounding is unambiguous; max rel <= 2e-3 and
relative L2 <= 5e-4 against the oracle's bf16 output)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle import formats as F  # noqa: E402
from quantized_routed_expert_route_gb300 import capi  # noqa: E402
from synth import counter as C  # noqa: E402
from tests import cases  # noqa: E402
from tests import tolerance as tol  # noqa: E402

DEV = "cuda"


def _stream():
    return torch.cuda.current_stream().cuda_stream


# ------------------------------------------------------------------ kernels in isolation

def test_q8_1_quantizer_bit_exact():
    r = np.random.default_rng(0)
    parts = [r.standard_normal(32 * 4000).astype(np.float32),
             (r.standard_normal(32 * 2000) * 1e-3).astype(np.float32),
             np.zeros(32 * 10, np.float32),
             # ramps whose x/d land on exact .5 ties
             np.tile((np.arange(32) - 16).astype(np.float32) * 0.25, 50),
             (r.integers(-127, 128, 32 * 500) * np.float32(0.5)).astype(np.float32),
             # values one ulp either side of exact .5 ties of x/d
             np.nextafter(np.tile((np.arange(32) - 16).astype(np.float32) * 0.25, 20), np.float32(np.inf)),
             np.nextafter(np.tile((np.arange(32) - 16).astype(np.float32) * 0.25, 20), np.float32(-np.inf)),
             # blocks whose d is tiny or subnormal
             (r.standard_normal(32 * 200) * 1e-38).astype(np.float32),
             (r.standard_normal(32 * 200) * 1e-44).astype(np.float32)]
    x = np.concatenate(parts)
    xd = torch.from_numpy(x).to(DEV)
    out = torch.empty(x.size // 32 * 36, dtype=torch.uint8, device=DEV)
    capi.moe_quantize_q8_1(xd.data_ptr(), x.size, out.data_ptr(), _stream())
    torch.cuda.synchronize()
    qs, d, s, _ = F.quantize_q8_1(x)
    want = F.q8_1_pack_blocks(qs, d, s).reshape(-1)
    got = out.cpu().numpy()
    assert np.array_equal(got, want), f"{int((got != want).sum())} bytes differ"


@pytest.mark.parametrize("wtype,k", [(F.TYPE_Q8_0, 256), (F.TYPE_Q8_0, 768), (F.TYPE_NVFP4, 2048),
                                     (F.TYPE_NVFP4, 768), (F.TYPE_Q4_K, 4096), (F.TYPE_Q4_K, 768),
                                     (F.TYPE_Q6_K, 2048), (F.TYPE_Q6_K, 768), (F.TYPE_Q4_0, 2048),
                                     (F.TYPE_Q4_0, 96), (F.TYPE_Q4_1, 256), (F.TYPE_Q5_0, 96),
                                     (F.TYPE_Q5_1, 256), (F.TYPE_Q5_K, 768), (F.TYPE_MXFP4, 96),
                                     (F.TYPE_MXFP4, 2048)])
def test_block_dots_bit_exact(wtype, k):
    rows = C.bank_bytes_np(11 + wtype, wtype, k, 0, 64)
    # every byte pattern: raw random codes, including all E2M1 signs and -0
    r = np.random.default_rng(1)
    a = r.standard_normal(k).astype(np.float32)
    qs, d, s, _ = F.quantize_q8_1(a)
    act = F.q8_1_pack_blocks(qs, d, s).reshape(-1)
    # banks are readable to the next 16-byte boundary past their end (MXFP4
    # blocks are read as aligned words)
    rows_d = torch.zeros(rows.size + 16, dtype=torch.uint8, device=DEV)
    rows_d[: rows.size].copy_(torch.from_numpy(rows.reshape(-1).copy()))
    act_d = torch.from_numpy(act).to(DEV)
    # Q6_K at k=768 (630-byte rows) and Q4_0 (18-byte blocks) put blocks at
    # every 2-byte alignment
    nb = k // 16 if wtype in (F.TYPE_NVFP4, F.TYPE_Q6_K) else k // 32
    assert nb == F.block_dots(wtype, rows[:1], k, np.zeros((k // 32, 32), np.int8)).shape[1]
    out = torch.empty((64, nb), dtype=torch.int32, device=DEV)
    capi.moe_debug_block_dots(wtype, rows_d.data_ptr(), 64, k, act_d.data_ptr(), out.data_ptr(), _stream())
    torch.cuda.synchronize()
    want = F.block_dots(wtype, rows, k, qs.reshape(-1))
    assert np.array_equal(out.cpu().numpy(), want)


# ------------------------------------------------------------------ whole layer

def _check_case(case, tokens=None, check_stages=True):
    res = cases.run_gpu(case, stages=check_stages)
    ref, ref_bits, st = cases.oracle(case, tokens)
    sel = np.arange(case.x.shape[0]) if tokens is None else np.asarray(tokens)
    beta, inter_err, amb = tol.output_bounds(case.geom, st)
    figs = tol.check_output(res["out"][sel], ref, beta)
    g = case.geom
    if check_stages and "inter" in res:
        if g.gate_up_type not in F.FLOAT_TYPES:
            for i, t in enumerate(sel):
                xi = st["x_act"][i]
                want = F.q8_1_pack_blocks(xi["qs"], xi["d"], xi["s"]).reshape(-1)
                assert np.array_equal(res["x_blocks"][t], want), f"x q8_1 blocks differ for token {t}"
        for i, t in enumerate(sel):
            for k in range(g.top_k):
                if not st["valid"][i, k]:
                    continue
                ginter = res["inter"][t, k].astype(np.float64)
                assert (np.abs(ginter - st["inter"][i, k]) <= inter_err[i, k]).all(), (t, k)
                if g.down_type not in F.FLOAT_TYPES:
                    blk = res["inter_blocks"][t, k]
                    gq = blk[:, 4:].view(np.int8).astype(np.int64).reshape(-1)
                    oq = st["inter_act"][i][k]["qs"].astype(np.int64).reshape(-1)
                    diff = gq != oq
                    assert (np.abs(gq - oq) <= 1).all()
                    assert not (diff & ~amb[i, k]).any(), f"unambiguous q8_1 code differs (route {t},{k})"
    figs["err_bits"] = res["err"]
    figs["launches"] = res["launches"]
    return figs


def test_tiny_q8_0_layer():
    """H=256 I=128 E=8 top-2 T=1, Q8_0 gate_up and down, no global scales."""
    case = cases.make_case(256, 128, 8, 2, F.TYPE_Q8_0, F.TYPE_Q8_0, 1, seed=0)
    case.sb[:] = 1.0
    figs = _check_case(case)
    assert figs["err_bits"] == 0


@pytest.mark.parametrize("T", [1, 8])
def test_qwen3_30b_a3b_shaped_nvfp4_layer(T):
    """H=2048 I=768 E=128 top-8, NVFP4 rows with per-expert weight_scale_2."""
    case = cases.make_case(2048, 768, 128, 8, F.TYPE_NVFP4, F.TYPE_NVFP4, T, seed=10 + T)
    figs = _check_case(case)
    assert figs["err_bits"] == 0


def test_fused_kernel_many_routes_cost_balanced_split():
    """Q8_0 banks have no grouped path, so 64 routes per pass still take the
    fused kernel (one launch) with its cost-balanced split of the pairs."""
    case = cases.make_case(2048, 768, 128, 8, F.TYPE_Q8_0, F.TYPE_Q8_0, 8, seed=15)
    figs = _check_case(case)
    assert figs["launches"] == 1
    assert figs["err_bits"] == 0


@pytest.mark.parametrize("wtype", [F.TYPE_Q4_K, F.TYPE_BF16])
def test_laguna_shaped_layer(wtype):
    """H=4096 I=768 E=256 top-10 T=1, one Q4_K layer and one BF16 layer."""
    case = cases.make_case(4096, 768, 256, 10, wtype, wtype, 1, seed=20 + wtype)
    figs = _check_case(case)
    assert figs["err_bits"] == 0


@pytest.mark.parametrize("T", [4, 16, 64])
def test_laguna_zipf_batches_sampled(T):
    """Zipf(1.1) routing, T tokens, Q4_K; the oracle checks a sample of tokens."""
    case = cases.make_case(4096, 768, 256, 10, F.TYPE_Q4_K, F.TYPE_Q4_K, T, seed=30 + T, routing="zipf")
    tokens = [0, T - 1] if T > 2 else list(range(T))
    _check_case(case, tokens=tokens)


@pytest.mark.parametrize("gu_t,dn_t", [(F.TYPE_Q4_K, F.TYPE_BF16), (F.TYPE_BF16, F.TYPE_Q4_K),
                                       (F.TYPE_NVFP4, F.TYPE_Q8_0), (F.TYPE_Q8_0, F.TYPE_NVFP4),
                                       (F.TYPE_BF16, F.TYPE_NVFP4), (F.TYPE_Q6_K, F.TYPE_Q4_0),
                                       (F.TYPE_Q4_0, F.TYPE_Q6_K), (F.TYPE_BF16, F.TYPE_Q6_K),
                                       (F.TYPE_Q6_K, F.TYPE_NVFP4), (F.TYPE_Q4_0, F.TYPE_Q8_0),
                                       (F.TYPE_Q5_K, F.TYPE_Q4_1), (F.TYPE_Q5_0, F.TYPE_MXFP4),
                                       (F.TYPE_MXFP4, F.TYPE_Q5_1), (F.TYPE_Q4_1, F.TYPE_Q5_K),
                                       (F.TYPE_F16, F.TYPE_Q4_K), (F.TYPE_Q8_0, F.TYPE_F32),
                                       (F.TYPE_F32, F.TYPE_NVFP4), (F.TYPE_Q6_K, F.TYPE_F16),
                                       (F.TYPE_BF16, F.TYPE_F32), (F.TYPE_F16, F.TYPE_F32)])
def test_mixed_type_pairs(gu_t, dn_t):
    """Gate_up and down of different types: the two-kernel path."""
    case = cases.make_case(512, 256, 16, 4, gu_t, dn_t, 5, seed=40 + 8 * gu_t + dn_t)
    _negate_q6k_scales(case)
    _check_case(case)


def _negate_q6k_scales(case):
    """Flip the sign of every other int8 scale of the routed Q6_K rows, in the
    oracle's copy and in the device bank (the synthetic encoder writes
    non-negative scales only)."""
    g = case.geom
    for rows_of, dev, wt, k, nrows in ((case.gu_rows, case.gu_dev, g.gate_up_type, g.H, 2 * g.I),
                                       (case.dn_rows, case.dn_dev, g.down_type, g.I, g.H)):
        if wt != F.TYPE_Q6_K:
            continue
        rb = F.row_bytes(wt, k)
        for e, rows in rows_of.items():
            sb = rows.reshape(nrows, k // 256, 210)
            assert np.shares_memory(sb, rows)
            sc = sb[..., 192:208].view(np.int8)
            sc[..., 1::2] = -sc[..., 1::2]
            dev[e * nrows * rb:(e + 1) * nrows * rb].copy_(torch.from_numpy(rows.reshape(-1).copy()))


@pytest.mark.parametrize("T", [1, 4])
def test_laguna_shaped_q4_k_gate_up_q6_k_down(T):
    """H=4096 I=768 E=256 top-10: Q4_K gate_up with Q6_K down (the pairing of
    a Q4_K_M checkpoint), with negative Q6_K scales; T=1 is one fused launch."""
    case = cases.make_case(4096, 768, 256, 10, F.TYPE_Q4_K, F.TYPE_Q6_K, T, seed=80 + T)
    _negate_q6k_scales(case)
    figs = _check_case(case)
    if T == 1:
        assert figs["launches"] == 1
    assert figs["err_bits"] == 0


@pytest.mark.parametrize("T", [1, 8])
def test_qwen3_30b_a3b_shaped_q6_k_layer(T):
    """H=2048 I=768 E=128 top-8, Q6_K gate_up and down with negative scales."""
    case = cases.make_case(2048, 768, 128, 8, F.TYPE_Q6_K, F.TYPE_Q6_K, T, seed=90 + T)
    _negate_q6k_scales(case)
    figs = _check_case(case)
    if T == 1:
        assert figs["launches"] == 1
    assert figs["err_bits"] == 0


@pytest.mark.parametrize("wtype", [F.TYPE_Q4_1, F.TYPE_Q5_0, F.TYPE_Q5_1, F.TYPE_Q5_K, F.TYPE_MXFP4])
def test_more_gguf_types_fused_layer(wtype):
    """H=2048 I=768 E=128 top-8, T=1, one fused launch, counter-based rows
    (every code pattern) for Q4_1, Q5_0, Q5_1, Q5_K and MXFP4 banks."""
    case = cases.make_case(2048, 768, 128, 8, wtype, wtype, 1, seed=140 + wtype)
    figs = _check_case(case)
    assert figs["launches"] == 1
    assert figs["err_bits"] == 0


@pytest.mark.parametrize("T", [1, 3])
@pytest.mark.parametrize("wtype", [F.TYPE_F16, F.TYPE_F32])
def test_float_row_layer(wtype, T):
    """H=2048 I=768 E=32 top-8 with F16 or F32 gate_up and down rows (float
    types of FreeToken PR #704's synthetic list, "Validation"): x reaches the
    rows as its bf16 values, the intermediate as fp32; T=1 is one fused
    launch."""
    case = cases.make_case(2048, 768, 32, 8, wtype, wtype, T, seed=150 + wtype + T)
    figs = _check_case(case)
    if T == 1:
        assert figs["launches"] == 1
    assert figs["err_bits"] == 0


@pytest.mark.parametrize("T", [1, 8])
def test_q4_0_layer_32_experts_top8(T):
    """Q4_0 gate_up and down, 32 experts, top-8, H=2048 I=768."""
    case = cases.make_case(2048, 768, 32, 8, F.TYPE_Q4_0, F.TYPE_Q4_0, T, seed=100 + T)
    figs = _check_case(case)
    if T == 1:
        assert figs["launches"] == 1
    assert figs["err_bits"] == 0


def test_q6_k_more_tokens_than_one_pass():
    """Q4_K gate_up + Q6_K down over three passes (150 tokens)."""
    case = cases.make_case(512, 256, 16, 4, F.TYPE_Q4_K, F.TYPE_Q6_K, 150, seed=110)
    _negate_q6k_scales(case)
    _check_case(case, tokens=[0, 63, 64, 149], check_stages=False)


@pytest.mark.parametrize("shape,gu_t,dn_t,T,launches", [
    ((2048, 768, 128, 8), F.TYPE_NVFP4, F.TYPE_NVFP4, 1, 1),   # fused
    ((512, 256, 16, 4), F.TYPE_NVFP4, F.TYPE_Q8_0, 5, None),   # two-kernel
    ((256, 256, 8, 4), F.TYPE_BF16, F.TYPE_BF16, 4, 4),        # dense, tensor cores
    ((512, 512, 16, 4), F.TYPE_Q4_K, F.TYPE_Q4_K, 8, 4),       # batched
    ((512, 512, 16, 4), F.TYPE_NVFP4, F.TYPE_NVFP4, 8, 4),     # batched
])
def test_gelu_tanh_glu_on_every_decode_path(shape, gu_t, dn_t, T, launches):
    """The gelu_tanh GLU in each path's gate_up epilogue."""
    H, I, E, K = shape
    case = cases.make_case(H, I, E, K, gu_t, dn_t, T, seed=120 + T + 3 * gu_t, glu=1)
    figs = _check_case(case)
    if launches is not None:
        assert figs["launches"] == launches
    assert figs["err_bits"] == 0


@pytest.mark.parametrize("src", ["host", "device"])
def test_fold_down_scale_equals_prefolded_bank(src):
    """moe_bank_fold_down_scale(per_expert_scale) gives the outputs, bit for
    bit, of a bank created with s_down * per_expert_scale (fp32), and those
    match the oracle on the folded scale bank."""
    from quantized_routed_expert_route_gb300.layer import MoeLayer
    from synth import banks as S
    case = cases.make_case(512, 256, 16, 4, F.TYPE_Q4_K, F.TYPE_Q6_K, 3, seed=130)
    g = case.geom
    pes = S.rng(131).uniform(0.25, 4.0, size=g.E).astype(np.float32)
    layer = MoeLayer(g.H, g.I, g.E, g.top_k, g.gate_up_type, g.down_type, case.gu_dev, case.dn_dev,
                     torch.from_numpy(case.sb).to(DEV), borrow=True, max_tokens=3)
    if src == "host":
        capi.moe_bank_fold_down_scale(layer.bank, pes.ctypes.data, capi.MOE_SRC_HOST, _stream())
    else:
        pes_d = torch.from_numpy(pes).to(DEV)
        capi.moe_bank_fold_down_scale(layer.bank, pes_d.data_ptr(), capi.MOE_SRC_DEVICE, _stream())
    x = torch.from_numpy(case.x.view(np.int16)).to(DEV).view(torch.bfloat16)
    out = layer.decode(x, torch.from_numpy(case.ids).to(DEV), torch.from_numpy(case.w).to(DEV))
    torch.cuda.synchronize()
    folded = out.view(torch.int16).cpu().numpy().view(np.uint16)
    layer.close()
    case.sb[:, 2] = case.sb[:, 2] * pes          # fp32 products
    figs = _check_case(case)
    res = cases.run_gpu(case, stages=False)
    assert np.array_equal(res["out"], folded)
    assert figs["err_bits"] == 0


@pytest.mark.parametrize("wtype", [F.TYPE_Q8_0, F.TYPE_NVFP4, F.TYPE_BF16, F.TYPE_Q4_0])
def test_ragged_geometry(wtype):
    """H and I not multiples of the 32-lane tiling, odd E, K and T."""
    case = cases.make_case(160, 96, 5, 3, wtype, wtype, 7, seed=50 + wtype)
    _check_case(case)


def test_more_tokens_than_one_pass():
    """T larger than one internal pass: split into passes, same results."""
    case = cases.make_case(256, 128, 16, 4, F.TYPE_NVFP4, F.TYPE_Q8_0, 150, seed=60)
    _check_case(case, tokens=[0, 63, 64, 149], check_stages=False)


def test_duplicate_expert_in_one_token():
    ids = [[3, 3, 1], [1, 0, 3]]
    case = cases.make_case(256, 128, 4, 3, F.TYPE_Q8_0, F.TYPE_Q8_0, 2, seed=70, ids=ids)
    _check_case(case)


def test_bad_id_sets_error_and_contributes_zero():
    ids = [[2, 99, 0], [-1, 1, 2]]
    case = cases.make_case(256, 128, 4, 3, F.TYPE_Q8_0, F.TYPE_NVFP4, 2, seed=80, ids=ids)
    figs = _check_case(case)
    assert figs["err_bits"] & capi.MOE_DEVERR_BAD_ID


def test_zero_tokens_is_a_noop():
    case = cases.make_case(256, 128, 4, 2, F.TYPE_Q8_0, F.TYPE_Q8_0, 1, seed=90)
    from quantized_routed_expert_route_gb300.layer import MoeLayer
    g = case.geom
    layer = MoeLayer(g.H, g.I, g.E, g.top_k, g.gate_up_type, g.down_type, case.gu_dev, case.dn_dev, None,
                     borrow=True)
    capi.moe_decode(layer.bank, 0, 0, 0, 0, 0, layer.ws.data_ptr(), layer.ws_bytes, _stream())
    torch.cuda.synchronize()
    assert layer.error_bits() == 0
    layer.close()


def test_graph_replay_equals_eager_and_runs_are_deterministic():
    case = cases.make_case(2048, 768, 128, 8, F.TYPE_NVFP4, F.TYPE_NVFP4, 8, seed=100)
    from quantized_routed_expert_route_gb300.layer import MoeLayer
    g = case.geom
    layer = MoeLayer(g.H, g.I, g.E, g.top_k, g.gate_up_type, g.down_type, case.gu_dev, case.dn_dev,
                     torch.from_numpy(case.sb).to(DEV), borrow=True)
    x = torch.from_numpy(case.x.view(np.int16)).to(DEV).view(torch.bfloat16)
    ids = torch.from_numpy(case.ids).to(DEV)
    w = torch.from_numpy(case.w).to(DEV)
    eager1 = layer.decode(x, ids, w).clone()
    eager2 = layer.decode(x, ids, w).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    out = torch.empty_like(eager1)
    with torch.cuda.stream(s):
        layer.decode(x, ids, w, out)          # warm-up on the capture stream
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            layer.decode(x, ids, w, out)
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager1.view(torch.int16), eager2.view(torch.int16))
    assert torch.equal(out.view(torch.int16), eager1.view(torch.int16))
    layer.close()


def test_decode_host_buffers_equal_device_decode_and_kernel_count():
    """moe_decode_host (pinned host x / ids / weights / out) gives the same bits
    as moe_decode on device buffers; moe_decode_kernel_count is 1 for a fused
    small batch and more for larger batches."""
    case = cases.make_case(2048, 768, 128, 8, F.TYPE_NVFP4, F.TYPE_NVFP4, 2, seed=110)
    from quantized_routed_expert_route_gb300.layer import MoeLayer
    g = case.geom
    layer = MoeLayer(g.H, g.I, g.E, g.top_k, g.gate_up_type, g.down_type, case.gu_dev, case.dn_dev,
                     torch.from_numpy(case.sb).to(DEV), borrow=True)
    x = torch.from_numpy(case.x.view(np.int16)).to(DEV).view(torch.bfloat16)
    ids = torch.from_numpy(case.ids).to(DEV)
    w = torch.from_numpy(case.w).to(DEV)
    want = layer.decode(x, ids, w).clone()
    T = case.x.shape[0]
    hx = torch.from_numpy(case.x.view(np.int16)).pin_memory()
    hids = torch.from_numpy(case.ids).pin_memory()
    hw = torch.from_numpy(case.w).pin_memory()
    hout = torch.zeros((T, g.H), dtype=torch.int16).pin_memory()
    iob = capi.moe_decode_io_bytes(layer.bank, T)
    io = torch.empty(iob, dtype=torch.uint8, device=DEV)
    capi.moe_decode_host(layer.bank, hx.data_ptr(), T, hids.data_ptr(), hw.data_ptr(), hout.data_ptr(),
                         io.data_ptr(), iob, layer.ws.data_ptr(), layer.ws_bytes, _stream())
    torch.cuda.synchronize()
    assert torch.equal(hout, want.view(torch.int16).cpu())
    assert capi.moe_decode_kernel_count(layer.bank, 1) >= 1
    assert capi.moe_decode_kernel_count(layer.bank, 0) == 0
    assert capi.moe_decode_kernel_count(layer.bank, 64) >= capi.moe_decode_kernel_count(layer.bank, 1)
    layer.close()


def test_decode_host_single_staged_buffer_equals_device_decode():
    """Host inputs laid out at moe_decode_io_offsets (one pinned buffer, one
    copy) give the same bits as moe_decode on device buffers."""
    case = cases.make_case(2048, 768, 128, 8, F.TYPE_NVFP4, F.TYPE_NVFP4, 3, seed=120)
    from quantized_routed_expert_route_gb300.layer import MoeLayer
    g = case.geom
    layer = MoeLayer(g.H, g.I, g.E, g.top_k, g.gate_up_type, g.down_type, case.gu_dev, case.dn_dev,
                     torch.from_numpy(case.sb).to(DEV), borrow=True)
    x = torch.from_numpy(case.x.view(np.int16)).to(DEV).view(torch.bfloat16)
    ids = torch.from_numpy(case.ids).to(DEV)
    w = torch.from_numpy(case.w).to(DEV)
    want = layer.decode(x, ids, w).clone()
    T, K = case.x.shape[0], g.top_k
    iob = capi.moe_decode_io_bytes(layer.bank, T)
    o_ids, o_w, o_out = capi.moe_decode_io_offsets(layer.bank, T)
    assert 2 * T * g.H <= o_ids and o_ids + 4 * T * K <= o_w and o_w + 4 * T * K <= o_out <= iob
    hin = torch.zeros(iob, dtype=torch.uint8).pin_memory()
    hin[: 2 * T * g.H] = torch.from_numpy(case.x.view(np.uint8).reshape(-1).copy())
    hin[o_ids: o_ids + 4 * T * K] = torch.from_numpy(case.ids.view(np.uint8).reshape(-1).copy())
    hin[o_w: o_w + 4 * T * K] = torch.from_numpy(case.w.view(np.uint8).reshape(-1).copy())
    hout = torch.zeros((T, g.H), dtype=torch.int16).pin_memory()
    io = torch.empty(iob, dtype=torch.uint8, device=DEV)
    base = hin.data_ptr()
    capi.moe_decode_host(layer.bank, base, T, base + o_ids, base + o_w, hout.data_ptr(), io.data_ptr(), iob,
                         layer.ws.data_ptr(), layer.ws_bytes, _stream())
    torch.cuda.synchronize()
    assert torch.equal(hout, want.view(torch.int16).cpu())
    layer.close()
