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


def _nvfp4_dequant(codes, scales, rows, K):
    c = np.empty((rows, K), dtype=np.int64)
    c[:, 0::2] = codes & 15
    c[:, 1::2] = codes >> 4
    v = F.e2m1_value(c).reshape(rows, K // 16, 16) * F.ue4m3_value(scales)[:, :, None]
    return v.reshape(rows, K)


@pytest.mark.parametrize("K,N,case", [(256, 128, "random"), (2048, 128, "random"), (512, 64, "random"),
                                      (256, 128, "row_scales"), (256, 128, "k_scales"), (512, 256, "random"),
                                      (256, 256, "row_scales"), (512, 256, "k_scales")])
def test_fp4_block_scaled_gemm_matches_f64(K, N, case):
    """The tcgen05 kind::mxf4nvf4 MMA with per-16 UE4M3 scales in tensor
    memory, against float64 of the decoded operands: every product of two
    scaled E2M1 values is exact in fp32, so the only error is the fp32
    accumulation, K * 2^-24 * sum|a*b| per element.  Structured scales (a
    distinct scale per row of A and of B, a distinct scale per 16-value block
    of K) check that every scale reaches its own rows and blocks."""
    r = np.random.default_rng(K + N + len(case))
    if case == "random":
        a = r.integers(0, 256, size=(128, K // 2), dtype=np.uint8)
        b = r.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
        sa = r.integers(0x28, 0x48, size=(128, K // 16), dtype=np.uint8)
        sb = r.integers(0x28, 0x48, size=(N, K // 16), dtype=np.uint8)
    else:
        a = np.full((128, K // 2), 0x22, np.uint8)     # every value 1.0
        b = np.full((N, K // 2), 0x22, np.uint8)
        sa = np.full((128, K // 16), 0x38, np.uint8)   # 1.0
        sb = np.full((N, K // 16), 0x38, np.uint8)
        if case == "row_scales":
            sa[:] = (((np.arange(128) % 8) + 3) << 3).astype(np.uint8)[:, None]
            sb[:] = (((np.arange(N) % 7) + 4) << 3).astype(np.uint8)[:, None]
        else:
            sa[:] = ((np.arange(K // 16) % 12 + 2) << 3).astype(np.uint8)[None, :]
    dev = [torch.from_numpy(v).to(DEV) for v in (a, sa, b, sb)]
    d = torch.full((128, N), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    capi.moe_debug_fp4_gemm(dev[0].data_ptr(), dev[1].data_ptr(), dev[2].data_ptr(), dev[3].data_ptr(), K, N,
                            d.data_ptr(), err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    A = _nvfp4_dequant(a, sa, 128, K)
    B = _nvfp4_dequant(b, sb, N, K)
    got = d.cpu().numpy().astype(np.float64)
    want = A @ B.T
    bound = K * 2.0 ** -24 * (np.abs(A) @ np.abs(B).T) + 1e-30
    assert np.isfinite(got).all()
    assert (np.abs(got - want) <= bound).all(), float(np.max(np.abs(got - want) / bound))


# ------------------------------------------------------------------ prompt path (grouped GEMMs)

from oracle import formats as F  # noqa: E402
from oracle import layer as OL  # noqa: E402
from tests import cases  # noqa: E402
from tests import tolerance as tol  # noqa: E402

# The prompt configuration's tolerances (relative L2 of the bf16 output against
# the oracle's bf16 output): 1e-2 for W4A4, 2e-3 for W4A8 and FP16.
TOL_L2 = {0: 1e-2, 1: 2e-3, 2: 2e-3}


def _stable_sort(ids, E):
    r = ids.reshape(-1).astype(np.int64)
    valid = (r >= 0) & (r < E)
    order = np.argsort(np.where(valid, r, E), kind="stable")
    order = order[valid[order]]
    off = np.zeros(E + 1, dtype=np.int64)
    off[1:] = np.cumsum(np.bincount(r[valid], minlength=E))
    return order, off


def _x_quantized(case, mode):
    x32 = F.bf16_bits_to_f64(case.x).astype(np.float32)
    if mode == 2:   # the FP16 mode exports x rounded to fp16
        return x32.astype(np.float16).view(np.uint8).reshape(-1)
    if mode == 0:
        codes, sc = OL.quantize_nvfp4_act(x32)
        packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
        return np.concatenate([packed, sc], axis=1).reshape(-1)
    qs, d, s, _ = F.quantize_q8_1(x32)
    return F.q8_1_pack_blocks(qs, d, s).reshape(-1)


def _check_prefill(case, mode, tokens=None):
    """The sort and the quantized x bit for bit; then, from the oracle's own
    stages (tests/tolerance.py, prefill_bounds), every bf16 output within its
    derived bound, equal to the oracle's bf16 output wherever that rounding is
    unambiguous, and the requantized intermediate equal to the oracle's
    except where an fp32 intermediate may round the other way; the prompt
    configuration's relative-L2 tolerance is kept as an aggregate line."""
    res = cases.run_prefill_gpu(case, mode)
    mode = 0 if mode == capi.MOE_PREFILL_W4A4_FIXED else mode   # the same arithmetic as W4A4
    g = case.geom
    T = case.x.shape[0]
    order, off = _stable_sort(case.ids, g.E)
    assert np.array_equal(res["off"], off), "expert row offsets differ"
    assert np.array_equal(res["perm"][: off[-1]], order), "sorted route order differs"
    assert np.array_equal(res["xq"], _x_quantized(case, mode)), "quantized activations differ"
    ref, ref_bits, st = cases.prefill_oracle(case, mode, tokens)
    sel = np.arange(T) if tokens is None else np.asarray(tokens)
    beta, flips, amb = tol.prefill_bounds(g, st, mode)
    figs = tol.check_output(res["out"][sel], ref, beta, l2_tol=TOL_L2[mode])
    # the requantized intermediate of the checked routes (the GPU exports it
    # as fp16 in sorted-row order; the W4A8 operand is q*d rounded once to fp16)
    pos = np.full(case.ids.size, -1, dtype=np.int64)
    pos[order] = np.arange(order.size)
    n_amb = n_tot = 0
    for i, t in enumerate(sel):
        for k in range(g.top_k):
            if not st["valid"][i, k]:
                continue
            row = res["i16"][pos[t * g.top_k + k]].astype(np.float64)
            want = st["inter_hat"][i, k]
            allowed = flips[i, k]
            if mode == 1:
                want = want.astype(np.float16).astype(np.float64)
                allowed = allowed + tol.ulp_fp16(np.abs(want) + allowed)
            diff = np.abs(row - want)
            a = amb[i, k]
            assert np.all(diff[~a] == 0), f"route ({t},{k}): {int(np.sum(diff[~a] != 0))} unambiguous codes differ"
            assert np.all(diff <= allowed * (1 + 1e-9) + 1e-300), f"route ({t},{k}): a code beyond its rounding"
            n_amb += int(a.sum())
            n_tot += a.size
    figs["inter_ambiguous_frac"] = n_amb / max(n_tot, 1)
    return res, figs


def _ragged_ids(T, E, K, seed):
    """Expert 0 gets every token's first route (more than two 128-row tiles),
    the rest spread unevenly, one expert gets none, one route is invalid."""
    r = np.random.default_rng(seed)
    ids = np.zeros((T, K), dtype=np.int32)
    for t in range(T):
        others = r.choice(np.arange(1, E - 1), size=K - 1, replace=False, p=None)
        ids[t, 1:] = others
    ids[T // 2, K - 1] = E + 3
    return ids


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_prefill_ragged_small(mode):
    """H=256 I=256 E=8 top-3, T=300: one expert with 300 rows (two tiles, the
    second partly filled), uneven others, an empty expert, a bad id."""
    T, E, K = 300, 8, 3
    case = cases.make_prefill_case(256, 256, E, K, T, seed=200 + mode, ids=_ragged_ids(T, E, K, 7))
    res, _ = _check_prefill(case, mode)
    assert res["err"] & capi.MOE_DEVERR_BAD_ID


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_prefill_ragged_small_gelu_tanh(mode):
    """The ragged small layer with the gelu_tanh GLU."""
    T, E, K = 300, 8, 3
    case = cases.make_prefill_case(256, 256, E, K, T, seed=210 + mode, ids=_ragged_ids(T, E, K, 8), glu=1)
    _check_prefill(case, mode)


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_prefill_qwen3_30b_a3b_shaped_chunk(mode):
    """H=2048 I=768 E=128 top-8, a 4096-token chunk (32768 routed rows); the
    oracle checks a sample of tokens, the sort and the quantized x in full."""
    case = cases.make_prefill_case(2048, 768, 128, 8, 4096, seed=300 + mode)
    res, _ = _check_prefill(case, mode, tokens=[0, 1, 2047, 4095])
    assert res["err"] == 0


def test_prefill_w4a4_route_sum_orders():
    """W4A4 with the fixed-order route sum gives the same bits on repeated
    calls; the completion-order sum (L2 reductions) is within the oracle's
    bound on its own (above) and differs from the fixed order only where the
    fp32 order of the K additions moves a bf16 rounding: by at most one bf16
    unit, on a small fraction of the outputs."""
    T, E, K = 300, 8, 3
    case = cases.make_prefill_case(256, 256, E, K, T, seed=230, ids=_ragged_ids(T, E, K, 9))
    a = cases.run_prefill_gpu(case, capi.MOE_PREFILL_W4A4_FIXED, stages=False)["out"]
    b = cases.run_prefill_gpu(case, capi.MOE_PREFILL_W4A4_FIXED, stages=False)["out"]
    assert np.array_equal(a, b), "fixed-order W4A4 is not repeatable"
    c = cases.run_prefill_gpu(case, capi.MOE_PREFILL_W4A4, stages=False)["out"]
    fa = F.bf16_bits_to_f64(a)
    fc = F.bf16_bits_to_f64(c)
    diff = fa != fc
    ulp = np.abs(fa) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(fa - fc)[diff] <= ulp[diff] * 1.0001), "orders differ by more than one bf16 unit"
    assert diff.mean() < 0.01, f"{diff.mean():.4f} of the outputs differ between the two orders"
