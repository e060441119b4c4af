"""GPU parity of the dense quantized linear (moe_linear) against the oracle
(oracle/linear.py), through the C ABI.

The GPU accumulates exact per-block integer dots scaled in fp32 (lanes in
sequence, then a warp tree) and rounds once to bf16; the bound on its fp32
error before that rounding is 2 (nb + 40) u32 sum_k |W||x_hat| |row_scale|
(nb = K/32 blocks), and tests/tolerance.check_output applies it (bit-exact
bf16 wherever the rounding is unambiguous, max rel <= 2e-3, rel L2 <= 5e-4)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle import formats as F  # noqa: E402
from oracle import linear as LIN  # noqa: E402
from quantized_routed_expert_route_gb300 import capi  # noqa: E402
from synth import banks as S  # noqa: E402
from synth import counter as C  # noqa: E402
from tests import tolerance as tol  # noqa: E402

DEV = "cuda"


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _run(wtype, rows_dev, N, K, rs_dev, x, T):
    xd = torch.from_numpy(x.view(np.int16)).to(DEV)
    out = torch.full((T, N), -1, dtype=torch.int16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    capi.moe_linear(wtype, rows_dev.data_ptr(), N, K, rs_dev.data_ptr() if rs_dev is not None else None,
                    xd.data_ptr(), T, out.data_ptr(), err.data_ptr(), _stream())
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16), int(err.item())


def _check(wtype, rows, K, rs, x, got, sel=None):
    """Oracle on the selected rows (all by default): rows are independent."""
    sel = np.arange(rows.shape[0]) if sel is None else np.asarray(sel)
    y, _, st = LIN.dense_linear(wtype, rows[sel], K, None if rs is None else rs[sel], x)
    nb = K // 32
    beta = 2.0 * (nb + 40) * tol.U32 * (np.abs(st["x_hat"]) @ np.abs(st["W"]).T) * np.abs(st["s"])[None, :]
    return tol.check_output(got[:, sel], y, beta)


def _rows(seed, wtype, K, N):
    rows = C.bank_bytes_np(seed, wtype, K, 0, N)
    dev = torch.empty(rows.size + 16, dtype=torch.uint8, device=DEV)
    dev[: rows.size].copy_(torch.from_numpy(rows.reshape(-1)))
    return rows, dev


@pytest.mark.parametrize("wtype,K,T", [(w, k, t) for w, k in [(F.TYPE_NVFP4, 2048), (F.TYPE_NVFP4, 160),
                                                             (F.TYPE_Q4_K, 2048), (F.TYPE_Q8_0, 768),
                                                             (F.TYPE_Q6_K, 768), (F.TYPE_Q4_0, 2048)]
                                       for t in (1, 3, 8)] +
                         [(F.TYPE_Q4_1, 768, 3), (F.TYPE_Q5_0, 2048, 1), (F.TYPE_Q5_1, 160, 8),
                          (F.TYPE_Q5_K, 768, 3), (F.TYPE_MXFP4, 2048, 1), (F.TYPE_MXFP4, 160, 3)])
def test_linear_matches_oracle(wtype, K, T):
    """N = 1000 rows (a ragged share per CTA and per ring slot), per-row
    scales of three parts (a fused qkv-like module); NVFP4 at K = 160 has
    rows that are not 16-byte aligned."""
    N = 1000
    rows, dev = _rows(40 + wtype + K, wtype, K, N)
    rs = np.concatenate([np.full(600, 0.37), np.full(250, 1.0), np.full(150, 2.5)]).astype(np.float32)
    x = S.hidden_bf16(50 + T, T, K)
    got, err = _run(wtype, dev[: rows.size], N, K, torch.from_numpy(rs).to(DEV), x, T)
    assert err == 0
    _check(wtype, rows, K, rs, x, got)


def test_linear_no_row_scale_and_single_row():
    K = 512
    for N in (1, 7):
        rows, dev = _rows(60 + N, F.TYPE_NVFP4, K, N)
        x = S.hidden_bf16(61, 2, K)
        got, err = _run(F.TYPE_NVFP4, dev[: rows.size], N, K, None, x, 2)
        assert err == 0
        _check(F.TYPE_NVFP4, rows, K, None, x, got)


def test_linear_full_size_sampled_rows():
    """A 48-layer stack of fused qkv projections (H=2048, q 4096 + k 512 +
    v 512 rows each) as one NVFP4 matrix of 245,760 rows (283 MB), T=1 and
    T=8; the oracle checks 64 sampled rows, all tokens."""
    N, K = 48 * 5120, 2048
    rb = F.row_bytes(F.TYPE_NVFP4, K)
    dev = torch.empty(N * rb + 16, dtype=torch.uint8, device=DEV)
    C.fill_bank_torch(dev[: N * rb], 71, F.TYPE_NVFP4, K)
    rs = S.rng(72).uniform(0.1, 2.0, size=N).astype(np.float32)
    sel = np.sort(S.rng(73).choice(N, size=64, replace=False))
    host_rows = np.zeros((N, rb), np.uint8)
    for r in sel:
        host_rows[r] = C.bank_bytes_np(71, F.TYPE_NVFP4, K, int(r), int(r) + 1)[0]
    for T in (1, 8):
        x = S.hidden_bf16(74 + T, T, K)
        got, err = _run(F.TYPE_NVFP4, dev[: N * rb], N, K, torch.from_numpy(rs).to(DEV), x, T)
        assert err == 0
        _check(F.TYPE_NVFP4, host_rows, K, rs, x, got, sel=sel)


def test_linear_argument_errors():
    K, N = 256, 16
    rows, dev = _rows(80, F.TYPE_Q8_0, K, N)
    x = torch.zeros((9, K), dtype=torch.int16, device=DEV)
    out = torch.zeros((9, N), dtype=torch.int16, device=DEV)
    lib = capi.library()
    s = _stream()
    assert lib.moe_linear(F.TYPE_Q8_0, dev.data_ptr(), N, K, None, x.data_ptr(), 0, out.data_ptr(), None, s) == 0
    assert lib.moe_linear(F.TYPE_Q8_0, dev.data_ptr(), N, K, None, x.data_ptr(), 9, out.data_ptr(), None, s) == \
        capi.MOE_EUNSUPPORTED
    assert lib.moe_linear(F.TYPE_BF16, dev.data_ptr(), N, K, None, x.data_ptr(), 1, out.data_ptr(), None, s) == \
        capi.MOE_EUNSUPPORTED
    assert lib.moe_linear(F.TYPE_Q8_0, dev.data_ptr() + 2, N, K, None, x.data_ptr(), 1, out.data_ptr(), None,
                          s) == capi.MOE_EINVAL
    assert lib.moe_linear(F.TYPE_Q4_K, dev.data_ptr(), N, 96, None, x.data_ptr(), 1, out.data_ptr(), None, s) == \
        capi.MOE_EINVAL
    assert lib.moe_linear(F.TYPE_Q8_0, None, N, K, None, x.data_ptr(), 1, out.data_ptr(), None, s) == capi.MOE_EINVAL
    torch.cuda.synchronize()
    assert int(out.abs().sum().item()) == 0          # nothing was written
