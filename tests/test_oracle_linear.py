"""Pins of the dense linear oracle (oracle/linear.py): brute force over
Python integers and fractions from the raw bytes, an exact closed form,
exact linearity in each row's scale, and a fused module equal to its parts."""
from fractions import Fraction

import numpy as np

from oracle import formats as F
from oracle import linear as LIN
from synth import banks as S


def _q8_0_rows(seed, N, K):
    r = np.random.default_rng(seed)
    w = (r.standard_normal((N, K)) * 0.05).astype(np.float32)
    out = np.zeros((N, K // 32, 34), np.uint8)
    for n in range(N):
        for b in range(K // 32):
            blk = w[n, 32 * b: 32 * b + 32]
            d = np.float16(np.abs(blk).max() / 127.0)
            q = np.clip(np.rint(blk / np.float32(d)), -127, 127).astype(np.int8)
            out[n, b, 0:2] = np.frombuffer(d.tobytes(), np.uint8)
            out[n, b, 2:] = q.view(np.uint8)
    return out.reshape(N, K // 32 * 34)


def test_tiny_q8_0_linear_brute_force_fractions():
    """Exact rational arithmetic from the row bytes: every fp16 scale and the
    q8_1 codes of x are exact rationals, so the fp64 oracle must agree to a
    few ulps."""
    N, K, T = 5, 96, 2
    rows = _q8_0_rows(3, N, K)
    x = S.hidden_bf16(4, T, K)
    rs = np.array([0.5, 1.0, 2.0, 0.001, 3.25], np.float32)
    y, _, _ = LIN.dense_linear(F.TYPE_Q8_0, rows, K, rs, x)
    for t in range(T):
        qs, d, _, _ = F.quantize_q8_1(F.bf16_bits_to_f64(x[t]).astype(np.float32))
        for n in range(N):
            acc = Fraction(0)
            for b in range(K // 32):
                blk = rows[n, 34 * b: 34 * b + 34]
                dw = Fraction(float(np.frombuffer(blk[0:2].tobytes(), np.float16)[0]))
                da = Fraction(float(np.uint16(d[b]).view(np.float16)))
                dot = sum(int(np.int8(np.uint8(c).view(np.int8))) * int(qs[b, i]) for i, c in enumerate(blk[2:]))
                acc += dw * da * dot
            want = float(acc * Fraction(float(rs[n])))
            assert abs(y[t, n] - want) <= 1e-13 * max(1.0, abs(want))


def test_unit_codes_integer_activation_closed_form():
    """One Q8_0 row of unit codes with d = 1 and x integers with |x| max 127
    in every block: q8_1 keeps x exactly (d_a = 1) and y = row_scale * sum(x)."""
    K = 128
    row = np.zeros((1, K // 32, 34), np.uint8)
    row[..., 0:2] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
    row[..., 2:] = 1
    r = np.random.default_rng(5)
    xi = r.integers(-127, 128, size=K).astype(np.float32)
    xi[::32] = 127.0                          # each block's amax is 127
    xbits = xi.view(np.uint32) >> 16          # integers up to 127 are exact in bf16
    y, bits, _ = LIN.dense_linear(F.TYPE_Q8_0, row.reshape(1, -1), K, np.array([0.75], np.float32),
                                  xbits.astype(np.uint16)[None, :])
    assert y[0, 0] == 0.75 * float(xi.sum())


def test_row_scale_linearity_and_fused_module_equals_parts():
    """Scaling row n's scale by a power of two scales y[:, n] exactly; the
    rows of three NVFP4 parts with their own scales, run as one fused linear,
    equal the three separate linears."""
    K, T = 256, 3
    r = np.random.default_rng(6)
    parts = []
    for n in (4, 2, 3):
        w = (r.standard_normal((n, K)) * 0.05).astype(np.float32)
        parts.append(S.convert_nvfp4(w, np.float32(np.abs(w).max() / (6 * 448))))
    scales = [np.float32(0.3), np.float32(1.0), np.float32(2.5)]
    x = S.hidden_bf16(7, T, K)
    fused_rows = np.concatenate(parts)
    rs = np.concatenate([np.full(p.shape[0], s, np.float32) for p, s in zip(parts, scales)])
    y, _, _ = LIN.dense_linear(F.TYPE_NVFP4, fused_rows, K, rs, x)
    off = 0
    for p, s in zip(parts, scales):
        yp, _, _ = LIN.dense_linear(F.TYPE_NVFP4, p, K, np.full(p.shape[0], s, np.float32), x)
        assert np.array_equal(y[:, off: off + p.shape[0]], yp)
        off += p.shape[0]
    rs2 = rs.copy()
    rs2[1] *= 4.0
    y2, _, _ = LIN.dense_linear(F.TYPE_NVFP4, fused_rows, K, rs2, x)
    assert np.array_equal(y2[:, 1], 4.0 * y[:, 1])
    assert np.array_equal(np.delete(y2, 1, axis=1), np.delete(y, 1, axis=1))
