"""Oracle: a dense quantized linear whose output rows carry their own fp32
scale, in fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

FreeToken PR #732, "Design": the scale of an NVFP4 tensor multiplies its
matmul result, y = (x @ W^T) * s, and a fused module that runs several
tensors as one matmul (qkv, gate_up) carries ggml_scale, one fp32 value per
output row (each part's scale, 1 for parts without one); its "Not covered"
list notes that the dense linears apply it in a separate elementwise kernel
after the GEMM.  The activation enters as in the decode path's prep_input
(FreeToken PR #704, "How it plugs into the CPU executor"): bf16 x quantized
to q8_1 per 32 values.

    y[t, n] = row_scale[n] * sum_k dequant(W)[n, k] * dequant(q8_1(x[t]))[k]
    out[t, n] = bf16(y[t, n])   (one rounding, ties to even)

A quantized row dotted with a q8_1 activation equals, up to rounding order,
the dot of the dequantized row with the dequantized activation; this oracle
computes that plain definition with an fp64 matmul.

Pins (tests/test_oracle_linear.py): brute force over Python integers and
fractions on a tiny Q8_0 case from the raw bytes; an exact closed form
(unit Q8_0 codes, integer activations); exact linearity in each row's scale;
the rows of a fused module equal the separate linears of its parts.
"""
from __future__ import annotations

import numpy as np

from . import formats as F


def dense_linear(wtype: int, rows, K: int, row_scale, x_bf16_bits):
    """rows: uint8 [N, row_bytes(wtype, K)] (a quantized type);
    row_scale: fp32 [N] or None (ones); x_bf16_bits: uint16 [T, K].
    Returns (y fp64 [T, N], out bf16 bits [T, N], {"x_hat": fp64 [T, K],
    "x_act": per-token q8_1 codes/scales})."""
    rows = np.asarray(rows, dtype=np.uint8)
    N = rows.shape[0]
    assert wtype != F.TYPE_BF16
    W = F.dequantize_rows(wtype, rows, K)                          # [N, K]
    x = F.bf16_bits_to_f64(np.asarray(x_bf16_bits, dtype=np.uint16)).reshape(-1, K)
    T = x.shape[0]
    s = np.ones(N) if row_scale is None else np.asarray(row_scale, dtype=np.float32).astype(np.float64)
    x_hat = np.zeros((T, K))
    acts = []
    for t in range(T):
        qs, d, sbits, _ = F.quantize_q8_1(x[t].astype(np.float32))
        x_hat[t] = F.dequantize_q8_1(qs, d).reshape(K)
        acts.append({"qs": qs, "d": d, "s": sbits})
    y = (x_hat @ W.T) * s[None, :]
    out = F.round_to_bf16(y)
    return y, F.f64_bf16_value_to_bits(out), {"x_hat": x_hat, "x_act": acts, "W": W, "s": s}
