"""Pins of the oracle's layer math: brute force over Python floats on the tiny
Q8_0 layer, the unit-scale BF16 special case against a numpy matmul
formula, invariants, and the W4A4 activation quantizer."""
import math

import numpy as np
import torch

from oracle import formats as F
from oracle import layer as L
from synth import banks as S


def _tiny(seed=0, T=1):
    H, I, E, K = 256, 128, 8, 2
    geom = L.Geometry(H, I, E, K, F.TYPE_Q8_0, F.TYPE_Q8_0)
    gu, dn, sb = S.converted_layer(seed, H, I, E, S.Q8_0, S.Q8_0)
    x = S.hidden_bf16(seed + 1, T, H)
    ids, w = S.softmax_topk_routing(seed + 2, T, E, K)
    return geom, gu, dn, sb, x, ids, w


def test_tiny_q8_0_layer_brute_force_python_floats():
    geom, gu, dn, sb, x, ids, w = _tiny()
    out, _, _ = L.moe_layer(geom, gu, dn, sb, x, ids, w)
    H, I = geom.H, geom.I
    xf = [float(v) for v in F.bf16_bits_to_f64(x[0])]
    qs, d, _, _ = F.quantize_q8_1(np.array(xf, np.float32))
    xa = [int(qs[b, i]) * float(np.uint16(d[b]).view(np.float16)) for b in range(H // 32) for i in range(32)]

    def q8_0_row(row):
        row = [int(v) for v in row]
        vals = []
        for b in range(len(row) // 34):
            dd = float(np.frombuffer(bytes(row[b * 34: b * 34 + 2]), np.float16)[0])
            for v in row[b * 34 + 2: b * 34 + 34]:
                vals.append(dd * (v - 256 if v > 127 else v))
        return vals

    want = [0.0] * H
    for k in range(geom.top_k):
        e = int(ids[0, k])
        h = [sum(a * b for a, b in zip(q8_0_row(gu[e, r]), xa)) for r in range(2 * I)]
        a = []
        for i in range(I):
            g, u = h[i] * float(sb[e, 0]), h[I + i] * float(sb[e, 1])
            a.append(g / (1.0 + math.exp(-g)) * u)
        aq, ad, _, _ = F.quantize_q8_1(np.array(a, np.float32))
        av = [int(aq[b, i]) * float(np.uint16(ad[b]).view(np.float16)) for b in range(I // 32) for i in range(32)]
        for j in range(H):
            y = sum(p * q for p, q in zip(q8_0_row(dn[e, j]), av))
            want[j] += y * float(sb[e, 2]) * float(w[0, k])
    assert np.allclose(out[0], want, rtol=1e-12, atol=1e-15)


def test_unit_scale_bf16_layer_equals_matmul_formula():
    H, I, E = 64, 32, 3
    r = np.random.default_rng(7)
    wgu = (r.standard_normal((E, 2 * I, H)) * 0.1).astype(np.float32)
    wd = (r.standard_normal((E, H, I)) * 0.1).astype(np.float32)
    gu = np.stack([S.convert_bf16(wgu[e]) for e in range(E)])
    dn = np.stack([S.convert_bf16(wd[e]) for e in range(E)])
    x = S.hidden_bf16(8, 2, H)
    geom = L.Geometry(H, I, E, 1, F.TYPE_BF16, F.TYPE_BF16)
    ids = np.array([[2], [0]], np.int32)
    w = np.ones((2, 1), np.float32)
    out, _, _ = L.moe_layer(geom, gu, dn, None, x, ids, w)
    # the same layer written with torch's bf16 decode and a numpy matmul
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    for t, e in enumerate([2, 0]):
        Wg = torch.from_numpy(wgu[e][:I]).bfloat16().double().numpy()
        Wu = torch.from_numpy(wgu[e][I:]).bfloat16().double().numpy()
        Wd = torch.from_numpy(wd[e]).bfloat16().double().numpy()
        hg, hu = Wg @ xt[t], Wu @ xt[t]
        ref = ((hg / (1 + np.exp(-hg))) * hu) @ Wd.T
        assert np.allclose(out[t], ref, rtol=1e-13, atol=1e-15)


def _gelu_erf(v):
    # the exact GELU, v * Phi(v), from the error function
    return 0.5 * v * (1.0 + np.vectorize(math.erf)(v / math.sqrt(2.0)))


def test_gelu_tanh_pins():
    """The tanh form approximates v * Phi(v) to within 4.8e-4 everywhere (the
    largest gap, 4.73e-4, sits near v = +-2.70); its odd part is exactly v/2,
    so gelu(v) - gelu(-v) = v; gelu(0) = 0 and gelu(v) -> v, 0 in the tails."""
    v = np.linspace(-12.0, 12.0, 240001)
    gt = L.gelu_tanh(v)
    gap = np.abs(gt - _gelu_erf(v))
    assert gap.max() <= 4.8e-4
    assert 4.6e-4 <= gap.max()                     # the tanh form, not the exact one
    assert abs(abs(v[np.argmax(gap)]) - 2.70) < 0.05   # the gap is even in v
    assert np.allclose(gt - L.gelu_tanh(-v), v, rtol=0, atol=1e-14)
    assert L.gelu_tanh(np.array([0.0]))[0] == 0.0
    assert abs(L.gelu_tanh(np.array([12.0]))[0] - 12.0) < 1e-12
    assert abs(L.gelu_tanh(np.array([-12.0]))[0]) < 1e-12


def test_unit_scale_bf16_gelu_layer_against_exact_gelu():
    """One route, unit scales, BF16 rows: the gelu_tanh layer is
    (gelu(x Wg^T) * (x Wu^T)) Wd^T up to the tanh form's 4.8e-4 gap, which
    reaches the output at most through |Wd| @ (4.8e-4 * |x Wu^T|)."""
    H, I, E = 64, 32, 2
    r = np.random.default_rng(9)
    wgu = (r.standard_normal((E, 2 * I, H)) * 0.3).astype(np.float32)
    wd = (r.standard_normal((E, H, I)) * 0.3).astype(np.float32)
    gu = np.stack([S.convert_bf16(wgu[e]) for e in range(E)])
    dn = np.stack([S.convert_bf16(wd[e]) for e in range(E)])
    x = S.hidden_bf16(10, 2, H)
    geom = L.Geometry(H, I, E, 1, F.TYPE_BF16, F.TYPE_BF16, glu=L.GLU_GELU_TANH)
    ids = np.array([[1], [0]], np.int32)
    out, _, _ = L.moe_layer(geom, gu, dn, None, x, ids, np.ones((2, 1), np.float32))
    silu_out, _, _ = L.moe_layer(L.Geometry(H, I, E, 1, F.TYPE_BF16, F.TYPE_BF16), gu, dn, None, x, ids,
                                 np.ones((2, 1), np.float32))
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    for t, e in enumerate([1, 0]):
        Wg = torch.from_numpy(wgu[e][:I]).bfloat16().double().numpy()
        Wu = torch.from_numpy(wgu[e][I:]).bfloat16().double().numpy()
        Wd = torch.from_numpy(wd[e]).bfloat16().double().numpy()
        hg, hu = Wg @ xt[t], Wu @ xt[t]
        ref = (_gelu_erf(hg) * hu) @ Wd.T
        bound = np.abs(Wd) @ (4.8e-4 * np.abs(hu)) + 1e-12
        assert (np.abs(out[t] - ref) <= bound).all()
        assert np.abs(silu_out[t] - ref).max() > 10 * bound.max()   # the kind is honoured


def test_fp16_prompt_mode_is_the_unquantized_layer_up_to_fp16_rounding():
    """In the FP16 mode x (bf16) is exact in fp16 and only the intermediate
    is rounded (relative error <= 2^-11 in the normal range), so the output
    differs from the unquantized layer by at most
    s_down * w * |Wd| @ ((2^-11 + 2^-23) |a| + 2^-25) (the fp32 cast of the
    intermediate comes first), and does differ."""
    H, I, E, K, T = 256, 256, 6, 2, 3
    gu, dn, sb = S.converted_layer(21, H, I, E, S.NVFP4, S.NVFP4)
    x = S.hidden_bf16(22, T, H)
    ids, w = S.softmax_topk_routing(23, T, E, K)
    geom = L.Geometry(H, I, E, K, F.TYPE_NVFP4, F.TYPE_NVFP4)
    out, _, st = L.moe_layer(geom, gu, dn, sb, x, ids, w, act_kind="fp16", stages=True)
    xt = F.bf16_bits_to_f64(x).reshape(T, H)
    assert np.array_equal(st["x_hat"], xt)
    for t in range(T):
        want = np.zeros(H)
        bound = np.zeros(H)
        for k in range(K):
            e = int(ids[t, k])
            Wgu = F.dequantize_rows(F.TYPE_NVFP4, gu[e], H)
            Wd = F.dequantize_rows(F.TYPE_NVFP4, dn[e], I)
            h = Wgu @ xt[t]
            g, u = h[:I] * float(sb[e, 0]), h[I:] * float(sb[e, 1])
            a = g / (1.0 + np.exp(-g)) * u
            f = float(sb[e, 2]) * float(w[t, k])
            want += (Wd @ a) * f
            bound += abs(f) * (np.abs(Wd) @ ((2.0 ** -11 + 2.0 ** -23) * np.abs(a) + 2.0 ** -25))
        assert (np.abs(out[t] - want) <= bound * (1 + 1e-9) + 1e-300).all()
        assert np.abs(out[t] - want).max() > 0


def test_f16_gate_up_f32_down_layer_keeps_activations_float():
    """F16 gate_up and F32 down rows (float rows): x is not quantized and the
    intermediate stays unquantized, so with unit scales and one route the
    layer is silu(x Wg^T) * (x Wu^T) Wd^T on the rows' exact values."""
    H, I, E = 64, 32, 2
    r = np.random.default_rng(11)
    wgu = (r.standard_normal((E, 2 * I, H)) * 0.1).astype(np.float16)
    wd = (r.standard_normal((E, H, I)) * 0.1).astype(np.float32)
    gu = wgu.view(np.uint8).reshape(E, 2 * I, 2 * H)
    dn = wd.view(np.uint8).reshape(E, H, 4 * I)
    x = S.hidden_bf16(12, 2, H)
    geom = L.Geometry(H, I, E, 1, F.TYPE_F16, F.TYPE_F32)
    ids = np.array([[1], [0]], np.int32)
    out, _, st = L.moe_layer(geom, gu, dn, None, x, ids, np.ones((2, 1), np.float32), stages=True)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(st["x_hat"], xt)
    for t, e in enumerate([1, 0]):
        Wg, Wu = wgu[e][:I].astype(np.float64), wgu[e][I:].astype(np.float64)
        hg, hu = Wg @ xt[t], Wu @ xt[t]
        ref = ((hg / (1 + np.exp(-hg))) * hu) @ wd[e].astype(np.float64).T
        assert np.allclose(out[t], ref, rtol=1e-13, atol=1e-15)


def test_layer_invariants():
    geom, gu, dn, sb, x, ids, w = _tiny(seed=3, T=3)
    base, _, _ = L.moe_layer(geom, gu, dn, sb, x, ids, w)
    # linear in the routing weight
    out2, _, _ = L.moe_layer(geom, gu, dn, sb, x, ids, w * 2)
    assert np.allclose(out2, 2 * base, rtol=1e-14)
    # linear in s_down
    sb2 = sb.copy()
    sb2[:, 2] *= 4
    out4, _, _ = L.moe_layer(geom, gu, dn, sb2, x, ids, w)
    assert np.allclose(out4, 4 * base, rtol=1e-14)
    # route order does not matter
    outp, _, _ = L.moe_layer(geom, gu, dn, sb, x, ids[:, ::-1].copy(), w[:, ::-1].copy())
    assert np.allclose(outp, base, rtol=1e-13, atol=1e-16)
    # a route with an out-of-range id contributes nothing
    ids_bad = ids.copy()
    ids_bad[:, 1] = 99
    outb, _, _ = L.moe_layer(geom, gu, dn, sb, x, ids_bad, w)
    g1 = L.Geometry(geom.H, geom.I, geom.E, 1, geom.gate_up_type, geom.down_type)
    out1, _, _ = L.moe_layer(g1, gu, dn, sb, x, ids[:, :1].copy(), w[:, :1].copy())
    assert np.allclose(outb, out1, rtol=1e-14)
    # scaling s_gate and s_up together by c with unit silu slope is not linear:
    # the GLU must see the scaled values (scales are applied before the GLU)
    sb3 = sb.copy()
    sb3[:, 0] *= 3
    out3, _, _ = L.moe_layer(geom, gu, dn, sb3, x, ids, w)
    assert not np.allclose(out3, 3 * base, rtol=1e-3)


def test_bf16_output_rounding_is_single_rne():
    geom, gu, dn, sb, x, ids, w = _tiny(seed=5)
    out, bits, _ = L.moe_layer(geom, gu, dn, sb, x, ids, w)
    ref = torch.from_numpy(out.astype(np.float32)).bfloat16().view(torch.int16).numpy().view(np.uint16)
    # fp64 -> bf16 once may differ from fp64 -> fp32 -> bf16 only in rare double-rounding cases
    assert (bits != ref).mean() < 1e-3


def test_nvfp4_activation_quantizer_pins():
    # a block whose amax is 6 has scale UE4M3(1.0) = 0x38 and grid values map exactly
    x = np.array([6, -4, 3, 2, 1.5, 1, 0.5, 0, -0.5, -1, -1.5, -2, -3, -6, 4, 0], np.float32)
    codes, sc = L.quantize_nvfp4_act(x)
    assert sc[0] == 0x38
    assert np.array_equal(F.e2m1_value(codes), x.astype(np.float64))
    # zero block -> scale 0, codes 0
    codes, sc = L.quantize_nvfp4_act(np.zeros(16, np.float32))
    assert sc[0] == 0 and not codes.any()
    # random blocks: every value within half an E2M1 step (times the scale) plus scale rounding
    r = np.random.default_rng(9)
    xb = r.standard_normal((300, 16)).astype(np.float32)
    codes, sc = L.quantize_nvfp4_act(xb)
    back = L.dequantize_nvfp4_act(codes, sc)
    sv = F.ue4m3_value(sc)          # [300, 1]: one scale per 16-value block
    step = np.where(np.abs(back) >= 4 * sv, 2 * sv, np.where(np.abs(back) >= 2 * sv, sv, 0.5 * sv))
    assert (np.abs(back - xb) <= step / 2 + 1e-12 + np.maximum(0, np.abs(xb) - 6 * sv)).all()
