"""Which GPU results count as correct, derived from the arithmetic.

The GPU computes in fp32 (block contributions accumulated in fp32, the GLU
activation in fp32, one bf16 rounding at the end); the oracle computes the same method in
fp64.  So a GPU output differs from the oracle's fp64 value by at most

  * the fp32 accumulation error of the down dot and the route sum,
  * for a BF16 down type, the fp32 error of the intermediate carried through
    the down dot,
  * for a quantized down type, the q8_1 codes of the intermediate that the
    fp32 and fp64 intermediates may legitimately round differently: a code
    whose pre-rounding value lies within the intermediate's fp32 error of a
    rounding boundary may go either way (and a block scale d whose fp16
    rounding is equally ambiguous may shift the whole block),
  * and the final bf16 rounding.

``output_bounds`` turns those into a per-element bound beta (before the bf16
rounding).  ``check_output`` then asserts: every GPU value is within beta plus
half a bf16 spacing of the oracle's fp64 value; wherever every value within
beta of the oracle's value rounds to the same bf16 number, the GPU value is
that number bit for bit; and the aggregate errors against the oracle's bf16
output meet the stated tolerances (max |err| / max |ref| <= 2e-3 over the
elements whose rounding is unambiguous, relative L2 <= 5e-4 over all).

All quantities are computed from the oracle's own stages: no GPU value feeds
the bounds.
"""
from __future__ import annotations

import numpy as np

from oracle import formats as F

U32 = 2.0 ** -24


def half_ulp_bf16(v):
    _, ex = np.frexp(np.abs(v))
    return np.exp2(np.maximum(ex.astype(np.float64) - 9.0, -134.0))


def ulp_fp16(v):
    _, ex = np.frexp(np.abs(v))
    return np.exp2(np.maximum(ex.astype(np.float64) - 11.0, -24.0))


def _act_slope_eval(g, kind):
    """The GLU activation at g, |its derivative|, and a bound on the error of
    its fp32 evaluation beyond a few relative roundings (which the caller
    adds).  SiLU: g*sigmoid(g), derivative sig*(1 + g*(1 - sig)).  gelu_tanh:
    0.5*g*(1 + tanh z), z = c0*(g + c1*g^3), derivative
    0.5*(1 + tanh z) + 0.5*g*(1 - tanh^2 z)*c0*(1 + 3*c1*g^2); z carries about
    6 roundings, tanhf 2 ulp, so the evaluation error is at most
    0.5*|g|*(6u*|z|*(1 - tanh^2 z) + 4u) plus a few roundings of the value
    (doubled below)."""
    if kind == 1:
        c0, c1 = np.sqrt(2.0 / np.pi), 0.044715
        with np.errstate(over="ignore", invalid="ignore"):
            z = c0 * (g + c1 * g ** 3)
            th = np.tanh(z)
            sech2 = 1.0 - th * th
            act = 0.5 * g * (1.0 + th)
            slope = np.abs(0.5 * (1.0 + th) + 0.5 * g * sech2 * c0 * (1.0 + 3.0 * c1 * g * g))
            ev = U32 * (np.abs(g) * (6.0 * np.abs(z) * sech2 + 4.0) + 6.0 * np.abs(act))
        return act, slope, np.nan_to_num(ev)
    with np.errstate(over="ignore"):
        sig = 1.0 / (1.0 + np.exp(-g))
    return g * sig, np.abs(sig * (1.0 + g * (1.0 - sig))), np.zeros_like(g)


def _inter_error(geom, st, t, k, xh, wgu, eps_h=None, x_err=0.0):
    """fp32 error bound of the intermediate act(g)*u of route (t, k).  eps_h
    bounds the relative accumulation error of the gate and up dots (default:
    the CUDA-core decode paths); x_err bounds |x_gpu - x_hat| per element
    (0 where the GPU's activations are exactly the oracle's)."""
    I = geom.I
    e = int(st["ids"][t, k])
    sg, su = abs(st["scales"][e, 0]), abs(st["scales"][e, 1])
    hg, hu = wgu[:I] @ xh, wgu[I:] @ xh
    g, u = hg * st["scales"][e, 0], hu * st["scales"][e, 1]
    Sg = sg * (np.abs(wgu[:I]) @ np.abs(xh))
    Su = su * (np.abs(wgu[I:]) @ np.abs(xh))
    if eps_h is None:
        nblk = geom.H // 32
        eps_h = 2.0 * (nblk + 40) * U32         # per-lane sequential sums, warp tree, scale products
    Eg = eps_h * Sg + sg * x_err * np.abs(wgu[:I]).sum(axis=1)   # bounds on |g_gpu - g|, |u_gpu - u|
    Eu = eps_h * Su + su * x_err * np.abs(wgu[I:]).sum(axis=1)
    act, dact, ev = _act_slope_eval(g, getattr(geom, "glu", 0))
    a = act * u
    return dact * np.abs(u) * Eg + np.abs(act) * Eu + ev * np.abs(u) + 16 * U32 * np.abs(a) + 1e-30


def q8_1_flip(a, da, qinfo):
    """q8_1 requantization of an intermediate the GPU holds in fp32 within da
    of the oracle's a: a code whose pre-rounding value lies within the
    intermediate's error of a rounding boundary may go either way (one step
    of d), and a block scale d whose fp16 rounding is equally ambiguous may
    shift every code of the block.  Returns (flip: bound on the change of
    each dequantized value, ambiguous mask)."""
    I = a.size
    nbd = I // 32
    a32 = a.astype(np.float32).astype(np.float64).reshape(nbd, 32)
    amax = np.abs(a32).max(axis=1)
    d = amax / 127.0
    dblk = (da.reshape(nbd, 32).max(axis=1) + U32 * amax) / 127.0 + 2 * U32 * d
    q = qinfo["qs"].astype(np.float64)                      # [nbd, 32]
    dh = F.fp16_bits_to_f64(qinfo["d"])                     # [nbd]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(d[:, None] > 0, a32 / d[:, None], 0.0)
        eta = np.where(d[:, None] > 0, (da.reshape(nbd, 32) + np.abs(q) * dblk[:, None]) / d[:, None], 0.0)
    frac = np.abs(ratio - np.floor(ratio) - 0.5)
    amb_code = frac <= eta + 8 * U32 * np.abs(ratio)
    u16 = ulp_fp16(d)
    mid_dist = np.abs(d - (np.floor(d / u16) + 0.5) * u16)
    amb_d = mid_dist <= dblk
    flip = (amb_code * dh[:, None] + amb_d[:, None] * (np.abs(q) + 1.0) * u16[:, None]).reshape(I)
    return flip, (amb_code | amb_d[:, None]).reshape(I)


def output_bounds(geom, st):
    """beta [T, H]: bound on |gpu_fp32_out - oracle_fp64_out| before bf16 rounding,
    plus per-route data for the intermediate checks."""
    T, K, H, I = st["ids"].shape[0], geom.top_k, geom.H, geom.I
    quant_down = geom.down_type not in F.FLOAT_TYPES
    beta = np.zeros((T, H))
    inter_err = np.zeros((T, K, I))
    amb = np.zeros((T, K, I), dtype=bool)
    nbd = I // 32
    for t in range(T):
        xh = st["x_hat"][t]
        for k in range(K):
            if not st["valid"][t, k]:
                continue
            e = int(st["ids"][t, k])
            wgu, wd = st["experts"][e]
            sws = abs(st["scales"][e, 2] * st["w"][t, k])
            da = _inter_error(geom, st, t, k, xh, wgu)
            inter_err[t, k] = da
            a = st["inter"][t, k]
            c_dn = 2.0 * (nbd + 40) * U32
            absW = np.abs(wd)
            if quant_down:
                flip, amb[t, k] = q8_1_flip(a, da, st["inter_act"][t][k])
                ahat = st["inter_hat"][t, k]
                beta[t] += sws * (absW @ flip + c_dn * (absW @ np.abs(ahat)))
            else:
                beta[t] += sws * (absW @ da + c_dn * (absW @ np.abs(a)))
            beta[t] += (K + 8) * U32 * np.abs(st["y"][t, k])
    return beta, inter_err, amb


def check_output(out_bits, ref, beta, max_rel_tol=2e-3, l2_tol=5e-4):
    """Assert the GPU bf16 output against the oracle; returns the figures."""
    gpu = F.bf16_bits_to_f64(np.asarray(out_bits, dtype=np.uint16)).reshape(ref.shape)
    ref16 = F.round_to_bf16(ref)
    bound = beta + half_ulp_bf16(np.abs(ref) + beta) * (1 + 1e-9) + 1e-30
    err = np.abs(gpu - ref)
    bad = err > bound
    assert not bad.any(), (
        f"{int(bad.sum())} outputs outside the derived bound; worst excess "
        f"{float((err - bound)[bad].max()):.3e} at {np.argwhere(bad)[:5].tolist()}")
    unique = F.round_to_bf16(ref - beta) == F.round_to_bf16(ref + beta)
    mism = unique & (gpu != ref16)
    assert not mism.any(), f"{int(mism.sum())} outputs differ from an unambiguous bf16 rounding"
    scale = max(np.abs(ref).max(), 1e-30)
    max_rel_all = float(np.abs(gpu - ref16).max() / scale)
    max_rel_unique = float((np.abs(gpu - ref16) * unique).max() / scale)
    rel_l2 = float(np.linalg.norm(gpu - ref16) / max(np.linalg.norm(ref16), 1e-30))
    assert max_rel_unique <= max_rel_tol, max_rel_unique
    assert rel_l2 <= l2_tol, rel_l2
    return {"max_rel_unique": max_rel_unique, "max_rel_all": max_rel_all, "rel_l2": rel_l2,
            "ambiguous_frac": float(1 - unique.mean())}


# ------------------------------------------------------------------ prompt path

def nvfp4_act_flip(a, da, ahat):
    """W4A4 requantization of an intermediate the GPU holds in fp32 within da
    of the oracle's a (per 16 values: scale = UE4M3(amax / 6), codes =
    E2M1(a / scale), both nearest-even with saturation, fp32 arithmetic): the
    block scale can be any UE4M3 value that rounding gives for an amax within
    the block's error, and each code any E2M1 value between those of a - da
    and a + da over that scale (both roundings are monotone).  Returns (flip:
    bound on the change of each dequantized value from ahat, ambiguous
    mask)."""
    ab, db, hb = a.reshape(-1, 16), da.reshape(-1, 16), ahat.reshape(-1, 16)
    amax = np.abs(ab).max(axis=1)
    damax = db.max(axis=1)
    lo = np.maximum(amax - damax, 0.0) / 6.0 * (1.0 - 8 * U32)
    hi = (amax + damax) / 6.0 * (1.0 + 8 * U32)
    c_lo = F.ue4m3_encode_rne_sat(lo.astype(np.float32)).astype(np.int64)
    c_hi = F.ue4m3_encode_rne_sat(hi.astype(np.float32)).astype(np.int64)
    assert np.all(c_hi - c_lo <= 1), "a block scale could take more than two values"
    flip = np.zeros_like(ab)
    for code in (c_lo, c_hi):
        sc = F.ue4m3_value(code)[:, None]
        safe = np.where(sc > 0, sc, 1.0)
        slack = db + 8 * U32 * np.abs(ab)
        v_lo = F.e2m1_value(F.e2m1_encode_rne_sat(((ab - slack) / safe).astype(np.float32))) * sc
        v_hi = F.e2m1_value(F.e2m1_encode_rne_sat(((ab + slack) / safe).astype(np.float32))) * sc
        flip = np.maximum(flip, np.maximum(np.abs(v_lo - hb), np.abs(v_hi - hb)))
    flip = flip.reshape(a.shape)
    return flip, flip > 0


def fp16_act_flip(a, da, ahat):
    """The FP16 prompt mode's one rounding of the fp32 intermediate to fp16
    (nearest even, monotone): any fp16 value between those of a - da and
    a + da."""
    slack = da + 4 * U32 * np.abs(a)
    with np.errstate(over="ignore"):
        v_lo = (a - slack).astype(np.float32).astype(np.float16).astype(np.float64)
        v_hi = (a + slack).astype(np.float32).astype(np.float16).astype(np.float64)
    flip = np.maximum(np.abs(v_lo - ahat), np.abs(v_hi - ahat))
    return flip, flip > 0


def prefill_bounds(geom, st, mode):
    """beta [T', H] for the prompt path (mode 0 W4A4, 1 W4A8, 2 FP16), like
    output_bounds: x as the mode quantizes it (the GPU's operands are exactly
    the oracle's: NVFP4 and fp16 values are exact in fp16, a q8_1 value q*d
    is carried as an fp16 pair hi + lo, exact unless lo underflows, by at
    most 2^-25); both grouped GEMMs accumulate exact products in fp32 on the
    tensor cores, with relative error at most 2*K*2^-24 of sum|a*b| over K
    terms (which also covers an accumulator that truncates); the scales and
    the GLU in fp32; the intermediate requantized by the mode's rule (the
    flips above); the down outputs times s_down * w and the route sum in
    fp32.  Returns (beta, flip [T', K, I], ambiguous mask [T', K, I])."""
    T, K, H, I = st["ids"].shape[0], geom.top_k, geom.H, geom.I
    eps_gu = 2.0 * (H + 16) * U32
    eps_dn = 2.0 * (I + 16) * U32
    pair_err = 2.0 ** -25 if mode == 1 else 0.0
    beta = np.zeros((T, H))
    flips = np.zeros((T, K, I))
    amb = np.zeros((T, K, I), dtype=bool)
    for t in range(T):
        xh = st["x_hat"][t]
        for k in range(K):
            if not st["valid"][t, k]:
                continue
            e = int(st["ids"][t, k])
            wgu, wd = st["experts"][e]
            da = _inter_error(geom, st, t, k, xh, wgu, eps_h=eps_gu, x_err=pair_err)
            a, ahat = st["inter"][t, k], st["inter_hat"][t, k]
            if mode == 0:
                flip, am = nvfp4_act_flip(a, da, ahat)
            elif mode == 1:
                flip, am = q8_1_flip(a, da, st["inter_act"][t][k])
            else:
                flip, am = fp16_act_flip(a, da, ahat)
            flips[t, k], amb[t, k] = flip, am
            sws = abs(st["scales"][e, 2] * st["w"][t, k])
            absW = np.abs(wd)
            beta[t] += sws * (absW @ (flip + pair_err) + eps_dn * (absW @ np.abs(ahat)))
            beta[t] += (K + 8) * U32 * np.abs(st["y"][t, k])
    return beta, flips, amb
