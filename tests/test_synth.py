"""The input generators: host and torch counter-based banks agree byte for
byte, converted NVFP4 blocks decode near their source weights, and the
routings have the stated structure."""
import numpy as np
import torch

from oracle import formats as F
from synth import banks as S
from synth import counter as C


def test_splitmix64_known_first_outputs():
    # SplitMix64 with seed 0: the widely published first outputs
    w = C.words_np(0, 0, 3)
    assert [int(v) for v in w] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_bank_host_equals_torch_cpu():
    for wtype, k in [(C.NVFP4, 256), (C.Q4_K, 512), (C.Q8_0, 256), (C.BF16, 64), (C.Q6_K, 512), (C.Q4_0, 256),
                     (C.Q4_1, 256), (C.Q5_0, 256), (C.Q5_1, 256), (C.Q5_K, 512), (C.MXFP4, 256),
                     (C.F16, 64), (C.F32, 64)]:
        rb = C._row_bytes(wtype, k)
        rows = 40
        t = torch.empty(rows * rb, dtype=torch.uint8)
        C.fill_bank_torch(t, 1234 + wtype, wtype, k, chunk_rows=16)
        full = C.bank_bytes_np(1234 + wtype, wtype, k, 0, rows)
        assert np.array_equal(t.numpy().reshape(rows, rb), full)
        part = C.bank_bytes_np(1234 + wtype, wtype, k, 13, 9)       # sub-range regenerates
        assert np.array_equal(part, full[13:22])


def test_counter_banks_decode_finite():
    for wtype, k in [(C.NVFP4, 256), (C.Q4_K, 512), (C.Q8_0, 256), (C.BF16, 64), (C.Q6_K, 512), (C.Q4_0, 256),
                     (C.Q4_1, 256), (C.Q5_0, 256), (C.Q5_1, 256), (C.Q5_K, 512), (C.MXFP4, 256),
                     (C.F16, 64), (C.F32, 64)]:
        rows = C.bank_bytes_np(99, wtype, k, 0, 64)
        v = F.dequantize_rows(wtype, rows, k)
        # NVFP4 rows exclude weight_scale_2 (applied to the projection output)
        limit = 12.0 if wtype == C.NVFP4 else 0.3
        assert np.isfinite(v).all() and 0 < np.abs(v).max() < limit


def test_converted_nvfp4_blocks_within_half_step():
    r = np.random.default_rng(0)
    w = (r.standard_normal((8, 256)) * 0.02).astype(np.float32)
    s2 = np.float32(np.abs(w).max() / np.float32(6 * 448))
    rows = S.convert_nvfp4(w, s2)
    back = F.dequantize_rows(F.TYPE_NVFP4, rows, 256) * float(s2)
    sv = F.ue4m3_value(rows[:, 128:]).repeat(16, axis=1) * float(s2)
    mag = np.abs(back)
    step = np.where(mag >= 4 * sv, 2 * sv, np.where(mag >= 2 * sv, sv, 0.5 * sv))
    assert (np.abs(back - w) <= step / 2 * (1 + 1e-5) + 1e-12).all()


def test_converted_q4k_reconstructs():
    r = np.random.default_rng(1)
    w = (r.standard_normal((4, 512)) * 0.02).astype(np.float32)
    back = F.dequantize_rows(F.TYPE_Q4_K, S.convert_q4k(w), 512)
    rel = np.linalg.norm(back - w) / np.linalg.norm(w)
    assert rel < 0.12


def test_converted_q6k_and_q4_0_reconstruct():
    r = np.random.default_rng(2)
    w = (r.standard_normal((4, 512)) * 0.02).astype(np.float32)
    for wtype, conv, tol in ((F.TYPE_Q6_K, S.convert_q6k, 0.03), (F.TYPE_Q4_0, S.convert_q4_0, 0.12)):
        back = F.dequantize_rows(wtype, conv(w), 512)
        assert np.linalg.norm(back - w) / np.linalg.norm(w) < tol


def test_routings():
    ids, w = S.softmax_topk_routing(0, 16, 128, 8)
    assert ids.shape == (16, 8) and np.allclose(w.sum(1), 1, atol=1e-6)
    assert all(len(set(row)) == 8 for row in ids)
    assert (np.diff(w, axis=1) <= 0).all()
    ids, w = S.zipf_routing(1, 64, 256, 10)
    assert all(len(set(row)) == 10 for row in ids) and np.allclose(w.sum(1), 1, atol=1e-6)
    # Zipf popularity: far fewer distinct experts than uniform routing would give
    assert len(np.unique(ids)) < 200


def test_converted_q4_1_q5_q5k_mxfp4_reconstruct():
    """The encoders of the other GGUF types round-trip N(0, 0.02) weights
    through the oracle's decoders within their code steps."""
    r = np.random.default_rng(3)
    w = (r.standard_normal((4, 512)) * 0.02).astype(np.float32)
    for wtype, enc, tol in [(F.TYPE_Q4_1, lambda v: S.convert_q4_1_q5(v, S.Q4_1), 0.08),
                            (F.TYPE_Q5_0, lambda v: S.convert_q4_1_q5(v, S.Q5_0), 0.06),
                            (F.TYPE_Q5_1, lambda v: S.convert_q4_1_q5(v, S.Q5_1), 0.04),
                            (F.TYPE_Q5_K, S.convert_q5k, 0.06),
                            (F.TYPE_MXFP4, S.convert_mxfp4, 0.15)]:
        rows = enc(w)
        assert rows.shape == (4, F.row_bytes(wtype, 512))
        back = F.dequantize_rows(wtype, rows, 512)
        rel = np.linalg.norm(back - w) / np.linalg.norm(w)
        assert rel < tol, (wtype, rel)
