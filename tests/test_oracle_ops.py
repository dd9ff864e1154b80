"""Pins of the oracle's single operations against closed forms, textbook special
cases and library routines (CPU only)."""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from speculative_decoding_spec_gb300 import synth
from speculative_decoding_spec_gb300.configs import BF16, F32, Q4_0


# ---------------- number formats ----------------
@pytest.mark.parametrize("bits,val", [(0x3F80, 1.0), (0xC000, -2.0), (0x3E80, 0.25),
                                      (0x4049, 3.140625), (0x0000, 0.0)])
def test_bf16_decode(bits, val):
    assert oracle.lib().or_bf16_to_double(bits) == val


@pytest.mark.parametrize("bits,val", [(0x3C00, 1.0), (0xC400, -4.0), (0x7BFF, 65504.0),
                                      (0x0001, 2.0 ** -24), (0x0400, 2.0 ** -14),
                                      (0x3555, 0.333251953125)])
def test_f16_decode(bits, val):
    assert oracle.lib().or_f16_to_double(bits) == val


def test_f16_decode_matches_library_on_all_finite_codes():
    codes = np.arange(0, 1 << 16, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = np.array([oracle.lib().or_f16_to_double(int(c)) for c in codes[::97]])
    fin = np.isfinite(ref[::97])
    assert np.array_equal(got[fin], ref[::97][fin])


def test_kv_rounding_bf16_ties_to_even_and_matches_torch():
    ulp = 2.0 ** -7
    assert oracle.round_kv(1.0 + ulp / 2, BF16) == 1.0            # tie -> even (1.0)
    assert oracle.round_kv(1.0 + 1.5 * ulp, BF16) == 1.0 + 2 * ulp  # tie -> even
    assert oracle.round_kv(1.0 + 0.6 * ulp, BF16) == 1.0 + ulp
    x = torch.randn(2000, generator=torch.Generator().manual_seed(5), dtype=torch.float32)
    ref = x.to(torch.bfloat16).float().numpy()
    got = np.array([oracle.round_kv(float(v), BF16) for v in x])
    assert np.array_equal(got.astype(np.float32), ref)
    assert oracle.round_kv(0.1, F32) == np.float32(0.1)


# ---------------- Q4_0 ----------------
def _one_block_q4(codes, scale):
    """A 1x32 Q4_0 matrix built byte by byte: byte i holds element i in its low
    nibble and element i+16 in its high nibble."""
    raw = bytearray(16)
    for i in range(16):
        raw[i] = (codes[i] & 0xF) | ((codes[i + 16] & 0xF) << 4)
    data = torch.tensor(list(raw), dtype=torch.uint8).view(1, 1, 16)
    sc = torch.tensor([scale], dtype=torch.float16).view(1, 1, 1)
    return synth.WTensor(Q4_0, 1, 1, 32, data, sc)


def test_q4_0_block_decode_and_nibble_order():
    codes = [(3 * i + 1) % 16 for i in range(32)]
    w = _one_block_q4(codes, 0.5)
    row = oracle.dequant_row(w, 0)
    assert np.array_equal(row, 0.5 * (np.array(codes) - 8.0))
    # all codes equal to 8 decode to exact zeros; 0 and 15 to the grid ends
    assert np.all(oracle.dequant_row(_one_block_q4([8] * 32, 3.0), 0) == 0.0)
    ends = oracle.dequant_row(_one_block_q4([0] * 16 + [15] * 16, 0.25), 0)
    assert np.all(ends[:16] == -2.0) and np.all(ends[16:] == 1.75)


def test_q4_0_blocks_on_16_value_grid():
    """Each 32-value block holds at most 16 distinct values, all on the grid
    scale * {-8..7} (the Q4_0 property the QAT repack relies on)."""
    w = synth.make_matrix(torch.Generator().manual_seed(1), Q4_0, 1, 8, 256, 0.02, "cpu")
    for n in range(8):
        row = oracle.dequant_row(w, n)
        for b in range(256 // 32):
            blk = row[b * 32:(b + 1) * 32]
            s = float(w.scales[0, n, b])
            assert len(set(blk.tolist())) <= 16
            q = blk / s
            assert np.all(np.abs(q - np.round(q)) < 1e-12)
            assert q.min() >= -8 and q.max() <= 7


# ---------------- linear ----------------
@pytest.mark.parametrize("dtype", [F32, BF16, Q4_0])
def test_linear_matches_numpy_matmul(dtype):
    g = torch.Generator().manual_seed(3)
    w = synth.make_matrix(g, dtype, 2, 48, 96, 0.05, "cpu")
    x = np.random.default_rng(0).standard_normal((5, 96))
    for layer in (0, 1):
        W = np.stack([oracle.dequant_row(w, n, layer) for n in range(48)])
        if dtype != Q4_0:
            ref_w = w.data[layer].float().numpy().astype(np.float64)
            assert np.array_equal(W, ref_w)
        y = oracle.linear(w, x, layer)
        assert np.allclose(y, x @ W.T, rtol=1e-13, atol=1e-13)


# ---------------- RMSNorm ----------------
def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(300)
    g = np.ones(300, np.float32)
    y = oracle.rmsnorm(x, g, 0.0)
    assert abs(np.sqrt(np.mean(y ** 2)) - 1.0) < 1e-14
    assert np.allclose(oracle.rmsnorm(7.5 * x, g, 0.0), y, rtol=1e-13)
    gg = rng.standard_normal(300).astype(np.float32)
    assert np.allclose(oracle.rmsnorm(x, gg, 0.0), y * gg.astype(np.float64), rtol=1e-13)


def test_rmsnorm_constant_vector_with_eps():
    # a constant vector c has mean square c^2, so the output is c / sqrt(c^2 + eps)
    g = np.ones(16, np.float32)
    y = oracle.rmsnorm(np.full(16, 2.0), g, 1e-6)
    assert np.allclose(y, 2.0 / math.sqrt(4.0 + 1e-6), rtol=1e-15)
    y = oracle.rmsnorm(np.full(16, -0.5), g, 0.25)
    assert np.allclose(y, -0.5 / math.sqrt(0.5), rtol=1e-15)


# ---------------- RoPE ----------------
def test_rope_two_dims_is_plane_rotation_by_pos_radians():
    for pos in (0, 1, 2, 7, 1000):
        v = oracle.rope([1.0, 0.0], pos)
        assert np.allclose(v, [math.cos(pos), math.sin(pos)], atol=1e-12)


def test_rope_rotate_half_pairing_and_invariants():
    hd = 8
    e0 = np.zeros(hd); e0[0] = 1.0
    v = oracle.rope(e0, 1)
    # element 0 pairs with element hd/2 (rotate-half), at unit frequency
    assert np.allclose(v, [math.cos(1), 0, 0, 0, math.sin(1), 0, 0, 0], atol=1e-15)
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    assert np.allclose(oracle.rope(q, 0), q)
    assert abs(np.linalg.norm(oracle.rope(q, 77)) - np.linalg.norm(q)) < 1e-12
    assert np.allclose(oracle.rope(oracle.rope(q, 30), 45), oracle.rope(q, 75), atol=1e-12)
    # attention scores depend only on the relative position
    s1 = oracle.rope(q, 100) @ oracle.rope(k, 60)
    s2 = oracle.rope(q, 1040) @ oracle.rope(k, 1000)
    assert abs(s1 - s2) < 1e-9


# ---------------- GELU ----------------
def test_gelu_exact_form():
    assert oracle.gelu(0.0) == 0.0
    assert abs(oracle.gelu(1.0) - 0.8413447460685429) < 1e-15      # Phi(1)
    assert abs(oracle.gelu(-1.0) - (-0.15865525393145707)) < 1e-15
    for x in (0.3, 1.7, 4.0):
        assert abs(oracle.gelu(x) - oracle.gelu(-x) - x) < 1e-14
    assert abs(oracle.gelu(12.0) - 12.0) < 1e-12
    # matches the library normal CDF
    for x in np.linspace(-5, 5, 41):
        assert abs(oracle.gelu(float(x)) - x * scipy.special.ndtr(x)) < 1e-14


# ---------------- attention ----------------
def test_attention_special_cases():
    rng = np.random.default_rng(4)
    hd = 16
    q = rng.standard_normal(hd)
    K = rng.standard_normal((1, hd)).astype(np.float32)
    V = rng.standard_normal((1, hd)).astype(np.float32)
    assert np.allclose(oracle.attend(q, K, V), V[0])
    # identical keys: uniform weights, output = mean of the values
    K = np.repeat(rng.standard_normal((1, hd)).astype(np.float32), 9, axis=0)
    V = rng.standard_normal((9, hd)).astype(np.float32)
    assert np.allclose(oracle.attend(q, K, V), V.astype(np.float64).mean(0), atol=1e-12)


def test_attention_matches_library_softmax():
    rng = np.random.default_rng(5)
    for n, hd in ((1, 64), (37, 64), (300, 128)):
        q = rng.standard_normal(hd) * 2
        K = rng.standard_normal((n, hd)).astype(np.float32)
        V = rng.standard_normal((n, hd)).astype(np.float32)
        p = scipy.special.softmax(K.astype(np.float64) @ q / math.sqrt(hd))
        assert np.allclose(oracle.attend(q, K, V), p @ V.astype(np.float64), atol=1e-12)


# ---------------- argmax ----------------
def test_argmax_lowest_index_on_ties_and_margin():
    assert oracle.argmax_f32([1.0, 3.0, 3.0, 2.0]) == (1, 0.0)
    t, m = oracle.argmax_f32([0.5, -1.0, 2.25, 2.0])
    assert t == 2 and abs(m - 0.25) < 1e-15
    # values equal once rounded to binary32 count as a tie
    t, _ = oracle.argmax_f32([1.0, 1.0 + 1e-12])
    assert t == 0
