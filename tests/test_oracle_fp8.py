"""Pins for the fp8 KV-cache oracle (CPU only): the e4m3fn codec against
torch's float8_e4m3fn conversions, the token-group quantizer against the
format's rounding bound and hand-worked values, fp8 attention against the
single-precision oracle on pools dequantized here by torch, and the append."""

import numpy as np
import pytest
import torch

import oracle
import oracle.fp8 as of8


def _torch_encode(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).float().numpy()


def test_encoder_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        np.clip(rng.standard_normal(200000).astype(np.float32) * 60, -448, 448),
        rng.uniform(-2.0 ** -5, 2.0 ** -5, 50000).astype(np.float32),        # subnormal range
        np.array([0.0, -0.0, 448.0, -448.0, 1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10,
                  2.0 ** -6, 2.0 ** -6 * (1 - 2.0 ** -5), 15 * 2.0 ** -10, 240.0, 232.0], np.float32),
    ])
    np.testing.assert_array_equal(oracle.e4m3_encode(x), _torch_encode(x))


def test_decoder_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    d, t = oracle.e4m3_decode(codes), _torch_decode(codes)
    assert np.array_equal(np.isnan(d), np.isnan(t)) and np.isnan(d).sum() == 2
    np.testing.assert_array_equal(d[~np.isnan(d)], t[~np.isnan(t)])
    assert oracle.e4m3_decode([0x7E])[0] == 448.0 and oracle.e4m3_decode([0x01])[0] == 2.0 ** -9


def test_quantizer_hand_worked_group():
    # max |x| = 7 gives scale 7 / 448 = 1/64 exactly; x * 64 = [224, -112, 0, 448]
    codes, scale = oracle.quantize_token_groups(np.array([[3.5, -1.75, 0.0, 7.0]], np.float32))
    assert scale[0] == np.float32(1 / 64)
    # 224 = 1.75 * 2^7 -> (7+7)<<3 | 6; -112 = -1.75 * 2^6 -> 0x80 | (6+7)<<3 | 6; 448 -> 0x7E
    assert codes[0].tolist() == [0x76, 0x80 | 0x6E, 0x00, 0x7E]


def test_quantizer_rounding_bound_and_group_max():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((300, 128)) * rng.uniform(0.01, 20, (300, 1))).astype(np.float32)
    x[0] = 0.0  # an all-zero group takes the 1e-10 floor
    codes, scale = oracle.quantize_token_groups(x)
    y = x.astype(np.float64) / scale.astype(np.float64)[:, None]
    v = of8.e4m3_decode(codes)
    a = np.abs(y)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    half_step = np.exp2(e - 4)  # half the code spacing at that magnitude (subnormals: 2^-10)
    assert np.all(np.abs(v - y) <= half_step * (1 + 1e-6) + 448 * 2.0 ** -23)
    gi = np.argmax(np.abs(x[1:]), axis=1)
    top = codes[1:][np.arange(299), gi]
    assert np.all((top & 0x7F) == 0x7E)  # the group maximum lands on +-448
    assert scale[0] == np.float32(1e-10) / np.float32(448) and np.all(codes[0] == 0)


def test_fp8_attention_equals_attention_on_torch_dequantized_pools():
    rng = np.random.default_rng(2)
    P, ps, H_kv, D, B, H_q = 12, 4, 2, 16, 3, 8
    k8 = rng.integers(0, 256, (P, ps, H_kv, D), dtype=np.uint8)
    v8 = rng.integers(0, 256, (P, ps, H_kv, D), dtype=np.uint8)
    for a in (k8, v8):
        a[(a & 0x7F) == 0x7F] = 0x7E  # no NaN codes in a cache written by the quantizer
    ks = rng.uniform(1e-3, 0.1, (P, ps, H_kv)).astype(np.float32)
    vs = rng.uniform(1e-3, 0.1, (P, ps, H_kv)).astype(np.float32)
    bt = rng.permutation(P).reshape(B, P // B)
    lens = np.array([13, 4, 9])
    q = rng.standard_normal((B, H_q, D))
    o, l = oracle.decode_attention_fp8(q, k8, v8, ks, vs, bt, lens, 0.3)
    kd = (_torch_decode(k8) * ks[..., None]).astype(np.float64)
    vd = (_torch_decode(v8) * vs[..., None]).astype(np.float64)
    o2, l2 = oracle.decode_attention(q, kd, vd, bt, lens, 0.3)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(l, l2)


def test_fp8_append_writes_quantized_rows_only():
    rng = np.random.default_rng(3)
    P, ps, H_kv, D, B = 10, 4, 2, 8, 3
    k8 = rng.integers(0, 127, (P, ps, H_kv, D), dtype=np.uint8)
    v8 = rng.integers(0, 127, (P, ps, H_kv, D), dtype=np.uint8)
    ks = rng.uniform(0.1, 1, (P, ps, H_kv)).astype(np.float32)
    vs = rng.uniform(0.1, 1, (P, ps, H_kv)).astype(np.float32)
    bt = np.array([[3, 7, 1], [0, 9, 2], [5, 6, 8]])
    pos = np.array([5, 0, 11])
    kn = rng.standard_normal((B, H_kv, D)).astype(np.float32)
    vn = rng.standard_normal((B, H_kv, D)).astype(np.float32)
    kp, vp, ks2, vs2 = oracle.kv_append_fp8(k8, v8, ks, vs, kn, vn, bt, pos, ps)
    changed = np.zeros((P, ps), bool)
    for b in range(B):
        page, row = bt[b, pos[b] // ps], pos[b] % ps
        changed[page, row] = True
        np.testing.assert_array_equal(kp[page, row], _torch_encode(np.clip(kn[b] / ks2[page, row][:, None], -448, 448)))
        np.testing.assert_array_equal(vp[page, row], _torch_encode(np.clip(vn[b] / vs2[page, row][:, None], -448, 448)))
        np.testing.assert_array_equal(ks2[page, row], np.max(np.abs(kn[b]), axis=1) / np.float32(448))
    np.testing.assert_array_equal(kp[~changed], k8[~changed])
    np.testing.assert_array_equal(vs2[~changed], vs[~changed])


def test_mutation_truncating_encoder_is_caught(monkeypatch):
    real = of8.e4m3_encode

    def truncating(x):
        x = np.asarray(x, np.float64)
        a = np.abs(x)
        e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
        step = np.exp2(e - 3)
        return real(np.trunc(a / step) * step * np.sign(x))  # toward zero, not to nearest even
    monkeypatch.setattr(oracle, "e4m3_encode", truncating)
    with pytest.raises(AssertionError):
        test_encoder_matches_torch_cast()


def _three_terms(x):
    """The three-term e4m3 split of float32 values (hi, then the rounding of
    what hi leaves, then of what both leave), with the oracle's codec; the
    differences are exact (Sterbenz), so float64 reproduces float32."""
    hi = of8.e4m3_decode(of8.e4m3_encode(x))
    r1 = x - hi
    mid = of8.e4m3_decode(of8.e4m3_encode(r1))
    r2 = r1 - mid
    lo = of8.e4m3_decode(of8.e4m3_encode(r2))
    return hi, mid, lo


def test_three_term_e4m3_split_precision():
    """The precision reading of the code-multiplying fp8 kernel: a query
    element (scaled to at most 2^8) or a weighted probability (at most
    2^8.5) split into three e4m3 terms is reconstructed within
    max(2^-12 |x|, 2^-10) (each rounding halves a 3-bit mantissa's spacing;
    below 2^-6 the subnormal grid's 2^-9 spacing sets the floor). Two terms
    would not meet it: the bound is tight enough to catch a dropped term."""
    rng = np.random.default_rng(7)
    mag = np.exp2(rng.uniform(-14.0, 8.5, 400000))
    x = (mag * np.where(rng.random(mag.size) < 0.5, -1.0, 1.0)).astype(np.float32).astype(np.float64)
    x = np.concatenate([x, [256.0, 255.9, 2.0 ** 8.5, 2.0 ** -6, 2.0 ** -9, 3 * 2.0 ** -10, 1.0 + 2.0 ** -11,
                            0.0, 1e-7]])
    hi, mid, lo = _three_terms(x)
    err3 = np.abs(x - (hi + mid + lo))
    bound = np.maximum(2.0 ** -12 * np.abs(x), 2.0 ** -10)
    assert np.all(err3 <= bound * (1 + 1e-9)), float(np.max(err3 / bound))
    err2 = np.abs(x - (hi + mid))
    big = np.abs(x) >= 4.0  # where the relative bound, not the subnormal floor, applies
    assert np.mean(err2[big] > bound[big]) > 0.5  # a split that stops at two terms fails it
