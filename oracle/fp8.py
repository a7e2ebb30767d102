"""fp8 (e4m3fn) KV cache: token-group quantization, the byte codec, and decode
attention over a quantized cache. TEST INFRASTRUCTURE ONLY (see the package
docstring).

tokenspeed 딥다이브 (fiv.co.kr), section 6-4 (GPU DSL and quantization, the
pseudo code of the token-group quantize kernel): a token group's scale is its
largest magnitude over the format's largest finite value (with a floor of
1e-10), the group is divided by the scale, clamped to the finite range and
cast to float8_e4m3fn; the reconstruction is the code's value times the scale,
in float32.

Readings (listed in the design notes): a token group is one token's row of one
kv head (D values), so the cache keeps one float32 scale per (page, row, kv
head) for K and one for V; the arithmetic of the page's pseudo code is float32
(PyTorch's default), so the scale and the division are float32 operations
rounded to nearest even, and the cast rounds to nearest even.

The e4m3fn format (OCP 8-bit floating point, "E4M3" with the "fn" finite
variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent
field 0 holds subnormals m * 2^-9; S.1111.111 is NaN (no infinities); the
largest finite value is 448 = 1.75 * 2^8.
"""

from __future__ import annotations

import numpy as np

from .attention import decode_attention, mla_decode_attention

E4M3_MAX = 448.0
SCALE_FLOOR = np.float32(1e-10)


def e4m3_decode(codes) -> np.ndarray:
    """Value of each e4m3fn byte as float64 (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = s * val
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def e4m3_encode(x) -> np.ndarray:
    """Round finite values with |x| <= 448 to the nearest e4m3fn code, ties to even.

    Works in float64, where every step below is exact for float32 inputs.
    """
    x = np.asarray(x, dtype=np.float64)
    if np.any(~np.isfinite(x)) or np.any(np.abs(x) > E4M3_MAX):
        raise ValueError("e4m3_encode takes finite values of magnitude <= 448")
    sign = np.signbit(x).astype(np.int64) << 7
    a = np.abs(x)
    out = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    # subnormal range: multiples of 2^-9 (rounding up to 8 * 2^-9 gives the smallest normal, code 8)
    out[sub] = np.rint(a[sub] * 2.0 ** 9).astype(np.int64)
    nrm = ~sub
    if np.any(nrm):
        an = a[nrm]
        e = np.floor(np.log2(an)).astype(np.int64)
        # guard log2 rounding at exact powers of two
        e = np.where(an < np.exp2(e.astype(np.float64)), e - 1, e)
        e = np.where(an >= np.exp2(e.astype(np.float64) + 1.0), e + 1, e)
        m = np.rint((an / np.exp2(e.astype(np.float64)) - 1.0) * 8.0).astype(np.int64)
        carry = m == 8
        e = np.where(carry, e + 1, e)
        m = np.where(carry, 0, m)
        out[nrm] = ((e + 7) << 3) | m
    return (sign | out).astype(np.uint8)


def quantize_token_groups(x):
    """Quantize groups along the last axis: returns (codes uint8 [..., D], scale float32 [...]).

    scale = max(max |group|, 1e-10) / 448, codes = e4m3(clamp(group / scale, -448, 448)),
    with the scale and the division as float32 operations.

    Pinned by: the codec against torch's float8_e4m3fn cast, the page's bound on the
    reconstruction (every element within half a code step of its group's scaled value),
    the group maximum landing on +-448 exactly, and a hand-worked group.
    """
    x = np.asarray(x, dtype=np.float32)
    gmax = np.max(np.abs(x), axis=-1)
    scale = np.maximum(gmax, SCALE_FLOOR).astype(np.float32) / np.float32(E4M3_MAX)
    y = (x / scale[..., None]).astype(np.float32)
    y = np.clip(y, np.float32(-E4M3_MAX), np.float32(E4M3_MAX))
    return e4m3_encode(y), scale.astype(np.float32)


def dequantize(codes, scale) -> np.ndarray:
    """The page's reconstruction: the code's value times its group's scale, in float32."""
    v = e4m3_decode(codes).astype(np.float32)
    return (v * np.asarray(scale, dtype=np.float32)[..., None]).astype(np.float32)


def kv_append_fp8(k_pool, v_pool, k_scale, v_scale, k_new, v_new, block_table, positions,
                  page_size):
    """Quantize one new token's K/V rows per sequence into an fp8 paged cache.

    Same placement as :func:`oracle.kv_append` (SwiftLLM page, section 3.1);
    each (token, kv head) row is one token group. Returns new arrays; inputs
    are not modified.

    Args: pools uint8 [P, ps, H_kv, D]; scales float32 [P, ps, H_kv];
    k_new, v_new [B, H_kv, D] (float; bf16 inputs are passed widened).
    """
    kp, vp = np.array(k_pool, copy=True), np.array(v_pool, copy=True)
    ks, vs = np.array(k_scale, copy=True), np.array(v_scale, copy=True)
    kq, kqs = quantize_token_groups(k_new)
    vq, vqs = quantize_token_groups(v_new)
    for b in range(len(positions)):
        pos = int(positions[b])
        page = int(block_table[b][pos // page_size])
        row = pos % page_size
        kp[page, row], ks[page, row] = kq[b], kqs[b]
        vp[page, row], vs[page, row] = vq[b], vqs[b]
    return kp, vp, ks, vs


def decode_attention_fp8(q, k_pool, v_pool, k_scale, v_scale, block_table, seq_lens, scale):
    """GQA decode over an fp8 cache: attention (fp64) over the page's float32
    reconstruction of every cached row.

    Pinned by: equality with :func:`oracle.decode_attention` on pools
    dequantized independently in the test, and the codec/quantizer pins.
    """
    kd = dequantize(k_pool, k_scale).astype(np.float64)
    vd = dequantize(v_pool, v_scale).astype(np.float64)
    return decode_attention(q, kd, vd, block_table, seq_lens, scale)


def mla_decode_attention_fp8(q_codes, q_scale, kv_codes, kv_scale, block_table, seq_lens, scale, d_v):
    """Absorbed-MLA decode on the fp8 input path: attention (fp64) over the
    page's float32 reconstruction of the query rows and the latent rows.

    TokenSpeed deep dive (wth2jhl.online), section 1: the MLA decode kernel
    takes bf16, fp16 or fp8 inputs. Reading (listed in the design notes): on
    the fp8 path both inputs are e4m3fn codes with token-group scales by the
    rule of tokenspeed 딥다이브 (fiv.co.kr), section 6-4, one group per row:
    one float32 scale per (sequence, head) query row of 576 values and one
    per cached latent row of 576 values. The values are the first ``d_v``
    columns of the same reconstructed latent rows.

    Args:
        q_codes: uint8 [B, H, Dqk]; q_scale: float32 [B, H];
        kv_codes: uint8 [P, page_size, Dqk]; kv_scale: float32 [P, page_size].

    Returns:
        (O [B, H, d_v] float64, LSE [B, H] float64).

    Pinned by: equality with :func:`oracle.mla_decode_attention` on inputs
    dequantized independently in the test (torch's float8_e4m3fn conversion),
    and a planted mistake (the latent scale left out of the values) caught.
    """
    qd = dequantize(q_codes, q_scale).astype(np.float64)
    cd = dequantize(kv_codes, kv_scale).astype(np.float64)
    return mla_decode_attention(qd, cd, block_table, seq_lens, scale, d_v)
