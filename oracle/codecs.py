"""Number formats used by the cache: bf16 and fp8 e4m3 (oracle; test infrastructure only).

[P2] "DeepSeek V4 稀疏注意力完全解剖", 第三层 (multiple quantisations: bf16 KV for
prefill, token-wise fp8 for decode) and [P1] §4.1 (the indexer "can use FP8").
The pages name the formats but not their encodings; the encodings follow the
bfloat16 bit layout (1 sign, 8 exponent, 7 fraction bits) and the OCP 8-bit
floating point specification, E4M3 variant (bias 7, no infinities, max 448,
S.1111.111 is NaN).

All rounding is round-to-nearest, ties-to-even, written as ``np.rint`` on the
significand (numpy's rint rounds half to even).

[P2] 第三层 also names an fp4 indexer cache ("indexer 用 fp4") without its encoding; it follows
the OCP Microscaling (MX) FP4 E2M1 element (bias 1, values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their
negatives, no infinities or NaN), two codes per byte with the even element in the low nibble, one
fp32 scale per row (amax / 6) as for the e4m3 rows.
"""
import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6      # 2^-6 is the smallest normal magnitude
E4M3_SUBNORMAL_QUANTUM = 2.0 ** -9


def bf16_round(x):
    """Round to the nearest bfloat16 value (ties to even); returns float64.

    A bfloat16 has an 8-bit significand (1 implicit + 7 stored).  frexp gives
    x = m * 2^e with 0.5 <= |m| < 1, so the significand is m * 2^8 rounded to an
    integer.  Overflow and bf16 subnormals do not occur for the cache's values.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def bf16_decode(bits):
    """bfloat16 bit patterns (uint16) to float64: the bits are the high half of an IEEE binary32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_encode(x):
    """float64 values to bfloat16 bit patterns (uint16), rounding to nearest even first."""
    r = bf16_round(x).astype(np.float32)          # exact: a bf16 value is a binary32 value
    return (r.view(np.uint32) >> 16).astype(np.uint16)


def e4m3_decode(codes):
    """Decode e4m3 bytes to float64: S EEEE MMM, bias 7.

    E == 0: subnormal, (-1)^S * 2^-6 * M/8.  E in 1..15: (-1)^S * 2^(E-7) * (1 + M/8),
    except E == 15, M == 7 which is NaN.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    E = (c >> 3) & 0xF
    M = c & 0x7
    mag = np.where(E == 0,
                   np.ldexp(M / 8.0, E4M3_MIN_NORMAL_EXP),
                   np.ldexp(1.0 + M / 8.0, E - 7))
    val = np.where(s == 1, -mag, mag)
    return np.where((E == 15) & (M == 7), np.nan, val)


def e4m3_round(x):
    """Round float64 values onto the e4m3 grid, RNE, saturating to +-448.

    Normal range (|x| >= 2^-6): 4 significant bits, so the significand m * 2^4 is
    rounded.  Subnormal range: multiples of 2^-9.  A result above 448 (including a
    round-up to 480) is clamped to 448, the "saturate to finite" conversion.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    m, e = np.frexp(a)
    normal = np.ldexp(np.rint(m * 16.0), e - 4)
    sub = np.rint(a / E4M3_SUBNORMAL_QUANTUM) * E4M3_SUBNORMAL_QUANTUM
    r = np.where(a < 2.0 ** E4M3_MIN_NORMAL_EXP, sub, normal)
    r = np.minimum(r, E4M3_MAX)
    return np.where(np.signbit(x), -r, r)


_E4M3_POSITIVE = e4m3_decode(np.arange(0x7F, dtype=np.uint8))   # codes 0..126, increasing


def e4m3_encode(x):
    """Encode float64 values to e4m3 bytes (RNE, saturating).  NaN input is not supported.

    The sign bit is kept when a negative value rounds to zero (code 0x80, -0).
    """
    r = e4m3_round(x)
    code = np.searchsorted(_E4M3_POSITIVE, np.abs(r)).astype(np.uint8)
    return np.where(np.signbit(r), code | 0x80, code).astype(np.uint8)


def fp8_row_scale(v):
    """Per-row scale for token-wise / entry-wise fp8: amax / 448 stored as fp32 (1 if amax == 0).

    The stored scale is an fp32 number, so the oracle rounds it to fp32 exactly as
    it will be read back.
    """
    v = np.asarray(v, dtype=np.float64)
    amax = np.max(np.abs(v), axis=-1)
    scale = np.where(amax > 0, amax / E4M3_MAX, 1.0)
    return scale.astype(np.float32).astype(np.float64)


def fp8_quantize_rows(v):
    """Quantise rows to (e4m3 codes, fp32 scale) with code = e4m3(v / scale)."""
    v = np.asarray(v, dtype=np.float64)
    scale = fp8_row_scale(v)
    codes = e4m3_encode(v / scale[..., None])
    return codes, scale


def fp8_dequantize_rows(codes, scale):
    """Row value = scale * decode(code), the token-wise fp8 reading of a cache row."""
    return e4m3_decode(codes) * np.asarray(scale, dtype=np.float64)[..., None]


# ---- fp4 e2m1 ------------------------------------------------------------------------------------
E2M1_MAX = 6.0


def e2m1_decode(codes):
    """Decode e2m1 codes (0..15) to float64: S EE M, bias 1; E == 0 is subnormal, 0.5 * M."""
    c = np.asarray(codes, dtype=np.int64) & 0xF
    s = (c >> 3) & 1
    E = (c >> 1) & 0x3
    M = c & 1
    mag = np.where(E == 0, 0.5 * M, np.ldexp(1.0 + M / 2.0, E - 1))
    return np.where(s == 1, -mag, mag)


def e2m1_round(x):
    """Round float64 values onto the e2m1 grid, RNE, saturating to +-6.

    Normal range (|x| >= 1): 2 significant bits, so the significand m * 2^2 of frexp is rounded.
    Subnormal range: multiples of 0.5.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    m, e = np.frexp(a)
    normal = np.ldexp(np.rint(m * 4.0), e - 2)
    sub = np.rint(a / 0.5) * 0.5
    r = np.where(a < 1.0, sub, normal)
    r = np.minimum(r, E2M1_MAX)
    return np.where(np.signbit(x), -r, r)


_E2M1_POSITIVE = e2m1_decode(np.arange(8))   # codes 0..7, increasing


def e2m1_encode(x):
    """Encode float64 values to e2m1 codes (uint8 0..15; RNE, saturating; the sign kept for -0)."""
    r = e2m1_round(x)
    code = np.searchsorted(_E2M1_POSITIVE, np.abs(r)).astype(np.uint8)
    return np.where(np.signbit(r), code | 0x8, code).astype(np.uint8)


def fp4_pack(codes):
    """[..., d] e2m1 codes -> [..., d / 2] bytes: element 2j in the low nibble, 2j + 1 in the high one."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def fp4_unpack(packed):
    """[..., d / 2] bytes -> [..., d] e2m1 codes."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def fp4_row_scale(v):
    """Per-row scale of fp4 rows: amax / 6 stored as fp32 (1 if amax == 0)."""
    v = np.asarray(v, dtype=np.float64)
    amax = np.max(np.abs(v), axis=-1)
    scale = np.where(amax > 0, amax / E2M1_MAX, 1.0)
    return scale.astype(np.float32).astype(np.float64)


def fp4_quantize_rows(v):
    """Quantise rows to (packed e2m1 bytes [..., d / 2], fp32 scale) with code = e2m1(v / scale)."""
    v = np.asarray(v, dtype=np.float64)
    scale = fp4_row_scale(v)
    return fp4_pack(e2m1_encode(v / scale[..., None])), scale


def fp4_dequantize_rows(packed, scale):
    """Row value = scale * e2m1(code)."""
    return e2m1_decode(fp4_unpack(packed)) * np.asarray(scale, dtype=np.float64)[..., None]
