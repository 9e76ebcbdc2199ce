"""Number formats used by the data path, in fp64 (test infrastructure only).

* bf16 -- GEMM outputs and activations are stored in bf16 (page "Blackwell 上的
  DeepGEMM FusedMoE（vLLM）", §1.1 table rows 6-8: mm1_out, mm2_out and the
  output are bf16).  Rounding is round-to-nearest-even (reading: the pages do
  not state it).
* e4m3fn -- FP8 activations/weights (same page, §2.6.2 views the activation
  buffer as ``torch.float8_e4m3fn``): 1 sign, 4 exponent (bias 7), 3 mantissa
  bits, no infinities, max 448.  Conversion reading: round-to-nearest-even with
  saturation to +-448.
* E2M1 -- MXFP4 weights (same page, TL;DR table: "E2M1 + E8M0/32"): 1 sign,
  2 exponent (bias 1), 1 mantissa bit.
* E8M0 -- power-of-two scale 2^(e-127); e = 255 is NaN and never produced.
* UE8M0 activation scale -- the fp32 scale rounded UP to a power of two (the
  page's FLOAT32_CEIL_UE8M0 format, §2.8(f)).
"""
from __future__ import annotations

import numpy as np

BF16_MAX = float.fromhex("0x1.fe00000000000p+127")
E4M3_MAX = 448.0
E2M1_MAX = 6.0


def round_fp32(v):
    """Round fp64 values to the nearest fp32 (IEEE round-to-nearest-even)."""
    return np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)


def _round_to_bits(v, sig_bits: int, min_quantum_exp: int):
    """Round to a binary format with ``sig_bits`` significant bits whose
    smallest quantum (subnormal spacing) is 2**min_quantum_exp; ties to even."""
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)                       # v = m * 2**e with 0.5 <= |m| < 1
    q_exp = np.maximum(e - sig_bits, min_quantum_exp)
    return np.ldexp(np.round(np.ldexp(v, -q_exp)), q_exp)   # np.round: half to even


def round_bf16(v):
    """fp64 -> nearest bf16 (8 significant bits, subnormal quantum 2^-133),
    ties to even, overflow to +-inf."""
    v = np.asarray(v, dtype=np.float64)
    r = _round_to_bits(v, 8, -133)
    return np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, v), r)


def round_e4m3(v):
    """fp64 -> nearest e4m3fn value (4 significant bits, subnormal quantum
    2^-9), ties to even, saturating to +-448."""
    r = _round_to_bits(v, 4, -9)
    return np.clip(r, -E4M3_MAX, E4M3_MAX)


def minifloat_decode(codes, exp_bits: int, man_bits: int, bias: int):
    """Decode sign/exponent/mantissa bit fields of a small float format.
    Exponent field 0 is subnormal; no special values are handled here."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where((c >> (exp_bits + man_bits)) & 1, -1.0, 1.0)
    ef = (c >> man_bits) & ((1 << exp_bits) - 1)
    mf = c & ((1 << man_bits) - 1)
    sub = mf.astype(np.float64) * 2.0 ** (1 - bias - man_bits)
    nrm = (1.0 + mf / 2.0 ** man_bits) * np.ldexp(1.0, (ef - bias).astype(np.int64))
    return sign * np.where(ef == 0, sub, nrm)


def _e4m3_decode_fields(codes):
    c = np.asarray(codes, dtype=np.int64)
    v = minifloat_decode(c, 4, 3, 7)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


_E4M3_TABLE = _e4m3_decode_fields(np.arange(256))


def e4m3_decode(codes):
    """uint8 e4m3fn codes -> fp64 values; 0x7F/0xFF decode to NaN.  Each code
    is decoded from its bit fields (``minifloat_decode``); uint8 arrays look
    the same values up in the table of all 256 codes."""
    c = np.asarray(codes)
    if c.dtype == np.uint8:
        return _E4M3_TABLE[c]
    return _e4m3_decode_fields(c)


def e4m3_encode(values):
    """Exact e4m3fn values (as produced by ``round_e4m3``) -> uint8 codes."""
    v = np.asarray(values, dtype=np.float64)
    a = np.abs(v)
    sign = np.where(np.signbit(v), 0x80, 0)
    _, e = np.frexp(a)
    exp_unb = e - 1                                 # a = 1.m * 2**exp_unb
    normal = a >= 2.0 ** -6
    biased = np.where(normal, exp_unb + 7, 0)
    man = np.where(normal, np.ldexp(a, -exp_unb) * 8 - 8, np.ldexp(a, 9))
    if not np.all(man == np.round(man)):
        raise ValueError("value not representable in e4m3fn")
    code = sign | (biased.astype(np.int64) << 3) | man.astype(np.int64)
    code = np.where(a == 0, sign, code)
    return code.astype(np.uint8)


def _e2m1_decode_fields(codes):
    return minifloat_decode(np.asarray(codes, dtype=np.int64) & 0xF, 2, 1, 1)


_E2M1_TABLE = _e2m1_decode_fields(np.arange(256))


def e2m1_decode(codes):
    """4-bit E2M1 codes -> fp64 values: +-{0, .5, 1, 1.5, 2, 3, 4, 6} (the
    high nibble of a byte is ignored; uint8 arrays use the table of the
    field decode)."""
    c = np.asarray(codes)
    if c.dtype == np.uint8:
        return _E2M1_TABLE[c]
    return _e2m1_decode_fields(c)


_E8M0_TABLE = np.ldexp(1.0, np.arange(256) - 127)


def e8m0_decode(codes):
    """E8M0 scale codes -> 2**(code - 127)."""
    c = np.asarray(codes)
    if c.dtype == np.uint8:
        return _E8M0_TABLE[c]
    return np.ldexp(1.0, c.astype(np.int64) - 127)


def unpack_fp4(packed, k: int):
    """[..., k/2] uint8 with the even element in the low nibble -> [..., k] codes."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (k,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def ceil_pow2(s):
    """Round positive values up to a power of two (exact)."""
    s = np.asarray(s, dtype=np.float64)
    m, e = np.frexp(s)
    return np.where(m == 0.5, s, np.ldexp(1.0, e))
