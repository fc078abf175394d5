"""Exact host codecs for the three storage formats of the compressed KV cache.

TEST INFRASTRUCTURE ONLY. This package is the oracle: a slow, plain, float64
CPU statement of what the decode path computes. Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it; the product path (the CUDA library and its binding) never does, and the two
share no code.

Sources for the formats:
  * vibecoco.ai, "DeepSeek V4 agent architecture", section
    "混合注意力：两种压缩，交替使用" (hybrid attention): both layer kinds keep most
    of each KV entry in FP8 and only the RoPE dims in BF16; the lightning
    indexer of CSA runs in FP4.
  * agents-report.net, "DeepSeek-V4：交錯壓縮注意力與低位元 KV 儲存…", section
    "核心技術：交錯壓縮注意力": KV is stored in a mixed low-bit format.
The pages name the formats but not their bit layouts. The layouts used here are
the public ones: OCP FP8 E4M3 ("e4m3fn": bias 7, no infinities, 0x7F/0xFF are
NaN, largest finite 448), OCP MX FP4 E2M1 (values 0, .5, 1, 1.5, 2, 3, 4, 6) and
bfloat16 (the top half of an IEEE binary32).

Every encoder rounds to nearest with ties to even and saturates to the largest
finite magnitude; the sign of a zero result is kept. Rounding is written out as
"divide by the quantum of the value's binade, round to an integer with ties to
even, multiply back", which is exact in float64 because every quantum is a power
of two.
"""
import numpy as np

E4M3_MAX = 448.0
E2M1_MAX = 6.0


def _round_to_grid(a, mant_bits, emin):
    """Round non-negative float64 ``a`` to the nearest number with ``mant_bits``
    fraction bits whose binade exponent is at least ``emin`` (values below
    2**emin share the quantum of binade ``emin``: the subnormal range).
    Ties go to the even multiple of the quantum, i.e. an even last mantissa bit."""
    a = np.asarray(a, dtype=np.float64)
    _, ex = np.frexp(a)                  # a = f * 2**ex with f in [0.5, 1)
    e = np.maximum(ex - 1, emin)         # binade exponent: a in [2**e, 2**(e+1))
    quantum = np.ldexp(1.0, e - mant_bits)
    return np.rint(a / quantum) * quantum  # np.rint rounds half to even


# ----------------------------------------------------------------------------- e4m3

def e4m3_decode(codes):
    """uint8 e4m3 codes -> float64 values (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 3) & 0xF
    M = (c & 7).astype(np.float64)
    mag = np.where(E == 0, M * 2.0 ** -9, (1.0 + M / 8.0) * np.ldexp(1.0, E - 7))
    mag = np.where((E == 15) & ((c & 7) == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(values):
    """float32 values -> uint8 e4m3 codes, round-to-nearest-even, saturating to
    +-448. Inputs must be finite."""
    v = np.asarray(values, dtype=np.float32)
    if not np.all(np.isfinite(v)):
        raise ValueError("e4m3_encode: non-finite input")
    sign = np.signbit(v).astype(np.int64)
    r = np.minimum(_round_to_grid(np.abs(v.astype(np.float64)), 3, -6), E4M3_MAX)
    _, ex = np.frexp(r)
    e = ex - 1
    normal = r >= 2.0 ** -6
    E = np.where(normal, e + 7, 0)
    M = np.where(normal, (r / np.ldexp(1.0, np.where(normal, e, 0)) - 1.0) * 8.0, r / 2.0 ** -9)
    code = (sign << 7) | (E.astype(np.int64) << 3) | M.astype(np.int64)
    return code.astype(np.uint8)


# ----------------------------------------------------------------------------- e2m1

def e2m1_decode(nibbles):
    """4-bit e2m1 codes (0..15, held in any integer array) -> float64."""
    c = np.asarray(nibbles).astype(np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    E = (c >> 1) & 3
    M = (c & 1).astype(np.float64)
    mag = np.where(E == 0, M * 0.5, (1.0 + M / 2.0) * np.ldexp(1.0, E - 1))
    return sign * mag


def e2m1_encode(values):
    """float32 values -> 4-bit e2m1 codes (uint8 0..15), round-to-nearest-even,
    saturating to +-6."""
    v = np.asarray(values, dtype=np.float32)
    if not np.all(np.isfinite(v)):
        raise ValueError("e2m1_encode: non-finite input")
    sign = np.signbit(v).astype(np.int64)
    r = np.minimum(_round_to_grid(np.abs(v.astype(np.float64)), 1, 0), E2M1_MAX)
    _, ex = np.frexp(r)
    e = ex - 1
    normal = r >= 1.0
    E = np.where(normal, e + 1, 0)
    M = np.where(normal, (r / np.ldexp(1.0, np.where(normal, e, 0)) - 1.0) * 2.0, r / 0.5)
    code = (sign << 3) | (E.astype(np.int64) << 1) | M.astype(np.int64)
    return code.astype(np.uint8)


# ----------------------------------------------------------------------------- bf16

def bf16_decode(bits):
    """uint16 bfloat16 bit patterns -> float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_encode(values):
    """float32 values -> uint16 bfloat16 bits, round-to-nearest-even (overflow
    gives infinity, as IEEE rounding does)."""
    v = np.asarray(values, dtype=np.float32)
    r = _round_to_grid(np.abs(v.astype(np.float64)), 7, -126)
    r32 = np.where(np.signbit(v), -r, r).astype(np.float32)  # exact: r has <= 8 significant bits
    return (r32.view(np.uint32) >> 16).astype(np.uint16)
