"""Oracle: exact number formats of the MX block-scaled path (plain, slow, CPU only).

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg
may import this module. The product path never does.

What the pages fix: activations are MXFP8 and weights FP4, multiplied by a block-scaled MMA
("New Deepseek 4.1 flash recipe", post 6, "How it works" item 1: mma.sync.kind::mxf8f6f4
.block_scale "for MXFP8 and FP8 x FP4"; "Dense projections" bullet: "MXFP8"). The pages do not
spell the encodings out, so this file takes the plain OCP Microscaling reading:

* E4M3  - 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities; S.1111.111 is NaN;
          largest finite 448; subnormals m * 2^-9.
* E2M1  - 1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}.
* UE8M0 - unsigned power of two 2^(b - 127); b = 255 is NaN and is never produced here.
* One UE8M0 scale per 32 consecutive elements along the reduction dimension.

Everything here is float64 and works from those closed forms; nothing is shared with the CUDA
path.
"""
from __future__ import annotations

import numpy as np

BLOCK = 32            # elements per UE8M0 scale
E4M3_MAX = 448.0
E2M1_MAX = 6.0
SCALE_MIN_EXP = -127  # UE8M0 byte 0
SCALE_MAX_EXP = 127   # UE8M0 byte 254


# ----------------------------------------------------------------------------------------------
# Decoding (closed forms)
# ----------------------------------------------------------------------------------------------
def e4m3_value(code: int) -> float:
    """Value of one E4M3 code, straight from the bit fields."""
    s = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e2m1_value(code: int) -> float:
    """Value of one E2M1 code (low 4 bits), straight from the bit fields."""
    s = -1.0 if (code >> 3) & 1 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * m * 0.5
    return s * (1.0 + m / 2.0) * 2.0 ** (e - 1)


def ue8m0_value(byte: int) -> float:
    if byte == 255:
        return float("nan")
    return 2.0 ** (byte - 127)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
UE8M0_TABLE = np.array([ue8m0_value(b) for b in range(256)], dtype=np.float64)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """Packed bytes [..., K/2] -> nibble codes [..., K]; element 2m is the LOW nibble of byte m."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    return E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def decode_ue8m0(scales: np.ndarray) -> np.ndarray:
    return UE8M0_TABLE[np.asarray(scales, dtype=np.uint8)]


def dequant_blocks(values: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """values [..., K] (already decoded element values) * 2^scale per 32-block -> float64."""
    v = np.asarray(values, dtype=np.float64)
    k = v.shape[-1]
    nb = scales.shape[-1]
    assert nb * BLOCK >= k
    sc = np.repeat(decode_ue8m0(scales), BLOCK, axis=-1)[..., :k]
    return v * sc


# ----------------------------------------------------------------------------------------------
# Encoding: round to nearest, ties to the even code
# ----------------------------------------------------------------------------------------------
def _encode_magnitude(mag: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Nearest grid index for non-negative magnitudes; ties go to the even index.

    `grid` lists every non-negative finite value of a format in code order (code i has value
    grid[i]); for E4M3 and E2M1 code order is value order and the code LSB is the mantissa LSB,
    so "even code" is round-half-to-even. Magnitudes above the top of the grid saturate to it.
    """
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.searchsorted(grid, mag, side="left")          # grid[hi-1] < mag <= grid[hi]
    hi = np.clip(hi, 1, len(grid) - 1)
    lo = hi - 1
    d_lo = mag - grid[lo]
    d_hi = grid[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(mag >= grid[-1], len(grid) - 1, idx)    # saturate (never reached under the scale rule)
    idx = np.where(mag <= 0.0, 0, idx)
    return idx.astype(np.uint8)


_E4M3_POS = E4M3_TABLE[:127]      # codes 0x00..0x7E: every non-negative finite E4M3 value
_E2M1_POS = E2M1_TABLE[:8]


def encode_e4m3(v: np.ndarray) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    code = _encode_magnitude(np.abs(v), _E4M3_POS)
    return (code | (np.signbit(v).astype(np.uint8) << 7)).astype(np.uint8)


def encode_e2m1(v: np.ndarray) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    code = _encode_magnitude(np.abs(v), _E2M1_POS)
    return (code | (np.signbit(v).astype(np.uint8) << 3)).astype(np.uint8)


# ----------------------------------------------------------------------------------------------
# Block scale rule
# ----------------------------------------------------------------------------------------------
def scale_exponent(amax: np.ndarray, qmax: float) -> np.ndarray:
    """Smallest integer s with amax <= qmax * 2^s, clamped to the UE8M0 range; amax = 0 -> -127.

    Reading of the pages: the FP4 KV writer was changed to "round like DeepSeek's reference
    quantizer" ("New Deepseek 4.1 flash recipe", post 4, "Quality and correctness"), and
    TileKernels "follows DeepSeek's reference term for term" (post 6, "Why TileLang"). The
    plainest reading is the power-of-two scale rounded UP from amax/qmax, so no element is ever
    clipped. Worked exactly: write amax = m * 2^E with m in [1, 2); then for E4M3 (qmax 448 =
    1.75 * 2^8) s = E - 8 + [m > 1.75], and for E2M1 (qmax 6 = 1.5 * 2^2) s = E - 2 + [m > 1.5].
    """
    a = np.asarray(amax, dtype=np.float64)
    frac, ex = np.frexp(a)                # a = frac * 2^ex, frac in [0.5, 1)
    m = frac * 2.0                        # a = m * 2^(ex - 1), m in [1, 2)
    big_e = ex - 1
    qfrac, qex = np.frexp(qmax)
    qm, qe = qfrac * 2.0, qex - 1         # qmax = qm * 2^qe (448 -> 1.75, 8; 6 -> 1.5, 2)
    s = big_e - qe + (m > qm).astype(np.int64)
    s = np.where(a == 0.0, SCALE_MIN_EXP, s)
    return np.clip(s, SCALE_MIN_EXP, SCALE_MAX_EXP).astype(np.int64)


def quantize_blocks(x: np.ndarray, fmt: str) -> tuple[np.ndarray, np.ndarray]:
    """Quantise rows of x (last dim a multiple of 32) to MX codes + UE8M0 scale bytes.

    Per 32-block: s = scale_exponent(max |x|); code = RNE(x * 2^-s). Scaling by a power of two is
    exact, so the only rounding is the element rounding. Returns (codes u8 [..., K] -- one nibble
    per byte for e2m1 -- and scale bytes u8 [..., K/32]).
    """
    x = np.asarray(x, dtype=np.float64)
    k = x.shape[-1]
    assert k % BLOCK == 0
    xb = x.reshape(x.shape[:-1] + (k // BLOCK, BLOCK))
    amax = np.max(np.abs(xb), axis=-1)
    if fmt == "e4m3":
        s = scale_exponent(amax, E4M3_MAX)
        enc = encode_e4m3
    elif fmt == "e2m1":
        s = scale_exponent(amax, E2M1_MAX)
        enc = encode_e2m1
    else:
        raise ValueError(fmt)
    scaled = xb * np.ldexp(1.0, -s)[..., None]
    codes = enc(scaled).reshape(x.shape)
    return codes, (s + 127).astype(np.uint8)


# ----------------------------------------------------------------------------------------------
# bf16 helpers (numpy has no bf16 dtype: bf16 travels as uint16 bit patterns)
# ----------------------------------------------------------------------------------------------
def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """float64 -> nearest bf16 (ties to even), returned as float64 values. Single rounding."""
    v = np.asarray(v, dtype=np.float64)
    _, ex = np.frexp(v)                           # |v| in [2^(ex-1), 2^ex)
    ex = np.maximum(ex, -125)                     # below 2^-126 the bf16 quantum is fixed (subnormals)
    q = np.ldexp(1.0, ex - 8)                     # 8 significant bits
    r = np.rint(v / q) * q                        # np.rint: ties to even
    return np.where(v == 0.0, v, r)


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    r = round_to_bf16(v).astype(np.float32)       # exact: a bf16 value is an fp32 value
    return (r.view(np.uint32) >> 16).astype(np.uint16)
