"""FP8 (e4m3) KV cache with a per-token scale.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

[KVS] "19.2 KV Cache 系统化管理" §19.2.4 (KV cache quantisation): storing the
cache at reduced precision cuts its size directly; its table lists FP8 at one
byte per element, half of FP16/BF16.  In its per-token example each token's
K vector and V vector are scaled on their own, and dequantisation multiplies
the scale back.  The formula itself is missing from the extracted page, so
this module takes the plainest reading of that sentence:

* one scale per token for its whole K vector ([Hkv, D], every head), and one
  for its V vector;
* absmax scaling onto the e4m3 range: ``amax = max|x|``,
  ``code = e4m3(x * (448 / amax))``, ``scale = amax / 448``, and the
  dequantised value is ``e4m3_value(code) * scale``;
* the codes are decided in float32 (the inputs are bf16 or fp32 and widen
  exactly; ``448 / amax``, ``amax / 448`` and each product are single
  correctly rounded float32 operations), rounding to the nearest e4m3 value,
  ties to even, saturating at +-448;
* ``amax == 0`` gives scale 0 and all-zero codes.

e4m3 ("E4M3", the 8-bit format with 4 exponent bits, bias 7, and 3 mantissa
bits, no infinities): sign s, exponent field E, mantissa field m.  E = 0 is
subnormal, ``m * 2**-9``; E = 1..15 is ``(1 + m/8) * 2**(E-7)``, except
E = 15, m = 7, which is NaN.  Largest finite value 448 (E = 15, m = 6),
smallest normal 2**-6, smallest subnormal 2**-9.
"""

import numpy as np

from .attention import paged_decode

E4M3_MAX = 448.0


def e4m3_decode(codes):
    """Value of each e4m3 code (uint8 array) as float64 (exact)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c >> 7, -1.0, 1.0)
    E = (c >> 3) & 15
    m = c & 7
    mag = np.where(E == 0, m * 2.0 ** -9, (8 + m) * np.exp2(E - 10.0))
    val = s * mag
    return np.where((E == 15) & (m == 7), np.nan, val)


def e4m3_encode(x):
    """Nearest e4m3 code to each (finite) value of x, ties to even, with
    magnitudes above 448 saturating to 448.  Works in float64, where every
    step below is exact for float32 inputs."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    neg = np.signbit(np.asarray(x, dtype=np.float64))
    a = np.minimum(a, E4M3_MAX)
    # exponent of the binade holding a (normals), floored at the subnormal one
    _, ex = np.frexp(np.where(a > 0, a, 1.0))          # a = f * 2**ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)
    quantum = np.exp2(e - 3.0)                          # 3 mantissa bits
    val = np.rint(a / quantum) * quantum                # rint: ties to even
    val = np.minimum(val, E4M3_MAX)
    # back to fields (val may have moved up one binade by rounding)
    _, ex2 = np.frexp(np.where(val > 0, val, 1.0))
    e2 = ex2 - 1
    normal = val >= 2.0 ** -6
    E = np.where(normal, e2 + 7, 0)
    m = np.where(normal, val / np.exp2(e2) * 8 - 8, val / 2.0 ** -9)
    code = (E.astype(np.int64) << 3) | m.astype(np.int64)
    code = np.where(val == 0, 0, code)
    return (code | (neg.astype(np.int64) << 7)).astype(np.uint8)


def quantize_token(x):
    """One token's K (or V) vector -> (codes uint8 of x's shape, scale f32),
    per the reading in the module docstring."""
    xf = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(xf))) if xf.size else np.float32(0)
    if amax == 0:
        return np.zeros(xf.shape, np.uint8), np.float32(0)
    inv = np.float32(E4M3_MAX) / amax
    scale = amax / np.float32(E4M3_MAX)
    y = (xf * inv).astype(np.float32)
    return e4m3_encode(y), np.float32(scale)


def dequantize(codes, scales):
    """Pool of codes [NB, bs, H, D] with scales [NB, bs] -> float64 values."""
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[:, :, None, None]


def reshape_and_cache_fp8(key, value, slot_mapping, k_codes, v_codes, k_scale, v_scale):
    """Quantise token t's key and value ([T, Hkv, D], bf16 or fp32 values)
    and write codes and scales into the slot ``slot_mapping[t]`` names
    (block slot // bs, offset slot % bs); negative slots are skipped.  The
    addressing is the append of [KVS] §19.2.3; the quantisation is §19.2.4.
    Returns new arrays (k_codes, v_codes, k_scale, v_scale)."""
    kc, vc = np.array(k_codes, copy=True), np.array(v_codes, copy=True)
    ks, vs = np.array(k_scale, copy=True), np.array(v_scale, copy=True)
    bs = kc.shape[1]
    for t in range(len(slot_mapping)):
        s = int(slot_mapping[t])
        if s < 0:
            continue
        blk, off = s // bs, s % bs
        kc[blk, off], ks[blk, off] = quantize_token(key[t])
        vc[blk, off], vs[blk, off] = quantize_token(value[t])
    return kc, vc, ks, vs


def paged_decode_fp8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens, scale):
    """Paged decode attention over an e4m3 pool: the dequantised pool
    (``e4m3_value(code) * token scale``, exact in float64) fed to the paged
    decode of [KVS] §19.2.3."""
    return paged_decode(q, dequantize(k_codes, k_scale), dequantize(v_codes, v_scale), block_tables,
                        context_lens, scale)
