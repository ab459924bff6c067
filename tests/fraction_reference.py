"""Exact-rational brute force for tiny inputs: an independent third check of
the C oracle.  Written separately from it (bit-level field extraction over the
whole 96-bit scale word, Python integers and fractions.Fraction throughout) so
that a slip in either implementation shows up as a disagreement.

Follows SKaiNET PR #562 "SIMD-fused Q4_K matmul kernel + Q4KMatmulKernel SPI",
section "Pipeline", and SKaiNET issue #1138 "[ternary-f32] Phase 2 …",
section "Tasks".
"""
from fractions import Fraction


def fp16(bits: int) -> Fraction:
    sign = -1 if bits >> 15 else 1
    e = (bits >> 10) & 31
    mant = bits & 1023
    assert e != 31, "Inf/NaN are outside the generator's range"
    if e == 0:
        return sign * Fraction(mant, 1 << 24)
    return sign * Fraction(1024 + mant, 1 << 10) * Fraction(2) ** (e - 15)


def _bits(word: int, lo: int, n: int) -> int:
    return (word >> lo) & ((1 << n) - 1)


def scales_mins(packed: bytes):
    """Eight (sc, m) pairs from the 12 packed bytes, read as one 96-bit
    little-endian word.  Byte i occupies bits 8i..8i+7."""
    word = int.from_bytes(bytes(packed), "little")
    out = []
    for s in range(8):
        if s < 4:
            sc = _bits(word, 8 * s, 6)
            m = _bits(word, 8 * (s + 4), 6)
        else:
            sc = _bits(word, 8 * (s + 4), 4) + (_bits(word, 8 * (s - 4) + 6, 2) << 4)
            m = _bits(word, 8 * (s + 4) + 4, 4) + (_bits(word, 8 * s + 6, 2) << 4)
        out.append((sc, m))
    return out


def block_values(blk: bytes):
    """The 256 exact values of one block."""
    blk = bytes(blk)
    d = fp16(blk[0] | blk[1] << 8)
    dmin = fp16(blk[2] | blk[3] << 8)
    sm = scales_mins(blk[4:16])
    qs = blk[16:144]
    vals = [None] * 256
    for j in range(4):
        for l in range(32):
            byte = qs[32 * j + l]
            for e, q in ((64 * j + l, byte % 16), (64 * j + 32 + l, byte // 16)):
                sc, m = sm[e // 32]
                vals[e] = d * sc * q - dmin * m
    return vals


def q4k_matmul(x_rows, W_rows, K: int):
    """y[t][o] exactly, with each weight rounded once to fp32 first (the
    oracle's dequantize-to-FP32 step).  x_rows: list of lists of floats,
    W_rows: list of byte strings."""
    import numpy as np
    nb = K // 256
    y = []
    for xt in x_rows:
        row_out = []
        for wrow in W_rows:
            acc = Fraction(0)
            for b in range(nb):
                vals = block_values(wrow[144 * b:144 * (b + 1)])
                for e, v in enumerate(vals):
                    w32 = Fraction(float(np.float32(float(v))))  # v is exact in double
                    acc += Fraction(float(xt[256 * b + e])) * w32
            row_out.append(acc)
        y.append(row_out)
    return y


def ternary_codes(row: bytes, K: int):
    codes = []
    for i in range(K):
        field = (row[i // 4] >> (2 * (i % 4))) & 3
        codes.append(field - 1)
    return codes


def q4_0_block_values(blk: bytes):
    """The 32 exact values of one Q4_0 block: fp16 d, then 16 bytes whose low
    nibbles are elements 0..15 and high nibbles elements 16..31; w = d·(q − 8)."""
    blk = bytes(blk)
    d = fp16(blk[0] | blk[1] << 8)
    vals = [None] * 32
    for l, byte in enumerate(blk[2:18]):
        vals[l] = d * (byte % 16 - 8)
        vals[16 + l] = d * (byte // 16 - 8)
    return vals


def q4_0_matmul(x_rows, W_rows, K: int):
    """y[t][o] exactly from Q4_0 rows (each weight exact in fp32 already)."""
    y = []
    for xt in x_rows:
        row_out = []
        for wrow in W_rows:
            acc = Fraction(0)
            for b in range(K // 32):
                for e, v in enumerate(q4_0_block_values(wrow[18 * b:18 * (b + 1)])):
                    acc += Fraction(float(xt[32 * b + e])) * v
            row_out.append(acc)
        y.append(row_out)
    return y


def q6k_block_values(blk: bytes):
    """The 256 exact values of one Q6_K block, read bit by bit: the whole ql
    area and qh area as little-endian integers, nibble and 2-bit fields taken
    at computed bit offsets."""
    blk = bytes(blk)
    ql = int.from_bytes(blk[0:128], "little")
    qh = int.from_bytes(blk[128:192], "little")
    scales = [b - 256 if b > 127 else b for b in blk[192:208]]
    d = fp16(blk[208] | blk[209] << 8)
    vals = []
    for v in range(256):
        n, g, l = v // 128, (v % 128) // 32, v % 32
        byte = 64 * n + (32 if g % 2 else 0) + l
        lo = _bits(ql, 8 * byte + (4 if g >= 2 else 0), 4)
        hi = _bits(qh, 8 * (32 * n + l) + 2 * g, 2)
        vals.append(d * scales[8 * n + 2 * g + l // 16] * (lo + 16 * hi - 32))
    return vals


def q6k_matmul(x_rows, W_rows, K: int):
    """y[t][o] exactly from Q6_K rows (each weight exact in fp32 already)."""
    y = []
    for xt in x_rows:
        row_out = []
        for wrow in W_rows:
            acc = Fraction(0)
            for b in range(K // 256):
                for e, v in enumerate(q6k_block_values(wrow[210 * b:210 * (b + 1)])):
                    acc += Fraction(float(xt[256 * b + e])) * v
            row_out.append(acc)
        y.append(row_out)
    return y
