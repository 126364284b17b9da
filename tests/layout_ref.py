"""A second, independent reading of the byte layouts written out in
include/qmv.h, used by the tests to build weight groups from chosen fields
(scales, codes) and to read fields back.  It decodes nothing into values: the
tests compute expected values from the fields themselves."""
from __future__ import annotations

import numpy as np

CODEBOOK = np.array([-127, -104, -83, -65, -49, -35, -22, -10,
                     1, 13, 25, 38, 53, 69, 89, 113], dtype=np.int64)


def f16_bits(v) -> int:
    return int(np.array(v, dtype=np.float64).astype(np.float16).view(np.uint16))


def f16_value(bits) -> float:
    return float(np.array(bits, dtype=np.uint16).view(np.float16).astype(np.float64))


def _set_bits(buf: bytearray, byte0: int, bit: int, nbits: int, v: int):
    for i in range(nbits):
        b = bit + i
        idx = byte0 + b // 8
        if (v >> i) & 1:
            buf[idx] |= 1 << (b % 8)
        else:
            buf[idx] &= ~(1 << (b % 8)) & 0xFF


def _get_bits(buf, byte0: int, bit: int, nbits: int) -> int:
    v = 0
    for i in range(nbits):
        b = bit + i
        v |= ((buf[byte0 + b // 8] >> (b % 8)) & 1) << i
    return v


def _put_codes(buf: bytearray, off: int, codes):
    """32 four-bit codes of one sub-block: byte i = c_i | c_{i+16} << 4."""
    for i in range(16):
        buf[off + i] = (int(codes[i]) & 0xF) | ((int(codes[i + 16]) & 0xF) << 4)


def _get_codes(buf, off: int):
    return [buf[off + (i % 16)] >> (0 if i < 16 else 4) & 0xF for i in range(32)]


def pack_q8_0(d_bits, q) -> bytes:
    """One Q8_0 group: d_bits[8] fp16 patterns, q[8][32] int8."""
    g = bytearray(272)
    for j in range(8):
        g[2 * j] = d_bits[j] & 0xFF
        g[2 * j + 1] = d_bits[j] >> 8
        for i in range(32):
            off = 16 * j + i if i < 16 else 128 + 16 * j + (i - 16)
            g[16 + off] = int(q[j][i]) & 0xFF
    return bytes(g)


def pack_q4_k(d_bits, dmin_bits, sc, m, q) -> bytes:
    """One Q4_K group: fp16 d, dmin; sc[8], m[8] in [0,63]; q[8][32] in [0,15]."""
    g = bytearray(144)
    g[0], g[1] = d_bits & 0xFF, d_bits >> 8
    g[2], g[3] = dmin_bits & 0xFF, dmin_bits >> 8
    for j in range(8):
        _set_bits(g, 4, 12 * j, 6, int(sc[j]))
        _set_bits(g, 4, 12 * j + 6, 6, int(m[j]))
        _put_codes(g, 16 + 16 * j, q[j])
    return bytes(g)


def pack_q5_k(d_bits, dmin_bits, sc, m, q) -> bytes:
    """One Q5_K group: fp16 d, dmin; sc[8], m[8] in [0,63]; q[8][32] in [0,31]
    (low four bits in the nibble area at 48, fifth bits at 16, 4 bytes per
    sub-block, bit i for weight i)."""
    g = bytearray(176)
    g[0], g[1] = d_bits & 0xFF, d_bits >> 8
    g[2], g[3] = dmin_bits & 0xFF, dmin_bits >> 8
    for j in range(8):
        _set_bits(g, 4, 12 * j, 6, int(sc[j]))
        _set_bits(g, 4, 12 * j + 6, 6, int(m[j]))
        _put_codes(g, 48 + 16 * j, [int(v) & 15 for v in q[j]])
        for i in range(32):
            _set_bits(g, 16 + 4 * j, i, 1, int(q[j][i]) >> 4)
    return bytes(g)


def unpack_q5_k(g):
    g = bytes(g)
    d, dmin = g[0] | (g[1] << 8), g[2] | (g[3] << 8)
    sc = [_get_bits(g, 4, 12 * j, 6) for j in range(8)]
    m = [_get_bits(g, 4, 12 * j + 6, 6) for j in range(8)]
    q = [[c | (_get_bits(g, 16 + 4 * j, i, 1) << 4) for i, c in enumerate(_get_codes(g, 48 + 16 * j))]
         for j in range(8)]
    return d, dmin, sc, m, q


def _q6_pos(j, i):
    """(byte offset of the word, bit) of the top two bits of weight i of block j."""
    e, word = i % 16, i // 16
    return 16 + 8 * j + 4 * word, 8 * (e % 4) + 2 * (e // 4)


def pack_q6_k(d_bits, sc, q) -> bytes:
    """One Q6_K group: fp16 d; sc[16] in [0,127] (one per 16 weights);
    q[256] in [0,63] (w = d sc (q - 32)), stored as v = (q - 32) mod 64."""
    g = bytearray(208)
    g[0], g[1] = d_bits & 0xFF, d_bits >> 8
    for i in range(16):
        _set_bits(g, 2, 7 * i, 7, int(sc[i]))
    for j in range(8):
        v = [(int(q[32 * j + i]) - 32) % 64 for i in range(32)]
        _put_codes(g, 80 + 16 * j, [x & 15 for x in v])
        for i in range(32):
            off, bit = _q6_pos(j, i)
            _set_bits(g, off, bit, 2, v[i] >> 4)
    return bytes(g)


def unpack_q6_k(g):
    g = bytes(g)
    d = g[0] | (g[1] << 8)
    sc = [_get_bits(g, 2, 7 * i, 7) for i in range(16)]
    q = []
    for j in range(8):
        low = _get_codes(g, 80 + 16 * j)
        for i in range(32):
            off, bit = _q6_pos(j, i)
            v = low[i] | (_get_bits(g, off, bit, 2) << 4)
            q.append((v + 32) % 64)
    return d, sc, q


def pack_q8_g(d_bits, q, gs) -> bytes:
    """One Q8 group with a scale per gs (64 or 128) weights: d_bits[8] fp16
    patterns, q[8 * gs] int8; 8 * gs weights, each 256 of them laid out as a
    Q8_0 payload."""
    n = 8 * gs
    g = bytearray(16 + n)
    for s_ in range(8):
        g[2 * s_], g[2 * s_ + 1] = d_bits[s_] & 0xFF, d_bits[s_] >> 8
    for el in range(n):
        half, j, i = el // 256, (el // 32) % 8, el % 32
        off = 16 * j + i if i < 16 else 128 + 16 * j + (i - 16)
        g[16 + 256 * half + off] = int(q[el]) & 0xFF
    return bytes(g)


def unpack_q8_g(g, gs):
    g = bytes(g)
    n = 8 * gs
    d = [g[2 * s_] | (g[2 * s_ + 1] << 8) for s_ in range(8)]
    q = []
    for el in range(n):
        half, j, i = el // 256, (el // 32) % 8, el % 32
        off = 16 * j + i if i < 16 else 128 + 16 * j + (i - 16)
        v = g[16 + 256 * half + off]
        q.append(v - 256 if v > 127 else v)
    return d, q


def pack_iq4_xs(d_bits, ls, c) -> bytes:
    """One IQ4_XS group (2 superblocks): d_bits[2]; ls[2][8] in [0,63];
    c[2][8][32] codebook indices."""
    g = bytearray(272)
    for s in range(2):
        g[8 * s] = d_bits[s] & 0xFF
        g[8 * s + 1] = d_bits[s] >> 8
        for j in range(8):
            _set_bits(g, 8 * s + 2, 6 * j, 6, int(ls[s][j]))
            _put_codes(g, 16 + 128 * s + 16 * j, c[s][j])
    return bytes(g)


def unpack_q8_0(g):
    g = [int(v) for v in bytes(bytearray(g))]
    d_bits = [g[2 * j] | (g[2 * j + 1] << 8) for j in range(8)]
    off = lambda j, i: 16 * j + i if i < 16 else 128 + 16 * j + (i - 16)
    q = [[int(np.int8(np.uint8(g[16 + off(j, i)]))) for i in range(32)] for j in range(8)]
    return d_bits, q


def unpack_q4_k(g):
    g = [int(v) for v in bytes(bytearray(g))]
    d_bits = g[0] | (g[1] << 8)
    dmin_bits = g[2] | (g[3] << 8)
    sc = [_get_bits(g, 4, 12 * j, 6) for j in range(8)]
    m = [_get_bits(g, 4, 12 * j + 6, 6) for j in range(8)]
    q = [_get_codes(g, 16 + 16 * j) for j in range(8)]
    return d_bits, dmin_bits, sc, m, q


def unpack_iq4_xs(g):
    g = [int(v) for v in bytes(bytearray(g))]
    d_bits = [g[8 * s] | (g[8 * s + 1] << 8) for s in range(2)]
    ls = [[_get_bits(g, 8 * s + 2, 6 * j, 6) for j in range(8)] for s in range(2)]
    c = [[_get_codes(g, 16 + 128 * s + 16 * j) for j in range(8)] for s in range(2)]
    return d_bits, ls, c


def q8_codes_natural(q):
    """Codes of the library's Q8 activation layout [n][K] back in element
    order.  Within every 256-element group (8 blocks of 32), element p of
    block l is stored at (p // 16) * 128 + l * 16 + p % 16 (the first halves
    of the 8 blocks, then the second halves), as include/qmv.h states."""
    q = np.asarray(q)
    n, K = q.shape
    l = np.arange(8)[:, None]
    p = np.arange(32)[None, :]
    pos = ((p // 16) * 128 + l * 16 + p % 16).reshape(-1)   # natural index l * 32 + p -> stored position
    g = q.reshape(n, K // 256, 256)
    return g[:, :, pos].reshape(n, K)
