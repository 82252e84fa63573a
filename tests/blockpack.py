"""Test-side block packers: build Q4_K / Q6_K / Q8_0 blocks from chosen field
values, written as the inverse of the layout reading (GGUF convention) and
independently of the oracle's unpackers, so hand-built blocks with known
weights can pin the oracle."""
import numpy as np


def f16_bits(v: float) -> int:
    return int(np.array([v], dtype=np.float16).view(np.uint16)[0])


def pack_q4k(d: float, dmin: float, sc, m, q) -> np.ndarray:
    """sc, m: 8 six-bit values; q: 256 four-bit quants (weight order)."""
    sc = [int(v) for v in sc]
    m = [int(v) for v in m]
    assert all(0 <= v < 64 for v in sc + m)
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (256,) and q.min() >= 0 and q.max() < 16
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = np.array([d], dtype=np.float16).view(np.uint8)
    blk[2:4] = np.array([dmin], dtype=np.float16).view(np.uint8)
    s = np.zeros(12, dtype=np.int64)
    for j in range(4):
        s[j] |= sc[j]                      # low 6 bits of byte j: scale j
        s[j + 4] |= m[j]                   # low 6 bits of byte j+4: min j
    for j in range(4, 8):
        s[j + 4] |= (sc[j] & 15) | ((m[j] & 15) << 4)   # byte j+4: low nibbles
        s[j - 4] |= (sc[j] >> 4) << 6      # top 2 bits of byte j-4: scale j high bits
        s[j] |= (m[j] >> 4) << 6           # top 2 bits of byte j: min j high bits
    blk[4:16] = s.astype(np.uint8)
    qs = np.zeros(128, dtype=np.int64)
    for i in range(256):
        grp, within = divmod(i, 64)
        if within < 32:
            qs[32 * grp + within] |= q[i]
        else:
            qs[32 * grp + within - 32] |= q[i] << 4
    blk[16:144] = qs.astype(np.uint8)
    return blk


def pack_q6k(d: float, sc, q6) -> np.ndarray:
    """sc: 16 int8 scales; q6: 256 six-bit codes 0..63 (weight = code - 32)."""
    sc = np.asarray(sc, dtype=np.int64)
    q6 = np.asarray(q6, dtype=np.int64)
    assert sc.shape == (16,) and sc.min() >= -128 and sc.max() <= 127
    assert q6.shape == (256,) and q6.min() >= 0 and q6.max() < 64
    ql = np.zeros(128, dtype=np.int64)
    qh = np.zeros(64, dtype=np.int64)
    for i in range(256):
        half, r = divmod(i, 128)
        quarter, l = divmod(r, 32)
        lo, hi = q6[i] & 15, q6[i] >> 4
        byte = 64 * half + (quarter & 1) * 32 + l
        ql[byte] |= lo if quarter < 2 else lo << 4
        qh[32 * half + l] |= hi << (2 * quarter)
    blk = np.zeros(210, dtype=np.uint8)
    blk[0:128] = ql.astype(np.uint8)
    blk[128:192] = qh.astype(np.uint8)
    blk[192:208] = sc.astype(np.int8).view(np.uint8)
    blk[208:210] = np.array([d], dtype=np.float16).view(np.uint8)
    return blk


def pack_q80(d: float, q) -> np.ndarray:
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (32,) and q.min() >= -128 and q.max() <= 127
    blk = np.zeros(34, dtype=np.uint8)
    blk[0:2] = np.array([d], dtype=np.float16).view(np.uint8)
    blk[2:34] = q.astype(np.int8).view(np.uint8)
    return blk
