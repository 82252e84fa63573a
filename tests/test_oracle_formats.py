"""Pins of the oracle's block codecs against facts outside the oracle: the
pages' block sizes, IEEE fp16 (numpy's converter), hand-built blocks with
closed-form weights, and exact rational arithmetic for the one fp32 rounding."""
from fractions import Fraction

import numpy as np
import pytest

import synth
from blockpack import f16_bits, pack_q4k, pack_q6k, pack_q80
from conftest import golden_lines

Q4_K, Q6_K, Q8_0 = 1, 2, 3
FMT = {"Q4_K": Q4_K, "Q6_K": Q6_K, "Q8_0": Q8_0}


def test_block_sizes_match_pages(orc):
    rows = [l.split() for l in golden_lines("formats.txt")]
    assert len(rows) == 3
    for name, nbytes, nelems in rows:
        f = FMT[name]
        assert orc.block_bytes(f) == int(nbytes)
        assert orc.block_elems(f) == int(nelems)
        # the generator lays out rows with the same sizes
        assert synth.row_bytes(f, 4 * int(nelems)) == 4 * int(nbytes)


def test_half_decode_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    assert np.array_equal(np.signbit(got[finite]), np.signbit(ref[finite]))


def _dq(orc, fmt, blk, cols=None):
    blk = np.ascontiguousarray(blk, dtype=np.uint8).reshape(1, -1)
    cols = cols or orc.block_elems(fmt) * (blk.size // orc.block_bytes(fmt))
    return orc.dequant(fmt, blk, 1, cols)[0]


# ---------------------------------------------------------------- Q8_0

def test_q80_closed_form(orc):
    q = np.arange(-127, 128, 8)[:32]
    q = np.concatenate([q, np.zeros(32 - q.size, dtype=np.int64)])
    for d in (0.5, 1.0, 0.0009765625, 2.0 ** -24, 65504.0, -3.0):
        w = _dq(orc, Q8_0, pack_q80(d, q))
        assert np.array_equal(w, (np.float64(np.float16(d)) * q).astype(np.float32))


def test_q80_extremes(orc):
    q = np.array([-128, 127] * 16)
    w = _dq(orc, Q8_0, pack_q80(1.0, q))
    assert np.array_equal(w, q.astype(np.float32))


# ---------------------------------------------------------------- Q4_K

def test_q4k_all_ones(orc):
    w = _dq(orc, Q4_K, pack_q4k(1.0, 0.0, [1] * 8, [0] * 8, np.ones(256, dtype=int)))
    assert np.array_equal(w, np.ones(256, dtype=np.float32))


def test_q4k_zero_scale_gives_minus_min(orc):
    m = [0, 1, 7, 15, 16, 31, 48, 63]
    q = np.random.default_rng(1).integers(0, 16, 256)
    w = _dq(orc, Q4_K, pack_q4k(0.75, 0.25, [0] * 8, m, q))
    for j in range(8):
        assert np.all(w[32 * j:32 * j + 32] == np.float32(-0.25 * m[j]))


def test_q4k_positions(orc):
    """a single nonzero quant at each of the 256 positions lands on that weight."""
    for i in range(256):
        q = np.zeros(256, dtype=int)
        q[i] = 5
        w = _dq(orc, Q4_K, pack_q4k(1.0, 0.0, [1] * 8, [0] * 8, q))
        nz = np.flatnonzero(w)
        assert nz.tolist() == [i] and w[i] == 5.0


def test_q4k_positions_raw_bytes(orc):
    """byte qs[32g+l]: low nibble is weight 64g+l, high nibble weight 64g+32+l
    (checked on raw bytes, without the test packer)."""
    base = pack_q4k(1.0, 0.0, [1] * 8, [0] * 8, np.zeros(256, dtype=int))
    for byte in range(128):
        g, l = divmod(byte, 32)
        blk = base.copy()
        blk[16 + byte] = 0x31      # low nibble 1, high nibble 3
        w = _dq(orc, Q4_K, blk)
        assert w[64 * g + l] == 1.0 and w[64 * g + 32 + l] == 3.0
        assert np.count_nonzero(w) == 2


def test_q4k_high_scale_fields_hand_typed(orc):
    """A Q4_K block typed byte by byte (no packer): d = dmin = 1.0 (fp16
    0x3C00), the twelve scale bytes below, and in every sub-block quants 0 in
    the first 16 weights and 2 in the last 16, so a sub-block decodes to -m
    and then 2 sc - m.  Sub-blocks 0..3 take sc, m from the low six bits of
    bytes 0..3 and 4..7; sub-blocks 4..7 take the low four bits from bytes
    8..11 (sc: low nibble, m: high nibble) and the top two bits from the top
    bits of bytes 0..3 (sc) and 4..7 (m).  The expected fields are worked
    out by hand in the comments."""
    scales = bytes([0xC1, 0x82, 0x43, 0x04,     # sc0..3 = 1, 2, 3, 4; top bits 3, 2, 1, 0
                    0x85, 0x46, 0xC7, 0x08,     # m0..3 = 5, 6, 7, 8; top bits 2, 1, 3, 0
                    0x9A, 0x3B, 0xFC, 0x0D])    # sc4..7 low 10, 11, 12, 13; m4..7 low 9, 3, 15, 0
    expect = {0: (1, 5), 1: (2, 6), 2: (3, 7), 3: (4, 8),
              4: (10 + 16 * 3, 9 + 16 * 2),     # (58, 41)
              5: (11 + 16 * 2, 3 + 16 * 1),     # (43, 19)
              6: (12 + 16 * 1, 15 + 16 * 3),    # (28, 63)
              7: (13 + 16 * 0, 0 + 16 * 0)}     # (13, 0)
    qs = bytes(([0x00] * 16 + [0x22] * 16) * 4)   # byte 32g + l: low nibble sub-block 2g, high 2g + 1
    blk = np.frombuffer(bytes([0x00, 0x3C, 0x00, 0x3C]) + scales + qs, dtype=np.uint8)
    assert blk.size == 144
    w = _dq(orc, Q4_K, blk)
    for j, (sc, m) in expect.items():
        assert (w[32 * j:32 * j + 16] == -m).all(), j
        assert (w[32 * j + 16:32 * j + 32] == 2 * sc - m).all(), j


def test_q4k_scale_min_roundtrip(orc):
    """random and exhaustive 6-bit scales/mins, recovered through two blocks:
    all q = 0 gives w = -dmin*m, all q = 1 gives w = d*sc - dmin*m."""
    r = np.random.default_rng(2)
    cases = [r.integers(0, 64, 16) for _ in range(300)]
    for v in range(64):                        # every value in every field position
        cases.append(np.full(16, v))
    for c in cases:
        sc, m = c[:8], c[8:]
        w0 = _dq(orc, Q4_K, pack_q4k(1.0, 1.0, sc, m, np.zeros(256, dtype=int)))
        w1 = _dq(orc, Q4_K, pack_q4k(1.0, 1.0, sc, m, np.ones(256, dtype=int)))
        for j in range(8):
            assert np.all(w0[32 * j:32 * j + 32] == -m[j])
            assert np.all(w1[32 * j:32 * j + 32] == sc[j] - m[j])


def test_q4k_uniform_bytes_give_uniform_fields(orc):
    """the generator's uniform scale bytes give every 6-bit value (bijective packing)."""
    W = synth.q4k(synth.rng(3), 64, 256 * 8)
    D = orc.dequant(Q4_K, W, 64, 256 * 8)
    assert np.isfinite(D).all()
    # weights of one sub-block take at most 16 distinct values (one per quant)
    for r in range(4):
        for j in range(8):
            assert np.unique(D[r, 32 * j:32 * j + 32]).size <= 16


def test_q4k_single_rounding(orc):
    """w = fp32(d*sc*q - dmin*m): the exact rational value rounded once to fp32."""
    r = np.random.default_rng(4)
    for _ in range(200):
        d = float(np.float16(r.uniform(1e-4, 2e-3)))
        dmin = float(np.float16(r.uniform(1e-4, 2e-3)))
        sc, m = r.integers(0, 64, 8), r.integers(0, 64, 8)
        q = r.integers(0, 16, 256)
        w = _dq(orc, Q4_K, pack_q4k(d, dmin, sc, m, q))
        for i in r.integers(0, 256, 16):
            j = i // 32
            exact = Fraction(d) * int(sc[j]) * int(q[i]) - Fraction(dmin) * int(m[j])
            # float(Fraction) is correctly rounded to fp64; this value fits in
            # 51 bits, so the fp64 is exact and the cast to fp32 rounds once.
            assert Fraction(float(exact)) == exact
            assert w[i] == np.float32(float(exact))


def test_q4k_subnormal_d(orc):
    d = 2.0 ** -24 * 3            # fp16 subnormal
    w = _dq(orc, Q4_K, pack_q4k(d, 0.0, [63] * 8, [0] * 8, np.full(256, 15)))
    assert np.all(w == np.float32(d * 63 * 15))


# ---------------------------------------------------------------- Q6_K

def test_q6k_positions(orc):
    for i in range(256):
        q6 = np.full(256, 32)          # weight 0 everywhere
        q6[i] = 32 + 7
        w = _dq(orc, Q6_K, pack_q6k(1.0, np.ones(16, dtype=int), q6))
        nz = np.flatnonzero(w)
        assert nz.tolist() == [i] and w[i] == 7.0


def test_q6k_positions_raw_bytes(orc):
    """raw-byte reading of the layout, without the test packer: ql[64h+l] low
    nibble -> weight 128h+l, ql[64h+32+l] low -> 128h+32+l, ql[64h+l] high ->
    128h+64+l, ql[64h+32+l] high -> 128h+96+l; qh[32h+l] bit pairs 0-1, 2-3,
    4-5, 6-7 are the high bits of those four weights."""
    base = np.zeros(210, dtype=np.uint8)
    base[192:208] = 1
    base[208:210] = np.array([1.0], dtype=np.float16).view(np.uint8)
    for h in range(2):
        for l in range(32):
            for quarter in range(4):
                blk = base.copy()
                byte = 64 * h + (quarter & 1) * 32 + l
                blk[byte] = 0x05 if quarter < 2 else 0x50
                blk[128 + 32 * h + l] = 0b10 << (2 * quarter)   # high bits = 2 -> +32
                w = _dq(orc, Q6_K, blk)
                target = 128 * h + 32 * quarter + l
                expect = np.full(256, -32.0, dtype=np.float32)
                expect[target] = (5 | (2 << 4)) - 32
                # untouched weights sharing a byte keep code 0 -> -32
                assert np.array_equal(w, expect), (h, l, quarter)


def test_q6k_scales_per_16(orc):
    sc = np.array([-128, 127, -1, 1, 0, 5, -63, 63, 2, -2, 17, -17, 100, -100, 64, -64])
    w = _dq(orc, Q6_K, pack_q6k(0.5, sc, np.full(256, 33)))    # q = 1
    assert np.array_equal(w, np.repeat(0.5 * sc, 16).astype(np.float32))


def test_q6k_code_roundtrip_and_extremes(orc):
    r = np.random.default_rng(5)
    for _ in range(100):
        q6 = r.integers(0, 64, 256)
        w = _dq(orc, Q6_K, pack_q6k(1.0, np.ones(16, dtype=int), q6))
        assert np.array_equal(w, (q6 - 32).astype(np.float32))
    w = _dq(orc, Q6_K, pack_q6k(2.0, np.full(16, -128), np.array([0, 63] * 128)))
    assert np.array_equal(w, np.array([2.0 * -128 * -32, 2.0 * -128 * 31] * 128, dtype=np.float32))


def test_q6k_generator_scale_range(orc):
    W = synth.q6k(synth.rng(6), 32, 512)
    sc = W.reshape(32, 2, 210)[:, :, 192:208].view(np.int8)
    assert sc.min() >= -63 and sc.max() <= 63


# ---------------------------------------------------------------- multi-block rows

@pytest.mark.parametrize("fmt", [Q4_K, Q6_K, Q8_0])
def test_rows_are_concatenated_blocks(orc, fmt):
    """a row of nb blocks dequantizes block by block (row stride nb * block bytes)."""
    cols = orc.block_elems(fmt) * 5
    W = synth.weights(synth.rng(7), fmt, 3, cols)
    D = orc.dequant(fmt, W, 3, cols)
    bb, be = orc.block_bytes(fmt), orc.block_elems(fmt)
    for r in range(3):
        for b in range(5):
            one = _dq(orc, fmt, W[r, b * bb:(b + 1) * bb])
            assert np.array_equal(D[r, b * be:(b + 1) * be], one)
