"""Host-side models of two invariants the batch-1 kernels rely on, checked
exhaustively over the sizes they meet (no GPU):

* the one-launch FFN's grid barrier: one 32-bit word, CTA 0 adds
  2^31 - (grid - 1) and every other CTA adds 1; from a word whose low 31
  bits are zero its top bit must flip exactly at the last arrival, in any
  arrival order, and leave the low bits zero for the next call;
* the bulk staging of x in place: the raw rows land at the top of the
  padded x area and are moved into 68-float group slots in rounds of
  2 * nct units (load the round, barrier, store it); no store may reach a
  raw value that a later round still has to read.
The index formulas restate the kernels' (column of value i of group G for
Q6_K: 256 blk + 128 h + 32 (i / 16) + l0 + i % 16)."""
import itertools

import numpy as np
import pytest

TOP = 0x80000000
MASK = 0xFFFFFFFF


def _run_barrier(start, grid, order):
    """arrivals in `order`; returns the arrival index at which the top bit
    first differs from every arriving CTA's old value's top bit, and the end value"""
    word = start
    olds = {}
    for n, cta in enumerate(order):
        inc = (TOP - (grid - 1)) & MASK if cta == 0 else 1
        olds[cta] = word
        word = (word + inc) & MASK
        released = [c for c, o in olds.items() if (word ^ o) & TOP]
        if released:
            return n, released, word, olds
    return None, [], word, olds


@pytest.mark.parametrize("grid", [1, 2, 3, 5, 10, 152, 304])
def test_grid_barrier_flips_exactly_at_the_last_arrival(grid):
    rng = np.random.default_rng(grid)
    orders = [list(range(grid)), list(range(grid))[::-1]] + [list(rng.permutation(grid)) for _ in range(20)]
    if grid <= 5:
        orders += [list(p) for p in itertools.permutations(range(grid))]
    for start in (0, TOP):
        for order in orders:
            n, released, end, olds = _run_barrier(start, grid, order)
            assert n == grid - 1, (start, order, n)           # nobody released before everyone arrived
            assert sorted(released) == list(range(grid))       # then every waiter sees the flip
            assert end & (TOP - 1) == 0 and (end ^ start) & TOP  # low bits back to zero, top bit flipped


def test_grid_barrier_needs_zero_low_bits():
    """a word that does not start with zero low bits releases too early
    (why lq_ffn_one_launch asks for a zeroed word)"""
    n, _, _, _ = _run_barrier(0x7FFFFFFF, 4, [1, 2, 3, 0])
    assert n == 0


def _qxcol(q6k, G, i):
    if q6k:
        blk, gm = G >> 2, G & 3
        h, l0 = gm >> 1, 16 * (gm & 1)
        return 256 * blk + 128 * h + 32 * (i >> 4) + l0 + (i & 15)
    return 64 * G + i


@pytest.mark.parametrize("q6k", [False, True])
@pytest.mark.parametrize("B", [1, 2, 4])
def test_bulk_staging_rounds_never_overwrite_unread_raw_values(q6k, B):
    for U in [4, 8, 12, 20, 28, 40, 64, 128, 160, 224]:
        cols = 64 * U
        for nct in [128, 160, 192, 224, 256, 288, 320]:
            units = B * U * 4
            base_raw = B * U * 4                        # raw rows start 4 floats per group above the slots
            written = np.zeros(B * U * 68, dtype=bool)  # float positions stored so far
            for base in range(0, units, 2 * nct):       # one round
                round_units = [e for e in range(base, min(base + 2 * nct, units))]
                # loads of the round: every float must still be raw (not yet overwritten)
                for e in round_units:
                    b, r = divmod(e, U * 4)
                    G, q = r >> 2, r & 3
                    src = base_raw + b * cols + _qxcol(q6k, G, 16 * q)
                    assert not written[src:src + 16].any(), (q6k, B, U, nct, e)
                # stores of the round, after the barrier
                for e in round_units:
                    b, r = divmod(e, U * 4)
                    G, q = r >> 2, r & 3
                    dst = (b * U + G) * 68 + 16 * q
                    written[dst:dst + 16] = True
            # every slot's 64 values were written exactly where the items read them
            slots = written.reshape(B * U, 68)
            assert slots[:, :64].all() and not slots[:, 64:].any()
