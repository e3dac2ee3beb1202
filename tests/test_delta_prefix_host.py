"""Host check of the in-register prefix sums the DELTA kernel uses (no GPU
needed): for a packed word of 2- or 4-bit column deltas, the kernel forms the
doubled running column of its entries from a few shifts, masks, one multiply
and byte extracts. This mirrors that arithmetic in numpy (32-bit wrap) for
every lane position of both decodes and compares it with the running sums of
the fields taken one by one, on random words and on the extremes (all fields
0, all fields at their maximum)."""
import numpy as np
import pytest

M32 = 0xFFFFFFFF


def byte(x, i):
    return (x >> (8 * i)) & 0xFF


def prefix4(w):
    """4-bit fields: P2 byte i = 2 x fields 0..2i+1, Q2 byte i = 2 x 0..2i."""
    lo = (w << 1) & 0x1E1E1E1E
    hi = (w >> 3) & 0x1E1E1E1E
    p2 = ((lo + hi) * 0x01010101) & M32
    return p2, (p2 - hi) & M32


def prefix2(w):
    """2-bit fields, adjacent pairs first summed into nibbles: P2 byte i =
    2 x fields 0..4i+3, Q2 byte i = 2 x fields 0..4i+1."""
    g = (w & 0x33333333) + ((w >> 2) & 0x33333333)
    lo = (g << 1) & 0x1E1E1E1E
    hi = (g >> 3) & 0x1E1E1E1E
    p2 = ((lo + hi) * 0x01010101) & M32
    return p2, (p2 - hi) & M32


def fields(w, bits):
    cap = (1 << bits) - 1
    return [(w >> (bits * k)) & cap for k in range(32 // bits)]


def words(bits):
    rng = np.random.default_rng(bits)
    out = [0, M32] + [int(v) for v in rng.integers(0, 1 << 32, 2000, dtype=np.uint64)]
    return out


@pytest.mark.parametrize("bits", [2, 4])
def test_lane_columns_match_running_sums(bits):
    for w in words(bits):
        run = np.cumsum(fields(w, bits)) * 2          # doubled running column
        if bits == 4:
            p2, q2 = prefix4(w)
            for q in range(4):                      # four lanes a word, two entries each
                assert byte(q2, q) == run[2 * q] and byte(p2, q) == run[2 * q + 1]
        else:
            p2, q2 = prefix2(w)
            for q in range(8):                      # eight lanes a word, two entries each
                t = p2 if q & 1 else q2
                o1 = byte(t, q >> 1)
                o0 = o1 - ((w >> (4 * q + 1)) & 6)
                assert o1 == run[2 * q + 1] and o0 == run[2 * q]
            # the lane-per-word decode: entries 4i+1 and 4i+3 from Q2 / P2,
            # 4i and 4i+2 by taking their upper neighbour back off
            for i in range(4):
                assert byte(q2, i) == run[4 * i + 1] and byte(p2, i) == run[4 * i + 3]
                assert byte(q2, i) - ((w >> (8 * i + 1)) & 6) == run[4 * i]
                assert byte(p2, i) - ((w >> (8 * i + 5)) & 6) == run[4 * i + 2]
        assert run[-1] < 256                        # no carry between bytes
