"""Shared-memory index arithmetic of two kernels, restated and checked on the
CPU: every copy lands in its own slot, every read finds the value that was
written for it, and a warp's reads spread over the 32 banks.

  * the weight-gradient operand quantisation (quant_t): a chunk of 128 rows x
    64 bf16 columns is copied as 16-byte pieces, piece k of row r at
    r*128 + 16*(k ^ (r/16 % 8)); a quantising thread (qt = tid % 8,
    cp = tid / 8) reads the 32-bit word holding columns 2cp, 2cp+1 of rows
    16qt .. 16qt+15;
  * the gathered dispatch of GEMM 1: lane l copies the eight 16-byte pieces of
    rows l, l+32, l+64, l+96 of a 128-row x 128-byte tile, piece c of row m at
    m*128 + 16*(c ^ (m % 8)), the 128-byte swizzle TMA writes and the MMA's
    shared-memory descriptor reads.
"""
import numpy as np


def test_quant_t_chunk_layout():
    chunk = 128 * 128
    owner = np.full(chunk // 16, -1, np.int64)
    # copies: thread tid moves piece k = tid % 8 of rows tid/8 + 32i
    for tid in range(256):
        k, rr = tid & 7, tid >> 3
        for i in range(4):
            r = rr + 32 * i
            place = r * 128 + ((k ^ ((r >> 4) & 7)) * 16)
            assert place % 16 == 0 and 0 <= place < chunk
            assert owner[place // 16] == -1, "two pieces in one slot"
            owner[place // 16] = r * 8 + k
    assert (owner >= 0).all()
    # reads: the word of columns 2cp, 2cp+1 in row r is byte 4*(cp % 4) of piece cp // 4
    for tid in range(256):
        qt, cp = tid & 7, tid >> 3
        word = (((cp >> 2) ^ qt) * 16) + (cp & 3) * 4
        for i in range(16):
            r = 16 * qt + i
            addr = r * 128 + word
            assert owner[addr // 16] == r * 8 + (cp >> 2)
            assert addr % 16 == (cp & 3) * 4
    # banks: for each i, a warp's 32 reads hit 32 different banks
    for w in range(8):
        for i in range(16):
            banks = set()
            for lane in range(32):
                tid = 32 * w + lane
                qt, cp = tid & 7, tid >> 3
                word = (((cp >> 2) ^ qt) * 16) + (cp & 3) * 4
                banks.add(((16 * qt + i) * 128 + word) // 4 % 32)
            assert len(banks) == 32


def test_gathered_rows_follow_the_128_byte_swizzle():
    tile = 128 * 128
    seen = np.zeros(tile // 16, np.int64)
    for lane in range(32):
        for i in range(4):
            m = lane + 32 * i
            for c in range(8):
                place = m * 128 + ((c ^ (m & 7)) * 16)
                # the 128-byte swizzle: 16-byte unit c of row m within its 1024-byte atom
                atom, row_in_atom = divmod(m, 8)
                assert place == atom * 1024 + row_in_atom * 128 + 16 * (c ^ row_in_atom)
                seen[place // 16] += 1
    assert (seen == 1).all()
