"""CPU model of the multi-launch mxfp4 kernels' code layout (ffn_mxfp4.cu).

A quad's four lanes (c = 0..3) load the four 16-byte scale blocks of a 64-byte
chunk of a weight row, one block per lane, and a 4x4 word transpose inside the
quad (an own-word rotation, three shuffles, a second rotation) leaves lane c
with word c (bytes 4c..4c+3, codes 8c..8c+7) of every block.  The model checks
that the transpose delivers exactly that word for every lane and block, that
each MMA pair of a block then sums that block's 32 codes only (so one scale
multiplies its fp32 sum), that the staged token chunk each lane reads holds the
elements its codes meet, and that the new row swizzle spreads a quarter-warp's
16-byte loads over all 32 banks."""
from __future__ import annotations

import itertools


def own_rotation(words, c):
    """Rotate a lane's four words left by c (two conditional rotations)."""
    a = words[1:] + words[:1] if c & 1 else list(words)
    return a[2:] + a[:2] if c & 2 else a


def quad_transpose(quad):
    """quad[lane] = the four words lane `lane` loaded (block `lane` of the chunk)."""
    q = [own_rotation(quad[c], c) for c in range(4)]
    out = []
    for c in range(4):
        q0 = q[c][0]
        v1 = q[(c - 1) & 3][1]  # shuffle i takes word i of lane (c - i) & 3
        v2 = q[(c - 2) & 3][2]
        v3 = q[(c - 3) & 3][3]
        r1, r2 = c & 1, c & 2
        a0 = v1 if r1 else q0
        a1 = q0 if r1 else v3
        a2 = v3 if r1 else v2
        a3 = v2 if r1 else v1
        out.append([a2, a3, a0, a1] if r2 else [a0, a1, a2, a3])
    return out


def test_quad_transpose_gives_word_c_of_every_block():
    quad = [[(blk, w) for w in range(4)] for blk in range(4)]
    out = quad_transpose(quad)
    for c in range(4):
        assert out[c] == [(qb, c) for qb in range(4)], c


def test_transpose_is_a_permutation_for_distinct_values():
    vals = list(range(16))
    for perm in itertools.islice(itertools.permutations(vals), 0, 200, 7):
        quad = [list(perm[4 * b:4 * b + 4]) for b in range(4)]
        out = quad_transpose(quad)
        assert sorted(v for row in out for v in row) == sorted(vals)
        for c in range(4):
            assert out[c] == [quad[qb][c] for qb in range(4)]


def mma_slots(c, byte):
    """k-slots of the block's MMA pair that byte `byte` (0..3) of lane c's word
    feeds: bytes 0, 1 -> MMA 0, bytes 2, 3 -> MMA 1; even byte -> slots
    {2c, 2c+1}, odd byte -> {2c+8, 2c+9} (one fp16x2 register per byte)."""
    mma = byte >> 1
    base = 2 * c if byte % 2 == 0 else 2 * c + 8
    return mma, (base, base + 1)


def test_each_mma_pair_sums_one_block_and_meets_the_right_tokens():
    # lane c holds codes 8c .. 8c+7 of block qb: byte b of its word = codes 8c+2b, 8c+2b+1
    for qb in range(4):
        seen = {0: {}, 1: {}}
        for c in range(4):
            for b in range(4):
                mma, slots = mma_slots(c, b)
                codes = (8 * c + 2 * b, 8 * c + 2 * b + 1)
                for s, code in zip(slots, codes):
                    assert s not in seen[mma]
                    seen[mma][s] = (qb, code)
        for mma in (0, 1):
            assert sorted(seen[mma]) == list(range(16))  # all 16 k-slots of the MMA
            assert {blk for blk, _ in seen[mma].values()} == {qb}  # one block only
        codes = sorted(code for mma in (0, 1) for _, code in seen[mma].values())
        assert codes == list(range(32))  # the pair covers the whole block
    # the token chunk lane c reads for block qb of chunk ch holds elements
    # 128 ch + 32 qb + 8c .. +8, and its 16-byte load gives the B registers in
    # the same slot order: register pair (x, y) for MMA 0, (z, w) for MMA 1
    for ch, qb, c in itertools.product(range(3), range(4), range(4)):
        q = ch * 16 + qb * 4 + c
        first = 8 * q
        assert first == 128 * ch + 32 * qb + 8 * c


def swz_mx(q, j):
    return q ^ ((j & 1) << 2)


def test_row_swizzle_spreads_a_quarter_warp_over_all_banks():
    """A quarter-warp is lanes g = 2i, 2i+1 (token rows n, n+1) x c = 0..3, reading
    chunk 4 qb + c of its row; rows are whole multiples of 128 bytes apart."""
    for cpr in (8, 40, 256, 512):  # chunks per staged row (d / 8)
        for ch in range(cpr // 16 + 1):
            for qb in range(4):
                q0 = ch * 16 + qb * 4
                if q0 + 3 >= cpr:
                    continue
                for n in range(0, 16, 2):
                    groups = set()
                    for row in (n, n + 1):
                        for c in range(4):
                            chunk = row * cpr + swz_mx(q0 + c, row)
                            assert swz_mx(q0 + c, row) < cpr
                            groups.add(chunk % 8)  # 16-byte bank group within 128 bytes
                    assert len(groups) == 8
