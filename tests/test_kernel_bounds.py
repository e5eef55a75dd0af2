"""CPU models of the single-launch kernels' index arithmetic (compute-
sanitizer is not available).  bf16: the shared-memory plan, the routing tables with
the shared expert and its split gate/up entries, and the extreme index of
every shared-memory, TMA, global-weight, h and ys access a unit makes, checked
against the size of its buffer.  The formulas are the kernel's (layer_fused.cu:
fused_plan, slot_addr, the producer's copies, the consumers' fragment loads and
stores).  Block-scaled weights, mxfp4 and 8-bit (layer_fused_bs.cu): the plan,
the gate/up and down stage layouts, the ldmatrix addresses in the 64-byte
swizzled boxes, the tensor-map coordinates, the swizzled x and h staging and
the hf / ys stores.  Routing comes from seeded draws of the sweep's kinds
(repeated-token and independent blocks)."""
from __future__ import annotations

import random

import pytest

FW, MAX_RING, MAX_CHUNKS_P2, GATE_TILE, MAX_BLOCK = 16, 8, 2, 8, 16
SMEM_BUDGET, SMEM_MAX = 220 * 1024, 227 * 1024


def pad(b):
    return b + 64 if b % 128 == 0 else b


def fused_plan(k, d, I, E):
    if d % 32 or I % 32 or I > 768 or k < 1 or k > MAX_BLOCK:
        return None
    NT = 1 if k <= 8 else 2
    C = d // 32
    nsl = (d + 1023) // 1024
    while nsl <= C and C % nsl:
        nsl += 1
    if nsl > C:
        return None
    ks = d // nsl
    if ks // 32 > FW * MAX_CHUNKS_P2:
        return None
    slot = max(16 * pad(ks * 2), 16 * I * 2)
    slot = (slot + 1023) & ~1023  # stage bases 1024-aligned (the mode-3 swizzle)
    scratch = NT * 8 * d * 2
    if NT == 2 and 8 * d * 2 + slot > scratch:
        scratch = 8 * d * 2 + slot
    scratch = max(scratch, k * E * 4, k * 8 * 16 * 4)
    scratch = (scratch + 127) & ~127
    redb = FW * NT * 32 * 16
    ring = next((r for r in range(MAX_RING - 1, 3, -1)
                 if 1024 + r * slot + scratch + redb + 16 * MAX_RING <= SMEM_BUDGET), 0)
    if ring < 4:
        return None
    return dict(NT=NT, nsl=nsl, ks=ks, slot=slot, scratch=scratch, ring=ring, redb=redb,
                smem=1024 + ring * slot + scratch + redb + 16 * MAX_RING)


def tables(idx, k, K, E, ns):
    """woken ids, offsets, sorted pair list (routed pairs t*K+s, then k*K+t)."""
    woken = sorted({e for row in idx for e in row})
    cnt = {e: sum(row.count(e) for row in idx) for e in woken}
    if ns:
        woken.append(E)
        cnt[E] = k
    off = [0]
    for e in woken:
        off.append(off[-1] + cnt[e])
    pos = {e: off[i] for i, e in enumerate(woken)}
    gat = [None] * off[-1]
    for q in range(k * K):
        e = idx[q // K][q % K]
        gat[pos[e]] = q
        pos[e] += 1
    for t in range(k * ns):
        gat[pos[E] + t] = k * K + t
    return woken, off, gat


def check_layer(k, d, I, E, K, idx, ns, tma):
    P = fused_plan(k, d, I, E)
    if P is None:
        return None
    NT, ks, nsl, slot, SH = P["NT"], P["ks"], P["nsl"], P["slot"], P["ring"]
    if tma == 3 and (d % 64 or ks % 64):
        tma = 1
    if tma in (1, 2) and (d % 256 or ks % 256):
        tma = 0
    rsx, rsg = d * 2, pad(ks * 2)
    row_b, blk_b = (512, 4096) if tma else (rsg, 512)
    up_off = 8 * ks * 2 if tma else 8 * rsg
    if tma == 3:
        # swizzled segments: every stage base (ring slots and the staged-x stage) 1024-aligned
        assert slot % 1024 == 0 and (8 * rsx) % 1024 == 0 and up_off % 1024 == 0
    assert P["smem"] + 5632 <= SMEM_MAX  # dynamic + the kernel's static 5.5 KB (routing tables)
    woken, off, gat = tables(idx, k, K, E, ns)
    nW, nP = len(woken), k * K + ns * k
    assert off[-1] == nP and sorted(gat) == list(range(k * K)) + [k * K + t for t in range(k * ns)]
    # ring size and gate/up entries, as the routing epilogue decides them
    extra = NT == 2 and P["scratch"] >= 8 * rsx + slot and SH < MAX_RING
    rmax = max([off[i + 1] - off[i] for i in range(nW - ns)] or [0])
    split = extra and ns and k > 8 and rmax <= 8
    mmax = rmax if split else max(off[i + 1] - off[i] for i in range(nW))
    S = SH + 1 if extra and mmax <= 8 else SH
    ent = [(woken[i], off[i], off[i + 1] - off[i]) for i in range(nW - ns)]
    if ns:
        ent += [(E, off[nW - 1], 8), (E, off[nW - 1] + 8, k - 8)] if split else [(E, off[nW - 1], k)]

    def stage_end(s, nbytes):  # last byte + 1 of a fill of stage s, and its limit
        base = s * slot if s < SH else SH * slot + 8 * rsx
        limit = (s + 1) * slot if s < SH else SH * slot + P["scratch"]
        return base + nbytes, limit

    for s in range(S):
        end, limit = stage_end(s, 16 * ks * 2 if tma else 16 * rsg)
        assert end <= limit, "gate/up fill overruns stage %d" % s
        end, limit = stage_end(s, 16 * I * 2)
        assert end <= limit, "down fill overruns stage %d" % s
    hcap = 2 * MAX_BLOCK * (K + ns) * I  # bf16 elements of ws.h (k_max * (K + ns) * I floats)
    cps = ks // 32
    for e, o, m in ent:
        assert 1 <= m <= (8 if S == SH + 1 else NT * 8), "entry of %d tokens" % m
        assert (e * I + I - 1) < (E + ns) * I  # last weight row of the entry's last unit
        # staged x rows of this entry (the extra stage starts at row 8)
        assert m * rsx <= P["scratch"] and (S == SH or m <= 8)
        # A fragments: row g = 7, lane column c = 3, each warp's last chunk
        for w in range(FW):
            c0, c1 = w * cps // FW, (w + 1) * cps // FW
            assert c1 - c0 <= MAX_CHUNKS_P2
            if c1 > c0:
                ch = c1 - 1
                if tma == 3:  # the largest offset over the MMA rows and lane columns
                    o_frag = max((ch >> 1) * 1024 + ((g >> 1) | ((g & 1) << 2)) * 128
                                 + ((((ch & 1) * 4 + c) ^ ((g >> 1) | ((g & 1) << 2))) << 4)
                                 for g in range(8) for c in range(4))
                else:
                    o_frag = 7 * row_b + (ch >> 3) * blk_b + (ch & 7) * 64 + 3 * 16
                assert o_frag + 16 <= up_off and up_off + o_frag + 16 <= min(slot, 2 * up_off)
        # B fragments: x chunk index of the last slice, XOR swizzle within the row
        swz = 4 if d % 64 == 0 else 0
        xq = (nsl - 1) * (ks // 8) + (cps - 1) * 4 + 3
        assert (xq ^ swz) < d // 8
        # h of the entry's last token, last column
        assert (o + m - 1) * I + I - 1 < hcap
        assert all(0 <= (q // K if q < k * K else q - k * K) < k for q in gat[o:o + m])
    C = I // 32
    for wi in range(nW):
        eo, em = off[wi], off[wi + 1] - off[wi]
        assert em <= NT * 8
        e = woken[wi]
        assert (e * d + d - 16) * I + 16 * I <= (E + ns) * d * I  # last down copy of the expert
        for wg in range(8):
            assert (wg + 1) * C // 8 - wg * C // 8 <= 3  # P3 chunks per warp
        for tok in range(em):
            pair = gat[eo + tok]
            assert pair * d + d - 1 < MAX_BLOCK * (K + ns) * d  # ys row end
            assert (eo + tok) * I + (C - 1) * 32 + 3 * 8 + 7 < hcap
    return S


def _draws(k, E, K, rnd):
    base = rnd.sample(range(E), K)
    rep = [base if rnd.random() < 0.8 else rnd.sample(range(E), K) for _ in range(k)]
    ind = [rnd.sample(range(E), K) for _ in range(k)]
    return rep, ind


@pytest.mark.parametrize("d", [256, 352, 1056, 2048, 2304])
@pytest.mark.parametrize("I", [64, 512, 768])
def test_fused_bf16_indices_stay_in_their_buffers(d, I):
    rnd = random.Random(d * 1000 + I)
    checked, extra_stage = 0, set()
    for E, K in ((8, 8), (16, 4), (128, 8), (256, 8)):
        for k in (1, 8, 9, 16):
            for idx in _draws(k, E, K, rnd):
                for ns in (0, 1):
                    for tma in (3, 1, 0):
                        S = check_layer(k, d, I, E, K, idx, ns, tma)
                        if S is not None:
                            checked += 1
                            extra_stage.add((k > 8, ns, S == fused_plan(k, d, I, E)["ring"] + 1))
    assert checked > 0
    # at k > 8 with independent rows the staged-x stage is in use, with and without
    # the shared expert (the split keeps it)
    assert (True, 0, True) in extra_stage and (True, 1, True) in extra_stage


# ---------------------------------------------------------------- block-scaled single-launch kernel
BS_GROUPS, BS_RING, BS_ROWS_G, BS_ROWS_D, BS_ROW_BYTES, BS_BOX, BS_MAX_D = 4, 8, 32, 64, 256, 64, 2048
BS_CODES, BS_STAGE, BS_SLOT = 16384, 17408, 18432
FMT = {"mxfp4": dict(CPS=512, BPI=4, SB=1, num=1, den=2), "q8": dict(CPS=256, BPI=2, SB=2, num=1, den=1)}


def bs_plan(fmt, k, d, I):
    """fused_bs_plan / bs_smem of layer_fused_bs.cu."""
    if d > BS_MAX_D or I > 512 or I < 64:
        return None
    if fmt == "mxfp4" and (d % 512 or I % 128):
        return None
    if fmt == "q8" and (d % 256 or I % 64 or (I > 256 and I % 256)):
        return None
    NT = 1 if k <= 8 else 2
    scratch = max(NT * 8 * d * 2, BS_GROUPS * NT * 8 * I * 2)
    scratch = (scratch + 127) & ~127
    smem = 1024 + BS_RING * BS_SLOT + scratch + 16 * BS_RING
    return None if smem + 8 * 1024 > SMEM_MAX else dict(NT=NT, scratch=scratch, smem=smem)


def sw64(box, row, j):
    """the kernel's sw64: chunk j of row `row` of a 64-byte-swizzled box."""
    return box + row * BS_BOX + ((j ^ ((row >> 1) & 3)) << 4)


def swz2(q, r):
    return q ^ ((r & 1) << 2)


def check_bs_layer(fmt, k, d, I, E, K, idx, ns):
    P = bs_plan(fmt, k, d, I)
    if P is None:
        return None
    F = FMT[fmt]
    NT, scratch = P["NT"], P["scratch"]
    assert P["smem"] + 7168 <= SMEM_MAX  # + the kernel's static shared memory
    woken, off, gat = tables(idx, k, K, E, ns)
    nW, nP = len(woken), k * K + ns * k
    Et = E + ns
    cb = lambda n: n * F["num"] // F["den"]  # code bytes of n elements
    # ---- gate/up stage: [4 boxes][32][64] gate | same for up | [32][16] gate scales | [32][16] up scales
    up_off, sc_off, scu_off = BS_CODES // 2, BS_CODES, BS_CODES + 512
    assert scu_off + 32 * 16 == BS_STAGE <= BS_SLOT and BS_SLOT % 1024 == 0
    for itb in range(4):
        for wq in range(4):
            for lane in range(32):
                a = sw64(up_off + itb * BS_ROWS_G * BS_BOX, wq * 8 + (lane & 7), lane >> 3)
                assert up_off <= a and a + 16 <= sc_off  # ldmatrix rows of the up codes
                assert (up_off + itb * BS_ROWS_G * BS_BOX) % 512 == 0  # swizzle atom alignment
    assert scu_off + 31 * 16 + 16 <= BS_STAGE  # lds128 of the last up-scale row
    nq = d // F["CPS"]
    assert cb(d) == nq * BS_ROW_BYTES
    # the code maps are 3-D, [row bytes / 64][rows][64]: one copy of 4 boxes per stage,
    # at chunk coordinate z = 4 q (x = 0, so the 16-byte rule holds), all inside the row
    chunks_g = cb(d) // BS_BOX
    assert cb(d) % BS_BOX == 0 and min(4, chunks_g) == 4
    for q in (0, nq - 1):
        assert 4 * q + 4 <= chunks_g
        assert (q * 16) % 16 == 0 and q * 16 + 16 <= d // 32 * F["SB"]
    # ---- down stage: [nb boxes][64][64] codes | [64][srs] scales
    rowb = cb(I)
    nqd = (rowb + BS_ROW_BYTES - 1) // BS_ROW_BYTES
    srow = I // 32 * F["SB"]
    srs = srow if nqd == 1 else 16
    assert (srow * 64) % 16 == 0 and (nqd == 1 or srow % 16 == 0)  # bulk size / tensor-map stride
    chunks_d = rowb // BS_BOX
    bz = min(4, chunks_d)  # the down map's box depth; the copy's byte count is bz full boxes
    assert rowb % BS_BOX == 0
    for q in range(nqd):
        nb = min(4, (rowb - q * BS_ROW_BYTES) // BS_BOX)
        assert 1 <= nb <= 4 and (rowb - q * BS_ROW_BYTES) % BS_BOX == 0
        assert nb == bz  # no partial last stage: every copy lands whole boxes that are read
        assert 4 * q + bz <= chunks_d  # the copy's chunks lie inside the row
        assert bz * BS_ROWS_D * BS_BOX <= BS_CODES and BS_CODES + BS_ROWS_D * srs <= BS_STAGE
        for itb in range(nb):
            for wq in range(4):
                for lane in (0, 7, 31):
                    for half in (0, 8):
                        a = sw64(itb * BS_ROWS_D * BS_BOX, wq * 16 + half + (lane & 7), lane >> 3)
                        assert 0 <= a and a + 16 <= nb * BS_ROWS_D * BS_BOX
            # scale words: rows up to 63, word itb
            assert BS_CODES + 63 * srs + itb * 4 + 4 <= BS_CODES + BS_ROWS_D * srs
            assert (63 * srs + itb * 4) % 4 == 0
            # blocks of this box: the B chunk index stays inside the staged h row
            for mb in range(F["BPI"]):
                hq = q * (F["CPS"] // 8) + (itb * F["BPI"] + mb) * 4 + 3
                assert swz2(hq, 1) < I // 8 and swz2(hq, 0) < I // 8
    # ---- staged x (P2) and h (P3) rows
    xrow, cpr = d * 2, d // 8
    assert k * xrow <= scratch and cpr % 64 == 0
    assert all(swz2(q, t) < cpr for q in range(cpr) for t in (0, 1))
    for q in (0, nq - 1):
        for blk in range(F["CPS"] // 32):
            xq = q * (F["CPS"] // 8) + blk * 4 + 3
            assert swz2(xq, 1) < cpr
    hrow, hcpr = I * 2, I // 8
    assert BS_GROUPS * NT * 8 * hrow <= scratch and hcpr % 8 == 0
    assert (BS_GROUPS - 1) * NT * 8 * hrow + (NT * 8 - 1) * hrow + hcpr * 16 <= scratch
    # ---- weights, h and ys
    tiles_g, tiles_d = I // BS_ROWS_G, d // BS_ROWS_D
    for wi in range(nW):
        e, eo, m = woken[wi], off[wi], off[wi + 1] - off[wi]
        assert m <= NT * 8
        assert e * I + (tiles_g - 1) * BS_ROWS_G + BS_ROWS_G <= Et * I  # gate/up box rows
        row = e * d + (tiles_d - 1) * BS_ROWS_D
        assert row + BS_ROWS_D <= Et * d and (row * srow) % 16 == 0
        for tok in range(m):
            pair = gat[eo + tok]
            assert 0 <= pair < nP
            assert (eo + tok) * I + (tiles_g - 1) * BS_ROWS_G + 3 * 8 + 7 < MAX_BLOCK * (K + ns) * I  # hf (fp32)
            assert pair * d + (tiles_d - 1) * BS_ROWS_D + 3 * 16 + 7 + 8 < MAX_BLOCK * (K + ns) * d  # ys
    return True


@pytest.mark.parametrize("fmt", ["mxfp4", "q8"])
@pytest.mark.parametrize("d", [512, 1024, 2048])
@pytest.mark.parametrize("I", [64, 128, 256, 384, 512])
def test_fused_block_scaled_indices_stay_in_their_buffers(fmt, d, I):
    rnd = random.Random(d * 7919 + I + (1 if fmt == "q8" else 0))
    checked = 0
    for E, K in ((4, 2), (16, 4), (256, 8)):
        for k in (1, 8, 9, 16):
            for idx in _draws(k, E, K, rnd):
                for ns in (0, 1):
                    checked += check_bs_layer(fmt, k, d, I, E, K, idx, ns) is not None
    ok = bs_plan(fmt, 16, d, I) is not None
    assert (checked > 0) == ok


def test_q8_block_order_matches_the_mma_k_slots():
    """The 8-bit kernel stores each 32-element block of a token row so that
    lane c's 16-byte chunk holds elements 4c..4c+3 and 16+4c..16+4c+3 (the k
    slots its two MMAs take from code chunks 2m and 2m+1); the shuffle
    permutation (q8_permute) reaches exactly that."""
    for lane in range(32):
        cc, base = lane & 3, lane & ~3
        s1, s2 = base + (cc >> 1), base + 2 + (cc >> 1)
        h = cc & 1
        # input chunk of lane L holds elements 8 (L & 3) .. +8 of its block, as 4 words of 2
        words = [(8 * (s1 & 3) + 2 * (2 * h + i), 8 * (s1 & 3) + 2 * (2 * h + i) + 1) for i in range(2)]
        words += [(8 * (s2 & 3) + 2 * (2 * h + i), 8 * (s2 & 3) + 2 * (2 * h + i) + 1) for i in range(2)]
        got = [e for w in words for e in w]
        assert got == [4 * cc, 4 * cc + 1, 4 * cc + 2, 4 * cc + 3, 16 + 4 * cc, 17 + 4 * cc, 18 + 4 * cc, 19 + 4 * cc]
