"""CPU model of the multi-launch bf16 gate/up kernel's staging (ffn_tma.cu):
each stage's gate and up matrices arrive as one 3-D tensor copy of 8 rows x
ks columns in 128-byte segments with the 128-byte swizzle, and MMA row g reads
stored row (g >> 1) | ((g & 1) << 2).  Checked for every d, d_ff the plan
takes: the consumer's fragment address fetches exactly the row piece the MMA
expects, the eight 16-byte loads of each quarter-warp hit distinct bank
groups, the h row each MMA row writes is its stored row (a permutation of the
unit's 8 rows), and the stages stay 1024-aligned inside the plan's shared
memory."""
from __future__ import annotations

import pytest

CONSUMER_WARPS, SMEM_BUDGET = 8, 220 * 1024


def pad(b):
    return b + 64 if b % 128 == 0 else b


HALF = SMEM_BUDGET // 2 + 1024


def tma_plan(k, d, I):
    """The gate/up part of ffn_tma.cu's tma_plan (ks, CTAs per SM, stage count, smem)."""
    NT = 1 if k <= 8 else 2
    C = d // 32
    nsl = (d + 1023) // 1024
    while nsl <= C and C % nsl:
        nsl += 1
    if nsl > C:
        return None
    ks, per_sm = d // nsl, 1
    xg2, redb2 = 2 * 8 * pad(d * 2), CONSUMER_WARPS * 2 * 32 * 16

    def two_fit(w):
        return 1024 + 2 * 16 * pad(w * 2) + xg2 + redb2 + 32 <= HALF

    if two_fit(ks):
        per_sm = 2
    elif ks > 512 and d % 512 == 0 and two_fit(512):
        ks, nsl, per_sm = 512, d // 512, 2
    xg = NT * 8 * pad(d * 2)
    redb = CONSUMER_WARPS * NT * 32 * 16
    budget = HALF if per_sm == 2 else SMEM_BUDGET
    for Sg in (4, 3, 2):
        smg = 1024 + Sg * 16 * pad(ks * 2) + xg + redb + 16 * Sg
        if smg <= budget:
            return dict(ks=ks, nsl=nsl, S=Sg, smem=smg, xg=xg, redb=redb, NT=NT, per_sm=per_sm)
    return None


def swizzle128(z, r, b):
    """Where the tensor copy puts byte b (0..127) of row r (0..7) of segment z:
    the 16-byte chunk index is XORed with the row inside each 1024-byte atom."""
    return z * 1024 + r * 128 + ((((b >> 4) ^ r) << 4) | (b & 15))


def stored_row(g):
    return (g >> 1) | ((g & 1) << 2)


def consumer_offset(g, c, ch):
    pr = stored_row(g)
    return (ch >> 1) * 1024 + pr * 128 + ((((ch & 1) * 4 + c) ^ pr) << 4)


@pytest.mark.parametrize("d", [512, 1024, 1536, 2048, 4096])
def test_swizzled_gateup_fragment_addresses(d):
    P = tma_plan(16, d, 1024)
    assert P is not None
    ks = P["ks"]
    assert ks % 64 == 0 and ks // 64 <= 256  # the map's box {64, 8, ks / 64}
    # inverse of the copy's placement for one matrix of a stage
    where = {}
    for z in range(ks // 64):
        for r in range(8):
            for b in range(0, 128, 16):
                where[swizzle128(z, r, b)] = (r, z * 64 + b // 2)  # (stored row, first column)
    assert len(where) == 8 * ks // 8  # every 16-byte piece lands once
    cps = ks // 32
    for w in range(CONSUMER_WARPS):
        c0, c1 = w * cps // CONSUMER_WARPS, (w + 1) * cps // CONSUMER_WARPS
        for ch in range(c0, c1):
            offs = []
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                o = consumer_offset(g, c, ch)
                assert o % 16 == 0 and 0 <= o and o + 16 <= 8 * ks * 2
                # the MMA wants row g's columns ch*32 + c*8 .. +7 of stored row pr
                assert where[o] == (stored_row(g), ch * 32 + c * 8)
                offs.append(o)
            for q in range(4):  # a quarter-warp's eight 16-byte loads: distinct bank groups
                groups = {(o // 16) % 8 for o in offs[8 * q:8 * q + 8]}
                assert len(groups) == 8


def test_stored_rows_are_a_permutation():
    assert sorted(stored_row(g) for g in range(8)) == list(range(8))
    # the quarter-warp pairs: MMA rows 2i and 2i+1 read stored rows i and i + 4
    assert all(stored_row(2 * i) == i and stored_row(2 * i + 1) == i + 4 for i in range(4))


@pytest.mark.parametrize("k", [1, 8, 16])
@pytest.mark.parametrize("d", [512, 1024, 1536, 2048, 4096])
def test_swizzled_stages_fit_and_align(k, d):
    P = tma_plan(k, d, 1024)
    if P is None:
        return
    ks, S = P["ks"], P["S"]
    stage = 32 * ks  # gate then up, unpadded
    assert stage % 1024 == 0 and (16 * ks) % 1024 == 0  # each matrix's box starts 1024-aligned
    assert stage <= 16 * pad(ks * 2)  # no more than the padded layout the plan reserves
    # aligned base (up to 1023 bytes of slack) + stages + x rows + reduction + barriers
    assert 1023 + S * stage + P["xg"] + P["redb"] + 16 * S <= P["smem"] <= SMEM_BUDGET
    if P["per_sm"] == 2:
        assert P["smem"] <= HALF and 2 * (P["smem"] + 1024) <= 228 * 1024  # + the per-CTA reserve


@pytest.mark.parametrize("d", [512, 1024, 1536, 2048, 3072, 4096])
def test_gateup_slice_depends_on_the_shape_only(d):
    """A block's rows equal single-token calls only if every k splits a row's sum
    the same way: the slice width (and so the warps' column chunks) is the same for
    k = 1..16; two CTAs per SM exactly where the two-token-tile plan fits half the
    budget (d = 2048 with 512-column slices), one elsewhere (d = 4096)."""
    plans = [tma_plan(k, d, 768) for k in (1, 2, 8, 9, 16)]
    assert all(P is not None for P in plans)
    assert len({(P["ks"], P["nsl"], P["per_sm"]) for P in plans}) == 1
    P = plans[-1]
    assert P["ks"] * P["nsl"] == d and P["ks"] % 32 == 0 and P["ks"] <= 1024
    if d == 2048:
        assert (P["ks"], P["per_sm"]) == (512, 2)
    if d == 4096:
        assert (P["ks"], P["per_sm"]) == (1024, 1)


def down_plan(I):
    """The down part of ffn_tma.cu's tma_plan, chosen for two token tiles:
    (rows per unit, CTAs per SM, stages per unit).  16 rows and two CTAs per SM when
    half the budget holds two full-d_ff stages; else, for d_ff a multiple of 128,
    two CTAs per SM with two half-d_ff stages per unit; else one CTA per SM with 32
    or 16 rows."""
    half = SMEM_BUDGET // 2 + 1024
    redb2, hb2 = CONSUMER_WARPS * 2 * 32 * 16, 2 * 8 * pad(I * 2)
    if 1024 + 2 * 16 * pad(I * 2) + hb2 + redb2 + 32 <= half:
        return 16, 2, 1
    if I % 128 == 0 and 1024 + 2 * 16 * pad(I) + hb2 + redb2 + 32 <= half:
        return 16, 2, 2
    for rs in (32, 16):
        if 2 * rs * pad(I * 2) + hb2 + redb2 + 32 <= SMEM_BUDGET:
            return rs, 1, 1
    return None


@pytest.mark.parametrize("I", [768, 1024, 1408, 1536])
@pytest.mark.parametrize("k", [1, 16])
def test_down_plan_fits_its_ctas_per_sm(I, k):
    """Two CTAs per SM only where both fit: the stages, h rows, reduction buffer and
    alignment slack of one CTA within half of the budget (and 227 KB per SM).  The
    plan depends on the shape only (k = 1 and 16 agree), and every measured shape
    keeps two CTAs per SM: full-d_ff stages up to d_ff = 1024, half-d_ff above."""
    rs, per_sm, dsl = down_plan(I)
    NT = 1 if k <= 8 else 2
    hb, redb = NT * 8 * pad(I * 2), CONSUMER_WARPS * NT * 32 * 16
    budget = SMEM_BUDGET // 2 + 1024 if per_sm == 2 else SMEM_BUDGET
    S = next(S for S in (4, 3, 2) if 1024 + S * rs * pad(I * 2 // dsl) + hb + redb + 16 * S <= budget)
    smem = 1024 + S * rs * pad(I * 2 // dsl) + hb + redb + 16 * S
    assert S >= 2 and smem <= budget
    assert per_sm == 2 and rs == 16 and 2 * (smem + 1024) <= 228 * 1024  # + the per-CTA reserve
    assert dsl == (1 if I <= 1024 else 2)
    assert (rs * (I // dsl) * 2) % 1024 == 0  # swizzled stages stay 1024-aligned


def down_offset(rw, g, c, ch, rs, upper):
    """The down consumer's swizzled fragment offset: row tile rw, MMA row g (+ 8
    when upper), lane column c, 32-column chunk ch."""
    pr = stored_row(g)
    x = ch * 4 + c
    o0 = (x >> 3) * (rs * 128) + (rw * 16 + pr) * 128 + (((x & 7) ^ pr) << 4)
    return o0 + (1024 if upper else 0)


@pytest.mark.parametrize("I", [768, 1024, 1408, 1536])
def test_swizzled_down_fragment_addresses(I):
    """Every lane's fragment offset in a down stage holds the weight row and the
    d_ff columns its MMA slot expects; with half-d_ff stages the columns of stage
    sl start at sl * I / 2, and the token (h) piece the lane reads is the same
    global column.  A quarter-warp's loads cover all eight 16-byte bank groups."""
    rs, _, dsl = down_plan(I)
    Ih = I // dsl
    assert Ih % 64 == 0 and Ih // 64 <= 256
    rtiles, kparts = rs // 16, CONSUMER_WARPS // (rs // 16)
    for sl in range(dsl):
        where = {}
        for z in range(Ih // 64):  # the box {64, rs, Ih/64} at z = sl * Ih/64, swizzled per 8-row atom
            for r in range(rs):
                for b in range(0, 128, 16):
                    off = z * rs * 128 + r * 128 + ((((b >> 4) ^ (r & 7)) << 4))
                    where[off] = (r, sl * Ih + z * 64 + b // 2)
        assert len(where) == rs * Ih // 8 and (rs * 128) % 1024 == 0
        Cs = Ih // 32
        for w in range(CONSUMER_WARPS):
            rw, kq = w % rtiles, w // rtiles
            for ch in range(kq * Cs // kparts, (kq + 1) * Cs // kparts):
                for upper in (0, 1):
                    offs = []
                    for lane in range(32):
                        g, c = lane >> 2, lane & 3
                        o = down_offset(rw, g, c, ch, rs, upper)
                        h_piece = (sl * Cs + ch) * 4 + c  # 16-byte piece of the h row
                        assert where[o] == (rw * 16 + 8 * upper + stored_row(g), h_piece * 8)
                        offs.append(o)
                    for q in range(4):
                        assert len({(o // 16) % 8 for o in offs[8 * q:8 * q + 8]}) == 8
