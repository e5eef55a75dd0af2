"""CPU models of the single-launch kernels' index arithmetic (compute-
sanitizer is not available).  bf16: the shared-memory plan, the routing tables with
the shared expert and its split gate/up entries, and the extreme index of
every shared-memory, TMA, global-weight, h and ys access a unit makes, checked
against the size of its buffer.  The formulas are the kernel's (layer_fused.cu:
fused_plan, slot_addr, the producer's copies, the consumers' fragment loads and
stores).  mxfp4 (layer_fused_mxfp4.cu): the plan, the gate/up and down stage
layouts, the tensor-map coordinates, the swizzled x and h staging and the hf /
ys stores.  Routing comes from seeded draws of the sweep's kinds
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
    slot = (slot + 127) & ~127
    scratch = NT * 8 * d * 2
    if NT == 2 and 8 * d * 2 + slot > scratch:
        scratch = 8 * d * 2 + slot
    scratch = max(scratch, k * E * 4, k * 8 * 16 * 4)
    scratch = (scratch + 127) & ~127
    redb = FW * NT * 32 * 16
    ring = next((r for r in range(MAX_RING - 1, 3, -1) if r * slot + scratch + redb + 16 * MAX_RING <= SMEM_BUDGET), 0)
    if ring < 4:
        return None
    return dict(NT=NT, nsl=nsl, ks=ks, slot=slot, scratch=scratch, ring=ring, redb=redb,
                smem=ring * slot + scratch + redb + 16 * MAX_RING)


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
    if tma and (d % 256 or ks % 256):
        tma = 0
    rsx, rsg = d * 2, pad(ks * 2)
    row_b, blk_b = (512, 4096) if tma else (rsg, 512)
    up_off = 8 * ks * 2 if tma else 8 * rsg
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
                    for tma in (1, 0):
                        S = check_layer(k, d, I, E, K, idx, ns, tma)
                        if S is not None:
                            checked += 1
                            extra_stage.add((k > 8, ns, S == fused_plan(k, d, I, E)["ring"] + 1))
    assert checked > 0
    # at k > 8 with independent rows the staged-x stage is in use, with and without
    # the shared expert (the split keeps it)
    assert (True, 0, True) in extra_stage and (True, 1, True) in extra_stage


# ---------------------------------------------------------------- mxfp4 single-launch kernel
MX_GROUPS, MX_RING, MX_CH, MX_ROWS, MX_COLS, MX_MAX_D = 4, 8, 4, 32, 512, 2048


def mx_plan(k, d, I):
    """fused_mx_plan / mx_smem of layer_fused_mxfp4.cu."""
    if d % MX_COLS or d > MX_MAX_D or I % 64 or I > 128 * MX_CH:
        return None
    NT = 1 if k <= 8 else 2
    slot = max(MX_ROWS * MX_COLS + MX_ROWS * MX_COLS // 16, 34 * I)
    slot = (slot + 127) & ~127
    ipad = (I + 127) // 128 * 128
    scratch = max(NT * 8 * d * 2, MX_GROUPS * NT * 8 * ipad * 2)
    scratch = (scratch + 127) & ~127
    smem = MX_RING * slot + scratch + 16 * MX_RING + (FW * 32 * 16 if NT == 2 else 0)
    return None if smem > SMEM_BUDGET else dict(NT=NT, slot=slot, scratch=scratch, smem=smem)


def swz(q, j):
    return q ^ (((q >> 3) & 1) | ((j & 1) << 1))


def check_mx_layer(k, d, I, E, K, idx, ns):
    P = mx_plan(k, d, I)
    if P is None:
        return None
    NT, slot, scratch = P["NT"], P["slot"], P["scratch"]
    woken, off, gat = tables(idx, k, K, E, ns)
    nW, nP = len(woken), k * K + ns * k
    # gate/up stage: [32][256] gate codes | [32][256] up codes | [32][16] gate scales | [32][16] up scales
    g_up = MX_ROWS * MX_COLS // 2
    g_sc, g_scu = 2 * g_up, 2 * g_up + MX_ROWS * MX_COLS // 32
    bytes_g = 2 * g_up + 2 * MX_ROWS * MX_COLS // 32
    assert bytes_g <= slot
    rw, c, j = 31, 3, MX_CH - 1  # the largest row, lane column and chunk
    assert g_up + rw * (MX_COLS // 2) + c * 16 + j * 64 + 16 <= g_sc       # up codes
    assert g_scu + rw * (MX_COLS // 32) + c + j * 4 + 1 <= bytes_g         # up scales
    # down stage: [64][I/2] codes | [64][I/32] scales
    rowb_d, srow_d = I // 2, I // 32
    d_sc, bytes_d = 64 * rowb_d, 64 * rowb_d + 64 * srow_d
    assert bytes_d <= slot
    CI = (I + 127) // 128
    for c in (0, 3):
        # with a ragged last 128-code chunk, lanes c >= 2 skip it (no codes there)
        jl = CI - 1 if (I % 128 == 0 or c < 2) else CI - 2
        if jl >= 0:
            assert 63 * rowb_d + c * 16 + jl * 64 + 16 <= d_sc  # codes of row 63
            assert d_sc + 63 * srow_d + c + jl * 4 + 1 <= bytes_d  # its scales
    # TMA coordinates: x bytes 16-aligned, boxes inside the matrices
    nq = d // MX_COLS
    for q in (0, nq - 1):
        assert (q * (MX_COLS // 2)) % 16 == 0 and (q * (MX_COLS // 32)) % 16 == 0
        assert q * (MX_COLS // 2) + 256 <= d // 2 and q * (MX_COLS // 32) + 16 <= d // 32
    # staged x rows (P2): k rows of d fp16, 16-byte pieces swizzled within groups of 4
    xrow = d * 2
    cpr = d // 8
    assert all(swz(q, t) < cpr for q in range(cpr) for t in (0, 1))
    assert k * xrow <= scratch
    # B reads of token t: bt = t*xrow + c*64 + ((tt ^ sw) << 4), plus chunk (q*4 + j)*256
    assert 3 * 64 + (3 << 4) + ((nq - 1) * MX_CH + MX_CH - 1) * 256 + 16 <= xrow
    # staged h rows (P3): per group NT*8 rows of CI*256 bytes
    hrow = CI * 256
    assert MX_GROUPS * NT * 8 * hrow <= scratch
    assert all(swz(q, n) < CI * 16 for q in range(CI * 16) for n in (0, 1))
    assert 3 * 64 + (3 << 4) + (CI - 1) * 256 + 16 <= hrow
    tiles_g, tiles_d = I // MX_ROWS, d // 64
    for wi in range(nW):
        e, eo, m = woken[wi], off[wi], off[wi + 1] - off[wi]
        assert m <= NT * 8
        assert e * I + (tiles_g - 1) * MX_ROWS + MX_ROWS <= (E + ns) * I  # gate/up box rows
        row = e * d + (tiles_d - 1) * 64
        assert (row + 64) * rowb_d <= (E + ns) * d * rowb_d and (row * srow_d) % 16 == 0 and (64 * srow_d) % 16 == 0
        for tok in range(m):
            pair = gat[eo + tok]
            assert 0 <= pair < nP
            assert (eo + tok) * I + (tiles_g - 1) * MX_ROWS + 3 * 8 + 7 < MAX_BLOCK * (K + ns) * I  # hf (fp32)
            assert pair * d + (tiles_d - 1) * 64 + 3 * 16 + 7 + 8 < MAX_BLOCK * (K + ns) * d       # ys
    return True


@pytest.mark.parametrize("d", [512, 1024, 2048])
@pytest.mark.parametrize("I", [64, 192, 448, 512])
def test_fused_mxfp4_indices_stay_in_their_buffers(d, I):
    rnd = random.Random(d * 7919 + I)
    checked = 0
    for E, K in ((4, 2), (16, 4), (256, 8)):
        for k in (1, 8, 9, 16):
            for idx in _draws(k, E, K, rnd):
                for ns in (0, 1):
                    checked += check_mx_layer(k, d, I, E, K, idx, ns) is not None
    assert checked > 0
