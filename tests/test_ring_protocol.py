"""CPU model of the mbarrier ring protocols of the single-launch kernels
(compute-sanitizer is not available, so the stage/phase bookkeeping is
checked here by exhaustion over unit counts and ring sizes).

A stage's full barrier completes once per fill; a waiter names the phase it
wants by its parity only.  That is sound when every warp that waits for a fill
of stage s also consumed the previous fill of s: it can then never be one
phase ahead of the barrier and pass a wait early.  The models below rebuild,
with the kernels' own formulas, the producer's fill sequence and each
consumer's stage sequence, and check:
  1. every consumer takes the fills meant for it, in issue order;
  2. every waiter of a fill consumed the previous fill of that stage;
  3. the per-stage parity each side tracks equals the fill's phase index.
The old bf16 down-phase scheme (one shared ring, groups alternating over it)
is kept as a negative control: with an odd ring it breaks rule 2."""
from __future__ import annotations

import pytest


def _check(fills, seqs):
    """fills: [(stage, waiters)] in issue order; seqs: waiter -> expected stages.
    Returns the number of broken waits (rules 2 and 3); rule 1 is asserted."""
    pos = {w: 0 for w in seqs}
    last, phase, bits = {}, {}, {w: 0 for w in seqs}
    pbits, violations = 0, 0
    for s, waiters in fills:
        ph = phase.get(s, 0)
        phase[s] = ph + 1
        assert ((pbits >> s) & 1) == (ph & 1)  # producer: parity of the phase it fills
        pbits ^= 1 << s
        prev = last.get(s)
        for w in waiters:
            assert seqs[w][pos[w]] == s, "consumer %s expects stage %d, fill is on %d" % (w, seqs[w][pos[w]], s)
            pos[w] += 1
            if prev is not None and w not in prev:
                violations += 1  # w skipped the previous fill of s
            if ((bits[w] >> s) & 1) != (ph & 1):
                violations += 1  # w would wait for the wrong parity
            bits[w] ^= 1 << s
        last[s] = set(waiters)
    assert all(pos[w] == len(seqs[w]) for w in seqs)
    return violations


def bf16_ring(n_gate, n_down, S, old_down_scheme=False):
    """layer_fused.cu: gate/up fills go round all S stages and every consumer
    warp waits for each; down unit j belongs to group j & 1, which owns the
    stages of its parity (pg / gs sequences)."""
    fills, ps = [], 0
    for _ in range(n_gate):
        fills.append((ps, ("g0", "g1")))
        ps = ps + 1 if ps + 1 < S else 0
    if old_down_scheme:
        for j in range(n_down):
            fills.append((ps, ("g%d" % (j & 1),)))
            ps = ps + 1 if ps + 1 < S else 0
    else:
        pg = [0, 1]
        for j in range(n_down):
            g = j & 1
            s = pg[g]
            pg[g] = s + 2 if s + 2 < S else g
            fills.append((s, ("g%d" % g,)))
    seqs = {}
    for grp in (0, 1):
        seq, cs = [], 0
        for _ in range(n_gate):
            seq.append(cs)
            cs = cs + 1 if cs + 1 < S else 0
        if old_down_scheme:
            st = cs
            for j in range(n_down):
                if (j & 1) == grp:
                    seq.append((st + j) % S)
        else:
            gs = grp
            for j in range(n_down):
                if (j & 1) == grp:
                    seq.append(gs)
                    gs = gs + 2 if gs + 2 < S else grp
        seqs["g%d" % grp] = seq
    return fills, seqs


@pytest.mark.parametrize("S", [4, 5, 6, 7, 8])
def test_bf16_ring_every_wait_follows_a_consumed_fill(S):
    for n_gate in range(0, 36):
        for n_down in range(0, 36):
            assert _check(*bf16_ring(n_gate, n_down, S)) == 0, (S, n_gate, n_down)


def test_old_shared_odd_ring_is_caught():
    # the scheme that let a group pass a wait one phase early (a GPU fault)
    bad = sum(_check(*bf16_ring(10, n_down, 5, old_down_scheme=True)) for n_down in range(4, 30))
    assert bad > 0
    # with an even ring the same alternation happens to stay sound
    assert all(_check(*bf16_ring(10, n, 4, old_down_scheme=True)) == 0 for n in range(30))


def mx_ring(units_g, units_d, nq, ring=8, groups=4):
    """layer_fused_bs.cu: rounds of one stage per group, round robin over
    the ring (a group without a unit in a round still gets a stage, filled
    empty); group q's stages are q, q + groups, ..."""
    R2 = -(-units_g // groups)
    R3 = -(-units_d // groups)
    fills, ps = [], 0
    for _ in range(R2):
        for _ in range(nq):
            for gq in range(groups):
                fills.append((ps, ("q%d" % gq,)))
                ps = (ps + 1) % ring
    for _ in range(R3):
        for gq in range(groups):
            fills.append((ps, ("q%d" % gq,)))
            ps = (ps + 1) % ring
    seqs = {}
    for grp in range(groups):
        seq, cs = [], grp
        for _ in range(R2 * nq + R3):
            seq.append(cs)
            cs = (cs + groups) % ring
        seqs["q%d" % grp] = seq
    return fills, seqs


def test_mxfp4_ring_groups_own_their_stages():
    for units_g in range(0, 40, 3):
        for units_d in range(0, 40, 5):
            for nq in (1, 2, 4):
                assert _check(*mx_ring(units_g, units_d, nq)) == 0


def test_mxfp4_down_units_wait_for_exactly_the_owner_ctas():
    """layer_fused_bs.cu: CTA b takes gate/up units [floor(bU/G),
    floor((b+1)U/G)).  Before a down group reads expert wi's h it waits for
    the flags of CTAs b0..b1, from the closed form owner(u) =
    floor(((u+1)G - 1)/U).  Every CTA holding one of the expert's units must be
    in that range (a missing one is a race on h), and both ends must hold one.
    A CTA strictly inside the range may hold no unit at all (more CTAs than
    units); it sets its flag as soon as its empty gate/up phase ends, so the
    wait for it is short and harmless."""
    for G in (1, 2, 7, 152, 160):
        for tiles_g in (1, 2, 16, 64, 96):
            for nW in (1, 2, 3, 9, 47, 103, 257):
                U = nW * tiles_g
                owner = [None] * U
                for b in range(G):
                    for u in range(b * U // G, (b + 1) * U // G):
                        assert owner[u] is None
                        owner[u] = b
                assert None not in owner
                assert all(owner[u] == ((u + 1) * G - 1) // U for u in range(0, U, max(1, U // 97)))
                for wi in {0, nW // 2, nW - 1}:
                    b0 = ((wi * tiles_g + 1) * G - 1) // U
                    b1 = (((wi + 1) * tiles_g) * G - 1) // U
                    owners = set(owner[wi * tiles_g:(wi + 1) * tiles_g])
                    assert owners <= set(range(b0, b1 + 1)) and b0 in owners and b1 in owners
                    for b in set(range(b0, b1 + 1)) - owners:
                        assert b * U // G == (b + 1) * U // G  # an idle CTA
