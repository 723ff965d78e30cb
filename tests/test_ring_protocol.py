"""The weight-gradient kernel's resident-slot ring, as a host-side model (no GPU).

The resident operand's k-blocks pass through a ring of RSLOTS shared-memory
slots that spans the work units a CTA pair runs in turn.  Three rules, the
same as in the kernel (csrc/gemm_res.cuh):

* fills go round the ring in order; a fill waits until the last UMMA that
  read its slot has released it;
* the gather warps signal a fill LAG = 2 fills later, and signal every
  outstanding fill when a unit's fills are done;
* the UMMA issuer waits for a unit's blocks on its first tile and releases
  each slot after the unit's last tile has read it (a streamed unit has one
  tile, so each of its blocks is released as soon as it is read).

The model runs both sides as a two-party scheduler and checks that it never
deadlocks, that no slot is refilled while a unit still reads it, and that
with six slots the next unit's first two blocks land while the running unit
computes (the point of a ring deeper than one unit).
"""

import random

import pytest

LAG = 2


def simulate(units, rslots, eager_gather=True):
    """units: list of (kblocks, ntiles).  eager_gather: the gather side moves
    whenever it can (as the kernel's gather warps do, independently of the
    issuer); otherwise only when the issuer is blocked.  Returns the event
    log, or raises on deadlock or on a slot refilled while in use."""
    fills = [(u, kb) for u, (kbs, _) in enumerate(units) for kb in range(kbs)]
    slot_of = {f: i % rslots for i, f in enumerate(fills)}
    released = {s: True for s in range(rslots)}    # slot free for its next fill
    signalled = set()                               # fills the issuer may read
    pending = []                                    # filled, not yet signalled
    in_use = {}                                     # slot -> fill it holds
    log = []
    gi = 0                                          # next fill index
    # issuer position: unit, tile, kb
    mu, mj, mk = 0, 0, 0

    def gather_step():
        nonlocal gi
        if gi >= len(fills):
            return False
        f = fills[gi]
        s = slot_of[f]
        if not released[s]:
            return False
        assert s not in in_use, f"slot {s} refilled while {in_use.get(s)} is in use"
        released[s] = False
        in_use[s] = f
        pending.append(f)
        log.append(("fill", f))
        gi += 1
        if len(pending) > LAG:
            signalled.add(pending.pop(0))
        last_of_unit = gi == len(fills) or fills[gi][0] != f[0]
        if last_of_unit:
            while pending:
                signalled.add(pending.pop(0))
        return True

    def issuer_step():
        nonlocal mu, mj, mk
        while mu < len(units) and (units[mu][0] == 0 or units[mu][1] == 0):
            mu += 1  # a unit with nothing to read: its tiles need no slot
        if mu >= len(units):
            return False
        kbs, nt = units[mu]
        f = (mu, mk)
        if mj == 0 and f not in signalled:
            return False
        log.append(("read", f, mj))
        if mj == nt - 1:  # last tile: the slot goes back to the ring
            s = slot_of[f]
            del in_use[s]
            released[s] = True
            log.append(("release", f))
        mk += 1
        if mk == kbs:
            mk = 0
            mj += 1
            if mj == nt:
                mj = 0
                mu += 1
        return True

    def issuer_done():
        return mu >= len(units) or all(k == 0 or t == 0 for k, t in units[mu:])

    while gi < len(fills) or not issuer_done():
        if eager_gather:
            progressed = gather_step() or issuer_step()
        else:
            progressed = issuer_step() or gather_step()
        if not progressed:
            raise RuntimeError(f"deadlock at fill {gi}, issuer unit {mu} tile {mj} kb {mk}")
    return log


def _random_units(rng, n):
    units = []
    for _ in range(n):
        kind = rng.random()
        if kind < 0.6:
            units.append((rng.randint(1, 4), rng.randint(1, 8)))    # resident unit
        elif kind < 0.9:
            units.append((rng.randint(5, 40), 1))                   # streamed tile
        else:
            units.append((0, rng.randint(1, 8)))                    # an expert with no rows
    return units


@pytest.mark.parametrize("eager", [True, False])
@pytest.mark.parametrize("rslots", [4, 5, 6, 7, 8])
def test_ring_never_deadlocks_nor_overwrites(rslots, eager):
    rng = random.Random(rslots)
    for _ in range(200):
        simulate(_random_units(rng, rng.randint(1, 20)), rslots, eager)


def test_ring_must_be_deeper_than_the_signal_lag():
    # a streamed unit longer than the ring: with RSLOTS <= LAG the gather
    # would wait for a slot whose fill it has not signalled yet
    for eager in (True, False):
        with pytest.raises(RuntimeError, match="deadlock"):
            simulate([(12, 1)], LAG, eager)


def _first_fill_before_last_tile(log, unit):
    """Index in the log of unit+1's first fill and of unit's last-tile first read."""
    first_fill = next(i for i, e in enumerate(log) if e[0] == "fill" and e[1][0] == unit + 1)
    last_tile = max(e[2] for e in log if e[0] == "read" and e[1][0] == unit)
    start_last = next(i for i, e in enumerate(log)
                      if e[0] == "read" and e[1][0] == unit and e[2] == last_tile)
    return first_fill, start_last


def test_six_slots_fetch_the_next_unit_during_the_current_one():
    units = [(4, 6)] * 5                      # balanced experts: 4 k-blocks, 6 tiles each
    # four slots: the next unit's first fill needs a slot the current unit
    # releases only on its last tile
    log4 = simulate(units, 4)
    ff, lt = _first_fill_before_last_tile(log4, 1)
    assert ff > lt
    # six slots: its first two blocks go into slots the current unit never used
    log6 = simulate(units, 6)
    ff, lt = _first_fill_before_last_tile(log6, 1)
    assert ff < lt
    early = [e for e in log6[:lt] if e[0] == "fill" and e[1][0] == 2]
    assert len(early) == 2
