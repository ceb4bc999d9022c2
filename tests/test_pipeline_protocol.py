"""Host simulation of the warp-role pipeline protocol (no GPU).

The kernel's roles talk only through mbarriers:
* operand ring: the producer waits ``consumed[s]`` with parity ``((phase // S) & 1) ^ 1``,
  fills slot ``s = phase % S`` and completes ``loaded[s]``; the MMA role waits
  ``loaded[s]`` with parity ``(phase // S) & 1``, reads slot ``s`` and completes
  ``consumed[s]``, with ``phase = w * k_blocks + k`` on both sides
  ("[Feature] Introduce tile scheduler #2441", gemm_tcgen5mma_ws_persistent.py,
  ``gemm_persistent`` TMA and MMA loops; the review comment on that file asks for
  ``phase % num_stages`` in the consumer too, which this model uses);
* accumulator double buffer: the MMA role waits ``tmem_empty[w & 1]`` with parity
  ``((w // 2) & 1) ^ 1`` and completes ``tmem_full[w & 1]``; the epilogue waits
  ``tmem_full[w & 1]`` with parity ``(w // 2) & 1`` and completes ``tmem_empty[w & 1]``.

An mbarrier is modelled by its phase counter: a wait on parity ``P`` passes when the
phase with that parity has completed, i.e. when ``P != phase_count & 1``.  The roles are
interleaved at random; the model checks that every read sees the data written for the
same (w, k), that no slot is refilled before it was read, and that nothing deadlocks.
"""

import random

import pytest


class Barrier:
    def __init__(self):
        self.phase = 0

    def passes(self, parity):
        return parity != (self.phase & 1)

    def complete(self):
        self.phase += 1


def slot_of(phase, S):
    return phase % S


def parity_of(phase, S):
    return (phase // S) & 1


def run_ring(S, k_blocks, waves, seed, consumer_slot=None):
    """Returns None if the protocol held, else a string naming the violation."""
    rng = random.Random(seed)
    loaded = [Barrier() for _ in range(S)]
    consumed = [Barrier() for _ in range(S)]
    data = [None] * S
    unread = [False] * S
    total = waves * k_blocks
    prod = 0
    cons = 0
    cslot = consumer_slot or (lambda w, k, phase: slot_of(phase, S))
    while cons < total:
        moves = []
        if prod < total and consumed[slot_of(prod, S)].passes(parity_of(prod, S) ^ 1):
            moves.append("p")
        if cons < total:
            w, k = divmod(cons, k_blocks)
            s = cslot(w, k, cons)
            if loaded[s].passes(parity_of(cons, S)):
                moves.append("c")
        if not moves:
            return f"deadlock at producer {prod}, consumer {cons}"
        if rng.choice(moves) == "p":
            s = slot_of(prod, S)
            if unread[s]:
                return f"slot {s} refilled before it was read (phase {prod})"
            data[s] = prod
            unread[s] = True
            loaded[s].complete()
            prod += 1
        else:
            w, k = divmod(cons, k_blocks)
            s = cslot(w, k, cons)
            if data[s] != cons:
                return f"phase {cons} read the data of phase {data[s]}"
            unread[s] = False
            consumed[s].complete()
            cons += 1
    return None


def run_accumulators(waves, seed):
    rng = random.Random(seed)
    full = [Barrier(), Barrier()]
    empty = [Barrier(), Barrier()]
    acc = [None, None]
    mma = 0
    epi = 0
    while epi < waves:
        moves = []
        if mma < waves and empty[mma & 1].passes(((mma // 2) & 1) ^ 1):
            moves.append("m")
        if epi < waves and full[epi & 1].passes((epi // 2) & 1):
            moves.append("e")
        if not moves:
            return f"deadlock at mma {mma}, epilogue {epi}"
        if rng.choice(moves) == "m":
            if acc[mma & 1] is not None:
                return f"accumulator {mma & 1} overwritten before it was drained (w={mma})"
            acc[mma & 1] = mma
            full[mma & 1].complete()
            mma += 1
        else:
            if acc[epi & 1] != epi:
                return f"w={epi} drained the accumulator of w={acc[epi & 1]}"
            acc[epi & 1] = None
            empty[epi & 1].complete()
            epi += 1
    return None


@pytest.mark.parametrize("S", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("k_blocks", [1, 2, 3, 4, 7, 32])
def test_ring_protocol_holds(S, k_blocks):
    for seed in range(40):
        assert run_ring(S, k_blocks, waves=5, seed=seed) is None


@pytest.mark.parametrize("waves", [1, 2, 3, 4, 9])
def test_accumulator_double_buffer_holds(waves):
    for seed in range(60):
        assert run_accumulators(waves, seed) is None


def test_consumer_indexing_slots_by_k_is_caught():
    # the slot function flagged in review: consumer reads k % S while the producer
    # writes phase % S; wrong whenever k_blocks % S != 0 and a CTA runs >= 2 tiles
    S, k_blocks = 4, 3
    bad = lambda w, k, phase: k % S
    failures = [run_ring(S, k_blocks, waves=3, seed=s, consumer_slot=bad) for s in range(20)]
    assert all(f is not None for f in failures)
    # ...and invisible when k_blocks is a multiple of S (why it went unnoticed)
    assert all(run_ring(4, 8, 3, s, consumer_slot=bad) is None for s in range(20))


def test_parities_match_the_generated_sm90_pipeline():
    # "tilelang" (generated kernel source of the 3-stage sm_90 GEMM): the consumer waits
    # barrier k % 3 with parity (k % 6) / 3 and the producer waits barrier k % 3 + 3 with
    # parity ((k % 6) / 3) ^ 1 -- the same functions as phase % S and (phase // S) & 1
    for k in range(1000):
        assert slot_of(k, 3) == k % 3
        assert parity_of(k, 3) == (k % 6) // 3
        assert parity_of(k, 3) ^ 1 == ((k % 6) // 3) ^ 1


# ---------------------------------------------------------------- unit-response ring
# Dynamic persistence: warp 3 fetches units by cancelling pending CTAs into a ring of
# ``slots`` 16-byte responses.  Fetch j (the unit after the CTA's iteration j) lands in slot
# ``j % slots`` and completes ``full[slot]``; each of ``consumers`` readers (producer, MMA,
# four epilogue warps) reads it after waiting ``full[slot]`` with parity
# ``(j // slots) & 1`` and arrives on ``empty[slot]`` (arrival count ``consumers``); the
# fetcher waits ``empty[slot]`` with parity ``((j // slots) & 1) ^ 1`` before reusing it.
# A response that cancelled nothing (``None``) ends the traversal of every role.
# ``first`` shifts the fetch numbering: the kernel once numbered fetches from 1, so the
# first use of slot 0 waited on parity 1, which a fresh barrier passes at once.


class CountBarrier(Barrier):
    def __init__(self, count):
        super().__init__()
        self.count = count
        self.arrived = 0

    def arrive(self):
        self.arrived += 1
        if self.arrived == self.count:
            self.arrived = 0
            self.complete()


def run_response_ring(slots, consumers, pending, seed, first=0):
    rng = random.Random(seed)
    full = [Barrier() for _ in range(slots)]
    empty = [CountBarrier(consumers) for _ in range(slots)]
    resp = [("unwritten",)] * slots
    unread = [0] * slots
    queue = list(range(100, 100 + pending))   # units of CTAs not launched yet
    fetched = []                              # response of each fetch, in order
    f_j, f_state, f_done = 0, "wait_empty", False
    c_j = [0] * consumers
    c_done = [False] * consumers
    while not (f_done and all(c_done)):
        moves = []
        i = f_j + first
        s, par = i % slots, (i // slots) & 1
        if not f_done:
            if f_state == "wait_empty" and empty[s].passes(par ^ 1):
                moves.append(("f_issue",))
            elif f_state == "in_flight":
                moves.append(("f_land",))
            elif f_state == "wait_full" and full[s].passes(par):
                moves.append(("f_read",))
        for c in range(consumers):
            if not c_done[c]:
                i = c_j[c] + first
                if full[i % slots].passes((i // slots) & 1):
                    moves.append(("c", c))
        if not moves:
            return f"deadlock: fetcher at {f_j} ({f_state}), readers at {c_j}"
        mv = rng.choice(moves)
        if mv[0] == "f_issue":
            if unread[s]:
                return f"slot {s} reissued while {unread[s]} readers still owe a read"
            f_state = "in_flight"
        elif mv[0] == "f_land":
            r = queue.pop(0) if queue else None
            resp[s] = (f_j, r)
            fetched.append(r)
            unread[s] = consumers
            full[s].complete()
            f_state = "wait_full"
        elif mv[0] == "f_read":
            if resp[s] != (f_j, fetched[f_j] if f_j < len(fetched) else "?"):
                return f"fetcher read {resp[s]} for fetch {f_j}"
            if resp[s][1] is None:
                f_done = True
            else:
                f_j, f_state = f_j + 1, "wait_empty"
        else:
            c = mv[1]
            i = c_j[c] + first
            sl = i % slots
            if resp[sl][0] != c_j[c]:
                return f"reader {c} took {resp[sl]} for fetch {c_j[c]}"
            unread[sl] -= 1
            empty[sl].arrive()
            if resp[sl][1] is None:
                c_done[c] = True
            c_j[c] += 1
    if fetched[:-1] != list(range(100, 100 + pending)) or fetched[-1] is not None:
        return f"fetched {fetched}"
    return None


@pytest.mark.parametrize("slots", [1, 2, 3])
@pytest.mark.parametrize("pending", [0, 1, 2, 3, 7])
def test_response_ring_holds(slots, pending):
    for seed in range(60):
        assert run_response_ring(slots, 6, pending, seed) is None


def test_response_ring_numbered_from_one_is_caught():
    # fetches numbered from 1: the first use of slot 0 waits on parity 1 and passes at
    # once on a fresh barrier, so a reader takes a response that was never written
    failures = [run_response_ring(2, 6, 3, seed, first=1) for seed in range(40)]
    assert all(f is not None for f in failures)


# ---------------------------------------------------------------- MXFP8 scale path
# The block-scaled kernel's roles: the producer arms loaded[s] (expect_tx, one arrival) and its
# TMA bytes land later; the transpose role waits atom_free[a] (a = phase % A) for the phase
# that last used the slot, writes the atoms and arrives on sf_ready[a]; the MMA role waits
# loaded[s] and sf_ready[a], reads both, and commits consumed[s] and atom_free[a].  The model
# tracks each barrier's pending arrivals and transaction bytes, so a phase that completes
# before the producer armed it is seen.  ``shared_loaded`` is the design that failed on the
# GPU: the transpose arriving on loaded[s] (count 2) instead of a barrier of its own, which
# lets it complete phase p of loaded[s] early once it runs S or more phases ahead.


class TxBarrier(Barrier):
    def __init__(self, count):
        super().__init__()
        self.count = count
        self.pending = count
        self.tx = 0
        self.armed = False

    def arrive(self, expect_tx=0, armed=False):
        self.tx += expect_tx
        self.armed = self.armed or armed
        self.pending -= 1
        return self._check()

    def land(self, nbytes):
        self.tx -= nbytes
        return self._check()

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            early = not self.armed
            self.pending = self.count
            self.armed = False
            self.complete()
            return "early" if early else "ok"
        return None


def run_mx_scales(S, A, k_total, seed, shared_loaded=False):
    rng = random.Random(seed)
    loaded = [TxBarrier(2 if shared_loaded else 1) for _ in range(S)]
    consumed = [Barrier() for _ in range(S)]
    sf_ready = [Barrier() for _ in range(A)]
    atom_free = [Barrier() for _ in range(A)]
    stage = [None] * S          # phase whose operands sit in stage s
    atoms = [None] * A          # phase whose scales sit in atom slot a
    in_flight = []              # (stage, phase) TMA fills not landed yet
    prod = tr = mma = 0
    while mma < k_total:
        moves = []
        if prod < k_total and consumed[prod % S].passes(((prod // S) & 1) ^ 1):
            moves.append("p")
        if in_flight:
            moves.append("land")
        if tr < k_total and (tr < A or atom_free[tr % A].passes(((tr // A) & 1) ^ 1)):
            moves.append("t")
        s, a = mma % S, mma % A
        ready = loaded[s].passes((mma // S) & 1)
        if not shared_loaded:
            ready = ready and sf_ready[a].passes((mma // A) & 1)
        if ready:
            moves.append("m")
        if not moves:
            return f"deadlock: producer {prod}, transpose {tr}, mma {mma}"
        mv = rng.choice(moves)
        if mv == "p":
            s = prod % S
            if loaded[s].arrive(expect_tx=1, armed=True) == "early":
                return f"loaded[{s}] completed before phase {prod} was armed"
            in_flight.append((s, prod))
            prod += 1
        elif mv == "land":
            s, ph = in_flight.pop(rng.randrange(len(in_flight)))
            stage[s] = ph
            if loaded[s].land(1) == "early":
                return f"loaded[{s}] completed early (phase {ph})"
        elif mv == "t":
            a = tr % A
            atoms[a] = tr
            if shared_loaded:
                if loaded[tr % S].arrive() == "early":
                    return f"loaded[{tr % S}] completed before phase {tr} was armed"
            else:
                sf_ready[a].complete()
            tr += 1
        else:
            s, a = mma % S, mma % A
            if stage[s] != mma:
                return f"MMA phase {mma} read the operands of phase {stage[s]}"
            if atoms[a] != mma:
                return f"MMA phase {mma} read the scales of phase {atoms[a]}"
            consumed[s].complete()
            atom_free[a].complete()
            mma += 1
    return None


@pytest.mark.parametrize("S,A", [(4, 8), (4, 4), (4, 3), (3, 8), (2, 5)])
def test_mx_scale_path_holds(S, A):
    for seed in range(150):
        assert run_mx_scales(S, A, 40, seed) is None, (S, A, seed)


def test_mx_scales_arriving_on_loaded_are_caught():
    # 8 atom slots let the transpose role run 7 phases ahead: with its arrival on loaded[s],
    # some interleaving completes a phase of loaded[s] before the producer armed it
    failures = [run_mx_scales(4, 8, 40, seed, shared_loaded=True) for seed in range(150)]
    assert any(f is not None for f in failures)


# ---------------------------------------------------------------- MXFP8 pair: scales by the epilogue
# The CTA-pair MXFP8 kernel (tg_mx_pair_kernel.cuh) writes the TMEM scale slots from its
# epilogue warps, through a scale ring of A = S + D slots that runs D phases ahead of the
# operand ring.  The producer loads the atoms of phases 0 .. D - 1 first; then per phase p it
# waits consumed[p % S] (parity ((p // S) & 1) ^ 1), loads the atoms of phase p + D into scale
# slot (p + D) % A (arming sf_loaded of that slot) and the operands of p (arming loaded[s]);
# the bytes land later in any order.  The MMA role waits tmem_empty with parity (w & 1) ^ 1
# before unit w (one accumulator), then per phase loaded[p % S] (parity (p // S) & 1) and
# sf_ready[p % A] (parity (p // A) & 1), and commits consumed[p % S]; after the unit's last
# phase it completes tmem_full.  The epilogue is one sequential agent: it polls, draining unit
# w once tmem_full passes with parity w & 1 and otherwise writing the scale slot of its next
# phase q once sf_loaded[q % A] passes with parity (q // A) & 1; after a drain it arrives on
# tmem_empty and stores four chunks, trying one scale slot before each chunk after the first.
# ``polling=False`` is the design that waits for tmem_full before writing any slot of the
# unit: it deadlocks.  ``slots`` below S + D lets a load overwrite atoms or a TMEM slot that is
# still in use.


def run_mx_pair_epilogue(S, k_stages, units, seed, D=2, polling=True, slots=None):
    rng = random.Random(seed)
    A = S + D if slots is None else slots
    consumed = [Barrier() for _ in range(S)]
    loaded = [TxBarrier(1) for _ in range(S)]
    sf_loaded = [TxBarrier(1) for _ in range(A)]
    sf_ready = [Barrier() for _ in range(A)]
    tmem_full, tmem_empty = Barrier(), Barrier()
    total = units * k_stages
    stage = [None] * S       # phase whose operands sit in ring slot s
    atoms = [None] * A       # phase whose atoms sit in shared-memory scale slot a
    slot = [None] * A        # phase whose scales sit in TMEM scale slot a
    in_flight = []           # (what, slot, phase) loads not landed yet
    prod = mma = ps = wd = 0
    sf_next = 0              # phase whose atoms the producer loads next
    entered = False          # the MMA role has passed tmem_empty for its current unit
    acc = None               # unit whose finished sum the accumulator holds
    chunks = 0               # chunks of the drained unit still to store

    def load_atoms():
        nonlocal sf_next
        if sf_next >= total:
            return None
        a = sf_next % A
        if sf_loaded[a].arrive(expect_tx=1, armed=True) == "early":
            return f"sf_loaded[{a}] completed before phase {sf_next} was armed"
        in_flight.append(("sf", a, sf_next))
        sf_next += 1
        return None

    def write_scale():
        nonlocal ps
        a = ps % A
        if atoms[a] != ps:
            return f"scale slot of phase {ps} written from the atoms of phase {atoms[a]}"
        if slot[a] is not None and mma <= slot[a]:
            return f"scale slot {a} rewritten (phase {ps}) before phase {slot[a]} was consumed"
        slot[a] = ps
        sf_ready[a].complete()
        ps += 1
        return None

    def scale_ready():
        return ps < total and sf_loaded[ps % A].passes((ps // A) & 1)

    for _ in range(D):
        err = load_atoms()
        if err:
            return err
    while wd < units:
        moves = []
        if prod < total and consumed[prod % S].passes(((prod // S) & 1) ^ 1):
            moves.append("p")
        if in_flight:
            moves.append("land")
        if mma < total:
            w, s, a = mma // k_stages, mma % S, mma % A
            if mma % k_stages == 0 and not entered:
                if tmem_empty.passes((w & 1) ^ 1):
                    moves.append("m")
            elif loaded[s].passes((mma // S) & 1) and sf_ready[a].passes((mma // A) & 1):
                moves.append("m")
        if chunks:
            moves.append("e")
        elif tmem_full.passes(wd & 1) or (polling and scale_ready()):
            moves.append("e")
        if not moves:
            return f"deadlock: producer {prod}, scales {ps}, mma {mma}, drain {wd}"
        mv = rng.choice(moves)
        if mv == "p":
            s = prod % S
            err = load_atoms()
            if err:
                return err
            if loaded[s].arrive(expect_tx=1, armed=True) == "early":
                return f"loaded[{s}] completed before phase {prod} was armed"
            in_flight.append(("op", s, prod))
            prod += 1
        elif mv == "land":
            what, s, ph = in_flight.pop(rng.randrange(len(in_flight)))
            if what == "op":
                stage[s] = ph
                done = loaded[s].land(1)
            else:
                if atoms[s] is not None and ps <= atoms[s]:
                    return f"atoms of phase {atoms[s]} overwritten before they were read"
                atoms[s] = ph
                done = sf_loaded[s].land(1)
            if done == "early":
                return f"{what}[{s}] completed early (phase {ph})"
        elif mv == "m":
            w, s, a = mma // k_stages, mma % S, mma % A
            if mma % k_stages == 0 and not entered:
                entered = True
                continue
            if stage[s] != mma:
                return f"MMA phase {mma} read the operands of phase {stage[s]}"
            if slot[a] != mma:
                return f"MMA phase {mma} read the scales of phase {slot[a]}"
            consumed[s].complete()
            mma += 1
            if mma % k_stages == 0:
                acc = w
                entered = False
                tmem_full.complete()
        elif chunks:
            if chunks < 4 and scale_ready():
                err = write_scale()
                if err:
                    return err
            chunks -= 1
            if chunks == 0:
                wd += 1
        elif tmem_full.passes(wd & 1):
            if acc != wd:
                return f"drain of unit {wd} read the accumulator of unit {acc}"
            tmem_empty.complete()
            chunks = 4
        else:
            err = write_scale()
            if err:
                return err
    return None


@pytest.mark.parametrize("S,D,k_stages", [(3, 2, 1), (3, 2, 2), (3, 2, 5), (3, 0, 3), (2, 3, 3),
                                          (4, 1, 7)])
def test_mx_pair_epilogue_scale_path_holds(S, D, k_stages):
    for seed in range(150):
        assert run_mx_pair_epilogue(S, k_stages, 6, seed, D=D) is None, (S, D, k_stages, seed)


def test_mx_pair_scales_written_only_after_the_drain_deadlock():
    assert run_mx_pair_epilogue(3, 4, 3, 0, polling=False).startswith("deadlock")


def test_mx_pair_scale_ring_shorter_than_operands_plus_lead_is_caught():
    # with A = S + D - 1 slots, loading phase p + D's atoms after consumed of p - S reuses the
    # slot of phase p - S + 1, which may not have been read yet
    failures = [run_mx_pair_epilogue(3, 4, 4, seed, D=2, slots=4) for seed in range(150)]
    assert any(f is not None and "deadlock" not in f for f in failures)


# ---------------------------------------------------------------- wide pair accumulator
# The wide pair kernel (tg_gemm_pair_wide_kernel.cuh) has one accumulator made of two N-halves
# (TMEM columns 0..255 and 256..511) in each CTA of the pair.  The MMA role (even CTA) writes
# half h of unit w from its first k-block on, after waiting tmem_empty[h] with parity
# (w & 1) ^ 1; after the unit it completes tmem_full in both CTAs.  Each CTA's epilogue waits
# tmem_full with parity w & 1, reads the halves the unit uses and arrives on tmem_empty[h] of
# the even CTA (count: both CTAs' epilogues); a half unit (one N-half) hands its unused half
# back at once, so both barriers complete once per unit.


def run_wide_accumulator(halves, k_blocks, seed, release_unused=True):
    """halves[w] in {1, 2}: the N-halves unit w uses.  Returns None or the first violation."""
    rng = random.Random(seed)
    units = len(halves)
    full = [Barrier(), Barrier()]                    # one per CTA, completed together
    empty = [CountBarrier(2), CountBarrier(2)]       # per N-half, in the even CTA
    acc = [[None, None], [None, None]]               # acc[cta][h] = [unit, k-blocks written, read?]
    mma = {"w": 0, "k": 0, "h": 0}
    epi = [{"w": 0, "h": 0, "waiting": True}, {"w": 0, "h": 0, "waiting": True}]
    while any(e["w"] < units for e in epi):
        moves = []
        w, k, h = mma["w"], mma["k"], mma["h"]
        if w < units:
            if k > 0 or empty[h].passes((w & 1) ^ 1):
                moves.append(("mma",))
        for c in (0, 1):
            e = epi[c]
            if e["w"] >= units:
                continue
            if e["waiting"]:
                if full[c].passes(e["w"] & 1):
                    moves.append(("epi_start", c))
            else:
                moves.append(("epi_half", c))
        if not moves:
            return f"deadlock: mma {mma}, epilogues {epi}"
        move = rng.choice(moves)
        if move[0] == "mma":
            for c in (0, 1):
                cur = acc[c][h]
                if k == 0:
                    if cur is not None and not cur[2]:
                        return f"unit {w} overwrote half {h} of CTA {c} before unit {cur[0]} was read"
                    acc[c][h] = [w, 1, False]
                else:
                    if cur is None or cur[0] != w:
                        return f"unit {w} accumulated into half {h} of CTA {c} owned by {cur}"
                    cur[1] += 1
            # next MMA step: halves in order inside a k-block, then the next k-block
            if h + 1 < halves[w]:
                mma["h"] = h + 1
            else:
                mma["h"] = 0
                if k + 1 < k_blocks:
                    mma["k"] = k + 1
                else:
                    full[0].complete()
                    full[1].complete()
                    mma.update(w=w + 1, k=0, h=0)
        elif move[0] == "epi_start":
            epi[move[1]]["waiting"] = False
        else:
            c = move[1]
            e = epi[c]
            hh = e["h"]
            if hh < halves[e["w"]]:
                cur = acc[c][hh]
                if cur is None or cur[0] != e["w"] or cur[1] != k_blocks:
                    return f"CTA {c} read half {hh} of unit {e['w']} as {cur}"
                cur[2] = True
                empty[hh].arrive()
            elif release_unused:
                empty[hh].arrive()
            if hh == 1:
                e.update(w=e["w"] + 1, h=0, waiting=True)
            else:
                e["h"] = 1
    return None


@pytest.mark.parametrize("halves", [[2], [2, 2, 2], [2, 2, 1], [1], [2, 1, 2, 1, 2], [1, 1, 2]])
@pytest.mark.parametrize("k_blocks", [1, 2, 5])
def test_wide_accumulator_protocol_holds(halves, k_blocks):
    for seed in range(60):
        assert run_wide_accumulator(halves, k_blocks, seed) is None


def test_wide_half_unit_must_hand_back_its_unused_half():
    # without the immediate hand-back, the unit after a half unit waits forever on half 1
    results = [run_wide_accumulator([2, 1, 2], 2, seed, release_unused=False) for seed in range(20)]
    assert all(r is not None and r.startswith("deadlock") for r in results)


# ---------------------------------------------------------------- wide pair: ring + accumulator
# The wide pair kernel's MMA role ties the operand ring to the accumulator hand-back: at the
# start of a whole unit it may run N-half 0 of the first ``defer`` k-blocks before the epilogues
# have handed N-half 1 of the previous unit back, holding those ring slots until half 1 has
# read them too (kWideDefer in tg_wide_config.h).  This model runs the producer, the MMA role
# in the kernel's issue order and both CTAs' epilogues as coroutines on modelled mbarriers,
# interleaved at random, and checks that every MMA reads the k-block of its own phase, that a
# slot is refilled only after every half that needs it has read it, that each half of the
# accumulator receives its unit's k-blocks in order before being read and is read only once
# complete, and that nothing deadlocks.


def run_wide_pipeline(halves, k_blocks, S, defer, seed, catch_up_commits=True):
    rng = random.Random(seed)
    units = len(halves)
    loaded = [Barrier() for _ in range(S)]
    consumed = [Barrier() for _ in range(S)]
    full = [Barrier(), Barrier()]
    empty = [CountBarrier(2), CountBarrier(2)]
    data = [None] * S
    need = [set() for _ in range(S)]        # halves that still have to read the slot
    acc = [[None, None], [None, None]]      # [unit, k-blocks written, read?] per CTA and half
    errors = []

    def fail(msg):
        errors.append(msg)
        raise StopIteration

    def producer():
        for w in range(units):
            for k in range(k_blocks):
                ph = w * k_blocks + k
                s = slot_of(ph, S)
                yield consumed[s], parity_of(ph, S) ^ 1
                if need[s]:
                    errors.append(f"slot {s} refilled (phase {ph}) before halves {need[s]} read it")
                    return
                data[s] = ph
                need[s] = set(range(halves[w]))
                loaded[s].complete()

    def op(w, h, k):
        ph = w * k_blocks + k
        s = slot_of(ph, S)
        if data[s] != ph:
            return f"unit {w} half {h} k {k} read slot {s} holding phase {data[s]}"
        need[s].discard(h)
        for c in (0, 1):
            cur = acc[c][h]
            if k == 0:
                if cur is not None and not cur[2]:
                    return f"unit {w} overwrote half {h} of CTA {c} before unit {cur[0]} was read"
                acc[c][h] = [w, 1, False]
            else:
                if cur is None or cur[0] != w or cur[1] != k:
                    return f"unit {w} half {h} k-block {k} accumulated onto {cur}"
                cur[1] += 1
        return None

    def commit(w, k):
        s = slot_of(w * k_blocks + k, S)
        if need[s]:
            return f"slot {s} released with halves {need[s]} unread"
        consumed[s].complete()
        return None

    def mma():
        for w in range(units):
            d = min(defer, k_blocks - 1) if halves[w] == 2 else 0
            for k in range(k_blocks):
                ph = w * k_blocks + k
                yield loaded[slot_of(ph, S)], parity_of(ph, S)
                if k == 0:
                    yield empty[0], (w & 1) ^ 1
                for m in (op(w, 0, k),):
                    if m:
                        errors.append(m)
                        return
                if halves[w] == 1:
                    m = commit(w, k)
                    if m:
                        errors.append(m)
                        return
                    continue
                if k < d:
                    continue
                if k == d:
                    yield empty[1], (w & 1) ^ 1
                    for j in range(d):
                        m = op(w, 1, j) or (commit(w, j) if catch_up_commits else None)
                        if m:
                            errors.append(m)
                            return
                m = op(w, 1, k) or commit(w, k)
                if m:
                    errors.append(m)
                    return
            full[0].complete()
            full[1].complete()

    def epilogue(c):
        for w in range(units):
            yield full[c], w & 1
            for h in (0, 1):
                if h < halves[w]:
                    cur = acc[c][h]
                    if cur is None or cur[0] != w or cur[1] != k_blocks:
                        errors.append(f"CTA {c} read half {h} of unit {w} as {cur}")
                        return
                    cur[2] = True
                empty[h].arrive()

    roles = {"producer": producer(), "mma": mma(), "epi0": epilogue(0), "epi1": epilogue(1)}
    waits = {}
    for name, g in list(roles.items()):
        waits[name] = next(g, None)
    while True:
        if errors:
            return errors[0]
        live = {n: wt for n, wt in waits.items() if wt is not None}
        if not live:
            return None
        ready = [n for n, (bar, par) in live.items() if bar.passes(par)]
        if not ready:
            return f"deadlock: waiting {sorted(live)}"
        n = rng.choice(ready)
        waits[n] = next(roles[n], None)


@pytest.mark.parametrize("defer", [0, 1, 2, 3])
@pytest.mark.parametrize("halves", [[2, 2, 2], [2, 1, 2], [1, 2, 2, 1], [2], [1, 1]])
@pytest.mark.parametrize("k_blocks", [1, 2, 3, 4, 7])
def test_wide_ring_and_accumulator_hold_with_deferred_half(defer, halves, k_blocks):
    for seed in range(25):
        assert run_wide_pipeline(halves, k_blocks, 4, defer, seed) is None


def test_wide_deferral_of_every_slot_deadlocks():
    # holding all S slots for half 1 leaves the producer nothing to refill: the reason the
    # deferral is kept below the ring depth
    results = [run_wide_pipeline([2, 2, 2], 8, 4, 4, seed) for seed in range(10)]
    assert all(r is not None and r.startswith("deadlock") for r in results)


def test_wide_catch_up_without_releasing_slots_is_caught():
    results = [run_wide_pipeline([2, 2, 2], 8, 4, 2, seed, catch_up_commits=False)
               for seed in range(10)]
    assert all(r is not None for r in results)
