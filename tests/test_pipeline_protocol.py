"""A randomised model of the grouped FFN kernel's barrier protocol (`ffn.cu`, no GPU).

It models the roles that meet at the kernel's mbarriers:
- the weight-chunk producer: ring of RC slots, `c_full` / `c_empty`;
- the token-row producer: ring of RX slots, arriving on `ready`;
- two dequant sets of 8 warps, taking alternate K blocks, each warp separately: wait
  `c_full` and, for A-slot reuse, `kb_done` of block it - A, then free the chunk and arrive
  on `ready`;
- two MMA threads: wait `ready`, then commit to `kb_done`.

Completions (copies landing, MMAs finishing, warps finishing their block) are delayed at
random. The model checks that every parity wait targets the current or the preceding phase
of its barrier (otherwise the hardware's parity test would pass at once), that no slot is
overwritten while it is read, that every warp reads the block it expects, and that the run
finishes. An odd weight ring of fewer than A + 2 slots breaks the first property: a dequant
set can reach a slot's next wait while the other set's block is still pending there. The
configurations below are the kernel's. If `TmCfg` changes, the source check fails until they
are updated here.
"""
import os
import random
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KD = 8   # kTmKD: ready / kb_done barriers

# (name, RX token-row slots, RC weight-chunk slots, A TMEM A slots), as TmCfg<kDown, kBf16>
CONFIGS = [("gate/up", 8, 8, 4), ("down", 4, 6, 2), ("gate/up bf16 weights", 8, 2, 4),
           ("down bf16 weights", 2, 2, 2)]


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phase, self.tx = name, count, count, 0, 0

    def _advance(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self):
        assert self.pending > 0, f"{self.name}: arrival beyond the count"
        self.pending -= 1
        self._advance()

    def expect(self, n):
        self.tx += n
        self.arrive()

    def complete(self, n):
        self.tx -= n
        self._advance()

    def done(self, phase, who):
        """Parity wait for `phase`; only the current or the preceding phase is meaningful."""
        assert self.phase - 1 <= phase <= self.phase, \
            f"{who} waits phase {phase} of {self.name}, which is at phase {self.phase}"
        return phase < self.phase


def run(RX, RC, A, KB, ntiles, seed):
    rnd = random.Random(seed)
    NB = KB * ntiles
    c_full = [Bar(f"c_full{i}", 1) for i in range(RC)]
    c_empty = [Bar(f"c_empty{i}", 8) for i in range(RC)]
    ready = [Bar(f"ready{i}", 9) for i in range(KD)]
    kb_done = [Bar(f"kb_done{i}", 2) for i in range(KD)]
    c_slot, c_readers = [None] * RC, [set() for _ in range(RC)]
    x_busy = [None] * RX
    events, t = [], 0
    st = dict(cp=0, xp=0, mma=[0, 0])
    deq = {(s, w): s for s in (0, 1) for w in range(8)}   # next block of each warp (its set's parity)
    for _ in range(400000):
        acts = []
        it = st["cp"]
        if it < NB and (it < RC or c_empty[it % RC].done(it // RC - 1, "weight producer")):
            def load(it=it, cs=it % RC):
                assert not c_readers[cs], f"weight slot {cs} overwritten while read (block {it})"
                c_slot[cs] = None
                c_full[cs].expect(1)

                def land(it=it, cs=cs):
                    c_slot[cs] = it
                    c_full[cs].complete(1)
                events.append((t + rnd.randint(1, 30), land))
                st["cp"] += 1
            acts.append(load)
        it = st["xp"]
        if it < NB and (it < RX or kb_done[(it - RX) % KD].done((it - RX) // KD, "token producer")):
            def rows(it=it):
                assert x_busy[it % RX] is None or x_busy[it % RX] <= it - RX, "token slot still read"
                ready[it % KD].expect(1)
                events.append((t + rnd.randint(1, 30), lambda it=it: ready[it % KD].complete(1)))
                st["xp"] += 1
            acts.append(rows)
        for (s, w), it in list(deq.items()):
            if it >= NB:
                continue
            cs = it % RC
            if c_full[cs].done(it // RC, f"dequant {s}.{w}") and \
                    (it < A or kb_done[(it - A) % KD].done((it - A) // KD, f"dequant {s}.{w}")):
                def dequant(s=s, w=w, it=it, cs=cs):
                    assert c_slot[cs] == it, f"dequant {s}.{w} finds block {c_slot[cs]} for block {it}"
                    c_readers[cs].add((s, w))

                    def release(s=s, w=w, it=it, cs=cs):
                        c_readers[cs].discard((s, w))
                        c_empty[cs].arrive()
                        ready[it % KD].arrive()
                    events.append((t + rnd.randint(0, 5), release))
                    deq[(s, w)] = min(it + 2, NB)
                acts.append(dequant)
        for m in (0, 1):
            it = st["mma"][m]
            if it < NB and ready[it % KD].done(it // KD, f"mma {m}"):
                def mma(m=m, it=it):
                    x_busy[it % RX] = it
                    events.append((t + rnd.randint(1, 20), lambda it=it: kb_done[it % KD].arrive()))
                    st["mma"][m] += 1
                acts.append(mma)
        due = [e for e in events if e[0] <= t]
        if not acts and not events:
            break
        if due and (not acts or rnd.random() < 0.5):
            e = rnd.choice(due)
            events.remove(e)
            e[1]()
        elif acts:
            rnd.choice(acts)()
        t += 1
    assert st["mma"] == [NB, NB] and st["cp"] == NB and st["xp"] == NB, f"stalled: {st}"


def test_configurations_match_the_kernel_source():
    src = open(os.path.join(ROOT, "quantized_grouped_gemm_gb300", "csrc", "ffn.cu")).read()
    assert re.search(r"static constexpr int A = kDown \? 2 : 4;", src)
    assert re.search(r"static constexpr int RX = kDown \? \(kBf16 \? 2 : 4\) : 8;", src)
    assert re.search(r"static constexpr int RC = kBf16 \? 2 : \(kDown \? 6 : 8\);", src)
    assert "constexpr int kTmKD = 8;" in src
    assert "mbar_init(&b->c_empty[i], kTmDeqSet)" in src and "mbar_init(&b->ready[i], kTmDeqSet + 1)" in src


@pytest.mark.parametrize("name,RX,RC,A", CONFIGS, ids=[c[0] for c in CONFIGS])
def test_kernel_ring_configurations_keep_the_protocol(name, RX, RC, A):
    for seed in range(60):
        run(RX, RC, A, KB=8, ntiles=5, seed=seed)


@pytest.mark.parametrize("RC,A", [(3, 2), (3, 4), (5, 4)])
def test_an_odd_weight_ring_below_a_plus_2_breaks_it(RC, A):
    """The condition the kernel asserts (the first bf16 down variant had RC = 3, A = 2)."""
    with pytest.raises(AssertionError):
        for seed in range(200):
            run(4, RC, A, KB=8, ntiles=5, seed=seed)


@pytest.mark.parametrize("RC,A", [(5, 2), (7, 4)])
def test_an_odd_weight_ring_of_a_plus_2_or_more_keeps_it(RC, A):
    for seed in range(60):
        run(8, RC, A, KB=8, ntiles=5, seed=seed)


# ----------------------------------------------------------------------------------------
# Accumulator slots and the down projection's staging ring.
#
# MMA thread m of tile t waits `d_empty` of its slot(s), issues the tile's K blocks, and
# commits `d_full` after the last one (the commit lands once those MMAs are done).  The
# epilogue drains the slots in the same order: it waits `d_full`, reads the accumulator, and
# arrives on `d_empty` after its last TMEM read of that slot.
#   down     slot ring of 4 (one matrix each): use j = 2 t + m, slot j % 4, phase j / 4; the
#            epilogue drains both matrices of a tile together and frees both slots at its end;
#   gate/up  2 slots; a tile with N <= 64 takes one slot for both matrices, a larger one both
#            (the running slot counter sc, per-slot use counts).
# The down epilogue stages each 32-token chunk in buffer (chunk % NSTG); before the chunk's
# barrier every issuing lane waits until its bulk operations of NSTG - 1 chunks back (or
# earlier) have read their buffer, so a buffer is never written while an operation reads it.
# ----------------------------------------------------------------------------------------
def run_slots(kind, ntiles, seed, NSTG=2, KB=4, wait_back=None):
    rnd = random.Random(seed)
    down = kind == "down"
    wait_back = NSTG if wait_back is None else wait_back   # the kernel: NSTG
    NDS = 4 if down else 2
    d_full = [Bar(f"d_full{i}", 1 if down else 2) for i in range(NDS)]
    d_empty = [Bar(f"d_empty{i}", 1) for i in range(NDS)]
    Ns = [rnd.choice([16, 32, 48, 64, 80, 96] + ([] if down else [112, 128])) for _ in range(ntiles)]
    reading = [False] * NDS            # the epilogue holds the slot
    written = [None] * NDS             # (tile, matrix) whose products the slot holds
    events, t = [], 0

    # tile t of thread m -> [(slot, phase)] it waits on (d_empty) and commits to (d_full)
    def gu_plan():
        sc, use, plan = 0, [0, 0], []
        for N in Ns:
            two = 2 * N > 128
            s0 = sc & 1
            s1 = s0 ^ 1 if two else s0
            slots = [(s0, use[s0])] + ([(s1, use[s1])] if two else [])
            plan.append(slots)
            use[s0] += 1
            if two:
                use[s1] += 1
            sc += 2 if two else 1
        return plan
    plan = gu_plan() if not down else None

    def uses(tile, m):
        if down:
            j = 2 * tile + m
            return [(j % 4, j // 4)]
        return plan[tile]

    mma = [dict(tile=0, kb=-1) for _ in range(2)]     # kb = -1: waiting for its slot(s)
    epi = dict(tile=0, m=0, state="wait", chunk=0, ci=0)
    bufs_reading = {}                  # buffer -> set of in-flight op ids
    lanes = {l: [] for l in range(4)}  # issuing lanes: list of (chunk, op id, done flag)
    opid = [0]

    def epi_slots():
        if down:
            return uses(epi["tile"], 0) + uses(epi["tile"], 1)
        return plan[epi["tile"]]

    for _ in range(200000):
        acts = []
        for m in (0, 1):
            st = mma[m]
            if st["tile"] >= ntiles:
                continue
            if st["kb"] < 0:
                us = uses(st["tile"], m)
                if all(d_empty[s].done(ph - 1, f"mma {m}") for s, ph in us if ph > 0):
                    def got(m=m, us=us):
                        for s, ph in us:
                            assert not reading[s], f"mma {m} writes slot {s} while the epilogue reads it"
                            written[s] = (mma[m]["tile"], m)
                        mma[m]["kb"] = 0
                    acts.append(got)
            elif st["kb"] < KB:
                def issue(m=m):
                    mma[m]["kb"] += 1
                    if mma[m]["kb"] == KB:
                        us = uses(mma[m]["tile"], m if down else m)
                        tl = t + rnd.randint(1, 40)
                        for s, ph in us:
                            events.append((tl, lambda s=s: d_full[s].arrive()))
                        mma[m]["tile"] += 1
                        mma[m]["kb"] = -1
                acts.append(issue)
        if epi["tile"] < ntiles:
            st = epi
            us = epi_slots()
            if st["state"] == "wait":
                if all(d_full[s].done(ph, "epilogue") for s, ph in us):
                    def start(us=us):
                        for s, ph in us:
                            reading[s] = True
                        epi["state"] = "drain"
                        epi["ci"] = 0
                    acts.append(start)
            else:
                N = Ns[epi["tile"]]
                nch = (N + 31) // 32 if down else 1
                c = epi["chunk"]
                b = c % NSTG
                last = epi["ci"] == nch - 1
                if st["state"] == "drain":
                    # write chunk c into buffer b (after its TMEM read); the last read frees the slot(s)
                    def write(b=b, c=c, last=last, us=us):
                        if down:
                            assert not bufs_reading.get(b), f"staging buffer {b} written while read (chunk {c})"
                        if last:
                            for s, ph in us:
                                reading[s] = False
                                d_empty[s].arrive()
                        epi["state"] = "issue" if down else "next"
                    acts.append(write)
                elif st["state"] == "issue":
                    # the issuing lanes wait for their operations of chunk c - (NSTG - 1) and earlier
                    # to have read their buffer, then the barrier, then this chunk's operations
                    if all(done for l in lanes for (cc, oid, done) in lanes[l] if cc <= c - (wait_back - 1)):
                        def issue_ops(b=b, c=c):
                            for l in lanes:
                                if rnd.random() < 0.9:
                                    opid[0] += 1
                                    oid = opid[0]
                                    bufs_reading.setdefault(b, set()).add(oid)
                                    rec = [c, oid, False]
                                    lanes[l].append(rec)

                                    def fin(b=b, oid=oid, rec=rec):
                                        bufs_reading[b].discard(oid)
                                        rec[2] = True
                                    events.append((t + rnd.randint(1, 60), fin))
                            epi["chunk"] += 1
                            epi["ci"] += 1
                            epi["state"] = "next" if epi["ci"] == nch else "drain"
                        acts.append(issue_ops)
                else:   # "next": the matrix (down) or the tile (gate/up) is drained
                    def nxt():
                        epi["tile"] += 1
                        epi["state"] = "wait"
                    acts.append(nxt)
        due = [e for e in events if e[0] <= t]
        if not acts and not events:
            break
        if due and (not acts or rnd.random() < 0.5):
            e = rnd.choice(due)
            events.remove(e)
            e[1]()
        elif acts:
            rnd.choice(acts)()
        t += 1
    assert epi["tile"] == ntiles and all(x["tile"] == ntiles for x in mma), f"stalled: {epi} {mma}"


def test_accumulator_slots_match_the_kernel_source():
    src = open(os.path.join(ROOT, "quantized_grouped_gemm_gb300", "csrc", "ffn.cu")).read()
    assert "static constexpr int NDS = kDown ? 4 : 2;" in src
    assert "static constexpr int NSTG = kDown ? 2 : 1;" in src
    assert "const int dsl = kDown ? (int)(dj % 4) : 0;" in src
    assert "mbar_init(&b->d_full[i], kDown ? 1 : 2)" in src


@pytest.mark.parametrize("kind", ["down", "gate/up"])
def test_accumulator_slot_protocol(kind):
    for seed in range(80):
        run_slots(kind, ntiles=12, seed=seed)


@pytest.mark.parametrize("NSTG", [2, 3, 4])
def test_down_staging_ring_is_never_written_while_read(NSTG):
    for seed in range(80):
        run_slots("down", ntiles=10, seed=seed, NSTG=NSTG)


def test_a_staging_ring_waited_one_chunk_too_late_breaks_it():
    """Waiting for the operations of NSTG chunks back (one chunk later than the kernel does)
    lets a buffer be written while an operation still reads it (NSTG = 2: the kernel waits for
    the previous chunk's operations before each barrier)."""
    with pytest.raises(AssertionError, match="written while read"):
        for seed in range(200):
            run_slots("down", ntiles=10, seed=seed, NSTG=2, wait_back=3)
