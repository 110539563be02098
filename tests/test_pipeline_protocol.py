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
           ("down bf16 weights", 2, 4, 2)]


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
    assert re.search(r"static constexpr int RC = kBf16 \? \(kDown \? 4 : 2\) : \(kDown \? 6 : 8\);", src)
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
