"""A CPU model of the mbarrier protocol of the prefill main kernel
(`relattn_fwd_tc_main_kernel`): producer, MMA issuer, the tensor core and the
softmax warps of two heads, written step for step after the kernel's waits,
arrives, issues and commits.  Random interleavings of the agents are run to
completion and checked for

* deadlock (every agent finishes),
* parity aliasing (a wait never sees a barrier more than one phase ahead of
  the phase it asks for, which the kernel's parity waits could not tell
  apart),
* buffer hazards: a K / V stage refilled while an MMA that reads it is still
  pending; S_w overwritten before the softmax has read it; P_w (over the
  first 64 columns of S_w) overwritten while a P V MMA still has to read it;
  O_w rescaled while a P V MMA of the previous tile is pending; O_w's final
  read before every P V has landed.

Each model step mirrors one action of the kernel; the assertions are the
hazards the kernel's comments argue away.  A mutated protocol (a wait
dropped) must fail, which pins the checker itself.
"""
import random

import pytest

K_STAGES, V_STAGES = 2, 3
WARPS = 4            # softmax warps per head (TMEM lane quarters)


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, 0, 0

    def arrive(self):
        self.pending += 1
        assert self.pending <= self.count
        if self.pending == self.count:
            self.pending, self.phase = 0, self.phase + 1

    def done(self, parity, want_phase):
        # try / test_wait.parity: true once the phase with that parity has
        # completed.  The kernel asks for phase `want_phase`; a barrier more
        # than one phase ahead would alias.
        assert self.phase <= want_phase + 1, "parity aliasing"
        return (self.phase & 1) != parity


class Model:
    def __init__(self, n, rng, drop=None):
        self.n, self.rng, self.drop = n, rng, drop
        B = {"q_full": Bar(1), "drain": Bar(1)}
        for s in range(K_STAGES):
            B[f"k_full{s}"], B[f"k_empty{s}"] = Bar(1), Bar(1)
        for s in range(V_STAGES):
            B[f"v_full{s}"], B[f"v_empty{s}"] = Bar(1), Bar(1)
        for w in range(2):
            B[f"s_full{w}"] = Bar(1)
            B[f"p_full{w}"] = Bar(WARPS)
            B[f"p_half{w}"] = Bar(WARPS)
            B[f"pv_tail{w}"] = Bar(1)
        self.B = B
        self.k_stage = [None] * K_STAGES     # tile held by each stage
        self.v_stage = [None] * V_STAGES
        self.tc = []                         # issued, not yet executed: ops and commits
        self.s_buf = [None, None]            # tile whose S is in S_w (None: being written)
        self.s_read = [set(), set()]         # warps that have read S_w of the current tile
        self.p_written = [{}, {}]            # (tile, half) -> warps that wrote it
        self.pv_done = [set(), set()]        # (tile, half) of finished P V
        self.pending = []                    # async TMA loads: (stage kind, stage, tile, bar)
        self.agents = [self.producer(), self.issuer()]
        for w in range(2):
            for q in range(WARPS):
                self.agents.append(self.softmax(w, q))

    # ---------------------------------------------------------------- agents
    def wait(self, name, parity, phase):
        while not self.B[name].done(parity, phase):
            yield

    def producer(self):
        self.pending.append(("q", 0, 0, "q_full"))
        for i in range(self.n):
            ks, vs = i % K_STAGES, i % V_STAGES
            if i >= K_STAGES and self.drop != "k_empty":
                yield from self.wait(f"k_empty{ks}", ((i // K_STAGES) - 1) & 1, (i // K_STAGES) - 1)
            # refilling a stage: no pending MMA may still read the tile in it
            assert not any(op[0] == "S" and op[2] == self.k_stage[ks] for op in self.tc
                           if op[0] == "S"), "K stage refilled under a pending S"
            self.k_stage[ks] = None
            self.pending.append(("k", ks, i, f"k_full{ks}"))
            if i >= V_STAGES and self.drop != "v_empty":
                yield from self.wait(f"v_empty{vs}", ((i // V_STAGES) - 1) & 1, (i // V_STAGES) - 1)
            assert not any(op[0] == "PV" and op[2] == self.v_stage[vs] for op in self.tc), \
                "V stage refilled under a pending P V"
            self.v_stage[vs] = None
            self.pending.append(("v", vs, i, f"v_full{vs}"))
            yield

    def issuer(self):
        yield from self.wait("q_full", 0, 0)

        def issue_s(w, i):
            ks = i % K_STAGES
            if w == 0:
                yield from self.wait(f"k_full{ks}", (i // K_STAGES) & 1, i // K_STAGES)
            assert self.k_stage[ks] == i
            self.tc.append(("S", w, i))
            self.tc.append(("commit", f"s_full{w}"))

        def issue_pv(w, i):
            vs = i % V_STAGES
            if w == 0:
                yield from self.wait(f"v_full{vs}", (i // V_STAGES) & 1, i // V_STAGES)
            assert self.v_stage[vs] == i
            if self.drop != "p_half":
                yield from self.wait(f"p_half{w}", i & 1, i)
            self.tc.append(("PV", w, i, 0))
            if self.drop != "p_full":
                yield from self.wait(f"p_full{w}", i & 1, i)
            self.tc.append(("PV", w, i, 1))
            if i == self.n - 1:
                self.tc.append(("commit", f"pv_tail{w}"))

        yield from issue_s(0, 0)
        yield from issue_s(1, 0)
        for i in range(self.n):
            for w in range(2):
                yield from issue_pv(w, i)
                if i + 1 < self.n:
                    yield from issue_s(w, i + 1)
        self.tc.append(("commit", "drain"))
        yield from self.wait("drain", 0, 0)

    def softmax(self, w, q):
        releaser = (w == 1 and q == 0)
        for i in range(self.n):
            yield from self.wait(f"s_full{w}", i & 1, i)
            if releaser:
                self.B[f"k_empty{i % K_STAGES}"].arrive()
                if i > 0:
                    self.B[f"v_empty{(i - 1) % V_STAGES}"].arrive()
            assert self.s_buf[w] == i, "softmax read a wrong S"
            self.s_read[w].add(q)
            yield
            # rescale of O_w: every P V of the previous tile has landed
            assert i == 0 or {(i - 1, 0), (i - 1, 1)} <= self.pv_done[w], "O rescaled under a pending P V"
            self.p_written[w].setdefault((i, 0), set()).add(q)
            self.B[f"p_half{w}"].arrive()
            yield
            self.p_written[w].setdefault((i, 1), set()).add(q)
            self.B[f"p_full{w}"].arrive()
            yield
        yield from self.wait(f"pv_tail{w}", 0, 0)
        # O_w is read out: every P V has landed
        assert all((i, h) in self.pv_done[w] for i in range(self.n) for h in (0, 1))

    # ------------------------------------------------------ asynchronous units
    def tensor_step(self):
        op = self.tc.pop(0)
        if op[0] == "commit":
            self.B[op[1]].arrive()
        elif op[0] == "S":
            _, w, i = op
            # S_w(i) overwrites the buffer: the previous tile's S was read by
            # all warps and its P has been consumed by both halves of P V
            if i > 0:
                assert self.s_read[w] == set(range(WARPS)), "S overwritten before it was read"
                assert {(i - 1, 0), (i - 1, 1)} <= self.pv_done[w], "P overwritten before P V read it"
            self.s_buf[w] = i
            self.s_read[w] = set()
        else:
            _, w, i, h = op
            assert self.p_written[w].get((i, h)) == set(range(WARPS)), "P V read P before it was written"
            self.pv_done[w].add((i, h))

    def tma_step(self):
        kind, st, tile, bar = self.pending.pop(self.rng.randrange(len(self.pending)))
        if kind == "k":
            self.k_stage[st] = tile
        elif kind == "v":
            self.v_stage[st] = tile
        self.B[bar].arrive()

    def run(self, max_steps=200000):
        live = list(self.agents)
        for _ in range(max_steps):
            choices = [("agent", a) for a in live]
            if self.tc:
                choices.append(("tc", None))
            if self.pending:
                choices.append(("tma", None))
            if not choices:
                return
            kind, a = self.rng.choice(choices)
            if kind == "tc":
                self.tensor_step()
            elif kind == "tma":
                self.tma_step()
            else:
                try:
                    next(a)
                except StopIteration:
                    live.remove(a)
            if not live and not self.tc and not self.pending:
                return
        raise AssertionError("deadlock (no progress within the step budget)")


@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
def test_main_kernel_protocol(n):
    for seed in range(40):
        Model(n, random.Random(1000 * n + seed)).run()


@pytest.mark.parametrize("drop", ["p_half", "p_full", "k_empty"])
def test_protocol_model_catches_a_dropped_wait(drop):
    """A protocol with one wait removed must fail in some interleaving."""
    failed = False
    for seed in range(200):
        try:
            Model(4, random.Random(seed), drop=drop).run()
        except AssertionError:
            failed = True
            break
    assert failed


def test_v_empty_wait_is_implied_by_the_k_ring():
    """With 2 K and 3 V stages the producer loads V(i) only after K(i), whose
    stage waited for S_1(i - 2) to land; S_1(i - 2) was issued after
    P V_1(i - 3), the last reader of V(i)'s stage.  So the V_EMPTY wait never
    holds the producer back in a way the hazard checks need: the model stays
    clean without it (the kernel keeps it as a guard)."""
    for n in (3, 5, 8):
        for seed in range(40):
            Model(n, random.Random(seed), drop="v_empty").run()
