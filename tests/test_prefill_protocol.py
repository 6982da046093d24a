"""The tensor-core kernel's barrier protocol, checked in a host-side model (no GPU).

tests/prefill_protocol_model.py replays the waits, arrivals and commits of prefill_tc_kernel's
roles under random interleavings of the roles, the TMA copies and the in-order tensor pipe.
The protocol as built must never deadlock, wait ahead of a barrier, alias a barrier phase, or
reuse a metadata slot, a K/V stage or an S/P buffer too early; and the model must catch each
planted protocol mistake (too few metadata slots, a V stage refilled without waiting for its PV,
a softmax waiting on the wrong phase, and the earlier V-cleaning handshake whose rotation role
skipped the V_FULL phases of tiles it did not clean), so that a pass means something.
"""
import random

import pytest

from tests import prefill_protocol_model as pm

CLEAN = {
    "none": lambda j: False,            # every page full (long documents)
    "all": lambda j: True,              # every tile has key-less V rows to clear
    "some": lambda j: j % 3 == 1,       # documents ending mid-tile now and then
}


def _schedules(n_runs, seed0=0):
    for seed in range(seed0, seed0 + n_runs):
        rng = random.Random(seed)
        yield seed, rng.choice([1, 2, 3, 4, 5, 8, 9, 16, 17]), rng.choice([1, 2]), rng.choice(sorted(CLEAN))


@pytest.mark.parametrize("part", range(4))
def test_protocol_as_built_is_safe_under_random_interleavings(part):
    """The kernel's configuration: a 3-stage K ring, a 2-stage V ring, 6 metadata slots, one
    producer issuing K and V (the instantiation without SPLIT_V, and every two-Q-tile CTA)."""
    for seed, n, nq, clean in _schedules(500, seed0=500 * part):
        try:
            pm.Sim(n, nq, CLEAN[clean], seed=seed, kst=3, slots=6).run()
        except pm.ProtocolError as e:
            pytest.fail(f"seed {seed}, {n} tiles, {nq} live Q tiles: {e}")


def test_key_halves_with_one_live_q_tile_are_safe():
    """Launches whose CTAs all have one live Q tile: the two softmax warpgroups each take half of
    every tile's keys (P complete after both), with one producer or the separate V producer."""
    for seed, n, _, clean in _schedules(600, seed0=5000):
        for vprod in (False, True):
            try:
                pm.Sim(n, 1, CLEAN[clean], seed=seed, kst=3, slots=6, vprod=vprod, kh=True).run()
            except pm.ProtocolError as e:
                pytest.fail(f"seed {seed}, {n} tiles, separate V producer {vprod}: {e}")


def test_model_catches_pv_after_one_key_half():
    class OneHalfEnough(pm.Sim):
        def __init__(self, *a, **kw):
            super().__init__(*a, **kw)
            self.P_FULL = [pm.Bar(f"P_FULL{i}", 1) for i in range(2)]  # planted: PV after one half
    caught = []
    for seed, n, _, clean in _schedules(300):
        try:
            OneHalfEnough(n, 1, CLEAN[clean], seed=seed, kst=3, slots=6, kh=True).run()
        except pm.ProtocolError as e:
            caught.append(str(e))
    assert any("P1" in c or "too many arrivals" in c for c in caught), caught[:3]


def _caught(make, n_runs=200):
    caught = 0
    for seed, n, nq, clean in _schedules(n_runs):
        try:
            make(n, nq, clean, seed).run()
        except pm.ProtocolError:
            caught += 1
    return caught


def test_separate_v_producer_is_safe_for_both_schedules():
    """V issued by a warp of its own that reads the block words itself: the SPLIT_V
    instantiation (one-Q-tile CTAs over long key ranges); safe for both schedules."""
    for seed, n, nq, clean in _schedules(300, seed0=9000):
        for vgate in (True, False):  # rotating kernels: V starts once Q is ready; the others at once
            try:
                pm.Sim(n, nq, CLEAN[clean], seed=seed, kst=3, slots=6, vprod=True, vgate=vgate).run()
            except pm.ProtocolError as e:
                pytest.fail(f"seed {seed}, {n} tiles, {nq} live Q tiles, vgate {vgate}: {e}")


def test_two_stage_k_ring_is_safe_too():
    for seed, n, nq, clean in _schedules(300, seed0=7000):
        try:
            pm.Sim(n, nq, CLEAN[clean], seed=seed, kst=2, slots=4).run()
        except pm.ProtocolError as e:
            pytest.fail(f"seed {seed}, {n} tiles, {nq} live Q tiles: {e}")


def test_model_catches_too_few_metadata_slots():
    """With the K ring two tiles ahead, the one-live-Q-tile schedule can publish tile j + 4's
    metadata while the softmax of tile j still reads its slot: 4 slots are too few."""
    assert _caught(lambda n, nq, clean, seed: pm.Sim(n, nq, CLEAN[clean], seed=seed, slots=4), 400) > 0


def test_model_catches_v_stage_refilled_before_its_pv():
    class NoVFreeWait(pm.Sim):
        def producer(self):
            def issue_k(j):
                s = j % self.kst
                if j >= self.kst:
                    yield ("wait", self.K_FREE[s], j // self.kst - 1)
                self.publish(j)
                self.K_FULL[s].arrive(expect_tx=1)
                self.issue_tma("K", j, self.K_FULL[s])
                yield ("step",)

            def issue_v(j):  # planted mistake: no wait for V_FREE
                s = j % 2
                self.read_slot(j, "issue_v")
                self.V_FULL[s].arrive(expect_tx=1)
                self.issue_tma("V", j, self.V_FULL[s])
                yield ("step",)

            ahead = self.kst - 1
            for j in range(min(ahead, self.n)):
                yield from issue_k(j)
            for j in range(self.n):
                if j + ahead < self.n:
                    yield from issue_k(j + ahead)
                yield from issue_v(j)

    assert _caught(lambda n, nq, clean, seed: NoVFreeWait(n, nq, CLEAN[clean], seed=seed)) > 0


def test_model_catches_softmax_waiting_on_the_wrong_phase():
    class EarlySoftmax(pm.Sim):
        def softmax(self, i):
            self.Q_READY.arrive()
            if i >= self.nq:
                return
            yield ("step",)
            for j in range(self.n):
                buf = i if self.nq == 2 else (j & 1)
                e = j if self.nq == 2 else (j >> 1)
                yield ("wait", self.S_FULL[buf], max(e - 1, 0))  # planted mistake: one phase early
                if self.s_buf.get(buf) != ("S", j):
                    raise pm.ProtocolError(f"softmax{i} reads S{buf} for tile {j}, holds {self.s_buf.get(buf)}")
                self.read_slot(j, f"softmax{i}")
                yield ("step",)
                if self.nq == 1 and j > 0:
                    yield ("wait", self.PV_DONE, j - 1)
                self.s_buf[buf] = ("P", j)
                self.P_FULL[buf].arrive()
            yield ("wait", self.FINAL, 0)

    assert _caught(lambda n, nq, clean, seed: EarlySoftmax(n, nq, CLEAN[clean], seed=seed)) > 0


class OldVClean(pm.Sim):
    """The earlier protocol, kept as a planted mistake.  The rotation role also zeroed the V
    rows of a tile that held no key, waiting V_FULL only for such tiles and then arriving on a
    V_READY barrier; the MMA thread waited V_READY (counting such tiles per stage) after V_FULL.
    Skipping the V_FULL phases of tiles it did not clean leaves the rotation role one phase
    AHEAD of the barrier when a clean tile follows an unclean one on the same stage whose V has
    not landed yet; a parity wait then passes at once and the role zeroes a stage that the
    earlier copy is still filling."""

    every_phase = False

    def __init__(self, *a, **kw):
        super().__init__(*a, **kw)
        self.V_READY = [pm.Bar(f"V_READY{s}", 1) for s in range(2)]
        self.cleaned = [0, 0]

    def v_users(self, j):
        return super().v_users(j) | ({"clean"} if self.clean_of(j) else set())

    def rotation(self):
        for j in range(self.n):
            s, sv = j % self.kst, j % 2
            yield ("wait", self.K_FULL[s], j // self.kst)
            self.read_slot(j, "rotation")
            yield ("step",)
            self.kstage_users[s].discard("rot")
            self.K_READY[s].arrive()
            if self.clean_of(j) or self.every_phase:
                yield ("wait", self.V_FULL[sv], j // 2)
                if self.vstage[sv] != j:
                    raise pm.ProtocolError(f"V clean of tile {j} finds stage holding {self.vstage[sv]}")
                if self.clean_of(j):
                    yield ("step",)
                    self.vstage_users[sv].discard("clean")
                    self.V_READY[sv].arrive()

    def mma_wait_v(self, jj):
        s = jj % 2
        yield ("wait", self.V_FULL[s], jj // 2)
        if self.clean_of(jj):
            yield ("wait", self.V_READY[s], self.cleaned[s])
            self.cleaned[s] += 1


class OldVCleanEveryPhase(OldVClean):
    """The same cleaning role, corrected: it consumes every V_FULL phase in tile order."""
    every_phase = True


def test_model_catches_the_old_v_clean_handshake():
    caught = []
    for seed, n, nq, clean in _schedules(400):
        try:
            OldVClean(n, nq, CLEAN[clean], seed=seed, kst=2).run()
        except pm.ProtocolError as e:
            caught.append(str(e))
    assert caught, "the model let the old V-clean handshake through"
    assert any("waiter ahead" in c and "V_FULL" in c for c in caught), caught[:3]


def test_v_clean_consuming_every_phase_is_safe():
    """Control for the test above: the model does not reject a V-cleaning role as such."""
    for seed, n, nq, clean in _schedules(400):
        try:
            OldVCleanEveryPhase(n, nq, CLEAN[clean], seed=seed, kst=2).run()
        except pm.ProtocolError as e:
            pytest.fail(f"seed {seed}, {n} tiles, {nq} live Q tiles, clean={clean}: {e}")


def test_model_flags_a_waiter_ahead_of_its_barrier():
    """Unit check of the parity rule: a wait registered for a phase the barrier has not begun."""
    class Ahead(pm.Sim):
        def rotation(self):
            yield ("wait", self.K_FULL[0], 1)  # phase 1 before phase 0 completed
    with pytest.raises(pm.ProtocolError, match="waiter ahead"):
        Ahead(4, 1, seed=0).run()
