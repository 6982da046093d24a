"""The tensor-core kernel's barrier protocol, checked in a host-side model (no GPU).

tests/prefill_protocol_model.py replays the waits, arrivals and commits of prefill_tc_kernel's
roles under random interleavings of the roles, the TMA copies and the in-order tensor pipe.
The protocol as built must never deadlock, alias a barrier phase, or reuse a metadata slot, a
K/V stage or an S/P buffer too early; and the model must catch each planted protocol mistake
(too few metadata slots, a V stage refilled without waiting for its PV, a softmax waiting on the
wrong phase), so that a pass means something.
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
    for seed, n, nq, clean in _schedules(500, seed0=500 * part):
        try:
            pm.Sim(n, nq, CLEAN[clean], seed=seed).run()
        except pm.ProtocolError as e:
            pytest.fail(f"seed {seed}, {n} tiles, {nq} live Q tiles, clean={clean}: {e}")


def _caught(make, n_runs=200):
    caught = 0
    for seed, n, nq, clean in _schedules(n_runs):
        try:
            make(n, nq, clean, seed).run()
        except pm.ProtocolError:
            caught += 1
    return caught


def test_model_catches_too_few_metadata_slots():
    assert _caught(lambda n, nq, clean, seed: pm.Sim(n, nq, CLEAN[clean], seed=seed, slots=2)) > 0


def test_model_catches_v_stage_refilled_before_its_pv():
    class NoVFreeWait(pm.Sim):
        def producer(self):
            def issue_k(j):
                s = j % 2
                if j >= 2:
                    yield ("wait", self.K_FREE[s], j // 2 - 1)
                self.publish(j)
                self.K_FULL[s].arrive(self, expect_tx=1)
                self.issue_tma("K", j, self.K_FULL[s])
                yield ("step",)

            def issue_v(j):  # planted mistake: no wait for V_FREE
                s = j % 2
                self.read_slot(j, "issue_v")
                self.V_FULL[s].arrive(self, expect_tx=1)
                self.issue_tma("V", j, self.V_FULL[s])
                yield ("step",)

            yield from issue_k(0)
            for j in range(self.n):
                if j + 1 < self.n:
                    yield from issue_k(j + 1)
                yield from issue_v(j)

    assert _caught(lambda n, nq, clean, seed: NoVFreeWait(n, nq, CLEAN[clean], seed=seed)) > 0


def test_model_catches_softmax_waiting_on_the_wrong_phase():
    class EarlySoftmax(pm.Sim):
        def softmax(self, i):
            self.Q_READY.arrive(self)
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
                self.P_FULL[buf].arrive(self)
            yield ("wait", self.FINAL, 0)

    assert _caught(lambda n, nq, clean, seed: EarlySoftmax(n, nq, CLEAN[clean], seed=seed)) > 0
