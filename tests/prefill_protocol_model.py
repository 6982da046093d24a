"""Discrete-event model of the tensor-core attention kernel's mbarrier protocol (test
infrastructure, host only).

The roles of prefill_tc_kernel (K/V producer, K rotation, softmax of each Q tile, MMA issuer)
are generators that yield ('wait', barrier, phase) or ('step',), in the same order of waits,
arrivals and commits as the kernel, for both schedules (two live Q tiles, and one live Q tile
whose scores alternate between the two S buffers).  Asynchronous engines: TMA copies land in
any order, each after a random latency (in scheduler steps; the bound is drawn per run, up to
tens of steps, so that a copy can stay in flight while the roles run several tiles ahead); the
tensor pipe runs MMAs in issue order and a commit arrives once every earlier MMA is done.  A
random scheduler interleaves everything.

Waits follow mbarrier.try_wait.parity exactly.  A wait for phase e of a barrier that has
completed k phases passes iff k - e is odd: besides the intended k = e + 1 it also passes when
the waiter is AHEAD of the barrier (k = e - 1, e - 3, ...: the phase asked for has not even
begun), and it blocks when the barrier is two phases past (k = e + 2: aliasing).  The model
raises on both: on any waiter registered while k < e, and on any k >= e + 2.

Checked besides: no deadlock; no metadata slot overwritten while a reader still needs it; no
K/V stage refilled before all its consumers are done; S/P tensor-memory buffers written in a
safe order; every QK^T and PV runs exactly once.

Subclasses may override the hooks (``v_users``, ``rotation``, ``mma_wait_v``, ``mma_saw``,
``producer``, ``softmax``) to plant a protocol mistake that the checks must catch.
"""
import random


class ProtocolError(Exception):
    pass


class Bar:
    def __init__(self, name, need):
        self.name, self.need = name, need
        self.arr, self.tx, self.k = 0, 0, 0

    def _check(self):
        if self.arr == self.need and self.tx == 0:
            self.arr = 0
            self.k += 1

    def arrive(self, expect_tx=0):
        self.arr += 1
        self.tx += expect_tx
        if self.arr > self.need:
            raise ProtocolError(f"{self.name}: too many arrivals")
        self._check()

    def complete_tx(self, b):
        self.tx -= b
        self._check()


class Sim:
    def __init__(self, ntiles, nq, clean=None, seed=0, slots=4, kst=3, vprod=False, vgate=True, kh=False):
        """ntiles K/V tiles, nq live Q tiles (1 or 2), `clean(j)`: whether tile j has key-less
        rows (used only by subclasses that model a V-cleaning role); kst K ring stages (the V
        ring has 2); slots metadata slots; vprod: V is issued by a producer of its own, which
        reads the block words itself (no metadata slot); vgate: that producer first waits for
        Q_READY (the rotating kernels); kh: with one live Q tile the two softmax roles each take
        half of every tile's keys."""
        self.rng = random.Random(seed)
        self.now = 0
        self.max_latency = self.rng.choice([0, 3, 12, 40])
        self.n, self.nq = ntiles, nq
        self.clean_of = clean or (lambda j: False)
        self.slots, self.kst, self.vprod, self.vgate = slots, kst, vprod, vgate
        self.K_FULL = [Bar(f"K_FULL{s}", 1) for s in range(kst)]
        self.K_READY = [Bar(f"K_READY{s}", 1) for s in range(kst)]
        self.K_FREE = [Bar(f"K_FREE{s}", 1) for s in range(kst)]
        self.V_FULL = [Bar(f"V_FULL{s}", 1) for s in range(2)]
        self.V_FREE = [Bar(f"V_FREE{s}", 1) for s in range(2)]
        self.S_FULL = [Bar(f"S_FULL{i}", 1) for i in range(2)]
        # kh (one live Q tile): both softmax roles work on every tile, each on half of its keys,
        # and P is complete once both have written theirs
        self.kh = kh and nq == 1
        self.P_FULL = [Bar(f"P_FULL{i}", 2 if self.kh else 1) for i in range(2)]
        self.PV_DONE = Bar("PV_DONE", 1)
        self.Q_READY = Bar("Q_READY", 2)
        self.FINAL = Bar("FINAL", 1)
        # state for hazard checks
        self.slot_tile = [None] * self.slots
        self.kstage = [None] * kst          # tile whose K is in the stage (landed)
        self.vstage = [None, None]
        self.kstage_users = [set() for _ in range(kst)]  # outstanding consumers of the stage's tile
        self.vstage_users = [set(), set()]
        self.tma = []      # pending copies: (kind, stage, tile, bar, earliest landing step)
        self.pipe = []     # tensor pipe FIFO: ('mma', fn) or ('commit', bar)
        self.s_buf = {}    # S/P buffer -> ('S', tile) / ('P', tile)
        self.done_qk = set()
        self.done_pv = set()

    # ------------------------------------------------------------------ hazards
    def read_slot(self, j, who):
        s = j % self.slots
        if self.slot_tile[s] != j:
            raise ProtocolError(f"{who} reads slot {s} for tile {j}, holds {self.slot_tile[s]}")

    def publish(self, j):
        self.slot_tile[j % self.slots] = j

    def v_users(self, j):
        """Consumers of a landed V tile."""
        return {"pv0"} | ({"pv1"} if self.nq == 2 else set())

    # ------------------------------------------------------------------ engines
    def issue_tma(self, kind, j, bar):
        st = j % (self.kst if kind == "K" else 2)
        users = self.kstage_users[st] if kind == "K" else self.vstage_users[st]
        if users:
            raise ProtocolError(f"{kind}({j}) issued into stage {st} while {sorted(users)} still use it")
        self.tma.append((kind, st, j, bar, self.now + self.rng.randint(0, self.max_latency)))

    def tma_ready(self):
        return [i for i, c in enumerate(self.tma) if c[4] <= self.now]

    def step_tma(self):
        i = self.rng.choice(self.tma_ready())
        kind, st, j, bar, _ = self.tma.pop(i)
        if kind == "K":
            if self.kstage_users[st]:
                raise ProtocolError(f"K({j}) lands in stage {st} while {sorted(self.kstage_users[st])} still use it")
            self.kstage[st] = j
            self.kstage_users[st] = {"rot", "qk0"} | ({"qk1"} if self.nq == 2 else set())
        else:
            self.vstage[st] = j
            self.vstage_users[st] = self.v_users(j)
        bar.complete_tx(1)

    def step_pipe(self):
        op = self.pipe.pop(0)
        if op[0] == "commit":
            op[1].arrive()
        else:
            op[1]()

    # ------------------------------------------------------------------ MMAs
    def qk(self, i, j, buf):
        def run():
            st = j % self.kst
            if self.kstage[st] != j or "rot" in self.kstage_users[st]:
                raise ProtocolError(f"QK{i}({j}) reads K stage {st} holding {self.kstage[st]} "
                                    f"(rotated: {'rot' not in self.kstage_users[st]})")
            prev = self.s_buf.get(buf)
            if prev is not None and prev[0] == "P" and (i, prev[1]) not in self.done_pv:
                raise ProtocolError(f"QK{i}({j}) overwrites P({prev[1]}) in S{buf} before its PV")
            if prev is not None and prev[0] in ("S", "P1"):
                raise ProtocolError(f"QK{i}({j}) overwrites S({prev[1]}) in S{buf} before the softmax read it")
            if (i, j) in self.done_qk:
                raise ProtocolError(f"QK{i}({j}) runs twice")
            self.s_buf[buf] = ("S", j)
            self.kstage_users[st].discard(f"qk{i}")
            self.done_qk.add((i, j))
        self.pipe.append(("mma", run))

    def pv(self, i, j, buf):
        def run():
            st = j % 2
            others = self.vstage_users[st] - {"pv0", "pv1"}
            if self.vstage[st] != j or others:
                raise ProtocolError(f"PV{i}({j}) reads V stage {st} holding {self.vstage[st]} "
                                    f"(still pending: {sorted(others)})")
            if self.s_buf.get(buf) != ("P", j):
                raise ProtocolError(f"PV{i}({j}) reads S{buf} holding {self.s_buf.get(buf)}")
            if (i, j) in self.done_pv:
                raise ProtocolError(f"PV{i}({j}) runs twice")
            self.vstage_users[st].discard(f"pv{i}")
            self.done_pv.add((i, j))
        self.pipe.append(("mma", run))

    def commit(self, bar):
        self.pipe.append(("commit", bar))

    # ------------------------------------------------------------------ actors
    def producer(self):
        n = self.n

        def issue_k(j):  # wait for the stage, publish the tile's metadata, load K
            s = j % self.kst
            if j >= self.kst:
                yield ("wait", self.K_FREE[s], j // self.kst - 1)
            self.publish(j)
            self.K_FULL[s].arrive(expect_tx=1)
            self.issue_tma("K", j, self.K_FULL[s])
            yield ("step",)

        # K runs kst - 1 tiles ahead of V: (kst = 3) K0, K1, K2, V0, K3, V1, ...
        ahead = self.kst - 1
        for j in range(min(ahead, n)):
            yield from issue_k(j)
        for j in range(n):
            if j + ahead < n:
                yield from issue_k(j + ahead)
            if not self.vprod:
                yield from self.issue_v(j, from_slot=True)

    def issue_v(self, j, from_slot):  # wait for the stage; clear empty page slots; load V
        s = j % 2
        if j >= 2:
            yield ("wait", self.V_FREE[s], j // 2 - 1)
        if from_slot:
            self.read_slot(j, "issue_v")
        self.V_FULL[s].arrive(expect_tx=1)
        self.issue_tma("V", j, self.V_FULL[s])
        yield ("step",)

    def vproducer(self):
        if self.vgate:  # the rotating kernels' V producer starts once Q is ready
            yield ("wait", self.Q_READY, 0)
        for j in range(self.n):
            yield from self.issue_v(j, from_slot=False)

    def rotation(self):
        for j in range(self.n):
            s = j % self.kst
            yield ("wait", self.K_FULL[s], j // self.kst)
            self.read_slot(j, "rotation")
            yield ("step",)  # rotate in place
            if self.kstage[s] != j:
                raise ProtocolError(f"rotation of K({j}) finds stage holding {self.kstage[s]}")
            self.kstage_users[s].discard("rot")
            self.K_READY[s].arrive()

    def softmax(self, i):
        self.Q_READY.arrive()
        if i >= self.nq and not self.kh:
            return
        yield ("step",)
        for j in range(self.n):
            buf = i if self.nq == 2 else (j & 1)
            e = j if self.nq == 2 else (j >> 1)
            yield ("wait", self.S_FULL[buf], e)
            if self.s_buf.get(buf) not in (("S", j), ("P1", j)):  # P1: the other half's P is in
                raise ProtocolError(f"softmax{i} reads S{buf} for tile {j}, holds {self.s_buf.get(buf)}")
            self.read_slot(j, f"softmax{i}")
            yield ("step",)
            if self.nq == 1 and j > 0:
                yield ("wait", self.PV_DONE, j - 1)
            self.read_slot(j, f"softmax{i}-mask")
            if self.kh and self.s_buf.get(buf) == ("S", j):
                self.s_buf[buf] = ("P1", j)
            else:
                self.s_buf[buf] = ("P", j)
            self.P_FULL[buf].arrive()
        yield ("wait", self.FINAL, 0)

    def mma_wait_v(self, jj):
        """The MMA thread's wait before PV of tile jj: V_FULL of its stage, every phase in order."""
        yield ("wait", self.V_FULL[jj % 2], jj // 2)

    def mma_saw(self, j):
        """Hook: the MMA thread has read tile j's metadata slot (just before its QK^T)."""

    def mma(self):
        n, nq = self.n, self.nq
        yield ("wait", self.Q_READY, 0)
        if nq == 1:
            def qk1(j):
                yield ("wait", self.K_READY[j % self.kst], j // self.kst)
                self.read_slot(j, "mma-qk1")
                self.mma_saw(j)
                self.qk(0, j, j & 1)
                self.commit(self.S_FULL[j & 1])
                self.commit(self.K_FREE[j % self.kst])

            yield from qk1(0)
            if n > 1:
                yield from qk1(1)
            for j in range(n):
                yield ("wait", self.P_FULL[j & 1], j >> 1)
                yield from self.mma_wait_v(j)
                self.pv(0, j, j & 1)
                self.commit(self.PV_DONE)
                self.commit(self.V_FREE[j % 2])
                if j + 2 < n:
                    yield from qk1(j + 2)
        else:
            yield ("wait", self.K_READY[0], 0)
            self.read_slot(0, "mma-qk")
            self.mma_saw(0)
            self.qk(0, 0, 0)
            self.commit(self.S_FULL[0])
            self.qk(1, 0, 1)
            self.commit(self.S_FULL[1])
            self.commit(self.K_FREE[0])
            for j in range(1, n):
                s, sp = j % self.kst, (j - 1) % 2
                yield ("wait", self.P_FULL[0], j - 1)
                yield from self.mma_wait_v(j - 1)
                self.pv(0, j - 1, 0)
                yield ("wait", self.K_READY[s], j // self.kst)
                self.read_slot(j, "mma-qk")
                self.mma_saw(j)
                self.qk(0, j, 0)
                self.commit(self.S_FULL[0])
                yield ("wait", self.P_FULL[1], j - 1)
                self.pv(1, j - 1, 1)
                self.commit(self.V_FREE[sp])
                self.qk(1, j, 1)
                self.commit(self.S_FULL[1])
                self.commit(self.K_FREE[s])
            jl = n - 1
            yield ("wait", self.P_FULL[0], jl)
            yield from self.mma_wait_v(jl)
            self.pv(0, jl, 0)
            yield ("wait", self.P_FULL[1], jl)
            self.pv(1, jl, 1)
            self.commit(self.V_FREE[jl % 2])
        self.commit(self.FINAL)
        yield ("wait", self.FINAL, 0)

    # ------------------------------------------------------------------ scheduler
    def actors(self):
        a = {"producer": self.producer(), "rotation": self.rotation(), "mma": self.mma(),
             "softmax0": self.softmax(0), "softmax1": self.softmax(1)}
        if self.vprod:
            a["vproducer"] = self.vproducer()
        return a

    def run(self, max_steps=200000):
        actors = self.actors()
        state = {name: None for name in actors}  # pending (barrier, phase) or None
        alive = set(actors)
        for steps in range(max_steps):
            self.now += 1
            runnable = []
            for name in sorted(alive):
                w = state[name]
                if w is None:
                    runnable.append(name)
                    continue
                bar, e = w
                if bar.k < e:
                    raise ProtocolError(
                        f"waiter ahead: {name} waits {bar.name} phase {e} while the barrier has completed "
                        f"only {bar.k} phases (a parity wait would "
                        f"{'pass at once' if (e - bar.k) % 2 else 'pass on the wrong phase'})")
                if bar.k >= e + 2:
                    raise ProtocolError(f"aliasing: {name} waits {bar.name} phase {e}, barrier at {bar.k}")
                if bar.k == e + 1:
                    runnable.append(name)
            engines = (["tma"] if self.tma_ready() else []) + (["pipe"] if self.pipe else [])
            if not runnable and not engines and self.tma:  # only copies in flight: time passes
                self.now = min(c[4] for c in self.tma)
                continue
            if not runnable and not engines:
                if alive:
                    raise ProtocolError("deadlock: " + ", ".join(
                        f"{n} on {state[n][0].name}[{state[n][1]}] (k={state[n][0].k})" for n in sorted(alive)))
                want = {(i, j) for i in range(self.nq) for j in range(self.n)}
                if self.done_pv != want or self.done_qk != want:
                    raise ProtocolError("not every QK^T / PV ran")
                return steps
            choice = self.rng.choice(runnable + engines * 2)
            if choice == "tma":
                self.step_tma()
                continue
            if choice == "pipe":
                self.step_pipe()
                continue
            state[choice] = None
            try:
                y = next(actors[choice])
            except StopIteration:
                alive.discard(choice)
                continue
            if y[0] == "wait":
                state[choice] = (y[1], y[2])
        raise ProtocolError("step limit")
