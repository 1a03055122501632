"""Happens-before model of a warp-specialised tcgen05 / TMA pipeline (CPU only).

A kernel's roles are written as Python generators that yield the barrier
operations and buffer accesses of the kernel, in its order.  `Model.run`
executes them under one random interleaving, with random completion times for
the asynchronous work (TMA copies, tcgen05 MMAs and commits, bulk reduce
copies; each run draws how fast that work is against the threads, from much
slower to much faster), and carries vector clocks through every
synchronisation:

* an mbarrier phase releases the join of its arrivals (a TMA copy's arrival
  carries the copy, a commit carries every MMA its issuer issued before it);
  a thread that waits for the phase acquires it;
* a named-barrier generation releases the join of its arrivals to the
  threads that bar.sync on it (bar.arrive does not wait, so does not acquire);
* a bulk-async group wait acquires the thread's own completed bulk copies.

MMAs issued by one thread write TMEM in issue order (accumulation into an
accumulator an earlier MMA wrote is the tensor core's contract), so a write
by an MMA is ordered after the writes of the earlier MMAs of its queue.
Nothing else orders them: an MMA that overwrites what an earlier MMA reads,
or reads what a thread wrote, needs a commit or a barrier like any access.

Checked on every run: no two conflicting accesses to a buffer are unordered
(a data race); a wait for phase n of an mbarrier starts with at least n
phases complete and returns before phase n + 1 completes (its parity cannot
alias); every arrival lands in the phase it is meant for; no thread arrives
twice in one named-barrier generation; nothing deadlocks; nothing is left
half-arrived at the end.

Actions a role yields:
  ("wait", bar, n)              wait for phase n of an mbarrier (n = -1: none yet)
  ("arrive", bar, n)            a thread's arrival, meant for phase n
  ("tma", bar, n, writes)       a TMA load: arrive.expect_tx on phase n; the
                                bytes land later (complete_tx)
  ("mma", queue, reads, writes, accs)   a tcgen05.mma issued into `queue`;
                                `accs`: the accumulators it adds into (writes,
                                listed apart for the reader)
  ("commit", queue, bar, n)     tcgen05.commit: arrives on phase n once every
                                MMA issued before it into `queue` is done
  ("nb_arrive", id, warps) / ("nb_sync", id, warps)   named barrier
  ("bulk", reads)               a bulk async copy out of shared memory
  ("bulk_wait",)                wait until this thread's bulk copies have read
                                their sources
  ("rd" | "wr", buffer)         a software access by the role
"""
import random


class Violation(Exception):
    pass


class Deadlock(Exception):
    pass


def _join(a, b):
    out = dict(a)
    for k, v in b.items():
        if out.get(k, 0) < v:
            out[k] = v
    return out


class _MBar:
    def __init__(self, count):
        self.count = count
        self.done = 0  # completed phases
        self.arrived = 0
        self.tx = 0
        self.acc = {}
        self.phase_vc = []


class Model:
    def __init__(self, counts, seed, queues=("S", "O")):
        self.rng = random.Random(seed)
        # weight of an asynchronous completion against a thread's step
        self.engine_weight = self.rng.choice([0.05, 0.3, 1.0, 3.0, 20.0])
        self.bars = {name: _MBar(c) for name, c in counts.items()}
        self.nb = {}  # id -> [generation, warps, arrived agents, accumulated clock]
        self.nb_vc = {}  # (id, generation) -> clock
        self.vc = {}  # agent -> vector clock
        self.hist = {}  # buffer -> accesses not yet subsumed by an ordered write
        self.queues = {q: [] for q in queues}
        self.queue_vc = {q: {} for q in queues}  # join of every MMA issued into the queue
        self.op_queue = {}  # MMA agent -> its queue
        self.inflight = []  # TMA loads: (bar, phase, clock)
        self.bulk = {}  # agent -> its bulk copies not yet waited for
        self.bulk_pending = []  # (agent, op) not yet complete
        self.blocked = {}  # agent -> ("mb", bar, n) | ("nb", id, generation) | ("bulk",)
        self.n_ops = 0

    # -- clocks
    def _release(self, agent):
        vc = dict(self.vc[agent])
        self.vc[agent][agent] += 1
        return vc

    def _new_agent(self, prefix, vc):
        self.n_ops += 1
        name = f"{prefix}{self.n_ops}"
        vc = dict(vc)
        vc[name] = 1
        self.vc[name] = vc
        return name

    def _access(self, agent, buf, write):
        vc = self.vc[agent]
        hist = self.hist.setdefault(buf, [])
        subsumes = write
        for a, e, w, aq in hist:
            if a == agent or not (write or w) or vc.get(a, 0) >= e:
                continue
            if write and w and aq is not None and aq == self.op_queue.get(agent):
                subsumes = False  # one issuer's MMAs write TMEM in order
                continue
            raise Violation(f"race on {buf}: {'write' if write else 'read'} by {agent} is not ordered after "
                            f"the {'write' if w else 'read'} by {a}")
        rec = (agent, vc[agent], write, self.op_queue.get(agent))
        if subsumes:
            self.hist[buf] = [rec]
        else:
            hist.append(rec)

    # -- mbarriers
    def _arrive(self, bar_name, n, vc, tx=0, done_tx=False):
        bar = self.bars[bar_name]
        if bar.done != n:
            raise Violation(f"arrival on {bar_name} meant for phase {n} lands in phase {bar.done}")
        if done_tx:
            bar.tx -= 1
        else:
            bar.arrived += 1
            bar.tx += tx
            if bar.arrived > bar.count:
                raise Violation(f"{bar_name}: more arrivals than its count in phase {n}")
        bar.acc = _join(bar.acc, vc)
        if bar.arrived == bar.count and bar.tx == 0:
            bar.phase_vc.append(bar.acc)
            bar.done += 1
            bar.arrived, bar.acc = 0, {}
            for agent, st in self.blocked.items():
                if st[0] == "mb" and st[1] == bar_name and bar.done > st[2] + 1:
                    raise Violation(f"{agent} waits for phase {st[2]} of {bar_name} with parity {st[2] & 1}, "
                                    f"but {bar.done} phases are complete: the parity aliases")

    # -- named barriers
    def _nb_arrive(self, agent, nid, warps):
        st = self.nb.setdefault(nid, [0, warps, set(), {}])
        if st[1] != warps:
            raise Violation(f"named barrier {nid} used with {st[1]} and {warps} warps")
        if agent in st[2]:
            raise Violation(f"overrun: {agent} arrives twice in generation {st[0]} of named barrier {nid}")
        st[2].add(agent)
        st[3] = _join(st[3], self._release(agent))
        gen = st[0]
        if len(st[2]) == warps:
            self.nb_vc[(nid, gen)] = st[3]
            st[0], st[2], st[3] = gen + 1, set(), {}
        return gen

    # -- one action of a role
    def _do(self, agent, act):
        kind = act[0]
        if kind == "wait":
            _, bar_name, n = act
            bar = self.bars[bar_name]
            if bar.done < n:
                raise Violation(f"{agent} waits for phase {n} of {bar_name} with only {bar.done} complete: "
                                "a parity wait would return on an earlier phase")
            self.blocked[agent] = ("mb", bar_name, n)
        elif kind == "arrive":
            self._arrive(act[1], act[2], self._release(agent))
        elif kind == "tma":
            _, bar_name, n, writes = act
            op = self._new_agent("tma", self._release(agent))
            for w in writes:
                self._access(op, w, True)
            self._arrive(bar_name, n, self.vc[agent], tx=1)
            self.inflight.append((bar_name, n, self.vc[op]))
        elif kind == "mma":
            _, qn, reads, writes, accs = act
            op = self._new_agent(f"mma{qn}", self._release(agent))
            self.op_queue[op] = qn
            for r in reads:
                self._access(op, r, False)
            for w in list(writes) + list(accs):
                self._access(op, w, True)
            self.queue_vc[qn] = _join(self.queue_vc[qn], self.vc[op])
            self.queues[qn].append(None)
        elif kind == "commit":
            _, qn, bar_name, n = act
            self.queues[qn].append((bar_name, n, dict(self.queue_vc[qn])))
        elif kind in ("nb_arrive", "nb_sync"):
            gen = self._nb_arrive(agent, act[1], act[2])
            if kind == "nb_sync":
                self.blocked[agent] = ("nb", act[1], gen)
        elif kind == "bulk":
            op = self._new_agent("bulk", self._release(agent))
            for r in act[1]:
                self._access(op, r, False)
            self.bulk.setdefault(agent, []).append(op)
            self.bulk_pending.append((agent, op))
        elif kind == "bulk_wait":
            self.blocked[agent] = ("bulk",)
        elif kind in ("rd", "wr"):
            self._access(agent, act[1], kind == "wr")
        else:
            raise AssertionError(act)

    def _runnable(self, name):
        st = self.blocked.get(name)
        if st is None:
            return True
        if st[0] == "mb":
            return self.bars[st[1]].done >= st[2] + 1
        if st[0] == "nb":
            return self.nb[st[1]][0] > st[2]
        return not any(a == name for a, _ in self.bulk_pending)

    def run(self, roles, max_steps=500000):
        for name in roles:
            self.vc[name] = {name: 1}
        live = dict(roles)
        for _ in range(max_steps):
            roles_ready = [("role", n) for n in sorted(live) if self._runnable(n)]
            engine = [("tc", qn) for qn, qu in self.queues.items() if qu]
            engine += [("tma", i) for i in range(len(self.inflight))]
            engine += [("bulk", i) for i in range(len(self.bulk_pending))]
            if not roles_ready and not engine:
                if live:
                    raise Deadlock({n: self.blocked.get(n) for n in live})
                break
            kind, x = self.rng.choices(roles_ready + engine,
                                       [1.0] * len(roles_ready) + [self.engine_weight] * len(engine))[0]
            if kind == "tc":
                entry = self.queues[x].pop(0)
                if entry is not None:  # a commit: every MMA before it is done
                    self._arrive(*entry)
            elif kind == "tma":
                bar_name, n, vc = self.inflight.pop(x)
                self._arrive(bar_name, n, vc, done_tx=True)
            elif kind == "bulk":
                self.bulk_pending.pop(x)
            else:
                st = self.blocked.pop(x, None)
                if st is not None and st[0] == "mb" and st[2] >= 0:
                    self.vc[x] = _join(self.vc[x], self.bars[st[1]].phase_vc[st[2]])
                elif st is not None and st[0] == "nb":
                    self.vc[x] = _join(self.vc[x], self.nb_vc[(st[1], st[2])])
                elif st is not None and st[0] == "bulk":
                    for op in self.bulk.pop(x, []):
                        self.vc[x] = _join(self.vc[x], self.vc[op])
                try:
                    act = next(live[x])
                except StopIteration:
                    del live[x]
                    continue
                self._do(x, act)
        else:
            raise AssertionError("step limit")
        for nid, st in self.nb.items():
            if st[2]:
                raise Violation(f"named barrier {nid} ends with an incomplete generation")
        for name, bar in self.bars.items():
            if bar.arrived or bar.tx:
                raise Violation(f"mbarrier {name} ends with arrivals pending")
        if self.bulk_pending:
            raise Violation("bulk copies still in flight at the end")
