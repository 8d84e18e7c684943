"""A model of the attention kernel's mbarrier protocol, explored under random
schedules on the CPU: a race detector for the synchronisation of
``attn_fwd.cuh`` (test infrastructure; it models the kernel, it does not run
it).

One persistent CTA runs a list of work items.  Each item has two query tiles
with ``nk0`` and ``nkv`` key tiles.  The roles are written as generators that
mirror the kernel's loops operation for operation:

- the producer (Q once per item into one of ``q_bufs`` buffers, K and V
  through a ring of ``stages``);
- the QK warp (S products in the order S0(0), S1(0), S0(1), ...);
- one P.V warp, or one per query tile (``split_pv``);
- the two softmax groups (copy S out, write P, read O in the epilogue).

With ``p_halves`` P is written and announced in two 64-key halves
(``p_half`` after the first, ``p_full`` after the second) and each P.V
product is issued as two MMAs, one per half, each after its half.

With ``order_pv`` the P.V product of key tile j waits until the tile's S
product of key tile j+1 has been issued, through ``qk_go`` barriers (the BF16
schedule).  ``qk_go`` sets how many barriers each tile has.

The engine's semantics:
- A barrier completes a phase when its expected arrivals are in.
- A wait for phase k is valid only while the barrier is at phase k or k+1.
  Parity waits cannot tell phases two apart: two behind would wait forever,
  one ahead would pass early. Any other phase is reported as aliasing.
- MMAs run one at a time in issue order (the tensor pipe).
- A commit arrives once every MMA its thread issued before it has run.
- TMA loads land at any later time.

Data checks, at the moment each access happens:
- an S product runs only after the previous S was copied out;
- a P.V product reads the P written for it, with its K/V stage holding the right tile;
- P is rewritten only after its P.V product ran;
- the epilogue reads O only after every P.V product of the item;
- the next item's first P.V product runs only after that read;
- a ring stage or Q is reloaded only after every product that reads it ran.

The failure path (``inject_timeout``): at a random moment one blocked wait
runs out of time and sets the CTA's abort word, as the kernel's bounded waits
do.
- From then on a wait that would block returns instead, and its role leaves
  its loop through the kernel's exit sequence.
- The producer then waits for the loads it may still have in flight (the last
  ``stages`` of K and of V, and the last ``q_bufs`` of Q).
- Each issuing warp commits and waits for its own MMAs.

At the CTA's exit, also after a normal run, no TMA load, MMA or commit
arrival may still be in flight: each would write to the shared or tensor
memory of the CTA that comes next.

``run`` returns None, or raises ``Violation`` for the first violation or deadlock.
"""
from __future__ import annotations

import random
from dataclasses import dataclass, field


class Violation(Exception):
    pass


@dataclass
class Barrier:
    name: str
    count: int
    pending: int = 0
    phase: int = 0  # completed phases

    def __post_init__(self):
        self.pending = self.count

    def arrive(self, n=1):
        self.pending -= n
        if self.pending < 0:
            raise Violation(f"{self.name}: more arrivals than expected in phase {self.phase}")
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count


@dataclass
class Protocol:
    """Which variant of the protocol to model (the kernel's is the default:
    4 ``qk_go`` barriers, one P.V warp, a ring of 4 stages)."""
    stages: int = 4
    q_bufs: int = 1
    p_halves: bool = False
    order_pv: bool = False
    qk_go: int = 4
    split_pv: bool = False
    # a variant measured on the GPU and not kept (the softmax compiled
    # slower): softmax 0 starts its epilogue only after tile 1 has written the
    # item's last P; softmax 1 arrives on p1_last after its last P of an item
    epi_after_p1: bool = False
    # planted mistake: the same wait as a parity wait on p_full1, which can be
    # two phases ahead when tile 1 has two more key tiles to go
    epi_wait_on_p_full1: bool = False
    # planted mistakes, for the tests that show the checker finds them
    skip_drain_wait: bool = False
    skip_o_done_wait: bool = False
    skip_q_empty_wait: bool = False
    # the failure path: one bounded wait runs out of time
    inject_timeout: bool = False
    skip_producer_drain: bool = False
    skip_mma_drain: bool = False


@dataclass
class _State:
    s_content: tuple | None = None  # (t, item, j) of the S product in S
    s_read: bool = True
    p: dict = field(default_factory=dict)        # t -> [(item, j), consumed, halves written]
    o_item: dict = field(default_factory=dict)   # t -> item accumulating in O_t
    o_done_n: dict = field(default_factory=dict) # t -> P.V products run for o_item
    o_free: dict = field(default_factory=dict)   # t -> epilogue has read O_t
    k_stage: dict = field(default_factory=dict)  # st -> (item, j)
    v_stage: dict = field(default_factory=dict)
    q: dict = field(default_factory=dict)        # Q buffer -> item
    reads_needed: dict = field(default_factory=dict)  # ('K'|'V'|'Q', version) -> n
    reads_done: dict = field(default_factory=dict)


def _wait(bar, k):
    return ("wait", bar, k)


class Model:
    def __init__(self, items, proto: Protocol, rng: random.Random):
        self.items, self.p, self.rng = items, proto, rng
        S = proto.stages
        B = Barrier
        self.bars = {
            **{f"q_full{i}": B(f"q_full{i}", 1) for i in range(proto.q_bufs)},
            **{f"q_empty{i}": B(f"q_empty{i}", 1) for i in range(proto.q_bufs)},
            **{f"k_full{i}": B(f"k_full{i}", 1) for i in range(S)},
            **{f"k_empty{i}": B(f"k_empty{i}", 1) for i in range(S)},
            **{f"v_full{i}": B(f"v_full{i}", 1) for i in range(S)},
            **{f"v_empty{w}_{i}": B(f"v_empty{w}_{i}", 1) for w in range(2) for i in range(S)},
            **{f"s_full{t}": B(f"s_full{t}", 1) for t in range(2)},
            **{f"s_drained{t}": B(f"s_drained{t}", 1) for t in range(2)},
            **{f"p_full{t}": B(f"p_full{t}", 1) for t in range(2)},
            **{f"p_half{t}": B(f"p_half{t}", 1) for t in range(2)},
            **{f"o_done{t}": B(f"o_done{t}", 1) for t in range(2)},
            **{f"o_free{t}": B(f"o_free{t}", 1) for t in range(2)},
            "p1_last": B("p1_last", 1),
            **{f"qk_go{t}_{i}": B(f"qk_go{t}_{i}", 1) for t in range(2) for i in range(proto.qk_go)},
            **{f"drain_{r}": B(f"drain_{r}", 1) for r in ("qk", "pv0", "pv1")},
        }
        self.abort = False
        self.n_k = self.n_v = self.n_q = 0  # loads the producer has issued
        self.st = _State()
        for t in range(2):
            self.st.p[t] = [None, True, 2]
            self.st.o_item[t] = None
            self.st.o_done_n[t] = 0
            self.st.o_free[t] = True
        self.pipe = []       # issued, not yet run: (seq, thread, kind, args)
        self.seq = 0
        self.last_issued = {}  # thread -> seq of its last issued MMA
        self.ran = -1        # seq of the last MMA run (the pipe is in order)
        self.commits = []    # (thread, seq bound, barrier), in issue order
        self.tmas = []       # (barrier, kind, stage, version)
        self.roles = {"producer": self._producer(), "qk": self._qk()}
        if proto.split_pv:
            self.roles["pv0"] = self._pv(0, (0,))
            self.roles["pv1"] = self._pv(1, (1,))
        else:
            self.roles["pv0"] = self._pv(0, (0, 1))
        self.roles["sm0"] = self._softmax(0)
        self.roles["sm1"] = self._softmax(1)
        self.next_op = {name: next(g) for name, g in self.roles.items()}

    # ---------------------------------------------------------------- roles
    def _nk(self, item, t):
        nk0, nkv = self.items[item]
        return nkv if t else nk0

    def _producer(self):
        S = self.p.stages
        kv_it = 0
        QB = self.p.q_bufs
        for item, (nk0, nkv) in enumerate(self.items):
            if item >= QB and not self.p.skip_q_empty_wait:
                yield _wait(f"q_empty{item % QB}", item // QB - 1)
            yield ("tma", f"q_full{item % QB}", "Q", item % QB, item)
            for j in range(nkv):
                st, use = kv_it % S, kv_it // S
                if use > 0:
                    yield _wait(f"k_empty{st}", use - 1)
                yield ("tma", f"k_full{st}", "K", st, (item, j))
                for w in range(2 if self.p.split_pv else 1):
                    if use > 0:
                        yield _wait(f"v_empty{w}_{st}", use - 1)
                yield ("tma", f"v_full{st}", "V", st, (item, j))
                kv_it += 1
        # also after a normal end: a wait elsewhere may still run out of time
        # while its last loads are in flight
        yield from self._producer_drain()
        yield ("done",)

    def _producer_drain(self):
        """The kernel's producer before it leaves, after a normal end or an
        abort: every copy it started must have landed before the CTA may
        exit."""
        if self.p.skip_producer_drain:
            return
        S = self.p.stages
        for i in range(max(0, self.n_k - S), self.n_k):
            yield ("wait_drain", f"k_full{i % S}", i // S)
        for i in range(max(0, self.n_v - S), self.n_v):
            yield ("wait_drain", f"v_full{i % S}", i // S)
        QB = self.p.q_bufs
        for i in range(max(0, self.n_q - QB), self.n_q):
            yield ("wait_drain", f"q_full{i % QB}", i // QB)

    def _mma_drain(self, name):
        """An issuing warp's last steps, after its loop ends or gives up: its
        MMAs must be complete before tensor memory is released."""
        if self.p.skip_mma_drain:
            return
        yield ("commit", name, f"drain_{name}")
        yield ("wait_drain", f"drain_{name}", 0)

    def _exit(self, name):
        """The role's wait gave up (abort word set): leave its loop."""
        def gen():
            if name == "producer":
                yield from self._producer_drain()
            elif name in ("qk", "pv0", "pv1"):
                yield from self._mma_drain(name)
            yield ("done",)
        self.roles[name] = gen()
        self.next_op[name] = next(self.roles[name])

    def _qk(self):
        S = self.p.stages
        kv_it, issued, last = 0, [0, 0], -1
        QB = self.p.q_bufs
        for item, (nk0, nkv) in enumerate(self.items):
            yield _wait(f"q_full{item % QB}", item // QB)
            for j in range(nkv):
                st, use = kv_it % S, kv_it // S
                yield _wait(f"k_full{st}", use)
                for t in range(2):
                    if j >= (nkv if t else nk0):
                        continue
                    if last >= 0 and not self.p.skip_drain_wait:
                        yield _wait(f"s_drained{last}", issued[last] - 1)
                    yield ("mma", "qk", "S", (t, item, j, st))
                    if self.p.order_pv:
                        yield ("arrive", f"qk_go{t}_{issued[t] % self.p.qk_go}")
                    yield ("commit", "qk", f"s_full{t}")
                    issued[t] += 1
                    last = t
                yield ("commit", "qk", f"k_empty{st}")
                kv_it += 1
            yield ("commit", "qk", f"q_empty{item % QB}")
        yield from self._mma_drain("qk")
        yield ("done",)

    def _pv(self, w, tiles):
        S, G = self.p.stages, self.p.qk_go
        name = f"pv{w}"
        kv_it, p_cnt, qk_base, go_seen = 0, [0, 0], [0, 0], [0, 0]
        for item, (nk0, nkv) in enumerate(self.items):
            for j in range(nkv):
                st, use = kv_it % S, kv_it // S
                yield _wait(f"v_full{st}", use)
                for t in tiles:
                    nk = nkv if t else nk0
                    if j >= nk:
                        continue
                    if self.p.p_halves:
                        yield _wait(f"p_half{t}", p_cnt[t])
                    else:
                        yield _wait(f"p_full{t}", p_cnt[t])
                    if j == 0 and item > 0:
                        yield _wait(f"o_free{t}", item - 1)
                    if self.p.order_pv:
                        upto = qk_base[t] + (j + 1 if j + 1 < nk else j)
                        while go_seen[t] <= upto:
                            yield _wait(f"qk_go{t}_{go_seen[t] % G}", go_seen[t] // G)
                            go_seen[t] += 1
                    if self.p.p_halves:
                        yield ("mma", name, "PVa", (t, item, j, st))
                        yield _wait(f"p_full{t}", p_cnt[t])
                        yield ("mma", name, "PVb", (t, item, j, st))
                    else:
                        yield ("mma", name, "PV", (t, item, j, st))
                    p_cnt[t] += 1
                    yield ("commit", name, f"o_done{t}")
                yield ("commit", name, f"v_empty{w}_{st}")
                kv_it += 1
            qk_base[0] += nk0
            qk_base[1] += nkv
        yield from self._mma_drain(name)
        yield ("done",)

    def _softmax(self, t):
        s_cnt = o_cnt = 0
        p1_cnt = 0  # tile 1's P writes up to this item (counted by softmax 0)
        for item in range(len(self.items)):
            nk = self._nk(item, t)
            for j in range(nk):
                yield _wait(f"s_full{t}", s_cnt)
                s_cnt += 1
                yield ("read_s", t, item, j)
                yield ("arrive", f"s_drained{t}")
                if j > 0 and not self.p.skip_o_done_wait:
                    yield _wait(f"o_done{t}", o_cnt - 1)
                if self.p.p_halves:
                    yield ("write_p_half", t, item, j, 0)
                    yield ("arrive", f"p_half{t}")
                    yield ("write_p_half", t, item, j, 1)
                else:
                    yield ("write_p", t, item, j)
                yield ("arrive", f"p_full{t}")
                if self.p.epi_after_p1 and t == 1 and j == nk - 1:
                    yield ("arrive", "p1_last")
                o_cnt += 1
            if self.p.epi_after_p1 and t == 0:
                if self.p.epi_wait_on_p_full1:
                    p1_cnt += self._nk(item, 1)
                    yield _wait("p_full1", p1_cnt - 1)
                else:
                    yield _wait("p1_last", item)
            yield _wait(f"o_done{t}", o_cnt - 1)
            yield ("read_o", t, item)
            yield ("arrive", f"o_free{t}")
        yield ("done",)

    # ---------------------------------------------------------------- checks
    def _need(self, kind, version, n):
        key = (kind, version)
        self.st.reads_needed[key] = self.st.reads_needed.get(key, 0) + n

    def _read(self, kind, version):
        key = (kind, version)
        self.st.reads_done[key] = self.st.reads_done.get(key, 0) + 1

    def _all_read(self, kind, version):
        key = (kind, version)
        return self.st.reads_done.get(key, 0) >= self.st.reads_needed.get(key, 0)

    def _tma_issue(self, bar, kind, stage, version):
        st = self.st
        if kind == "Q":
            self.n_q += 1
        elif kind == "K":
            self.n_k += 1
        else:
            self.n_v += 1
        if kind == "Q":
            old = st.q.get(stage)
            if old is not None and not self._all_read("Q", old):
                raise Violation(f"Q buffer {stage} reloaded for item {version} while products "
                                f"still read item {old}")
            st.q[stage] = version
            nk0, nkv = self.items[version]
            self._need("Q", version, nk0 + nkv)
        else:
            table = st.k_stage if kind == "K" else st.v_stage
            old = table.get(stage)
            if old is not None and not self._all_read(kind, old):
                raise Violation(f"{kind} stage {stage} reloaded with {version} while {old} is still read")
            table[stage] = version
            item, j = version
            nk0, nkv = self.items[item]
            self._need(kind, version, (1 if j < nk0 else 0) + 1)
        self.tmas.append(bar)

    def _run_mma(self, thread, kind, args):
        st = self.st
        t, item, j, stage = args
        if kind == "S":
            if not st.s_read:
                raise Violation(f"S({t},{item},{j}) overwrites S{st.s_content} before it was copied out")
            qbuf = item % self.p.q_bufs
            if st.k_stage.get(stage) != (item, j) or st.q.get(qbuf) != item:
                raise Violation(f"S({t},{item},{j}) reads K stage {stage}={st.k_stage.get(stage)}, "
                                f"Q buffer {qbuf}={st.q.get(qbuf)}")
            self._read("K", (item, j))
            self._read("Q", item)
            st.s_content, st.s_read = (t, item, j), False
        else:
            # PV: the whole product; PVa / PVb: its halves (keys 0-63 / 64-127)
            pc, consumed, halves = st.p[t]
            need = 1 if kind == "PVa" else 2
            if pc != (item, j) or consumed or halves < need:
                raise Violation(f"{kind}({t},{item},{j}) reads P_{t}={pc} (consumed {consumed}, "
                                f"{halves} halves written)")
            if st.v_stage.get(stage) != (item, j):
                raise Violation(f"{kind}({t},{item},{j}) reads V stage {stage}={st.v_stage.get(stage)}")
            first = kind in ("PV", "PVa")
            if j == 0 and first:
                if not st.o_free[t]:
                    raise Violation(f"PV({t},{item},0) overwrites O_{t} before the epilogue read it")
                st.o_item[t], st.o_done_n[t], st.o_free[t] = item, 0, False
            elif st.o_item[t] != item:
                raise Violation(f"{kind}({t},{item},{j}) accumulates into O_{t} of item {st.o_item[t]}")
            if kind in ("PV", "PVb"):
                st.o_done_n[t] += 1
                st.p[t][1] = True
                self._read("V", (item, j))

    def _role_op(self, name, op):
        st = self.st
        kind = op[0]
        if kind == "arrive":
            self.bars[op[1]].arrive()
        elif kind == "tma":
            self._tma_issue(*op[1:])
        elif kind == "mma":
            self.seq += 1
            self.pipe.append((self.seq, op[1], op[2], op[3]))
            self.last_issued[op[1]] = self.seq
        elif kind == "commit":
            self.commits.append((op[1], self.last_issued.get(op[1], -1), op[2]))
        elif kind == "read_s":
            _, t, item, j = op
            if st.s_content != (t, item, j) or st.s_read:
                raise Violation(f"softmax {t} copies out S{st.s_content} expecting ({t},{item},{j})")
            st.s_read = True
        elif kind == "write_p" or (kind == "write_p_half" and op[4] == 0):
            t, item, j = op[1:4]
            pc, consumed, _ = st.p[t]
            if pc is not None and not consumed:
                raise Violation(f"softmax {t} writes P({item},{j}) over P{pc} before its P.V ran")
            st.p[t] = [(item, j), False, 2 if kind == "write_p" else 1]
        elif kind == "write_p_half":
            t, item, j = op[1:4]
            if st.p[t][0] != (item, j) or st.p[t][2] != 1:
                raise Violation(f"softmax {t} writes the second half of P({item},{j}) over {st.p[t]}")
            st.p[t][2] = 2
        elif kind == "read_o":
            _, t, item = op
            if st.o_item[t] != item or st.o_done_n[t] != self._nk(item, t):
                raise Violation(f"epilogue {t} reads O of item {item} after "
                                f"{st.o_done_n[t]} of {self._nk(item, t)} P.V products")
            st.o_free[t] = True
        else:
            raise AssertionError(op)

    # ---------------------------------------------------------------- engine
    def _wait_state(self, op):
        """True if the wait passes now; checks that it is not aliased."""
        bar, k = self.bars[op[1]], op[2]
        if bar.phase not in (k, k + 1):
            raise Violation(f"wait for phase {k} of {bar.name} while it has completed {bar.phase} "
                            f"phases: a parity wait cannot tell these apart")
        return bar.phase == k + 1

    def run(self, max_steps=200000):
        """Random schedule: every role and every kind of asynchronous event
        gets a random speed for the whole run, so that schedules where one
        role lags far behind the others (the ones that expose aliasing) come
        up often.  With ``inject_timeout`` one blocked wait gives up at a
        random step."""
        speed = {name: self.rng.choice((0.02, 0.2, 1.0)) for name in self.roles}
        for kind in ("pipe", "commit", "tma"):
            speed[kind] = self.rng.choice((0.05, 0.3, 1.0))
        timeout_at = self.rng.randint(0, 600) if self.p.inject_timeout else None
        done = set()
        for step in range(max_steps):
            choices, blocked = [], []
            for name in list(self.next_op):
                op = self.next_op[name]
                if name in done:
                    continue
                if op[0] == "done":
                    done.add(name)
                    continue
                if op[0] in ("wait", "wait_drain") and not self._wait_state(op):
                    if op[0] == "wait" and self.abort:
                        self._exit(name)  # the bounded wait sees the abort word
                        choices.append(("none", name))
                    elif op[0] == "wait":
                        blocked.append(name)
                    continue
                choices.append(("role", name))
            if len(done) == len(self.roles):
                # every role has finished: the CTA exits now
                if self.tmas:
                    raise Violation(f"the CTA exits with TMA loads in flight: {self.tmas}")
                if self.pipe:
                    raise Violation(f"the CTA exits with MMAs in flight: {self.pipe}")
                if self.commits:
                    raise Violation(f"the CTA exits with commit arrivals pending: {self.commits}")
                return None
            if timeout_at is not None and step >= timeout_at and blocked:
                # this wait's time limit runs out: it sets the abort word
                self.abort = True
                self._exit(self.rng.choice(blocked))
                timeout_at = None
                continue
            if self.pipe:
                choices.append(("pipe", None))
            for i, (thread, bound, _) in enumerate(self.commits):
                # a thread's commits arrive in order, each once its MMAs ran
                if bound <= self.ran and all(c[0] != thread for c in self.commits[:i]):
                    choices.append(("commit", i))
            for i in range(len(self.tmas)):
                choices.append(("tma", i))
            if not choices:
                stuck = {n: op for n, op in self.next_op.items() if n not in done}
                raise Violation(f"deadlock: {stuck}")
            weights = [speed.get(arg, 1.0) if what in ("role", "none") else speed[what]
                       for what, arg in choices]
            what, arg = self.rng.choices(choices, weights)[0]
            if what == "none":
                continue
            if what == "role":
                op = self.next_op[arg]
                if op[0] not in ("wait", "wait_drain"):
                    self._role_op(arg, op)
                self.next_op[arg] = next(self.roles[arg])
            elif what == "pipe":
                seq, thread, kind, args = self.pipe.pop(0)
                self._run_mma(thread, kind, args)
                self.ran = seq
            elif what == "commit":
                _, _, bar = self.commits.pop(arg)
                self.bars[bar].arrive()
            else:
                self.bars[self.tmas.pop(arg)].arrive()
        raise Violation("step limit")


def random_items(rng, n_items, max_tiles, causal):
    items = []
    for _ in range(n_items):
        nkv = rng.randint(1, max_tiles)
        nk0 = nkv - 1 if causal and nkv > 1 and rng.random() < 0.8 else nkv
        items.append((nk0, nkv))
    return items


def check(proto: Protocol, seeds, n_items=4, max_tiles=4):
    """Explore ``seeds`` random item lists and schedules; the first violation
    as (seed, items, message), else None."""
    for seed in seeds:
        rng = random.Random(seed)
        items = random_items(rng, n_items, max_tiles, causal=rng.random() < 0.7)
        try:
            Model(items, proto, rng).run()
        except Violation as e:
            return seed, items, str(e)
    return None
