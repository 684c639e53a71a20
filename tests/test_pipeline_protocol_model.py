"""CPU model of the forward kernel's barrier protocol (no GPU).

A discrete-event restatement of attn_fwd_kernel.cuh's roles and mbarriers:

* the producer: Q once, then K_j into a 3-slot ring and V_j into a 2-slot
  ring.  K_j waits for the release of K_(j-3)'s slot; V_j for the release of
  V_(j-2)'s slot, which the key-split build signals on its own barrier and the
  other builds with step j - 1's release commit on K_(j-1)'s slot;
* the MMA issuer (one thread, mma_role): step 0 issues S_s(0) for each
  sub-tile that reads tile 0; step j >= 1 waits for K_j, then per sub-tile the
  PV of tile j - 1 (after V_(j-1), waited once per step; its first half after
  that sub-tile's first half of P, the rest after all of P) and S of tile j,
  and makes one release commit on K_j's slot; the
  key-split build runs its own loop (alternate tiles per sub-tile, PV's V
  release per tile);
* one softmax group per sub-tile: waits for each of its S, releases the
  first half of its P, then all of it (the key split: all of it at once).

Commits arrive when every earlier tensor operation has left the tensor pipe,
which runs them in issue order.  Loads complete after random delays, and the
roles advance in random order.

Checked over the tile schedules of the square, non-causal, windowed,
global-token and key-split builds: the run ends (no deadlock); no wait ever
sees a barrier two phases ahead (the parity test would alias); a K or V slot
is rewritten only after every product reading the tile it held has left the
tensor pipe; and each sub-tile's PV(t) is issued before its S of the next tile
it reads (S overwrites P)."""

import random

import pytest

K_ST, V_ST = 3, 2


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, k):
        """Has the k-th phase (0-based) completed?  The kernel's parity wait
        can only tell phase k from k + 2 if the barrier is at most one phase
        past k."""
        assert self.phase <= k + 1, "a waiter fell two phases behind (parity alias)"
        return self.phase > k


def schedule_cases():
    """(n_tot, reads[sub] = the streamed tiles each sub-tile reads, key split?)."""
    cases = []
    for n in (1, 2, 3, 4, 5, 8, 13):
        cases.append((n, [list(range(n - 1)) if n > 1 else [], list(range(n))], False))  # square causal
        cases.append((n, [list(range(n)), list(range(n))], False))                          # non-causal
        cases.append((n, [list(range(n)), []], False))                                      # sub-tile 1 past the end
        cases.append((n, [list(range(min(2, n))), list(range(max(0, n - 3), n))], False))   # windows
        cases.append((n, [list(range(0, n, 2)), list(range(1, n, 2))], True))               # key split
        if n >= 4:                                                                          # global + window phases
            cases.append((n, [[0, 1] + list(range(2, n - 1)), [0] + list(range(3, n))], False))
    return cases


def run(n_tot, reads, ks_build, seed, v_step_back=1):
    rng = random.Random(seed)
    bars = {"q_full": Barrier(1)}
    for i in range(K_ST):
        bars[f"k_full{i}"], bars[f"k_empty{i}"] = Barrier(1), Barrier(1)
    for i in range(V_ST):
        bars[f"v_full{i}"], bars[f"v_empty{i}"] = Barrier(1), Barrier(1)
    for s in range(2):
        bars[f"s_full{s}"], bars[f"p_full{s}"], bars[f"o_done{s}"] = Barrier(1), Barrier(1), Barrier(1)
        bars[f"p_half{s}"] = Barrier(1)
    pipe, inflight = [], []
    k_slot, v_slot = [None] * K_ST, [None] * V_ST
    left = {}      # ("k" | "v", tile) -> number of products reading it that left the pipe
    events = []
    own = [{t: n for n, t in enumerate(r)} for r in reads]

    def readers(kind, t):
        return sum(1 for s in range(2) if t in own[s])

    def wait(name, k):
        while not bars[name].done(k):
            yield

    def producer():
        inflight.append([rng.randint(1, 5), "q_full"])
        for j in range(n_tot):
            ks, vs = j % K_ST, j % V_ST
            if j >= K_ST:
                yield from wait(f"k_empty{ks}", (j - K_ST) // K_ST)
            if k_slot[ks] is not None:
                assert left.get(("k", k_slot[ks]), 0) == readers("k", k_slot[ks]), "K slot rewritten early"
            k_slot[ks] = j
            inflight.append([rng.randint(1, 8), f"k_full{ks}"])
            if j >= V_ST:
                if ks_build:
                    yield from wait(f"v_empty{vs}", (j - 2) // V_ST)
                else:
                    yield from wait(f"k_empty{(j - v_step_back) % K_ST}", (j - v_step_back) // K_ST)
            if v_slot[vs] is not None:
                assert left.get(("v", v_slot[vs]), 0) == readers("v", v_slot[vs]), "V slot rewritten early"
            v_slot[vs] = j
            inflight.append([rng.randint(1, 8), f"v_full{vs}"])

    def mma(op, s, t):
        pipe.append(("mma", op, t))
        events.append((s, op, t))

    def issuer():
        if n_tot == 0:
            return
        yield from wait("q_full", 0)
        if ks_build:
            for jl in range((n_tot + 1) // 2 + 1):
                for s in range(2):
                    tp = 2 * (jl - 1) + s
                    if jl > 0 and tp < n_tot:
                        yield from wait(f"v_full{tp % V_ST}", tp // V_ST)
                        yield from wait(f"p_full{s}", jl - 1)
                        mma("pv", s, tp)
                        if jl - 1 == len(reads[s]) - 1:
                            pipe.append(("commit", None, f"o_done{s}"))
                        pipe.append(("commit", None, f"v_empty{tp % V_ST}"))
                    tn = 2 * jl + s
                    if tn < n_tot:
                        yield from wait(f"k_full{tn % K_ST}", tn // K_ST)
                        mma("s", s, tn)
                        pipe.append(("commit", None, f"s_full{s}"))
                        pipe.append(("commit", None, f"k_empty{tn % K_ST}"))
                    yield
        else:
            yield from wait("k_full0", 0)
            for s in range(2):
                if 0 in own[s]:
                    mma("s", s, 0)
                    pipe.append(("commit", None, f"s_full{s}"))
            pipe.append(("commit", None, "k_empty0"))
            for j in range(1, n_tot + 1):
                i, has_k = j - 1, j < n_tot
                if has_k:
                    yield from wait(f"k_full{j % K_ST}", j // K_ST)
                v_ready = False
                for s in range(2):
                    if i in own[s]:
                        if not v_ready:
                            yield from wait(f"v_full{i % V_ST}", i // V_ST)
                        v_ready = True
                        yield from wait(f"p_half{s}", own[s][i])
                        mma("pv_first_half", s, i)
                        yield from wait(f"p_full{s}", own[s][i])
                        mma("pv", s, i)
                        if own[s][i] == len(reads[s]) - 1:
                            pipe.append(("commit", None, f"o_done{s}"))
                    if has_k and j in own[s]:
                        mma("s", s, j)
                        pipe.append(("commit", None, f"s_full{s}"))
                if has_k:
                    pipe.append(("commit", None, f"k_empty{j % K_ST}"))
                yield
        for t in range(max(0, n_tot - K_ST), n_tot):
            yield from wait(f"k_empty{t % K_ST}", t // K_ST)
        if ks_build:
            for t in range(max(0, n_tot - V_ST), n_tot):
                yield from wait(f"v_empty{t % V_ST}", t // V_ST)
        for s in range(2):
            if reads[s]:
                yield from wait(f"o_done{s}", 0)

    def softmax(s):
        for li in range(len(reads[s])):
            yield from wait(f"s_full{s}", li)
            for _ in range(rng.randint(0, 3)):
                yield
            if not ks_build:
                bars[f"p_half{s}"].arrive()
                for _ in range(rng.randint(0, 3)):
                    yield
            bars[f"p_full{s}"].arrive()
        if reads[s]:
            yield from wait(f"o_done{s}", 0)

    def tensor_pipe():
        while True:
            if pipe and rng.random() < 0.6:
                kind, op, what = pipe.pop(0)
                if kind == "commit":
                    bars[what].arrive()
                elif op != "pv_first_half":
                    key = ("k" if op == "s" else "v", what)
                    left[key] = left.get(key, 0) + 1
            yield

    def loads():
        while True:
            for f in list(inflight):
                f[0] -= 1
                if f[0] <= 0:
                    inflight.remove(f)
                    bars[f[1]].arrive()
            yield

    roles = [producer(), issuer(), softmax(0), softmax(1)]
    aux = [tensor_pipe(), loads()]
    alive = list(roles)
    for _ in range(200000):
        if not alive:
            break
        for a in aux:
            next(a)
        r = rng.choice(alive)
        try:
            next(r)
        except StopIteration:
            alive.remove(r)
    assert not alive, f"deadlock: {len(alive)} roles still waiting"
    for s in range(2):
        mine = [e for e in events if e[0] == s]
        for a, b in zip(reads[s], reads[s][1:]):
            assert mine.index((s, "pv", a)) < mine.index((s, "s", b))
            if not ks_build:
                assert mine.index((s, "pv_first_half", a)) < mine.index((s, "pv", a))
        if reads[s]:
            assert (s, "pv", reads[s][-1]) in mine


@pytest.mark.parametrize("case", range(len(schedule_cases())))
def test_protocol_ends_without_aliasing_or_early_slot_reuse(case):
    n_tot, reads, ks_build = schedule_cases()[case]
    for seed in range(12):
        run(n_tot, reads, ks_build, seed)


def test_a_release_one_step_early_is_caught():
    """Planted mistake: the producer reuses V_(j-2)'s slot after step j - 2's
    commit instead of step j - 1's, whose commit is the first to cover the
    PV of tile j - 2."""
    n_tot, reads = 8, [list(range(7)), list(range(8))]
    caught = 0
    for seed in range(40):
        try:
            run(n_tot, reads, False, seed, v_step_back=2)
        except AssertionError:
            caught += 1
    assert caught > 0
