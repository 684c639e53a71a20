"""CPU model of the backward kernel's barrier protocol (no GPU).

A discrete-event restatement of attn_bwd_kernel.cuh's roles and mbarriers,
with every tensor-memory region and shared-memory stage carrying a tag of
what it holds, checked at each read:

* the producer: K and V once; per step i, Q_i into Q stage i mod 2 after the
  release of step i - 2 (q_empty), dO_i into dO stage i mod 2 likewise
  (do_empty);
* the MMA issuer (one thread): S_0 first; per step dP_i (after dO_i and the
  read-out of dQ_(i-1), which dP^T overwrites), dV_i (after P^T_i), the next
  step's S^T (after the dS phase has read P^T_i back), then dK_i and dQ_i
  (after dS_i) and the step's release commits;
* two compute warpgroups (one half of the query columns each): P phase
  (S^T -> P^T in place), then the dS phase: P^T read back, dP^T read, dS^T
  written over it, dS written into shared memory (over dO_i once dV_i has
  read it, or into a tile of its own once dQ_(i-1) has read the last dS);
* the dQ warpgroup: dQ_i read out of the dP^T region.

The tensor pipe runs its operations in issue order; a commit arrives when it
reaches the head of the pipe (every earlier operation has completed).  Loads
land after random delays; the roles advance in random order.

Checked: the run ends (no deadlock); no wait ever sees a barrier two phases
ahead (the parity test would alias); every read, by the tensor core or by a
warpgroup, finds the value of the step it expects.  Three planted mistakes
(the next S^T issued without waiting for the P^T read-back; dS written over
dO_i before dV_i has read it; dQ_i issued before dK_i, so that it overwrites
dS^T first) must each be caught.  (Releasing the dO stage right after dV_i
would go unnoticed: the producer refills a step's Q stage first, and that
release follows dQ_i.)"""

import random

import pytest


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
        assert self.phase <= k + 1, "a waiter fell two phases behind (parity alias)"
        return self.phase > k


def run(steps, seed, ds_in_do=True, early_s=False, skip_dv_wait=False, dq_before_dk=False):
    rng = random.Random(seed)
    bars = {"kv_full": Barrier(1), "s_full": Barrier(1), "dp_full": Barrier(1), "dv_done": Barrier(1),
            "p_ready": Barrier(2), "p_read": Barrier(2), "ds_ready": Barrier(2), "dq_full": Barrier(1),
            "dq_empty": Barrier(1), "kv_done": Barrier(1)}
    for s in range(2):
        for b in ("q_full", "q_empty", "do_full", "do_empty"):
            bars[f"{b}{s}"] = Barrier(1)
    # tags: tensor memory halves, shared-memory stages (halves for dO, which dS replaces)
    tm = {("S", h): None for h in range(2)} | {("DP", h): None for h in range(2)}
    sm = {"K": None, "V": None} | {("Q", s): None for s in range(2)}
    sm |= {("dO", s, h): None for s in range(2) for h in range(2)}
    sm |= {("dS", h): None for h in range(2)}  # the separate dS tile (D < 128)
    pipe, inflight = [], []

    def expect(store, key, want):
        assert store[key] == want, f"{key} holds {store[key]}, expected {want}"

    def wait(name, k):
        while not bars[name].done(k):
            yield

    def ds_key(i, h):
        return ("dO", i & 1, h) if ds_in_do else ("dS", h)

    def producer():
        inflight.append([rng.randint(1, 6), [("K", ("K",)), ("V", ("V",))], "kv_full"])
        for i in range(steps):
            s = i & 1
            if i >= 2:
                yield from wait(f"q_empty{s}", (i >> 1) - 1)
            inflight.append([rng.randint(1, 8), [(("Q", s), ("Q", i))], f"q_full{s}"])
            if i >= 2:
                yield from wait(f"do_empty{s}", (i >> 1) - 1)
            inflight.append([rng.randint(1, 8), [(("dO", s, h), ("dO", i)) for h in range(2)], f"do_full{s}"])
            yield

    # tensor-pipe operations: (reads of shared memory, reads of tensor memory, writes of tensor memory)
    def op_s(i):
        return ([("K", ("K",)), (("Q", i & 1), ("Q", i))], [], [(("S", h), ("S", i)) for h in range(2)])

    def op_dp(i):
        return ([("V", ("V",))] + [(("dO", i & 1, h), ("dO", i)) for h in range(2)], [],
                [(("DP", h), ("dP", i)) for h in range(2)])

    def op_dv(i):
        return ([(("dO", i & 1, h), ("dO", i)) for h in range(2)], [(("S", h), ("P", i)) for h in range(2)], [])

    def op_dk(i):
        return ([(("Q", i & 1), ("Q", i))], [(("DP", h), ("dS", i)) for h in range(2)], [])

    def op_dq(i):
        return ([("K", ("K",))] + [(ds_key(i, h), ("dS", i)) for h in range(2)], [],
                [(("DP", h), ("dQ", i)) for h in range(2)])

    def issue(op):
        pipe.append(("op", op))

    def commit(name):
        pipe.append(("commit", name))

    def issuer():
        yield from wait("kv_full", 0)
        yield from wait("q_full0", 0)
        issue(op_s(0))
        commit("s_full")
        for i in range(steps):
            s = i & 1
            yield from wait(f"do_full{s}", i >> 1)
            if i > 0:
                yield from wait("dq_empty", i - 1)
            issue(op_dp(i))
            commit("dp_full")
            yield from wait("p_ready", i)
            issue(op_dv(i))
            commit("dv_done")
            if i + 1 < steps:
                if not early_s:
                    yield from wait("p_read", i)
                yield from wait(f"q_full{(i + 1) & 1}", (i + 1) >> 1)
                issue(op_s(i + 1))
                commit("s_full")
            yield from wait("ds_ready", i)
            if dq_before_dk:
                issue(op_dq(i))
                issue(op_dk(i))
            else:
                issue(op_dk(i))
                issue(op_dq(i))
            commit("dq_full")
            commit(f"q_empty{s}")
            commit(f"do_empty{s}")
        commit("kv_done")
        for i in range(max(0, steps - 2), steps):
            yield from wait(f"q_empty{i & 1}", i >> 1)
            yield from wait(f"do_empty{i & 1}", i >> 1)

    def pause(n=3):
        for _ in range(rng.randint(0, n)):
            yield

    def compute(h):
        for i in range(steps):
            yield from wait("s_full", i)
            expect(tm, ("S", h), ("S", i))
            yield from pause()
            tm[("S", h)] = ("P", i)
            bars["p_ready"].arrive()
            yield from wait("dp_full", i)
            expect(tm, ("S", h), ("P", i))
            yield from pause()
            expect(tm, ("S", h), ("P", i))   # still there up to the read-back's last column
            bars["p_read"].arrive()
            expect(tm, ("DP", h), ("dP", i))
            yield from pause()
            tm[("DP", h)] = ("dS", i)
            if ds_in_do:
                if not skip_dv_wait:
                    yield from wait("dv_done", i)
            elif i > 0:
                yield from wait("dq_full", i - 1)
            sm[ds_key(i, h)] = ("dS", i)
            yield from pause()
            bars["ds_ready"].arrive()
        if steps:
            yield from wait("kv_done", 0)

    def dq_role():
        for i in range(steps):
            yield from wait("dq_full", i)
            for h in range(2):
                expect(tm, ("DP", h), ("dQ", i))
            yield from pause()
            bars["dq_empty"].arrive()

    def tensor_pipe():
        busy = 0
        while True:
            if pipe and busy == 0 and rng.random() < 0.5:
                kind, what = pipe.pop(0)
                if kind == "commit":
                    bars[what].arrive()
                else:
                    reads_sm, reads_tm, writes_tm = what
                    for key, want in reads_sm:
                        expect(sm, key, want)
                    for key, want in reads_tm:
                        expect(tm, key, want)
                    for key, val in writes_tm:
                        tm[key] = val
                    busy = rng.randint(0, 3)
            elif busy:
                busy -= 1
            yield

    def loads():
        while True:
            for f in list(inflight):
                f[0] -= 1
                if f[0] <= 0:
                    inflight.remove(f)
                    for key, val in f[1]:
                        sm[key] = val
                    bars[f[2]].arrive()
            yield

    roles = [producer(), issuer(), compute(0), compute(1), dq_role()] if steps else []
    aux = [tensor_pipe(), loads()]
    alive = list(roles)
    for _ in range(400000):
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


@pytest.mark.parametrize("steps", [1, 2, 3, 4, 7, 12])
@pytest.mark.parametrize("ds_in_do", [True, False])
def test_protocol_ends_and_every_read_sees_its_step(steps, ds_in_do):
    for seed in range(15):
        run(steps, seed, ds_in_do=ds_in_do)


@pytest.mark.parametrize("mistake", ["early_s", "skip_dv_wait", "dq_before_dk"])
def test_planted_protocol_mistakes_are_caught(mistake):
    caught = 0
    for seed in range(60):
        try:
            run(6, seed, **{mistake: True})
        except AssertionError:
            caught += 1
    assert caught > 0
