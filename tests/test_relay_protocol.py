"""The shared-memory relay of the GEMM epilogue (tc_gemm.cuh), as a protocol.

With the relay, a copying warp reads TMEM lane quarter q and hands it, 32
columns at a time, to a computing warp through two shared-memory slots. Four
64-thread named barriers carry the hand-off: full(s) (bar.arrive by the
copier, bar.sync by the computer) and empty(s) (the reverse). The copier
passes all 8 chunks of every tile with a non-empty contraction, waiting on
empty(s) before it refills a slot, and at the end it waits on empty(s) once
more for each slot it used. The computer takes chunks in column order, and
releases unread any chunk that its policy skips or does not reach.

Named barriers have no timeout, so a mismatch would hang the kernel. This
test executes both warps' barrier sequences in random interleavings. It checks
that they never deadlock, that no warp counts twice toward one barrier phase,
that a slot is refilled only after it was released, that every chunk read is
the one written, and that every barrier ends with no pending arrivals.
"""
import random

import pytest

CHUNKS = 8  # 256 accumulator columns / 32


def copier_ops(tiles):
    ops, used = [], set()
    for zero, _ in tiles:
        if zero:
            continue
        for ch in range(CHUNKS):
            s = ch & 1
            if s in used:
                ops.append(("sync", ("empty", s)))
            used.add(s)
            ops += [("put", s, ch), ("arrive", ("full", s))]
    ops += [("sync", ("empty", s)) for s in (0, 1) if s in used]
    return ops


def computer_ops(tiles):
    ops = []
    for zero, loads in tiles:
        if zero:
            continue
        taken = 0

        def skip_to(ch):
            nonlocal taken
            while taken < ch:
                s = taken & 1
                ops.extend([("sync", ("full", s)), ("release", s), ("arrive", ("empty", s))])
                taken += 1

        for ch in loads:  # increasing chunk indices
            skip_to(ch)
            s = taken & 1
            ops.extend([("sync", ("full", s)), ("get", s, ch), ("release", s),
                        ("arrive", ("empty", s))])
            taken += 1
        skip_to(CHUNKS)
    return ops


def execute(tiles, rng, computer=computer_ops):
    prog = {"copier": copier_ops(tiles), "computer": computer(tiles)}
    pc = {w: 0 for w in prog}
    phase = {}    # barrier -> warps counted toward its current phase
    blocked = {}  # warp -> barrier it waits on
    slot = {0: None, 1: None}
    while True:
        ready = [w for w in prog if pc[w] < len(prog[w]) and w not in blocked]
        if not ready:
            assert not blocked, f"deadlock: pc={pc} blocked={blocked}"
            break
        w = rng.choice(ready)
        op = prog[w][pc[w]]
        kind = op[0]
        if kind in ("sync", "arrive"):
            members = phase.setdefault(op[1], [])
            assert w not in members, f"{w} counted twice toward {op[1]}"
            members.append(w)
            if len(members) == 2:  # 64 threads: both warps
                phase[op[1]] = []
                for other, b in list(blocked.items()):
                    if b == op[1]:
                        del blocked[other]
                        pc[other] += 1
                pc[w] += 1
            elif kind == "sync":
                blocked[w] = op[1]
            else:
                pc[w] += 1
        elif kind == "put":
            assert slot[op[1]] is None, f"slot {op[1]} refilled before release"
            slot[op[1]] = op[2]
            pc[w] += 1
        elif kind == "get":
            assert slot[op[1]] == op[2], f"read chunk {slot[op[1]]}, wanted {op[2]}"
            pc[w] += 1
        else:  # release
            slot[op[1]] = None
            pc[w] += 1
    assert all(not m for m in phase.values()), f"pending arrivals: {phase}"
    assert slot == {0: None, 1: None}


def random_tiles(rng):
    tiles = []
    for _ in range(rng.randint(1, 7)):
        zero = rng.random() < 0.15            # empty contraction: no relay at all
        k = rng.randint(0, CHUNKS)            # chunks the policy loads
        loads = list(range(k)) if rng.random() < 0.7 else sorted(rng.sample(range(CHUNKS), k))
        tiles.append((zero, loads))
    return tiles


@pytest.mark.parametrize("seed", range(4))
def test_relay_protocol_random_interleavings(seed):
    rng = random.Random(seed)
    for _ in range(600):
        execute(random_tiles(rng), rng)


def test_relay_protocol_catches_a_missing_release():
    """A computer that does not release the chunks its policy skips leaves the
    copier waiting on a slot: the checker must report it."""
    def no_release_of_skipped(t):
        ops = []
        for zero, loads in t:
            if zero:
                continue
            for i, ch in enumerate(loads):
                s = i & 1
                ops.extend([("sync", ("full", s)), ("get", s, ch), ("release", s),
                            ("arrive", ("empty", s))])
        return ops

    with pytest.raises(AssertionError):
        execute([(False, [0, 1]), (False, [0])], random.Random(0), no_release_of_skipped)
