"""A model of the split-barrier protocol of the wide row-panel pass
(memory_efficient_optimizer_gb300/csrc/row_panel.cuh, run_chunk_split), run
on the CPU under random interleavings of the warps.

Per sub-panel q every warp writes its row shares into share buffer q % B,
arrives on mbarrier q % 2 (completed by all warps' arrivals), and one
iteration later waits for that phase and reads every warp's shares of q.  The
model checks, for every interleaving it draws:

- every read of sub-panel q's shares finds sub-panel q's values (a buffer is
  rewritten only after every warp has read it);
- an arrival for q finds its mbarrier in q's phase (the phase of q - 2 on the
  same mbarrier has completed), so it is not counted toward an earlier one;
- a wait for q never finds its mbarrier two phases ahead (the parity test
  stays unambiguous);
- no warp waits forever (every interleaving finishes).

With B = 4 (the kernel's kShareBufs) no interleaving breaks these; with
B = 3 some do, which shows the checks can fail.
"""
import random

import pytest


class Violation(AssertionError):
    pass


def run_schedule(n_warps, n_sub, bufs, rng):
    """One random interleaving.  Each warp's program, iteration k = 0..n_sub:
    (k < n_sub) write shares of k and arrive for k; (k > 0) wait for k - 1,
    then read the shares of k - 1.  Steps are atomic; the scheduler picks any
    warp whose next step can run."""
    share = [[None] * n_warps for _ in range(bufs)]
    phase = [0, 0]      # completed phases of mbarrier 0 and 1
    arrived = [0, 0]    # arrivals counted toward the current phase
    # per warp: (iteration k, step within the iteration)
    pc = [(0, 0) for _ in range(n_warps)]

    def steps(k):
        s = []
        if k < n_sub:
            s.append("arrive")
        if k > 0:
            s += ["wait", "read"]
        return s

    def runnable(w):
        k, i = pc[w]
        if k > n_sub:
            return False
        st = steps(k)
        if i >= len(st):
            return True  # moves to the next iteration
        if st[i] == "wait":
            q = k - 1
            return phase[q % 2] > q // 2
        return True

    while True:
        ready = [w for w in range(n_warps) if runnable(w)]
        if not ready:
            if all(pc[w][0] > n_sub for w in range(n_warps)):
                return
            raise Violation("deadlock")
        w = rng.choice(ready)
        k, i = pc[w]
        st = steps(k)
        if i >= len(st):
            pc[w] = (k + 1, 0)
            continue
        op = st[i]
        if op == "arrive":
            q = k
            b = q % 2
            if phase[b] != q // 2:
                raise Violation(f"arrival for {q} while mbarrier {b} has completed {phase[b]} phases")
            share[q % bufs][w] = q
            arrived[b] += 1
            if arrived[b] == n_warps:
                arrived[b] = 0
                phase[b] += 1
        elif op == "wait":
            q = k - 1
            if phase[q % 2] > q // 2 + 1:
                raise Violation(f"wait for {q}: mbarrier two phases ahead")
        else:  # read
            q = k - 1
            got = share[q % bufs]
            if any(v != q for v in got):
                raise Violation(f"warp {w} read shares {got} for sub-panel {q}")
        pc[w] = (k, i + 1)


@pytest.mark.parametrize("n_warps", [2, 3, 14])
def test_four_share_buffers_hold_under_every_drawn_interleaving(n_warps):
    rng = random.Random(1234 + n_warps)
    for _ in range(400 if n_warps < 14 else 60):
        run_schedule(n_warps, n_sub=rng.randint(1, 12), bufs=4, rng=rng)


def test_three_share_buffers_are_caught():
    rng = random.Random(99)
    failures = 0
    for _ in range(2000):
        try:
            run_schedule(3, n_sub=10, bufs=3, rng=rng)
        except Violation:
            failures += 1
    assert failures > 0
