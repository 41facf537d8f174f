"""The backward kernels' hand-over protocol, checked on a model under random interleavings.

Each CTA of the two backward kernels has compute warps (E) and an MMA warp (M)
that hand work to each other through named barriers (`bar.arrive` by the
side handing over, `bar.sync` by the side taking over) and wait for MMA
products through mbarriers.  A named barrier completes when both sides have
arrived; if one side arrives twice before the other arrives once, the counts
mix two uses and a thread can be left waiting for good.  The mbarrier waits
are bounded: after a timeout they return at once (the degraded mode), so the
protocol must be safe by its named barriers alone.

The model replays each side's sequence of barrier operations (transcribed from
the kernels' loops, per chunk) under random schedules, with MMA completions in
issue order, in normal mode (mbarrier waits block until the product is done)
and degraded mode (they return at once), and checks that no side arrives
twice at a barrier before the other side's arrival, that no wait for a
product falls two phases behind in normal mode, and that every run ends.
The same model finds the hazard in the form with one barrier shared by all
of a chunk's compute -> MMA hand-overs.
"""
import random

import pytest


def _run(e_ops, m_ops, degraded, seed):
    rnd = random.Random(seed)
    done, mma_queue, named = {}, [], {}
    agents = {"E": e_ops, "M": m_ops}
    cur = {"E": None, "M": None}
    finished = set()
    for _ in range(100000):
        if len(finished) == 2:
            return "ok"
        choices = [a for a in agents if a not in finished] + (["mma"] if mma_queue else [])
        rnd.shuffle(choices)
        moved = False
        for c in choices:
            if c == "mma":  # the oldest product completes
                bar = mma_queue.pop(0)
                done[bar] = done.get(bar, 0) + 1
                moved = True
                break
            if cur[c] is None:
                cur[c] = next(agents[c], None)
                if cur[c] is None:
                    finished.add(c)
                    moved = True
                    break
            kind, name, *arg = cur[c]
            if kind == "wait":  # for product number arg[0] committed to mbarrier `name`
                n = done.get(name, 0)
                if not degraded and n >= arg[0] + 2:
                    return "fell two phases behind"
                if n >= arg[0] + 1 or degraded:
                    cur[c] = None
                    moved = True
                    break
                continue
            if kind == "commit":
                mma_queue.append(name)
                cur[c] = None
                moved = True
                break
            st = named.setdefault(name, {"E": False, "M": False, "gen": 0, "wait": {}})
            if c not in st["wait"]:  # arrive (and for sync: start waiting)
                if st[c]:
                    return "double arrival"
                st[c] = True
                gen = st["gen"]
                if st["E"] and st["M"]:
                    st["E"] = st["M"] = False
                    st["gen"] += 1
                if kind == "arrive":
                    cur[c] = None
                    moved = True
                    break
                st["wait"][c] = gen
            if st["gen"] > st["wait"][c]:
                del st["wait"][c]
                cur[c] = None
                moved = True
                break
        if not moved:
            return "deadlock"
    return "did not end"


def suffix_protocol(n, ids):
    em, em2, em3 = ids

    def e():
        for i in range(n):
            yield ("sync", "ME")
            yield ("wait", "PT", i)
            yield ("arrive", em)
            yield ("wait", "dPT", i)
            yield ("arrive", em2)
            yield ("wait", "dV", i)
            yield ("wait", "dK", i)
            yield ("wait", "R", i)
            yield ("arrive", em3)

    def m():
        for i in range(n):
            yield ("commit", "PT")
            yield ("arrive", "ME")
            yield ("commit", "dPT")
            yield ("sync", em)
            yield ("commit", "dV")
            yield ("sync", em2)
            yield ("commit", "dK")
            yield ("commit", "R")
            yield ("wait", "R", i)
            yield ("sync", em3)

    return e(), m()


def prefix_protocol(n, ids):
    em, em2, em3 = ids

    def e():
        for i in range(n):
            yield ("sync", "ME")
            yield ("arrive", em)       # g written
            yield ("wait", "mma", 2 * i)
            yield ("arrive", em2)      # dP packed
            yield ("wait", "mma", 2 * i + 1)
            yield ("arrive", em3)      # dQ staged, S copied

    def m():
        for i in range(n):
            if i > 0:
                yield ("wait", "rbar", i - 1)
            yield ("arrive", "ME")
            yield ("sync", em)
            yield ("commit", "mma")    # [dP | dqf]
            yield ("wait", "mma", 2 * i)
            yield ("sync", em2)
            yield ("commit", "mma")    # dqf += dP kf
            yield ("commit", "rbar")
            yield ("sync", em3)
        yield ("wait", "rbar", n - 1)

    return e(), m()


KERNEL_IDS = ("EM", "EM2", "EM3")


@pytest.mark.parametrize("protocol", [suffix_protocol, prefix_protocol])
@pytest.mark.parametrize("degraded", [False, True])
def test_protocol_is_safe_under_any_schedule(protocol, degraded):
    for n in (1, 2, 3, 5):
        for seed in range(150):
            assert _run(*protocol(n, KERNEL_IDS), degraded, seed) == "ok", (n, seed)


@pytest.mark.parametrize("protocol", [suffix_protocol, prefix_protocol])
def test_model_finds_the_hazard_of_one_shared_barrier(protocol):
    results = {_run(*protocol(n, ("EM", "EM", "EM")), True, seed) for n in (2, 3) for seed in range(300)}
    assert "double arrival" in results
