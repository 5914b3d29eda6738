"""Model check of the barrier protocol of the persistent decode kernel (csrc/decode.cuh).

The producer warp and the 8 consumer warps of a CTA hand over ring stages (a K+V tile
pair each) and two item slots (a work item's new-token row) through mbarriers, and the
consumers meet at one named barrier per item.  This test restates each warp's sequence of
waits and arrivals as a generator, for every ring depth the kernel uses (3, 4, 6) and
random item/tile layouts (including items with no tile), and runs them under many random
interleavings with the hardware's parity-wait semantics: an mbarrier with arrival count c
completes a phase every c arrivals, and a wait for completion number `need` passes as soon
as the completion count has the same parity, so a pass at a count other than `need` (a
waiter that skipped or fell behind a phase) is a protocol error, as is a state in which no
warp can move.
"""
import random

import pytest

CONSUMERS = 8


def roles(items, S):
    """items: tiles per work item of one CTA, in order."""
    def producer():
        n = 0
        for k, tiles in enumerate(items):
            slot = k & 1
            yield ("wait", f"qempty{slot}", k >> 1)  # slot free (the previous user released it)
            yield ("arrive", f"qfull{slot}")          # new-token row and position published
            for _ in range(tiles):
                s = n % S
                yield ("wait", f"empty{s}", n // S)
                yield ("arrive", f"full{s}")           # K and V tile landed
                n += 1

    def consumer():
        n = 0
        for k, tiles in enumerate(items):
            slot = k & 1
            yield ("wait", f"qfull{slot}", (k >> 1) + 1)
            for _ in range(tiles):
                s = n % S
                yield ("wait", f"full{s}", n // S + 1)
                yield ("arrive", f"empty{s}")
                n += 1
            yield ("arrive", f"qempty{slot}")
            yield ("arrive", "merge")                   # the named barrier of the item merge
            yield ("wait", "merge", k + 1)

    gens = {"producer": producer()}
    for c in range(CONSUMERS):
        gens[f"consumer{c}"] = consumer()
    return gens


COUNTS = {"qfull": 1, "full": 1, "qempty": CONSUMERS, "empty": CONSUMERS, "merge": CONSUMERS}


def count_of(bar):
    return COUNTS[bar.rstrip("0123456789")]


def run(gens, seed):
    rng = random.Random(seed)
    cur = {k: next(g, None) for k, g in gens.items()}
    arrivals = {}
    while True:
        live = [k for k, op in cur.items() if op is not None]
        if not live:
            return None
        ready = []
        for k in live:
            op = cur[k]
            if op[0] == "wait":
                done = arrivals.get(op[1], 0) // count_of(op[1])
                if op[1] == "merge":  # bar.sync counts arrivals itself: no parity aliasing
                    if done >= op[2]:
                        ready.append(k)
                elif (done - op[2]) % 2 == 0:
                    if done != op[2]:
                        return f"{k} passes {op[1]} for completion {op[2]} at completion {done}"
                    ready.append(k)
            else:
                ready.append(k)
        if not ready:
            return "deadlock: " + ", ".join(f"{k} at {cur[k]}" for k in live)
        k = rng.choice(ready)
        if cur[k][0] == "arrive":
            arrivals[cur[k][1]] = arrivals.get(cur[k][1], 0) + 1
        cur[k] = next(gens[k], None)


@pytest.mark.parametrize("S", [3, 4, 6])
def test_decode_protocol_has_no_deadlock_or_phase_alias(S):
    rng = random.Random(S)
    layouts = [[16] * 7, [1] * 9, [0, 3, 0, 0, 5], [2, 17, 1], [S, S, S, S], [S + 1, S - 1, 1, 0]]
    layouts += [[rng.randint(0, 20) for _ in range(rng.randint(1, 8))] for _ in range(8)]
    for items in layouts:
        for seed in range(10):
            err = run(roles(items, S), seed)
            assert err is None, (S, items, seed, err)


def test_model_catches_a_consumer_that_skips_the_slot_release():
    # consumers that never release an item slot: the producer's third item must wait forever
    def broken(items, S):
        gens = roles(items, S)

        def consumer():
            n = 0
            for k, tiles in enumerate(items):
                slot = k & 1
                yield ("wait", f"qfull{slot}", (k >> 1) + 1)
                for _ in range(tiles):
                    s = n % S
                    yield ("wait", f"full{s}", n // S + 1)
                    yield ("arrive", f"empty{s}")
                    n += 1
        for c in range(CONSUMERS):
            gens[f"consumer{c}"] = consumer()
        return gens

    assert run(broken([1, 1, 1], 4), 0).startswith("deadlock")


def test_model_catches_a_ring_deeper_than_the_waits_assume():
    # a producer that runs two laps ahead (no wait on empty) overwrites a stage the
    # consumers have not read: the consumers then see a completion they did not expect
    def eager(items, S):
        gens = roles(items, S)

        def producer():
            for k, tiles in enumerate(items):
                slot = k & 1
                yield ("wait", f"qempty{slot}", k >> 1)
                yield ("arrive", f"qfull{slot}")
                for t in range(tiles):
                    yield ("arrive", f"full{t % S}")
        gens["producer"] = producer()
        return gens

    assert any(run(eager([3 * 4], 4), seed) is not None for seed in range(20))
