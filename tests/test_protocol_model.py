"""Model check of the barrier protocol of the warp-specialised attention kernel.

The kernel in ``csrc/attn_ws.cuh`` runs five roles per CTA (TMA producer, rotary warps,
MMA issuer, two softmax warpgroups) that hand buffers to one another through mbarriers.
This test restates each role's sequence of barrier waits and arrivals as a generator and
runs them under many random interleavings, with the hardware's parity-wait semantics: a
wait for completion number ``need`` passes as soon as the completion count ``c`` has the
same parity, so a pass with ``c != need`` (a waiter two phases behind, or one that skipped
a phase) is a protocol error, as is a state where no role can move (a deadlock).

It covers every ring depth the host may pick (1..4 K slots, 1..4 V slots) and unit lists
with and without a second query tile.  Single-slot rings are the sensitive case: moving
the K/V readiness checks from the MMA issuer into the softmax warps, for instance, makes
the keeper wait for a V tile that the producer only loads after a K slot that the keeper
itself would release, and this model reports that as a deadlock.
"""
import random

import pytest


def units_for(S, ts):
    """(n0, n1, nkv) of the units with query-tile pairs ts, as the kernel decodes them."""
    out = []
    for t in ts:
        n0 = 2 * t + 1
        n1 = 2 * t + 2 if (2 * t + 1) * 128 < S else 0
        out.append((n0, n1, max(n0, n1)))
    return out


def roles(units, NK, NV):
    def producer():
        ks = vs = 0
        kuse, vuse = [0] * NK, [0] * NV
        for ul, (n0, n1, nkv) in enumerate(units):
            # K_0 of the unit first: its slot frees before the previous unit's last S
            yield ("wait", f"K_EMPTY{ks}", kuse[ks])
            kuse[ks] += 1
            yield ("arrive", f"K_FULL{ks}")
            ks = (ks + 1) % NK
            yield ("wait", "Q_EMPTY", ul)
            yield ("arrive", "Q_FULL")
            for j in range(1, nkv + 1):  # K_j before V_{j-1}
                if j < nkv:
                    yield ("wait", f"K_EMPTY{ks}", kuse[ks])
                    kuse[ks] += 1
                    yield ("arrive", f"K_FULL{ks}")
                    ks = (ks + 1) % NK
                if j >= 1:
                    yield ("wait", f"V_EMPTY{vs}", vuse[vs])
                    vuse[vs] += 1
                    yield ("arrive", f"V_FULL{vs}")
                    vs = (vs + 1) % NV

    def rotary():
        ks = 0
        kuse = [0] * NK
        for ul, (n0, n1, nkv) in enumerate(units):
            # the producer's order: K_0, the query tiles, then K_1 ...
            items = ["K"] + ["Q"] + ["K"] * (nkv - 1)
            for item in items:
                if item == "Q":
                    yield ("wait", "Q_FULL", ul + 1)
                    yield ("arrive", "Q_READY0")
                    if n1:
                        yield ("arrive", "Q_READY1")
                    continue
                kuse[ks] += 1
                yield ("wait", f"K_FULL{ks}", kuse[ks])
                yield ("arrive", f"K_READY{ks}")
                ks = (ks + 1) % NK

    def mma():
        ks = vs = 0
        kuse, vuse = [0] * NK, [0] * NV
        p_cnt, q_cnt = [0, 0], [0, 0]
        for ul, (n0, n1, nkv) in enumerate(units):
            for j in range(nkv + 1):
                if j < nkv:
                    yield ("wait", f"K_READY{ks}", kuse[ks] + 1)
                if j >= 1:
                    yield ("wait", f"V_FULL{vs}", vuse[vs] + 1)
                for tau, n in enumerate((n0, n1)):
                    if n == 0:
                        continue
                    if 1 <= j <= n:  # PV_tau(j-1) after P_tau(j-1)
                        p_cnt[tau] += 1
                        yield ("wait", f"P_FULL{tau}", p_cnt[tau])
                        if j == n:
                            yield ("arrive", f"O_FINAL{tau}")
                    if j < n:  # S_tau(j)
                        if j == 0:
                            q_cnt[tau] += 1
                            yield ("wait", f"Q_READY{tau}", q_cnt[tau])
                        yield ("arrive", f"S_FULL{tau}")
                if j < nkv:
                    yield ("arrive", f"K_EMPTY{ks}")
                    kuse[ks] += 1
                    ks = (ks + 1) % NK
                if j >= 1:
                    yield ("arrive", f"V_EMPTY{vs}")
                    vuse[vs] += 1
                    vs = (vs + 1) % NV
                if j == nkv - 1:
                    yield ("arrive", "Q_EMPTY")

    def softmax(tau):
        s_use = o_use = 0
        for n0, n1, nkv in units:
            n = n0 if tau == 0 else n1
            if n == 0:
                continue
            for j in range(n):
                s_use += 1
                yield ("wait", f"S_FULL{tau}", s_use)
                yield ("arrive", f"P_FULL{tau}")
            o_use += 1
            yield ("wait", f"O_FINAL{tau}", o_use)

    return {"producer": producer(), "rotary": rotary(), "mma": mma(),
            "softmax0": softmax(0), "softmax1": softmax(1)}


def run_roles(gens, seed):
    """Runs the roles to completion under one random schedule; returns None or the error."""
    rng = random.Random(seed)
    cur = {k: next(g, None) for k, g in gens.items()}
    done = {}
    while True:
        live = [k for k, op in cur.items() if op is not None]
        if not live:
            return None
        ready = []
        for k in live:
            op = cur[k]
            if op[0] == "wait":
                c = done.get(op[1], 0)
                if (c - op[2]) % 2 == 0:  # the parity wait passes
                    if c != op[2]:
                        return f"{k} passes {op[1]} for completion {op[2]} at count {c}"
                    ready.append(k)
            else:
                ready.append(k)
        if not ready:
            return "deadlock: " + ", ".join(f"{k} at {cur[k]}" for k in live)
        k = rng.choice(ready)
        if cur[k][0] == "arrive":
            done[cur[k][1]] = done.get(cur[k][1], 0) + 1
        cur[k] = next(gens[k], None)


@pytest.mark.parametrize("NK", [1, 2, 3, 4])
@pytest.mark.parametrize("NV", [1, 2, 3, 4])
def test_protocol_has_no_deadlock_or_phase_alias(NK, NV):
    rng = random.Random(100 * NK + NV)
    for S in (128, 129, 200, 256, 300, 384, 650, 1100, 2048):
        T = (S + 255) // 256
        mixes = [list(range(T - 1, -1, -1)), [T - 1] * 3, [0, 0, T - 1, 0]]
        mixes += [[rng.randrange(T) for _ in range(rng.randint(1, 5))] for _ in range(3)]
        for ts in mixes:
            for seed in range(12):
                err = run_roles(roles(units_for(S, ts), NK, NV), seed)
                assert err is None, (S, ts, NK, NV, seed, err)


def test_model_catches_a_skipped_phase():
    # A consumer that waits only on every second phase of a single-slot ring must be
    # flagged: the parity wait cannot tell "two more phases done" from "none".
    def gens():
        def prod():
            for i in range(4):
                yield ("wait", "EMPTY", i)
                yield ("arrive", "FULL")

        def cons():
            for i in range(0, 4, 2):
                yield ("wait", "FULL", i + 1)
                yield ("arrive", "EMPTY")
                yield ("arrive", "EMPTY")
        return {"producer": prod(), "consumer": cons()}

    assert any(run_roles(gens(), seed) is not None for seed in range(20))
