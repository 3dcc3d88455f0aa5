"""Exhaustive interleaving model of the forward attention kernel's hand-off protocol (CPU).

The kernel (csrc/attention.cu) runs five roles per CTA: a loader (work items, Q, K/V stages),
a thread issuing Q K^T, a thread issuing P V, and four softmax warps.  They meet at mbarriers
waited on by parity, and the MMAs and TMA loads complete asynchronously.  This model writes each
role's sequence of barrier operations as the kernel performs them, for a few small work lists,
and explores every interleaving of the roles' steps, the issuers' MMA / commit completions (in
order within each issuing thread, in any order between the two) and the TMA loads' completions.
It fails on:
  * a deadlock: no step possible while some role has not finished;
  * a parity wait that finds its barrier two or more phases past the awaited one (the hardware
    wait would then block until a later phase, or return for the wrong one);
  * a data hazard: S read before its Q K^T completed, P written over an S buffer whose
    previous P V has not completed, Q K^T issued into a buffer whose previous P V has not
    completed, P V issued before its values are loaded, O read before the item's P V products
    completed or overwritten before the softmax read the previous item's O, a K/V stage or Q
    buffer reloaded while an MMA that reads it has not completed.
Sub-block g uses S buffer g mod 3 and phase g // 3 of its barriers; a K/V stage holds SUBS
sub-blocks (NST stages); Q is double-buffered; the item ring has RING slots.
"""
import itertools

import pytest

SUBS, NST, NQ = 2, 2, 2


class Bar:
    def __init__(self, name, count):
        self.name, self.count = name, count


def build_programs(items, ring, warps, rescale, mutation=None):
    """The roles' action lists.  Actions:
    ('wait', bar, n)     until phase n of bar has completed (n < 0: no wait)
    ('arrive', bar)      one arrival
    ('mma', thread, key) issue an MMA (completes later, in order within the thread)
    ('commit', thread, bar)  arrive on bar once the thread's earlier MMAs have completed
    ('tma', bar, key)    start a load that arrives on bar when it completes
    ('check', kind, arg) a hazard condition on the state
    ('mark', key)        record a point a hazard condition refers to
    ``mutation`` plants one mistake in the protocol, for the tests that the model catches it."""
    bars = {}

    def bar(name, count):
        if name not in bars:
            bars[name] = Bar(name, count)
        return name

    n_items = len(items)
    g0 = list(itertools.accumulate([0] + items))[:-1]
    it_full = [bar(f"it_full{k}", 1) for k in range(ring)]
    it_empty = [bar(f"it_empty{k}", 2 + warps - (mutation == "it_empty_count")) for k in range(ring)]
    q_full = [bar(f"q_full{k}", 1) for k in range(NQ)]
    q_empty = [bar(f"q_empty{k}", 1) for k in range(NQ)]
    kv_full = [bar(f"kv_full{k}", 1) for k in range(NST)]
    kv_empty = [bar(f"kv_empty{k}", 1) for k in range(NST)]
    s_full = [bar(f"s_full{k}", 1) for k in range(3)]
    p_full = [bar(f"p_full{k}", warps) for k in range(3)]
    pv_done = [bar(f"pv_done{k}", 1) for k in range(3)]
    o_full, o_empty = bar("o_full", 1), bar("o_empty", warps)

    # stage of each sub-block, and which sub-blocks each stage fill holds
    stage_of, fills = {}, []
    st = 0
    for i, n in enumerate(items):
        for j in range((n + SUBS - 1) // SUBS):
            subs = [g0[i] + u for u in range(j * SUBS, min(n, (j + 1) * SUBS))]
            for gg in subs:
                stage_of[gg] = (st, len(fills))
            fills.append((st, subs))
            st = (st + 1) % NST

    def ring_uses(i):  # slot and use count of ring entry i (the end marker is entry n_items)
        return i % ring, i // ring

    producer = []
    fill = 0
    for i in range(n_items + 1):
        slot, use = ring_uses(i)
        producer += [("wait", it_empty[slot], use - 1), ("arrive", it_full[slot])]
        if i == n_items:
            break
        qb, quse = i % NQ, i // NQ
        producer += [("wait", q_empty[qb], quse - 1), ("check", "q_load", i), ("tma", q_full[qb], ("Q", i))]
        for j in range((items[i] + SUBS - 1) // SUBS):
            s, _ = fills[fill]
            fuse = sum(1 for f in fills[:fill] if f[0] == s)
            if mutation != "loader_skips_kv_empty":
                producer.append(("wait", kv_empty[s], fuse - 1))
            producer += [("check", "kv_load", fill), ("tma", kv_full[s], ("KV", fill))]
            fill += 1

    def issuer(qk):
        prog = []
        for i in range(n_items + 1):
            slot, use = ring_uses(i)
            prog += [("wait", it_full[slot], use), ("arrive", it_empty[slot])]
            if i == n_items:
                break
            n = items[i]
            if qk:
                prog.append(("wait", q_full[i % NQ], i // NQ))
            for u in range(n):
                gg = g0[i] + u
                b, h = gg % 3, u % SUBS
                s, f = stage_of[gg]
                fuse = sum(1 for ff in fills[:f] if ff[0] == s)
                stage_done = h == SUBS - 1 or u == n - 1
                if qk:
                    if mutation == "qk_waits_for_p_only":
                        prog.append(("wait", p_full[b], gg // 3 - 1))
                    else:
                        prog.append(("wait", pv_done[b], gg // 3 - 1))
                else:
                    prog.append(("wait", p_full[b], gg // 3))
                    if u == 0 and i > 0 and mutation != "pv_skips_o_empty":
                        prog.append(("wait", o_empty, i - 1))
                if h == 0:
                    prog.append(("wait", kv_full[s], fuse))
                if qk:
                    prog += [("check", "qk_issue", gg), ("mma", "qk", ("QK", gg)), ("commit", "qk", s_full[b])]
                    if u == n - 1:
                        prog.append(("commit", "qk", q_empty[i % NQ]))
                else:
                    prog += [("check", "pv_issue", gg), ("mma", "pv", ("PV", gg)), ("commit", "pv", pv_done[b])]
                    if stage_done:
                        prog.append(("commit", "pv", kv_empty[s]))
                    if u == n - 1:
                        prog.append(("commit", "pv", o_full))
        return prog

    def softmax(w):
        prog = []
        for i in range(n_items + 1):
            slot, use = ring_uses(i)
            prog += [("wait", it_full[slot], use), ("arrive", it_empty[slot])]
            if i == n_items:
                break
            for u in range(items[i]):
                gg = g0[i] + u
                b = gg % 3
                if mutation != "softmax_skips_s_full":
                    prog.append(("wait", s_full[b], gg // 3))
                prog.append(("check", "read_s", gg))
                if rescale and u > 0:
                    prog += [("wait", pv_done[(gg - 1) % 3], (gg - 1) // 3), ("check", "rescale", gg)]
                prog += [("check", "write_p", gg), ("arrive", p_full[b])]
            if mutation != "softmax_skips_o_full":
                prog.append(("wait", o_full, i))
            prog += [("check", "read_o", i), ("mark", ("o_read", i, w)), ("arrive", o_empty)]
        return prog

    progs = {"load": producer, "qk": issuer(True), "pv": issuer(False)}
    for w in range(warps):
        progs[f"sm{w}"] = softmax(w)
    return progs, bars, fills, g0


def explore(items, ring, warps, rescale, mutation=None, limit=3_000_000):
    """Visit every reachable state; returns their number.  Raises AssertionError on a deadlock,
    a parity wait two phases behind its barrier, or a hazard."""
    progs, bars, fills, g0 = build_programs(items, ring, warps, rescale, mutation)
    roles = sorted(progs)
    ridx = {r: k for k, r in enumerate(roles)}
    bar_names = sorted(bars)
    bidx = {n: k for k, n in enumerate(bar_names)}
    key_bar = {a[2]: a[1] for a in progs["load"] if a[0] == "tma"}
    # the issuers' queues: every mma / commit in issue order
    queue = {t: [a for a in progs[t] if a[0] in ("mma", "commit")] for t in ("qk", "pv")}
    qpos = {t: {a[2]: k for k, a in enumerate(queue[t]) if a[0] == "mma"} for t in ("qk", "pv")}
    issued_at = {t: [sum(1 for a in progs[t][:pc] if a[0] in ("mma", "commit")) for pc in range(len(progs[t]) + 1)]
                 for t in ("qk", "pv")}
    n_items = len(items)
    item_of = {gg: i for i in range(n_items) for gg in range(g0[i], g0[i] + items[i])}
    fill_of = {gg: f for f, (_, subs) in enumerate(fills) for gg in subs}
    o_read_pc = {}  # (item, warp) -> pc just after that warp's read of the item's O
    for r in roles:
        for pc, a in enumerate(progs[r]):
            if a[0] == "mark":
                o_read_pc[(a[1][1], a[1][2])] = pc + 1

    def done(comp, t, key):  # MMA `key` of thread t has completed
        return comp[0 if t == "qk" else 1] > qpos[t][key]

    def hazard_free(kind, arg, pcs, comp, loaded):
        if kind == "read_s":
            return done(comp, "qk", ("QK", arg))
        if kind in ("write_p", "qk_issue_buffer"):
            return arg < 3 or done(comp, "pv", ("PV", arg - 3))
        if kind == "qk_issue":
            i = item_of[arg]
            return ((arg < 3 or done(comp, "pv", ("PV", arg - 3))) and ("Q", i) in loaded
                    and ("KV", fill_of[arg]) in loaded)
        if kind == "rescale":
            return done(comp, "pv", ("PV", arg - 1))
        if kind == "pv_issue":
            i = item_of[arg]
            if arg == g0[i] and i > 0 and any(pcs[ridx[f"sm{w}"]] < o_read_pc[(i - 1, w)] for w in range(warps)):
                return False  # O still being read by a softmax warp
            return ("KV", fill_of[arg]) in loaded
        if kind == "read_o":
            return all(done(comp, "pv", ("PV", gg)) for gg in range(g0[arg], g0[arg] + items[arg]))
        if kind == "kv_load":
            s = fills[arg][0]
            prev = [k for k in range(arg) if fills[k][0] == s]
            return not prev or all(done(comp, "qk", ("QK", gg)) and done(comp, "pv", ("PV", gg))
                                   for gg in fills[prev[-1]][1])
        if kind == "q_load":
            return arg < NQ or all(done(comp, "qk", ("QK", gg)) for gg in range(g0[arg - NQ], g0[arg - NQ] + items[arg - NQ]))
        raise AssertionError(kind)

    def arrive(barst, name):
        b = list(barst)
        k, miss = b[bidx[name]]
        miss -= 1
        if miss == 0:
            k, miss = k + 1, bars[name].count
        b[bidx[name]] = (k, miss)
        return tuple(b)

    # state: pcs, completed MMA/commit counts (qk, pv), loads in flight, loads completed,
    # barriers as (completed phases, arrivals still missing in the current phase)
    start = (tuple(0 for _ in roles), (0, 0), frozenset(), frozenset(),
             tuple((0, bars[n].count) for n in bar_names))
    seen = {start}
    stack = [start]
    while stack:
        pcs, comp, inflight, loaded, barst = stack.pop()
        succ = []
        for ri, r in enumerate(roles):  # a role's next step
            pc = pcs[ri]
            if pc == len(progs[r]):
                continue
            a = progs[r][pc]
            npcs = pcs[:ri] + (pc + 1,) + pcs[ri + 1:]
            if a[0] == "wait":
                k = barst[bidx[a[1]]][0]
                if a[2] >= 0 and k >= a[2] + 2:
                    raise AssertionError(f"{r}: waits for phase {a[2]} of {a[1]}, which has completed {k} phases")
                if a[2] < 0 or k >= a[2] + 1:
                    succ.append((npcs, comp, inflight, loaded, barst))
            elif a[0] == "arrive":
                succ.append((npcs, comp, inflight, loaded, arrive(barst, a[1])))
            elif a[0] in ("mma", "commit", "mark"):
                succ.append((npcs, comp, inflight, loaded, barst))
            elif a[0] == "tma":
                succ.append((npcs, comp, inflight | {a[2]}, loaded, barst))
            elif a[0] == "check":
                if not hazard_free(a[1], a[2], pcs, comp, loaded):
                    raise AssertionError(f"{r}: hazard {a[1]}({a[2]})")
                succ.append((npcs, comp, inflight, loaded, barst))
            else:
                raise AssertionError(a)
        for t, ci in (("qk", 0), ("pv", 1)):  # an issuer's oldest queued MMA or commit completes
            if comp[ci] < issued_at[t][pcs[ridx[t]]]:
                e = queue[t][comp[ci]]
                ncomp = (comp[0] + (ci == 0), comp[1] + (ci == 1))
                succ.append((pcs, ncomp, inflight, loaded, arrive(barst, e[2]) if e[0] == "commit" else barst))
        for key in inflight:  # a load completes
            succ.append((pcs, comp, inflight - {key}, loaded | {key}, arrive(barst, key_bar[key])))
        if not succ:
            if all(pcs[ri] == len(progs[r]) for ri, r in enumerate(roles)):
                continue
            raise AssertionError("deadlock: " + "; ".join(
                f"{r} at {progs[r][pcs[ri]] if pcs[ri] < len(progs[r]) else 'end'}" for ri, r in enumerate(roles)))
        for nxt in succ:
            if nxt not in seen:
                seen.add(nxt)
                stack.append(nxt)
                if len(seen) > limit:
                    raise RuntimeError("state space too large for the test")
    return len(seen)


# (sub-blocks of each work item, item ring slots, softmax warps, rescale wait on every sub-block)
CONFIGS = [
    ([2, 1], 2, 1, False),
    ([3, 1], 2, 1, True),
    ([4, 1, 2], 2, 1, True),
    ([3, 2], 2, 2, False),
    ([1, 2, 1], 4, 2, True),
]


@pytest.mark.parametrize("items,ring,warps,rescale", CONFIGS)
def test_protocol_has_no_deadlock_aliasing_or_hazard(items, ring, warps, rescale):
    assert explore(items, ring, warps, rescale) > 1000


@pytest.mark.parametrize("mutation,items,warps", [
    ("qk_waits_for_p_only", [4, 2], 1),      # Q K^T overwrites S/P before P V read P
    ("softmax_skips_s_full", [2, 1], 1),     # S read before Q K^T completed
    ("softmax_skips_o_full", [2, 1], 1),     # O read before the item's P V products completed
    ("loader_skips_kv_empty", [3, 2, 1], 1),  # a K/V stage reloaded under its MMAs
    ("it_empty_count", [1, 1, 1], 2),        # the ring slot refilled before every role read it
])
def test_the_model_catches_a_planted_mistake(mutation, items, warps):
    with pytest.raises(AssertionError):
        explore(items, 2, warps, False, mutation)


@pytest.mark.parametrize("warps", [1, 2])
def test_the_pv_threads_o_empty_wait_is_implied(warps):
    # P V of an item's first sub-block waits for P of that sub-block from every softmax warp,
    # and a warp writes it only after reading the previous item's O: without the o_empty wait
    # nothing changes
    explore([1, 2, 1], 2, warps, True, "pv_skips_o_empty")
