"""Exhaustive interleaving models of the kernels' hand-off protocols (CPU): the forward
attention kernel first, then the backward dQ and dK/dV kernels, the projection GEMM, the fused
post-attention chain and the whole-stack kernel.

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


def run_model(progs, bars, key_bar, issuers, hazard_free, limit=3_000_000):
    """Visit every reachable state of the roles ``progs`` (name -> action list); returns their
    number.  ``issuers`` are the roles whose mma / commit actions queue up and complete in order;
    ``key_bar`` maps a load to the barrier it arrives on; ``hazard_free(kind, arg, pcs, comp,
    loaded)`` evaluates a check action (pcs by role name, comp: completed queue entries by
    issuer, loaded: the completed loads).  Raises AssertionError on a deadlock, a parity wait two
    phases behind its barrier, or a hazard."""
    roles = sorted(progs)
    ridx = {r: k for k, r in enumerate(roles)}
    bar_names = sorted(bars)
    bidx = {n: k for k, n in enumerate(bar_names)}
    queue = {t: [a for a in progs[t] if a[0] in ("mma", "commit")] for t in issuers}
    issued_at = {t: [sum(1 for a in progs[t][:pc] if a[0] in ("mma", "commit")) for pc in range(len(progs[t]) + 1)]
                 for t in issuers}

    def arrive(barst, name):
        b = list(barst)
        k, miss = b[bidx[name]]
        miss -= 1
        if miss == 0:
            k, miss = k + 1, bars[name].count
        b[bidx[name]] = (k, miss)
        return tuple(b)

    # state: pcs, completed queue entries per issuer, loads in flight, loads completed,
    # barriers as (completed phases, arrivals still missing in the current phase)
    start = (tuple(0 for _ in roles), tuple(0 for _ in issuers), frozenset(), frozenset(),
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
                if not hazard_free(a[1], a[2], dict(zip(roles, pcs)), dict(zip(issuers, comp)), loaded):
                    raise AssertionError(f"{r}: hazard {a[1]}({a[2]})")
                succ.append((npcs, comp, inflight, loaded, barst))
            else:
                raise AssertionError(a)
        for ci, t in enumerate(issuers):  # an issuer's oldest queued MMA or commit completes
            if comp[ci] < issued_at[t][pcs[ridx[t]]]:
                e = queue[t][comp[ci]]
                ncomp = comp[:ci] + (comp[ci] + 1,) + comp[ci + 1:]
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


def mark_pcs(progs):
    """(mark key) -> (role, pc just after the mark)."""
    return {a[1]: (r, pc + 1) for r in progs for pc, a in enumerate(progs[r]) if a[0] == "mark"}


def explore(items, ring, warps, rescale, mutation=None):
    """The forward kernel's protocol on the work list ``items`` (sub-blocks per item)."""
    progs, bars, fills, g0 = build_programs(items, ring, warps, rescale, mutation)
    key_bar = {a[2]: a[1] for a in progs["load"] if a[0] == "tma"}
    qpos = {t: {a[2]: k for k, a in enumerate([a for a in progs[t] if a[0] in ("mma", "commit")]) if a[0] == "mma"}
            for t in ("qk", "pv")}
    n_items = len(items)
    item_of = {gg: i for i in range(n_items) for gg in range(g0[i], g0[i] + items[i])}
    fill_of = {gg: f for f, (_, subs) in enumerate(fills) for gg in subs}
    marks = mark_pcs(progs)

    def done(comp, t, key):  # MMA `key` of thread t has completed
        return comp[t] > qpos[t][key]

    def hazard_free(kind, arg, pcs, comp, loaded):
        if kind == "read_s":
            return done(comp, "qk", ("QK", arg))
        if kind == "write_p":
            return arg < 3 or done(comp, "pv", ("PV", arg - 3))
        if kind == "qk_issue":
            return ((arg < 3 or done(comp, "pv", ("PV", arg - 3))) and ("Q", item_of[arg]) in loaded
                    and ("KV", fill_of[arg]) in loaded)
        if kind == "rescale":
            return done(comp, "pv", ("PV", arg - 1))
        if kind == "pv_issue":
            i = item_of[arg]
            if arg == g0[i] and i > 0:
                for w in range(warps):
                    r, pc = marks[("o_read", i - 1, w)]
                    if pcs[r] < pc:
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
            return arg < NQ or all(done(comp, "qk", ("QK", gg))
                                   for gg in range(g0[arg - NQ], g0[arg - NQ] + items[arg - NQ]))
        raise AssertionError(kind)

    return run_model(progs, bars, key_bar, ["qk", "pv"], hazard_free)


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


# ---------------------------------------------------------------------------------------------
# The backward dQ kernel (csrc/attention_bwd.cu, dQ mode): a loader (resident Q and dO per work
# item, K_j / V_j tiles per 64-key step into a ring of BWD_NST stages), one MMA-issuing thread and
# the elementwise warps.  Step s of an item computes S into S buffer s mod 2 (counted from the
# item's first step) as soon as its tiles are in, dP into the single dP buffer once the warps hold
# the previous step's dP in registers (dp_read), releases the step to the warps (s_full) only
# after the previous step's dS is written (x_full), then accumulates dQ += dS K of the previous
# step.  The warps read S and dP, arrive on dp_read, write dS over S, arrive on x_full, and read
# out the accumulator at the end of the item (acc_full / acc_empty).
BWD_NST = 3


def build_dq(items, warps, mutation=None):
    bars = {}

    def bar(name, count):
        bars[name] = Bar(name, count)
        return name

    res_full, res_empty = bar("res_full", 1), bar("res_empty", 1)
    s_full, x_full, dp_read = bar("s_full", 1), bar("x_full", warps), bar("dp_read", warps)
    acc_full, acc_empty = bar("acc_full", 1), bar("acc_empty", warps)
    b_full = [bar(f"b_full{k}", 1) for k in range(BWD_NST)]
    b_empty = [bar(f"b_empty{k}", 1) for k in range(BWD_NST)]
    t0 = list(itertools.accumulate([0] + items))[:-1]  # global index of each item's first step
    buf = {t0[i] + s: s % 2 for i in range(len(items)) for s in range(items[i])}

    load = []
    for i, n in enumerate(items):
        load += [("wait", res_empty, i - 1), ("check", "res_load", i), ("tma", res_full, ("R", i))]
        for s in range(n):
            t = t0[i] + s
            load += [("wait", b_empty[t % BWD_NST], t // BWD_NST - 1), ("check", "stage_load", t),
                     ("tma", b_full[t % BWD_NST], ("B", t))]

    mma = []
    for i, n in enumerate(items):
        mma.append(("wait", res_full, i))
        if i > 0:
            mma.append(("wait", acc_empty, i - 1))
        for s in range(n + 1):
            t = t0[i] + s
            if s < n:
                mma += [("wait", b_full[t % BWD_NST], t // BWD_NST), ("check", "s_issue", t), ("mma", "mma", ("S", t))]
                if s > 0:
                    mma.append(("wait", dp_read, t - 1))
                mma += [("check", "dp_issue", t), ("mma", "mma", ("DP", t))]
            elif s > 0:
                mma.append(("wait", dp_read, t - 1))
            if s > 0 and mutation != "s_full_before_x_full":
                mma.append(("wait", x_full, t - 1))
            if s < n:
                mma.append(("commit", "mma", s_full))
            if s > 0 and mutation == "s_full_before_x_full":
                mma.append(("wait", x_full, t - 1))
            if s > 0:
                mma += [("check", "acc_issue", t - 1), ("mma", "mma", ("ACC", t - 1)),
                        ("commit", "mma", b_empty[(t - 1) % BWD_NST])]
        mma += [("commit", "mma", res_empty), ("commit", "mma", acc_full)]

    def elementwise(w):
        prog = []
        for i, n in enumerate(items):
            for s in range(n):
                t = t0[i] + s
                # S (first half) and all of dP are loaded, then dp_read; S's second half is
                # loaded and dS written over S after it
                prog.append(("wait", s_full, t))
                if mutation == "dp_read_before_load":
                    prog.append(("arrive", dp_read))
                prog += [("check", "ew_read", t), ("mark", ("dp_read", t, w))]
                if mutation != "dp_read_before_load":
                    prog.append(("arrive", dp_read))
                prog += [("check", "ew_write", t), ("mark", ("x", t, w)), ("arrive", x_full)]
            prog += [("wait", acc_full, i), ("check", "acc_read", i), ("mark", ("acc_read", i, w)), ("arrive", acc_empty)]
        return prog

    progs = {"load": load, "mma": mma}
    for w in range(warps):
        progs[f"ew{w}"] = elementwise(w)
    return progs, bars, t0, buf


def explore_dq(items, warps, mutation=None):
    """The dQ kernel's protocol on the work list ``items`` (steps per item)."""
    progs, bars, t0, buf = build_dq(items, warps, mutation)
    key_bar = {a[2]: a[1] for a in progs["load"] if a[0] == "tma"}
    entries = [a for a in progs["mma"] if a[0] in ("mma", "commit")]
    qpos = {a[2]: k for k, a in enumerate(entries) if a[0] == "mma"}
    mma_pc = {a[2]: pc for pc, a in enumerate(progs["mma"]) if a[0] == "mma"}
    marks = mark_pcs(progs)
    n_steps = sum(items)
    item_of = {t0[i] + s: i for i in range(len(items)) for s in range(items[i])}

    def done(comp, key):
        return comp["mma"] > qpos[key]

    def issued(pcs, key):
        return pcs["mma"] > mma_pc[key]

    def passed(pcs, key):  # every warp is past the mark
        return all(pcs[r] >= pc for (k, r, pc) in ((k, *marks[k]) for k in marks)
                   if k[0] == key[0] and k[1:-1] == key[1:])

    def prev_user(t):  # the previous step that used t's S buffer
        return max((u for u in range(t) if buf[u] == buf[t]), default=None)

    def next_user(t):
        return min((u for u in range(t + 1, n_steps) if buf[u] == buf[t]), default=None)

    def hazard_free(kind, arg, pcs, comp, loaded):
        if kind == "s_issue":  # S buffer: the warps are done with its previous step
            u = prev_user(arg)
            return ("B", arg) in loaded and ("R", item_of[arg]) in loaded and (
                u is None or (passed(pcs, ("x", u)) and issued(pcs, ("ACC", u))))
        if kind == "dp_issue":  # the dP buffer: every warp holds the previous step's dP
            return arg == 0 or passed(pcs, ("dp_read", arg - 1))
        if kind == "ew_read":
            nu = next_user(arg)
            return (done(comp, ("S", arg)) and done(comp, ("DP", arg))
                    and (nu is None or not issued(pcs, ("S", nu)))
                    and (arg + 1 >= n_steps or not issued(pcs, ("DP", arg + 1))))
        if kind == "ew_write":
            nu = next_user(arg)
            return nu is None or not issued(pcs, ("S", nu))
        if kind == "acc_issue":  # dS written by every warp; a new item's accumulator read out
            i = item_of[arg]
            if arg == t0[i] and i > 0 and not passed(pcs, ("acc_read", i - 1)):
                return False
            return passed(pcs, ("x", arg))
        if kind == "acc_read":
            return all(done(comp, ("ACC", t)) for t in range(t0[arg], t0[arg] + items[arg]))
        if kind == "stage_load":
            u = arg - BWD_NST
            return u < 0 or all(done(comp, (k, u)) for k in ("S", "DP", "ACC"))
        if kind == "res_load":
            return arg == 0 or all(done(comp, (k, t)) for k in ("S", "DP")
                                   for t in range(t0[arg - 1], t0[arg - 1] + items[arg - 1]))
        raise AssertionError(kind)

    return run_model(progs, bars, key_bar, ["mma"], hazard_free)


@pytest.mark.parametrize("items,warps", [([3], 1), ([2, 1], 1), ([1, 3], 2), ([2, 2], 2), ([4, 1, 2], 1)])
def test_dq_protocol_has_no_deadlock_aliasing_or_hazard(items, warps):
    assert explore_dq(items, warps) > 100


@pytest.mark.parametrize("mutation,items,warps", [
    # step s released before the warps' dS of step s - 1 is seen: one warp runs a step ahead,
    # and x_full's phase completes on its two arrivals (two warps), or wraps (one warp)
    ("s_full_before_x_full", [4], 2),
    ("s_full_before_x_full", [4], 1),
    ("dp_read_before_load", [3], 1),    # dP overwritten before the warps hold it
])
def test_the_dq_model_catches_a_planted_mistake(mutation, items, warps):
    with pytest.raises(AssertionError):
        explore_dq(items, warps, mutation)


# ---------------------------------------------------------------------------------------------
# The backward dK/dV kernel (csrc/attention_bwd.cu, dK/dV mode): resident K and V per work item,
# Q_j / dO_j tiles per 64-query step in a ring of DKV_NST stages, one MMA-issuing thread, the
# elementwise warps.  Each step: the warps stage the step's log-sum-exp and row sums in one of two
# shared buffers (each warp writes part, every warp reads all of it) and meet at a named barrier
# before reading; the MMA thread computes S^T and dP^T of step s into
# the single S and dP buffers after the previous step's accumulating MMAs (dV += P^T dO,
# dK += dS^T Q), which it issues once the warps have written P^T and dS^T over S and dP (x_full).
DKV_NST = 2


def build_dkv(items, warps, mutation=None):
    bars = {}

    def bar(name, count):
        bars[name] = Bar(name, count)
        return name

    res_full, res_empty = bar("res_full", 1), bar("res_empty", 1)
    s_full, x_full = bar("s_full", 1), bar("x_full", warps)
    acc_full, acc_empty = bar("acc_full", 1), bar("acc_empty", warps)
    ebar = bar("elem_bar", warps)  # the named barrier, arrive-and-wait
    b_full = [bar(f"b_full{k}", 1) for k in range(DKV_NST)]
    b_empty = [bar(f"b_empty{k}", 1) for k in range(DKV_NST)]
    t0 = list(itertools.accumulate([0] + items))[:-1]

    load = []
    for i, n in enumerate(items):
        load += [("wait", res_empty, i - 1), ("check", "res_load", i), ("tma", res_full, ("R", i))]
        for s in range(n):
            t = t0[i] + s
            load += [("wait", b_empty[t % DKV_NST], t // DKV_NST - 1), ("check", "stage_load", t),
                     ("tma", b_full[t % DKV_NST], ("B", t))]

    mma = []
    for i, n in enumerate(items):
        mma.append(("wait", res_full, i))
        if i > 0:
            mma.append(("wait", acc_empty, i - 1))
        for s in range(n + 1):
            t = t0[i] + s
            if s < n:
                mma.append(("wait", b_full[t % DKV_NST], t // DKV_NST))
            step = [("check", "s_issue", t), ("mma", "mma", ("S", t)), ("commit", "mma", s_full)] if s < n else []
            if mutation == "s_before_acc":
                mma += step
            if s > 0:
                mma += [("wait", x_full, t - 1), ("check", "acc_issue", t - 1), ("mma", "mma", ("ACC", t - 1)),
                        ("commit", "mma", b_empty[(t - 1) % DKV_NST])]
            if mutation != "s_before_acc":
                mma += step
        mma += [("commit", "mma", res_empty), ("commit", "mma", acc_full)]

    def elementwise(w):
        prog = []
        for i, n in enumerate(items):
            for s in range(n):
                t = t0[i] + s
                # each warp stages its part of the step's values, which every warp then reads
                prog += [("check", "sf_write", t), ("mark", ("sfw", t, w))]
                if mutation != "no_named_barrier":
                    prog += [("arrive", ebar), ("wait", ebar, t)]
                prog += [("wait", s_full, t), ("check", "ew_read", t), ("mark", ("sf", t, w)),
                         ("mark", ("x", t, w)), ("arrive", x_full)]
            prog += [("wait", acc_full, i), ("check", "acc_read", i), ("mark", ("acc_read", i, w)), ("arrive", acc_empty)]
        return prog

    progs = {"load": load, "mma": mma}
    for w in range(warps):
        progs[f"ew{w}"] = elementwise(w)
    return progs, bars, t0


def explore_dkv(items, warps, mutation=None):
    """The dK/dV kernel's protocol on the work list ``items`` (steps per item)."""
    progs, bars, t0 = build_dkv(items, warps, mutation)
    key_bar = {a[2]: a[1] for a in progs["load"] if a[0] == "tma"}
    entries = [a for a in progs["mma"] if a[0] in ("mma", "commit")]
    qpos = {a[2]: k for k, a in enumerate(entries) if a[0] == "mma"}
    mma_pc = {a[2]: pc for pc, a in enumerate(progs["mma"]) if a[0] == "mma"}
    marks = mark_pcs(progs)
    item_of = {t0[i] + s: i for i in range(len(items)) for s in range(items[i])}

    def done(comp, key):
        return comp["mma"] > qpos[key]

    def issued(pcs, key):
        return pcs["mma"] > mma_pc[key]

    def passed(pcs, key):
        return all(pcs[r] >= pc for k, (r, pc) in marks.items() if k[0] == key[0] and k[1:-1] == key[1:])

    def hazard_free(kind, arg, pcs, comp, loaded):
        if kind == "s_issue":  # S and dP hold P^T, dS^T of the previous step until its MMAs read them
            return (("B", arg) in loaded and ("R", item_of[arg]) in loaded
                    and (arg == 0 or (passed(pcs, ("x", arg - 1)) and issued(pcs, ("ACC", arg - 1)))))
        if kind == "ew_read":  # S and dP computed and not yet overwritten; every warp's staging written
            nxt = ("S", arg + 1)
            return (done(comp, ("S", arg)) and (nxt not in mma_pc or not issued(pcs, nxt))
                    and passed(pcs, ("sfw", arg)))
        if kind == "acc_issue":
            i = item_of[arg]
            if arg == t0[i] and i > 0 and not passed(pcs, ("acc_read", i - 1)):
                return False
            return passed(pcs, ("x", arg))
        if kind == "acc_read":
            return all(done(comp, ("ACC", t)) for t in range(t0[arg], t0[arg] + items[arg]))
        if kind == "stage_load":
            u = arg - DKV_NST
            return u < 0 or (done(comp, ("S", u)) and done(comp, ("ACC", u)))
        if kind == "res_load":
            return arg == 0 or all(done(comp, ("S", t)) for t in range(t0[arg - 1], t0[arg - 1] + items[arg - 1]))
        if kind == "sf_write":  # staging buffer t mod 2: every warp is done with step t - 2
            return arg < 2 or passed(pcs, ("sf", arg - 2))
        raise AssertionError(kind)

    return run_model(progs, bars, key_bar, ["mma"], hazard_free)


@pytest.mark.parametrize("items,warps", [([3], 1), ([2, 1], 2), ([1, 3], 2), ([4, 1, 2], 1)])
def test_dkv_protocol_has_no_deadlock_aliasing_or_hazard(items, warps):
    assert explore_dkv(items, warps) > 100


@pytest.mark.parametrize("mutation,items,warps", [
    ("s_before_acc", [3], 1),        # S^T overwrites P^T before dV += P^T dO has read it
    ("no_named_barrier", [3], 2),    # a warp reads the step's staged values before another wrote its part
])
def test_the_dkv_model_catches_a_planted_mistake(mutation, items, warps):
    with pytest.raises(AssertionError):
        explore_dkv(items, warps, mutation)


# ---------------------------------------------------------------------------------------------
# The projection GEMM (csrc/gemm.cu): a loader filling a ring of GEMM_STAGES k-block stages, one
# MMA-issuing thread accumulating each tile's k-blocks into one of two tensor-memory
# accumulators, and the epilogue warps reading a finished accumulator.  Per tile the MMA thread
# waits until the epilogue has read the accumulator's previous tile (acce), then for each
# k-block waits for the stage (full), issues, and frees the stage (commit empty); it commits accf
# after the last k-block.  The epilogue warps wait accf, read, and arrive on acce.
GEMM_STAGES = 3


def build_gemm(tiles, num_k, warps, mutation=None):
    bars = {}

    def bar(name, count):
        bars[name] = Bar(name, count)
        return name

    full = [bar(f"full{k}", 1) for k in range(GEMM_STAGES)]
    empty = [bar(f"empty{k}", 1) for k in range(GEMM_STAGES)]
    accf = [bar(f"accf{k}", 1) for k in range(2)]
    acce = [bar(f"acce{k}", warps) for k in range(2)]
    load, mma = [], []
    j = 0  # k-block load index over the CTA's tiles
    for t in range(tiles):
        for kb in range(num_k):
            load += [("wait", empty[j % GEMM_STAGES], j // GEMM_STAGES - 1), ("check", "stage_load", j),
                     ("tma", full[j % GEMM_STAGES], ("K", j))]
            j += 1
    j = 0
    for t in range(tiles):
        a = t % 2
        if mutation != "mma_skips_acce":
            mma.append(("wait", acce[a], t // 2 - 1))
        for kb in range(num_k):
            s = j % GEMM_STAGES
            mma.append(("wait", full[s], j // GEMM_STAGES))
            if mutation == "empty_before_mma":
                mma.append(("commit", "mma", empty[s]))
            mma += [("check", "mma_issue", (t, kb, j)), ("mma", "mma", ("M", j))]
            if mutation != "empty_before_mma":
                mma.append(("commit", "mma", empty[s]))
            j += 1
        mma.append(("commit", "mma", accf[a]))

    def epilogue(w):
        prog = []
        for t in range(tiles):
            prog += [("wait", accf[t % 2], t // 2), ("check", "acc_read", t), ("mark", ("acc_read", t, w)),
                     ("arrive", acce[t % 2])]
        return prog

    progs = {"load": load, "mma": mma}
    for w in range(warps):
        progs[f"epi{w}"] = epilogue(w)
    return progs, bars


def explore_gemm(tiles, num_k, warps, mutation=None):
    """The GEMM's protocol for ``tiles`` tiles of ``num_k`` k-blocks on one CTA."""
    progs, bars = build_gemm(tiles, num_k, warps, mutation)
    key_bar = {a[2]: a[1] for a in progs["load"] if a[0] == "tma"}
    entries = [a for a in progs["mma"] if a[0] in ("mma", "commit")]
    qpos = {a[2]: k for k, a in enumerate(entries) if a[0] == "mma"}
    marks = mark_pcs(progs)

    def done(comp, key):
        return comp["mma"] > qpos[key]

    def passed(pcs, key):
        return all(pcs[r] >= pc for k, (r, pc) in marks.items() if k[0] == key[0] and k[1:-1] == key[1:])

    def hazard_free(kind, arg, pcs, comp, loaded):
        if kind == "stage_load":  # the stage's previous k-block has been read by its MMAs
            return arg < GEMM_STAGES or done(comp, ("M", arg - GEMM_STAGES))
        if kind == "mma_issue":  # operands loaded; the first k-block overwrites the accumulator
            t, kb, j = arg
            if ("K", j) not in loaded:
                return False
            return kb > 0 or t < 2 or passed(pcs, ("acc_read", t - 2))
        if kind == "acc_read":
            return all(done(comp, ("M", arg * num_k + kb)) for kb in range(num_k))
        raise AssertionError(kind)

    return run_model(progs, bars, key_bar, ["mma"], hazard_free)


@pytest.mark.parametrize("tiles,num_k,warps", [(3, 2, 1), (4, 1, 2), (2, 4, 2), (5, 2, 1)])
def test_gemm_protocol_has_no_deadlock_aliasing_or_hazard(tiles, num_k, warps):
    assert explore_gemm(tiles, num_k, warps) > 100


@pytest.mark.parametrize("mutation", ["mma_skips_acce", "empty_before_mma"])
def test_the_gemm_model_catches_a_planted_mistake(mutation):
    with pytest.raises(AssertionError):
        explore_gemm(4, 2, 2, mutation)


# ---------------------------------------------------------------------------------------------
# The fused post-attention chain (csrc/postchain.cu, d_model 128, pre-LN): a loader (the
# attention output tile O per tile; weight blocks through a two-slot ring in the order Wo, W1_0,
# W1_1, then W2_c and W1_(c+2) per d_ff chunk c, then the next layer's W_qkv in three blocks), an
# issuer for o_proj / FFN-out / next-layer QKV (one thread), an issuer for FFN-in (another), and
# the epilogue warps, which meet at one named barrier in each row-statistics exchange (two slot
# pairs, used alternately).  Tensor memory: A1 / t / OUT and then N (the next QKV's input) in
# [0, 128), N2 [128, 256), G [256, 384), GP [384, 512); the next layer's q, k, v are computed
# into [128, 256), [256, 384), [384, 512).
def build_chain(tiles, nch, warps, fuse, mutation=None):
    bars = {}

    def bar(name, count):
        bars[name] = Bar(name, count)
        return name

    o_full, o_free = bar("o_full", 1), bar("o_free", 1)
    acc_full, acc_read = bar("acc_full", 1), bar("acc_read", warps)
    out_full, out_read = bar("out_full", 1), bar("out_read", warps)
    g_full, g_read = bar("g_full", 1), bar("g_read", warps)
    gp_ready, gp_free = bar("gp_ready", warps), bar("gp_free", 1)
    n_ready = bar("n_ready", warps)
    qkv_full = [bar(f"qkv_full{j}", 1) for j in range(3)]
    r_full = [bar(f"r_full{k}", 1) for k in range(2)]
    r_empty = [bar(f"r_empty{k}", 1) for k in range(2)]
    epi = bar("epi_bar", warps)  # the named barrier, arrive-and-wait

    order = [("Wo",), ("W1", 0)] + ([("W1", 1)] if nch > 1 else [])
    for c in range(nch):
        order.append(("W2", c))
        if c + 2 < nch:
            order.append(("W1", c + 2))
    if fuse:
        order += [("Q", j) for j in range(3)]
    units = len(order)
    pos = {u: k for k, u in enumerate(order)}
    # the issuers' own index formulas agree with the loader's order
    for k in range(nch):
        assert pos[("W1", k)] == (1 if k == 0 else (2 if k == 1 else 2 * k))
        assert pos[("W2", k)] == (3 + 2 * k if k <= nch - 2 else 2 * nch)

    load = []
    for ts in range(tiles):
        load += [("wait", o_free, ts - 1), ("check", "o_load", ts), ("tma", o_full, ("O", ts))]
        for k in range(units):
            g = ts * units + k
            load += [("wait", r_empty[g % 2], g // 2 - 1), ("check", "ring_load", g), ("tma", r_full[g % 2], ("U", g))]

    def take(g):
        return [("wait", r_full[g % 2], g // 2)]

    mma1, mma2 = [], []
    for ts in range(tiles):
        g0 = ts * units
        if ts > 0:
            mma1.append(("wait", out_read, ts - 1))
        mma1 += [("wait", o_full, ts)] + take(g0) + [
            ("check", "op_issue", ts), ("mma", "mma1", ("OP", ts)), ("commit", "mma1", r_empty[g0 % 2]),
            ("commit", "mma1", o_free), ("commit", "mma1", acc_full)]
        for c in range(nch):
            g = g0 + pos[("W2", c)]
            mma1 += [("wait", gp_ready, ts * nch + c)] + take(g) + [
                ("check", "f2_issue", (ts, c)), ("mma", "mma1", ("F2", ts, c)), ("commit", "mma1", r_empty[g % 2]),
                ("commit", "mma1", gp_free)]
        mma1.append(("commit", "mma1", out_full))
        if fuse:
            mma1.append(("wait", n_ready, ts))
            for j in range(3):
                g = g0 + pos[("Q", j)]
                mma1 += take(g) + [("check", "qkv_issue", (ts, j)), ("mma", "mma1", ("QKV", ts, j)),
                                   ("commit", "mma1", r_empty[g % 2]), ("commit", "mma1", qkv_full[j])]
            if mutation != "next_oproj_before_qkv_done":
                mma1.append(("wait", qkv_full[2], ts))

        def ffn1(k):
            g = g0 + pos[("W1", k)]
            return take(g) + [("check", "f1_issue", (ts, k)), ("mma", "mma2", ("F1", ts, k)),
                              ("commit", "mma2", r_empty[g % 2]), ("commit", "mma2", g_full)]
        mma2 += [("wait", acc_read, ts)] + ffn1(0)
        for c in range(nch):
            if mutation != "ffn1_before_g_read":
                mma2.append(("wait", g_read, ts * nch + c))
            if c + 1 < nch:
                mma2 += ffn1(c + 1)

    def epilogue(w):
        prog, n = [], 0  # n: row-statistics exchanges so far

        def stats():
            nonlocal n
            step = [("check", "red_write", n)]
            if mutation != "no_named_barrier":
                step += [("arrive", epi), ("wait", epi, n)]
            step.append(("mark", ("red_read", n, w)))
            n += 1
            return step
        for ts in range(tiles):
            prog += [("wait", acc_full, ts), ("check", "read_a1", ts), ("mark", ("a1w", ts, w))]
            prog += stats()
            prog += [("check", "n2_write", ts), ("mark", ("n2w", ts, w)), ("arrive", acc_read)]
            for c in range(nch):
                k = ts * nch + c
                prog += [("wait", g_full, k), ("check", "read_g", (ts, c)), ("mark", ("gread", ts, c, w)),
                         ("arrive", g_read)]
                if k > 0 and mutation != "gp_write_without_gp_free":
                    prog.append(("wait", gp_free, k - 1))
                prog += [("check", "gp_write", (ts, c)), ("mark", ("gpw", ts, c, w)), ("arrive", gp_ready)]
            prog += [("wait", out_full, ts), ("check", "read_out", ts), ("mark", ("outread", ts, w)),
                     ("arrive", out_read)]
            if fuse:
                prog += stats()
                prog += [("mark", ("nw", ts, w)), ("arrive", n_ready)]
                for j in range(3):
                    prog += [("wait", qkv_full[j], ts), ("check", "read_qkv", (ts, j)), ("mark", ("qkvread", ts, j, w))]
        return prog

    progs = {"load": load, "mma1": mma1, "mma2": mma2}
    for w in range(warps):
        progs[f"epi{w}"] = epilogue(w)
    return progs, bars, units, pos


def explore_chain(tiles, nch, warps, fuse, mutation=None):
    """The chain's protocol for ``tiles`` tiles of ``nch`` d_ff chunks on one CTA."""
    progs, bars, units, pos = build_chain(tiles, nch, warps, fuse, mutation)
    key_bar = {a[2]: a[1] for a in progs["load"] if a[0] == "tma"}
    qpos = {t: {a[2]: k for k, a in enumerate([a for a in progs[t] if a[0] in ("mma", "commit")]) if a[0] == "mma"}
            for t in ("mma1", "mma2")}
    mma_pc = {a[2]: (t, pc) for t in ("mma1", "mma2") for pc, a in enumerate(progs[t]) if a[0] == "mma"}
    marks = mark_pcs(progs)
    unit_mma = {}  # ring unit -> the MMA that reads it
    for ts in range(tiles):
        for u, k in pos.items():
            key = {"Wo": ("OP", ts), "W1": ("F1", ts, u[-1]), "W2": ("F2", ts, u[-1]), "Q": ("QKV", ts, u[-1])}[u[0]]
            unit_mma[ts * units + k] = key

    def owner(key):
        return "mma2" if key[0] == "F1" else "mma1"

    def done(comp, key):
        t = owner(key)
        return comp[t] > qpos[t][key]

    def issued(pcs, key):
        t, pc = mma_pc[key]
        return pcs[t] > pc

    def passed(pcs, key):
        return all(pcs[r] >= pc for k, (r, pc) in marks.items() if k[0] == key[0] and k[1:-1] == key[1:])

    def loaded_unit(ts, u, loaded):
        return ("U", ts * units + pos[u]) in loaded

    def hazard_free(kind, arg, pcs, comp, loaded):
        if kind == "o_load":
            return arg == 0 or done(comp, ("OP", arg - 1))
        if kind == "ring_load":
            return arg < 2 or done(comp, unit_mma[arg - 2])
        if kind == "op_issue":  # A1 free: OUT read, and N read by the previous tile's QKV MMAs
            ts = arg
            if ("O", ts) not in loaded or not loaded_unit(ts, ("Wo",), loaded):
                return False
            return ts == 0 or (passed(pcs, ("outread", ts - 1)) and
                               (not fuse or all(done(comp, ("QKV", ts - 1, j)) for j in range(3))))
        if kind == "read_a1":
            return done(comp, ("OP", arg))
        if kind == "n2_write":  # N2 free: FFN-in of the previous tile done, its q read by every warp
            ts = arg
            return ts == 0 or (all(done(comp, ("F1", ts - 1, k)) for k in range(nch)) and
                               (not fuse or passed(pcs, ("qkvread", ts - 1, 0))))
        if kind == "f1_issue":
            ts, k = arg
            if not loaded_unit(ts, ("W1", k), loaded) or not passed(pcs, ("n2w", ts)):
                return False
            if k > 0:
                return passed(pcs, ("gread", ts, k - 1))
            return ts == 0 or (passed(pcs, ("gread", ts - 1, nch - 1)) and
                               (not fuse or passed(pcs, ("qkvread", ts - 1, 1))))
        if kind == "read_g":
            ts, c = arg
            nxt = ("F1", ts, c + 1)
            return done(comp, ("F1", ts, c)) and (c + 1 >= nch or not issued(pcs, nxt))
        if kind == "gp_write":  # GP free: FFN-out of the previous chunk done, the previous tile's v read
            ts, c = arg
            k = ts * nch + c
            prev = (ts, c - 1) if c > 0 else (ts - 1, nch - 1)
            if k > 0 and not done(comp, ("F2",) + prev):
                return False
            return not (fuse and c == 0 and ts > 0) or passed(pcs, ("qkvread", ts - 1, 2))
        if kind == "f2_issue":
            ts, c = arg
            return (loaded_unit(ts, ("W2", c), loaded) and passed(pcs, ("gpw", ts, c))
                    and passed(pcs, ("a1w", ts)))
        if kind == "read_out":
            return all(done(comp, ("F2", arg, c)) for c in range(nch))
        if kind == "qkv_issue":  # N written; q over N2 after FFN-in; k over G after its last read
            ts, j = arg
            if not loaded_unit(ts, ("Q", j), loaded) or not passed(pcs, ("nw", ts)):
                return False
            if j == 0:
                return all(done(comp, ("F1", ts, k)) for k in range(nch))
            if j == 1:
                return passed(pcs, ("gread", ts, nch - 1))
            return True  # v over GP: FFN-out of the last chunk was issued before, by this thread
        if kind == "read_qkv":  # (their regions' next writers check that every warp has read them)
            ts, j = arg
            return done(comp, ("QKV", ts, j))
        if kind == "red_write":  # slot pair n % 2: every warp has read exchange n - 2
            return arg < 2 or passed(pcs, ("red_read", arg - 2))
        raise AssertionError(kind)

    return run_model(progs, bars, key_bar, ["mma1", "mma2"], hazard_free)


@pytest.mark.parametrize("tiles,nch,warps,fuse", [(2, 1, 1, True), (2, 2, 1, True), (2, 3, 1, False),
                                                  (2, 2, 2, True), (3, 1, 2, False)])
def test_chain_protocol_has_no_deadlock_aliasing_or_hazard(tiles, nch, warps, fuse):
    assert explore_chain(tiles, nch, warps, fuse) > 100


@pytest.mark.parametrize("mutation,tiles,nch,warps,fuse", [
    ("next_oproj_before_qkv_done", 2, 1, 1, True),  # o_proj overwrites N under the QKV products
    ("no_named_barrier", 2, 1, 2, True),            # a warp writes N2 while another reads q
    ("ffn1_before_g_read", 1, 2, 1, False),         # G overwritten before the epilogue read it
    ("gp_write_without_gp_free", 1, 2, 1, False),   # GP rewritten under FFN-out
])
def test_the_chain_model_catches_a_planted_mistake(mutation, tiles, nch, warps, fuse):
    with pytest.raises(AssertionError):
        explore_chain(tiles, nch, warps, fuse, mutation)


# ---------------------------------------------------------------------------------------------
# The whole-stack kernel (csrc/stack.cu, S <= 128, d_model 128, pre-LN): per sequence and layer
# ("tile-layer" s), one MMA thread issues k, v, q (into accumulators A and B of tensor memory),
# per head S = Q K^T into A, P V into B and the row sums, o_proj onto the residual R and FFN-out;
# another issues FFN-in into A; the epilogue warps drain k and v to shared memory, q into
# tensor memory, run each head's softmax (a named-barrier exchange of the row maximum, P over S),
# form O / l, and run the chain's three phases; the sequence's output leaves through per-warp
# stages that reuse the K tiles' shared memory.  Tensor memory: R [0, 128); N, then Q [128, 192)
# and O / l [192, 256), then N2, in [128, 256); A [256, 384): k, q, S / P of each head, G;
# B [384, 512): v, each head's O, GP.  HEADS heads per layer (the kernel has four; the model two).
STACK_HEADS = 2


def build_stack(seqs, layers, nch, warps, mutation=None):
    bars = {}

    def bar(name, count):
        bars[name] = Bar(name, count)
        return name

    H = STACK_HEADS
    per_tile = ["n_ready", "k_read", "kv_ready", "q_ready", "o_ready", "acc_read"]
    b = {n: bar(n, warps) for n in per_tile}
    for n in ["acc_k", "acc_v", "acc_q", "acc_full", "out_full", "s_full", "g_full", "gp_free"]:
        b[n] = bar(n, 1)
    for n in ["p_full", "g_read", "gp_ready"]:
        b[n] = bar(n, warps)
    pv_done = [bar(f"pv_done{h}", 1) for h in range(H)]
    r_full = [bar(f"r_full{k}", 1) for k in range(2)]
    r_empty = [bar(f"r_empty{k}", 1) for k in range(2)]
    epi = bar("epi_bar", warps)

    order = [("K",), ("V",), ("Q",), ("Wo",), ("W1", 0)] + ([("W1", 1)] if nch > 1 else [])
    for c in range(nch):
        order.append(("W2", c))
        if c + 2 < nch:
            order.append(("W1", c + 2))
    units = len(order)
    pos = {u: k for k, u in enumerate(order)}
    assert units == 4 + 2 * nch
    for k in range(nch):  # the issuers' index formulas agree with the loader's order
        assert pos[("W1", k)] == 3 + (1 if k == 0 else (2 if k == 1 else 2 * k))
        assert pos[("W2", k)] == 3 + (3 + 2 * k if k <= nch - 2 else 2 * nch)
    tl = seqs * layers  # tile-layers

    load = []
    for s in range(tl):
        for k in range(units):
            g = s * units + k
            load += [("wait", r_empty[g % 2], g // 2 - 1), ("check", "ring_load", g), ("tma", r_full[g % 2], ("U", g))]

    def take(g):
        return [("wait", r_full[g % 2], g // 2)]

    def mm(t, key, g=None):
        acts = [("check", "issue", key), ("mma", t, key)]
        if g is not None:
            acts.append(("commit", t, r_empty[g % 2]))
        return acts

    mma1, mma2 = [], []
    for s in range(tl):
        g0 = s * units
        mma1.append(("wait", b["n_ready"], s))
        mma1 += take(g0) + mm("mma1", ("K", s), g0) + [("commit", "mma1", b["acc_k"])]
        mma1 += take(g0 + 1) + mm("mma1", ("V", s), g0 + 1) + [("commit", "mma1", b["acc_v"])]
        if mutation != "q_before_k_read":
            mma1.append(("wait", b["k_read"], s))
        mma1 += take(g0 + 2) + mm("mma1", ("Q", s), g0 + 2) + [("commit", "mma1", b["acc_q"])]
        mma1.append(("wait", b["kv_ready"], s))
        if mutation != "s_before_q_ready":
            mma1.append(("wait", b["q_ready"], s))
        for h in range(H):
            mma1 += mm("mma1", ("S", s, h)) + [("commit", "mma1", b["s_full"]), ("wait", b["p_full"], s * H + h)]
            mma1 += mm("mma1", ("PV", s, h)) + [("commit", "mma1", pv_done[h])]
        mma1 += [("wait", b["o_ready"], s)] + take(g0 + 3) + mm("mma1", ("OP", s), g0 + 3) + [
            ("commit", "mma1", b["acc_full"])]
        for c in range(nch):
            g = g0 + pos[("W2", c)]
            mma1 += [("wait", b["gp_ready"], s * nch + c)] + take(g) + mm("mma1", ("F2", s, c), g) + [
                ("commit", "mma1", b["gp_free"])]
        mma1.append(("commit", "mma1", b["out_full"]))
        if mutation != "ffn1_skips_acc_read":
            mma2.append(("wait", b["acc_read"], s))
        for c in range(nch):
            if c > 0:
                mma2.append(("wait", b["g_read"], s * nch + c - 1))
            g = g0 + pos[("W1", c)]
            mma2 += take(g) + mm("mma2", ("F1", s, c), g) + [("commit", "mma2", b["g_full"])]
        mma2.append(("wait", b["g_read"], s * nch + nch - 1))

    def epilogue(w):
        prog, n = [], 0

        def exchange():  # a named-barrier exchange through two alternating slot pairs
            nonlocal n
            acts = [("check", "red_write", n)]
            if mutation != "no_named_barrier":
                acts += [("arrive", epi), ("wait", epi, n)]
            acts.append(("mark", ("red_read", n, w)))
            n += 1
            return acts
        for i in range(seqs):
            for l in range(layers):
                s = i * layers + l
                prog += exchange() + [("check", "nr_write", s), ("mark", ("nw", s, w)), ("arrive", b["n_ready"])]
                prog += [("wait", b["acc_k"], s), ("check", "done", ("K", s)), ("mark", ("kread", s, w)),
                         ("arrive", b["k_read"]), ("check", "sk_write", s), ("mark", ("skw", s, w)),
                         ("wait", b["acc_v"], s), ("check", "done", ("V", s)), ("check", "sv_write", s),
                         ("mark", ("svw", s, w)), ("arrive", b["kv_ready"])]
                prog += [("wait", b["acc_q"], s), ("check", "done", ("Q", s)), ("check", "q_write", s),
                         ("mark", ("qw", s, w)), ("arrive", b["q_ready"])]
                for h in range(H):
                    prog += [("wait", b["s_full"], s * H + h), ("check", "read_s", (s, h)),
                             ("mark", ("sread", s, h, w))]
                    prog += exchange()
                    prog += [("check", "p_write", (s, h)), ("mark", ("pw", s, h, w)), ("arrive", b["p_full"])]
                for h in range(H):
                    if mutation != "o_without_pv_done":
                        prog.append(("wait", pv_done[h], s))
                    prog.append(("check", "done", ("PV", s, h)))
                prog += [("mark", ("ow", s, w)), ("arrive", b["o_ready"])]
                prog += [("wait", b["acc_full"], s), ("check", "done", ("OP", s)), ("mark", ("p1r", s, w))]
                prog += exchange() + [("check", "n2_write", s), ("mark", ("n2w", s, w)), ("arrive", b["acc_read"])]
                for c in range(nch):
                    k = s * nch + c
                    prog += [("wait", b["g_full"], k), ("check", "read_g", (s, c)), ("mark", ("gread", s, c, w)),
                             ("arrive", b["g_read"])]
                    if k > 0:
                        prog.append(("wait", b["gp_free"], k - 1))
                    prog += [("check", "gp_write", (s, c)), ("mark", ("gpw", s, c, w)), ("arrive", b["gp_ready"])]
                prog += [("wait", b["out_full"], s)] + [("check", "done", ("F2", s, c)) for c in range(nch)]
            prog += exchange() + [("check", "stage_write", i), ("mark", ("stw", i, w))]
        return prog

    progs = {"load": load, "mma1": mma1, "mma2": mma2}
    for w in range(warps):
        progs[f"epi{w}"] = epilogue(w)
    return progs, bars, units, pos


def explore_stack(seqs, layers, nch, warps, mutation=None):
    """The whole-stack kernel's protocol for ``seqs`` sequences of ``layers`` layers on one CTA."""
    progs, bars, units, pos = build_stack(seqs, layers, nch, warps, mutation)
    H = STACK_HEADS
    key_bar = {a[2]: a[1] for a in progs["load"] if a[0] == "tma"}
    qpos = {t: {a[2]: k for k, a in enumerate([a for a in progs[t] if a[0] in ("mma", "commit")]) if a[0] == "mma"}
            for t in ("mma1", "mma2")}
    mma_pc = {a[2]: (t, pc) for t in ("mma1", "mma2") for pc, a in enumerate(progs[t]) if a[0] == "mma"}
    marks = mark_pcs(progs)
    unit_mma = {}
    for s in range(seqs * layers):
        for u, k in pos.items():
            unit_mma[s * units + k] = {"K": ("K", s), "V": ("V", s), "Q": ("Q", s), "Wo": ("OP", s),
                                       "W1": ("F1", s) + u[1:], "W2": ("F2", s) + u[1:]}[u[0]]

    def done(comp, key):
        t = "mma2" if key[0] == "F1" else "mma1"
        return comp[t] > qpos[t][key]

    def issued(pcs, key):
        t, pc = mma_pc[key]
        return pcs[t] > pc

    def passed(pcs, key):
        return all(pcs[r] >= pc for k, (r, pc) in marks.items() if k[0] == key[0] and k[1:-1] == key[1:])

    def unit_loaded(s, u, loaded):
        return ("U", s * units + pos[u]) in loaded

    def issue_ok(key, pcs, comp, loaded):
        kind, s = key[0], key[1]
        if kind == "K":  # A free: the previous tile-layer's last G read; N written
            return (unit_loaded(s, ("K",), loaded) and passed(pcs, ("nw", s))
                    and (s == 0 or passed(pcs, ("gread", s - 1, nch - 1))))
        if kind == "V":  # B: its previous content, GP, was read by this thread's FFN-out before
            return unit_loaded(s, ("V",), loaded) and passed(pcs, ("nw", s))
        if kind == "Q":  # A again: k drained by every warp
            return unit_loaded(s, ("Q",), loaded) and passed(pcs, ("kread", s))
        if kind == "S":  # q and the K tiles written; A held q (h = 0) or P of the previous head
            return passed(pcs, ("qw", s)) and passed(pcs, ("skw", s))
        if kind == "PV":  # P written by every warp, V tiles in shared memory
            return passed(pcs, ("pw", s, key[2])) and passed(pcs, ("svw", s))
        if kind == "OP":  # O / l pairs written by every warp; R holds the residual
            return unit_loaded(s, ("Wo",), loaded) and passed(pcs, ("ow", s)) and passed(pcs, ("nw", s))
        if kind == "F1":  # N2 written; A: P of the last head read by its P V, or G read
            c = key[2]
            if not unit_loaded(s, ("W1", c), loaded) or not passed(pcs, ("n2w", s)):
                return False
            return done(comp, ("PV", s, H - 1)) if c == 0 else passed(pcs, ("gread", s, c - 1))
        if kind == "F2":  # GP written by every warp; R holds t 2^s2 (phase 1 done)
            c = key[2]
            return unit_loaded(s, ("W2", c), loaded) and passed(pcs, ("gpw", s, c)) and passed(pcs, ("n2w", s))
        raise AssertionError(key)

    def hazard_free(kind, arg, pcs, comp, loaded):
        if kind == "issue":
            return issue_ok(arg, pcs, comp, loaded)
        if kind == "done":
            return done(comp, arg)
        if kind == "ring_load":
            return arg < 2 or done(comp, unit_mma[arg - 2])
        if kind == "nr_write":  # N over N2 of the previous tile-layer (FFN-in done reading it)
            s = arg
            return s == 0 or all(done(comp, ("F1", s - 1, c)) for c in range(nch))
        if kind == "sk_write":  # the K tiles: the previous S products done, the output stages written
            s = arg
            if s > 0 and not all(done(comp, ("S", s - 1, h)) for h in range(H)):
                return False
            i = s // layers
            return s % layers or i == 0 or passed(pcs, ("stw", i - 1))
        if kind == "sv_write":
            s = arg
            return s == 0 or all(done(comp, ("PV", s - 1, h)) for h in range(H))
        if kind == "q_write":  # Q over N, which the k, v, q products have read
            return done(comp, ("Q", arg))
        if kind == "read_s":
            s, h = arg
            return done(comp, ("S", s, h)) and (h + 1 >= H or not issued(pcs, ("S", s, h + 1)))
        if kind == "p_write":  # P over S columns other warps read
            s, h = arg
            return passed(pcs, ("sread", s, h))
        if kind == "n2_write":  # N2 over Q and O / l: the S products and o_proj have read them
            s = arg
            return done(comp, ("OP", s)) and all(done(comp, ("S", s, h)) for h in range(H))
        if kind == "read_g":
            s, c = arg
            return done(comp, ("F1", s, c)) and (c + 1 >= nch or not issued(pcs, ("F1", s, c + 1)))
        if kind == "gp_write":  # GP over each head's O (read by every warp) or the previous GP
            s, c = arg
            k = s * nch + c
            prev = (s, c - 1) if c > 0 else (s - 1, nch - 1)
            if k > 0 and not done(comp, ("F2",) + prev):
                return False
            return c > 0 or passed(pcs, ("ow", s))
        if kind == "stage_write":  # the output stages over the K tiles
            i = arg
            s = i * layers + layers - 1
            return all(done(comp, ("S", s, h)) for h in range(H))
        if kind == "red_write":
            return arg < 2 or passed(pcs, ("red_read", arg - 2))
        raise AssertionError(kind)

    return run_model(progs, bars, key_bar, ["mma1", "mma2"], hazard_free)


@pytest.mark.parametrize("seqs,layers,nch,warps", [(1, 2, 1, 1), (2, 1, 2, 1), (1, 2, 2, 2), (2, 2, 1, 1)])
def test_stack_protocol_has_no_deadlock_aliasing_or_hazard(seqs, layers, nch, warps):
    assert explore_stack(seqs, layers, nch, warps) > 100


@pytest.mark.parametrize("mutation,seqs,layers,nch,warps", [
    ("q_before_k_read", 1, 1, 1, 1),       # q overwrites k before every warp drained it
    ("no_named_barrier", 1, 1, 1, 2),      # P over S columns another warp has not read
    ("s_before_q_ready", 1, 1, 1, 1),      # S computed before q is in tensor memory
    ("ffn1_skips_acc_read", 1, 1, 1, 1),   # FFN-in before N2 is written
    ("o_without_pv_done", 1, 1, 1, 1),     # O read before P V completed
])
def test_the_stack_model_catches_a_planted_mistake(mutation, seqs, layers, nch, warps):
    with pytest.raises(AssertionError):
        explore_stack(seqs, layers, nch, warps, mutation)
