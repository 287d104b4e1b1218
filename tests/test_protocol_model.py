"""Race checks of the synchronisation protocols by exhaustive-ish random
interleaving, on the CPU (compute-sanitizer is not available, and a GPU run
shows one schedule at a time).

Each (rank, call) of a chain is a process of small atomic steps: stores,
polls that block until a condition holds, reads.  A scheduler runs a random
runnable process one step at a time, over many seeds.  A process of call e
starts, in serial mode, once every rank has finished call e - 1 (the kernel
boundary), in overlap mode once its own rank has finished call e - 1 (the
hand-off of CTA (r, k) to CTA (r, k) of the next call).  Found:

* a race: a store over a slot whose previous message was not read yet, or a
  read of an input or output of the wrong call;
* a deadlock: nothing can run before every process has finished.

Models (one CTA index; the protocols are per CTA index):

* LL: epoch-tagged packets into recv[receiver][e & 1][sender]; the reader
  polls until the slot carries epoch e ("Every Microsecond Counts", page 1,
  section "Four barrier-free mechanisms", parts 1 and 3).
* sentinel: raw values into the same slots; the reader polls until the slot
  is not the sentinel, reads, and refills it with the sentinel (part 2).
* two-shot pull (the TMA AllReduce and the two-shot fused normalisation):
  rank q publishes its input for call e and stores arrive[q] = e; owner j
  reads every rank's input once arrive[q] >= e and writes its share of every
  rank's output, then stores cmpl[p][j] = e; rank p finishes only once every
  owner's cmpl[p][j] >= e ("SiFAR", page 3, "Limits of existing algorithms";
  page 1 part 4: counters reaching N, kept as flags).

* DB and BASELINE: raw data, then a top barrier of epoch flags (DB, two
  buffers) or one buffer with a top and a bottom barrier (BASELINE).
* two-shot over flagged lines: reduce-scatter into the owner's lines, then an
  all-gather into every rank's lines, both epoch-tagged.
* two-shot over sentinels: the same two phases with raw values into
  sentinel-prefilled slots, each refilled by its reader.
* atomic accumulation: every rank adds into the owner's line and bumps its
  counter; the owner reads at counter = R, clears the line, all-gathers.

Each model also runs with a planted mistake (a single buffer under overlap,
no refill, no bottom barrier on one buffer, no completion wait, no arrival
wait, no all-gather wait, no clear) that the search must catch, so the
checker itself is shown to see races.
"""
import random

import pytest


class Race(AssertionError):
    pass


class Deadlock(AssertionError):
    pass


def run(procs_of, R, calls, overlap, seed, max_steps=200000):
    """procs_of(r, e, state) -> generator; yields a callable (block until it
    returns True) or None (a step boundary)."""
    rng = random.Random(seed)
    state = {"done": [0] * R}
    live = {}            # (r, e) -> [generator, pending condition]
    started = set()

    def can_start(r, e):
        if overlap:
            return state["done"][r] >= e - 1
        return all(d >= e - 1 for d in state["done"])

    for _ in range(max_steps):
        for r in range(R):
            e = state["done"][r] + 1
            while (r, e) in started:
                e += 1
            if e <= calls and (r, e) not in started and can_start(r, e) and \
                    all((r, f) not in live for f in range(1, e)):
                live[(r, e)] = [procs_of(r, e, state), None]
                started.add((r, e))
        runnable = [key for key, (g, cond) in live.items() if cond is None or cond()]
        if not runnable:
            if not live and all(d == calls for d in state["done"]):
                return
            raise Deadlock(f"seed {seed}: nothing can run; waiting: {sorted(live)}")
        key = rng.choice(runnable)
        g = live[key][0]
        try:
            live[key][1] = next(g)
        except StopIteration:
            r, e = key
            state["done"][r] = e
            del live[key]
    raise AssertionError("step limit")


# ------------------------------------------------------------------ LL
def ll_model(R, single_buffer=False):
    def procs_of(r, e, st):
        slots = st.setdefault("slots", {})
        par = 0 if single_buffer else e & 1
        peers = [q for q in range(R) if q != r]
        for p in peers:                                   # sends
            s = slots.setdefault((p, par, r), {"epoch": 0, "unread": False})
            if s["unread"]:
                raise Race(f"rank {r} call {e} overwrote rank {p}'s unread epoch {s['epoch']}")
            s.update(epoch=e, unread=True)
            yield None
        for q in random.Random(r * 1000 + e).sample(peers, len(peers)):      # receives, any order
            key = (r, par, q)
            yield (lambda key=key: slots.get(key, {}).get("epoch") == e)
            s = slots[key]
            if s["epoch"] != e:
                raise Race(f"rank {r} call {e} read epoch {s['epoch']} from {q}")
            s["unread"] = False
    return procs_of


# ------------------------------------------------------------ sentinel
SENT = None


def sentinel_model(R, refill=True):
    def procs_of(r, e, st):
        slots = st.setdefault("slots", {})
        par = e & 1
        peers = [q for q in range(R) if q != r]
        for p in peers:
            key = (p, par, r)
            if slots.get(key, SENT) is not SENT:
                raise Race(f"rank {r} call {e} stored over {slots[key]} (not yet read or refilled)")
            slots[key] = (r, e)
            yield None
        for q in random.Random(r * 7919 + e).sample(peers, len(peers)):
            key = (r, par, q)
            yield (lambda key=key: slots.get(key, SENT) is not SENT)
            if slots[key] != (q, e):
                raise Race(f"rank {r} call {e} read {slots[key]} from {q}")
            yield None
            if refill:
                slots[key] = SENT
            else:
                slots[key] = ("stale", q, e)      # a reader that forgets the refill
    return procs_of


# ------------------------------------------------------------ two-shot pull
def pull_model(R, completion_wait=True, arrival_wait=True):
    def procs_of(r, e, st):
        inp = st.setdefault("input", [0] * R)
        out = st.setdefault("out", [[0] * R for _ in range(R)])      # out[p][owner share] = call written
        arrive = st.setdefault("arrive", [0] * R)
        cmpl = st.setdefault("cmpl", [[0] * R for _ in range(R)])
        # rank r's stream: the previous call's output is consumed, then this
        # call's input produced
        if e > 1 and any(v != e - 1 for v in out[r]):
            raise Race(f"rank {r} consumed call {e - 1}'s output while it held {out[r]}")
        inp[r] = e
        yield None
        arrive[r] = e
        yield None
        order = random.Random(r * 104729 + e).sample(range(R), R)
        for q in order:                                   # owner r reads share r of every rank
            if arrival_wait:
                yield (lambda q=q: arrive[q] >= e)
            if inp[q] != e:
                raise Race(f"owner {r} call {e} read rank {q}'s input of call {inp[q]}")
            yield None
        for p in order:                                   # and writes share r of every rank's output
            out[p][r] = e
            yield None
        for p in range(R):
            cmpl[p][r] = e
        yield None
        if completion_wait:
            for q in range(R):
                yield (lambda q=q: cmpl[r][q] >= e)
    return procs_of


SEEDS = range(300)


@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("R", [2, 3, 4])
def test_ll_double_buffer_has_no_race(R, overlap):
    for seed in SEEDS:
        run(ll_model(R), R, calls=6, overlap=overlap, seed=seed)


def test_ll_single_buffer_races_under_overlap():
    """The forced single buffer: safe with kernel boundaries, a race once
    calls overlap (the GPU test of the same knob sees a timeout or a wrong
    value)."""
    for seed in SEEDS:
        run(ll_model(3, single_buffer=True), 3, calls=6, overlap=False, seed=seed)
    caught = 0
    for seed in SEEDS:
        try:
            run(ll_model(3, single_buffer=True), 3, calls=6, overlap=True, seed=seed)
        except (Race, Deadlock):
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("R", [2, 3, 4])
def test_sentinel_refill_has_no_race(R, overlap):
    for seed in SEEDS:
        run(sentinel_model(R), R, calls=6, overlap=overlap, seed=seed)


def test_sentinel_without_refill_is_caught():
    with pytest.raises(Race):
        for seed in SEEDS:
            run(sentinel_model(3, refill=False), 3, calls=6, overlap=False, seed=seed)


@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("R", [2, 3, 4])
def test_two_shot_pull_has_no_race(R, overlap):
    for seed in SEEDS:
        run(pull_model(R), R, calls=6, overlap=overlap, seed=seed)


@pytest.mark.parametrize("planted", ["no completion wait", "no arrival wait"])
def test_two_shot_pull_planted_mistakes_are_caught(planted):
    kw = {"completion_wait": planted != "no completion wait", "arrival_wait": planted != "no arrival wait"}
    caught = 0
    for seed in SEEDS:
        try:
            run(pull_model(3, **kw), 3, calls=6, overlap=True, seed=seed)
        except Race:
            caught += 1
    assert caught > 0, planted


# ------------------------------------------------- two-shot over sentinels
def twoshot_sentinel_model(R, double_buffer=True, refill=True, empty_owner=False, ag_wait=True):
    """The pages' two-phase LLBuffer algorithm ("Every Microsecond Counts",
    page 1, "Unified primitives and API design", table of variants: sentinel
    synchronisation + double buffering): rank q stores share j raw into owner
    j's slot rs[j][par][q]; the owner polls until none of its R - 1 slots
    holds the sentinel, reads and refills them, then stores the reduced share
    into ag[p][par][j] of every rank p, which polls, reads and refills.  With
    empty_owner, the last rank's share is empty (a message shorter than
    (R - 1) chunks): nobody sends it a share and nobody waits for its
    all-gather."""
    def procs_of(r, e, st):
        rs = st.setdefault("rs", {})
        ag = st.setdefault("ag", {})
        par = e & 1 if double_buffer else 0
        peers = [q for q in range(R) if q != r]
        owns = lambda j: not (empty_owner and j == R - 1)

        def put(region, key, val):
            if region.get(key, SENT) is not SENT:
                raise Race(f"rank {r} call {e} stored over {region[key]} at {key} (not read or refilled)")
            region[key] = val

        def take(region, key, want):
            if region[key] != want:
                raise Race(f"rank {r} call {e} read {region[key]} at {key}, wanted {want}")
            region[key] = SENT if refill else ("stale",) + want

        for j in peers:
            if owns(j):
                put(rs, (j, par, r), (r, e))
                yield None
        if owns(r):
            for q in random.Random(r * 31 + e).sample(peers, len(peers)):
                yield (lambda q=q: rs.get((r, par, q), SENT) is not SENT)
                take(rs, (r, par, q), (q, e))
                yield None
            for p in peers:
                put(ag, (p, par, r), (r, e))
                yield None
        for j in random.Random(r * 37 + e).sample(peers, len(peers)):
            if owns(j) and ag_wait:
                yield (lambda j=j: ag.get((r, par, j), SENT) is not SENT)
                take(ag, (r, par, j), (j, e))
                yield None
    return procs_of


@pytest.mark.parametrize("empty_owner", [False, True])
@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("R", [2, 3, 4])
def test_twoshot_sentinel_has_no_race(R, overlap, empty_owner):
    for seed in SEEDS:
        run(twoshot_sentinel_model(R, empty_owner=empty_owner), R, calls=6, overlap=overlap, seed=seed)


@pytest.mark.parametrize("planted", ["no refill", "no all-gather wait"])
def test_twoshot_sentinel_planted_mistakes_are_caught(planted):
    kw = {"refill": planted != "no refill", "ag_wait": planted != "no all-gather wait"}
    caught = 0
    for seed in SEEDS:
        try:
            run(twoshot_sentinel_model(3, **kw), 3, calls=6, overlap=True, seed=seed)
        except (Race, Deadlock):
            caught += 1
    assert caught > 0, planted


@pytest.mark.parametrize("empty_owner", [False, True])
def test_twoshot_sentinel_all_gather_orders_slot_reuse(empty_owner):
    """As for the two-shot over flagged lines, the all-gather alone orders the
    reuse of every slot: a single buffer is race-free too, so the second
    buffer is extra safety, not a requirement (a sender reaches call e + 1
    only after the owner's call-e all-gather, sent after its call-e reads;
    an owner's call-e + 1 all-gather follows every rank's call-e + 1 send,
    which follows that rank's call-e reads)."""
    for seed in SEEDS:
        run(twoshot_sentinel_model(3, double_buffer=False, empty_owner=empty_owner), 3, calls=6, overlap=True,
            seed=seed)


# ------------------------------------------------------------ DB / BASELINE
def flag_model(R, double_buffer=True, bottom=False):
    """Raw data into recv[receiver][parity][sender], then a top barrier of
    epoch flags (DB: ready flags after the data; "SiFAR", page 3, Technique
    1), and for BASELINE one buffer and a bottom barrier after the reads
    (page 1, "Global memory barriers")."""
    def procs_of(r, e, st):
        slots = st.setdefault("slots", {})
        top = st.setdefault("top", {})
        bot = st.setdefault("bot", {})
        par = e & 1 if double_buffer else 0
        peers = [q for q in range(R) if q != r]
        for p in peers:
            s = slots.setdefault((p, par, r), {"call": 0, "unread": False})
            if s["unread"]:
                raise Race(f"rank {r} call {e} overwrote rank {p}'s unread call {s['call']}")
            s.update(call=e, unread=True)
            yield None
        for p in peers:
            top[(p, r)] = e
        yield None
        for q in peers:
            yield (lambda q=q: top.get((r, q), 0) >= e)
        for q in peers:
            s = slots[(r, par, q)]
            if s["call"] != e:
                raise Race(f"rank {r} call {e} read call {s['call']} from {q}")
            s["unread"] = False
            yield None
        if bottom:
            for p in peers:
                bot[(p, r)] = e
            yield None
            for q in peers:
                yield (lambda q=q: bot.get((r, q), 0) >= e)
    return procs_of


@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("R", [2, 3, 4])
@pytest.mark.parametrize("proto", ["db", "baseline"])
def test_flag_protocols_have_no_race(proto, R, overlap):
    kw = {"double_buffer": True, "bottom": False} if proto == "db" else {"double_buffer": False, "bottom": True}
    for seed in SEEDS:
        run(flag_model(R, **kw), R, calls=6, overlap=overlap, seed=seed)


def test_one_buffer_without_bottom_barrier_is_caught():
    caught = 0
    for seed in SEEDS:
        try:
            run(flag_model(3, double_buffer=False, bottom=False), 3, calls=6, overlap=True, seed=seed)
        except Race:
            caught += 1
    assert caught > 0


# ------------------------------------------------ two-shot over flagged lines
def twoshot_model(R, double_buffer=True, ag_wait=True):
    """Reduce-scatter: rank q sends share j to owner j's slot rs[j][par][q]
    (epoch-tagged lines); the owner polls all R - 1, folds, and all-gathers
    the result into ag[p][par][j] for every rank p, which polls all owners."""
    def procs_of(r, e, st):
        rs = st.setdefault("rs", {})
        ag = st.setdefault("ag", {})
        par = e & 1 if double_buffer else 0
        peers = [q for q in range(R) if q != r]

        def put(region, key):
            s = region.setdefault(key, {"epoch": 0, "unread": False})
            if s["unread"]:
                raise Race(f"rank {r} call {e} overwrote unread epoch {s['epoch']} at {key}")
            s.update(epoch=e, unread=True)

        def take(region, key):
            s = region[key]
            if s["epoch"] != e:
                raise Race(f"rank {r} call {e} read epoch {s['epoch']} at {key}")
            s["unread"] = False

        for j in peers:
            put(rs, (j, par, r))
            yield None
        for q in peers:
            yield (lambda q=q: rs.get((r, par, q), {}).get("epoch") == e)
            take(rs, (r, par, q))
        for p in peers:
            put(ag, (p, par, r))
            yield None
        for j in peers:
            if ag_wait:
                yield (lambda j=j: ag.get((r, par, j), {}).get("epoch") == e)
                take(ag, (r, par, j))
    return procs_of


@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("R", [2, 3, 4])
def test_twoshot_lines_have_no_race(R, overlap):
    for seed in SEEDS:
        run(twoshot_model(R), R, calls=6, overlap=overlap, seed=seed)


def test_twoshot_phases_order_slot_reuse():
    """Finding: the two phases alone order every slot's reuse (a rank starts
    call e + 1 only after every owner's all-gather of call e, which the owner
    sends only after reading that rank's reduce-scatter lines of call e), so
    even one buffer is race-free in this model; the kernel double-buffers
    anyway.  A rank that skips the all-gather wait is caught."""
    for seed in SEEDS:
        run(twoshot_model(3, double_buffer=False), 3, calls=6, overlap=True, seed=seed)
    caught = 0
    for seed in SEEDS:
        try:
            run(twoshot_model(3, double_buffer=False, ag_wait=False), 3, calls=6, overlap=True, seed=seed)
        except (Race, Deadlock):
            caught += 1
    assert caught > 0


# ------------------------------------------------------- atomic accumulation
def atomic_model(R, clear=True, double_buffer=True):
    """LL128 atomic (page 1, part 4): every rank adds its part into owner j's
    accumulator line acc[j][par] and bumps its counter; the owner waits for
    counter == R, reads the sum, clears the line (data and counter) and
    all-gathers with epoch flags."""
    def procs_of(r, e, st):
        acc = st.setdefault("acc", {})
        ag = st.setdefault("ag", {})
        par = e & 1 if double_buffer else 0
        peers = [q for q in range(R) if q != r]
        for j in range(R):                                # adds, own line included
            line = acc.setdefault((j, par), {"parts": [], "count": 0})
            if any(c != e for _, c in line["parts"]):
                raise Race(f"rank {r} call {e} added into owner {j}'s line holding {line['parts']}")
            line["parts"].append((r, e))
            line["count"] += 1
            yield None
        line = acc[(r, par)]
        yield (lambda line=line: line["count"] >= R)
        if sorted(line["parts"]) != [(q, e) for q in range(R)]:
            raise Race(f"owner {r} call {e} read {sorted(line['parts'])}")
        if clear:
            line["parts"], line["count"] = [], 0
        else:
            line["count"] = 0                             # a reader that forgets the data
        yield None
        for p in peers:
            ag[(p, par, r)] = e
        yield None
        for j in peers:
            yield (lambda j=j: ag.get((r, par, j), 0) == e)
    return procs_of


@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("R", [2, 3, 4])
def test_atomic_lines_have_no_race(R, overlap):
    for seed in SEEDS:
        run(atomic_model(R), R, calls=6, overlap=overlap, seed=seed)


def test_atomic_missing_clear_is_caught():
    caught = 0
    for seed in SEEDS:
        try:
            run(atomic_model(3, clear=False), 3, calls=6, overlap=True, seed=seed)
        except (Race, Deadlock):
            caught += 1
    assert caught > 0


def test_atomic_all_gather_orders_line_reuse():
    """Finding, as for the two-shot lines: the all-gather already orders the
    reuse of an accumulator line (the owner clears it before its all-gather,
    and every adder waits for that all-gather before its next call), so one
    buffer is race-free in this model too."""
    for seed in SEEDS:
        run(atomic_model(3, double_buffer=False), 3, calls=6, overlap=True, seed=seed)


# ------------------------------------------- overlap hand-off and geometry
def run_ctas(R, Ks, units, overlap, cross_geometry, seed, max_steps=400000):
    """LL over CTAs: call e (epoch e) runs Ks[e - 1] CTAs per rank; CTA k of
    every rank handles units u with u % K == k.  In overlap mode CTA (r, k)
    of call e starts once CTA (r, k) of call e - 1 is done, but only when
    the two calls have the same geometry (the host's overlap key); otherwise
    (or in serial mode) it starts once every CTA of every earlier call is done.
    cross_geometry=True plants the mistake of overlapping across a change."""
    rng = random.Random(seed)
    calls = len(Ks)
    done = {}                       # (r, k) -> last epoch finished by that CTA index
    finished = set()                # (r, k, e)
    slots = {}
    live, started = {}, set()

    def all_done_before(e):
        return all((r, k, f) in finished for f in range(1, e) for r in range(R) for k in range(Ks[f - 1]))

    def can_start(r, k, e):
        if e > 1 and overlap and (Ks[e - 1] == Ks[e - 2] or cross_geometry):
            return k < Ks[e - 2] and (r, k, e - 1) in finished or (k >= Ks[e - 2] and all_done_before(e))
        return all_done_before(e)

    def proc(r, k, e):
        K = Ks[e - 1]
        par = e & 1
        mine = [u for u in range(units) if u % K == k]
        peers = [q for q in range(R) if q != r]
        for u in mine:
            for p in peers:
                s = slots.setdefault((p, par, r, u), {"epoch": 0, "unread": False})
                if s["unread"]:
                    raise Race(f"CTA ({r},{k}) call {e} overwrote unread epoch {s['epoch']} of unit {u} at rank {p}")
                s.update(epoch=e, unread=True)
                yield None
        for u in mine:
            for q in peers:
                key = (r, par, q, u)
                yield (lambda key=key: slots.get(key, {}).get("epoch") == e)
                slots[key]["unread"] = False

    for _ in range(max_steps):
        for e in range(1, calls + 1):
            for r in range(R):
                for k in range(Ks[e - 1]):
                    if (r, k, e) not in started and can_start(r, k, e):
                        live[(r, k, e)] = [proc(r, k, e), None]
                        started.add((r, k, e))
        runnable = [key for key, (g, cond) in live.items() if cond is None or cond()]
        if not runnable:
            if len(finished) == sum(R * K for K in Ks):
                return
            raise Deadlock(f"seed {seed}: waiting {sorted(live)}")
        key = rng.choice(runnable)
        try:
            live[key][1] = next(live[key][0])
        except StopIteration:
            finished.add(key)
            done[key[:2]] = key[2]
            del live[key]
    raise AssertionError("step limit")


GEOMETRIES = [[2, 2, 1, 1, 2, 2, 2, 1], [1, 2, 2, 1, 2, 1, 1, 2], [2, 2, 2, 2, 2, 2, 2, 2]]


@pytest.mark.parametrize("Ks", GEOMETRIES)
def test_overlap_hand_off_only_within_one_geometry_is_safe(Ks):
    for seed in range(150):
        run_ctas(3, Ks, units=4, overlap=True, cross_geometry=False, seed=seed)
        run_ctas(3, Ks, units=4, overlap=False, cross_geometry=False, seed=seed)


def test_overlap_across_a_geometry_change_is_caught():
    caught = 0
    for seed in range(150):
        try:
            run_ctas(3, GEOMETRIES[0], units=4, overlap=True, cross_geometry=True, seed=seed)
        except (Race, Deadlock):
            caught += 1
    assert caught > 0


# --------------------------------------------- cluster statistics exchange
def run_cluster(CL, rows, seed, early_exit=False, max_steps=200000):
    """The row statistics exchange of the fused kernels: per row, every CTA of
    a cluster stores its partial into a slot of every cluster CTA (st.async),
    counted by the target's mbarrier of that round, waits for its own
    mbarrier, reads the slots; two rounds (maxima, sums) per row, one
    mbarrier each, whose phase advances once per row.  Checked: a store for
    row j reaches a CTA only after that CTA has read its row j - 1 slots of
    the round (else it would overwrite them or count in the wrong phase),
    and never after the CTA has exited.  early_exit plants a CTA that leaves
    without its last wait."""
    rng = random.Random(seed)
    ctas = [{"read": [0, 0], "count": [dict(), dict()], "slot": [dict(), dict()], "exited": False}
            for _ in range(CL)]

    def proc(c):
        for row in range(rows):
            for rnd in (0, 1):
                for d in rng.sample(range(CL), CL):
                    dst = ctas[d]
                    if dst["exited"]:
                        raise Race(f"CTA {c} stored row {row} round {rnd} into exited CTA {d}")
                    if dst["read"][rnd] < row:
                        raise Race(f"CTA {c} stored row {row} round {rnd} before CTA {d} read row {row - 1}")
                    dst["slot"][rnd][c] = row
                    dst["count"][rnd][row] = dst["count"][rnd].get(row, 0) + 1
                    yield None
                me = ctas[c]
                if early_exit and c == 0 and row == rows - 1 and rnd == 1:
                    break
                yield (lambda me=me, rnd=rnd, row=row: me["count"][rnd].get(row, 0) == CL)
                if any(v != row for v in me["slot"][rnd].values()):
                    raise Race(f"CTA {c} row {row} round {rnd} read {me['slot'][rnd]}")
                me["read"][rnd] = row + 1
                yield None
        ctas[c]["exited"] = True

    live = {c: [proc(c), None] for c in range(CL)}
    for _ in range(max_steps):
        runnable = [c for c, (g, cond) in live.items() if cond is None or cond()]
        if not runnable:
            if not live:
                return
            raise Deadlock(f"seed {seed}: {sorted(live)}")
        c = rng.choice(runnable)
        try:
            live[c][1] = next(live[c][0])
        except StopIteration:
            del live[c]
    raise AssertionError("step limit")


@pytest.mark.parametrize("CL", [1, 2, 4, 8])
def test_cluster_exchange_has_no_race(CL):
    for seed in range(300):
        run_cluster(CL, rows=4, seed=seed)


def test_cluster_exchange_early_exit_is_caught():
    caught = 0
    for seed in range(300):
        try:
            run_cluster(4, rows=3, seed=seed, early_exit=True)
        except (Race, Deadlock):
            caught += 1
    assert caught > 0
