"""Host-side model of the attention kernel's K/V ring (k6_attn_single.cu).

The kernel's producer loads a unit's K/V tiles in the order K_0 K_1, then V_j
followed by K_{j+2}, into a 6-slot ring; the Q.K^T warp consumes the K tiles,
the P.V warp the V tiles.  A slot is freed by an mbarrier arrival: K(n)'s by
the softmax group that sees S(n) done, V(n)'s by the Q.K^T warp once it has
seen P(n).V done (before it issues S(n+3)).  Each slot's kv_full barrier is
tested by phase parity only, so a wait for a slot's load is unambiguous only if
the slot's previous load has already landed when the wait starts.

This model writes each thread's waits in the kernel's program order as a
dependency graph and checks, for every sequence of up to three chunks of 1-7
tiles and a few long ones:
- the load-index formulas (k_load, v_load) agree with the producer's order;
- every load the producer issues finds its slot freed by someone;
- the graph has no cycle (no thread waits on itself);
- no wait can match an earlier phase of its slot.
With six slots every slot holds one kind of tile, and a lead of 2 or 3 passes.
The kernel's earlier 5-slot ring, where K and V take turns in a slot, passes
with a lead of 2 only: a lead of 3 is shown to break the last condition.
"""
import collections
import itertools
import sys

NSTAGE, NSBUF = 6, 3   # the kernel's ring slots and S buffers


def k_load(t, T, A):
    return t if t < A else 2 * t - A + 1


def v_load(j, T, A):
    lead = min(A, T)
    more = max(T - A, 0)
    return lead + j + min(j, more)


def producer_order(Ts, A):
    loads, tile = [], 0
    for T in Ts:
        loads += [("K", tile + t) for t in range(min(A, T))]
        for j in range(T):
            loads.append(("V", tile + j))
            if j + A < T:
                loads.append(("K", tile + j + A))
        tile += T
    return loads, tile


def model(Ts, A, nstage=NSTAGE):
    """Dependency graph of the kernel's waits: node -> set of nodes it waits for."""
    loads, N = producer_order(Ts, A)
    idx = {l: i for i, l in enumerate(loads)}
    deps = collections.defaultdict(set)

    def dep(a, b):
        deps[a].add(b)

    release = {idx[("K", n)]: ("wake", n) for n in range(N)}
    release.update({idx[("V", m)]: ("S_release", m + NSBUF) for m in range(N - NSBUF)})
    consumer = {}
    for i in range(len(loads)):
        if i:
            dep(("load", i), ("load", i - 1))        # the producer issues loads in order
        if i >= nstage:
            assert i - nstage in release, ("a load needs a slot nobody frees", Ts, i)
            dep(("load", i), release[i - nstage])
        dep(("landed", i), ("load", i))
    for n in range(N):
        consumer[idx[("K", n)]] = ("S", n)
        consumer[idx[("V", n)]] = ("PV", n)
        # Q.K^T thread, in order: wait P(n-3).V, free V(n-3); wait K(n); issue S(n)
        if n:
            dep(("S_release", n), ("S", n - 1))
        if n >= NSBUF:
            dep(("S_release", n), ("PV_done", n - NSBUF))
        dep(("wait_K", n), ("S_release", n))
        dep(("S", n), ("wait_K", n))
        dep(("S", n), ("landed", idx[("K", n)]))
        # softmax: tile n after S(n), the max of tile n-1, and its group's previous tile
        dep(("wake", n), ("S", n))
        if n:
            dep(("wake", n), ("wake", n - 1))
        if n >= 2:
            dep(("wake", n), ("P", n - 2))
        dep(("P", n), ("wake", n))
        # P.V thread, in order: wait V(n), then the parts of P(n); issue P(n).V
        if n:
            dep(("wait_V", n), ("PV", n - 1))
        dep(("PV", n), ("wait_V", n))
        dep(("PV", n), ("landed", idx[("V", n)]))
        dep(("PV", n), ("P", n))
        dep(("PV_done", n), ("PV", n))
    return loads, idx, deps, consumer, N


def ancestors(deps, root):
    seen, stack = set(), [root]
    while stack:
        for y in deps.get(stack.pop(), ()):
            if y not in seen:
                seen.add(y)
                stack.append(y)
    return seen


def acyclic(deps):
    sys.setrecursionlimit(max(10000, sys.getrecursionlimit()))
    state = {}

    def visit(x):
        st = state.get(x)
        if st == 1:
            return False
        if st == 2:
            return True
        state[x] = 1
        ok = all(visit(y) for y in deps.get(x, ()))
        state[x] = 2
        return ok

    nodes = set(deps) | {b for v in deps.values() for b in v}
    return all(visit(x) for x in nodes)


def aliasing(Ts, A, nstage=NSTAGE):
    """The first wait that could match an earlier phase of its slot, or None."""
    loads, idx, deps, consumer, N = model(Ts, A, nstage)
    for i, (kind, n) in enumerate(loads):
        if i < nstage:
            continue
        wait = ("wait_K" if kind == "K" else "wait_V", n)
        if consumer[i - nstage] not in ancestors(deps, wait):
            return loads[i], loads[i - nstage]
    return None


CASES = [list(Ts) for k in range(1, 4) for Ts in itertools.product(range(1, 8), repeat=k)] + \
    [[17], [51, 51], [52, 51, 51, 52]]


def test_load_index_formulas_match_the_producer_order():
    for T in range(1, 80):
        loads, _ = producer_order([T], 2)
        for t in range(T):
            assert loads[k_load(t, T, 2)] == ("K", t)
            assert loads[v_load(t, T, 2)] == ("V", t)
        # the closed forms in the kernel for a lead of 2
        for t in range(T):
            assert k_load(t, T, 2) == (t if t < 2 else 2 * t - 1)
            assert v_load(t, T, 2) == (t + 2 if t + 2 < T else T) + t


def test_every_slot_is_freed_and_no_wait_cycles():
    for Ts in CASES:
        for A in (2, 3):
            _, _, deps, _, _ = model(Ts, A)   # model() asserts that every needed slot is freed
            assert acyclic(deps), (Ts, A)


def test_no_wait_can_match_an_earlier_phase():
    for Ts in CASES:
        for A in (2, 3):
            assert aliasing(Ts, A) is None, (Ts, A)


def test_with_six_slots_a_steady_state_slot_holds_one_kind():
    # inside a unit, loads 2 .. 2T-3 alternate V and K, so there a slot's load
    # and the load six before it are the same kind: K(n) follows K(n-3), V(n)
    # follows V(n-3).  (The first two loads and a unit's tail, where only V
    # loads remain, shift the pattern; the checks above cover those.)
    for T in range(3, 40):
        loads, _ = producer_order([T], 2)
        for i in range(2 + NSTAGE, 2 * T - 2):
            assert loads[i][0] == loads[i - NSTAGE][0], (T, i)
            assert loads[i][1] == loads[i - NSTAGE][1] + 3, (T, i)


def test_five_slots_alias_with_a_lead_of_three():
    # the earlier 5-slot ring: with K three tiles ahead, the P.V warp could wait
    # for V(n) while K(n) (the slot's previous load) is still in flight
    for Ts in CASES:
        assert aliasing(Ts, 2, nstage=5) is None, Ts
    found = aliasing([5], 3, nstage=5)
    assert found == (("V", 2), ("K", 2))


def pair_model(Ts, A, nstage=NSTAGE, remote_release=True):
    """Two CTAs of a cluster running the same units (the kernel's multicast
    form): each loads one panel of every tile into both, so a load lands in a
    CTA only once both CTAs issued their panels, and a slot is refilled only
    once the consumers of both CTAs released it (remote_release=False drops the
    partner's release, a mistake the checks below must catch)."""
    loads, idx, deps, consumer, N = model(Ts, A, nstage)
    pair = collections.defaultdict(set)
    for node, ds in deps.items():
        for cta in (0, 1):
            for d in ds:
                pair[(cta, node)].add((cta, d))
    for i in range(len(loads)):
        for cta in (0, 1):
            pair[(cta, ("landed", i))].add((1 - cta, ("load", i)))    # the partner's panel
            if i >= nstage and remote_release:
                release = next(iter(deps[("load", i)] - {("load", i - 1)}))
                pair[(cta, ("load", i))].add((1 - cta, release))      # the partner's release
    return pair, loads, consumer


def pair_refill_races(Ts, A, remote_release=True, nstage=NSTAGE):
    """Loads whose multicast could overwrite a slot the partner still reads: CTA
    X's load i writes slot i % nstage in both CTAs, so the partner's consumer of
    load i - nstage must come before it."""
    pair, loads, consumer = pair_model(Ts, A, nstage, remote_release)
    races = []
    for i in range(nstage, len(loads)):
        for cta in (0, 1):
            if (1 - cta, consumer[i - nstage]) not in ancestors(pair, (cta, ("load", i))):
                races.append((cta, loads[i]))
    return races


def test_cluster_pair_has_no_wait_cycle():
    for Ts in CASES:
        assert acyclic(pair_model(Ts, 2)[0]), Ts


def test_cluster_pair_never_refills_a_slot_the_partner_reads():
    for Ts in CASES:
        assert pair_refill_races(Ts, 2) == [], Ts


def test_without_the_partner_release_a_refill_races():
    assert pair_refill_races([7], 2, remote_release=False)
