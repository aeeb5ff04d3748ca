"""The streaming slot pool's replacement policy (host only, no GPU), through
the C ABI's smoe_cache_simulate: a free slot first (lowest index), else evict
the resident expert used least often, ties to the one used least recently,
then to the lower slot, never an expert of the current request. Checked
against a small model written here from that rule, on a worked example and
on seeded random request streams, and for its invariants and errors."""
import numpy as np
import pytest

import int4_routed_expert_router_gb300 as smoe


def model(n_layers, E, n_slots, requests):
    """The rule written out directly (a dictionary of resident experts)."""
    slot_of, uses, last, owner = {}, {}, {}, {}
    free = list(range(n_slots))
    out, hits, misses = [], 0, 0
    for tick, (layer, ids) in enumerate(requests, start=1):
        ids = list(ids)
        if len(set(ids)) > n_slots:
            raise MemoryError
        pinned = set()
        for e in ids:                                  # resident ones first
            s = slot_of.get((layer, e))
            if s is not None:
                hits += 1
                uses[s] += 1
                last[s] = tick
                pinned.add(s)
        placed = set()
        for e in ids:
            s = slot_of.get((layer, e))
            if s is not None:
                if s in placed:
                    hits += 1
                    uses[s] += 1
                    last[s] = tick
                continue
            misses += 1
            if free:
                s = free.pop(0)
            else:
                s = min((x for x in owner if x not in pinned), key=lambda x: (uses[x], last[x], x))
                del slot_of[owner[s]]
            owner[s] = (layer, e)
            slot_of[(layer, e)] = s
            uses[s], last[s] = 1, tick
            pinned.add(s)
            placed.add(s)
        out += [slot_of[(layer, e)] for e in ids]
    return np.asarray(out, np.int32), hits, misses


def test_worked_example():
    reqs = [(0, [0, 1]), (0, [0, 2]), (1, [3]), (0, [1])]
    slots, hits, misses = smoe.cache_simulate(2, 4, 3, reqs)
    # [0,1] fill slots 0,1; expert 0 hits, 2 takes slot 2; (1,3) evicts (0,1) (one use,
    # oldest); (0,1) comes back into slot 2, whose expert was used once at tick 2
    assert slots.tolist() == [0, 1, 0, 2, 1, 2]
    assert (hits, misses) == (1, 5)


@pytest.mark.parametrize("seed", range(6))
def test_matches_the_rule_on_random_streams(seed):
    rng = np.random.default_rng(seed)
    n_layers, E = int(rng.integers(1, 4)), int(rng.integers(4, 40))
    n_slots = int(rng.integers(8, 3 * E))
    reqs = []
    for _ in range(200):
        layer = int(rng.integers(0, n_layers))
        n = int(rng.integers(1, min(8, n_slots) + 1))
        # skewed choice, with occasional repeats inside a request
        ids = rng.zipf(1.5, size=n) % E
        if len(set(ids.tolist())) > n_slots:
            continue
        reqs.append((layer, ids.tolist()))
    got, gh, gm = smoe.cache_simulate(n_layers, E, n_slots, reqs)
    want, wh, wm = model(n_layers, E, n_slots, reqs)
    assert np.array_equal(got, want)
    assert (gh, gm) == (wh, wm)
    assert gh + gm == sum(len(ids) for _, ids in reqs)


def test_invariants_every_request_resident_and_slots_distinct():
    rng = np.random.default_rng(9)
    E, n_slots = 64, 20
    reqs = [(0, rng.choice(E, 10, replace=False).tolist()) for _ in range(100)]
    slots, _, _ = smoe.cache_simulate(1, E, n_slots, reqs)
    o = 0
    for _, ids in reqs:
        s = slots[o:o + len(ids)]
        o += len(ids)
        assert (s >= 0).all() and (s < n_slots).all()
        assert len(set(s.tolist())) == len(ids)      # distinct experts, distinct slots


def test_hot_experts_stay_resident():
    """A frequently used expert survives a long stream of one-off experts."""
    reqs = []
    for i in range(50):
        reqs.append((0, [0]))
        reqs.append((0, [1 + i]))
    slots, hits, misses = smoe.cache_simulate(1, 64, 4, reqs)
    assert all(slots[2 * i] == slots[0] for i in range(50))
    assert hits == 49 and misses == 51


def test_errors():
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.cache_simulate(1, 8, 2, [(0, [0, 1, 2])])       # three distinct experts, two slots
    assert ei.value.status == smoe.ENOMEM
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.cache_simulate(1, 8, 4, [(0, [8])])             # id out of range
    assert ei.value.status == smoe.EINVAL
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.cache_simulate(2, 8, 4, [(2, [0])])             # layer out of range
    assert ei.value.status == smoe.EINVAL
