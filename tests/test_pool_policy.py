"""The expert slot pool's host-side policy (no GPU): fmoe_pool_plan against a
plain least-recently-used simulation written here, plus its edge cases.

Planning touches no device: the slot and host-blob pointers given to
fmoe_pool_init are only stored (nonzero, aligned stand-ins here)."""
import numpy as np
import pytest

from quantized_moe_expert_05_b300 import build

FAKE_SLOTS = 1 << 20          # never dereferenced by planning
FAKE_HOST = 1 << 21


@pytest.fixture(scope="module")
def fm():
    build.build()
    from quantized_moe_expert_05_b300 import fmoe
    return fmoe


def pool(fm, S, E, blob=256):
    return fm.SlotPool(S, E, blob, FAKE_SLOTS, FAKE_HOST)


class RefLRU:
    """Least recently used with protection of the last `keep` requests: the
    policy stated in include/fmoe.h, restated independently."""

    def __init__(self, S, E):
        self.S, self.E = S, E
        self.expert_of = [None] * S
        self.last = [0] * S
        self.tick = 0
        self.hits = self.misses = 0

    def plan(self, ids, keep):
        now = self.tick + 1
        lo = max(1, now - keep)
        where = {e: s for s, e in enumerate(self.expert_of) if e is not None}
        distinct = list(dict.fromkeys(ids))
        missing = [e for e in distinct if e not in where]
        resident_slots = {where[e] for e in distinct if e in where}
        free = [s for s in range(self.S)
                if (self.expert_of[s] is None or self.last[s] < lo) and s not in resident_slots]
        if len(free) < len(missing):
            return None
        self.tick = now
        for e in distinct:
            if e in where:
                self.hits += 1
                self.last[where[e]] = now
        loads = []
        for e in ids:
            if e in where:
                continue
            cands = [s for s in range(self.S) if self.expert_of[s] is None or self.last[s] < lo]
            s = min(cands, key=lambda c: (0 if self.expert_of[c] is None else self.last[c], c))
            if self.expert_of[s] is not None:
                del where[self.expert_of[s]]
            self.expert_of[s] = e
            where[e] = s
            self.last[s] = now
            loads.append((e, s))
            self.misses += 1
        return [where[e] for e in ids], loads


def test_empty_pool_fills_lowest_slots_then_evicts_least_recent(fm):
    p = pool(fm, 4, 10)
    assert p.plan([1, 2]) == ([0, 1], [(1, 0), (2, 1)])
    assert p.plan([3]) == ([2], [(3, 2)])
    assert p.plan([4]) == ([3], [(4, 3)])
    # slots 0 and 1 were last used by request 1: the lower one goes first
    assert p.plan([5]) == ([0], [(5, 0)])
    # expert 2 is resident: a hit, no load
    assert p.plan([2]) == ([1], [])
    assert p.stats() == {"hits": 1, "misses": 5, "requests": 5}


def test_duplicates_load_once(fm):
    p = pool(fm, 3, 8)
    slots, loads = p.plan([7, 7, 3, 7])
    assert loads == [(7, 0), (3, 1)] and slots == [0, 0, 1, 0]


def test_keep_protects_the_previous_request(fm):
    p = pool(fm, 3, 8)
    p.plan([0, 1, 2])
    # keep = 1: the slots of the previous request may still be computed on
    with pytest.raises(fm.FmoeError):
        p.plan([3], keep=1)
    # keep = 0: slot 0 (least recent, lowest) is evicted
    assert p.plan([3], keep=0) == ([0], [(3, 0)])


def test_refused_request_changes_nothing(fm):
    p = pool(fm, 2, 8)
    p.plan([4, 5])
    before = p.stats()
    with pytest.raises(fm.FmoeError):
        p.plan([1, 2, 3])                 # three distinct experts, two slots
    assert p.stats() == before
    assert p.plan([4]) == ([0], [])        # expert 4 still resident


def test_bad_ids_are_refused(fm):
    p = pool(fm, 4, 8)
    with pytest.raises(fm.FmoeError):
        p.plan([8])
    with pytest.raises(fm.FmoeError):
        p.plan([-1])


@pytest.mark.parametrize("S,E,K,T,keep", [(16, 64, 4, 1, 1), (8, 64, 4, 1, 0), (32, 512, 4, 4, 1),
                                          (128, 512, 4, 1, 1), (12, 40, 10, 1, 0)])
def test_plan_matches_reference_lru_under_zipf(fm, S, E, K, T, keep):
    rng = np.random.default_rng(S * 1000 + E + K + T)
    rank = rng.permutation(E)
    p_e = (rank + 1.0) ** -1.1
    p_e /= p_e.sum()
    ours, ref = pool(fm, S, E), RefLRU(S, E)
    for step in range(300):
        ids = []
        for _ in range(T):
            ids += list(rng.choice(E, size=K, replace=False, p=p_e))
        want = ref.plan([int(i) for i in ids], keep)
        if want is None:
            with pytest.raises(fm.FmoeError):
                ours.plan(ids, keep)
            continue
        assert ours.plan(ids, keep) == want, step
    st = ours.stats()
    assert (st["hits"], st["misses"]) == (ref.hits, ref.misses)


def test_slot_logits_keep_the_picks_only(fm):
    p = pool(fm, 6, 10)
    ids = np.array([[7, 2], [2, 9]], dtype=np.int32)
    slots, _ = p.plan(ids.flatten().tolist())
    slots = np.array(slots, dtype=np.int32).reshape(2, 2)
    logits = np.arange(20, dtype=np.float32).reshape(2, 10) * 0.5 - 3.0
    sl = p.slot_logits(logits, ids, slots)
    lowest = np.finfo(np.float32).min
    for t in range(2):
        for s in range(6):
            picked = [k for k in range(2) if slots[t, k] == s]
            want = logits[t, ids[t, picked[0]]] if picked else lowest
            assert sl[t, s] == want
