"""The expert cache's host planning (k3moe_cache_plan / k3moe_cache_publish), without a GPU.

The policy, after the pages' LRU cache for the experts ("kimi-k3-in-c" README, Part II
section 12): a slot holds an expert, is empty, or is in flight; a call marks its resident
experts used, then reserves a slot for each missing expert in ascending expert order (an
empty slot first, else the least recently used slot that the call does not use and that is
not in flight), and publishes what arrived.  A small Python model of those rules is run side
by side with the library on random call sequences; the state (which slot holds which expert,
each slot's last use) and every planned copy must agree.
"""
import numpy as np
import pytest

import mxfp4_routed_expert_gemv_gb300 as k3

EMPTY, INFLIGHT = k3.SLOT_EMPTY, k3.SLOT_INFLIGHT


class Model:
    def __init__(self, E, C):
        self.E, self.C = E, C
        self.expert_of = [EMPTY] * C
        self.used_at = [0] * C
        self.clock = 0

    def slot_of(self, e):
        for s in range(self.C):
            if self.expert_of[s] == e:
                return s
        return -1

    def plan(self, idx):
        valid = [e for e in idx if 0 <= e < self.E]
        distinct = sorted(set(valid))
        inflight = sum(1 for v in self.expert_of if v == INFLIGHT)
        if len(distinct) + inflight > self.C:
            return None
        now = self.clock + 1
        missing = []
        for e in distinct:
            s = self.slot_of(e)
            if s >= 0:
                self.used_at[s] = now
            else:
                missing.append(e)
        fetch = []
        for e in missing:
            empties = [s for s in range(self.C) if self.expert_of[s] == EMPTY]
            if empties:
                v = empties[0]
            else:
                cands = [s for s in range(self.C) if self.expert_of[s] >= 0 and self.used_at[s] < now]
                v = min(cands, key=lambda s: (self.used_at[s], s))
            self.expert_of[v] = INFLIGHT
            self.used_at[v] = now
            fetch.append((e, v))
        self.clock = now
        slot_of = {e: v for e, v in fetch}
        slot_idx = [(slot_of[e] if e in slot_of else self.slot_of(e)) if 0 <= e < self.E else -1 for e in idx]
        return slot_idx, fetch

    def publish(self, fetch, n_ok):
        for j, (e, s) in enumerate(fetch):
            self.expert_of[s] = e if j < n_ok else EMPTY


def _check_state(cache, model):
    assert cache.expert_of.tolist() == model.expert_of
    assert cache.used_at.astype(np.int64).tolist() == model.used_at
    assert cache.clock == model.clock
    for e in range(model.E):
        s = model.slot_of(e)
        if s >= 0:
            assert cache.slot_of[e] == s
        elif e not in [x for x in model.expert_of if x >= 0]:
            assert cache.slot_of[e] == -1 or model.expert_of[cache.slot_of[e]] == INFLIGHT


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_plan_matches_the_policy_on_random_calls(seed):
    rng = np.random.default_rng(seed)
    E, C = 40, 12
    cache = k3.ExpertCache(E, C)
    model = Model(E, C)
    hot = rng.choice(E, size=8, replace=False)
    for call in range(300):
        n = int(rng.integers(1, 24))
        # skewed: most indices from a hot set, some anywhere, a few out of range
        idx = np.where(rng.random(n) < 0.7, rng.choice(hot, size=n), rng.integers(0, E, size=n))
        if rng.random() < 0.1:
            idx[rng.integers(0, n)] = rng.choice([-1, E, E + 7])
        idx = idx.astype(np.int32)
        want = model.plan(idx.tolist())
        if want is None:
            before = (cache.expert_of.copy(), cache.slot_of.copy(), cache.used_at.copy(), cache.clock)
            with pytest.raises(k3.K3moeError) as ei:
                cache.plan(idx)
            assert ei.value.status == 2
            after = (cache.expert_of, cache.slot_of, cache.used_at, cache.clock)
            for a, b in zip(before[:3], after[:3]):
                assert np.array_equal(a, b), "a refused plan changed the state"
            assert before[3] == after[3]
            continue
        slot_idx, fe, fs = cache.plan(idx)
        assert slot_idx.tolist() == want[0]
        assert list(zip(fe.tolist(), fs.tolist())) == want[1]
        n_ok = len(fe) if rng.random() > 0.05 else int(rng.integers(0, len(fe) + 1))
        cache.publish(fe, fs, n_ok)
        model.publish(want[1], n_ok)
        _check_state(cache, model)


def test_first_call_fills_empty_slots_in_expert_order_and_repeat_fetches_nothing():
    cache = k3.ExpertCache(20, 8)
    slot_idx, fe, fs = cache.plan(np.array([9, 3, 17, 3, 5], np.int32))
    assert fe.tolist() == [3, 5, 9, 17] and fs.tolist() == [0, 1, 2, 3]
    assert slot_idx.tolist() == [2, 0, 3, 0, 1]
    cache.publish(fe, fs)
    slot_idx, fe, fs = cache.plan(np.array([17, 9, 5, 3], np.int32))
    assert fe.size == 0 and slot_idx.tolist() == [3, 2, 1, 0]
    cache.publish(fe, fs)


def test_least_recently_used_slot_is_evicted_never_one_the_call_uses():
    cache = k3.ExpertCache(10, 3)
    for e in (0, 1, 2):  # slots 0, 1, 2 used at clocks 1, 2, 3
        _, fe, fs = cache.plan(np.array([e], np.int32))
        cache.publish(fe, fs)
    _, fe, fs = cache.plan(np.array([0], np.int32))  # expert 0 used again: clock 4
    cache.publish(fe, fs)
    _, fe, fs = cache.plan(np.array([5, 2], np.int32))  # 1 is the oldest; 2 is in this call
    assert fe.tolist() == [5] and fs.tolist() == [1]
    cache.publish(fe, fs)
    assert cache.expert_of.tolist() == [0, 5, 2] and cache.slot_of[1] == -1


def test_more_experts_than_slots_is_refused_and_in_flight_slots_are_kept():
    cache = k3.ExpertCache(10, 4)
    with pytest.raises(k3.K3moeError):
        cache.plan(np.arange(5, dtype=np.int32))
    assert cache.expert_of.tolist() == [EMPTY] * 4 and cache.clock == 0
    _, fe, fs = cache.plan(np.array([1, 2], np.int32))  # not published: two slots in flight
    assert (cache.expert_of == INFLIGHT).sum() == 2
    with pytest.raises(k3.K3moeError):
        cache.plan(np.array([3, 4, 5], np.int32))  # 3 + 2 in flight > 4
    slot_idx, fe2, fs2 = cache.plan(np.array([3, 4], np.int32))
    assert sorted(fs2.tolist()) == sorted(set(range(4)) - set(fs.tolist()))
    cache.publish(fe, fs, 1)  # the second copy failed: its slot is empty again
    cache.publish(fe2, fs2)
    assert cache.expert_of[fs[0]] == 1 and cache.expert_of[fs[1]] == EMPTY
    assert cache.slot_of[2] == -1


def test_invalid_indices_map_to_minus_one_and_are_not_fetched():
    cache = k3.ExpertCache(6, 3)
    slot_idx, fe, fs = cache.plan(np.array([-1, 6, 2, 100, 2], np.int32))
    assert slot_idx.tolist() == [-1, -1, 0, -1, 0] and fe.tolist() == [2]


def test_argument_checks():
    with pytest.raises(k3.K3moeError) as ei:
        k3.ExpertCache(4, 5)  # more slots than experts: refused at the reset
    assert ei.value.status == 1
    cache = k3.ExpertCache(4, 2)
    with pytest.raises(k3.K3moeError):
        cache.publish(np.array([7], np.int32), np.array([0], np.int32))  # no such expert
