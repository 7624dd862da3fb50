"""The expert cache's slot policy (host only, through colibri_moe_cache_simulate) against an independent
implementation of the rule and against closed forms.  The rule ("Colibri walkthrough" page, section 3.1:
slots keep last_used and hit_count; eviction prefers a low hit_count and an old last_used): among the slots
the current forward does not use, an empty slot first, else the smallest last_used + weight * hit_count
(hit_count = forwards that used the expert since it entered the slot), ties to the older last_used, then
the lower slot."""
import numpy as np
import pytest

import quantized_expert_ffn_bias_gb300 as coli


@pytest.fixture(scope="module", autouse=True)
def _lib():
    try:
        coli.lib()
    except (RuntimeError, OSError) as e:
        pytest.skip(f"library not built: {e}")


def reference(E, n_slots, weight, sets):
    slot_expert = [-1] * n_slots
    last = [0] * n_slots
    cnt = [0] * n_slots
    where = {}
    hits = misses = 0
    for step, ids in enumerate(sets, start=1):
        busy = set()
        for e in ids:
            if e in where:
                s = where[e]
                busy.add(s)
                last[s] = step
                cnt[s] += 1
                hits += 1
        for e in ids:
            if e in where:
                continue
            free = [s for s in range(n_slots) if s not in busy]
            empty = [s for s in free if slot_expert[s] < 0]
            if empty:
                s = empty[0]
            else:
                s = min(free, key=lambda i: (last[i] + weight * cnt[i], last[i], i))
            if slot_expert[s] >= 0:
                del where[slot_expert[s]]
            slot_expert[s] = e
            where[e] = s
            last[s] = step
            cnt[s] = 1
            busy.add(s)
            misses += 1
    return hits, misses


def _trace(rng, E, k, n, skew):
    p = 1.0 / np.arange(1, E + 1) ** skew
    p /= p.sum()
    perm = rng.permutation(E)
    return [sorted(perm[rng.choice(E, size=k, replace=False, p=p)].tolist()) for _ in range(n)]


@pytest.mark.parametrize("weight", [0.0, 0.5, 1.0, 3.0])
@pytest.mark.parametrize("skew", [0.0, 1.1])
def test_policy_matches_reference(weight, skew):
    rng = np.random.default_rng(int(weight * 10) + int(skew * 100))
    E, k, S = 32, 4, 10
    sets = _trace(rng, E, k, 300, skew)
    assert coli.colibri_moe_cache_simulate(E, S, weight, sets) == reference(E, S, weight, sets)


def test_policy_closed_forms():
    # the same set every step: only the first step misses
    assert coli.colibri_moe_cache_simulate(16, 4, 1.0, [[1, 5, 9]] * 10) == (27, 3)
    # enough slots for every expert: each distinct expert misses once
    rng = np.random.default_rng(0)
    sets = _trace(rng, 20, 3, 100, 0.0)
    distinct = len(set(e for s in sets for e in s))
    assert coli.colibri_moe_cache_simulate(20, 20, 2.0, sets) == (sum(map(len, sets)) - distinct, distinct)
    # plain LRU (weight 0) with one slot and a cycle of two experts: every lookup misses
    assert coli.colibri_moe_cache_simulate(4, 1, 0.0, [[0], [1]] * 5) == (0, 10)


def test_weighting_keeps_hot_experts():
    """Two hot experts, used in a warm-up and then every fourth forward, interleaved with a scan of one-off
    experts: plain LRU lets the scan flush them, the frequency weighting keeps them (the page reports higher
    hit rates for the weighted rule than for plain LRU)."""
    hot = [0, 1]
    sets = [hot] * 5
    cold = 10
    for i in range(200):
        if i % 4 == 0:
            sets.append(hot)
        else:
            sets.append([cold, cold + 1])
            cold += 2
    E = cold + 2
    h_lru, _ = coli.colibri_moe_cache_simulate(E, 4, 0.0, sets)
    h_w, _ = coli.colibri_moe_cache_simulate(E, 4, 2.0, sets)
    # LRU: the warm-up repeats and the hot forward right after them (5 x 2); weighted: also the 49 later
    # hot forwards
    assert h_lru == 2 * 5
    assert h_w == 2 * 5 + 2 * 49
    assert reference(E, 4, 2.0, sets)[0] == h_w


def test_simulate_refuses_too_few_slots():
    with pytest.raises(coli.ColiError) as e:
        coli.colibri_moe_cache_simulate(8, 2, 0.0, [[0, 1, 2]])
    assert e.value.status == coli.COLI_EUNSUPPORTED
