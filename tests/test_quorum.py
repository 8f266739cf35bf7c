"""Cyclic quorum-set decomposition: the host-side set check and schedule (no GPU).

The properties are checked against the definition written out here independently of the library:
a perfect difference set modulo c has every non-zero residue exactly once among its ordered
differences; subproblem s (base-c digits s_e) owns the chunks whose digits t_e lie in s_e + D; the
schedule must compute every needed (query chunk, key chunk) pair exactly once, inside a subproblem
that owns both chunks.
"""
import itertools

import pytest

cq = pytest.importorskip("exact_long_context_tcgen05_gb300")

# Perfect difference sets (Singer sets of prime-power orders 1, 2, 3, 4, 5), checked below.
SETS = {3: (0, 1), 7: (0, 1, 3), 13: (0, 1, 3, 9), 21: (0, 1, 4, 14, 16), 31: (0, 1, 3, 8, 12, 18)}


def is_perfect_difference_set(c, D):
    diffs = [(b - a) % c for a, b in itertools.permutations(D, 2)]
    return len(set(D)) == len(D) and sorted(diffs) == list(range(1, c))


def digits(t, c, itr):
    out = []
    for _ in range(itr):
        out.append(t % c)
        t //= c
    return out


def owned_chunks(s, c, D, itr):
    """Chunks of subproblem s by the definition: every digit t_e in s_e + D (mod c)."""
    sd = digits(s, c, itr)
    per_digit = [[(sd[e] + a) % c for a in D] for e in range(itr)]
    out = set()
    for combo in itertools.product(*per_digit):
        out.add(sum(x * c ** e for e, x in enumerate(combo)))
    return out


@pytest.mark.parametrize("c", sorted(SETS))
def test_registered_sets_are_perfect_difference_sets(c):
    D = SETS[c]
    assert is_perfect_difference_set(c, D)
    assert cq.cqsa_quorum_check(c, D) == cq.CQSA_OK


@pytest.mark.parametrize("c,D", [(7, (0, 1, 2)), (8, (0, 1, 3)), (7, (0, 1, 1)), (7, (0, 1, 7)), (13, (0, 1, 3, 8)),
                                 (6, (0, 1, 3))])
def test_invalid_sets_rejected(c, D):
    assert not is_perfect_difference_set(c, D)
    with pytest.raises(cq.CqsaError):
        cq.cqsa_quorum_check(c, D)


@pytest.mark.parametrize("c,itr", [(3, 1), (3, 2), (3, 3), (7, 1), (7, 2), (13, 1), (31, 1)])
@pytest.mark.parametrize("causal", [True, False])
def test_schedule_covers_every_pair_once(c, itr, causal):
    D = SETS[c]
    T = c ** itr
    for n_chunks in sorted({T, max(1, T - 1), max(1, T // 2 + 1)}):
        sched = cq.cqsa_quorum_schedule(c, D, itr, n_chunks, causal)
        pairs = [(q, k) for _, q, k in sched]
        need = [(q, k) for q in range(n_chunks) for k in range(n_chunks) if (k <= q or not causal)]
        assert sorted(pairs) == sorted(need), "every needed pair exactly once"
        owned = {}
        for s, q, k in sched:
            assert 0 <= s < T
            if s not in owned:
                owned[s] = owned_chunks(s, c, D, itr)
            assert q in owned[s] and k in owned[s], (s, q, k)
        assert [s for s, _, _ in sched] == sorted(s for s, _, _ in sched), "grouped by subproblem"


@pytest.mark.parametrize("c,itr", [(3, 2), (7, 1), (7, 2), (13, 1)])
def test_subproblem_sizes_match_the_cost_model(c, itr):
    """Each subproblem owns l^itr of the c^itr chunks and each chunk lies in l^itr subproblems, so the
    subproblems together cover c^itr * (l^itr)^2 chunk pairs: (l^2/c)^itr of all (c^itr)^2 pairs."""
    D = SETS[c]
    l, T = len(D), c ** itr
    count = [0] * T
    total = 0
    for s in range(T):
        own = owned_chunks(s, c, D, itr)
        assert len(own) == l ** itr
        total += len(own) ** 2
        for t in own:
            count[t] += 1
    assert all(x == l ** itr for x in count)
    assert total * c ** itr == (l * l) ** itr * T * T


def test_schedule_rejects_bad_depth():
    with pytest.raises(cq.CqsaError):
        cq.cqsa_quorum_schedule(7, (0, 1, 3), 0, 7, True)
    with pytest.raises(cq.CqsaError):
        cq.cqsa_quorum_schedule(7, (0, 1, 3), 1, 8, True)  # more chunks than c^itr
    with pytest.raises(cq.CqsaError):
        cq.cqsa_quorum_schedule(7, (0, 1, 3), 9, 7, True)  # c^itr beyond the supported range
