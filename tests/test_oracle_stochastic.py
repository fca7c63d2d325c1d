"""Pins for the oracle's stochastic (rejection-sampling) verification.

Against: small cases worked by hand (each acceptance threshold, residual and
inversion written out below), the greedy limit (a one-hot target turns the walk
into the greedy walk of the independent greedy oracle), and the property the
pages claim for the method: the emitted tokens follow the target distribution
whatever the draft distribution is (sampled; on the three-sibling case below a
walk that forgets to take a rejected draft out of the draft distribution puts
0.54 on a token whose target probability is 0.3).
"""
import numpy as np
import pytest

from oracle import stochastic as S
from oracle import verify as GV
import workloads as W


def _logits(*rows):
    """fp32 logits whose softmax at T=1 is each given probability row."""
    return np.log(np.asarray(rows, np.float64)).astype(np.float32)


def _walk(parent, draft, logits, q, coins, T=1.0, max_depth=4):
    path, L, bonus, st, am, sm = S.walk_stochastic(parent, draft, logits, np.asarray(q, np.float64), coins, T,
                                                   max_depth)
    return path.tolist(), L, bonus, st


# p_root = [.5 .3 .2], q_root = [.2 .6 .2]; the root's children carry tokens 1 then 2.
P0, Q0 = [0.5, 0.3, 0.2], [0.2, 0.6, 0.2]


def test_hand_both_rejected():
    # child 1 (x=1): accept iff coin*0.6 < 0.3; coin 0.6 rejects.  Residual
    # max(p - q, 0) = [.3 0 0] -> r = [1 0 0]; q' = [.2 0 .2]/.4 = [.5 0 .5].
    # child 2 (x=2): coin*0.5 < r(2) = 0 never holds.  Residual stays [1 0 0]:
    # the bonus is token 0 whatever coins[0] is.
    for c0 in (0.0, 0.5, 0.999):
        got = _walk([-1, 0, 0], [0, 1, 2], _logits(P0, P0, P0), [Q0] * 3, [c0, 0.6, 0.3])
        assert got == ([0, -1, -1, -1, -1], 0, 0, 0)


def test_hand_first_accepted_then_leaf_bonus():
    # coin 0.4: 0.24 < 0.3 accepts child 1, a leaf; the bonus is drawn from
    # p_1 = [.1 .6 .3] (cumulative .1 .7 1): coins[0] = .65 -> 1, .05 -> 0, .75 -> 2.
    lg = _logits(P0, [0.1, 0.6, 0.3], P0)
    for c0, tok in ((0.65, 1), (0.05, 0), (0.75, 2)):
        assert _walk([-1, 0, 0], [0, 1, 2], lg, [Q0] * 3, [c0, 0.4, 0.9]) == ([0, 1, -1, -1, -1], 1, tok, 0)


def test_hand_second_sibling_accepted():
    # children carry tokens 1 then 0.  Child 1 rejected as above, so r = [1 0 0],
    # q' = [.5 0 .5]; child 2 (x=0): coin*0.5 < 1 always accepts.  Its bonus
    # comes from p_2 = [.25 .25 .5] (cumulative .25 .5 1): coins[0] = .45 -> 1.
    lg = _logits(P0, P0, [0.25, 0.25, 0.5])
    assert _walk([-1, 0, 0], [0, 1, 0], lg, [Q0] * 3, [0.45, 0.6, 0.99]) == ([0, 2, -1, -1, -1], 1, 1, 0)


def test_hand_partial_residual_and_draft_renormalisation():
    # p = [.5 .3 .2], q = [.1 .2 .7]; children carry tokens 2 then 1.
    # child 1 (x=2): accept iff coin*0.7 < 0.2; coin .5 rejects.  Residual
    # max(p - q, 0) = [.4 .1 0] -> r = [.8 .2 0]; q' = [.1 .2 0]/.3 = [1/3 2/3 0].
    # child 2 (x=1): accept iff coin*(2/3) < 0.2, i.e. coin < 0.3.
    p, q = [0.5, 0.3, 0.2], [0.1, 0.2, 0.7]
    lg = _logits(p, p, p)
    assert _walk([-1, 0, 0], [0, 2, 1], lg, [q] * 3, [0.1, 0.5, 0.25])[:2] == ([0, 2, -1, -1, -1], 1)
    # coin .35 rejects (a draft distribution left unrenormalised, [.1 .2 0], or
    # left unchanged would have accepted).  Residual max([.8 .2 0] - [1/3 2/3 0], 0)
    # = [.467 0 0] -> r = [1 0 0]: the bonus is 0.
    assert _walk([-1, 0, 0], [0, 2, 1], lg, [q] * 3, [0.99, 0.5, 0.35]) == ([0, -1, -1, -1, -1], 0, 0, 0)
    # one child only (x=2), rejected: the bonus is drawn from r = [.8 .2 0]
    # (cumulative .8 1): coins[0] = .85 -> 1, .75 -> 0 (p itself would give 2 and 1).
    lg2 = _logits(p, p)
    assert _walk([-1, 0], [0, 2], lg2, [q] * 2, [0.85, 0.5])[2] == 1
    assert _walk([-1, 0], [0, 2], lg2, [q] * 2, [0.75, 0.5])[2] == 0


def test_hand_temperature():
    # logits [0, ln 2, ln 4]: T=1 -> p = [1 2 4]/7 (cumulative .143 .429 1);
    # T=0.5 -> [1 4 16]/21 (.048 .238 1); T=2 -> [1 1.414 2]/4.414 (.227 .547 1).
    # coins[0] = 0.25 gives 1, 2, 1.
    lg = np.array([[0.0, np.log(2.0), np.log(4.0)]], np.float32)
    for T, tok in ((1.0, 1), (0.5, 2), (2.0, 1)):
        assert _walk([-1], [0], lg, [[1 / 3] * 3], [0.25], T=T) == ([0, -1, -1, -1, -1], 0, tok, 0)


def test_hand_point_mass_draft_and_zero_coin():
    # q_root = one-hot at token 1, so after child 1 is rejected no draft mass is
    # left: q' = 0 and a later child is accepted iff the residual gives its token
    # any mass.  p = [.2 .5 .3]: child 1 (x=1) accepts iff coin*1 < .5; coin .7
    # rejects; residual max(p - [0 1 0], 0) = [.2 0 .3] -> r = [.4 0 .6].
    p, q = [0.2, 0.5, 0.3], [0.0, 1.0, 0.0]
    lg = _logits(p, p, p)
    assert _walk([-1, 0, 0], [0, 1, 2], lg, [q] * 3, [0.0, 0.7, 0.9])[:2] == ([0, 2, -1, -1, -1], 1)
    # a single child: the bonus from r = [.4 0 .6] with coins[0] = 0 is the first
    # token with mass, 0; with coins[0] = .4 it is 2 (cumulative .4 .4 1).
    assert _walk([-1, 0], [0, 1], lg[:2], [q] * 2, [0.0, 0.7])[2] == 0
    assert _walk([-1, 0], [0, 1], lg[:2], [q] * 2, [0.4, 0.7])[2] == 2


def test_invalid_tree_and_path_too_long():
    lg = _logits(P0, P0, P0)
    assert _walk([-1, 2, 0], [0, 1, 2], lg, [Q0] * 3, [0.5, 0.1, 0.1]) == ([-1] * 5, 0, 0, -3)
    assert _walk([-1, 0, 0], [0, 1, 3], lg, [Q0] * 3, [0.5, 0.1, 0.1]) == ([-1] * 5, 0, 0, -3)
    assert _walk([-1, 0, 0], [0, -1, 2], lg, [Q0] * 3, [0.5, 0.1, 0.1]) == ([-1] * 5, 0, 0, -3)
    assert _walk([-1, 0, 0], [7, 1, 2], lg, [Q0] * 3, [0.5, 0.99, 0.99])[3] == 0   # the root's token is unused
    # chain 0 -> 1 -> 2 with one-hot-ish acceptance (coin 0) accepts both drafts
    assert _walk([-1, 0, 1], [0, 1, 1], lg, [Q0] * 3, [0.65, 0.0, 0.0])[:2] == ([0, 1, 2, -1, -1], 2)
    path, L, bonus, st = _walk([-1, 0, 1], [0, 1, 1], lg, [Q0] * 3, [0.65, 0.0, 0.0], max_depth=1)
    assert (path, L, st) == ([-1, -1], 2, -2) and bonus == 1


def test_greedy_limit_equals_greedy_walk():
    """A one-hot target (a logit 800 above the rest underflows every other
    probability to 0) accepts exactly the draft equal to the argmax and draws
    the argmax as the bonus, whatever q and the coins are."""
    g = np.random.default_rng(11)
    for trial in range(300):
        n = int(g.integers(1, 14))
        V = 6
        parent = W.tree_random_recursive(g, n)
        draft = W.draft_tokens(g, parent, V)
        lg = g.standard_normal((n, V)).astype(np.float32)
        am = g.integers(0, V, n)
        for u in range(n):   # often make the argmax one of u's children's tokens
            kids = [c for c in range(n) if parent[c] == u]
            if kids and g.random() < 0.7:
                am[u] = draft[kids[int(g.integers(0, len(kids)))]]
        lg[np.arange(n), am] += 800.0
        q = g.dirichlet(np.ones(V), n)
        coins = g.random(n)
        md = int(g.integers(0, n + 1))
        got = _walk(parent, draft, lg, q, coins, max_depth=md)
        path, L, bonus, st = GV.accept_walk(parent, draft, GV.greedy_argmax(lg), md)
        assert got == (path.tolist(), L, bonus, st), trial


def _draw_children(g, parent, q, V):
    draft = np.zeros(len(parent), np.int64)
    for u in range(len(parent)):
        kids = [c for c in range(len(parent)) if parent[c] == u]
        if kids:
            draft[kids] = g.choice(V, size=len(kids), replace=False, p=q[u])
    return draft


@pytest.mark.parametrize("seed", [0, 1])
def test_emitted_tokens_follow_target_distribution(seed):
    """The first emitted token (accepted draft or bonus) is distributed as
    p_root, and given that the walk entered child c, the next one as p_c.
    Here a node's target row depends only on its own token (as a model's next
    distribution depends on its context), so the second token given the first
    t must follow that row for t."""
    g = np.random.default_rng(100 + seed)
    V, n_samp = 5, 20000
    parent = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3])
    p_root = g.dirichlet(np.full(V, 0.7))
    p_next = g.dirichlet(np.full(V, 0.7), V)          # row t: target after token t
    q_root = g.dirichlet(np.full(V, 0.7))
    q_next = g.dirichlet(np.full(V, 0.7), V)
    first = np.zeros(V)
    second = np.zeros((V, V))
    for _ in range(n_samp):
        # per sample: rows of depth-1 nodes follow their own (yet to be drawn) token
        q = np.tile(q_root, (10, 1))
        d1 = _draw_children(g, parent[:4], q[:4], V)
        rows_p = np.tile(p_root, (10, 1))
        for c in (1, 2, 3):
            q[c] = q_next[d1[c]]
            rows_p[c] = p_next[d1[c]]
        draft = _draw_children(g, parent, q, V)
        draft[1:4] = d1[1:4]
        coins = g.random(10)
        path, L, bonus, st, _, _ = S.walk_stochastic(parent, draft, np.log(rows_p).astype(np.float32), q, coins,
                                                     1.0, 4)
        assert st == 0
        y1 = int(draft[path[1]]) if L >= 1 else bonus
        first[y1] += 1
        if L >= 1:
            y2 = int(draft[path[2]]) if L >= 2 else bonus
            second[y1, y2] += 1
    f = first / n_samp
    sigma = np.sqrt(p_root * (1 - p_root) / n_samp)
    assert np.all(np.abs(f - p_root) <= 5 * sigma + 1e-3), (f, p_root)
    for t in range(V):
        m = second[t].sum()
        if m < 500:
            continue
        ft = second[t] / m
        sig = np.sqrt(p_next[t] * (1 - p_next[t]) / m)
        assert np.all(np.abs(ft - p_next[t]) <= 5 * sig + 2e-3), (t, ft, p_next[t])


def test_single_draft_acceptance_rate():
    """One child drawn from q is accepted with probability sum_x min(p(x), q(x))."""
    g = np.random.default_rng(7)
    V, n = 6, 20000
    p = g.dirichlet(np.ones(V))
    q = g.dirichlet(np.ones(V))
    lg = np.log(np.stack([p, p])).astype(np.float32)
    hits = 0
    for _ in range(n):
        x = int(g.choice(V, p=q))
        hits += _walk([-1, 0], [0, x], lg, [q, q], g.random(2))[1]
    expect = np.minimum(p, q).sum()
    assert abs(hits / n - expect) <= 5 * np.sqrt(expect * (1 - expect) / n)


def test_batched_matches_per_tree_and_generator_contract():
    g = W.rng(3, "stoch-oracle")
    parents = np.stack([W.tree_random_levels(g, 24, 5) for _ in range(3)])
    si = W.stochastic_inputs(3, parents, 200, temperature=0.7)
    acc, L, bonus, st, m = S.verify_stochastic(si.draft, si.logits, si.q, parents, si.coins, si.temperature, 5)
    for b in range(3):
        path, l, bo, s, am, sm = S.walk_stochastic(parents[b], si.draft[b], si.logits[b], si.q[b], si.coins[b],
                                                   si.temperature, 5)
        assert acc[b].tolist() == path.tolist() and (L[b], bonus[b], st[b]) == (l, bo, s)
        # siblings distinct, every draft token has positive draft probability under its parent
        for u in range(24):
            kids = [c for c in range(24) if parents[b][c] == u]
            toks = si.draft[b][kids]
            assert len(set(toks.tolist())) == len(kids)
            assert np.all(si.q[b, u, toks] > 0)
    assert np.all((si.coins >= 0) & (si.coins < 1))
    np.testing.assert_allclose(si.q.astype(np.float64).sum(-1), 1.0, atol=1e-4)


def test_first_token_distribution_three_siblings():
    """Target and draft disagree strongly; three siblings are drawn without
    replacement from q.  The first emitted token must still follow p."""
    g = np.random.default_rng(5)
    p = np.array([0.05, 0.15, 0.3, 0.5])
    q = np.array([0.6, 0.25, 0.1, 0.05])
    lg = np.log(np.tile(p, (4, 1))).astype(np.float32)
    n = 20000
    cnt = np.zeros(4)
    for _ in range(n):
        draft = np.array([0, *g.choice(4, size=3, replace=False, p=q)])
        path, L, bonus, st, _, _ = S.walk_stochastic([-1, 0, 0, 0], draft, lg, np.tile(q, (4, 1)), g.random(4),
                                                     1.0, 3)
        cnt[int(draft[path[1]]) if L else bonus] += 1
    sigma = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(cnt / n - p) <= 5 * sigma), cnt / n
