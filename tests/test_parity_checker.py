"""The parity checker itself, on the CPU: it accepts the oracle's own walk and
rejects walks with planted mistakes (a wrong token, logits off by 2 ulp)."""
import numpy as np

import oracle
import parity
import synth


def _walk(x, **kw):
    return oracle.walk(synth.bits(x.W1), synth.bits(x.W2), synth.bits(x.base), x.anchor.numpy(),
                       x.temperature.numpy(), x.seed, **kw)


def test_accepts_the_oracle_itself():
    x = synth.make_custom(V=600, gamma=4, B=4, seed=21, temperatures=(0.0, 1.0, 0.6, 0.0),
                          noise_seed=5)
    t, lg, _ = _walk(x)
    rep = parity.check(x, t, lg)
    assert rep.ok(), rep
    assert rep.logits_exact == rep.logits_checked and rep.steps_exact == rep.steps_checked


def test_rejects_a_wrong_greedy_token():
    x = synth.make_custom(V=600, gamma=4, B=1, seed=22)
    t, lg, _ = _walk(x)
    vals = parity.bf16_vals(lg[0, 2])
    wrong = int(np.argmin(vals))          # far from the maximum
    t2 = t.copy()
    t2[0, 2] = wrong
    rep = parity.check(x, t2, None)
    assert not rep.ok() and rep.failures[0][0] == "greedy token"


def test_rejects_a_wrong_sampled_token():
    x = synth.make_custom(V=600, gamma=3, B=2, seed=23, temperatures=(1.0,), noise_seed=9)
    t, lg, sc = _walk(x, want_scores=True)
    t2 = t.copy()
    t2[1, 1] = int(np.argmin(sc[1, 1]))
    rep = parity.check(x, t2, None)
    assert not rep.ok() and rep.failures[0][0] == "sampled token"


def test_logit_tolerance():
    x = synth.make_custom(V=300, gamma=2, B=1, seed=24)
    t, lg, _ = _walk(x)
    one = lg.copy()
    v = 17
    one[0, 0, v] = one[0, 0, v] + 1     # next bf16 pattern: 1 ulp away
    assert parity.check(x, t, one).ok()
    two = lg.copy()
    two[0, 1, v] = two[0, 1, v] + 2     # 2 ulp away
    rep = parity.check(x, t, two)
    assert not rep.ok() and rep.failures[0][0] == "logit"


def test_near_tie_rule_accepts_the_runner_up_of_a_tie():
    # W2 = 0 and a base with two equal maxima: either token is a near-tie;
    # the oracle picks the smaller id, a GPU picking the other must pass.
    V, gamma = 50, 1
    x = synth.make_custom(V=V, gamma=gamma, B=1, seed=25)
    import torch
    x.W2.zero_()
    base = torch.zeros(1, gamma, V)
    base[0, 0, 10] = 3.0
    base[0, 0, 20] = 3.0 + 2.0**-6       # 1 bf16 ulp above at 3.0
    x.base = base.to(torch.bfloat16)
    t, lg, _ = _walk(x)
    assert int(t[0, 0]) == 20
    rep = parity.check(x, np.array([[10]], np.int32), lg)
    assert rep.ok() and rep.near_ties == 1


def test_group_sampler_accepts_the_oracle_itself():
    x = synth.make_custom(V=603, gamma=4, B=4, seed=25, temperatures=(0.6, 1.0, 0.0, 1.0),
                          noise_seed=6)
    t, lg, _ = _walk(x, sampler=1)
    rep = parity.check(x, t, lg, sampler=1)
    assert rep.ok(), rep
    assert rep.steps_exact == rep.steps_checked


def test_group_sampler_rejects_a_token_of_another_group():
    x = synth.make_custom(V=603, gamma=3, B=2, seed=26, temperatures=(1.0,), noise_seed=10)
    O = oracle.default()
    t, lg, _, grp = O.walk(synth.bits(x.W1), synth.bits(x.W2), synth.bits(x.base),
                           x.anchor.numpy(), x.temperature.numpy(), x.seed, sampler=1,
                           want_groups=True)
    # the pick of the group with the lowest score: far from a near-tie
    k = 1
    j = int(np.argmin(grp[0][1, k]))
    t2 = t.copy()
    t2[1, k] = int(grp[1][1, k, j])
    rep = parity.check(x, t2, None, sampler=1)
    assert not rep.ok() and rep.failures[0][0] == "group-sampled token"
    # and the Gumbel-max rule does not accept the group sampler's walk wholesale
    assert not parity.check(x, t, None, sampler=0).ok()


# ------------------------------------------------------- recurrent heads --

def _cell_walk(x, cell, M):
    return oracle.walk_cell(synth.bits(x.W1), synth.bits(x.W2), synth.bits(x.base),
                            x.anchor.numpy(), x.temperature.numpy(), x.seed, cell, M=M)


def test_cell_accepts_the_oracle_itself():
    x = synth.make_custom(V=500, gamma=4, B=3, seed=25, temperatures=(0.0, 1.0, 0.6),
                          noise_seed=6)
    M = synth.bits(synth.make_cell_matrix(7))
    for cell in (1, 2):
        t, lg, _, st, _ = _cell_walk(x, cell, M)
        rep = parity.check(x, t, lg, cell=cell, M=M, gpu_states=st)
        assert rep.ok(), rep
        assert rep.states_exact == rep.states_checked == 3 * 4 * 256


def test_cell_rejects_a_wrong_state_element():
    x = synth.make_custom(V=500, gamma=3, B=1, seed=26)
    M = synth.bits(synth.make_cell_matrix(8))
    for cell in (1, 2):
        t, lg, _, st, ex = _cell_walk(x, cell, M)
        st2 = st.copy()
        i = int(np.argmax(np.abs(ex[0, 1])))   # a large element: far from any midpoint? flip it
        st2[0, 1, i] = st2[0, 1, i] + 1        # the next bf16 pattern
        rep = parity.check(x, t, None, cell=cell, M=M, gpu_states=st2)
        assert not rep.ok() and any(f[0] == "state" for f in rep.failures), rep


def test_cell_accepts_a_flip_at_a_midpoint_only():
    # gated head, M = 0: h_0 = x / 2 exactly, so no flip is allowed at step 0;
    # an element whose exact value is a bf16 midpoint allows either neighbour
    x = synth.make_custom(V=300, gamma=2, B=1, seed=27)
    M = np.zeros((256, 256), np.uint16)
    t, lg, _, st, ex = _cell_walk(x, 1, M)
    st2 = st.copy()
    st2[0, 0, 5] ^= 1                          # a flip where the value is exact
    rep = parity.check(x, t, None, cell=1, M=M, gpu_states=st2)
    assert not rep.ok()
    # step 1: (h_0 + x_1) / 2 is a midpoint wherever the sum needs one more bit
    mids = [i for i in range(256)
            if parity.bf16_vals(st[0, 1, i:i + 1])[0] != ex[0, 1, i] and ex[0, 1, i] != 0]
    assert mids, "expected a rounded element at step 1"
    i = mids[0]
    lo_hi = sorted([int(st[0, 1, i]), int(st[0, 1, i]) + 1, int(st[0, 1, i]) - 1],
                   key=lambda h: abs(parity.bf16_vals([h])[0] - ex[0, 1, i]))
    other = lo_hi[1]                            # the other neighbour of the exact value
    st3 = st.copy()
    st3[0, 1, i] = other
    rep = parity.check(x, t, None, cell=1, M=M, gpu_states=st3)
    assert rep.ok() and rep.states_flipped == 1, rep


def test_cell_with_group_sampler_accepts_the_oracle_itself():
    x = synth.make_custom(V=400, gamma=3, B=3, seed=28, temperatures=(0.0, 1.0, 0.6),
                          noise_seed=8)
    M = synth.bits(synth.make_cell_matrix(9))
    t, lg, _, st, _ = oracle.walk_cell(synth.bits(x.W1), synth.bits(x.W2), synth.bits(x.base),
                                       x.anchor.numpy(), x.temperature.numpy(), x.seed, 2, M=M,
                                       sampler=1)
    rep = parity.check(x, t, lg, cell=2, M=M, gpu_states=st, sampler=1)
    assert rep.ok() and rep.steps_exact == rep.steps_checked, rep


def test_gru_accepts_the_oracle_and_rejects_a_wrong_state():
    x = synth.make_custom(V=420, gamma=4, B=2, seed=29, temperatures=(0.0, 1.0), noise_seed=3)
    M = synth.bits(synth.make_cell_matrix(10, rows=768))
    X = synth.bits(synth.make_cell_tables(420, 11))
    t, lg, _, st, ex = oracle.walk_cell(synth.bits(x.W1), synth.bits(x.W2), synth.bits(x.base),
                                        x.anchor.numpy(), x.temperature.numpy(), x.seed, 3,
                                        M=M, X=X)
    rep = parity.check(x, t, lg, cell=3, M=M, X=X, gpu_states=st)
    assert rep.ok() and rep.states_exact == rep.states_checked, rep
    st2 = st.copy()
    i = int(np.argmax(np.abs(ex[1, 2])))
    st2[1, 2, i] = st2[1, 2, i] + 1
    rep = parity.check(x, t, None, cell=3, M=M, X=X, gpu_states=st2)
    assert not rep.ok() and any(f[0] == "state" for f in rep.failures), rep


def test_every_request_check_accepts_the_oracle_and_rejects_planted_tokens():
    """check_all_tokens (the tokens-only, whole-batch check used at full size)
    passes the oracle's own walk, counts every step, and catches a wrong token
    in any request, greedy or sampled."""
    x = synth.make_custom(V=700, gamma=5, B=9, seed=25, temperatures=(0.0, 0.6, 1.0),
                          noise_seed=11)
    t, _, sc = _walk(x, want_logits=False, want_scores=True)
    rep = parity.check_all_tokens(x, t)
    assert rep.ok() and rep.steps_checked == 9 * 5 and rep.steps_exact == 9 * 5, rep
    for b, k in ((0, 3), (4, 1), (8, 4)):          # greedy, sampled at 0.6, sampled at 1.0
        t2 = t.copy()
        t2[b, k] = int(np.argmin(sc[b, k])) if x.temperature[b] > 0 else \
            int(np.argmin(parity.bf16_vals(_walk(x)[1][b, k])))
        rep = parity.check_all_tokens(x, t2)
        assert not rep.ok() and rep.failures[0][1] == b and rep.failures[0][2] == k, rep
    t3 = t.copy()
    t3[2, 0] = x.base.shape[2]                     # out of range
    assert parity.check_all_tokens(x, t3).failures[0][0] == "token out of range"


def test_state_rule_near_zero_takes_any_rounding_within_the_bound():
    # a state element near zero, where the fp32 error bound 2^-20 spans many
    # bf16 spacings: a rounding of any value within the bound passes, one
    # beyond it fails (no previous state, zero inputs: the bound is 2^-20)
    O = oracle.default()
    r = 256
    M = np.zeros((r, r), np.uint16)
    x_tok = np.zeros(r, np.uint16)
    ex = np.full(r, 3.0e-7)
    oh = O.bf16_rne(ex)
    for shift, ok in ((0.9 * parity.CELL_TOL, True), (-0.9 * parity.CELL_TOL, True),
                      (3.0 * parity.CELL_TOL, False)):
        gh = oh.copy()
        gh[7] = O.bf16_rne(np.array([3.0e-7 + shift]))[0]
        assert gh[7] != oh[7]
        rep = parity.Report()
        parity._check_states(O, rep, 1, M, None, None, x_tok, gh, oh, ex, 0, 0)
        assert rep.ok() == ok, (shift, rep)
