"""Compare a CUDA walk with the CPU oracle, element by element.

The rule (from the walk's numerics: fp32 accumulation in any order on the GPU,
an fp64 sum in the oracle, then two bf16 roundings on both sides):

* logits: a GPU logit passes if it is within 1 bf16 ulp of the oracle logit
  (ulp taken at the larger magnitude), or if it equals bf16(base + b') where
  b' is the other bf16 neighbour of the exact projection (an fp32
  accumulation may legitimately round the bias to either neighbour when the
  exact value sits near a rounding boundary);
* tokens: step by step, with the oracle fed the GPU's previous token (teacher
  forcing), the GPU token must be the oracle's argmax, except at a near-tie:
  greedy, the GPU token's oracle logit is within 2 bf16 ulp of the maximum;
  sampled, its oracle score is within the fp32 error bound of the two scores
  (logit error / T + 2^-18 (1 + |g|) + 2 fp32 ulp, for each of the two).
"""
import math

import numpy as np

import oracle
import synth


def bf16_vals(h):
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def bf16_ulp(x):
    """Spacing of bf16 at |x| (normal range; 2^-133 below it)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    ulp = np.exp2(e - 7)
    return np.where(a >= 2.0**-126, ulp, 2.0**-133)


def f32_ulp(x):
    return np.spacing(np.abs(np.asarray(x, dtype=np.float32))).astype(np.float64)


def _other_neighbour_logit(O, u_bits, W2, base_bits, v):
    """bf16(base + b') with b' the other bf16 neighbour of the exact W2[v].u."""
    u = bf16_vals(u_bits)
    acc = float(np.dot(bf16_vals(W2[v]), u))
    n1 = int(O.bf16_rne(np.array([acc]))[0])
    v1 = bf16_vals([n1])[0]
    if v1 == acc:
        return None
    # neighbour on the other side of acc
    step = math.copysign(1, acc - v1)
    if v1 == 0:
        n2 = 0x0001 if step > 0 else 0x8001
    else:
        away = (acc - v1) * v1 > 0      # moving away from zero
        n2 = n1 + 1 if away else n1 - 1
    other = bf16_vals([n2])[0]
    return int(O.bf16_rne(np.array([bf16_vals([base_bits])[0] + other]))[0])


class Report:
    def __init__(self):
        self.logits_checked = 0
        self.logits_exact = 0
        self.logits_ulp = 0
        self.logits_neighbour = 0
        self.steps_checked = 0
        self.steps_exact = 0
        self.near_ties = 0
        self.states_checked = 0
        self.states_exact = 0
        self.states_flipped = 0
        self.failures = []

    def ok(self):
        return not self.failures

    def __repr__(self):
        return ("Report(logits=%d exact=%d 1ulp=%d neighbour=%d steps=%d exact=%d near_ties=%d "
                "states=%d exact=%d flipped=%d failures=%d %s)" % (
                    self.logits_checked, self.logits_exact, self.logits_ulp,
                    self.logits_neighbour, self.steps_checked, self.steps_exact,
                    self.near_ties, self.states_checked, self.states_exact,
                    self.states_flipped, len(self.failures), self.failures[:5]))


# Group sampler (sampler = 1): the GPU's group score carries fp32 errors of a
# few ulp of |logit / T| plus the noise error (<= 0.08 of 2^-18 (1 + |g|),
# measured over every uniform) and ~1e-6 from the hardware exp2 / log2; the
# in-group pick compares running sums of fp32 weights with U2 * S, each within
# ~2e-6 S of the fp64 values.  The bounds below are about 8x those.
GROUP_SCORE_TOL = 2.0**-16
GROUP_PICK_TOL = 1e-5


# Recurrent heads: the GPU's p = M[i, :] . h is an fp32 sum 13 additions deep
# (8 in order per lane, then a 5-level butterfly), so its error is below
# 13 * 2^-24 * sum_j |M_ij h_j| < 2^-20 * sum_j |M_ij h_j|; the gate or tanh,
# the products and the add each add a few fp32 ulps of values below
# 1 + |p| + |x| + |h|.  A state element is right when it is the bf16
# rounding of some value within this bound of the exact one: for elements
# far from zero that allows only the other neighbour, and only when the exact
# value lies within the bound of the midpoint; near zero, where the bound
# spans several bf16 spacings, any rounding inside it.
CELL_TOL = 2.0**-20


def _check_states(O, rep, cell, M, W1, gh_prev, x_tok, gh, oh, oex, b, k):
    """GPU state gh [r] against the oracle's update oh / oex of the GPU's own
    previous state gh_prev (None at step 0) and token input rows x_tok ([r],
    or [3, r] for the GRU)."""
    rep.states_checked += gh.size
    same = gh == oh
    rep.states_exact += int(same.sum())
    bad = np.nonzero(~same)[0]
    if bad.size == 0:
        return
    r = gh.size
    Mv = bf16_vals(M).reshape(-1, r, r)                 # one or three gate matrices
    hp = np.zeros(r) if gh_prev is None else bf16_vals(gh_prev)
    p = np.abs(Mv @ hp).sum(axis=0)
    mass = (np.abs(Mv) @ np.abs(hp)).sum(axis=0)
    x = np.abs(bf16_vals(x_tok).reshape(-1, r)).sum(axis=0)
    gv, ov = bf16_vals(gh), bf16_vals(oh)
    for i in bad:
        ex = float(oex[i])
        tol = CELL_TOL * (mass[i] + 1.0 + p[i] + x[i] + abs(hp[i]))
        lo, hi = bf16_vals(O.bf16_rne(np.array([ex - tol, ex + tol])))   # rounding is monotone
        if lo <= gv[i] <= hi:
            rep.states_flipped += 1
            continue
        rep.failures.append(("state", b, k, int(i), float(gv[i]), float(ov[i]), ex))


def check(inputs: "synth.WalkInputs", gpu_tokens, gpu_logits=None, requests=None,
          nthreads=0, O=None, report=None, sampler=0, cell=0, M=None, gpu_states=None,
          X=None):
    """Check the GPU's tokens [B, gamma] (and logits [B, gamma, V]) for `requests`.

    sampler 0: per-token Gumbel-max; 1: group inverse-CDF (a GPU token may
    differ from the oracle's only at a group-score near-tie, then being that
    group's pick, or next to a pick whose running sum sits at the threshold).
    cell 1, 2 or 3 (a recurrent head with matrix M, bits [r, r] or [3r, r],
    and for the GRU the token tables X, bits [3, V, r]): gpu_states
    [B, gamma, r] are the GPU's states; each step's state is checked against
    the oracle's update of the GPU's previous state and token (see CELL_TOL),
    and the step's logits against the oracle's projection of the GPU state.
    Returns a Report; ``report.ok()`` is the verdict.
    """
    O = O or oracle.default()
    rep = report or Report()
    B, gamma, V = inputs.base.shape
    requests = list(range(B)) if requests is None else list(requests)
    W1 = synth.bits(inputs.W1)
    W2 = synth.bits(inputs.W2)
    base_all = synth.bits(inputs.base)
    gpu_tokens = np.asarray(gpu_tokens)
    for b in requests:
        T = float(inputs.temperature[b])
        toks = gpu_tokens[b].astype(np.int32)
        if np.any(toks < 0) or np.any(toks >= V):
            rep.failures.append(("token out of range", b, toks.tolist()))
            continue
        gs = None
        if cell != 0:
            gs = np.asarray(gpu_states[b]).astype(np.uint16)
            group = sampler == 1 and T != 0.0
            res = O.walk_cell(
                W1, W2, base_all[b:b + 1], np.array([inputs.anchor[b]], np.int32),
                np.array([T], np.float32), inputs.seed, cell, M=M, forced=toks[None, :],
                forced_state=gs[None], want_scores=T != 0.0 and not group,
                nthreads=nthreads, req0=b, sampler=sampler, want_groups=group, X=X)
            ot, ol, osc, ost, oex = res[:5]
            ot, ol, osc = ot[0], ol[0], (osc[0] if osc is not None else None)
            grp = tuple(g_[0] for g_ in res[5]) if group else None
        else:
            ot, ol, osc, grp = _oracle_request(O, W1, W2, base_all, inputs, b, toks, nthreads,
                                               sampler)
        rep.steps_checked += gamma
        for k in range(gamma):
            ok_row = ol[k]
            prev = int(inputs.anchor[b]) if k == 0 else int(toks[k - 1])
            if cell != 0:
                xt = X[:, prev] if cell == 3 else W1[prev]
                _check_states(O, rep, cell, M, W1, gs[k - 1] if k > 0 else None, xt,
                              gs[k], ost[0, k], oex[0, k], b, k)
            if gpu_logits is not None:
                gl = np.asarray(gpu_logits[b, k])
                u = gs[k] if cell != 0 else W1[prev]
                _check_logits(O, rep, u, W2, base_all[b, k], gl, ok_row, b, k)
            g = int(toks[k])
            if g == int(ot[k]):
                rep.steps_exact += 1
                continue
            if T != 0.0 and sampler == 1:
                gs, gp, gm = grp[0][k], grp[1][k], grp[2][k]
                o = int(ot[k])
                jo, jg = o // 8, g // 8

                def near_pick(j, tok):
                    return tok == int(gp[j]) or (gm[j] <= GROUP_PICK_TOL and
                                                 abs(tok - int(gp[j])) == 1)

                if jg == jo:
                    good = near_pick(jo, g)
                else:
                    tol = GROUP_SCORE_TOL * (2.0 + abs(float(gs[jo])) + abs(float(gs[jg])))
                    good = float(gs[jo]) - float(gs[jg]) <= tol and near_pick(jg, g)
                if good:
                    rep.near_ties += 1
                    continue
                rep.failures.append(("group-sampled token", b, k, g, o, float(gs[jo]),
                                     float(gs[jg])))
                continue
            if T == 0.0:
                vals = bf16_vals(ok_row)
                m1, lg = vals.max(), vals[g]
                if m1 - lg <= 2 * bf16_ulp(max(abs(m1), abs(lg))):
                    rep.near_ties += 1
                    continue
                rep.failures.append(("greedy token", b, k, g, int(ot[k]), float(m1), float(lg)))
            else:
                s = osc[k].astype(np.float64)
                o = int(ot[k])
                lv = bf16_vals(ok_row)

                def tol(v):
                    gv = s[v] - lv[v] / T
                    dl = 0.0
                    if gpu_logits is not None:
                        dl = abs(bf16_vals([gpu_logits[b, k, v]])[0] - lv[v]) / T
                    return dl + 2.0**-18 * (1 + abs(gv)) + 2 * f32_ulp(s[v])

                if s[o] - s[g] <= tol(o) + tol(g):
                    rep.near_ties += 1
                    continue
                rep.failures.append(("sampled token", b, k, g, o, float(s[o]), float(s[g])))
    return rep


def check_all_tokens(inputs: "synth.WalkInputs", gpu_tokens, nthreads=0, O=None, sampler=0):
    """Every request's tokens, teacher-forced, at any size: one tokens-only
    oracle walk of the whole batch (the oracle fed the GPU's previous token at
    every step), then the full rule of `check` (near-ties from the oracle's
    logits or scores) for the requests where some step differs.  Returns a
    Report whose steps_checked is B * gamma."""
    O = O or oracle.default()
    rep = Report()
    B, gamma, V = inputs.base.shape
    toks = np.asarray(gpu_tokens).astype(np.int32)
    bad = [b for b in range(B) if np.any(toks[b] < 0) or np.any(toks[b] >= V)]
    for b in bad:
        rep.failures.append(("token out of range", b, toks[b].tolist()))
    if bad:
        return rep
    ot = O.walk(synth.bits(inputs.W1), synth.bits(inputs.W2), synth.bits(inputs.base),
                inputs.anchor.numpy(), inputs.temperature.numpy(), inputs.seed, forced=toks,
                want_logits=False, nthreads=nthreads, sampler=sampler)[0]
    differ = [b for b in range(B) if not np.array_equal(ot[b], toks[b])]
    same = B - len(differ)
    rep.steps_checked += same * gamma
    rep.steps_exact += same * gamma
    if differ:
        check(inputs, toks, None, requests=differ, nthreads=nthreads, O=O, report=rep,
              sampler=sampler)
    return rep


def _oracle_request(O, W1, W2, base_all, inputs, b, toks, nthreads, sampler=0):
    """Oracle walk of request b alone (at request index b), teacher-forced."""
    T = float(inputs.temperature[b])
    group = sampler == 1 and T != 0.0
    res = O.walk(W1, W2, base_all[b:b + 1], np.array([inputs.anchor[b]], np.int32),
                 np.array([T], np.float32), inputs.seed, forced=toks[None, :],
                 want_scores=T != 0.0 and not group, nthreads=nthreads, req0=b,
                 sampler=sampler, want_groups=group)
    ot, ol, osc = res[0], res[1], res[2]
    grp = tuple(a[0] for a in res[3]) if group else None
    return ot[0], ol[0], (osc[0] if osc is not None else None), grp


def _check_logits(O, rep, u, W2, base_row, gl, ol, b, k):
    gv = bf16_vals(gl)
    ov = bf16_vals(ol)
    n = gv.size
    rep.logits_checked += n
    exact = gv == ov
    rep.logits_exact += int(exact.sum())
    bad = np.nonzero(~exact)[0]
    if bad.size == 0:
        return
    within = np.abs(gv[bad] - ov[bad]) <= bf16_ulp(np.maximum(np.abs(gv[bad]), np.abs(ov[bad])))
    rep.logits_ulp += int(within.sum())
    for v in bad[~within]:
        alt = _other_neighbour_logit(O, u, W2, int(base_row[v]), int(v))
        if alt is not None and alt == int(gl[v]):
            rep.logits_neighbour += 1
            continue
        rep.failures.append(("logit", b, k, int(v), float(gv[v]), float(ov[v])))
