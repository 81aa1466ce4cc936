"""Pins of the CPU oracle against things other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
if that oracle disagrees with what the pages or the mathematics fix.  The
pins are written so that a plausible slip anywhere in the oracle (a dropped
rounding, a wrong sign or index, a swapped operand, a wrong tie rule, a wrong
constant or counter layout in the noise) fails at least one of them;
``test_oracle_mutations.py`` plants such slips in copies of the oracle and
checks exactly that.

Independent references used here:
  * PyTorch's fp32 -> bf16 cast (round to nearest even) and a nearest-value
    search over the 65,536 bf16 bit patterns;
  * Triton's Philox4x32-10 (``tl.philox``), run by Triton's CPU interpreter;
  * scipy's Gumbel distribution and chi-square test;
  * exact rational arithmetic (``fractions.Fraction``) for a brute-force walk.
"""
import json
import math
import os
import subprocess
import sys
from fractions import Fraction

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")


# ------------------------------------------------------------------ bf16 ---

def _bf16_table():
    """All finite bf16 values, sorted, with their bit patterns."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        vals = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ok = np.isfinite(vals)
    bits, vals = bits[ok], vals[ok]
    # drop -0.0 so each value appears once (+0.0 kept); sign of zero handled apart
    keep = ~((vals == 0) & (bits == 0x8000))
    bits, vals = bits[keep], vals[keep]
    order = np.argsort(vals, kind="stable")
    return vals[order], bits[order]


_TABLE = None


def nearest_bf16_bits(x: float) -> int:
    """bf16 nearest to the double x, ties to the even bit pattern (search)."""
    global _TABLE
    if _TABLE is None:
        _TABLE = _bf16_table()
    vals, bits = _TABLE
    if math.isnan(x):
        return 0x7FC0
    if x == 0:
        return 0x8000 if math.copysign(1.0, x) < 0 else 0
    fx = Fraction(x)
    top = Fraction(vals[-1])                      # largest finite bf16
    half_ulp_top = Fraction(2) ** 119             # half the spacing at the top
    if fx >= top + half_ulp_top:
        return 0x7F80
    if fx <= -(top + half_ulp_top):
        return 0xFF80
    i = int(np.searchsorted(vals, x, side="left"))
    if i < len(vals) and vals[i] == x:
        return int(bits[i])
    lo, hi = i - 1, i
    dlo = fx - Fraction(vals[lo])
    dhi = Fraction(vals[hi]) - fx
    if dlo < dhi:
        pick = lo
    elif dhi < dlo:
        pick = hi
    else:
        pick = lo if (int(bits[lo]) & 1) == 0 else hi
    b = int(bits[pick])
    if b == 0 and x < 0:
        return 0x8000                             # rounds to -0
    return b


def pin_bf16_hand(O):
    """Hand cases: ties to even, a non-tie just above a tie, signs, overflow."""
    cases = [
        (1.0 + 2**-8, 0x3F80),          # tie between 1 and 1+2^-7 -> even (1.0)
        (1.0 + 3 * 2**-8, 0x3F82),      # tie between 1+2^-7 and 1+2^-6 -> 1+2^-6
        (1.0 + 2**-8 + 2**-40, 0x3F81),  # just above the tie -> up; an fp32 detour would tie
        (-2.5, 0xC020),
        (3.0, 0x4040),
        (-0.0, 0x8000),
        (0.0, 0x0000),
        (3.5e38, 0x7F80),               # above the largest finite bf16 -> inf
        (2.0**-133, 0x0001),            # smallest subnormal
        (2.0**-134, 0x0000),            # half of it: tie to even (zero)
        (3 * 2.0**-135, 0x0001),        # 0.75 of it -> up
    ]
    got = O.bf16_rne(np.array([c[0] for c in cases]))
    for (x, want), g in zip(cases, got):
        assert int(g) == want, "bf16_rne(%r) = %#06x, want %#06x" % (x, int(g), want)


def pin_bf16_vs_torch(O):
    """Every fp32 high half with tie / near-tie / random low halves vs torch."""
    hi = np.arange(65536, dtype=np.uint32) << 16
    rng = np.random.default_rng(7)
    lows = [0x0000, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x0001]
    pats = [hi | lo for lo in lows] + [hi | rng.integers(0, 65536, 65536, dtype=np.uint32)]
    x32 = np.concatenate(pats).astype(np.uint32).view(np.float32)
    x32 = x32[np.isfinite(x32)]
    want = torch.from_numpy(x32.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.bf16_rne(x32.astype(np.float64))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, "bf16_rne disagrees with torch on %d fp32 values, e.g. %r" % (
        bad.size, x32[bad[:3]])


def pin_bf16_vs_search(O):
    """Doubles that fp32 cannot hold (incl. near midpoints) vs nearest-value search."""
    rng = np.random.default_rng(11)
    xs = list(rng.standard_normal(2000) * np.exp(rng.uniform(-60, 60, 2000)))
    # midpoints of adjacent bf16 values, nudged by a few fp64 ulps either way
    b = rng.integers(0, 0x7F7F, 1000).astype(np.uint32)
    lo = (b << 16).view(np.float32).astype(np.float64)
    hi = ((b + 1) << 16).view(np.float32).astype(np.float64)
    mid = (lo + hi) / 2
    for m in mid:
        xs += [m, np.nextafter(m, np.inf), np.nextafter(m, -np.inf), -m]
    xs = np.array(xs, dtype=np.float64)
    got = O.bf16_rne(xs)
    for x, g in zip(xs, got):
        want = nearest_bf16_bits(float(x))
        assert int(g) == want, "bf16_rne(%r) = %#06x, nearest is %#06x" % (x, int(g), want)


# ---------------------------------------------------------------- Philox ---

_TRITON_SCRIPT = r"""
import json, os, sys
os.environ["TRITON_INTERPRET"] = "1"
import numpy as np, torch, triton, triton.language as tl

@triton.jit
def _k(c_ptr, seed_lo_ptr, seed_hi_ptr, out_ptr, N: tl.constexpr):
    i = tl.arange(0, N)
    c0 = tl.load(c_ptr + 4 * i + 0).to(tl.uint32)
    c1 = tl.load(c_ptr + 4 * i + 1).to(tl.uint32)
    c2 = tl.load(c_ptr + 4 * i + 2).to(tl.uint32)
    c3 = tl.load(c_ptr + 4 * i + 3).to(tl.uint32)
    k0 = tl.load(seed_lo_ptr + i).to(tl.uint32)
    k1 = tl.load(seed_hi_ptr + i).to(tl.uint32)
    a, b, c, d = tl.random.philox_impl(c0, c1, c2, c3, k0, k1, 10)
    tl.store(out_ptr + 4 * i + 0, a.to(tl.int64) & 0xFFFFFFFF)
    tl.store(out_ptr + 4 * i + 1, b.to(tl.int64) & 0xFFFFFFFF)
    tl.store(out_ptr + 4 * i + 2, c.to(tl.int64) & 0xFFFFFFFF)
    tl.store(out_ptr + 4 * i + 3, d.to(tl.int64) & 0xFFFFFFFF)

req = json.load(sys.stdin)
ctr = np.array(req["ctr"], dtype=np.int64).reshape(-1, 4)
key = np.array(req["key"], dtype=np.int64).reshape(-1, 2)
n = ctr.shape[0]
out = torch.zeros(n * 4, dtype=torch.int64)
_k[(1,)](torch.from_numpy(ctr.reshape(-1).copy()), torch.from_numpy(key[:, 0].copy()),
         torch.from_numpy(key[:, 1].copy()), out, N=n)
json.dump(out.tolist(), sys.stdout)
"""

_PHILOX_REF = None


def philox_reference():
    """(ctr, key, out) from Triton's Philox4x32-10 on the CPU interpreter."""
    global _PHILOX_REF
    if _PHILOX_REF is not None:
        return _PHILOX_REF
    rng = np.random.default_rng(3)
    n = 256
    ctr = rng.integers(0, 2**32, (n, 4), dtype=np.uint64)
    key = rng.integers(0, 2**32, (n, 2), dtype=np.uint64)
    # the walk's own layouts: small counters (v>>2, k, b, 0) and a few seeds
    ctr[:64, 1] %= 16
    ctr[:64, 2] %= 256
    ctr[:64, 3] = 0
    # the group sampler's counters (j >> 1, k, b, 1)
    ctr[64:96, 1] %= 16
    ctr[64:96, 2] %= 256
    ctr[64:96, 3] = 1
    key[:8] = [[1234, 0], [0, 0], [1, 0], [0xFFFFFFFF, 0xFFFFFFFF],
               [1234, 1], [7, 9], [2**31, 5], [42, 42]]
    env = dict(os.environ, TRITON_INTERPRET="1")
    req = json.dumps({"ctr": ctr.reshape(-1).tolist(), "key": key.reshape(-1).tolist()})
    res = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], input=req, env=env,
                         capture_output=True, text=True, timeout=600)
    if res.returncode != 0:
        raise RuntimeError("triton interpreter failed: " + res.stderr[-2000:])
    out = np.array(json.loads(res.stdout), dtype=np.uint64).reshape(n, 4)
    _PHILOX_REF = (ctr.astype(np.uint32), key.astype(np.uint32), out.astype(np.uint32))
    return _PHILOX_REF


def pin_philox_vs_triton(O):
    """Philox4x32-10 equals Triton's implementation on 256 counter/key pairs."""
    ctr, key, want = philox_reference()
    got = O.philox4x32_10(ctr, key)
    bad = np.nonzero((got != want).any(axis=1))[0]
    assert bad.size == 0, "philox differs from triton on %d of %d inputs" % (bad.size, len(ctr))


def pin_noise_layout(O):
    """Token v of request b at step k reads word v&3 of counter (v>>2, k, b, 0)."""
    ctr, key, want = philox_reference()
    for i in range(64):
        c0, k, b, _ = (int(x) for x in ctr[i])
        seed = int(key[i, 0]) | (int(key[i, 1]) << 32)
        for w in range(4):
            v = 4 * c0 + w
            if v >= 2**31:
                continue
            got = O.noise_bits(seed, b, k, v)
            assert got == int(want[i, w]), "noise bits of (b=%d,k=%d,v=%d) wrong" % (b, k, v)


def pin_uniform(O):
    """U is the midpoint of bin x>>9 of 2^23 bins: exact, inside (0,1), uniform."""
    for x, want in [(0, 2.0**-24), (0x1FF, 2.0**-24), (0x200, 3 * 2.0**-24),
                    (0xFFFFFFFF, 1 - 2.0**-24), (0x80000000, 0.5 + 2.0**-24)]:
        assert O.uniform(x) == want, "uniform(%#x) = %r, want %r" % (x, O.uniform(x), want)
    # uniformity of the walk's noise over many tokens: chi-square on 256 bins
    from scipy import stats
    us = np.array([O.uniform(O.noise_bits(99, 3, 2, v)) for v in range(65536)])
    assert us.min() > 0 and us.max() < 1
    counts = np.bincount((us * 256).astype(int), minlength=256)
    p = stats.chisquare(counts).pvalue
    assert p > 1e-4, "noise uniforms fail chi-square (p=%g)" % p


def pin_gumbel(O):
    """g = -log(-log U) follows the standard Gumbel law; g(1/e) = 0; g rises with U."""
    from scipy import stats
    assert O.gumbel(math.exp(-1.0)) == 0.0 or abs(O.gumbel(float(np.float32(math.exp(-1))))) < 1e-6
    us = (2 * np.arange(0, 2**23, 97) + 1) * 2.0**-24
    gs = np.array([O.gumbel(float(u)) for u in us])
    assert np.all(np.diff(gs) > 0), "gumbel(U) must increase with U"
    ks = stats.kstest(gs, stats.gumbel_r.cdf)
    assert ks.statistic < 2e-3, "gumbel(U) on a uniform grid is not Gumbel (D=%g)" % ks.statistic


# ------------------------------------------------------------------ walks ---

def load_hand_walk():
    """Parse tests/golden/hand_walk.txt into arrays (values as float64)."""
    W1 = {}
    W2 = {}
    base = {}
    logit = {}
    anchor = tokens = None
    with open(os.path.join(GOLDEN, "hand_walk.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tag, *rest = line.split()
            if tag == "W1":
                W1[int(rest[0])] = [float(x) for x in rest[1:]]
            elif tag == "W2":
                W2[int(rest[0])] = [float(x) for x in rest[1:]]
            elif tag == "base":
                base[int(rest[0])] = [float(x) for x in rest[1:]]
            elif tag == "logit":
                logit[int(rest[0])] = [float(x) for x in rest[1:]]
            elif tag == "anchor":
                anchor = int(rest[0])
            elif tag == "tokens":
                tokens = [int(x) for x in rest]
    return W1, W2, base, logit, anchor, tokens


def _to_bf16_bits(vals):
    t = torch.tensor(np.asarray(vals, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.tensor(np.asarray(vals, dtype=np.float32))), \
        "fixture value not representable in bf16"
    return t.view(torch.int16).numpy().view(np.uint16)


def _from_bits(h):
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def pin_hand_walk(O):
    """The hand-computed three-step walk of tests/golden/hand_walk.txt."""
    W1d, W2d, based, logitd, anchor, tokens = load_hand_walk()
    V, r, gamma = 4, 256, 3
    W1 = np.zeros((V, r), np.float32)
    W2 = np.zeros((V, r), np.float32)
    for i in range(V):
        W1[i, :2] = W1d[i]
        W2[i, :2] = W2d[i]
    base = np.array([[based[k] for k in range(gamma)]], np.float32)
    t, lg, _ = O.walk(_to_bf16_bits(W1), _to_bf16_bits(W2), _to_bf16_bits(base),
                      np.array([anchor], np.int32), np.zeros(1, np.float32), 0)
    assert list(t[0]) == tokens, "hand walk tokens %r, want %r" % (list(t[0]), tokens)
    want = np.array([logitd[k] for k in range(gamma)])
    assert np.array_equal(_from_bits(lg[0]), want), "hand walk logits %r, want %r" % (
        _from_bits(lg[0]), want)


def _fraction_walk(W1v, W2v, basev, anchor, gamma):
    """Brute force: exact transition table M[p][v], then walk by lookup.

    M[p][v] = bf16(W2[v] . W1[p]) built W1-major with exact rationals and the
    nearest-value search; logits = bf16(base + M), argmax ties to lowest id.
    """
    V = W2v.shape[0]
    M = np.zeros((V, V), np.float64)
    for p in range(V):                                   # W1-major order
        u = [Fraction(float(x)) for x in W1v[p]]
        for v in range(V):
            acc = sum((Fraction(float(w)) * uj for w, uj in zip(W2v[v], u)), Fraction(0))
            M[p, v] = _from_bits([nearest_bf16_bits(float(acc))])[0] if acc != 0 else 0.0
    prev = anchor
    toks, logits = [], []
    for k in range(gamma):
        row = np.array([_from_bits([nearest_bf16_bits(float(Fraction(float(basev[k, v])) +
                                                              Fraction(float(M[prev, v]))))])[0]
                        for v in range(V)])
        tok = int(np.argmax(row))                        # first maximum
        toks.append(tok)
        logits.append(row)
        prev = tok
    return toks, np.array(logits)


def pin_fig2_bruteforce(O):
    """The Fig. 2 shape of "Weights That Stay" (V=12, r=4, three steps), brute force."""
    V, r_used, r, gamma = 12, 4, 256, 3
    for seed in range(6):
        g = torch.Generator("cpu").manual_seed(100 + seed)
        W1 = torch.zeros(V, r)
        W2 = torch.zeros(V, r)
        W1[:, :r_used] = torch.randn(V, r_used, generator=g) / 2
        W2[:, :r_used] = torch.randn(V, r_used, generator=g)
        base = torch.randn(1, gamma, V, generator=g)
        if seed % 2:
            base = torch.round(base * 4) / 4                    # coarse: many ties
        W1b, W2b, bb = (x.to(torch.bfloat16) for x in (W1, W2, base))
        anchor = int(torch.randint(0, V, (1,), generator=g))
        bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
        t, lg, _ = O.walk(bits(W1b), bits(W2b), bits(bb), np.array([anchor], np.int32),
                          np.zeros(1, np.float32), 0)
        toks, logits = _fraction_walk(W1b.float().numpy()[:, :r_used],
                                      W2b.float().numpy()[:, :r_used],
                                      bb.float().numpy()[0], anchor, gamma)
        assert list(t[0]) == toks, "seed %d: tokens %r, brute force %r" % (seed, list(t[0]), toks)
        assert np.array_equal(_from_bits(lg[0]), logits), "seed %d: logits differ" % seed


def pin_w2_zero(O):
    """W2 = 0: logits equal base exactly and tokens are argmax(base_k), first max."""
    V, r, gamma, B = 1000, 256, 5, 3
    g = torch.Generator("cpu").manual_seed(5)
    W1 = (torch.randn(V, r, generator=g) / 16).to(torch.bfloat16)
    W2 = torch.zeros(V, r, dtype=torch.bfloat16)
    base = torch.round(torch.randn(B, gamma, V, generator=g) * 8) / 8   # ties likely
    base = base.to(torch.bfloat16)
    anchor = torch.randint(0, V, (B,), generator=g).int().numpy()
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    t, lg, _ = O.walk(bits(W1), bits(W2), bits(base), anchor, np.zeros(B, np.float32), 0)
    bf = base.float().numpy()
    # values, not bits: bf16(-0 + 0) is +0
    assert np.array_equal(_from_bits(lg), bf.astype(np.float64)), \
        "with W2 = 0 the logits must equal base"
    assert np.array_equal(t, np.argmax(bf, axis=2)), "with W2 = 0 tokens are argmax(base)"


def pin_spike(O):
    """A +40 spike at a chosen token of each step's base always wins."""
    V, r, gamma, B = 2048, 256, 6, 2
    g = torch.Generator("cpu").manual_seed(6)
    W1 = (torch.randn(V, r, generator=g) / 16).to(torch.bfloat16)
    W2 = torch.randn(V, r, generator=g).to(torch.bfloat16)
    base = torch.randn(B, gamma, V, generator=g)
    pos = torch.randint(0, V, (B, gamma), generator=g)
    for b in range(B):
        for k in range(gamma):
            base[b, k, pos[b, k]] += 40.0
    base = base.to(torch.bfloat16)
    anchor = torch.randint(0, V, (B,), generator=g).int().numpy()
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    for T in (0.0, 1.0):
        t, _, _ = O.walk(bits(W1), bits(W2), bits(base), anchor, np.full(B, T, np.float32), 9)
        assert np.array_equal(t, pos.numpy()), "spike tokens not chosen at T=%g" % T


def pin_batch_independence(O):
    """A request's walk is the same alone (at its own request index) and in a batch."""
    import synth
    x = synth.make_custom(V=777, gamma=4, B=5, seed=8, temperatures=(0.0, 1.0, 0.6))
    bits = synth.bits
    t, lg, _ = O.walk(bits(x.W1), bits(x.W2), bits(x.base), x.anchor.numpy(),
                      x.temperature.numpy(), 31)
    for b in range(5):
        tb, lb, _ = O.walk(bits(x.W1), bits(x.W2), bits(x.base[b:b + 1]),
                           x.anchor.numpy()[b:b + 1], x.temperature.numpy()[b:b + 1], 31,
                           req0=b)
        assert np.array_equal(tb[0], t[b]) and np.array_equal(lb[0], lg[b]), \
            "request %d differs alone vs in the batch" % b


def pin_permutation(O):
    """Relabelling the vocabulary relabels the tokens (on tie-free walks)."""
    import synth
    checked = 0
    for seed in range(20, 40):
        x = synth.make_custom(V=513, gamma=4, B=1, seed=seed)
        bits = synth.bits
        t, lg, _ = O.walk(bits(x.W1), bits(x.W2), bits(x.base), x.anchor.numpy(),
                          x.temperature.numpy(), 0)
        vals = _from_bits(lg[0])
        top2 = np.sort(vals, axis=1)[:, -2:]
        if np.any(top2[:, 0] == top2[:, 1]):
            continue                                         # a tie: order matters
        perm = np.random.default_rng(seed).permutation(513)   # new id i = old perm[i]
        inv = np.argsort(perm)
        W1p, W2p = x.W1[perm], x.W2[perm]
        basep = x.base[:, :, perm]
        anchorp = inv[x.anchor.numpy()].astype(np.int32)
        tp, _, _ = O.walk(bits(W1p), bits(W2p), bits(basep), anchorp,
                          x.temperature.numpy(), 0)
        assert np.array_equal(perm[tp[0]], t[0]), "permuted walk seed %d differs" % seed
        checked += 1
        if checked >= 4:
            break
    assert checked >= 4, "too few tie-free walks to check"


def _softmax(x):
    e = np.exp(x - x.max())
    return e / e.sum()


def pin_sampling_law(O):
    """Sampled tokens follow softmax(logit / T) (chi-square, 120,000 draws)."""
    from scipy import stats
    V, r, n = 12, 4, 120000
    base_row = torch.linspace(-1.5, 1.5, V).to(torch.bfloat16)
    W = np.zeros((V, r), np.uint16)
    base = np.broadcast_to(base_row.view(torch.int16).numpy().view(np.uint16), (n, 1, V)).copy()
    anchor = np.zeros(n, np.int32)
    for T in (0.6, 1.0):
        t, _, _ = O.walk(W, W, base, anchor, np.full(n, T, np.float32), 2024, nthreads=0)
        counts = np.bincount(t[:, 0], minlength=V)
        p = _softmax(base_row.float().numpy().astype(np.float64) / T)
        res = stats.chisquare(counts, p * n)
        assert res.pvalue > 1e-3, "T=%g: token counts off softmax (p=%g)" % (T, res.pvalue)


def pin_t_to_zero(O):
    """As T -> 0+ the sample becomes the greedy argmax."""
    import synth
    x = synth.make_custom(V=300, gamma=3, B=4, seed=12)
    bits = synth.bits
    tg, lg, _ = O.walk(bits(x.W1), bits(x.W2), bits(x.base), x.anchor.numpy(),
                       np.zeros(4, np.float32), 0)
    vals = np.sort(_from_bits(lg), axis=2)
    gap = (vals[:, :, -1] - vals[:, :, -2]).min()
    assert gap > 0, "pick a tie-free seed"
    T = float(gap / 100.0)                       # noise range ~30 << gap / T
    ts, _, _ = O.walk(bits(x.W1), bits(x.W2), bits(x.base), x.anchor.numpy(),
                      np.full(4, T, np.float32), 77)
    assert np.array_equal(ts, tg), "T -> 0+ must give the greedy walk"


def pin_overflowing_quotient(O):
    """Temperatures so small that fp32(logit / T) overflows for the larger
    logits.  The Gumbel score is that fp32 quotient plus noise, so every logit
    whose quotient overflows scores +inf and the finite ones cannot reach it:
    the smallest such id wins, whatever the noise.  The group sampler forms z
    in fp64, where the quotients stay finite and ordered: it takes the argmax."""
    V, r, gamma, B = 96, 256, 3, 4
    g = torch.Generator("cpu").manual_seed(31)
    W1 = (torch.randn(V, r, generator=g) / 16).to(torch.bfloat16)
    W2 = torch.zeros(V, r, dtype=torch.bfloat16)          # logits = base exactly
    vals = torch.tensor([-2.0, -0.5, 0.0, 0.25, 1.0, 3.0])
    base = vals[torch.randint(0, len(vals), (B, gamma, V), generator=g)]
    base[:, :, :5] = -1.0                                   # the first ids never positive
    top = torch.randint(5, V, (B, gamma), generator=g)
    for b in range(B):
        for k in range(gamma):
            base[b, k, top[b, k]] = 8.0                     # one unique maximum per row
    base = base.to(torch.bfloat16)
    anchor = torch.randint(0, V, (B,), generator=g).int().numpy()
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    temps = np.array([1e-40, 3e-39, 2.0**-127, 1e-45], np.float32)
    bf = base.float().numpy()
    with np.errstate(over="ignore"):
        q = (bf.astype(np.float64) / temps.astype(np.float64)[:, None, None]).astype(np.float32)
    assert np.isposinf(q).any(axis=2).all(), "every row needs an overflowing logit"
    first_pos = np.argmax(np.isposinf(q), axis=2)
    for seed in (0, 5):
        t, _, _ = O.walk(bits(W1), bits(W2), bits(base), anchor, temps, seed)
        assert np.array_equal(t, first_pos), \
            "overflowing quotient: tokens %r, first +inf ids %r" % (t.tolist(), first_pos.tolist())
        tg, _, _ = O.walk(bits(W1), bits(W2), bits(base), anchor, temps, seed, sampler=1)
        assert np.array_equal(tg, top.numpy()), "group sampler at tiny T must take the argmax"


def pin_forced(O):
    """Teacher forcing with a walk's own tokens reproduces that walk."""
    import synth
    x = synth.make_custom(V=400, gamma=5, B=3, seed=13, temperatures=(0.0, 1.0, 0.6))
    bits = synth.bits
    t, lg, sc = O.walk(bits(x.W1), bits(x.W2), bits(x.base), x.anchor.numpy(),
                       x.temperature.numpy(), 5, want_scores=True)
    tf, lf, sf = O.walk(bits(x.W1), bits(x.W2), bits(x.base), x.anchor.numpy(),
                        x.temperature.numpy(), 5, forced=t, want_scores=True)
    assert np.array_equal(t, tf) and np.array_equal(lg, lf) and np.array_equal(sc, sf)
    # the scores' argmax (first) is the token
    assert np.array_equal(np.argmax(sc, axis=2), t)


def pin_errors(O):
    """Bad anchors and temperatures are rejected."""
    import oracle
    W = np.zeros((4, 8), np.uint16)
    base = np.zeros((1, 1, 4), np.uint16)
    for anchor, T in [(4, 0.0), (-1, 0.0), (0, -1.0), (0, float("nan")), (0, float("inf"))]:
        try:
            O.walk(W, W, base, np.array([anchor], np.int32), np.array([T], np.float32), 0)
        except oracle.OracleError:
            continue
        raise AssertionError("anchor=%r T=%r was accepted" % (anchor, T))



def pin_group_layout(O):
    """Group j of request b at step k takes its two uniforms from words 2(j&1)
    and 2(j&1)+1 of counter (j >> 1, k, b, 1)."""
    ctr, key, want = philox_reference()
    for i in range(64, 96):
        c0, k, b, c3 = (int(x) for x in ctr[i])
        assert c3 == 1
        seed = int(key[i, 0]) | (int(key[i, 1]) << 32)
        for par in range(2):
            j = 2 * c0 + par
            u1, u2 = O.group_uniforms(seed, b, k, j)
            assert u1 == O.uniform(int(want[i, 2 * par])) and \
                u2 == O.uniform(int(want[i, 2 * par + 1])), \
                "group uniforms of (b=%d,k=%d,j=%d) wrong" % (b, k, j)


def pin_group_sampling_law(O):
    """Group inverse-CDF sampling: tokens follow softmax(logit / T) (chi-square,
    120,000 draws), with full and ragged last groups."""
    from scipy import stats
    r, n = 4, 120000
    for V in (12, 20):
        base_row = torch.linspace(-1.5, 1.2, V).to(torch.bfloat16)
        W = np.zeros((V, r), np.uint16)
        base = np.broadcast_to(base_row.view(torch.int16).numpy().view(np.uint16),
                               (n, 1, V)).copy()
        anchor = np.zeros(n, np.int32)
        for T in (0.6, 1.0):
            t, _, _ = O.walk(W, W, base, anchor, np.full(n, T, np.float32), 2025, nthreads=0,
                             sampler=1)
            counts = np.bincount(t[:, 0], minlength=V)
            p = _softmax(base_row.float().numpy().astype(np.float64) / T)
            res = stats.chisquare(counts, p * n)
            assert res.pvalue > 1e-3, "V=%d T=%g: group sampler off softmax (p=%g)" % (
                V, T, res.pvalue)


def pin_group_t_to_zero(O):
    """Group sampler: as T -> 0+ the sample becomes the greedy argmax."""
    import synth
    x = synth.make_custom(V=300, gamma=3, B=4, seed=12)
    bits = synth.bits
    tg, lg, _ = O.walk(bits(x.W1), bits(x.W2), bits(x.base), x.anchor.numpy(),
                       np.zeros(4, np.float32), 0)
    vals = np.sort(_from_bits(lg), axis=2)
    gap = (vals[:, :, -1] - vals[:, :, -2]).min()
    assert gap > 0, "pick a tie-free seed"
    T = float(gap / 100.0)
    ts, _, _ = O.walk(bits(x.W1), bits(x.W2), bits(x.base), x.anchor.numpy(),
                      np.full(4, T, np.float32), 77, sampler=1)
    assert np.array_equal(ts, tg), "group sampler: T -> 0+ must give the greedy walk"


def pin_group_batch_independence(O):
    """Group sampler: a request's walk is the same alone and in a batch."""
    import synth
    x = synth.make_custom(V=777, gamma=4, B=5, seed=8, temperatures=(1.0, 0.6, 0.0))
    bits = synth.bits
    t, _, _ = O.walk(bits(x.W1), bits(x.W2), bits(x.base), x.anchor.numpy(),
                     x.temperature.numpy(), 31, sampler=1)
    for b in range(5):
        tb, _, _ = O.walk(bits(x.W1), bits(x.W2), bits(x.base[b:b + 1]),
                          x.anchor.numpy()[b:b + 1], x.temperature.numpy()[b:b + 1], 31,
                          req0=b, sampler=1)
        assert np.array_equal(tb[0], t[b]), "request %d differs alone vs in the batch" % b

# ------------------------------------------------------ recurrent heads ---
# The recurrent cells of "Keeping the Draft Walk on Chip", section "Beyond
# DSpark: other serial heads" (readings in oracle.c's header): special cases
# where a cell walk reduces to the pinned Markov walk or to a closed form.

def _cell_inputs(V, gamma, seed, spike_token=None, w1=None):
    """W1, W2, base, anchor (bits) for one request; with spike_token, a +40
    spike at that token in every step's base and the anchor at that token."""
    g = torch.Generator("cpu").manual_seed(seed)
    r = 256
    W1 = (torch.randn(V, r, generator=g) / 16) if w1 is None else w1
    W2 = torch.randn(V, r, generator=g)
    base = torch.randn(1, gamma, V, generator=g)
    anchor = int(torch.randint(0, V, (1,), generator=g))
    if spike_token is not None:
        base[0, :, spike_token] += 40.0
        anchor = spike_token
    bits = lambda t: t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)
    return bits(W1), bits(W2), bits(base), np.array([anchor], np.int32)


def _bits_of(t):
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def pin_cell_rnn_zero_matrix(O):
    """RNN head with M = 0 is the Markov walk over the table bf16(tanh(W1))."""
    V, gamma = 500, 5
    W1, W2, base, anchor = _cell_inputs(V, gamma, 41)
    W1[:7] = _bits_of(torch.full((7, 256), 3.0))               # saturating rows too
    M = np.zeros((256, 256), np.uint16)
    T = np.zeros(1, np.float32)
    t, lg, _, st, _ = O.walk_cell(W1, W2, base, anchor, T, 0, 2, M=M)
    W1t = O.bf16_rne(np.tanh(_from_bits(W1)).ravel()).reshape(W1.shape)
    tm, lm, _ = O.walk(W1t, W2, base, anchor, T, 0)
    assert np.array_equal(t, tm) and np.array_equal(lg, lm), \
        "RNN with M = 0 must walk like Markov over tanh(W1)"
    prev = [int(anchor[0])] + [int(v) for v in t[0, :-1]]
    assert np.array_equal(st[0], W1t[prev]), "RNN with M = 0: state must be tanh(W1[prev])"


def pin_cell_gated_half(O):
    """Gated head with M = 0 (gate 1/2) on a constant token path: the state is
    the geometric series x (1 - 2^-(k+1)), exact in bf16 for k <= 7; each step
    projects it like a Markov step whose W1 row is that state."""
    V, gamma, t0 = 300, 8, 17
    g = torch.Generator("cpu").manual_seed(42)
    W1f = torch.randn(V, 256, generator=g) / 16
    vals = torch.tensor([1.0, 2.0, 4.0, 8.0, -1.0, -2.0, -4.0, -8.0]) / 64
    W1f[t0] = vals[torch.randint(0, 8, (256,), generator=g)]
    W1, W2, base, anchor = _cell_inputs(V, gamma, 43, spike_token=t0, w1=W1f)
    M = np.zeros((256, 256), np.uint16)
    T = np.zeros(1, np.float32)
    t, lg, _, st, _ = O.walk_cell(W1, W2, base, anchor, T, 0, 1, M=M)
    assert np.all(t == t0), "the spike must hold the token path"
    x = _from_bits(W1[t0])
    for k in range(gamma):
        want = x * (1.0 - 2.0 ** -(k + 1))
        assert np.array_equal(_from_bits(st[0, k]), want), "gated M = 0: state %d" % k
        W1k = W1.copy()
        W1k[t0] = st[0, k]
        _, lk, _ = O.walk(W1k, W2, base[:, k:k + 1], anchor, T, 0)
        assert np.array_equal(lk[0, 0], lg[0, k]), "gated: step %d must project its state" % k


def pin_cell_gated_saturation(O):
    """Gated head, M = c * ones with W1 >= 0: from step 1 the gate is 1 (fp64:
    1 - z < 1e-17) and the state is W1[prev], the Markov walk's latent; with
    M = -c * ones the gate is 0 and the state stays h_0 = W1[anchor] / 2."""
    V, gamma = 400, 6
    g = torch.Generator("cpu").manual_seed(44)
    W1f = torch.randn(V, 256, generator=g).abs() / 16
    W1, W2, base, anchor = _cell_inputs(V, gamma, 45, w1=W1f)
    T = np.zeros(1, np.float32)
    for c in (64.0, -64.0):
        M = _bits_of(torch.full((256, 256), c))
        t, lg, _, st, _ = O.walk_cell(W1, W2, base, anchor, T, 0, 1, M=M)
        h0 = _from_bits(W1[anchor[0]]) / 2
        assert np.array_equal(_from_bits(st[0, 0]), h0), "gated: h_0 = W1[anchor] / 2"
        if c > 0:
            prev = [int(v) for v in t[0, :-1]]
            assert np.array_equal(st[0, 1:], W1[prev]), "gated, open gate: state = W1[prev]"
            _, lm, _ = O.walk(W1, W2, base, anchor, T, 0, forced=t)
            assert np.array_equal(lm[0, 1:], lg[0, 1:]), "gated, open gate: Markov logits"
        else:
            for k in range(1, gamma):
                assert np.array_equal(st[0, k], st[0, 0]), "gated, shut gate: state frozen"


def pin_cell_rnn_permutation(O):
    """RNN head with M = a * P (row i holds a at column pi(i)) on a constant
    token path: element i follows the scalar map h_i <- tanh(a h_pi(i) + x_i)."""
    V, gamma, t0 = 300, 6, 123
    W1, W2, base, anchor = _cell_inputs(V, gamma, 46, spike_token=t0)
    g = torch.Generator("cpu").manual_seed(47)
    pi = torch.randperm(256, generator=g).numpy()
    a = 0.75
    Mf = torch.zeros(256, 256)
    Mf[torch.arange(256), torch.from_numpy(pi)] = a
    T = np.zeros(1, np.float32)
    t, _, _, st, _ = O.walk_cell(W1, W2, base, anchor, T, 0, 2, M=_bits_of(Mf))
    assert np.all(t == t0), "the spike must hold the token path"
    x = _from_bits(W1[t0])
    h = np.zeros(256)
    for k in range(gamma):
        h = _from_bits(O.bf16_rne(np.tanh(a * h[pi] + x)))
        assert np.array_equal(_from_bits(st[0, k]), h), "RNN permutation: state %d" % k


def _gru_tables(V, seed, r_fill=None, z_fill=None):
    """The GRU's three token tables [3, V, 256] ~ N(0,1)/16, with the r- and
    z-tables optionally set to a constant."""
    g = torch.Generator("cpu").manual_seed(seed)
    X = torch.randn(3, V, 256, generator=g) / 16
    if r_fill is not None:
        X[0] = r_fill
    if z_fill is not None:
        X[1] = z_fill
    return _bits_of(X)


def pin_cell_gru_reduces_to_rnn(O):
    """GRU with M = 0 and a shut update gate (X_z = -40: z < 5e-18) is the
    Markov walk over the table bf16(tanh(X_n)), whatever the reset gate."""
    V, gamma = 450, 5
    W1, W2, base, anchor = _cell_inputs(V, gamma, 50)
    M = np.zeros((768, 256), np.uint16)
    T = np.zeros(1, np.float32)
    for r_fill in (None, -40.0, 40.0):
        X = _gru_tables(V, 51, r_fill=r_fill, z_fill=-40.0)
        t, lg, _, st, _ = O.walk_cell(W1, W2, base, anchor, T, 0, 3, M=M, X=X)
        Xn = O.bf16_rne(np.tanh(_from_bits(X[2])).ravel()).reshape(V, 256)
        tm, lm, _ = O.walk(Xn, W2, base, anchor, T, 0)
        assert np.array_equal(t, tm) and np.array_equal(lg, lm), \
            "GRU with M = 0, z = 0 must walk like Markov over tanh(X_n)"
        prev = [int(anchor[0])] + [int(v) for v in t[0, :-1]]
        assert np.array_equal(st[0], Xn[prev]), "GRU with M = 0, z = 0: state = tanh(X_n[prev])"


def pin_cell_gru_hold(O):
    """GRU with an open update gate (X_z = +40) keeps h = h_{-1} = 0: logits
    equal base and tokens are argmax(base)."""
    V, gamma = 300, 4
    W1, W2, base, anchor = _cell_inputs(V, gamma, 52)
    g = torch.Generator("cpu").manual_seed(53)
    M = _bits_of(torch.randn(768, 256, generator=g) / 16)
    X = _gru_tables(V, 54, z_fill=40.0)
    T = np.zeros(1, np.float32)
    t, lg, _, st, _ = O.walk_cell(W1, W2, base, anchor, T, 0, 3, M=M, X=X)
    assert not np.any(_from_bits(st)), "GRU, open update gate: the state stays 0"
    assert np.array_equal(_from_bits(lg[0]), _from_bits(base[0])), "GRU hold: logits = base"
    assert np.array_equal(t[0], np.argmax(_from_bits(base[0]), axis=1)), "GRU hold: argmax"


def pin_cell_gru_permutation(O):
    """GRU with U_r = U_z = 0, U_n = a * P, a shut update gate and an open
    reset gate on a constant token path: element i follows the scalar map
    h_i <- tanh(x_n,i + a h_pi(i)); with the reset gate shut instead,
    h_i = tanh(x_n,i) every step."""
    V, gamma, t0 = 300, 6, 77
    W1, W2, base, anchor = _cell_inputs(V, gamma, 55, spike_token=t0)
    g = torch.Generator("cpu").manual_seed(56)
    pi = torch.randperm(256, generator=g).numpy()
    a = 0.75
    Mf = torch.zeros(768, 256)
    Mf[512 + torch.arange(256), torch.from_numpy(pi)] = a
    M = _bits_of(Mf)
    T = np.zeros(1, np.float32)
    for r_fill in (40.0, -40.0):
        X = _gru_tables(V, 57, r_fill=r_fill, z_fill=-40.0)
        t, _, _, st, _ = O.walk_cell(W1, W2, base, anchor, T, 0, 3, M=M, X=X)
        assert np.all(t == t0), "the spike must hold the token path"
        xn = _from_bits(X[2, t0])
        h = np.zeros(256)
        for k in range(gamma):
            pre = xn + a * h[pi] if r_fill > 0 else xn
            h = _from_bits(O.bf16_rne(np.tanh(pre)))
            assert np.array_equal(_from_bits(st[0, k]), h), \
                "GRU permutation (reset %+g): state %d" % (r_fill, k)


def pin_cell_batch_and_forcing(O):
    """Each request keeps its own state (alone == in a batch), and forcing a
    walk with its own tokens and states changes nothing."""
    import synth
    x = synth.make_custom(V=333, gamma=4, B=3, seed=48, temperatures=(0.0, 1.0, 0.6))
    g = torch.Generator("cpu").manual_seed(49)
    M1 = _bits_of(torch.randn(256, 256, generator=g) / 16)
    M3 = _bits_of(torch.randn(768, 256, generator=g) / 16)
    X = _gru_tables(333, 58)
    bits = synth.bits
    for cell in (1, 2, 3):
        M = M3 if cell == 3 else M1
        kw = {"M": M, "X": X if cell == 3 else None}
        args = (bits(x.W1), bits(x.W2))
        t, lg, _, st, _ = O.walk_cell(*args, bits(x.base), x.anchor.numpy(),
                                      x.temperature.numpy(), 77, cell, **kw)
        for b in range(3):
            tb, lb, _, sb, _ = O.walk_cell(*args, bits(x.base[b:b + 1]),
                                           x.anchor.numpy()[b:b + 1],
                                           x.temperature.numpy()[b:b + 1], 77, cell, req0=b,
                                           **kw)
            assert np.array_equal(tb[0], t[b]) and np.array_equal(lb[0], lg[b]) and \
                np.array_equal(sb[0], st[b]), "cell %d: request %d differs alone" % (cell, b)
        tf, lf, _, sf, _ = O.walk_cell(*args, bits(x.base), x.anchor.numpy(),
                                       x.temperature.numpy(), 77, cell, forced=t,
                                       forced_state=st, **kw)
        assert np.array_equal(tf, t) and np.array_equal(lf, lg) and np.array_equal(sf, st), \
            "cell %d: forcing a walk with itself changed it" % cell


ALL_PINS = [
    pin_bf16_hand, pin_bf16_vs_torch, pin_bf16_vs_search,
    pin_philox_vs_triton, pin_noise_layout, pin_uniform, pin_gumbel,
    pin_hand_walk, pin_fig2_bruteforce, pin_w2_zero, pin_spike,
    pin_batch_independence, pin_permutation, pin_sampling_law, pin_t_to_zero,
    pin_overflowing_quotient, pin_forced, pin_errors, pin_group_layout, pin_group_sampling_law, pin_group_t_to_zero,
    pin_group_batch_independence, pin_cell_rnn_zero_matrix, pin_cell_gated_half,
    pin_cell_gated_saturation, pin_cell_rnn_permutation, pin_cell_gru_reduces_to_rnn,
    pin_cell_gru_hold, pin_cell_gru_permutation, pin_cell_batch_and_forcing,
]
