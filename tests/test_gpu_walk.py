"""Parity of the CUDA walk with the CPU oracle, through the C ABI (GPU only).

Small shapes are compared on every logit and every step.  The five full-size
workloads, in the launch configuration the benchmark times, are compared on
every logit of sampled requests (the oracle replays one request at its own
request index) and on every token of every request (one teacher-forced,
tokens-only oracle walk of the whole batch).
"""
import dataclasses
import numpy as np
import pytest
import torch

import parity
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session")
def walkmod():
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    from serial_draft_head_gb300 import walk
    walk.load(build_if_missing=True)
    return walk


def make_walk(walkmod, x, max_B=None, max_gamma=None, kernel=None):
    w = walkmod.Walk(x.W1.cuda(), x.W2.cuda(), max_B or x.B, max_gamma or x.gamma)
    if kernel == "stream":
        w.set_kernel(walkmod.KERNEL_STREAM)
    elif kernel == "batched":
        w.set_kernel(walkmod.KERNEL_BATCHED)
    return w


def gpu_run(w, x, want_logits=True, seed=None):
    B, gamma, V = x.base.shape
    base = x.base.cuda()
    anchor = x.anchor.cuda()
    temp = x.temperature.cuda()
    tokens = torch.full((B, gamma), -2, dtype=torch.int32, device="cuda")
    logits = torch.empty(B, gamma, V, dtype=torch.bfloat16, device="cuda") if want_logits else None
    w.run(base, anchor, temp, x.seed if seed is None else seed, tokens, logits)
    st = w.status()
    lg = logits.view(torch.int16).cpu().numpy().view(np.uint16) if want_logits else None
    return st, tokens.cpu().numpy(), lg


SMALL = [
    # V, gamma, B, temperatures, seed
    (12, 3, 1, (0.0,), 1),                 # the Fig. 2 shape of "Weights That Stay", r = 256
    (1000, 5, 3, (0.0, 1.0, 0.6), 2),
    (5003, 7, 8, (0.6, 0.0, 1.0), 3),      # ragged shards
    (152 * 33 + 17, 4, 17, (0.0, 1.0), 4),  # every SM busy plus a ragged tail, B > 16
    (20000, 3, 2, (1.0,), 5),
    (4096, 2, 33, (0.0, 0.6, 1.0), 6),
    (2048, 1, 256, (0.0, 0.6, 1.0), 7),    # the largest batch
    (3000, 64, 1, (0.0,), 8),              # the longest walk
    (130000, 3, 1, (0.0,), 9),             # 152 CTAs, 6 shared-memory strips each
    (90001, 2, 5, (0.0, 1.0), 10),         # odd V: plain base loads
    (77778, 3, 12, (0.6, 0.0), 11),        # two n-tiles (8 < B <= 16)
    (3001, 2, 130, (0.0, 0.6, 1.0), 12),   # B = 130: MMA N = 144, ragged column quarters
]


@pytest.mark.parametrize("kernel", ["planned", "stream", "batched"])
@pytest.mark.parametrize("V,gamma,B,temps,seed", SMALL)
def test_small_every_logit(walkmod, V, gamma, B, temps, seed, kernel):
    x = synth.make_custom(V=V, gamma=gamma, B=B, seed=seed, temperatures=temps,
                          noise_seed=1000 + seed)
    w = make_walk(walkmod, x, kernel=kernel)
    st, toks, lg = gpu_run(w, x)
    assert st == 0, walkmod.dspark_walk_strerror(st)
    rep = parity.check(x, toks, lg)
    assert rep.ok(), rep
    w.close()


@pytest.mark.parametrize("V,max_B,B,temps", [
    (160000, 16, 16, (0.0, 1.0, 0.6)),   # no shared strips, 4 streamed strips per warp
    (160000, 16, 3, (0.6, 0.0)),
    (200000, 1, 1, (0.6,)),              # 1 shared, 5 streamed strips per warp (4 + 1)
    (230000, 2, 2, (0.0, 0.6)),          # 1 shared, 6 streamed strips per warp (4 + 2)
])
def test_streamed_tier_every_logit(walkmod, V, max_B, B, temps):
    """Shards larger than the chip: the rows the chip cannot hold are streamed
    through each warp's ring every step; every logit and token of every
    request checked."""
    x = synth.make_custom(V=V, gamma=3, B=B, seed=21, temperatures=temps, noise_seed=1021)
    w = walkmod.Walk(x.W1.cuda(), x.W2.cuda(), max_B, x.gamma)
    plan = w.plan()
    assert plan["kernel"] == walkmod.KERNEL_RESIDENT and plan["rows_stream"] > 0, plan
    assert plan["rows_tmem"] == 512, plan          # the mma.sync kernel's streamed tier
    st, toks, lg = gpu_run(w, x)
    assert st == 0, walkmod.dspark_walk_strerror(st)
    rep = parity.check(x, toks, lg)
    assert rep.ok(), rep
    w.close()


GREEDY_TOKENS_ONLY = [
    # V, gamma, B, seed: all greedy and no logits requested, so the resident
    # kernel takes its keys straight from the epilogues (no key pass)
    (12, 3, 1, 31),
    (5003, 7, 8, 32),
    (152 * 33 + 17, 4, 16, 33),   # two accumulator n-tiles, ragged tail
    (3000, 64, 1, 34),
    (130000, 3, 1, 35),
    (90001, 2, 5, 36),
    (200000, 3, 1, 37),           # streamed tier: a group of 4 strips and one of 1
    (230000, 3, 2, 38),           # streamed tier, two requests: groups of 4 and 2
    (180000, 3, 4, 39),           # streamed tier, four requests
    (160000, 3, 12, 40),          # streamed tier, two n-tiles, no shared strips
]


@pytest.mark.parametrize("V,gamma,B,seed", GREEDY_TOKENS_ONLY)
def test_greedy_tokens_without_logits(walkmod, V, gamma, B, seed):
    x = synth.make_custom(V=V, gamma=gamma, B=B, seed=seed, temperatures=(0.0,))
    w = make_walk(walkmod, x)
    st, toks, _ = gpu_run(w, x, want_logits=False)
    assert st == 0, walkmod.dspark_walk_strerror(st)
    rep = parity.check(x, toks)
    assert rep.ok(), rep
    w.close()


def test_tiny_config(walkmod):
    x = synth.make_inputs("tiny")
    w = make_walk(walkmod, x)
    assert w.plan()["kernel"] == walkmod.KERNEL_RESIDENT
    st, toks, lg = gpu_run(w, x)
    assert st == 0
    rep = parity.check(x, toks, lg)
    assert rep.ok(), rep


# ------------------------------------------------------- full-size configs --

_WEIGHTS = {}


def full_inputs(name, B, round_index=0):
    cfg = synth.CONFIGS[name]
    if name not in _WEIGHTS:
        _WEIGHTS.clear()
        W1, W2, _ = synth.make_weights(cfg.V, cfg.r, cfg.seed)
        _WEIGHTS[name] = (W1, W2)
    return synth.make_inputs(cfg, B=B, round_index=round_index, weights=_WEIGHTS[name])


_WALKS = {}


def full_walk(walkmod, name, x):
    cfg = synth.CONFIGS[name]
    if name not in _WALKS:
        for w in _WALKS.values():
            w.close()
        _WALKS.clear()
        _WALKS[name] = walkmod.Walk(x.W1.cuda(), x.W2.cuda(), max(cfg.batches), cfg.gamma)
    return _WALKS[name]


def _sample_requests(B, temps):
    pick = {0, B - 1}
    pick.update(range(min(B, len(temps))))          # one of each temperature
    pick.update(range(max(0, B - len(temps)), B))
    if B > 8:
        pick.add(B // 2)
    return sorted(pick)


@pytest.mark.parametrize("round_index,want_logits", [(0, True), (1, True), (99, True),
                                                    (2, False), (50, False)])
def test_qwen3_resident(walkmod, round_index, want_logits):
    x = full_inputs("qwen3_resident", 1, round_index)
    w = full_walk(walkmod, "qwen3_resident", x)
    plan = w.plan()
    assert plan["kernel"] == walkmod.KERNEL_RESIDENT and plan["rows_stream"] == 0
    assert plan["rows_tmem"] == 512, plan          # the mma.sync resident kernel
    st, toks, lg = gpu_run(w, x, want_logits=want_logits)
    assert st == 0
    rep = parity.check(x, toks, lg)
    assert rep.ok(), rep


@pytest.mark.parametrize("B", [1, 4, 8, 16])
@pytest.mark.parametrize("want_logits", [True, False])
def test_long_block(walkmod, B, want_logits):
    x = full_inputs("long_block", B)
    w = full_walk(walkmod, "long_block", x)
    assert w.plan()["rows_tmem"] == 512               # the mma.sync resident kernel
    st, toks, lg = gpu_run(w, x, want_logits=want_logits)
    assert st == 0
    rep = parity.check(x, toks, lg, requests=_sample_requests(B, (0.0,)))
    assert rep.ok(), rep
    full = parity.check_all_tokens(x, toks)
    assert full.ok() and full.steps_checked == B * x.gamma, full


@pytest.mark.parametrize("B", [1, 8])
@pytest.mark.parametrize("want_logits", [True, False])
def test_partial(walkmod, B, want_logits):
    x = full_inputs("partial", B)
    w = full_walk(walkmod, "partial", x)
    plan = w.plan()
    assert plan["kernel"] == walkmod.KERNEL_RESIDENT and plan["rows_stream"] > 0
    assert plan["rows_tmem"] == 512, plan          # the mma.sync kernel's streamed tier
    st, toks, lg = gpu_run(w, x, want_logits=want_logits)
    assert st == 0
    rep = parity.check(x, toks, lg, requests=_sample_requests(B, (0.0,)))
    assert rep.ok(), rep
    full = parity.check_all_tokens(x, toks)
    assert full.ok() and full.steps_checked == B * x.gamma, full


@pytest.mark.parametrize("B", [1, 16, 64, 128, 253])
def test_sampled(walkmod, B):
    x = full_inputs("sampled", B)
    w = full_walk(walkmod, "sampled", x)
    st, toks, lg = gpu_run(w, x)
    assert st == 0
    rep = parity.check(x, toks, lg, requests=_sample_requests(B, (0.0, 0.6, 1.0)))
    assert rep.ok(), rep
    full = parity.check_all_tokens(x, toks)
    assert full.ok() and full.steps_checked == B * x.gamma, full


def test_sampled_full_batch_zero_projection_property(walkmod):
    """With W2 = 0 every greedy token is argmax(base): checked for all 253 requests."""
    x = full_inputs("sampled", 253)
    x.temperature.zero_()
    w = walkmod.Walk(x.W1.cuda(), torch.zeros_like(x.W2).cuda(), 253, x.gamma)
    st, toks, _ = gpu_run(w, x, want_logits=False)
    assert st == 0
    want = np.argmax(x.base.float().numpy(), axis=2)
    assert np.array_equal(toks, want)
    w.close()


# --------------------------------------------------------- round behaviour --

def test_graph_replay_and_parity_alternation(walkmod):
    """A captured round replays correctly many times with no memset in between."""
    x = synth.make_custom(V=7000, gamma=5, B=4, seed=40, temperatures=(0.0, 1.0),
                          noise_seed=77)
    w = make_walk(walkmod, x)
    base, anchor, temp = x.base.cuda(), x.anchor.cuda(), x.temperature.cuda()
    tokens = torch.full((4, 5), -2, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        w.run(base, anchor, temp, x.seed, tokens, stream=s)  # warm-up outside capture
    s.synchronize()
    eager = tokens.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        w.run(base, anchor, temp, x.seed, tokens, stream=s)
    for _ in range(5):
        tokens.fill_(-2)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(tokens, eager)
    assert w.status() == 0
    rep = parity.check(x, eager.cpu().numpy())
    assert rep.ok(), rep


def test_seed_per_round_graph_replays_draw_fresh_noise(walkmod):
    """With the per-round seed mode, one captured graph replayed with a fixed
    seed keys round n's noise on seed + n; each replay matches the oracle at
    that key, and the sampled tokens change from replay to replay."""
    x = synth.make_custom(V=6007, gamma=4, B=3, seed=42, temperatures=(0.6, 1.0, 0.0),
                          noise_seed=5)
    w = make_walk(walkmod, x)
    w.set_seed_mode(walkmod.SEED_PER_ROUND)
    base, anchor, temp = x.base.cuda(), x.anchor.cuda(), x.temperature.cuda()
    tokens = torch.full((3, 4), -2, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    r0 = w.round(s)
    with torch.cuda.stream(s):
        w.run(base, anchor, temp, x.seed, tokens, stream=s)      # round r0, eager
    s.synchronize()
    first = tokens.cpu().numpy()
    assert parity.check(dataclasses.replace(x, seed=x.seed + r0), first).ok()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        w.run(base, anchor, temp, x.seed, tokens, stream=s)
    seen = [first]
    for _ in range(3):
        r = w.round(s)
        tokens.fill_(-2)
        g.replay()
        torch.cuda.synchronize()
        got = tokens.cpu().numpy()
        rep = parity.check(dataclasses.replace(x, seed=x.seed + r), got)
        assert rep.ok(), (r, rep)
        seen.append(got)
    assert w.round(s) == r0 + 4 and w.status() == 0
    assert any(not np.array_equal(seen[0][:2], t[:2]) for t in seen[1:])


def test_gumbel_noise_every_uniform(walkmod):
    """The kernels' Gumbel noise against float64 -log(-log U) for all 2^23
    uniforms: within a quarter of the 2^-18 (1 + |g|) error the token
    comparison allows."""
    m = torch.arange(1 << 23, dtype=torch.int64)
    bits = ((m << 9) | 0x155).to(torch.int32).cuda()       # the low 9 bits are unused
    noise = torch.empty(1 << 23, dtype=torch.float32, device="cuda")
    walkmod.dspark_walk_gumbel_noise(bits, noise)
    g = noise.cpu().numpy().astype(np.float64)
    mm = m.numpy().astype(np.float64)
    t = (16777216.0 - 2.0 * mm - 1.0) / 16777216.0           # 1 - U, exact
    ref = -np.log(-np.log1p(-t))
    err = np.abs(g - ref) / (2.0**-18 * (1.0 + np.abs(ref)))
    assert np.all(np.isfinite(g))
    assert err.max() <= 0.25, (err.max(), int(np.argmax(err)))


def test_unit_rates_are_plausible(walkmod):
    """The roofline's tier rates and the rendezvous latencies come out of the
    probe finite and in the range one GPU of this class can give: an mma.sync
    needs at least one cycle of an SM's tensor pipe, the ldmatrix-fed one no
    less, a cross-SM hop is slower than an L2 round trip, and neither takes
    microseconds."""
    r = walkmod.dspark_walk_unit_rates()
    for k, v in r.items():
        assert np.isfinite(v) and v > 0, (k, v)
    assert 1.0 <= r["hmma_rf_cycles"] <= 16.0, r
    assert r["hmma_smem_cycles"] >= r["hmma_rf_cycles"] * 0.9, r
    assert 2.0 <= r["tc_tmem_a_cycles"] <= 200.0, r
    assert 200.0 <= r["sm_mhz"] <= 4000.0, r
    rtt_ns = r["l2_load_round_trip_cycles"] / r["sm_mhz"] * 1000.0
    assert 20.0 <= rtt_ns <= 2000.0, r
    assert rtt_ns < r["cross_sm_hop_ns"] <= 10000.0, r


def test_handles_with_different_shared_memory_needs(walkmod):
    """A kernel's shared-memory limit is process-wide: creating a handle that
    needs less must not break a handle (or the allocation-free entry) that
    needs more."""
    big = synth.make_custom(V=60000, gamma=2, B=16, seed=43, temperatures=(0.0, 1.0))
    w_big = make_walk(walkmod, big)                  # resident, two n-tiles
    w_big_s = make_walk(walkmod, big, kernel="stream")
    small = synth.make_custom(V=60000, gamma=2, B=1, seed=44)
    w_small = make_walk(walkmod, small)              # created afterwards, needs less
    for w in (w_big, w_big_s):
        st, toks, lg = gpu_run(w, big)
        assert st == 0
        assert parity.check(big, toks, lg).ok()
    st, toks, _ = gpu_run(w_small, small, want_logits=False)
    assert st == 0 and parity.check(small, toks).ok()
    for w in (w_big, w_big_s, w_small):
        w.close()


def test_rounds_back_to_back(walkmod):
    """Consecutive rounds with fresh inputs on one handle each match the oracle."""
    cfg_x = synth.make_custom(V=9001, gamma=3, B=2, seed=41, temperatures=(0.0, 0.6))
    w = make_walk(walkmod, cfg_x)
    for i in range(4):
        x = synth.make_custom(V=9001, gamma=3, B=2, seed=41, temperatures=(0.0, 0.6),
                              noise_seed=i)
        x.base = synth.make_custom(V=9001, gamma=3, B=2, seed=500 + i).base
        st, toks, lg = gpu_run(w, x)
        assert st == 0
        assert parity.check(x, toks, lg).ok()


def test_untouched_memory(walkmod):
    """Nothing past [B, gamma] tokens or [B, gamma, V] logits is written."""
    x = synth.make_custom(V=3333, gamma=3, B=3, seed=42, temperatures=(0.0, 1.0))
    w = make_walk(walkmod, x, max_B=8, max_gamma=8)
    tok = torch.full((3 * 3 + 64,), 12345, dtype=torch.int32, device="cuda")
    lgt = torch.full((3 * 3 * 3333 + 512,), 7.0, dtype=torch.bfloat16, device="cuda")
    w.run(x.base.cuda(), x.anchor.cuda(), x.temperature.cuda(), x.seed, tok[:9].view(3, 3),
          lgt[:3 * 3 * 3333].view(3, 3, 3333))
    assert w.status() == 0
    assert torch.all(tok[9:] == 12345)
    assert torch.all(lgt[3 * 3 * 3333:] == 7.0)


def test_host_buffers_match_device_buffers(walkmod):
    x = synth.make_custom(V=4321, gamma=4, B=5, seed=43, temperatures=(0.0, 0.6, 1.0))
    w = make_walk(walkmod, x)
    st, toks, lg = gpu_run(w, x)
    assert st == 0
    base = x.base.pin_memory()
    out = torch.full((5, 4), -2, dtype=torch.int32).pin_memory()
    outl = torch.empty(5, 4, 4321, dtype=torch.bfloat16).pin_memory()
    st2 = walkmod.dspark_walk_run_host(w.h, base, x.anchor.pin_memory(),
                                       x.temperature.pin_memory(), x.seed, out, 5, 4, outl)
    assert st2 == 0
    assert np.array_equal(out.numpy(), toks)
    assert np.array_equal(outl.view(torch.int16).numpy().view(np.uint16), lg)
    # pageable host buffers take the staged copies instead of in-place reads
    out2 = torch.full((5, 4), -2, dtype=torch.int32)
    st3 = walkmod.dspark_walk_run_host(w.h, x.base.clone(), x.anchor.clone(),
                                       x.temperature.clone(), x.seed, out2, 5, 4, None)
    assert st3 == 0 and np.array_equal(out2.numpy(), toks)
    w.close()


@pytest.mark.parametrize("kernel", ["planned", "stream", "batched"])
def test_host_buffers_every_kernel_and_errors(walkmod, kernel):
    """dspark_walk_run_host on pinned buffers (read and written in place) for
    every kernel, a larger walk whose base is staged, and a bad anchor's
    status coming back through it (then cleared)."""
    x = synth.make_custom(V=20011, gamma=3, B=6, seed=44, temperatures=(0.0, 1.0))
    w = make_walk(walkmod, x, kernel=kernel)
    out = torch.full((6, 3), -2, dtype=torch.int32).pin_memory()
    st = walkmod.dspark_walk_run_host(w.h, x.base.pin_memory(), x.anchor.pin_memory(),
                                      x.temperature.pin_memory(), x.seed, out, 6, 3, None)
    assert st == 0
    assert parity.check(x, out.numpy()).ok()
    bad = x.anchor.clone()
    bad[2] = x.base.shape[2] + 5
    st = walkmod.dspark_walk_run_host(w.h, x.base.pin_memory(), bad.pin_memory(),
                                      x.temperature.pin_memory(), x.seed, out, 6, 3, None)
    assert st == walkmod.EANCHOR and np.all(out.numpy() == -1)
    st = walkmod.dspark_walk_run_host(w.h, x.base.pin_memory(), x.anchor.pin_memory(),
                                      x.temperature.pin_memory(), x.seed, out, 6, 3, None)
    assert st == 0 and parity.check(x, out.numpy()).ok()
    w.close()
    # 18 MB of base logits: above the in-place limit, staged through device memory
    y = synth.make_custom(V=151936, gamma=4, B=15, seed=45, temperatures=(0.0,))
    w = make_walk(walkmod, y)
    out = torch.full((15, 4), -2, dtype=torch.int32).pin_memory()
    st = walkmod.dspark_walk_run_host(w.h, y.base.pin_memory(), y.anchor.pin_memory(),
                                      y.temperature.pin_memory(), y.seed, out, 15, 4, None)
    assert st == 0
    assert parity.check(y, out.numpy(), requests=[0, 7, 14]).ok()
    w.close()


# ------------------------------------------------------------------ errors --

def test_bad_anchor_and_temperature_are_reported(walkmod):
    x = synth.make_custom(V=2000, gamma=3, B=2, seed=44)
    w = make_walk(walkmod, x)
    x.anchor[1] = 2000
    st, toks, _ = gpu_run(w, x, want_logits=False)
    assert st == walkmod.EANCHOR and np.all(toks == -1)
    x.anchor[1] = 5
    x.temperature[0] = -1.0
    st, toks, _ = gpu_run(w, x, want_logits=False)
    assert st == walkmod.ETEMP and np.all(toks == -1)
    x.temperature[0] = float("nan")
    st, toks, _ = gpu_run(w, x, want_logits=False)
    assert st == walkmod.ETEMP
    x.temperature[0] = 0.0
    st, toks, lg = gpu_run(w, x)          # the handle still works afterwards
    assert st == 0 and parity.check(x, toks, lg).ok()


def test_host_side_errors(walkmod):
    x = synth.make_custom(V=500, gamma=2, B=2, seed=45)
    w = make_walk(walkmod, x)
    base, anchor, temp = x.base.cuda(), x.anchor.cuda(), x.temperature.cuda()
    tok = torch.empty(2, 2, dtype=torch.int32, device="cuda")
    with pytest.raises(walkmod.WalkError) as e:
        walkmod.dspark_walk_run(w.h, base, anchor, temp, 0, tok, 3, 2)      # B > max_B
    assert e.value.code == walkmod.EINVAL
    with pytest.raises(walkmod.WalkError):
        walkmod.dspark_walk_run(w.h, base, anchor, temp, 0, tok, 2, 3)      # gamma > max
    with pytest.raises(walkmod.WalkError):
        walkmod.dspark_walk_run(w.h, 0, anchor, temp, 0, tok, 2, 2)         # NULL base
    with pytest.raises(walkmod.WalkError) as e:
        walkmod.dspark_walk_create(x.W1.cuda(), x.W2.cuda(), 500, 128, 2, 2)  # r != 256
    assert e.value.code == walkmod.EUNSUPPORTED


@pytest.mark.parametrize("B", [1, 2, 5, 8, 12])
def test_exact_ties_go_to_the_smallest_token(walkmod, B):
    """W2 = 0, so every logit is its base value.  Each step plants the same
    maximum at rows of one lane in several tiers of one CTA's shard (tensor
    memory, a later tensor-memory strip's second row half, the register
    strip, a shared strip) and in a later CTA; the smallest token id must win,
    exactly (the near-tie rule would accept any of them).  Greedy rounds
    without logits take the fused epilogue."""
    V, gamma = 151936, 8
    x = synth.make_custom(V=V, gamma=gamma, B=B, seed=70 + B)
    g = torch.Generator().manual_seed(700 + B)
    base = (torch.rand(B, gamma, V, generator=g) * -7.0 - 1.0).to(torch.bfloat16)
    w = walkmod.Walk(x.W1.cuda(), torch.zeros_like(x.W2).cuda(), B, gamma)
    plan = w.plan()
    R, n = plan["rows_per_cta"], plan["n_cta"]
    want = np.zeros((B, gamma), dtype=np.int64)
    for b in range(B):
        for k in range(gamma):
            c = (7 * k + 13 * b) % (n - 3)
            wp, gl = (k + b) % 8, (3 * k + b) % 8
            local = [640 + 16 * (wp + 8) + gl, 64 * wp + 32 + gl + 8, 512 + 16 * wp + gl,
                     64 * wp + gl]
            toks = [c * R + r for r in local if r < R] + [(c + 3) * R + 64 * wp + gl]
            toks = [v for v in toks if v < V]
            base[b, k, toks] = 2.0
            want[b, k] = min(toks)
    x.base = base
    st, toks, _ = gpu_run(w, x, want_logits=False)
    assert st == 0
    assert np.array_equal(toks, want), (toks, want)
    w.close()


@pytest.mark.parametrize("kernel", ["planned", "stream", "batched"])
@pytest.mark.parametrize("V", [1, 2, 7])
def test_degenerate_vocabularies(walkmod, V, kernel):
    """V = 1 (every token is 0), V = 2, V = 7 (one ragged group of the group
    sampler), greedy and sampled requests, on every kernel."""
    x = synth.make_custom(V=V, gamma=3, B=3, seed=60 + V, temperatures=(0.0, 1.0, 0.6),
                          noise_seed=60)
    w = make_walk(walkmod, x, kernel=kernel)
    st, toks, lg = gpu_run(w, x)
    assert st == 0
    assert parity.check(x, toks, lg).ok()
    if V == 1:
        assert not toks.any()
    if kernel != "stream":
        w.set_sampler(walkmod.SAMPLER_GROUP)
        st, toks, lg = gpu_run(w, x)
        assert st == 0
        assert parity.check(x, toks, lg, sampler=1).ok()
    w.close()


@pytest.mark.parametrize("kernel", ["planned", "stream", "batched"])
@pytest.mark.parametrize("B", [6, 12, 20])
def test_tiny_temperatures(walkmod, B, kernel):
    """Temperatures down to fp32 subnormals: fl(1/T) overflows below 2^-128 and
    logit / T overflows for most logits below 2^-127, so the Gumbel scores
    tie at +inf and the smallest such token wins; 1e-30 keeps the scores
    finite.  The group sampler where logit / T stays finite in fp32."""
    x = synth.make_custom(V=3001, gamma=3, B=B, seed=71, noise_seed=71,
                          temperatures=(1e-40, 3e-39, 2.0**-127, 1e-30, 0.0, 1.0))
    w = make_walk(walkmod, x, kernel=kernel)
    st, toks, lg = gpu_run(w, x)
    assert st == 0, walkmod.dspark_walk_strerror(st)
    rep = parity.check(x, toks, lg)
    assert rep.ok(), rep
    if kernel != "stream":
        y = synth.make_custom(V=3001, gamma=3, B=B, seed=71, noise_seed=72,
                              temperatures=(1e-30, 1e-20, 0.0, 2.0**-100))
        w.set_sampler(walkmod.SAMPLER_GROUP)
        st, toks, lg = gpu_run(w, y)
        assert st == 0
        rep = parity.check(y, toks, lg, sampler=1)
        assert rep.ok(), rep
    w.close()


def test_empty_batch_and_walk_are_rejected(walkmod):
    x = synth.make_custom(V=500, gamma=2, B=2, seed=46)
    w = make_walk(walkmod, x)
    base, anchor, temp = x.base.cuda(), x.anchor.cuda(), x.temperature.cuda()
    tok = torch.empty(2, 2, dtype=torch.int32, device="cuda")
    for B, gamma in ((0, 2), (2, 0), (-1, 2)):
        with pytest.raises(walkmod.WalkError) as e:
            walkmod.dspark_walk_run(w.h, base, anchor, temp, 0, tok, B, gamma)
        assert e.value.code == walkmod.EINVAL
    w.close()


def test_lost_arrival_times_out_and_recovers(walkmod):
    """A CTA that never posts makes the round end with ETIMEOUT, not hang."""
    x = synth.make_custom(V=8000, gamma=4, B=2, seed=46, temperatures=(0.0, 1.0))
    w = make_walk(walkmod, x)
    walkmod.dspark_walk_set_limits(w.h, 50_000_000, 1)      # 50 ms; CTA 1 skips
    st, toks, _ = gpu_run(w, x, want_logits=False)
    assert st == walkmod.ETIMEOUT
    assert np.all(toks == -1)
    walkmod.dspark_walk_set_limits(w.h, 200_000_000, -1)
    for _ in range(2):                                     # both parities clean again
        st, toks, lg = gpu_run(w, x)
        assert st == 0
        assert parity.check(x, toks, lg).ok()


def test_lost_arrival_one_greedy_request(walkmod):
    """One greedy request without logits (the next step's projection runs
    while warp 0 waits): a CTA that never posts still ends the round with
    ETIMEOUT, and the next rounds run clean."""
    x = synth.make_custom(V=151936, gamma=5, B=1, seed=48, temperatures=(0.0,))
    w = make_walk(walkmod, x)
    walkmod.dspark_walk_set_limits(w.h, 50_000_000, 3)      # 50 ms; CTA 3 skips
    st, toks, _ = gpu_run(w, x, want_logits=False)
    assert st == walkmod.ETIMEOUT
    assert np.all(toks == -1)
    walkmod.dspark_walk_set_limits(w.h, 200_000_000, -1)
    for _ in range(2):
        st, toks, _ = gpu_run(w, x, want_logits=False)
        assert st == 0
        assert parity.check(x, toks).ok()
    w.close()


def test_lost_arrival_with_streamed_tier(walkmod):
    """A round aborted while streamed chunks are in flight ends with ETIMEOUT
    (the ring's copies are waited for before the CTAs exit), and the next
    rounds run clean."""
    x = synth.make_custom(V=200000, gamma=3, B=1, seed=47, temperatures=(0.6,))
    w = make_walk(walkmod, x)
    assert w.plan()["rows_stream"] > 0
    walkmod.dspark_walk_set_limits(w.h, 50_000_000, 5)      # 50 ms; CTA 5 skips
    st, toks, _ = gpu_run(w, x, want_logits=False)
    assert st == walkmod.ETIMEOUT
    assert np.all(toks == -1)
    walkmod.dspark_walk_set_limits(w.h, 200_000_000, -1)
    for _ in range(2):
        st, toks, lg = gpu_run(w, x)
        assert st == 0
        assert parity.check(x, toks, lg).ok()
    w.close()


# ---------------------------------------------------- group inverse-CDF --

GROUP_SHAPES = [
    # V, gamma, B, temperatures, seed
    (1000, 4, 3, (0.6, 1.0, 0.0), 51),
    (5003, 5, 8, (1.0, 0.6), 52),                  # ragged last group (5003 = 8 * 625 + 3)
    (152 * 33 + 17, 3, 17, (0.6, 0.0, 1.0), 53),   # B > 16: the batched kernel
    (4096, 2, 64, (1.0, 0.6, 0.0), 54),
    (130000, 2, 2, (1.0,), 55),
    (200000, 2, 1, (0.6,), 56),                    # the streamed tier
]


@pytest.mark.parametrize("kernel", ["planned", "batched"])
@pytest.mark.parametrize("V,gamma,B,temps,seed", GROUP_SHAPES)
def test_group_sampler_every_logit(walkmod, V, gamma, B, temps, seed, kernel):
    x = synth.make_custom(V=V, gamma=gamma, B=B, seed=seed, temperatures=temps,
                          noise_seed=2000 + seed)
    w = make_walk(walkmod, x, kernel=kernel)
    w.set_sampler(walkmod.SAMPLER_GROUP)
    st, toks, lg = gpu_run(w, x)
    assert st == 0, walkmod.dspark_walk_strerror(st)
    rep = parity.check(x, toks, lg, sampler=1)
    assert rep.ok(), rep
    w.close()


@pytest.mark.parametrize("B", [16, 64, 253])
def test_group_sampler_sampled_config(walkmod, B):
    x = full_inputs("sampled", B)
    w = full_walk(walkmod, "sampled", x)
    w.set_sampler(walkmod.SAMPLER_GROUP)
    try:
        st, toks, lg = gpu_run(w, x)
    finally:
        w.set_sampler(walkmod.SAMPLER_GUMBEL)
    assert st == 0
    rep = parity.check(x, toks, lg, requests=_sample_requests(B, (0.0, 0.6, 1.0)), sampler=1)
    assert rep.ok(), rep
    full = parity.check_all_tokens(x, toks, sampler=1)
    assert full.ok() and full.steps_checked == B * x.gamma, full


def test_group_sampler_not_on_the_streamed_kernel(walkmod):
    x = synth.make_custom(V=1000, gamma=2, B=2, seed=57, temperatures=(1.0,))
    w = make_walk(walkmod, x, kernel="stream")
    w.set_sampler(walkmod.SAMPLER_GROUP)
    with pytest.raises(walkmod.WalkError) as e:
        gpu_run(w, x)
    assert e.value.code == walkmod.EUNSUPPORTED
    w.close()


# ------------------------------------------------------- recurrent heads --

CELL_SHAPES = [
    # V, gamma, B, temperatures, seed
    (12, 3, 1, (0.0,), 61),                       # fewer CTAs than rows of M
    (1000, 5, 3, (0.0, 1.0, 0.6), 62),
    (5003, 7, 8, (0.6, 0.0, 1.0), 63),
    (152 * 33 + 17, 4, 16, (0.0, 1.0), 64),       # two n-tiles, the largest resident batch
    (130000, 6, 2, (0.0, 0.6), 65),               # 128 of the CTAs own two rows of M
    (200000, 3, 1, (0.6,), 66),                   # the streamed tier
    (160000, 3, 5, (0.0, 0.6), 67),               # the streamed tier, five requests
]


def cell_weights(cell, V, seed):
    """(M, X) of a recurrent head: X (the GRU's token tables) is None otherwise."""
    if cell == 3:
        return synth.make_cell_matrix(seed, rows=768), synth.make_cell_tables(V, seed + 1)
    return synth.make_cell_matrix(seed), None


def cell_run(walkmod, w, x, cell, M, want_logits=True, X=None):
    B, gamma, _ = x.base.shape
    Md = M.cuda()
    states = torch.empty(B, gamma, 256, dtype=torch.bfloat16, device="cuda")
    w.set_cell(cell, Md, None if X is None else X.cuda())
    w.set_state_output(states)
    try:
        st, toks, lg = gpu_run(w, x, want_logits=want_logits)
    finally:
        w.set_state_output(None)
        w.set_cell(walkmod.CELL_MARKOV)
    return st, toks, lg, synth.bits(states.cpu())


@pytest.mark.parametrize("cell", [1, 2, 3])
@pytest.mark.parametrize("V,gamma,B,temps,seed", CELL_SHAPES)
def test_cell_every_logit_and_state(walkmod, V, gamma, B, temps, seed, cell):
    """Gated (1), RNN (2) and GRU (3) heads: every state element, logit and token."""
    x = synth.make_custom(V=V, gamma=gamma, B=B, seed=seed, temperatures=temps,
                          noise_seed=3000 + seed)
    M, X = cell_weights(cell, V, seed)
    w = make_walk(walkmod, x)
    st, toks, lg, states = cell_run(walkmod, w, x, cell, M, X=X)
    assert st == 0, walkmod.dspark_walk_strerror(st)
    rep = parity.check(x, toks, lg, cell=cell, M=synth.bits(M), gpu_states=states,
                       X=None if X is None else synth.bits(X))
    assert rep.ok(), rep
    assert rep.states_checked == B * gamma * 256
    w.close()


@pytest.mark.parametrize("cell", [1, 2, 3])
def test_cell_long_block(walkmod, cell):
    """V = 151,936, gamma = 16, B = 16 on the recurrent heads (sampled requests)."""
    x = full_inputs("long_block", 16)
    w = full_walk(walkmod, "long_block", x)
    M, X = cell_weights(cell, x.base.shape[2], 100 + cell)
    st, toks, lg, states = cell_run(walkmod, w, x, cell, M, X=X)
    assert st == 0
    rep = parity.check(x, toks, lg, requests=_sample_requests(16, (0.0,)), cell=cell,
                       M=synth.bits(M), gpu_states=states,
                       X=None if X is None else synth.bits(X))
    assert rep.ok(), rep


def test_markov_state_output_is_the_gathered_row(walkmod):
    """With the Markov head the state output is u_k = W1[prev_k]."""
    x = synth.make_custom(V=3000, gamma=5, B=3, seed=67, temperatures=(0.0, 1.0))
    w = make_walk(walkmod, x)
    states = torch.empty(3, 5, 256, dtype=torch.bfloat16, device="cuda")
    w.set_state_output(states)
    st, toks, _ = gpu_run(w, x, want_logits=False)
    assert st == 0
    W1 = synth.bits(x.W1)
    s = synth.bits(states.cpu())
    for b in range(3):
        prev = [int(x.anchor[b])] + [int(t) for t in toks[b, :-1]]
        assert np.array_equal(s[b], W1[prev])
    w.close()


def test_cell_rejections(walkmod):
    """Recurrent heads run on the resident kernel only; bad arguments are refused."""
    x = synth.make_custom(V=4096, gamma=2, B=17, seed=68, temperatures=(0.0,))
    w = make_walk(walkmod, x)                       # max_B 17: B = 17 takes the batched kernel
    M = synth.make_cell_matrix(9).cuda()
    with pytest.raises(walkmod.WalkError) as e:
        walkmod.dspark_walk_set_cell(w.h, 7, M)
    assert e.value.code == walkmod.EINVAL
    with pytest.raises(walkmod.WalkError) as e:
        walkmod.dspark_walk_set_cell(w.h, walkmod.CELL_RNN, None)
    assert e.value.code == walkmod.EINVAL
    with pytest.raises(walkmod.WalkError) as e:                # the GRU needs its tables
        walkmod.dspark_walk_set_cell(w.h, walkmod.CELL_GRU,
                                     synth.make_cell_matrix(9, rows=768).cuda(), None)
    assert e.value.code == walkmod.EINVAL
    w.set_cell(walkmod.CELL_RNN, M)
    with pytest.raises(walkmod.WalkError) as e:
        gpu_run(w, x)
    assert e.value.code == walkmod.EUNSUPPORTED
    w.set_cell(walkmod.CELL_MARKOV)
    st, toks, lg = gpu_run(w, x)                    # the Markov head still runs there
    assert st == 0 and parity.check(x, toks, lg).ok()
    w.close()


def test_cell_graph_replay_and_group_sampler(walkmod):
    """A recurrent head inside a captured CUDA graph replays identically (the
    exchange buffer needs no reset), and it composes with the group sampler."""
    x = synth.make_custom(V=9000, gamma=6, B=3, seed=69, temperatures=(0.0, 1.0, 0.6),
                          noise_seed=79)
    M = synth.make_cell_matrix(69)
    Md = M.cuda()
    w = make_walk(walkmod, x)
    states = torch.empty(3, 6, 256, dtype=torch.bfloat16, device="cuda")
    w.set_cell(walkmod.CELL_GATED, Md)
    w.set_state_output(states)
    base, anchor, temp = x.base.cuda(), x.anchor.cuda(), x.temperature.cuda()
    tokens = torch.full((3, 6), -2, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        w.run(base, anchor, temp, x.seed, tokens, stream=s)
    s.synchronize()
    eager, eager_states = tokens.clone(), states.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        w.run(base, anchor, temp, x.seed, tokens, stream=s)
    for _ in range(4):
        tokens.fill_(-2)
        states.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(tokens, eager) and torch.equal(states, eager_states)
    assert w.status() == 0
    rep = parity.check(x, eager.cpu().numpy(), cell=1, M=synth.bits(M),
                       gpu_states=synth.bits(eager_states.cpu()))
    assert rep.ok(), rep
    del g
    # the same head with the group inverse-CDF sampler
    w.set_sampler(walkmod.SAMPLER_GROUP)
    st, toks, lg = gpu_run(w, x)
    assert st == 0
    rep = parity.check(x, toks, lg, cell=1, M=synth.bits(M), sampler=1,
                       gpu_states=synth.bits(states.cpu()))
    assert rep.ok(), rep
    w.close()
