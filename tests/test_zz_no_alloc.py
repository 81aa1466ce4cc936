"""The allocation-free entry point (GPU only).

dspark_walk_run_noalloc is for callers that may not allocate device memory
(code inside an allocator or its callbacks, processes whose device memory all
belongs to a caching pool, paths that must never wait on the driver's
allocator).  Its rendezvous slots are a fixed block inside the library, shared
by every call and looked up in the caller's current context on every call.
These tests check its tokens and logits against the oracle and against the
handle-based entry point, on two calls in a row, at its stated maxima, that a
call allocates no device memory, and that it keeps working after the device
is reset.  This file is collected last on purpose.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import parity
import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def walkmod():
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    from serial_draft_head_gb300 import walk
    walk.load(build_if_missing=True)
    return walk


def _handle_run(walk, x):
    w = walk.Walk(x.W1.cuda(), x.W2.cuda(), x.B, x.gamma)
    tok = torch.full((x.B, x.gamma), -2, dtype=torch.int32, device="cuda")
    lg = torch.empty(x.B, x.gamma, x.V, dtype=torch.bfloat16, device="cuda")
    w.run(x.base.cuda(), x.anchor.cuda(), x.temperature.cuda(), x.seed, tok, lg)
    assert w.status() == 0
    w.close()
    return tok.cpu().numpy(), lg.view(torch.int16).cpu().numpy().view(np.uint16)


def _noalloc_run(walk, x, dev, tok, lg):
    W1, W2, base, anchor, temp = dev
    tok.fill_(-2)
    walk.dspark_walk_run_noalloc(W1, W2, x.V, 256, base, anchor, temp, x.seed, tok, x.B, x.gamma,
                                 lg)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), (None if lg is None else
                               lg.view(torch.int16).cpu().numpy().view(np.uint16))


def _device(x):
    return (x.W1.cuda(), x.W2.cuda(), x.base.cuda(), x.anchor.cuda(), x.temperature.cuda())


def test_noalloc_matches_oracle_and_handle_path_twice_in_a_row(walkmod):
    """The same round twice in a row (the second call finds the first one's
    state in the shared block and must clear it), then another shape: every
    token and logit of both calls passes the parity rule against the oracle,
    the two calls agree exactly, and the handle-based entry point (which may
    run another kernel, another fp32 summation order) agrees with it within
    the rule's neighbour case."""
    for i, (V, B, gamma) in enumerate([(5003, 6, 5), (20011, 3, 7)]):
        x = synth.make_custom(V=V, gamma=gamma, B=B, seed=60 + i, temperatures=(0.0, 0.6, 1.0),
                              noise_seed=900 + i)
        dev = _device(x)
        tok = torch.empty(B, gamma, dtype=torch.int32, device="cuda")
        lg = torch.empty(B, gamma, V, dtype=torch.bfloat16, device="cuda")
        first = _noalloc_run(walkmod, x, dev, tok, lg)
        second = _noalloc_run(walkmod, x, dev, tok, lg)
        assert np.array_equal(first[0], second[0]) and np.array_equal(first[1], second[1])
        rep = parity.check(x, first[0], first[1])
        assert rep.ok(), rep
        want_tok, want_lg = _handle_run(walkmod, x)
        rep_want = parity.check(x, want_tok, want_lg)
        assert rep_want.ok(), rep_want
        gv, wv = parity.bf16_vals(first[1]), parity.bf16_vals(want_lg)
        ulp = parity.bf16_ulp(np.maximum(np.abs(gv), np.abs(wv)))
        far = int(np.sum(np.abs(gv - wv) > 2 * ulp))
        assert far <= rep.logits_neighbour + rep_want.logits_neighbour


def test_noalloc_at_its_maxima(walkmod):
    """B = 64 and gamma = 16, the largest round the fixed block holds (its key
    slots used to the end): every token of every request against the oracle,
    every logit of a few requests, on two calls in a row."""
    x = synth.make_custom(V=20011, gamma=16, B=64, seed=66, temperatures=(0.0, 0.6, 1.0),
                          noise_seed=913)
    dev = _device(x)
    tok = torch.empty(64, 16, dtype=torch.int32, device="cuda")
    lg = torch.empty(64, 16, 20011, dtype=torch.bfloat16, device="cuda")
    first = _noalloc_run(walkmod, x, dev, tok, lg)
    second = _noalloc_run(walkmod, x, dev, tok, lg)
    assert np.array_equal(first[0], second[0]) and np.array_equal(first[1], second[1])
    full = parity.check_all_tokens(x, first[0])
    assert full.ok() and full.steps_checked == 64 * 16, full
    rep = parity.check(x, first[0], first[1], requests=[0, 1, 2, 31, 62, 63])
    assert rep.ok(), rep


def test_noalloc_allocates_no_device_memory(walkmod):
    """After one warm-up call (the first call in a context may load kernels),
    further calls at other batch sizes and walk lengths leave the device's free
    memory exactly as it was."""
    x = synth.make_custom(V=9001, gamma=16, B=64, seed=67, temperatures=(0.0, 1.0),
                          noise_seed=917)
    dev = _device(x)
    tok = torch.empty(64 * 16, dtype=torch.int32, device="cuda")
    lg = torch.empty(64 * 16 * 9001, dtype=torch.bfloat16, device="cuda")

    def call(B, gamma, logits):
        base = dev[2][:B, :gamma].contiguous() if gamma < 16 else dev[2][:B]
        walkmod.dspark_walk_run_noalloc(dev[0], dev[1], x.V, 256, base, dev[3][:B], dev[4][:B],
                                        x.seed, tok[:B * gamma], B, gamma,
                                        lg[:B * gamma * x.V] if logits else None)

    bases = {(B, g): dev[2][:B, :g].contiguous() for B, g in ((1, 3), (3, 16), (7, 5), (64, 16))}
    for B in (1, 2, 4, 8, 64):                       # one call per kernel instantiation
        call(B, 2, False)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for (B, g), base in bases.items():
        for logits in (False, True):
            walkmod.dspark_walk_run_noalloc(dev[0], dev[1], x.V, 256, base, dev[3][:B],
                                            dev[4][:B], x.seed + B, tok[:B * g], B, g,
                                            lg[:B * g * x.V] if logits else None)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert bool((tok[:64 * 16] >= 0).all())


_RESET_CHILD = r'''
import ctypes, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
import parity, synth
from serial_draft_head_gb300 import walk
L = walk.load(build_if_missing=False)
rt = ctypes.CDLL("libcudart.so.13")
rt.cudaMalloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t]
rt.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
rt.cudaFree.argtypes = [ctypes.c_void_p]
x = synth.make_custom(V=3001, gamma=4, B=3, seed=68, temperatures=(0.0, 1.0), noise_seed=921)
host = [np.ascontiguousarray(synth.bits(x.W1)), np.ascontiguousarray(synth.bits(x.W2)),
        np.ascontiguousarray(synth.bits(x.base)), x.anchor.numpy().astype(np.int32),
        x.temperature.numpy().astype(np.float32)]
def once():
    ptrs = []
    for a in host + [np.zeros((3, 4), np.int32)]:
        p = ctypes.c_void_p()
        assert rt.cudaMalloc(ctypes.byref(p), a.nbytes) == 0
        assert rt.cudaMemcpy(p, a.ctypes.data, a.nbytes, 1) == 0
        ptrs.append(p)
    rc = L.dspark_walk_run_noalloc(ptrs[0], ptrs[1], 3001, 256, ptrs[2], ptrs[3], ptrs[4],
                                   x.seed, ptrs[5], 3, 4, None, None)
    assert rc == 0, rc
    assert rt.cudaDeviceSynchronize() == 0
    out = np.zeros((3, 4), np.int32)
    assert rt.cudaMemcpy(out.ctypes.data, ptrs[5], out.nbytes, 2) == 0
    for p in ptrs:
        rt.cudaFree(p)
    return out
a = once()
assert rt.cudaDeviceReset() == 0
b = once()
assert np.array_equal(a, b), (a, b)
rep = parity.check(x, b)
assert rep.ok(), rep
print("reset ok")
'''


def test_noalloc_after_a_device_reset(walkmod):
    """In a fresh process that owns all of its device memory through the CUDA
    runtime: a call, cudaDeviceReset (which ends the context the scratch
    block's address belonged to), then a call in the new context gives the
    same tokens, which pass the oracle."""
    res = subprocess.run([sys.executable, "-c", _RESET_CHILD, ROOT], capture_output=True,
                         text=True, timeout=300)
    assert res.returncode == 0 and "reset ok" in res.stdout, res.stdout + res.stderr


def test_noalloc_rejects_sizes_above_its_maximum(walkmod):
    with pytest.raises(walkmod.WalkError) as e:
        walkmod.dspark_walk_run_noalloc(16, 16, 100, 256, 16, 16, 16, 0, 16, 65, 4)
    assert e.value.code == walkmod.ELIMIT
    with pytest.raises(walkmod.WalkError) as e:
        walkmod.dspark_walk_run_noalloc(16, 16, 100, 256, 16, 16, 16, 0, 16, 4, 17)
    assert e.value.code == walkmod.ELIMIT
