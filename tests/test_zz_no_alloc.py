"""The allocation-free entry point against the handle-based one (GPU only).

dspark_walk_run_noalloc serves callers that may not allocate device memory;
its rendezvous slots live in a fixed block inside the library, shared by
every call.  Two calls in a row must each give the same tokens and logits as
dspark_walk_run on the same inputs.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import parity
import synth

pytestmark = pytest.mark.gpu


def _handle_run(walk, x):
    w = walk.Walk(x.W1.cuda(), x.W2.cuda(), x.B, x.gamma)
    tok = torch.full((x.B, x.gamma), -2, dtype=torch.int32, device="cuda")
    lg = torch.empty(x.B, x.gamma, x.V, dtype=torch.bfloat16, device="cuda")
    w.run(x.base.cuda(), x.anchor.cuda(), x.temperature.cuda(), x.seed, tok, lg)
    assert w.status() == 0
    w.close()
    return tok.cpu().numpy(), lg.view(torch.int16).cpu().numpy().view(np.uint16)


def test_noalloc_matches_handle_path_twice_in_a_row():
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    from serial_draft_head_gb300 import walk
    walk.load(build_if_missing=True)
    for i, (V, B, gamma) in enumerate([(5003, 6, 5), (20011, 3, 7)]):
        x = synth.make_custom(V=V, gamma=gamma, B=B, seed=60 + i, temperatures=(0.0, 0.6, 1.0),
                              noise_seed=900 + i)
        # the handle path may run another kernel (another fp32 summation
        # order), so logits agree within the parity tolerance, not bit for bit
        want_tok, want_lg = _handle_run(walk, x)
        W1, W2 = x.W1.cuda(), x.W2.cuda()
        tok = torch.full((B, gamma), -2, dtype=torch.int32, device="cuda")
        lg = torch.empty(B, gamma, V, dtype=torch.bfloat16, device="cuda")
        walk.dspark_walk_run_noalloc(W1, W2, V, 256, x.base.cuda(), x.anchor.cuda(),
                                     x.temperature.cuda(), x.seed, tok, B, gamma, lg)
        torch.cuda.synchronize()
        got_tok = tok.cpu().numpy()
        got_lg = lg.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got_tok, want_tok)
        # both sides pass the parity rule against the oracle; where they
        # differ by more than 2 bf16 ulp, one side took the other bf16
        # neighbour of the exact projection (the rule's cancellation case)
        rep_got = parity.check(x, got_tok, got_lg)
        rep_want = parity.check(x, want_tok, want_lg)
        assert rep_got.ok(), rep_got
        assert rep_want.ok(), rep_want
        gv, wv = parity.bf16_vals(got_lg), parity.bf16_vals(want_lg)
        ulp = parity.bf16_ulp(np.maximum(np.abs(gv), np.abs(wv)))
        far = int(np.sum(np.abs(gv - wv) > 2 * ulp))
        assert far <= rep_got.logits_neighbour + rep_want.logits_neighbour


def test_noalloc_rejects_sizes_above_its_maximum():
    from serial_draft_head_gb300 import walk
    with pytest.raises(walk.WalkError) as e:
        walk.dspark_walk_run_noalloc(16, 16, 100, 256, 16, 16, 16, 0, 16, 65, 4)
    assert e.value.code == walk.ELIMIT
    with pytest.raises(walk.WalkError) as e:
        walk.dspark_walk_run_noalloc(16, 16, 100, 256, 16, 16, 16, 0, 16, 4, 17)
    assert e.value.code == walk.ELIMIT
