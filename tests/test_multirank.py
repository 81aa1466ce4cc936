"""Replicas across ranks (gloo, world size 2, CPU only).

The walk shards only into independent replicas: each rank walks its own
requests (at their global request index, so the Philox noise is the same as
in one big batch) with no collective on the data path.  These tests check
that sharded results equal the single-process walk, and that the benchmark's
reference arm runs under torchrun with two ranks.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    x = synth.make_custom(V=700, gamma=4, B=6, seed=71, temperatures=(0.0, 1.0, 0.6),
                          noise_seed=5)
    mine = [b for b in range(x.B) if b % world == rank]
    toks = {}
    for b in mine:      # each request alone, at its own request index
        t, _, _ = oracle.walk(synth.bits(x.W1), synth.bits(x.W2), synth.bits(x.base[b:b + 1]),
                              x.anchor.numpy()[b:b + 1], x.temperature.numpy()[b:b + 1], x.seed,
                              want_logits=False, req0=b)
        toks[b] = t[0].tolist()
    # results leave the ranks only for the check (not part of the walk)
    gathered = [None] * world
    dist.all_gather_object(gathered, toks)
    if rank == 0:
        merged = {}
        for d in gathered:
            merged.update(d)
        with open(os.path.join(out_dir, "tokens.json"), "w") as f:
            json.dump({str(k): v for k, v in merged.items()}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_match_single_process(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    merged = json.load(open(tmp_path / "tokens.json"))
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    x = synth.make_custom(V=700, gamma=4, B=6, seed=71, temperatures=(0.0, 1.0, 0.6),
                          noise_seed=5)
    t, _, _ = oracle.walk(synth.bits(x.W1), synth.bits(x.W2), synth.bits(x.base),
                          x.anchor.numpy(), x.temperature.numpy(), x.seed, want_logits=False)
    for b in range(x.B):
        assert merged[str(b)] == t[b].tolist()


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "2", "--warmup", "1", "--workload", "tiny"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
