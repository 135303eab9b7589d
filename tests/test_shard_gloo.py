"""KV-head sharding on two CPU ranks (gloo): each rank runs the oracle's
verification and selection on its own KV heads, the results are gathered, and
they must equal the unsharded computation exactly.  Checks the host-side
shard bookkeeping that a multi-GPU run of one stream would use."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import ts_synth as syn
from oracle import ts_oracle as orc
from self_speculative_ultra_gb300 import shard


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    w = syn.scaled(syn.WORKLOADS["tiny"], Hq=12, Hkv=3, L=700, B=200, planted=4)
    inp = syn.attention_inputs(w)
    return w, inp


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, inp = _case()
    q, k, v = (orc.bf16_to_f64(inp[n]) for n in ("q", "k", "v"))
    qs, ks, vs = shard.shard_layer(q, k, v, rank, world)
    O, LSE, imp = orc.verify_attention(qs, ks, vs, inp["L"], inp["parents"], w.n_imp)
    idx = np.stack([orc.select_partial(imp[h].astype(np.float32), inp["L"], w.B, w.S, w.R)
                    for h in range(ks.shape[0])])
    parts = [None] * world
    dist.all_gather_object(parts, (O, LSE, imp, idx))
    if rank == 0:
        np.save(os.path.join(out_dir, "O.npy"), np.concatenate([p[0] for p in parts], axis=1))
        np.save(os.path.join(out_dir, "LSE.npy"), np.concatenate([p[1] for p in parts], axis=1))
        np.save(os.path.join(out_dir, "imp.npy"), np.concatenate([p[2] for p in parts], axis=0))
        np.save(os.path.join(out_dir, "idx.npy"), np.concatenate([p[3] for p in parts], axis=0))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("Hkv,world", [(3, 2), (8, 3), (5, 5)])
def test_kv_head_ranges_partition(Hkv, world):
    got = [shard.kv_head_range(Hkv, r, world) for r in range(world)]
    assert got[0][0] == 0 and got[-1][1] == Hkv
    assert all(a[1] == b[0] for a, b in zip(got, got[1:]))
    sizes = [b - a for a, b in got]
    assert max(sizes) - min(sizes) <= 1


def test_two_rank_head_shard_equals_unsharded(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    w, inp = _case()
    q, k, v = (orc.bf16_to_f64(inp[n]) for n in ("q", "k", "v"))
    O, LSE, imp = orc.verify_attention(q, k, v, inp["L"], inp["parents"], w.n_imp)
    idx = np.stack([orc.select_partial(imp[h].astype(np.float32), inp["L"], w.B, w.S, w.R)
                    for h in range(w.Hkv)])
    np.testing.assert_array_equal(np.load(tmp_path / "O.npy"), O)
    np.testing.assert_array_equal(np.load(tmp_path / "LSE.npy"), LSE)
    np.testing.assert_array_equal(np.load(tmp_path / "imp.npy"), imp)
    np.testing.assert_array_equal(np.load(tmp_path / "idx.npy"), idx)
