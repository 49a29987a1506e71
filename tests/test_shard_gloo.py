"""Two gloo ranks on the CPU run the exchange step of the vocabulary-sharded
cross-entropy: each rank holds one column shard of the same rows, forms its
shard statistics, all-gathers them in rank order, merges them in shard order
and forms the row losses and its own shard's gradient.  Both ranks must
obtain identical losses and merged statistics, and the joined gradients must
equal the unsharded oracle's.  (The kernels of each step are the C ABI's
ce_shard_stats / ce_merge_stats / ce_shard_fwd_bwd, tested on the GPU; here
the fp64 oracle stands in for them, so the test runs without a GPU.)"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

KEYS = ("x_max", "argmax", "lse", "sum_z", "z_y")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, cuts, out_dir):
    from oracle import ce as oc
    from oracle import ce_shard as osh
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        g = np.random.default_rng(7)
        N, V = 24, 301
        x = g.normal(0, 2.5, (N, V))
        lab = g.integers(0, V, N)
        lab[[2, 11]] = -100
        lab[5] = cuts[0]           # label on the second shard's first column
        lab[6] = cuts[0] - 1       # and on the first shard's last column
        edges = [0] + list(cuts) + [V]
        a, b = edges[rank], edges[rank + 1]
        st = osh.shard_stats(x[:, a:b], a, lab, softcap=20.0)
        mine = torch.tensor(np.stack([st[k].astype(np.float64) for k in KEYS], axis=1))
        gathered = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(gathered, mine)
        parts = [{k: t[:, i].numpy().copy() for i, k in enumerate(KEYS)} for t in gathered]
        for p in parts:
            p["argmax"] = p["argmax"].astype(np.int64)
        merged = osh.merge_stats(parts)
        loss = osh.row_loss(merged, lab, V, label_smoothing=0.1)
        n_valid, _ = oc.count(lab, V, -100)
        s = oc.scale("mean", 1.0, n_valid)
        valid = (lab != -100) & (lab >= 0) & (lab < V)
        grad = osh.shard_grad(x[:, a:b], a, V, lab, merged["lse"], np.where(valid, s, 0.0),
                              label_smoothing=0.1, softcap=20.0)
        np.save(os.path.join(out_dir, f"loss{rank}.npy"), loss)
        np.save(os.path.join(out_dir, f"argmax{rank}.npy"), merged["argmax"])
        np.save(os.path.join(out_dir, f"grad{rank}.npy"), grad)
        if rank == 0:
            np.save(os.path.join(out_dir, "x.npy"), x)
            np.save(os.path.join(out_dir, "lab.npy"), lab)
    finally:
        dist.destroy_process_group()


def test_two_rank_exchange_matches_the_unsharded_oracle(tmp_path):
    from oracle import ce as oc
    oc.build()  # before the ranks start, so they do not build it concurrently
    cuts = [150]
    mp.start_processes(_worker, args=(2, _free_port(), cuts, str(tmp_path)), nprocs=2,
                       start_method="spawn")
    l0, l1 = np.load(tmp_path / "loss0.npy"), np.load(tmp_path / "loss1.npy")
    assert np.array_equal(l0, l1)  # every rank holds the same losses
    assert np.array_equal(np.load(tmp_path / "argmax0.npy"), np.load(tmp_path / "argmax1.npy"))
    x, lab = np.load(tmp_path / "x.npy"), np.load(tmp_path / "lab.npy")
    ref = oc.ce_fwd_bwd(x, "f64", x.shape[1], lab, label_smoothing=0.1, softcap=20.0)
    np.testing.assert_allclose(l0, ref["loss"], rtol=1e-12, atol=1e-12)
    assert np.array_equal(np.load(tmp_path / "argmax0.npy"), ref["argmax"])
    grad = np.concatenate([np.load(tmp_path / "grad0.npy"), np.load(tmp_path / "grad1.npy")], axis=1)
    np.testing.assert_allclose(grad, ref["grad"], rtol=1e-11, atol=1e-15)
