"""Expert-parallel decomposition of the layer on two gloo ranks (CPU).

Each rank routes every token the same way, computes only the pairs whose
expert lies in its half of the expert range, and the ranks sum their partial
deltas with one all-reduce ("Running a 2.78-Trillion-Parameter Model Across Two
Desks", Act II: one activation goes out, the weighted sum of the far experts
comes back).  The sum must equal the unsharded layer (to rounding: the order of
the sum changes).  With shared experts, their pairs (every token, gate 1) are
split with the routed ones by expert id.  Also checks bench.py's max-over-ranks
timing helper."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _recipe(shared):
    import seeded_inputs as si
    r = si.LayerRecipe("ep", d=64, ff=64, E=12, k=3, T=6, x_dtype="f32", w_dtype="f32", seed=21, scale_lo=119,
                       scale_hi=125)
    return r.with_(n_shared=2, bias="zipf", bias_mode="select", seed=22) if shared else r


def _worker(rank, world, port, out_dir, shared):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import seeded_inputs as si
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r = _recipe(shared)
    x = si.layer_x(r)
    W = si.layer_router_w(r)
    _, idx, g = oracle.router(x, W, si.layer_bias(r), r.k, bias_mode=r.bias_mode)
    # every token's pairs: the routed slots, then the shared experts with gate 1
    S = r.n_shared
    idx = np.concatenate([idx, np.broadcast_to(np.arange(r.E, r.E + S, dtype=np.int32), (r.T, S))], axis=1)
    g = np.concatenate([g, np.ones((r.T, S))], axis=1)
    n_exp = r.E + S
    per = n_exp // world
    e0, e1 = rank * per, (rank + 1) * per if rank < world - 1 else n_exp
    recs = {e: si.layer_record(r, e) for e in range(e0, e1)}  # only this rank's experts
    part = oracle.partial_delta(x, idx, g, r.d, r.ff, r.k + S, recs, e0, e1)
    t = torch.from_numpy(part)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    slowest = bench.dist_max(float(rank + 1), world)
    np.save(os.path.join(out_dir, f"rank{rank}.npy"), t.numpy())
    np.save(os.path.join(out_dir, f"max{rank}.npy"), np.array([slowest]))
    dist.destroy_process_group()


@pytest.mark.parametrize("shared", [False, True])
def test_two_rank_expert_split_equals_full_layer(tmp_path, shared):
    import oracle
    import seeded_inputs as si
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path), shared), nprocs=world,
                       start_method="spawn")
    r = _recipe(shared)
    recs = [si.layer_record(r, e) for e in range(r.E + r.n_shared)]
    _, _, y, _ = oracle.layer_forward(si.layer_x(r), si.layer_router_w(r), si.layer_bias(r), r.d, r.ff, r.E, r.k,
                                      recs, n_shared=r.n_shared, bias_mode=r.bias_mode)
    for rank in range(world):
        got = np.load(tmp_path / f"rank{rank}.npy")
        np.testing.assert_allclose(got, y, rtol=0, atol=1e-12 * np.max(np.abs(y)))
        assert np.load(tmp_path / f"max{rank}.npy")[0] == world  # max over ranks of (rank + 1)
