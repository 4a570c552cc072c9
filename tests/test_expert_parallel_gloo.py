"""Expert-parallel decomposition of the layer on two gloo ranks (CPU).

Each rank routes every token the same way, computes only the pairs whose
expert lies in its half of the expert range, and the ranks sum their partial
deltas with one all-reduce ("Running a 2.78-Trillion-Parameter Model Across Two
Desks", Act II: one activation goes out, the weighted sum of the far experts
comes back).  The sum must equal the unsharded layer (to rounding: the order of
the sum changes).  Also checks bench.py's max-over-ranks timing helper."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import seeded_inputs as si
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r = si.LayerRecipe("ep", d=64, ff=64, E=12, k=3, T=6, x_dtype="f32", w_dtype="f32", seed=21, scale_lo=119,
                       scale_hi=125)
    x = si.layer_x(r)
    W = si.layer_router_w(r)
    _, idx, g = oracle.router(x, W, None, r.k)
    per = r.E // world
    e0, e1 = rank * per, (rank + 1) * per if rank < world - 1 else r.E
    recs = {e: si.layer_record(r, e) for e in range(e0, e1)}  # only this rank's experts
    part = oracle.partial_delta(x, idx, g, r.d, r.ff, r.k, recs, e0, e1)
    t = torch.from_numpy(part)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    slowest = bench.dist_max(float(rank + 1), world)
    np.save(os.path.join(out_dir, f"rank{rank}.npy"), t.numpy())
    np.save(os.path.join(out_dir, f"max{rank}.npy"), np.array([slowest]))
    dist.destroy_process_group()


def test_two_rank_expert_split_equals_full_layer(tmp_path):
    import oracle
    import seeded_inputs as si
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    r = si.LayerRecipe("ep", d=64, ff=64, E=12, k=3, T=6, x_dtype="f32", w_dtype="f32", seed=21, scale_lo=119,
                       scale_hi=125)
    recs = [si.layer_record(r, e) for e in range(r.E)]
    _, _, y, _ = oracle.layer_forward(si.layer_x(r), si.layer_router_w(r), None, r.d, r.ff, r.E, r.k, recs)
    for rank in range(world):
        got = np.load(tmp_path / f"rank{rank}.npy")
        np.testing.assert_allclose(got, y, rtol=0, atol=1e-12 * np.max(np.abs(y)))
        assert np.load(tmp_path / f"max{rank}.npy")[0] == world  # max over ranks of (rank + 1)
