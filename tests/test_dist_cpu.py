"""Multi-process host logic of bench.py on the CPU (gloo, world size 2).

The layer shards by (batch, head) slice with no exchange on the data path, so
bench.py runs one replica per rank: each rank draws its own batch (weak
scaling), the ranks meet only at barriers, and the reported step time is the
max over ranks of the per-rank mean."""
import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    try:
        import bench
        from softmax_attention_hybrid_gb300.inputs import custom_workload, make_inputs

        r, w, local = bench.dist_info()
        bench.dist_init(w, "gloo")
        step_ms = bench.max_over_ranks(1.5 + rank, w, torch.device("cpu"))
        bench.barrier(w)
        # each rank's batch comes from its own seed (bench.py: make_inputs(w, seed=rank))
        wl = custom_workload(1, 2, 16, dtype="fp32", frozen=(1,))
        x = make_inputs(wl, seed=r)
        fp = torch.tensor([float(x["q"].double().sum())])
        allfp = [torch.zeros(1) for _ in range(w)]
        torch.distributed.all_gather(allfp, fp)
        torch.distributed.destroy_process_group()
        queue.put((rank, r, w, local, step_ms, [float(t) for t in allfp]))
    except Exception as e:  # reported to the parent, which fails the test
        queue.put((rank, "error", repr(e)))


def test_two_rank_replicas_take_the_max_step_time():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = [queue.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort(key=lambda t: t[0])
    for res in results:
        assert res[1] != "error", res
    for rank, (_, r, w, local, step_ms, fps) in enumerate(results):
        assert (r, w, local) == (rank, 2, rank)
        assert step_ms == 2.5           # the slower rank decides the step time
        assert fps[0] != fps[1]         # the replicas hold different batches
    assert results[0][5] == results[1][5]
