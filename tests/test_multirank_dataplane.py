"""The multi-GPU partition of the path, on CPU with gloo (world size 2): Ulysses
rank r owns heads [r*H/P, (r+1)*H/P) for all S rows, computes their attention,
and the post-attention All-to-All sends block p of its rows (sequence shard p) to
rank p, which places it at heads r*H/P.. of its [B, S/P, H, D] shard (X-Stage,
abstract; gist.science technical summary, "Key Contributions" item 3).

The attention of each rank is the oracle's (fp64, on the rank's head slice);
the exchange is point-to-point sends and receives over gloo (which has no
all-to-all).  Every rank's received shard must equal the oracle's whole path
(attention of all heads, then the explicit re-shard) bit for bit: attention of a
head does not depend on which other heads sit in the same tensor.

A second test makes one rank leave between steps: the other rank's next
exchange must end with an error within the process group's short timeout (a
host-side failure; no GPU is involved).
"""
import datetime
import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

B, S, H, D, P = 1, 64, 4, 16, 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _inputs():
    sys.path.insert(0, ROOT)
    import dit_inputs as di
    w = di.Workload("dp", B=B, H=H, S=S, D=D, P=P, scale=0.25, seed=77)
    return di.random_qkv(w), w.scale


def _exchange(dist, torch, L_r, rank, world):
    """Post-attention All-to-All of rank `rank`'s head block L_r [B, S, Hl, D]:
    returns its sequence shard [B, S/P, H, D]."""
    Sl, Hl = S // world, H // world
    out = np.empty((B, Sl, H, D), dtype=np.float64)
    out[:, :, rank * Hl:(rank + 1) * Hl] = L_r[:, rank * Sl:(rank + 1) * Sl]
    reqs, bufs = [], {}
    for peer in range(world):
        if peer == rank:
            continue
        send = torch.from_numpy(np.ascontiguousarray(L_r[:, peer * Sl:(peer + 1) * Sl]))
        bufs[peer] = torch.empty((B, Sl, Hl, D), dtype=torch.float64)
        reqs.append(dist.isend(send, peer))
        reqs.append(dist.irecv(bufs[peer], peer))
    for r in reqs:
        r.wait()
    for peer, buf in bufs.items():
        out[:, :, peer * Hl:(peer + 1) * Hl] = buf.numpy()
    return out


def _rank_attention(q, k, v, scale, rank, world):
    import oracle
    Hl = H // world
    sl = slice(rank * Hl, (rank + 1) * Hl)
    return oracle.attention(np.ascontiguousarray(q[:, :, sl]), np.ascontiguousarray(k[:, :, sl]),
                            np.ascontiguousarray(v[:, :, sl]), scale, nthreads=1)


def _dataplane_worker(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import oracle
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    (q, k, v), scale = _inputs()
    shard = _exchange(dist, torch, _rank_attention(q, k, v, scale, rank, world), rank, world)
    ref = oracle.attention_a2a(q, k, v, scale, world, nthreads=1)[rank]
    queue.put((rank, bool(np.array_equal(shard, ref)), float(np.abs(shard - ref).max())))
    dist.barrier()
    dist.destroy_process_group()


def test_head_partition_and_post_attention_exchange_gloo_world2():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dataplane_worker, args=(r, P, port, queue)) for r in range(P)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    res = sorted(queue.get(timeout=10) for _ in range(P))
    assert [r[0] for r in res] == list(range(P))
    assert all(r[1] for r in res), res


def _leaving_worker(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import time
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=5))
    (q, k, v), scale = _inputs()
    L = _rank_attention(q, k, v, scale, rank, world)
    _exchange(dist, torch, L, rank, world)          # step 1: both ranks take part
    if rank == 1:
        queue.put((rank, "left"))
        queue.close()
        queue.join_thread()                         # the message is out before the process is
        os._exit(0)                                 # leaves between steps, no goodbye
    t0 = time.time()
    try:
        _exchange(dist, torch, L, rank, world)      # step 2: the peer is gone
        queue.put((rank, "no error"))
    except Exception as e:  # noqa: BLE001 - any error ends the step; the test checks that one came
        queue.put((rank, f"error after {time.time() - t0:.1f} s: {type(e).__name__}"))
    queue.close()
    queue.join_thread()
    os._exit(0)


def test_rank_leaving_between_steps_ends_the_next_exchange_with_an_error():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_leaving_worker, args=(r, P, port, queue)) for r in range(P)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode is not None for p in procs), "a rank hung"
    res = dict(queue.get(timeout=10) for _ in range(P))
    assert res[1] == "left"
    assert res[0].startswith("error after"), res[0]
    assert float(res[0].split()[2]) < 60.0
