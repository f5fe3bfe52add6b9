"""Two Ulysses ranks as two processes on one GPU: each process owns its output
sequence shard, maps the other process's shard through CUDA IPC, and its
attention kernel stores the rows of the other rank's sequence block straight
into that process's memory (xs_attn_ulysses_rank_fwd; X-Stage, abstract, and the
gist.science technical summary, "Key Contributions" item 3: the tile owner's
stores go to the rank that owns the tile's rows).

No kernel waits for another: each rank records an interprocess event after its
launch and the other rank's stream waits for that event before the shard is
read.  Host-side barriers (gloo) order the setup and the teardown, so no
process frees or leaves memory the other may still write.  Each rank checks its
own shard bit for bit against the fused kernel run on the whole tensors in its
own process, on index-coded inputs and on random inputs.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
B, S, H, D, P = 1, 2048, 8, 128, 2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker_main(rank, port, queues, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import datetime
    import math
    import numpy as np
    import torch
    import torch.distributed as dist
    import dit_inputs as di
    import dit_attention_ulysses_gb300 as xs

    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=P, timeout=datetime.timedelta(seconds=120))
    peer = 1 - rank
    Hl, Sl = H // P, S // P
    to_dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    checks = []
    try:
        for kind in ("layout", "random"):
            if kind == "layout":
                q, k, v, scale = di.layout_code_inputs_torch(B, S, H, D)
            else:
                w = di.Workload("ipc", B=B, H=H, S=S, D=D, P=P, scale=1 / math.sqrt(D), seed=41)
                q, k, v = (to_dev(x) for x in di.random_qkv(w))
                scale = w.scale
            # this rank's shard, shared with the peer through CUDA IPC
            mine = torch.full((B, Sl, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
            torch.cuda.synchronize()
            queues[peer].put(mine)
            theirs = queues[rank].get(timeout=60)
            dist.barrier()                                   # both mappings exist
            ptrs = [0, 0]
            ptrs[rank], ptrs[peer] = mine.data_ptr(), theirs.data_ptr()
            sl = slice(rank * Hl, (rank + 1) * Hl)
            stream = torch.cuda.current_stream()
            xs.xs_attn_ulysses_rank_fwd(q[:, :, sl].contiguous(), k[:, :, sl].contiguous(),
                                        v[:, :, sl].contiguous(), ptrs, H, rank, scale, stream=stream)
            done = torch.cuda.Event(interprocess=True)
            done.record(stream)
            queues[peer].put(done.ipc_handle())              # recorded before its handle is sent
            peer_done = torch.cuda.Event.from_ipc_handle(torch.cuda.current_device(), queues[rank].get(timeout=60))
            stream.wait_event(peer_done)                     # the peer's stores into `mine` are done
            torch.cuda.synchronize()
            status = xs.xs_attn_get_device_error()
            ref = [torch.empty((B, Sl, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
            xs.xs_attn_a2a_fwd(q, k, v, ref, scale)
            torch.cuda.synchronize()
            checks.append((kind, status, bool(torch.equal(mine.view(torch.int16), ref[rank].view(torch.int16)))))
            dist.barrier()                                   # both ranks have read their shards
            del theirs, peer_done
            torch.cuda.synchronize()
            dist.barrier()                                   # mappings released before `mine` goes
            del mine
    finally:
        results.put((rank, checks))
        dist.destroy_process_group()


def test_two_process_ranks_store_into_each_others_shards():
    ctx = mp.get_context("spawn")
    queues = [ctx.Queue() for _ in range(P)]
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker_main, args=(r, port, queues, results)) for r in range(P)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = dict(results.get(timeout=10) for _ in range(P))
    for r in range(P):
        assert [c[0] for c in res[r]] == ["layout", "random"], res
        for kind, status, equal in res[r]:
            assert status == 0 and equal, (r, kind, status, equal)
