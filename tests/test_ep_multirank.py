"""Expert-parallel protocol (invariant_moe_gb300.ep) on CPU gloo ranks:
every rank's output, with its experts split over 2 or 4 ranks, has the bits
of the same rank computing alone with all experts.  The per-rank data steps
are tests/ep_host_ops.py's (oracle experts, fp32 slot-order sum), so what is
checked is the protocol itself: split sizes, the order rows travel in and
come back in, the return to (token, slot) order and the slot-order sum
("Batch-invariance generation with vLLM fused-MoE backend at improved
performance", sections "Summary" and "Usage": expert parallelism over 8
GPUs)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _inputs(rank, M, H, E, I, k, kind):
    from tests import synthetic as syn
    w = syn.moe_weights(H, E, I, seed=5, unit=True)          # the same on every rank
    x = syn.moe_tokens(M, H, seed=100 + rank, unit=True)
    if kind == "rand":
        ids, wts = syn.random_routing(M, E, k, seed=200 + rank)
    else:  # every token routed to the experts of rank 0 only
        g = syn.gen(300 + rank)
        el = E // 4 if kind == "rank0_only_of4" else E // 2
        ids = torch.stack([torch.randperm(el, generator=g)[:k] for _ in range(M)]).to(torch.int32)
        wts = torch.rand(M, k, generator=g)
    return w, x, ids, wts


def _worker(rank, world, port, q, case):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from invariant_moe_gb300 import ep
        from tests.ep_host_ops import HostOps, LocalComm
        oracle.build()
        H, E, I, k, kind = case
        M = 11 + 9 * rank                      # ragged: every rank its own batch
        w, x, ids, wts = _inputs(rank, M, H, E, I, k, kind)
        el = E // world
        ops = HostOps(oracle)
        comm = ep.TorchComm()
        out = ep.ep_moe_forward(x, ids, wts, w.w13[rank * el:(rank + 1) * el].contiguous(),
                                w.w2[rank * el:(rank + 1) * el].contiguous(), E, comm, ops)
        alone = ep.ep_moe_forward(x, ids, wts, w.w13, w.w2, E, LocalComm(), ops)
        d = ep.dispatch(ops, x, ids, wts, E, world)
        q.put((rank, bool(torch.equal(out, alone)), d.send_counts, M * k, None))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, False, None, None, repr(e)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,case", [
    (2, (64, 8, 32, 2, "rand")),
    (4, (64, 8, 32, 2, "rand")),
    (2, (64, 8, 32, 3, "rank0_only")),       # rank 1 receives no rows
    (4, (128, 16, 64, 4, "rank0_only_of4")),
])
def test_ep_ranks_match_one_rank(oracle_mod, world, case):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q, case)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, same, counts, pairs, err in res:
        assert err is None, f"rank {rank}: {err}"
        assert same, f"rank {rank}: expert-parallel output differs from the one-rank output"
        assert sum(counts) == pairs and len(counts) == world
        if case[-1].startswith("rank0_only"):
            assert counts[1:] == [0] * (world - 1)


def test_split_counts():
    from invariant_moe_gb300 import ep
    offsets = [0, 3, 3, 7, 10, 10, 12, 15, 20]       # E = 8
    assert ep.split_counts(offsets, 8, 2) == [10, 10]
    assert ep.split_counts(offsets, 8, 4) == [3, 7, 2, 8]
    assert ep.split_counts(offsets, 8, 1) == [20]
    with pytest.raises(ValueError):
        ep.split_counts(offsets, 8, 3)
