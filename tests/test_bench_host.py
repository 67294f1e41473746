"""Host logic of bench.py that needs no GPU: packing a step's transfers into one buffer each way."""
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _workload():
    wl = bench.Workload(None, "t")
    g = torch.Generator().manual_seed(0)
    ins = [torch.randn(3, 5, generator=g).to(torch.bfloat16), torch.arange(7, dtype=torch.int32),
           torch.rand(2, 9, generator=g)]
    for t in ins:
        wl.h2d.append((torch.empty_like(t), t.clone()))        # (device side, host side)
    outs = [torch.full((4, 3), 2.5).to(torch.bfloat16), torch.ones(1, dtype=torch.int64)]
    for t in outs:
        wl.d2h.append((torch.empty_like(t), t.clone()))        # (host side, device side)
    return wl, ins, outs


def test_pack_keeps_contents_and_aligns_views():
    wl, ins, outs = _workload()
    dev_in = [p[0] for p in wl.h2d]
    hi, ho = wl.pack_transfers(align=256, device="cpu")
    assert hi == 3 * 256 and ho == 2 * 256
    dbuf, hbuf = wl.h2d_buf
    base_d, base_h = dbuf.data_ptr(), hbuf.data_ptr()
    for i, ((d, h), want) in enumerate(zip(wl.h2d, ins)):
        assert d is dev_in[i]                                  # same objects: closures still see them
        assert d.data_ptr() - base_d == 256 * i and h.data_ptr() - base_h == 256 * i
        assert torch.equal(h, want) and d.shape == want.shape and d.dtype == want.dtype
    odbuf, ohbuf = wl.d2h_buf
    for i, ((h, d), want) in enumerate(zip(wl.d2h, outs)):
        assert d.data_ptr() - odbuf.data_ptr() == 256 * i and h.data_ptr() - ohbuf.data_ptr() == 256 * i
        assert torch.equal(d, want)


def test_one_copy_each_way_moves_every_tensor():
    wl, ins, outs = _workload()
    wl.pack_transfers(align=256, device="cpu")
    dbuf, hbuf = wl.h2d_buf
    dbuf.zero_()
    dbuf.copy_(hbuf)                                           # the step's single input copy
    for (d, _), want in zip(wl.h2d, ins):
        assert torch.equal(d, want)
    for (_, d), v in zip(wl.d2h, (7.0, 3)):
        d.fill_(v)                                             # a kernel writing its output
    odbuf, ohbuf = wl.d2h_buf
    ohbuf.copy_(odbuf)                                         # the step's single output copy
    assert torch.all(wl.d2h[0][0] == 7.0) and torch.all(wl.d2h[1][0] == 3)


def test_transfer_groups_follow_readers_and_writers():
    wl, ins, outs = _workload()
    wl.launches = [None] * 5
    wl.h2d_at = [0, 0, 3]              # the first two inputs are read by launch 0: one copy
    wl.d2h_after = [2]                 # the second output defaults to the last launch
    wl.pack_transfers(align=256, device="cpu")
    gin, gout = wl.transfer_groups()
    assert gin == [(0, 0, 512), (3, 512, 768)]
    assert gout == [(2, 0, 256), (4, 256, 512)]


def _replica_rank(rank, world, port, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        bench.barrier(True, device="cpu")
        ms = bench.max_over_ranks(1.0 + rank, True, device="cpu")       # rank 1 is the slow one
        out.put((rank, ms, bench.whole_job_tflops(2e12, world, ms)))
    finally:
        dist.destroy_process_group()


def test_replicas_report_the_slowest_rank_and_the_whole_job():
    """bench.py --gpus 2 runs two replicas: both see the slower rank's time and the value counts
    the work of both (gloo on the CPU stands in for NCCL)."""
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_replica_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.0, 2.0]
    assert all(abs(r[2] - 2e12 * 2 / 2e-3 / 1e12) < 1e-9 for r in res)      # 2000 TFLOPS


def test_reference_arm_prints_only_on_rank_0(capsys):
    import argparse
    bench.run_reference(argparse.Namespace(workload="decode", warmup=3, steps=1, gpus=2), rank=1)
    assert capsys.readouterr().out == ""
