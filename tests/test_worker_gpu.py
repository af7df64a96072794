"""wf_decode_worker: a persistent decode grid that takes its tasks while it runs
(the GPU-driven control loop of the Weaver summary, Awesome System Papers wiki,
WEAVER, "核心方法": spin on a task counter, run the attention found there, bump a
completion counter).

The feeder is this test's host thread: it copies task records and then the
`posted` count into device memory with cudaMemcpyAsync on a second stream while
the worker grid runs on its own stream.  Every output is checked against the fp64
oracle's decode of the same sequence.  The failure path is exercised without any
fault: a worker that is never fed gives up after its idle limit, reports
WF_DEV_TIMEOUT and returns, and the device keeps working.
"""
import math
import time

import numpy as np
import pytest

import oracle
from paged_kv_cache_wf_gb300 import binding as wf
from paged_kv_cache_wf_gb300 import workloads as W
from tests import _gpu as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = G.torch_mod()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_kv_cache_wf_gb300 import build
    build.build()


def _setup(lay, seed):
    torch = G.torch_mod()
    vals = W.draw_layer_values(lay, np.random.default_rng(seed))
    kp, vp = G.build_dev_pools(lay, vals)
    q = G.to_dev(vals.q, lay.geom.dtype)
    out = torch.full_like(q, float("nan"))
    bt = torch.from_numpy(lay.block_tables).cuda()
    hk, hv = oracle.build_pools(lay, vals)
    return vals, kp, vp, q, out, bt, hk, hv


def _records(lay, out_rows):
    # task b: decode q[b] over sequence b's table row into out[out_rows[b]]
    return np.stack([lay.seq_lens, np.arange(lay.B), np.arange(lay.B), out_rows], axis=1).astype(np.int32)


def test_worker_fed_while_running_matches_oracle():
    torch = G.torch_mod()
    lens = [1, 15, 16, 17, 100, 255, 256, 257, 700, 1024, 1500, 3000, 33, 64, 65, 2, 5, 900, 128, 129]
    lay = W.custom_layout(32, 8, 128, 16, W.BF16, lens, seed=61)
    vals, kp, vp, q, out, bt, hk, hv = _setup(lay, 61)
    n = lay.B
    out_rows = np.arange(n)[::-1].copy()          # out[n-1-b] <- sequence b
    recs = _records(lay, out_rows)
    tasks = torch.zeros((n, 4), dtype=torch.int32, device="cuda")
    mailbox = torch.zeros(4, dtype=torch.int32, device="cuda")
    host_tasks = torch.from_numpy(recs).pin_memory()
    cuts = [0, 3, 9, 15, n]
    posted = [torch.tensor([c], dtype=torch.int32).pin_memory() for c in cuts[1:]]
    stop = torch.tensor([1], dtype=torch.int32).pin_memory()
    st = G.dev_status()
    worker, feeder = torch.cuda.Stream(), torch.cuda.Stream()
    scale = 1.0 / math.sqrt(lay.geom.D)
    torch.cuda.synchronize()
    with torch.cuda.stream(worker):
        wf.wf_decode_worker(out, q, kp, vp, bt, tasks, mailbox, scale, num_workers=6,
                            idle_timeout_ns=5_000_000_000, dev_status=st)
    for i in range(len(cuts) - 1):
        time.sleep(0.005)   # the worker is running and waiting meanwhile
        with torch.cuda.stream(feeder):
            tasks[cuts[i]:cuts[i + 1]].copy_(host_tasks[cuts[i]:cuts[i + 1]], non_blocking=True)
            mailbox[0:1].copy_(posted[i], non_blocking=True)   # after its records, same stream
        feeder.synchronize()
    with torch.cuda.stream(feeder):
        mailbox[1:2].copy_(stop, non_blocking=True)
    feeder.synchronize()
    worker.synchronize()
    assert wf.wf_device_status_fetch(st) == 0
    mb = mailbox.cpu().numpy()
    assert mb[0] == n and mb[3] == n, mb                  # every posted task done
    ref = oracle.paged_decode(vals.q, hk, hv, lay.block_tables, lay.seq_lens, scale, W.BF16)
    got = G.from_dev(out, W.BF16)[out_rows]
    G.assert_close(got, ref, W.BF16, "worker fed while running")


def test_worker_drains_preposted_tasks_and_flags_a_bad_record():
    """All tasks (one with an out-of-range length) posted and `stop` set before the
    launch: the worker runs the good ones, flags the bad one, and leaves."""
    torch = G.torch_mod()
    lay = W.tiny_decode(0)                                # fp32 pools: 1e-4 tolerance
    vals, kp, vp, q, out, bt, hk, hv = _setup(lay, 62)
    n = lay.B
    recs = _records(lay, np.arange(n))
    recs = np.concatenate([recs, [[lay.M * lay.geom.P + 1, 0, 0, 0]]]).astype(np.int32)
    tasks = torch.from_numpy(recs).cuda()
    mailbox = torch.tensor([n + 1, 1, 0, 0], dtype=torch.int32, device="cuda")
    st = G.dev_status()
    scale = 1.0 / math.sqrt(lay.geom.D)
    wf.wf_decode_worker(out, q, kp, vp, bt, tasks, mailbox, scale, num_workers=3,
                        idle_timeout_ns=2_000_000_000, dev_status=st)
    assert wf.wf_device_status_fetch(st) == wf.WF_DEV_BAD_TASK
    assert int(mailbox[3]) == n + 1
    ref = oracle.paged_decode(vals.q, hk, hv, lay.block_tables, lay.seq_lens, scale, W.F32)
    G.assert_close(G.from_dev(out, W.F32), ref, W.F32, "worker, preposted tasks")


def test_worker_stopped_with_nothing_posted_exits_cleanly():
    torch = G.torch_mod()
    lay = W.custom_layout(8, 2, 64, 16, W.BF16, [10, 20], seed=63)
    vals, kp, vp, q, out, bt, hk, hv = _setup(lay, 63)
    tasks = torch.zeros((4, 4), dtype=torch.int32, device="cuda")
    mailbox = torch.tensor([0, 1, 0, 0], dtype=torch.int32, device="cuda")
    st = G.dev_status()
    wf.wf_decode_worker(out, q, kp, vp, bt, tasks, mailbox, 0.125, num_workers=8,
                        idle_timeout_ns=2_000_000_000, dev_status=st)
    assert wf.wf_device_status_fetch(st) == 0
    assert int(mailbox[3]) == 0
    assert torch.isnan(out.float()).all()              # nothing was written


def test_worker_never_fed_times_out_and_the_device_keeps_working():
    """No task ever comes: each CTA gives up after the idle limit, sets
    WF_DEV_TIMEOUT and returns; a decode afterwards on the same stream is correct."""
    torch = G.torch_mod()
    lay = W.custom_layout(32, 8, 128, 16, W.BF16, [40, 300], seed=64)
    vals, kp, vp, q, out, bt, hk, hv = _setup(lay, 64)
    tasks = torch.zeros((8, 4), dtype=torch.int32, device="cuda")
    mailbox = torch.zeros(4, dtype=torch.int32, device="cuda")
    st = G.dev_status()
    limit_ns = 50_000_000
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    wf.wf_decode_worker(out, q, kp, vp, bt, tasks, mailbox, 0.088, num_workers=4, idle_timeout_ns=limit_ns,
                        dev_status=st)
    status = wf.wf_device_status_fetch(st)
    waited = time.perf_counter() - t0
    assert status == wf.WF_DEV_TIMEOUT
    assert waited >= limit_ns * 1e-9 * 0.9, waited
    mb = mailbox.cpu().numpy()
    assert mb[2] == 4 and mb[3] == 0, mb                # each CTA claimed one task, none ran
    assert torch.isnan(out.float()).all()
    # the context is intact: the ordinary decode call on the same stream
    ref = oracle.paged_decode(vals.q, hk, hv, lay.block_tables, lay.seq_lens, 0.088, W.BF16)
    res = G.run_decode(lay, vals, (kp, vp), 0.088)
    G.assert_close(G.from_dev(res, W.BF16), ref, W.BF16, "decode after a timed-out worker")
