"""Continuous batching with churn, end to end on the GPU: the native block manager
hands out blocks and slots as requests arrive, grow one token per step, fork
(prefix sharing, copy-on-write of a shared partial block) and leave; every step
runs wf_copy_blocks, wf_reshape_and_cache and wf_paged_decode (the tensor-core
kernel with its work-item queue) on the device, and the oracle does the same
copies, scatters and decodes on host pools (tiny-vllm-py "Mental Model" and
"Prefix Sharing"; ember "The core idea").

Pools start as NaN everywhere and blocks are reused after frees, so a read of a
slot the manager did not hand to that sequence shows up as NaN or as a mismatch.
"""
import math

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


@pytest.mark.parametrize("seed", [0, 1])
def test_churn_steps_through_the_block_manager(seed):
    torch = G.torch_mod()
    H_q, H_kv, D, P, N = 32, 8, 128, 16, 160
    g = W.Geometry(H_q=H_q, H_kv=H_kv, D=D, P=P, N=N, dtype=W.BF16)
    rng = np.random.default_rng(seed)
    bm = wf.BlockManager(N, P, shuffle_seed=77 + seed)
    host_k, host_v = W.empty_pool(g), W.empty_pool(g)
    dev_k, dev_v = G.to_dev(host_k, W.BF16), G.to_dev(host_v, W.BF16)
    st = G.dev_status()
    scale = 1.0 / math.sqrt(D)
    live = []
    next_id = 0
    copies = forks = 0
    for step in range(10):
        # departures
        for s in list(live):
            if rng.random() < 0.15:
                bm.free(s)
                live.remove(s)
        new_slots, pairs = [], []
        # forks: a child shares its parent's blocks (prefix sharing)
        if live and rng.random() < 0.5:
            parent = int(rng.choice(live))
            bm.fork(parent, next_id)
            live.append(next_id)
            next_id += 1
            forks += 1
        # arrivals with prompts (they attend over their prompt this step)
        arrived = set()
        for _ in range(int(rng.integers(1, 3))):
            n = int(rng.integers(1, 300))
            if bm.num_free() < -(-n // P) + 4:
                break
            slots, pair = bm.append(next_id, n)
            assert pair is None
            new_slots.append(slots)
            live.append(next_id)
            arrived.add(next_id)
            next_id += 1
        # keep room for one more token per running sequence (and its copy)
        while bm.num_free() < 2 * len(live) + 2:
            victim = int(rng.choice([x for x in live if x not in arrived]))
            bm.free(victim)
            live.remove(victim)
        # every other running sequence decodes one token
        for s in live:
            if s not in arrived:
                slots, pair = bm.append(s, 1)
                new_slots.append(slots)
                if pair is not None:
                    pairs.append(pair)
        # copy-on-write copies first, then this step's rows
        if pairs:
            pr = np.array(pairs, np.int32)
            wf.wf_copy_blocks(dev_k, dev_v, torch.from_numpy(pr).cuda(), st)
            oracle.copy_blocks(host_k, host_v, pr, W.BF16)
            copies += len(pairs)
        slots = np.concatenate(new_slots).astype(np.int64)
        T = slots.shape[0]
        k = W._draw(rng, (T, H_kv, D), W.BF16, 1.0)
        v = W._draw(rng, (T, H_kv, D), W.BF16, 1.0)
        wf.wf_reshape_and_cache(G.to_dev(k, W.BF16), G.to_dev(v, W.BF16), dev_k, dev_v,
                                torch.from_numpy(slots).cuda(), st)
        oracle.reshape_and_cache(k, v, host_k, host_v, slots, W.BF16)
        # decode every live sequence
        lens = [bm.seq_len(s) for s in live]
        M = max(-(-x // P) for x in lens)
        bt, sl = bm.tables(live, M, N - 1)
        q = W._draw(rng, (len(live), H_q, D), W.BF16, 1.0)
        out_dev = torch.empty((len(live), H_q, D), dtype=torch.bfloat16, device="cuda")
        msl = int(sl.max())
        ws = torch.empty(wf.wf_paged_decode_workspace_size(len(live), H_q, msl, wf.pool_desc(dev_k)),
                         dtype=torch.uint8, device="cuda")
        wf.wf_paged_decode(out_dev, G.to_dev(q, W.BF16), dev_k, dev_v, torch.from_numpy(bt).cuda(),
                           torch.from_numpy(sl).cuda(), msl, scale, ws, st)
        ref = oracle.paged_decode(q, host_k, host_v, bt, sl, scale, W.BF16)
        G.assert_close(G.from_dev(out_dev, W.BF16), ref, W.BF16, f"step {step}")
        assert wf.wf_device_status_fetch(st) == 0
    # the pools agree byte for byte on every slot a live sequence owns
    bt, sl = bm.tables(live, max(-(-bm.seq_len(s) // P) for s in live), N - 1)
    owned = np.zeros((N, P), bool)
    for row, n in zip(bt, sl):
        for p in range(int(n)):
            owned[row[p // P], p % P] = True
    kk = G.storage_bytes(dev_k).reshape(N, P, -1)
    assert np.array_equal(kk[owned], host_k.view(np.uint8).reshape(N, P, -1)[owned])
    assert forks > 0 and copies > 0
