"""Seeded random geometries and lengths through the decode and the prefill, each
checked against the fp64 oracle at the bf16 tolerances: head counts, groups, head
sizes, block sizes and length mixes the fixed cases do not pin, drawn from a
generator with a fixed seed per case (so a failure reproduces by its id).
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


def _geometry(rng):
    H_kv = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16]))
    grp = int(rng.choice([1, 2, 4, 8]))
    while H_kv * grp > 64:
        grp //= 2
    D = int(rng.choice([64, 128]))
    P = int(rng.choice([16, 16, 32, 64, 128, 1, 5]))
    return H_kv * grp, H_kv, D, P


def _lengths(rng, B, hi):
    # log-uniform over [1, hi]: short and long sequences in one batch
    return np.maximum(1, np.round(np.exp(rng.uniform(0.0, math.log(hi), size=B)))).astype(int)


@pytest.mark.parametrize("seed", list(range(16)))
def test_decode_random_geometry(seed):
    rng = np.random.default_rng(1000 + seed)
    H_q, H_kv, D, P = _geometry(rng)
    B = int(rng.integers(1, 13))
    sl = _lengths(rng, B, 3000)
    lay = W.custom_layout(H_q, H_kv, D, P, W.BF16, list(map(int, sl)), seed=seed)
    vals = W.draw_layer_values(lay, np.random.default_rng(2000 + seed))
    scale = 1.0 / math.sqrt(D)
    st = G.dev_status()
    pools = G.build_dev_pools(lay, vals, st)
    got = G.from_dev(G.run_decode(lay, vals, pools, scale, st), W.BF16)
    kh, vh = oracle.build_pools(lay, vals)
    ref = oracle.paged_decode(vals.q, kh, vh, lay.block_tables, lay.seq_lens, scale, W.BF16)
    G.assert_close(got, ref, W.BF16, f"decode H_q={H_q} H_kv={H_kv} D={D} P={P} B={B}")
    assert wf.wf_device_status_fetch(st) == 0


@pytest.mark.parametrize("seed", list(range(12)))
def test_prefill_random_geometry(seed):
    rng = np.random.default_rng(3000 + seed)
    H_q, H_kv, D, P = _geometry(rng)
    B = int(rng.integers(1, 7))
    ql = _lengths(rng, B, 300)
    ql[rng.integers(0, B)] = int(rng.integers(0, 3))   # a request with no or few new tokens
    c = np.maximum(_lengths(rng, B, 900) - 1, 1 - ql)   # every sequence holds a position
    lay = W.custom_layout(H_q, H_kv, D, P, W.BF16, list(map(int, ql + c)), list(map(int, ql)), seed=seed)
    vals = W.draw_layer_values(lay, np.random.default_rng(4000 + seed))
    scale = 1.0 / math.sqrt(D)
    st = G.dev_status()
    pools = G.build_dev_pools(lay, vals, st)
    got = G.from_dev(G.run_prefill(lay, vals, pools, scale, st), W.BF16)
    kh, vh = oracle.build_pools(lay, vals)
    ref = oracle.paged_prefill(vals.q, kh, vh, lay.block_tables, lay.seq_lens, lay.cu_q_lens, scale, W.BF16)
    G.assert_close(got, ref, W.BF16, f"prefill H_q={H_q} H_kv={H_kv} D={D} P={P} B={B}")
    assert wf.wf_device_status_fetch(st) == 0
