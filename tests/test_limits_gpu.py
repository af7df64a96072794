"""The limits of the arguments: sequences whose length is the table's whole span
(seq_len = M * P, the last block full), max_seq_len at the bound M * P, and a pool
whose every block but the spare is in use, the highest id N - 1 included.  Decode
(tensor-core and CUDA-core kernels) and prefill match the oracle there."""
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


def _full_layout(H_q, H_kv, D, P, M, others, q_lens, seed):
    """The first sequence spans all M table entries; the pool has one spare block."""
    lens = [M * P] + list(others)
    for s in range(seed, seed + 64):   # a permutation that puts id N - 1 in a table
        lay = W.custom_layout(H_q, H_kv, D, P, W.BF16, lens, q_lens, seed=s, spare_blocks=1)
        if lay.block_tables.shape[1] == M and (lay.block_tables == lay.geom.N - 1).any():
            return lay
    raise AssertionError("no seed put block N - 1 in a table")


@pytest.mark.parametrize("H_q,H_kv,D,P", [
    (32, 8, 128, 16),    # tensor-core decode
    (12, 12, 64, 7),     # CUDA-core decode (MHA, P % 16 != 0)
])
def test_decode_at_the_table_and_pool_limits(H_q, H_kv, D, P):
    M = 40
    lay = _full_layout(H_q, H_kv, D, P, M, [1, P, 3 * P + 1, M * P], None, seed=5)
    assert int(lay.seq_lens.max()) == M * P == lay.max_seq_len
    vals = W.draw_layer_values(lay, np.random.default_rng(6))
    scale = 1.0 / math.sqrt(D)
    st = G.dev_status()
    pools = G.build_dev_pools(lay, vals, st)
    out = G.run_decode(lay, vals, pools, scale, st, max_seq_len=M * P)
    assert wf.wf_device_status_fetch(st) == 0
    kp, vp = oracle.build_pools(lay, vals)
    ref = oracle.paged_decode(vals.q, kp, vp, lay.block_tables, lay.seq_lens, scale, W.BF16)
    G.assert_close(G.from_dev(out, W.BF16), ref, W.BF16, "decode at the limits")


def test_prefill_at_the_table_and_pool_limits():
    P, M = 16, 24
    # a request that is all new rows over the whole table, one with a prefix that
    # ends the table exactly, and a single-row request
    lay = _full_layout(16, 4, 128, P, M, [M * P, 33], [M * P, 100, 1], seed=9)
    assert int(lay.seq_lens.max()) == M * P
    vals = W.draw_layer_values(lay, np.random.default_rng(10))
    scale = 1.0 / math.sqrt(128)
    st = G.dev_status()
    pools = G.build_dev_pools(lay, vals, st)
    out = G.run_prefill(lay, vals, pools, scale, st)
    assert wf.wf_device_status_fetch(st) == 0
    kp, vp = oracle.build_pools(lay, vals)
    ref = oracle.paged_prefill(vals.q, kp, vp, lay.block_tables, lay.seq_lens, lay.cu_q_lens, scale, W.BF16)
    G.assert_close(G.from_dev(out, W.BF16), ref, W.BF16, "prefill at the limits")
