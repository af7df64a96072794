"""Seeded synthetic inputs for paged KV-cache attention.

This module is the one piece that both the CUDA path's tests/bench and the
fp64 oracle are fed from.  It holds no attention arithmetic: it draws
sequence lengths, builds block tables with a host-side block allocator (the
role the scheduler / model runner plays in weft and ember), names the slot of
every token the runner would write (``slot = block_id * P + offset``, the
runner's bookkeeping, "write: scatter via slot_mapping" in weft's cache-layout
table), and draws q/K/V values.  Everything is a pure function of a seed.

Pool geometry follows weft's per-layer paged view ``[N, P, H_kv, D]``
(weft, "Cache layouts" table).  bf16 values are produced by rounding float32
draws to nearest-even once, here, and are carried as uint16 bit patterns so
that both sides read exactly the same numbers.

The five named workloads mirror the ones this library is measured on
(tiny fp32 decode; GPT-2-small, Llama-3.2-1B and Llama-3-8B shaped bf16
decode; a mixed prefill+decode step at Llama-3-8B shapes).  The Weaver
traces (BurstGPT, Azure-Conv) are not available offline; the length
distributions below stand in for them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Tuple

import numpy as np

F32 = "f32"
BF16 = "bf16"


# ---------------------------------------------------------------------------
# dtype plumbing (no attention arithmetic)
# ---------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round-to-nearest-even), as uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    out = ((u + (((u >> 16) & 1) + np.uint32(0x7FFF))) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def storage_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of stored values (float32 or bf16 bits) to float64."""
    if dtype == F32:
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    return bf16_bits_to_f32(a).astype(np.float64)


def elt_size(dtype: str) -> int:
    return 4 if dtype == F32 else 2


def np_storage_dtype(dtype: str):
    return np.float32 if dtype == F32 else np.uint16


NAN_BITS = {F32: np.float32(np.nan), BF16: np.uint16(0x7FC0)}


# ---------------------------------------------------------------------------
# geometry and layout
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class Geometry:
    H_q: int
    H_kv: int
    D: int
    P: int          # block size (tokens per block)
    N: int          # blocks in the per-layer pool
    dtype: str      # "f32" | "bf16"
    L: int = 1      # layers (one pool per layer)
    value_scale: float = 1.0

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def row_elems(self) -> int:
        """Elements of one slot of one pool (all KV heads of one position)."""
        return self.H_kv * self.D

    @property
    def pool_elems(self) -> int:
        return self.N * self.P * self.H_kv * self.D


@dataclasses.dataclass
class Layout:
    """Lengths, block tables and slots of one step (no values).

    ``seq_lens[b]`` counts the tokens of sequence b in the cache AFTER this
    step's write; ``q_lens[b]`` is how many of them are new this step (1 for a
    decode row).  Request b's new tokens are positions
    ``seq_lens[b]-q_lens[b] .. seq_lens[b]-1``; the rest is its cached prefix.
    """
    geom: Geometry
    seq_lens: np.ndarray       # int32 [B]
    q_lens: np.ndarray         # int32 [B]
    block_tables: np.ndarray   # int32 [B, M]; unused entries point at a spare block
    spare_block: int           # a block no live position uses (stays NaN-poisoned)

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def M(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def prefix_lens(self) -> np.ndarray:
        return (self.seq_lens - self.q_lens).astype(np.int32)

    @property
    def cu_q_lens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    @property
    def cu_prefix(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.prefix_lens)]).astype(np.int64)

    @property
    def T_total(self) -> int:
        return int(self.q_lens.sum())

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.B else 0

    @property
    def max_q_len(self) -> int:
        return int(self.q_lens.max()) if self.B else 0

    def slot_of(self, b: int, pos: np.ndarray) -> np.ndarray:
        """The runner's slot bookkeeping: where position ``pos`` of sequence b lives."""
        P = self.geom.P
        pos = np.asarray(pos, dtype=np.int64)
        return self.block_tables[b, pos // P].astype(np.int64) * P + pos % P

    def new_slots(self) -> np.ndarray:
        """slot_mapping for this step's new tokens, request-major (int64 [T_total])."""
        out = [self.slot_of(b, np.arange(self.prefix_lens[b], self.seq_lens[b]))
               for b in range(self.B)]
        return np.concatenate(out).astype(np.int64) if out else np.zeros(0, np.int64)

    def prefix_slots(self) -> np.ndarray:
        """Slots of every cached prefix position, request-major (int64 [sum prefix])."""
        out = [self.slot_of(b, np.arange(0, self.prefix_lens[b])) for b in range(self.B)]
        return np.concatenate(out).astype(np.int64) if out else np.zeros(0, np.int64)


@dataclasses.dataclass
class LayerValues:
    """One layer's values in storage dtype (float32 or bf16 bits)."""
    q: np.ndarray        # [T_total, H_q, D]
    k_new: np.ndarray    # [T_total, H_kv, D]
    v_new: np.ndarray
    k_prefix: np.ndarray # [sum prefix, H_kv, D]  request-major, position-major
    v_prefix: np.ndarray


# ---------------------------------------------------------------------------
# block allocator fixture (host side; stands in for ember's block manager)
# ---------------------------------------------------------------------------
class BlockAllocator:
    """O(1) LIFO free-list allocator over block ids 0..N-1, shuffled at start."""

    def __init__(self, N: int, rng: np.random.Generator):
        self.free = list(rng.permutation(N).astype(np.int64))
        self.N = N

    def alloc(self) -> int:
        if not self.free:
            raise RuntimeError("block pool exhausted")
        return int(self.free.pop())

    def release(self, blocks):
        self.free.extend(int(b) for b in blocks)

    def __len__(self):
        return len(self.free)


def _blocks_for(n_tokens: int, P: int) -> int:
    return -(-int(n_tokens) // P)


def _tables_from_lists(lists: List[List[int]], spare: int) -> np.ndarray:
    M = max([len(x) for x in lists] + [1])
    bt = np.full((len(lists), M), spare, dtype=np.int32)
    for b, blocks in enumerate(lists):
        bt[b, :len(blocks)] = blocks
    return bt


def layout_from_permutation(geom: Geometry, seq_lens, q_lens, rng) -> Layout:
    """Tables take consecutive runs of one random permutation of the pool's block ids.

    The last id of the permutation is kept back as the spare (poison) block.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    perm = rng.permutation(geom.N).astype(np.int64)
    spare = int(perm[-1])
    lists, k = [], 0
    for L in seq_lens:
        nb = _blocks_for(L, geom.P)
        if k + nb > geom.N - 1:
            raise ValueError("pool too small for the requested lengths")
        lists.append([int(x) for x in perm[k:k + nb]])
        k += nb
    return Layout(geom, seq_lens, q_lens, _tables_from_lists(lists, spare), spare)


def layout_with_churn(geom_fn, seq_lens, q_lens, rng, headroom: float = 1.25) -> Layout:
    """Build fragmented tables by allocating, freeing and reallocating under churn.

    Procedure (a reading of "allocating, freeing and reallocating under churn"):
      1. N = ceil(headroom * blocks needed) + 1; shuffled LIFO free list.
      2. Fill the pool to about 90% with dummy sequences of the same length
         distribution (lengths drawn by permuting the real ones), then free a
         random half of them.
      3. Grow the real sequences round-robin, one block per turn; whenever the
         free list runs dry, free a random surviving dummy.
    The result interleaves every table with the others' blocks.
    ``geom_fn(N)`` returns the Geometry for a pool of N blocks.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    probe = geom_fn(1)
    P = probe.P
    need = [_blocks_for(L, P) for L in seq_lens]
    N = int(math.ceil(headroom * sum(need))) + 1
    geom = geom_fn(N)
    alloc = BlockAllocator(N, rng)
    spare = alloc.alloc()
    # 2. dummies up to ~90% full
    dummies: List[List[int]] = []
    target = int(0.9 * (N - 1))
    while True:
        room = target - ((N - 1) - len(alloc))
        if room <= 0:
            break
        nb = min(max(1, need[int(rng.integers(len(need)))]), room)
        dummies.append([alloc.alloc() for _ in range(nb)])
    order = rng.permutation(len(dummies))
    keep = []
    for i, d in enumerate(order):
        if i % 2 == 0:
            alloc.release(dummies[d])
        else:
            keep.append(dummies[d])
    dummies = keep
    # 3. grow the real sequences round-robin
    lists: List[List[int]] = [[] for _ in seq_lens]
    remaining = list(need)
    while any(r > 0 for r in remaining):
        for b in range(len(lists)):
            if remaining[b] <= 0:
                continue
            while len(alloc) == 0:
                if not dummies:
                    raise RuntimeError("churn fixture ran out of blocks")
                j = int(rng.integers(len(dummies)))
                alloc.release(dummies.pop(j))
            lists[b].append(alloc.alloc())
            remaining[b] -= 1
    return Layout(geom, seq_lens, q_lens, _tables_from_lists(lists, spare), spare)


# ---------------------------------------------------------------------------
# values
# ---------------------------------------------------------------------------
def _draw(rng, shape, dtype: str, scale: float) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if scale != 1.0:
        x = (x * np.float32(scale)).astype(np.float32)
    return x if dtype == F32 else f32_to_bf16_bits(x)


def draw_layer_values(layout: Layout, rng) -> LayerValues:
    g = layout.geom
    T = layout.T_total
    npre = int(layout.prefix_lens.sum())
    s = g.value_scale
    return LayerValues(
        q=_draw(rng, (T, g.H_q, g.D), g.dtype, s),
        k_new=_draw(rng, (T, g.H_kv, g.D), g.dtype, s),
        v_new=_draw(rng, (T, g.H_kv, g.D), g.dtype, s),
        k_prefix=_draw(rng, (npre, g.H_kv, g.D), g.dtype, s),
        v_prefix=_draw(rng, (npre, g.H_kv, g.D), g.dtype, s),
    )


def empty_pool(geom: Geometry) -> np.ndarray:
    """A pool filled with NaN (every slot no live position owns stays NaN)."""
    shape = (geom.N, geom.P, geom.H_kv, geom.D)
    return np.full(shape, NAN_BITS[geom.dtype], dtype=np_storage_dtype(geom.dtype))


def dense_sequence(layout: Layout, vals: LayerValues, b: int, which: str) -> np.ndarray:
    """Sequence b's K (or V) rows by logical position, straight from the drawn values.

    Never touches a pool: prefix rows then new rows, in position order.
    """
    pre = vals.k_prefix if which == "k" else vals.v_prefix
    new = vals.k_new if which == "k" else vals.v_new
    cp, cq = layout.cu_prefix, layout.cu_q_lens
    return np.concatenate([pre[cp[b]:cp[b + 1]], new[cq[b]:cq[b + 1]]], axis=0)


# ---------------------------------------------------------------------------
# the named workloads
# ---------------------------------------------------------------------------
def tiny_decode(seed: int = 0) -> Layout:
    """Tiny fp32 decode: B=4, cached {5,17,33,64}, H_q=4, H_kv=2, D=64, P=16, N=32."""
    rng = np.random.default_rng(seed)
    geom = Geometry(H_q=4, H_kv=2, D=64, P=16, N=32, dtype=F32, L=1)
    cached = np.array([5, 17, 33, 64], dtype=np.int32)
    return layout_from_permutation(geom, cached + 1, np.ones(4, np.int32), rng)


def gpt2_decode(seed: int = 0) -> Layout:
    """GPT-2-small decode: MHA 12 heads, D=64, L=12, P=16, bf16, B=32, ctx ~ U{64..1024}."""
    rng = np.random.default_rng(seed)
    B = 32
    cached = rng.integers(64, 1025, size=B).astype(np.int32)
    seq = cached + 1
    P = 16
    N = sum(_blocks_for(L, P) for L in seq) + 1     # exactly what is needed, plus the spare
    geom = Geometry(H_q=12, H_kv=12, D=64, P=P, N=N, dtype=BF16, L=12,
                    value_scale=1.0 / math.sqrt(64))
    return layout_from_permutation(geom, seq, np.ones(B, np.int32), rng)


def llama1b_decode(seed: int = 0) -> Layout:
    """Llama-3.2-1B decode: H_q=32, H_kv=8, D=64, L=16, P=16, bf16, B=64, ctx log-uniform [32,4096]."""
    rng = np.random.default_rng(seed)
    B = 64
    cached = np.round(np.exp(rng.uniform(math.log(32), math.log(4096), size=B))).astype(np.int32)
    seq = cached + 1
    P = 16
    N = int(math.ceil(1.1 * sum(_blocks_for(L, P) for L in seq))) + 1
    geom = Geometry(H_q=32, H_kv=8, D=64, P=P, N=N, dtype=BF16, L=16)
    return layout_from_permutation(geom, seq, np.ones(B, np.int32), rng)


def _llama8b_geom(N: int, P: int = 16) -> Geometry:
    return Geometry(H_q=32, H_kv=8, D=128, P=P, N=N, dtype=BF16, L=32)


def llama8b_decode(B: int = 231, seed: int = 0) -> Layout:
    """Llama-3-8B large-batch decode: H_q=32, H_kv=8, D=128, L=32, P=16, bf16.

    Prompt ~ lognormal(median 1000, sigma 1.0) capped at 8192, plus output
    ~ U{1..512}; tables fragmented by the churn fixture.
    """
    rng = np.random.default_rng(seed)
    prompt = np.clip(np.round(rng.lognormal(math.log(1000.0), 1.0, size=B)), 1, 8192)
    output = rng.integers(1, 513, size=B)
    cached = (prompt + output).astype(np.int32)
    seq = cached + 1
    return layout_with_churn(_llama8b_geom, seq, np.ones(B, np.int32), rng)


def mixed_step(seed: int = 0, n_prefill: int = 8, n_decode: int = 120) -> Tuple[Layout, Layout]:
    """Mixed continuous-batching step at Llama-3-8B shapes (bf16).

    8 prefill requests: new tokens ~ U{128..2048} on cached prefixes ~ U{0..2048};
    120 decode sequences with contexts ~ U{256..8192}.  One pool, one churned
    allocation for both groups.  Returns (prefill_layout, decode_layout), which
    share the pool geometry.
    """
    rng = np.random.default_rng(seed)
    n_new = rng.integers(128, 2049, size=n_prefill).astype(np.int32)
    prefix = rng.integers(0, 2049, size=n_prefill).astype(np.int32)
    ctx = rng.integers(256, 8193, size=n_decode).astype(np.int32)
    seq = np.concatenate([prefix + n_new, ctx + 1]).astype(np.int32)
    ql = np.concatenate([n_new, np.ones(n_decode, np.int32)]).astype(np.int32)
    both = layout_with_churn(_llama8b_geom, seq, ql, rng)
    pf = Layout(both.geom, seq[:n_prefill], ql[:n_prefill],
                both.block_tables[:n_prefill].copy(), both.spare_block)
    dc = Layout(both.geom, seq[n_prefill:], ql[n_prefill:],
                both.block_tables[n_prefill:].copy(), both.spare_block)
    return pf, dc


# ---------------------------------------------------------------------------
# device-side values for the large workloads (host RNG would take minutes)
# ---------------------------------------------------------------------------
def live_slot_mask(layouts) -> np.ndarray:
    """bool [N*P]: slots that hold a cached prefix position of some sequence."""
    layouts = layouts if isinstance(layouts, (list, tuple)) else [layouts]
    g = layouts[0].geom
    live = np.zeros(g.N * g.P, dtype=bool)
    for lay in layouts:
        live[lay.prefix_slots()] = True
    return live


def device_pools(layouts, seed: int, device="cuda"):
    """K and V pools on the device: N(0,1)*scale bf16/f32 draws from a seeded torch
    generator in every slot that holds a cached prefix position, NaN elsewhere
    (this step's new slots included: the step's scatter fills them)."""
    import torch
    layouts = layouts if isinstance(layouts, (list, tuple)) else [layouts]
    g = layouts[0].geom
    tdt = torch.float32 if g.dtype == F32 else torch.bfloat16
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    dead = torch.from_numpy(~live_slot_mask(layouts)).to(device)
    pools = []
    for _ in range(2):
        pool = torch.empty((g.N * g.P, g.H_kv, g.D), dtype=tdt, device=device)
        pool.normal_(0.0, g.value_scale, generator=gen)
        pool[dead] = float("nan")
        pools.append(pool.view(g.N, g.P, g.H_kv, g.D))
    return pools[0], pools[1]


def device_step_values(layout: Layout, seed: int, device="cuda"):
    """q [T_total, H_q, D], k_new, v_new [T_total, H_kv, D] on the device (seeded torch draws)."""
    import torch
    g = layout.geom
    tdt = torch.float32 if g.dtype == F32 else torch.bfloat16
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    T = layout.T_total
    out = []
    for shape in ((T, g.H_q, g.D), (T, g.H_kv, g.D), (T, g.H_kv, g.D)):
        t = torch.empty(shape, dtype=tdt, device=device)
        t.normal_(0.0, g.value_scale, generator=gen)
        out.append(t)
    return tuple(out)


WORKLOADS = {
    "tiny": "tiny fp32 paged decode (B=4, H_q=4, H_kv=2, D=64, P=16, N=32)",
    "gpt2": "GPT-2-small-shaped decode (MHA 12 heads, D=64, L=12, B=32, bf16)",
    "llama1b": "Llama-3.2-1B-shaped decode (H_q=32, H_kv=8, D=64, L=16, B=64, bf16)",
    "llama8b": "Llama-3-8B-shaped decode (H_q=32, H_kv=8, D=128, L=32, bf16, B in {118,231})",
    "mixed": "mixed step at Llama-3-8B shapes (8 prefills + 120 decodes, bf16)",
}


# ---------------------------------------------------------------------------
# prefix sharing with copy-on-write (tiny-vllm-py, "Prefix Sharing"; ember's next
# steps: "copy-on-write block tables")
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class SharedPrefixStep:
    """R requests share a cached prefix of c tokens, then each decodes one token.

    Before the step every table points at the same prefix blocks (request 0 owns
    them).  If c % P != 0 the last prefix block is partly filled and every other
    request must write into it: it gets a private copy first (copy-on-write), and
    its table is switched to the copy.  ``post`` is the step's decode layout (its
    tables after the switch); ``cow_pairs`` the (source, destination) blocks to copy;
    ``prefix_slots`` where the shared prefix was written (request 0's table).
    """
    geom: Geometry
    prefix_len: int
    pre_tables: np.ndarray     # int32 [R, M] before copy-on-write
    post: Layout               # decode layout after it (seq_lens = c + 1)
    cow_pairs: np.ndarray      # int32 [n, 2] (src, dst)
    prefix_slots: np.ndarray   # int64 [c]


def shared_prefix_step(H_q: int, H_kv: int, D: int, P: int, dtype: str, n_req: int, prefix_len: int,
                       seed: int = 0, spare_blocks: int = 3) -> SharedPrefixStep:
    rng = np.random.default_rng(seed)
    c = int(prefix_len)
    shared = _blocks_for(c, P)
    partial = c % P != 0
    # blocks: the shared prefix, plus per request either a copy of the partial tail
    # (requests 1..R-1) or a fresh block for position c (when the prefix ends on a
    # block boundary), plus spares
    extra = (n_req - 1) if partial else n_req
    N = shared + extra + spare_blocks
    geom = Geometry(H_q=H_q, H_kv=H_kv, D=D, P=P, N=N, dtype=dtype)
    alloc = BlockAllocator(N, rng)
    prefix_blocks = [alloc.alloc() for _ in range(shared)]
    pre_lists = [list(prefix_blocks) for _ in range(n_req)]
    post_lists = [list(prefix_blocks) for _ in range(n_req)]
    pairs = []
    for r in range(n_req):
        if partial:
            if r > 0:
                dst = alloc.alloc()
                pairs.append((prefix_blocks[-1], dst))
                post_lists[r][-1] = dst
        else:
            post_lists[r].append(alloc.alloc())
    spare = alloc.alloc()
    seq_lens = np.full(n_req, c + 1, dtype=np.int32)
    post = Layout(geom, seq_lens, np.ones(n_req, np.int32), _tables_from_lists(post_lists, spare), spare)
    pre_tables = _tables_from_lists(pre_lists, spare)
    prefix_slots = (np.asarray(prefix_blocks, np.int64)[np.arange(c) // P] * P + np.arange(c) % P).astype(np.int64)
    return SharedPrefixStep(geom, c, pre_tables, post, np.asarray(pairs, np.int32).reshape(-1, 2), prefix_slots)


def draw_shared_prefix_values(step: SharedPrefixStep, rng) -> LayerValues:
    """Values of a shared-prefix step: one prefix (repeated per request, so the
    contiguous brute force sees every request's full sequence), one new token and
    one query per request."""
    g = step.geom
    R, c, s = step.post.B, step.prefix_len, g.value_scale
    kp = _draw(rng, (c, g.H_kv, g.D), g.dtype, s)
    vp = _draw(rng, (c, g.H_kv, g.D), g.dtype, s)
    return LayerValues(
        q=_draw(rng, (R, g.H_q, g.D), g.dtype, s),
        k_new=_draw(rng, (R, g.H_kv, g.D), g.dtype, s),
        v_new=_draw(rng, (R, g.H_kv, g.D), g.dtype, s),
        k_prefix=np.concatenate([kp] * R, axis=0) if R else kp[:0],
        v_prefix=np.concatenate([vp] * R, axis=0) if R else vp[:0],
    )


def cow_copy_workload(H_kv: int = 8, D: int = 128, P: int = 16, n_pairs: int = 4096, seed: int = 0):
    """Block pairs for timing the copy: n_pairs distinct sources and distinct
    destinations drawn from a pool of 3 * n_pairs blocks (Llama-3-8B shapes: 32 KB a
    block and pool)."""
    rng = np.random.default_rng(seed)
    N = 3 * n_pairs
    perm = rng.permutation(N).astype(np.int32)
    pairs = np.stack([perm[:n_pairs], perm[n_pairs:2 * n_pairs]], axis=1)
    geom = Geometry(H_q=4 * H_kv, H_kv=H_kv, D=D, P=P, N=N, dtype=BF16)
    return geom, pairs


# ---------------------------------------------------------------------------
# small custom layouts used by tests
# ---------------------------------------------------------------------------
def custom_layout(H_q: int, H_kv: int, D: int, P: int, dtype: str, seq_lens, q_lens=None,
                  seed: int = 0, spare_blocks: int = 3, value_scale: float = 1.0) -> Layout:
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    q_lens = np.ones_like(seq_lens) if q_lens is None else np.asarray(q_lens, dtype=np.int32)
    N = sum(_blocks_for(L, P) for L in seq_lens) + spare_blocks
    geom = Geometry(H_q=H_q, H_kv=H_kv, D=D, P=P, N=N, dtype=dtype, value_scale=value_scale)
    return layout_from_permutation(geom, seq_lens, q_lens, np.random.default_rng(seed))
