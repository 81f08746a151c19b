"""Seeded synthetic inputs shared by the oracle checks, the GPU tests and the
benchmark.

This module draws data and lays out cache structures (ring offsets, page
tables, tree parents); it holds none of the attention arithmetic. Everything is
drawn with a CPU `torch.Generator`: values are fp32 N(0, 1) rounded to bf16
(round-to-nearest-even) and returned as numpy uint16 bit patterns; metadata is
int32. Slots and pages that hold no token are filled with a bf16 NaN, so a
kernel that reads them instead of skipping them produces NaN.

Workloads (each a seeded recipe; seed = the workload's index unless given):
  * single sliding layer: 1 stream, 8 q / 2 KV heads, head_dim 256, a ring of
    511 slots with 300 written from a uniform random start, RoPE on 256 dims
    with theta 1e4 at position 300, sigmoid gate logits N(0, 1);
  * hybrid 28-layer step: [sliding x3, full] x7, 8 q / 2 KV heads, head_dim 256;
    sliding rings full (511), full layers paged (16-token pages, permuted);
  * paged batched decode: 64 streams, lengths U[64, 4096], 16-token pages,
    permuted page table, 16 q / 8 KV heads, head_dim 128, theta 1e6, no gate;
  * tree verify: 16 streams x 16 rows, best-first trees (parent drawn uniformly
    among earlier nodes of depth < 7), prefix U[512, 8192], 24 q / 4 KV heads,
    head_dim 256, RoPE on 64 dims theta 5e6;
  * long context: 8 q / 2 KV heads, head_dim 256, 64-token pages, 1,048,576
    tokens at 1 stream or 262,144 at 8.
"""
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

NAN_BF16 = 0x7FC0


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, gen: torch.Generator, chunk: int = 1 << 26) -> np.ndarray:
    """fp32 N(0,1) rounded to bf16, as uint16 bits. Large draws go in chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn(e - s, generator=gen, dtype=torch.float32).to(torch.bfloat16)
        out[s:e] = x.view(torch.int16).numpy().view(np.uint16)
    return out.reshape(shape)


def randint(lo: int, hi: int, size, gen: torch.Generator) -> np.ndarray:
    """Uniform integers in [lo, hi] (inclusive)."""
    return torch.randint(lo, hi + 1, tuple(np.atleast_1d(size)), generator=gen).numpy().astype(np.int32)


def randperm(n: int, gen: torch.Generator) -> np.ndarray:
    return torch.randperm(n, generator=gen).numpy().astype(np.int32)


# --------------------------------------------------------------------- layers

@dataclass
class RopeSpec:
    rotary_dim: int
    theta: float


SLIDING_ROPE = RopeSpec(256, 1e4)   # sliding layers: all 256 dims, theta 1e4
FULL_ROPE = RopeSpec(64, 5e6)       # full layers: first quarter, theta 5e6


@dataclass
class DecodeInputs:
    """New-token inputs of one decode call."""
    q: np.ndarray        # [B, Hq, D] u16
    k_new: np.ndarray    # [B, Hkv, D] u16
    v_new: np.ndarray    # [B, Hkv, D] u16
    gate: Optional[np.ndarray]  # [B, Hq] u16 or None
    pos: np.ndarray      # [B] i32


@dataclass
class RingCache:
    k: np.ndarray            # [rows, Hkv, R, D] u16
    v: np.ndarray
    head: np.ndarray         # [B] i32: slot the new entry goes to
    count: np.ndarray        # [B] i32: valid slots (the `count` before head)
    stream_rows: np.ndarray  # [B] i32

    @property
    def R(self):
        return self.k.shape[2]


@dataclass
class PagedCache:
    k: np.ndarray            # [num_pages, Hkv, P, D] u16
    v: np.ndarray
    block_table: np.ndarray  # [B, max_pages] i32 (-1 past the stream's pages)
    seq_len: np.ndarray      # [B] i32 cached tokens

    @property
    def P(self):
        return self.k.shape[2]


@dataclass
class DecodeCase:
    Hq: int
    Hkv: int
    D: int
    rope: RopeSpec
    cache: object            # RingCache or PagedCache
    inputs: DecodeInputs
    meta: dict = field(default_factory=dict)

    @property
    def kind(self):
        return "ring" if isinstance(self.cache, RingCache) else "paged"


def decode_inputs(gen, B, Hq, Hkv, D, pos, gate: bool) -> DecodeInputs:
    q = randn_bf16((B, Hq, D), gen)
    k = randn_bf16((B, Hkv, D), gen)
    v = randn_bf16((B, Hkv, D), gen)
    g = randn_bf16((B, Hq), gen) if gate else None
    return DecodeInputs(q, k, v, g, np.asarray(pos, np.int32).reshape(B))


NAN_E4M3 = 0x7F


def rand_e4m3(shape, gen: torch.Generator, max_exp: int = 8) -> np.ndarray:
    """Random E4M3 codes as uint8, drawn as bit fields: a uniform sign, an
    exponent field in [0, max_exp] (magnitudes below 2^(max_exp - 6)) and a
    uniform 3-bit mantissa."""
    n = int(np.prod(shape))
    sign = torch.randint(0, 2, (n,), generator=gen).numpy().astype(np.uint8)
    exp = torch.randint(0, max_exp + 1, (n,), generator=gen).numpy().astype(np.uint8)
    man = torch.randint(0, 8, (n,), generator=gen).numpy().astype(np.uint8)
    return ((sign << 7) | (exp << 3) | man).reshape(shape)


def e4m3_pool_like(pool_bf16: np.ndarray, gen: torch.Generator, max_exp: int = 8) -> np.ndarray:
    """An E4M3 pool with the same written slots as a bf16 pool: random codes
    where the bf16 pool holds data, NaN (0x7f) where it holds NaN."""
    out = rand_e4m3(pool_bf16.shape, gen, max_exp)
    out[pool_bf16 == NAN_BF16] = NAN_E4M3
    return out


def ring_cache(gen, B, Hkv, D, R, counts, heads=None, n_rows=None, stream_rows=None) -> RingCache:
    """Ring of R slots per (row, KV head). Stream b holds counts[b] entries that
    end just before heads[b] (a uniform random head if not given); every other
    slot is NaN. Extra rows (n_rows > B) are NaN-filled decoys."""
    counts = np.asarray(counts, np.int32).reshape(B)
    if heads is None:
        heads = randint(0, R - 1, B, gen)
    heads = np.asarray(heads, np.int32).reshape(B)
    n_rows = B if n_rows is None else n_rows
    if stream_rows is None:
        stream_rows = np.arange(B, dtype=np.int32)
    stream_rows = np.asarray(stream_rows, np.int32)
    k = np.full((n_rows, Hkv, R, D), NAN_BF16, np.uint16)
    v = np.full((n_rows, Hkv, R, D), NAN_BF16, np.uint16)
    for b in range(B):
        n = int(counts[b])
        if n == 0:
            continue
        slots = (int(heads[b]) - n + np.arange(n)) % R
        k[stream_rows[b]][:, slots] = randn_bf16((Hkv, n, D), gen)
        v[stream_rows[b]][:, slots] = randn_bf16((Hkv, n, D), gen)
    return RingCache(k, v, heads, counts, stream_rows)


def paged_cache(gen, B, Hkv, D, P, seq_lens, room: int = 1, spare_pages: int = 3,
                permute: bool = True) -> PagedCache:
    """Paged leases: stream b owns ceil((seq_lens[b] + room) / P) pages, drawn
    from a randomly permuted physical pool (room = slots kept free after the
    cached tokens for the entries a call writes back). Unused page slots, the
    free room and spare pages are NaN."""
    seq_lens = np.asarray(seq_lens, np.int32).reshape(B)
    npages = [(int(n) + room + P - 1) // P for n in seq_lens]
    total = sum(npages) + spare_pages
    phys = randperm(total, gen) if permute else np.arange(total, dtype=np.int32)
    max_pages = max(npages) if B else 1
    bt = np.full((B, max(max_pages, 1)), -1, np.int32)
    k = np.full((total, Hkv, P, D), NAN_BF16, np.uint16)
    v = np.full((total, Hkv, P, D), NAN_BF16, np.uint16)
    nxt = 0
    for b in range(B):
        bt[b, : npages[b]] = phys[nxt: nxt + npages[b]]
        nxt += npages[b]
        n = int(seq_lens[b])
        if n == 0:
            continue
        kk = randn_bf16((n, Hkv, D), gen)
        vv = randn_bf16((n, Hkv, D), gen)
        t = np.arange(n)
        pages = bt[b, t // P]
        k[pages, :, t % P, :] = kk
        v[pages, :, t % P, :] = vv
    return PagedCache(k, v, bt, seq_lens)


def tree_parents(gen, T: int, max_depth: int = 7) -> np.ndarray:
    """A best-first draft tree of T nodes in creation order: node 0 is the root;
    node i picks its parent uniformly among earlier nodes of depth < max_depth."""
    parent = np.full(T, -1, np.int32)
    depth = np.zeros(T, np.int32)
    for i in range(1, T):
        cand = [j for j in range(i) if depth[j] < max_depth]
        pick = int(torch.randint(0, len(cand), (1,), generator=gen))
        parent[i] = cand[pick]
        depth[i] = depth[parent[i]] + 1
    return parent


def chain_parents(T: int) -> np.ndarray:
    return np.arange(-1, T - 1, dtype=np.int32)


def star_parents(T: int) -> np.ndarray:
    p = np.zeros(T, np.int32)
    p[0] = -1
    return p


@dataclass
class VerifyCase:
    Hq: int
    Hkv: int
    D: int
    rope: RopeSpec
    cache: PagedCache          # prefix; seq_len = prefix_len
    q: np.ndarray              # [S, T, Hq, D]
    k: np.ndarray              # [S, T, Hkv, D] (not rotated)
    v: np.ndarray
    parent: np.ndarray         # [S, T]
    gate: Optional[np.ndarray]  # [S, T, Hq]
    meta: dict = field(default_factory=dict)


# ------------------------------------------------------------------ workloads

def single_sliding_layer(seed: int = 0) -> DecodeCase:
    """1 stream, 8 q / 2 KV heads, head_dim 256, ring of 511, 300 written from a
    uniform random start, RoPE 256 dims theta 1e4 at position 300, gate on."""
    gen = generator(seed)
    B, Hq, Hkv, D, R = 1, 8, 2, 256, 511
    start = int(randint(0, R - 1, 1, gen)[0])
    head = (start + 300) % R
    cache = ring_cache(gen, B, Hkv, D, R, [300], heads=[head])
    inputs = decode_inputs(gen, B, Hq, Hkv, D, [300], gate=True)
    return DecodeCase(Hq, Hkv, D, SLIDING_ROPE, cache, inputs, {"start": start})


HYBRID_PATTERN = ["sliding", "sliding", "sliding", "full"] * 7


def hybrid_layer(seed: int, layer: int, B: int, context: int) -> DecodeCase:
    """Layer `layer` of the 28-layer hybrid step at `context` cached tokens:
    sliding layers hold a full ring (511 = window - 1) unless the context is
    shorter; full layers hold `context` tokens in 16-token permuted pages."""
    gen = generator(seed * 1000 + layer)
    Hq, Hkv, D = 8, 2, 256
    if HYBRID_PATTERN[layer] == "sliding":
        R = 511
        n = min(context, R)
        cache = ring_cache(gen, B, Hkv, D, R, [n] * B)
        inputs = decode_inputs(gen, B, Hq, Hkv, D, [context] * B, gate=True)
        return DecodeCase(Hq, Hkv, D, SLIDING_ROPE, cache, inputs, {"layer": layer})
    cache = paged_cache(gen, B, Hkv, D, 16, [context] * B)
    inputs = decode_inputs(gen, B, Hq, Hkv, D, [context] * B, gate=True)
    return DecodeCase(Hq, Hkv, D, FULL_ROPE, cache, inputs, {"layer": layer})


def paged_batched(seed: int = 2, B: int = 64, lo: int = 64, hi: int = 4096) -> DecodeCase:
    """64 streams, ragged lengths U[64, 4096], 16-token permuted pages, 16 q / 8
    KV heads, head_dim 128, RoPE on all 128 dims theta 1e6, no gate."""
    gen = generator(seed)
    Hq, Hkv, D = 16, 8, 128
    lens = randint(lo, hi, B, gen)
    cache = paged_cache(gen, B, Hkv, D, 16, lens)
    inputs = decode_inputs(gen, B, Hq, Hkv, D, lens, gate=False)
    return DecodeCase(Hq, Hkv, D, RopeSpec(128, 1e6), cache, inputs)


def tree_verify(seed: int = 3, S: int = 16, T: int = 16, lo: int = 512, hi: int = 8192,
                trees: str = "random", gate: bool = False) -> VerifyCase:
    """16 streams x 16 rows of best-first trees over paged prefixes U[512, 8192],
    24 q / 4 KV heads, head_dim 256, RoPE first 64 dims theta 5e6."""
    gen = generator(seed)
    Hq, Hkv, D = 24, 4, 256
    lens = randint(lo, hi, S, gen)
    cache = paged_cache(gen, S, Hkv, D, 16, lens, room=T)
    if trees == "random":
        parent = np.stack([tree_parents(gen, T) for _ in range(S)])
    elif trees == "chain":
        parent = np.stack([chain_parents(T)] * S)
    else:
        parent = np.stack([star_parents(T)] * S)
    q = randn_bf16((S, T, Hq, D), gen)
    k = randn_bf16((S, T, Hkv, D), gen)
    v = randn_bf16((S, T, Hkv, D), gen)
    g = randn_bf16((S, T, Hq), gen) if gate else None
    return VerifyCase(Hq, Hkv, D, FULL_ROPE, cache, q, k, v, parent, g)


def long_context(seed: int = 4, B: int = 1, context: int = 1 << 20) -> DecodeCase:
    """8 q / 2 KV heads, head_dim 256, 64-token pages; 1,048,576 tokens at one
    stream or 262,144 at eight. Full-layer RoPE (64 dims, theta 5e6)."""
    gen = generator(seed)
    Hq, Hkv, D = 8, 2, 256
    cache = paged_cache(gen, B, Hkv, D, 64, [context] * B)
    inputs = decode_inputs(gen, B, Hq, Hkv, D, [context] * B, gate=False)
    return DecodeCase(Hq, Hkv, D, FULL_ROPE, cache, inputs)


# ------------------------------------------------------------------ device-side generation

def hybrid_step_device(seed: int, B: int, context: int, device="cuda"):
    """The 28-layer hybrid step drawn directly on the GPU (same recipe as
    hybrid_layer: bf16 N(0,1) K/V, full sliding rings of 511 slots with a
    uniform random head per stream, full layers in 16-token pages from a
    randomly permuted pool, gate logits N(0,1), positions = context). Returns a
    list of per-layer dicts of device tensors."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    Hq, Hkv, D = 8, 2, 256

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)

    layers = []
    for kind in HYBRID_PATTERN:
        L = {"kind": kind, "q": randn(B, Hq, D), "k_new": randn(B, Hkv, D),
             "v_new": randn(B, Hkv, D), "gate": randn(B, Hq),
             "pos": torch.full((B,), context, dtype=torch.int32, device=device)}
        if kind == "sliding":
            R = 511
            n = min(context, R)
            L.update(rope=SLIDING_ROPE, R=R, k=randn(B, Hkv, R, D), v=randn(B, Hkv, R, D),
                     head=torch.randint(0, R, (B,), generator=g, device=device, dtype=torch.int32),
                     count=torch.full((B,), n, dtype=torch.int32, device=device),
                     rows=torch.arange(B, dtype=torch.int32, device=device))
        else:
            P = 16
            per = (context + 1 + P - 1) // P
            total = B * per + 3
            perm = torch.randperm(total, generator=g, device=device).to(torch.int32)
            L.update(rope=FULL_ROPE, P=P, k=randn(total, Hkv, P, D), v=randn(total, Hkv, P, D),
                     block_table=perm[: B * per].reshape(B, per).contiguous(),
                     seq_len=torch.full((B,), context, dtype=torch.int32, device=device))
        layers.append(L)
    return layers


def e4m3_device(gen, shape, device="cuda"):
    """Random E4M3 codes drawn on the device (uniform bytes, NaN codes
    0x7f / 0xff replaced by zero)."""
    t = torch.randint(0, 256, tuple(shape), generator=gen, device=device, dtype=torch.int32).to(torch.uint8)
    t[(t & 0x7F) == 0x7F] = 0
    return t


def paged_device(gen, B, Hkv, D, P, lens, room=1, device="cuda"):
    """Paged pools drawn on the device (bf16 N(0,1) everywhere), page table
    from a random permutation; lens is a host list of cached lengths."""
    lens = [int(n) for n in lens]
    npages = [(n + room + P - 1) // P for n in lens]
    total = sum(npages) + 3
    perm = torch.randperm(total, generator=gen, device=device).to(torch.int32)
    bt = torch.full((B, max(npages)), -1, dtype=torch.int32, device=device)
    nxt = 0
    for b in range(B):
        bt[b, :npages[b]] = perm[nxt:nxt + npages[b]]
        nxt += npages[b]
    k = torch.randn(total, Hkv, P, D, generator=gen, device=device).to(torch.bfloat16)
    v = torch.randn(total, Hkv, P, D, generator=gen, device=device).to(torch.bfloat16)
    seq = torch.tensor(lens, dtype=torch.int32, device=device)
    return k, v, bt, seq
