"""Seeded synthetic inputs for the DSA indexer path.

This module only draws random numbers and lays them out as a batch: it holds
none of the indexer's arithmetic (no quantisation, no scores, no top-k, no
index conversion). Both the CUDA path and the CPU oracle take their inputs
from here, so the two sides see byte-identical data.

Random numbers come from a counter-based generator (SplitMix64 finaliser over
``seed, stream, counter``), so every tensor is reproducible element by element
on any machine, independently of numpy's own generators. Normals use the
Box-Muller transform in fp64 and are rounded to bf16 (round to nearest even)
where the path consumes bf16.

Shapes follow DeepSeek-V3.2's indexer: 64 query heads of dim 128 sharing one
K row per token (MQA), head weights ``w`` in fp32, a paged K cache of 64-slot
blocks reached through a block table, decode requests first in the batch.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os

import numpy as np

N_HEADS = 64
HEAD_DIM = 128
ROPE_DIM = 64
BLOCK_SIZE = 64

# Stream ids: one independent counter space per tensor of a batch.
STREAM_Q = 1
STREAM_K_CTX = 2
STREAM_K_NEW = 3
STREAM_W = 4
STREAM_LEN = 5
STREAM_PERM = 6

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (Steele, Lea, Flood 2014)."""
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _stream_key(seed: int, stream: int) -> np.uint64:
    base = np.array([(int(seed) & 0xFFFFFFFFFFFF) * 1024 + int(stream)], dtype=np.uint64)
    return _mix64(base)[0]


def random_u64(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """``n`` 64-bit words ``mix64(key + (start+i+1)*gamma)``."""
    key = _stream_key(seed, stream)
    z = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    t = np.empty_like(z)
    with np.errstate(over="ignore"):
        np.multiply(z, _GAMMA, out=z)
        np.add(z, key, out=z)
        for shift, mul in ((30, _M1), (27, _M2), (31, None)):
            np.right_shift(z, np.uint64(shift), out=t)
            np.bitwise_xor(z, t, out=z)
            if mul is not None:
                np.multiply(z, mul, out=z)
    return z


def uniform01(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """Uniform doubles in (0, 1] with 53 random bits."""
    u = random_u64(seed, stream, n, start) >> np.uint64(11)
    return (u.astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def _normal_chunk(seed: int, stream: int, out: np.ndarray, p0: int, p1: int, n: int) -> None:
    u = uniform01(seed, stream, 2 * (p1 - p0), start=2 * p0)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    a = (2.0 * math.pi) * u[1::2]
    lo = 2 * p0
    hi = min(n, 2 * p1)
    z = np.empty(2 * (p1 - p0), dtype=np.float64)
    np.multiply(r, np.cos(a), out=z[0::2])
    np.multiply(r, np.sin(a), out=z[1::2])
    out[lo:hi] = z[: hi - lo]


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """``n`` standard normals (fp64) by Box-Muller; chunks run on a thread pool."""
    out = np.empty(n, dtype=np.float64)
    pairs = (n + 1) // 2
    spans = [(p0, min(pairs, p0 + _CHUNK)) for p0 in range(0, pairs, _CHUNK)]
    if len(spans) <= 1:
        for p0, p1 in spans:
            _normal_chunk(seed, stream, out, p0, p1, n)
        return out
    workers = min(len(spans), os.cpu_count() or 1, 16)
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        list(ex.map(lambda sp: _normal_chunk(seed, stream, out, sp[0], sp[1], n), spans))
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64/fp32 values to bf16 (via fp32, ties to even); uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def uniform_int(seed: int, stream: int, lo: int, hi: int, n: int) -> np.ndarray:
    """``n`` integers uniform on [lo, hi] (inclusive)."""
    span = hi - lo + 1
    u = uniform01(seed, stream, n)
    return (lo + np.minimum(np.floor((1.0 - u) * span), span - 1)).astype(np.int64)


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """A seeded permutation of ``range(n)``: argsort of random 64-bit keys."""
    return np.argsort(random_u64(seed, stream, n), kind="stable").astype(np.int64)


def rope_cos_sin(max_pos: int, theta: float = 10000.0) -> np.ndarray:
    """The rotary angles as a model holds them: float32 [max_pos, 64], row p =
    cos(p * f_i) for i < 32, then sin(p * f_i), f_i = theta^(-2i/64) (fp64,
    rounded to fp32). Input preparation: the path receives this table."""
    half = ROPE_DIM // 2
    inv = theta ** (-2.0 * np.arange(half, dtype=np.float64) / ROPE_DIM)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def rope_neox(x: np.ndarray, positions: np.ndarray, theta: float = 10000.0) -> np.ndarray:
    """Rotary position embedding on dims ``[0, ROPE_DIM)`` of the last axis (fp64).

    Input preparation only: the indexer receives q and k after rotation. The
    rotated subspace is the leading ``ROPE_DIM`` dims; pairs are (i, i+32)
    (half-split), with inverse frequency ``theta^(-2i/ROPE_DIM)``.
    ``x`` has shape ``[N, ..., HEAD_DIM]`` and ``positions`` ``[N]``.
    """
    half = ROPE_DIM // 2
    inv = theta ** (-2.0 * np.arange(half, dtype=np.float64) / ROPE_DIM)
    ang = positions.astype(np.float64)[:, None] * inv[None, :]
    shape = (x.shape[0],) + (1,) * (x.ndim - 2) + (half,)
    c = np.cos(ang).reshape(shape)
    s = np.sin(ang).reshape(shape)
    y = x.copy()
    a = x[..., :half]
    b = x[..., half:ROPE_DIM]
    y[..., :half] = a * c - b * s
    y[..., half:ROPE_DIM] = b * c + a * s
    return y


@dataclasses.dataclass
class Batch:
    """One step's input for one indexer layer, host-side numpy arrays.

    Requests ``[0, num_decodes)`` are decodes (one query token each), the rest
    are prefills; query token ``i`` of request ``r`` sits at position
    ``seq_lens[r] - q_len[r] + i``.  ``ctx_*`` is the K of the tokens already
    in the cache before this step (the cache state), ``k_new`` the K of this
    step's query tokens, which the path writes at ``slot_mapping``.
    """

    name: str
    topk: int
    num_decodes: int
    seq_lens: np.ndarray          # int32 [B]
    query_start_loc: np.ndarray   # int32 [B+1]
    req_id_per_token: np.ndarray  # int32 [T]
    positions: np.ndarray         # int64 [T]
    block_table: np.ndarray       # int32 [B, bt_stride]
    num_blocks: int
    q: np.ndarray                 # uint16 (bf16 bits) [T, 64, 128]
    w: np.ndarray                 # float32 [T, 64]
    k_new: np.ndarray             # uint16 (bf16 bits) [T, 128]
    slot_mapping: np.ndarray      # int64 [T]
    ctx_k: np.ndarray             # uint16 (bf16 bits) [Nctx, 128]
    ctx_slots: np.ndarray         # int64 [Nctx]
    block_size: int = BLOCK_SIZE

    @property
    def num_reqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.query_start_loc).astype(np.int64)

    def row_lengths(self) -> np.ndarray:
        """Number of visible keys for each query row (position + 1)."""
        return (self.positions + 1).astype(np.int64)

    def num_pairs(self) -> int:
        """Causal (query token, key) pairs scored by one indexer pass."""
        return int(self.row_lengths().sum())


def make_batch(
    seed: int,
    decode_seq_lens,
    prefills,
    topk: int,
    *,
    name: str = "batch",
    identity_table: bool = False,
    rope: bool = False,
    spare_blocks: int = 0,
    bt_pad: int = 0,
    table_seed: int | None = None,
    with_data: bool = True,
) -> Batch:
    """Build a seeded batch.

    ``decode_seq_lens``: context length (including the new token) of each
    decode request.  ``prefills``: list of ``(seq_len, q_len)`` with
    ``q_len <= seq_len``; the first ``seq_len - q_len`` tokens are already in
    the cache.  Pages of all requests are drawn from one seeded permutation of
    ``[0, num_blocks)`` unless ``identity_table``.  ``with_data=False`` draws
    the metadata only: ``q``, ``w``, ``k_new`` and ``ctx_k`` keep their
    leading dimension and have width 0.
    """
    seq = [int(x) for x in decode_seq_lens] + [int(s) for s, _ in prefills]
    qlen = [1] * len(decode_seq_lens) + [int(q) for _, q in prefills]
    for s, q in zip(seq, qlen):
        if not (1 <= q <= s):
            raise ValueError("need 1 <= q_len <= seq_len")
    B = len(seq)
    bs = BLOCK_SIZE
    pages = [(s + bs - 1) // bs for s in seq]
    total_pages = sum(pages)
    num_blocks = total_pages + spare_blocks
    if identity_table:
        perm = np.arange(num_blocks, dtype=np.int64)
    else:
        perm = permutation(seed if table_seed is None else table_seed, STREAM_PERM, num_blocks)
    bt_stride = max(pages, default=1) + bt_pad
    block_table = np.full((B, bt_stride), -1, dtype=np.int32)
    cur = 0
    for r in range(B):
        block_table[r, : pages[r]] = perm[cur : cur + pages[r]]
        cur += pages[r]

    qsl = np.zeros(B + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(qlen)
    T = int(qsl[-1])
    req = np.repeat(np.arange(B, dtype=np.int32), qlen)
    pos = np.concatenate(
        [np.arange(s - q, s, dtype=np.int64) for s, q in zip(seq, qlen)]
    ) if B else np.zeros(0, dtype=np.int64)

    slot_new = block_table[req, pos // bs].astype(np.int64) * bs + pos % bs
    ctx_req = np.repeat(np.arange(B, dtype=np.int64), [s - q for s, q in zip(seq, qlen)])
    ctx_positions = (
        np.concatenate([np.arange(0, s - q, dtype=np.int64) for s, q in zip(seq, qlen)])
        if B else np.zeros(0, np.int64)
    )
    ctx_slots = block_table[ctx_req, ctx_positions // bs].astype(np.int64) * bs + ctx_positions % bs
    n_ctx = int(ctx_slots.shape[0])

    if not with_data:
        return Batch(
            name=name, topk=int(topk), num_decodes=len(decode_seq_lens), seq_lens=np.asarray(seq, dtype=np.int32),
            query_start_loc=qsl, req_id_per_token=req, positions=pos, block_table=block_table,
            num_blocks=num_blocks, q=np.zeros((T, 0, 0), np.uint16), w=np.zeros((T, 0), np.float32),
            k_new=np.zeros((T, 0), np.uint16), slot_mapping=slot_new, ctx_k=np.zeros((n_ctx, 0), np.uint16),
            ctx_slots=ctx_slots)
    qf = normal(seed, STREAM_Q, T * N_HEADS * HEAD_DIM).reshape(T, N_HEADS, HEAD_DIM)
    kn = normal(seed, STREAM_K_NEW, T * HEAD_DIM).reshape(T, HEAD_DIM)
    kc = normal(seed, STREAM_K_CTX, n_ctx * HEAD_DIM).reshape(n_ctx, HEAD_DIM)
    if rope:
        qf = rope_neox(qf, pos)
        kn = rope_neox(kn, pos)
        kc = rope_neox(kc, ctx_positions)
    w = normal(seed, STREAM_W, T * N_HEADS).astype(np.float32).reshape(T, N_HEADS)
    return Batch(
        name=name,
        topk=int(topk),
        num_decodes=len(decode_seq_lens),
        seq_lens=np.asarray(seq, dtype=np.int32),
        query_start_loc=qsl,
        req_id_per_token=req,
        positions=pos,
        block_table=block_table,
        num_blocks=num_blocks,
        q=bf16_bits(qf),
        w=w,
        k_new=bf16_bits(kn),
        slot_mapping=slot_new,
        ctx_k=bf16_bits(kc),
        ctx_slots=ctx_slots,
    )


# --------------------------------------------------------------------------
# The five workloads, at full size and scaled down.  Seed 0 for the T=512
# prefill, seeds 1-4 for the others; layer l of the stack uses 1000*5 + l.
# --------------------------------------------------------------------------

def prefill512(scale: float = 1.0) -> Batch:
    """Single request, causal prefill of 512 tokens with RoPE, identity table, top-128."""
    T = max(8, int(512 * scale))
    return make_batch(0, [], [(T, T)], 128, name="prefill512", identity_table=True, rope=True)


def decode32(scale: float = 1.0, n_reqs: int = 32) -> Batch:
    """32 decode requests, context uniform on [4096, 8192], permuted table, top-2048."""
    lo, hi = int(4096 * scale), int(8192 * scale)
    lens = uniform_int(1, STREAM_LEN, max(2, lo), max(2, hi), n_reqs)
    topk = 2048 if scale >= 1.0 else max(16, int(2048 * scale) // 4 * 4)
    return make_batch(1, lens, [], topk, name="decode32")


def prefill4x8k(scale: float = 1.0, n_reqs: int = 4) -> Batch:
    """4 causal prefills of 8192 tokens (fresh requests), shuffled pages, top-2048."""
    L = max(8, int(8192 * scale))
    topk = 2048 if scale >= 1.0 else max(16, int(2048 * scale) // 4 * 4)
    return make_batch(2, [], [(L, L)] * n_reqs, topk, name="prefill4x8k")


def decode8x128k(scale: float = 1.0, n_reqs: int = 8) -> Batch:
    """8 decode requests at 131072 context, random table, top-2048."""
    L = max(2, int(131072 * scale))
    topk = 2048 if scale >= 1.0 else max(16, int(2048 * scale) // 4 * 4)
    return make_batch(3, [L] * n_reqs, [], topk, name="decode8x128k")


STACK_LAYERS = 61
STACK_FREQ = 4


def stack_layer(layer: int, scale: float = 1.0, n_decode: int = 64, with_data: bool = True) -> Batch:
    """One F layer's batch of the 61-layer stack: 64 decodes at 32768 + a 4096-token prefill.

    Every F layer has its own seeded q, w, new K and K cache (seed 5000+layer);
    all layers share the step's metadata (lengths and block table, seed 5).
    """
    L = max(2, int(32768 * scale))
    P = max(8, int(4096 * scale))
    topk = 2048 if scale >= 1.0 else max(16, int(2048 * scale) // 4 * 4)
    return make_batch(1000 * 5 + layer, [L] * n_decode, [(P, P)], topk, name=f"stack61.l{layer}", table_seed=5,
                      with_data=with_data)


WORKLOADS = {
    "prefill512": prefill512,
    "decode32": decode32,
    "prefill4x8k": prefill4x8k,
    "decode8x128k": decode8x128k,
}
