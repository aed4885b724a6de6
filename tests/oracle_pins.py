"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
if the oracle disagrees with a hand-worked value, a closed form, a library
routine or a brute-force enumeration. ``test_oracle_pins.py`` runs them on
the real oracle; ``test_oracle_mutants.py`` runs them on deliberately broken
builds and requires that each break is caught.

Sources: the web pages "IndexCache：DeepSeek 稀疏注意力中的跨层索引复用"
(atomage.cn; its `Indexer`, FP8 indexer-cache, `SparseAttnIndexer` and layer
schedule snippets), "PR #37735 完整报告" (prhub.com.cn; 关键源码片段 and
风险与影响), the vLLM API page "vllm.v1.attention.backends.mla.index_group"
(`_convert_once`), the OCP 8-bit floating point specification, and the OCP
Microscaling Formats (MX) specification (the E2M1 element of the FP4 cache).
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np
import torch

from dsa_sparse_attention_quant_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
SOFTMAX_SCALE = 128 ** -0.5
HEAD_NORM = 64 ** -0.5


def read_golden(name: str):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def torch_e4m3(values: np.ndarray) -> np.ndarray:
    """Library E4M3 conversion (round to nearest even) with saturation to +-448."""
    t = torch.from_numpy(np.ascontiguousarray(values, np.float32))
    return t.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def torch_e4m3_value(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def bf16(x) -> np.ndarray:
    return synth.bf16_bits(np.asarray(x, np.float64))


# ----------------------------------------------------------------- E4M3

def pin_e4m3_golden(ora):
    for value, code, *_ in read_golden("e4m3_codes.txt"):
        got = ora.e4m3_encode(float(value))
        assert got == int(code, 16), f"e4m3({value}) = {got:#04x}, expected {code}"


def pin_e4m3_values_vs_library(ora):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    lib = torch_e4m3_value(codes)
    mine = np.array([ora.e4m3_value(int(c)) for c in codes])
    assert np.array_equal(np.signbit(mine), np.signbit(lib))
    assert np.array_equal(mine, lib)
    assert math.isnan(ora.e4m3_value(0x7F)) and math.isnan(ora.e4m3_value(0xFF))
    # round trip of every finite code
    for c in codes:
        assert ora.e4m3_encode(ora.e4m3_value(int(c))) == int(c)


def pin_e4m3_all_bf16_vs_library(ora):
    """Every finite bf16 value (the quantiser only ever sees bf16 / 2^k) vs torch."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    vals = (bits << np.uint32(16)).view(np.float32)
    vals = vals[np.isfinite(vals)]
    assert np.array_equal(ora.e4m3_encode_array(vals), torch_e4m3(vals))


def pin_e4m3_random_fp32_brute_force(ora, n: int = 4000):
    """Nearest finite E4M3 by linear scan, ties to the even code, on random fp32."""
    table = [(c, ora_free_value(c)) for c in range(0x7F)]  # non-negative finite codes
    u = synth.uniform01(99, 7, 2 * n)
    mags = np.exp2(u[:n] * 22.0 - 12.0) * (1.0 + u[n:])
    vals = np.where(np.arange(n) % 2 == 0, mags, -mags).astype(np.float32)
    for v in vals:
        a = abs(float(v))
        best = None
        for c, cv in table:
            d = abs(cv - a)
            if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
                best = (d, c)
        want = (best[1] if a < 448.0 else 0x7E) | (0x80 if v < 0 else 0)
        assert ora.e4m3_encode(float(v)) == want, (float(v), want)


def ora_free_value(c: int) -> float:
    """E4M3 value of a non-negative finite code by the OCP formula (test's own)."""
    e, m = c >> 3, c & 7
    return (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)


# ----------------------------------------------------------------- scales

def pin_ue8m0_worked(ora):
    cases = [
        (1.0, 2.0 ** -8),       # 1/448 lies in (2^-9, 2^-8]
        (2.0, 2.0 ** -7),
        (448.0, 1.0),           # exactly a power of two: kept
        (1.75, 2.0 ** -8),      # 1.75/448 = 2^-8 exactly
        (1.7578125, 2.0 ** -7), # next bf16 above 1.75: rounds up
        (0.0, 2.0 ** -42),      # amax floored at 1e-10: 1e-10/448 in (2^-43, 2^-42]
        (3.0e38, 2.0 ** 120),   # 3e38/448 = 6.7e35 in (2^119, 2^120]
    ]
    for amax, want in cases:
        assert ora.ue8m0_scale(amax) == want, (amax, ora.ue8m0_scale(amax), want)


def pin_ue8m0_invariants(ora, n: int = 3000):
    u = synth.uniform01(5, 1, n)
    amaxs = np.exp2(u * 60.0 - 30.0).astype(np.float32)
    for a in amaxs:
        s = ora.ue8m0_scale(float(a))
        m, e = math.frexp(s)
        assert m == 0.5, "scale must be a power of two"
        assert float(a) / s <= 448.0
        assert float(a) / s > 224.0, "scale must be the smallest power of two that fits"


def pin_quant_group_worked(ora):
    x = np.zeros(128, np.float32)
    x[0] = 1.0
    codes, s = ora.quant_group(x)
    assert codes[0] == 0x78 and not codes[1:].any()
    assert np.float32(s).view(np.uint32) == 0x3B800000
    x[0] = 2.0
    codes, s = ora.quant_group(x)
    assert codes[0] == 0x78 and np.float32(s).view(np.uint32) == 0x3C000000
    x[:] = 0
    x[7] = 448.0
    x[8] = -1.0
    codes, s = ora.quant_group(x)
    assert s == 1.0 and codes[7] == 0x7E and codes[8] == 0xB8
    # mixed signs: amax 1 -> scale 2^-8; -1 -> -256 (0xF8); 0.5 -> 128 (0x70); 0.75 -> 192 (0x74)
    x[:] = 0
    x[0], x[1], x[2] = -1.0, 0.5, 0.75
    codes, s = ora.quant_group(x)
    assert s == 2.0 ** -8 and list(codes[:3]) == [0xF8, 0x70, 0x74]


def pin_quant_group_vs_library(ora, n_groups: int = 64):
    """Groups of N(0,1) bf16 values: codes = torch E4M3 of x / (power-of-two scale)."""
    x = synth.bf16_to_f32(bf16(synth.normal(11, 1, n_groups * 128))).reshape(n_groups, 128)
    x[3] *= 1e-20
    x[4] *= 1e20
    x[5] = 0.0
    for g in range(n_groups):
        codes, s = ora.quant_group(x[g])
        amax = float(np.abs(x[g]).max())
        assert s >= max(amax, 1e-10) / 448.0 * (1 - 1e-7)
        assert np.array_equal(codes, torch_e4m3(x[g] / np.float32(s)))
        # dequantised error bound: half an E4M3 step (relative 2^-4) of each value
        deq = torch_e4m3_value(codes) * s
        assert np.all(np.abs(deq - x[g]) <= np.abs(x[g]) * 2.0 ** -4 + s * 2.0 ** -10)


# ----------------------------------------------------------------- cache layout

def pin_slot_layout(ora):
    # 132 bytes per slot (128 K bytes + one fp32 scale), 64 slots per page = 8448 bytes;
    # inside a page the 64 K rows come first, then the 64 scales.
    assert ora.slot_offsets(0) == (0, 8192)
    assert ora.slot_offsets(1) == (128, 8196)
    assert ora.slot_offsets(63) == (63 * 128, 8192 + 63 * 4)
    assert ora.slot_offsets(64) == (8448, 8448 + 8192)
    assert ora.slot_offsets(65) == (8576, 16644)


def pin_k_quant_write_worked(ora):
    cache = ora.new_cache(2)
    k = np.zeros((4, 128), np.float64)
    k[0, 0] = 1.0          # -> code 0x78 at byte 0, scale 2^-8
    k[1, 5] = -2.0         # padding token: must not be written
    k[2, 127] = 448.0      # -> code 0x7E, scale 1.0
    k[3, 0] = 1.0          # slot past the cache: skipped and counted
    slots = np.array([5, -1, 70, 128], np.int64)
    bad = ora.k_quant_write(bf16(k), slots, cache)
    assert bad == 1
    flat = cache.reshape(-1)
    want = np.zeros_like(flat)
    want[5 * 128 + 0] = 0x78
    want[8192 + 5 * 4: 8192 + 5 * 4 + 4] = np.frombuffer(np.float32(2.0 ** -8).tobytes(), np.uint8)
    want[8448 + 6 * 128 + 127] = 0x7E
    want[8448 + 8192 + 6 * 4: 8448 + 8192 + 6 * 4 + 4] = np.frombuffer(np.float32(1.0).tobytes(), np.uint8)
    assert np.array_equal(flat, want)


# ----------------------------------------------------------------- scores

def _cache_with_keys(ora, keys_f64, block_table_row, num_blocks):
    """Write keys at logical positions 0..n-1 through one request's block table."""
    n = keys_f64.shape[0]
    pos = np.arange(n)
    slots = block_table_row[pos // 64].astype(np.int64) * 64 + pos % 64
    cache = ora.new_cache(num_blocks)
    assert ora.k_quant_write(bf16(keys_f64), slots, cache) == 0
    return cache


def pin_logits_hand_case(ora):
    # q head 0 = (2, 0, ...), every other head 0; k = (1, 0, ...); w_0 = 1:
    # I = 1 * ReLU(2 * 1) * 128^-1/2 * 64^-1/2 = 0.0220971 (to 7 digits).
    q = np.zeros((64, 128))
    q[0, 0] = 2.0
    k = np.zeros((1, 128))
    k[0, 0] = 1.0
    w = np.zeros(64, np.float32)
    w[0] = 1.0
    bt = np.array([0], np.int32)
    cache = _cache_with_keys(ora, k, bt, 1)
    qc, qs = ora.q_quant(bf16(q))
    got = ora.logits_row(qc, qs, w, cache, bt, 1)
    assert abs(got[0] - 0.0220971) < 5e-8
    # ReLU: a negative dot product contributes nothing
    q[0, 0] = -2.0
    qc, qs = ora.q_quant(bf16(q))
    assert ora.logits_row(qc, qs, w, cache, bt, 1)[0] == 0.0
    # a negative head weight flips the sign of a positive contribution
    q[0, 0] = 2.0
    w[0] = -1.0
    qc, qs = ora.q_quant(bf16(q))
    assert abs(ora.logits_row(qc, qs, w, cache, bt, 1)[0] + 0.0220971) < 5e-8
    # two heads: 3*ReLU(2*1) + 0.5*ReLU(-4*1) + 2*ReLU(1.5*1) = 9 -> 9 / (sqrt(128)*8)
    q[:] = 0
    q[0, 0], q[1, 0], q[2, 0] = 2.0, -4.0, 1.5
    w[:] = 0
    w[0], w[1], w[2] = 3.0, 0.5, 2.0
    qc, qs = ora.q_quant(bf16(q))
    assert abs(ora.logits_row(qc, qs, w, cache, bt, 1)[0] - 9.0 * SOFTMAX_SCALE * HEAD_NORM) < 1e-12


def pin_logits_matmul_special_case(ora):
    """All inputs positive and exactly representable after quantisation, so the
    ReLU is the identity: I = c * (w^T Q) K^T, a plain float64 matmul."""
    n_keys = 150
    grid = np.arange(8) * 0.25  # {0, .25, ..., 1.75}: x * 256 is an exact E4M3 value
    u = synth.uniform01(3, 1, 64 * 128 + n_keys * 128)
    Q = grid[(u[: 64 * 128] * 8).astype(int) % 8].reshape(64, 128)
    K = grid[(u[64 * 128:] * 8).astype(int) % 8].reshape(n_keys, 128)
    Q[:, 0] = 1.75  # amax 1.75 per row -> scale 2^-8, lossless
    K[:, 0] = 1.75
    w = (0.5 + synth.uniform01(3, 2, 64)).astype(np.float32)
    bt = np.array([2, 0, 1], np.int32)  # a permuted block table
    cache = _cache_with_keys(ora, K, bt, 3)
    qc, qs = ora.q_quant(bf16(Q))
    got = ora.logits_row(qc, qs, w, cache, bt, n_keys)
    want = SOFTMAX_SCALE * HEAD_NORM * ((w.astype(np.float64) @ Q) @ K.T)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=0)


def pin_logits_scale_folding(ora):
    """The pages fold q_scale, softmax_scale and n_head^-0.5 into the weights
    before the op: I = k_scale * sum_h w'_h ReLU(codes_q . codes_k) with
    w' = w * q_scale * softmax_scale * n_head^-0.5. Codes are decoded with the
    library's E4M3 type, not the oracle's decoder."""
    n_keys = 200
    Q = synth.normal(21, 1, 64 * 128).reshape(64, 128)
    Q[7] *= 1e-3   # spread the per-head scales
    Q[9] *= 40.0
    K = synth.normal(21, 2, n_keys * 128).reshape(n_keys, 128)
    K[::3] *= 9.0
    w = synth.normal(21, 3, 64).astype(np.float32)
    bt = np.array([3, 1, 0, 2], np.int32)
    cache = _cache_with_keys(ora, K, bt, 4)
    qc, qs = ora.q_quant(bf16(Q))
    got = ora.logits_row(qc, qs, w, cache, bt, n_keys)
    wf = w.astype(np.float64) * qs.astype(np.float64) * SOFTMAX_SCALE * HEAD_NORM
    cq = torch_e4m3_value(qc)
    pos = np.arange(n_keys)
    slots = bt[pos // 64].astype(np.int64) * 64 + pos % 64
    flat = cache.reshape(-1)
    kcodes = np.stack([flat[(s // 64) * 8448 + (s % 64) * 128:][:128] for s in slots])
    kscale = np.array([np.frombuffer(flat[(s // 64) * 8448 + 8192 + (s % 64) * 4:][:4].tobytes(), np.float32)[0]
                       for s in slots], np.float64)
    ck = torch_e4m3_value(kcodes)
    want = kscale * (np.maximum(cq @ ck.T, 0.0).T @ wf)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-300)


def pin_indexer_causal_rows(ora):
    """A prefill of 70 tokens: row t sees exactly keys 0..t (its own included)."""
    b = synth.make_batch(41, [], [(70, 70)], 8, identity_table=False)
    cache = ora.fill_cache(b)
    topk, scores = ora.indexer(b, cache, with_scores=True)
    for t in range(70):
        n = t + 1
        assert np.all(scores[t, n:] == 0.0)
        want = ora.topk_row(scores[t, :n], 8)
        assert np.array_equal(topk[t], want)
        assert set(topk[t][topk[t] >= 0].tolist()) <= set(range(n))
        assert int((topk[t] >= 0).sum()) == min(8, n)
    assert list(topk[0]) == [0] + [-1] * 7
    # the row's own key is visible: a key that dominates every head lands in the top-1
    q = synth.bf16_to_f32(b.q[69]).astype(np.float64)
    kbig = np.maximum(q.mean(axis=0), 0) * 50 + 1e-3
    b.k_new[69] = bf16(kbig)
    b.w[69] = np.abs(b.w[69])
    cache = ora.fill_cache(b)
    t69 = ora.indexer(b, cache, rows=np.array([69]))
    assert t69[0][0] == 69


def pin_indexer_block_table_invariance(ora):
    """The same request under two different block tables scores identically."""
    b1 = synth.make_batch(52, [300], [], 16, identity_table=True)
    b2 = synth.make_batch(52, [300], [], 16, identity_table=False, spare_blocks=3)
    assert not np.array_equal(b1.block_table[0], b2.block_table[0, :5])
    s1 = ora.indexer(b1, ora.fill_cache(b1), with_scores=True)[1]
    s2 = ora.indexer(b2, ora.fill_cache(b2), with_scores=True)[1]
    assert np.array_equal(s1, s2)


# ----------------------------------------------------------------- FP4 cache

E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # codes 0..7 (OCP MX, FP4 E2M1)


def _e2m1_brute(v: float) -> int:
    """Nearest E2M1 code by enumeration: smallest distance, then the even code;
    magnitudes past 6 saturate. The test's own rule, not the oracle's."""
    sign = 0x8 if math.copysign(1.0, v) < 0 else 0
    a = min(abs(v), 6.0)
    best = min(range(8), key=lambda c: (abs(E2M1_MAGNITUDES[c] - a), c & 1))
    return sign | best


def pin_e2m1_golden(ora):
    for value, code, *_ in read_golden("e2m1_codes.txt"):
        got = ora.e2m1_encode(float(np.float32(float(value))))
        assert got == int(code, 16), (value, hex(got), code)
    for c in range(16):
        want = (-1.0 if c & 8 else 1.0) * E2M1_MAGNITUDES[c & 7]
        got = ora.e2m1_value(c)
        assert got == want and math.copysign(1.0, got) == (-1.0 if c & 8 else 1.0), (c, got)


def pin_e2m1_brute_force(ora, n: int = 3000):
    grid = np.arange(-8 * 64, 8 * 64 + 1) / 64.0  # every multiple of 1/64 in [-8, 8]: all halfway points
    rnd = (synth.normal(91, 1, n) * np.exp2(synth.uniform01(91, 2, n) * 8 - 4)).astype(np.float32)
    for v in np.concatenate([grid.astype(np.float32), rnd]):
        assert ora.e2m1_encode(float(v)) == _e2m1_brute(float(v)), float(v)


def pin_ue8m0_e2m1(ora, n: int = 3000):
    cases = [
        (6.0, 1.0),           # 6/6 = 1: kept
        (1.0, 0.25),          # 1/6 in (2^-3, 2^-2]
        (3.0, 0.5),           # 3/6 = 2^-1 exactly
        (3.015625, 1.0),      # next bf16 above 3: rounds up
        (12.0, 2.0),
        (0.0, 2.0 ** -35),    # amax floored at 1e-10: 1e-10/6 in (2^-36, 2^-35]
    ]
    for amax, want in cases:
        assert ora.ue8m0_scale_e2m1(amax) == want, (amax, ora.ue8m0_scale_e2m1(amax), want)
    u = synth.uniform01(92, 1, n)
    for a in np.exp2(u * 60.0 - 30.0).astype(np.float32):
        s = ora.ue8m0_scale_e2m1(float(a))
        assert math.frexp(s)[0] == 0.5, "scale must be a power of two"
        assert 3.0 < float(a) / s <= 6.0, "scale must be the smallest power of two that fits"


def pin_quant_group_e2m1_vs_brute_force(ora, n_groups: int = 24):
    x = synth.bf16_to_f32(bf16(synth.normal(93, 1, n_groups * 128))).reshape(n_groups, 128)
    x[2] *= 1e-12
    x[3] = 0.0
    for g in range(n_groups):
        packed, s = ora.quant_group_e2m1(x[g])
        assert packed.shape == (64,)
        assert s == ora.ue8m0_scale_e2m1(float(np.abs(x[g]).max()))
        codes = [_e2m1_brute(float(np.float32(v) / np.float32(s))) for v in x[g]]
        assert list(packed & 15) == codes[0::2] and list(packed >> 4) == codes[1::2]
        deq = np.array([(-1.0 if c & 8 else 1.0) * E2M1_MAGNITUDES[c & 7] for c in codes]) * s
        assert np.all(np.abs(deq - x[g]) <= 0.25 * np.abs(x[g]) + 0.25 * s)


def pin_fp4_slot_layout(ora):
    # 68 bytes per slot (64 bytes of E2M1 pairs + one fp32 scale), 64 slots per page = 4352
    # bytes; inside a page the 64 K rows come first, then the 64 scales.
    assert ora.slot_offsets(0, "fp4") == (0, 4096)
    assert ora.slot_offsets(1, "fp4") == (64, 4100)
    assert ora.slot_offsets(63, "fp4") == (63 * 64, 4096 + 63 * 4)
    assert ora.slot_offsets(64, "fp4") == (4352, 4352 + 4096)
    assert ora.slot_offsets(65, "fp4") == (4416, 8452)


def pin_fp4_k_quant_write_worked(ora):
    cache = ora.new_cache(2, "fp4")
    assert cache.shape == (2, 4352)
    k = np.zeros((4, 128), np.float64)
    k[0, 0], k[0, 1], k[0, 3] = 1.0, -0.5, 3.0   # amax 3 -> scale 0.5: codes 0x4, 0xA, 0x0, 0x7
    k[1, 5] = -2.0                                # padding token: must not be written
    k[2, 126], k[2, 127] = 1.0, -12.0             # amax 12 -> scale 2: 0.5 -> 0x1, -6 -> 0xF
    k[3, 0] = 1.0                                 # slot past the cache: skipped and counted
    slots = np.array([5, -1, 70, 128], np.int64)
    assert ora.k_quant_write(bf16(k), slots, cache) == 1
    flat = cache.reshape(-1)
    want = np.zeros_like(flat)
    want[5 * 64 + 0] = 0xA4   # dims 0 (low nibble) and 1 (high nibble)
    want[5 * 64 + 1] = 0x70   # dims 2 and 3
    want[4096 + 5 * 4: 4096 + 5 * 4 + 4] = np.frombuffer(np.float32(0.5).tobytes(), np.uint8)
    want[4352 + 6 * 64 + 63] = 0xF1
    want[4352 + 4096 + 6 * 4: 4352 + 4096 + 6 * 4 + 4] = np.frombuffer(np.float32(2.0).tobytes(), np.uint8)
    assert np.array_equal(flat, want)


def pin_fp4_scores_equal_fp8_on_shared_values(ora):
    """Keys whose values both caches hold exactly (E2M1 magnitudes times a
    power of two, with 6 * 2^j the row's amax) dequantise identically from the
    FP4 and the FP8 cache, so every score and every top-k row of the indexer
    agree exactly between the two: the FP4 decode is tied to the pinned FP8
    path."""
    b = synth.make_batch(94, [150, 1], [(90, 20)], 16)
    u = synth.uniform01(94, 7, (b.ctx_k.shape[0] + b.k_new.shape[0]) * 128)
    mags = np.array(E2M1_MAGNITUDES)[(u * 8).astype(int) % 8]
    sign = np.where(synth.uniform01(94, 8, u.size) < 0.5, -1.0, 1.0)
    vals = (mags * sign).reshape(-1, 128)
    vals[:, 5] = 6.0                                     # amax 6 * 2^j in every row
    j = (np.arange(vals.shape[0]) % 5 - 2).astype(np.float64)
    vals *= np.exp2(j)[:, None]
    n_ctx = b.ctx_k.shape[0]
    b.ctx_k = bf16(vals[:n_ctx])
    b.k_new = bf16(vals[n_ctx:])
    c8 = ora.fill_cache(b)
    c4 = ora.fill_cache(b, fmt="fp4")
    t8, s8 = ora.indexer(b, c8, with_scores=True)
    t4, s4 = ora.indexer(b, c4, with_scores=True)
    assert np.array_equal(s8, s4) and np.array_equal(t8, t4)
    assert np.abs(s8).max() > 0
    # and a single row through logits_row on both caches
    qc, qs = ora.q_quant(b.q[0])
    bt = b.block_table[b.req_id_per_token[0]]
    n = int(b.positions[0]) + 1
    assert np.array_equal(ora.logits_row(qc, qs, b.w[0], c8, bt, n), ora.logits_row(qc, qs, b.w[0], c4, bt, n))


def pin_fp4_scores_vs_library(ora):
    """The FP4 cache's codes unpacked by the test (low nibble first) and
    decoded by table; the score is then a float64 matmul of dequantised
    values (ReLU per head, weighted sum over heads)."""
    n_keys = 130
    Q = synth.normal(95, 1, 64 * 128).reshape(64, 128)
    K = synth.normal(95, 2, n_keys * 128).reshape(n_keys, 128)
    K[::4] *= 7.0
    w = synth.normal(95, 3, 64).astype(np.float32)
    bt = np.array([2, 0, 1], np.int32)
    pos = np.arange(n_keys)
    slots = bt[pos // 64].astype(np.int64) * 64 + pos % 64
    cache = ora.new_cache(3, "fp4")
    assert ora.k_quant_write(bf16(K), slots, cache) == 0
    qc, qs = ora.q_quant(bf16(Q))
    got = ora.logits_row(qc, qs, w, cache, bt, n_keys)
    flat = cache.reshape(-1)
    table = np.array([(-1.0 if c & 8 else 1.0) * E2M1_MAGNITUDES[c & 7] for c in range(16)])
    kd = np.zeros((n_keys, 128))
    for i, s in enumerate(slots):
        row = flat[(s // 64) * 4352 + (s % 64) * 64:][:64]
        codes = np.stack([row & 15, row >> 4], axis=1).reshape(-1)
        ks = np.frombuffer(flat[(s // 64) * 4352 + 4096 + (s % 64) * 4:][:4].tobytes(), np.float32)[0]
        kd[i] = table[codes] * np.float64(ks)
    qd = torch_e4m3_value(qc) * qs.astype(np.float64)[:, None]
    want = SOFTMAX_SCALE * HEAD_NORM * (np.maximum(qd @ kd.T, 0.0).T @ w.astype(np.float64))
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-300)


# ----------------------------------------------------------------- top-k

def pin_topk_brute_force(ora, trials: int = 60):
    u = synth.uniform01(77, 1, trials * 16)
    for t in range(trials):
        n = 1 + t % 16
        k = 1 + (t * 7) % 9
        # coarse values so that ties happen often
        sc = np.floor(u[t * 16: t * 16 + n] * 5.0) - 2.0
        got = ora.topk_row(sc, k)
        m = min(k, n)
        assert list(got[m:]) == [-1] * (k - m)
        best = None
        for sub in itertools.combinations(range(n), m):
            inside = sc[list(sub)]
            outside = np.delete(sc, list(sub))
            if outside.size and inside.min() < outside.max():
                continue
            key = sum(sub)
            if best is None or key < best[0]:
                best = (key, set(sub))
        assert set(got[:m].tolist()) == best[1], (sc, k, got)
        # reported in score order, lower index first among equal scores
        for a, b_ in zip(got[: m - 1], got[1:m]):
            assert sc[a] > sc[b_] or (sc[a] == sc[b_] and a < b_)


def pin_topk_vs_argsort(ora):
    sc = synth.normal(78, 1, 5000)
    sc[::7] = np.round(sc[::7], 1)  # many exact ties
    for k in (1, 64, 2048, 5000, 6000):
        got = ora.topk_row(sc, k)
        want = np.argsort(-sc, kind="stable")[: min(k, 5000)]
        assert np.array_equal(got[: min(k, 5000)], want)
        assert np.all(got[min(k, 5000):] == -1)


# ----------------------------------------------------------------- conversion

def pin_convert_worked(ora):
    bt = np.array([[3, 0, -1], [1, 2, 4]], np.int32)
    logical = np.array([[0, 63, 64, 100, -1],
                        [5, 64, -1, -1, 130]], np.int32)
    req = np.array([0, 1], np.int32)
    phys, valid = ora.convert(logical, req, bt)
    assert phys.tolist() == [[192, 255, 0, 36, -1], [69, 128, -1, -1, 258]]
    assert valid.tolist() == [4, 3]
    # a physical block holding twice the rows (block_stride_rows = 128)
    phys, _ = ora.convert(logical, req, bt, block_stride_rows=128)
    assert phys.tolist() == [[384, 447, 0, 36, -1], [133, 256, -1, -1, 514]]
    # identity block table: physical == logical
    ident = np.arange(8, dtype=np.int32)[None, :]
    lg = np.array([[0, 1, 500, 63, 64, -1]], np.int32)
    phys, valid = ora.convert(lg, np.array([0], np.int32), ident)
    assert phys.tolist() == lg.tolist() and valid.tolist() == [5]


# ----------------------------------------------------------------- schedule

def pin_schedule(ora):
    # 61 layers, freq 4, default offset 2: skip iff max(l-1, 0) % 4 != 0
    fs, prod = ora.schedule(61, True, 4)
    full = [0, 1, 5, 9, 13, 17, 21, 25, 29, 33, 37, 41, 45, 49, 53, 57]
    assert [i for i, c in enumerate(fs) if c == "F"] == full
    assert fs.count("F") == 16 and fs.count("S") == 45
    for l in range(61):
        assert prod[l] == max(f for f in full if f <= l)
    fs, _ = ora.schedule(10, True, 2)
    assert fs == "FFSFSFSFSF"
    fs, _ = ora.schedule(9, True, 3)
    assert fs == "FFSSFSSFS"
    fs, _ = ora.schedule(8, True, 1)
    assert fs == "F" * 8
    fs, _ = ora.schedule(12, False, 4)
    assert fs == "F" * 12
    fs, _ = ora.schedule(9, True, 4, offset=1)  # skip iff l % 4 != 0
    assert fs == "FSSSFSSSF"
    fs, prod = ora.schedule(6, True, 4, pattern="FSSFFS")
    assert fs == "FSSFFS" and prod.tolist() == [0, 0, 0, 3, 4, 4]
    fs, prod = ora.schedule(3, False, 4, pattern="FSS")  # IndexCache off: pattern ignored
    assert fs == "FFF"
    for bad in [dict(n_layers=4, pattern="FSXF"), dict(n_layers=4, pattern="FSS"),
                dict(n_layers=4, pattern="SFFF"), dict(n_layers=4, freq=0),
                dict(n_layers=4, freq=2, offset=0)]:
        kw = dict(use_index_cache=True, freq=4)
        kw.update(bad)
        try:
            ora.schedule(**kw)
        except ValueError:
            continue
        raise AssertionError(f"schedule accepted {bad}")


def _bf16_float(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def pin_rope_hand_cases(ora):
    # unit vectors in dims 0 and 32 rotated by (cos, sin) = (0.6, 0.8): the pair
    # of dim i is dim i + 32, dim i takes x*cos - y*sin, dim i + 32 y*cos + x*sin
    x = np.zeros((4, 128), np.uint16)
    x[0, 0] = 0x3F80      # e_0
    x[1, 32] = 0x3F80     # e_32
    x[2, 5] = 0x4000      # 2 * e_5
    x[3, 64] = 0x3F80     # e_64: outside the rotated dims
    cs = np.zeros((2, 64), np.float32)
    cs[:, :32] = 1.0      # position 0: the identity
    cs[1, :32], cs[1, 32:] = 0.6, 0.8
    out, bad = ora.rope(x, np.array([1, 1, 1, 1], np.int64), cs, 1)
    assert bad == 0
    bf = lambda v: int(synth.bf16_bits(np.array([v]))[0])
    assert out[0, 0] == bf(0.6) and out[0, 32] == bf(0.8)
    assert out[1, 0] == bf(-0.8) and out[1, 32] == bf(0.6)
    assert out[2, 5] == bf(1.2) and out[2, 37] == bf(1.6)
    assert np.array_equal(out[3], x[3])
    assert np.count_nonzero(out[0]) == 2 and np.count_nonzero(out[1]) == 2
    ident, _ = ora.rope(x, np.zeros(4, np.int64), cs, 1)
    assert np.array_equal(ident, x)
    # a position outside the table: copied and counted
    same, bad = ora.rope(x[:2], np.array([2], np.int64), cs, 2)
    assert bad == 2 and np.array_equal(same, x[:2])


def pin_rope_error_bound(ora, n: int = 2000):
    # against the exact rotation in fp64: each output is the exact value up to
    # the fp32 steps (< 2^-22 relative to |x||c| + |y||s|) and one bf16 rounding
    # (half an ulp, <= 2^-8 relative); rows share a position per token of 3 rows
    rng = np.random.default_rng(3)
    x = synth.bf16_bits(rng.standard_normal((n, 128)) * 4.0)
    cs = synth.rope_cos_sin(512)
    pos = rng.integers(0, 512, size=(n + 2) // 3).astype(np.int64)
    out, bad = ora.rope(x, pos, cs, 3)
    assert bad == 0
    xf = _bf16_float(x).astype(np.float64)
    p = pos[np.arange(n) // 3]
    c = cs[p, :32].astype(np.float64)
    s = cs[p, 32:].astype(np.float64)
    x1, x2 = xf[:, :32], xf[:, 32:64]
    y1, y2 = x1 * c - x2 * s, x2 * c + x1 * s
    g = _bf16_float(out).astype(np.float64)
    for got, ref, scale in ((g[:, :32], y1, np.abs(x1 * c) + np.abs(x2 * s)),
                            (g[:, 32:64], y2, np.abs(x2 * c) + np.abs(x1 * s))):
        tol = np.abs(ref) * 2.0 ** -8 * (1 + 2.0 ** -20) + scale * 2.0 ** -22 + 1e-30
        assert np.all(np.abs(got - ref) <= tol)
    assert np.array_equal(out[:, 64:], x[:, 64:])
    # the rotation keeps each pair's length (to the rounding above)
    r_in = np.hypot(x1, x2)
    r_out = np.hypot(g[:, :32], g[:, 32:64])
    assert np.all(np.abs(r_out - r_in) <= r_in * 2.0 ** -7 + 1e-30)


def pin_gather_rows_vs_library(ora):
    # numpy's take along the row axis, zero rows for -1 and out-of-range ids
    rng = np.random.default_rng(5)
    rows = rng.integers(0, 256, size=(300, 160), dtype=np.uint8)
    phys = rng.integers(-1, 300, size=(7, 33)).astype(np.int32)
    phys[2, 3], phys[4, 0] = 300, -5  # out of range: zeros, counted
    out, bad = ora.gather_rows(rows, phys, 144)
    ok = (phys >= 0) & (phys < 300)
    ref = np.zeros((7, 33, 144), np.uint8)
    ref[ok] = np.take(rows[:, :144], phys[ok], axis=0)
    assert bad == 2 and np.array_equal(out, ref)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
