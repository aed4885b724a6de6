"""The FP4 indexer K cache on the GPU against the oracle.

"IndexCache：DeepSeek 稀疏注意力中的跨层索引复用" hands `sparse_attn_indexer` a
`use_fp4_cache` flag and nothing more of the format; both sides take the same
reading: E2M1 codes (OCP MX FP4), one ue8m0 scale per token's 128 values
(amax/6 rounded up to a power of two), dim 2i in the low nibble, pages of 64
rows of 64 code bytes followed by the 64 fp32 scales (4352 bytes).

Bit-exact: every byte of the cache (codes and scales), written standalone, with
RoPE, and fused into the indexer's prologue and the layer-stack runner. Within
the usual tolerance: the scores; top-k sets equal up to ties at the boundary.
"""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_quant_gb300 as dsa
import oracle
from dsa_sparse_attention_quant_gb300 import synth
from oracle import compare
from tests.gpu_harness import DEV, DeviceBatch, bf16_tensor
from tests.test_gpu_parity import check_batch
from tests.test_gpu_stack import run_stack

pytestmark = pytest.mark.gpu


def _k_rows_with_scale_boundaries(n: int, seed: int) -> np.ndarray:
    """bf16 K rows: N(0,1) rows spread over many binades, plus rows whose
    amax sits on or next to 6 * 2^j (the scale boundary), a zero row and a
    row of one huge and many tiny values."""
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((n, 128)) * np.exp2(rng.integers(-12, 12, n))[:, None]
    for i, j in enumerate(range(-6, 6)):
        r = 12 + 3 * i
        if r + 2 >= n:
            break
        k[r] = rng.uniform(-1, 1, 128) * 2.0 ** j
        k[r, 7] = 6.0 * 2.0 ** j                       # amax exactly 6 * 2^j: scale 2^j
        k[r + 1] = k[r]
        k[r + 1, 7] = 6.0 * 2.0 ** j * (1 + 2 ** -7)   # next bf16 above: scale 2^(j+1)
        k[r + 2] = k[r]
        k[r + 2, 7] = 1.5 * 2.0 ** (j + 2) * (1 - 2 ** -8)  # just below: scale 2^j
    k[1] = 0.0
    k[2] = 1e-6
    k[2, 0] = 3e4
    return synth.bf16_bits(k)


def test_fp4_k_write_bit_exact():
    n, num_blocks = 300, 7
    k = _k_rows_with_scale_boundaries(n, 31)
    rng = np.random.default_rng(32)
    slots = rng.permutation(num_blocks * 64)[:n].astype(np.int64)
    slots[4] = -1                      # padding token
    slots[9] = num_blocks * 64 + 3     # past the cache: skipped, flagged
    want = oracle.new_cache(num_blocks, "fp4")
    assert oracle.k_quant_write(k, slots, want) == 1
    cache = dsa.new_k_cache(num_blocks, "fp4", device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.indexer_k_quant_write(bf16_tensor(k), torch.from_numpy(slots).to(DEV), cache, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1  # DSA_DEVERR_SLOT_RANGE
    got = cache.cpu().numpy()
    assert np.array_equal(got, want), f"{int((got != want).sum())} cache bytes differ"


def test_fp4_rope_write_bit_exact():
    n, num_blocks, max_pos = 200, 4, 8192
    rng = np.random.default_rng(33)
    k = synth.bf16_bits(rng.standard_normal((n, 128)) * 2.0)
    pos = rng.integers(0, max_pos, n).astype(np.int64)
    slots = rng.permutation(num_blocks * 64)[:n].astype(np.int64)
    cs = synth.rope_cos_sin(max_pos)
    rot, bad = oracle.rope(k, pos, cs, 1)
    assert bad == 0
    want = oracle.new_cache(num_blocks, "fp4")
    oracle.k_quant_write(rot, slots, want)
    cache = dsa.new_k_cache(num_blocks, "fp4", device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.indexer_k_rope_quant_write(bf16_tensor(k), torch.from_numpy(pos).to(DEV), torch.from_numpy(cs).to(DEV),
                                   torch.from_numpy(slots).to(DEV), cache, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(cache.cpu().numpy(), want)


def test_fp4_decode_batch_scaled():
    check_batch(synth.decode32(scale=0.1), fmt="fp4")


def test_fp4_prefill_chunks_with_ragged_tails():
    hb = synth.make_batch(2, [], [(700, 700), (333, 333), (129, 129)], 128, name="prefill-small")
    check_batch(hb, fmt="fp4")


def test_fp4_mixed_batch():
    hb = synth.make_batch(7, [3000, 1, 64, 65, 777], [(900, 130), (257, 257)], 256)
    check_batch(hb, fmt="fp4")


def test_fp4_scores_match_fp8_on_shared_values():
    """Keys both caches hold exactly (E2M1 magnitudes times 2^j, amax 6 * 2^j)
    give the same scores from either cache on the GPU as well."""
    hb = synth.make_batch(94, [150, 1], [(300, 60)], 64)
    rng = np.random.default_rng(35)
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    for name in ("ctx_k", "k_new"):
        n = getattr(hb, name).shape[0]
        v = mags[rng.integers(0, 8, (n, 128))] * np.where(rng.random((n, 128)) < 0.5, -1.0, 1.0)
        v[:, 3] = 6.0
        v *= np.exp2(rng.integers(-3, 3, n))[:, None]
        setattr(hb, name, synth.bf16_bits(v))
    out = {}
    for fmt in ("fp8", "fp4"):
        db = DeviceBatch(hb, fmt=fmt)
        q8, _, wf = db.quant_fold()
        dsa.indexer_k_quant_write(db.k_new, db.slot_mapping, db.k_cache, db.dev_err)
        out[fmt] = dsa.indexer_logits(db.batch, q8, wf, db.k_cache, dev_err=db.dev_err).cpu().numpy()
        assert dsa.check_device_error(db.dev_err) == 0
    for t in range(hb.num_tokens):
        n = int(hb.positions[t]) + 1
        np.testing.assert_allclose(out["fp4"][t, :n], out["fp8"][t, :n], rtol=1e-6, atol=1e-30)


def test_fp4_stack_freq4_scaled():
    fs = run_stack(9, 4, scale=0.05, n_decode=6, fmt="fp4")
    assert fs == "FFSSSFSSS"


def test_fp4_full_size_decode_rows_sampled():
    """decode8x128k at full size with the FP4 cache: scores and top-k of
    sampled rows against the oracle (the oracle scores those rows only)."""
    hb = synth.decode8x128k()
    rows = np.array([0, 5], np.int64)
    db = DeviceBatch(hb, fmt="fp4")
    res = db.run(with_logits=True)
    assert res["dev_err"] == 0
    cache = oracle.fill_cache(hb, fmt="fp4")
    assert np.array_equal(res["cache"], cache)
    _, scores = oracle.indexer(hb, cache, rows=rows, with_scores=True)
    lens = hb.positions[rows] + 1
    for i, t in enumerate(rows):
        ok, worst, at = compare.check_scores(res["logits"][t, :lens[i]], scores[i, :lens[i]])
        assert ok, f"row {t}: score error {worst:.3g}x tolerance at key {at}"
    assert not compare.check_topk(res["topk"][rows], scores, lens, hb.topk)


def test_fp4_full_size_prefill_rows_sampled():
    """prefill4x8k at full size with the FP4 cache (K quantised into it by the
    fused prologue): every cache byte, and scores and top-k of sampled rows of
    every request against the oracle."""
    from tests.test_gpu_fullsize import sampled_rows

    hb = synth.prefill4x8k()
    check_batch(hb, rows=sampled_rows(hb, 8, 37), check_logits=True, fmt="fp4")
