"""Parity of the CUDA path with the CPU oracle on seeded inputs.

Bit-exact: FP8 codes and ue8m0 scales of q and of the K cache (every byte of
the cache), the folded head weights, and the logical->physical conversion.
Within tolerance (2e-3 of max(|I|, mean |I| of the row)): the scores. Set
equality up to oracle ties within that tolerance at the k-th boundary: top-k.
"""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_quant_gb300 as dsa
import oracle
from dsa_sparse_attention_quant_gb300 import synth
from oracle import compare
from tests.gpu_harness import DEV, DeviceBatch

pytestmark = pytest.mark.gpu


def fold_reference(w, q_scale):
    """The pages' weight fold in fp32, operation by operation."""
    w = w.astype(np.float32)
    return ((w * q_scale.astype(np.float32)) * np.float32(128 ** -0.5)) * np.float32(0.125)


def conversion_table(hb, row):
    """Oracle physical id of every logical id of one query row."""
    n = int(hb.positions[row]) + 1
    ids = np.arange(n, dtype=np.int32)[None, :]
    phys, _ = oracle.convert(ids, np.array([hb.req_id_per_token[row]], np.int32), hb.block_table)
    return phys[0]


def check_batch(hb, rows=None, check_logits=True, fmt="fp8"):
    """The whole path on ``hb`` with an FP8 or FP4 K cache against the oracle."""
    db = DeviceBatch(hb, fmt=fmt)
    res = db.run(with_logits=check_logits)
    assert res["dev_err"] == 0, f"device error word {res['dev_err']:#x}"
    cache = oracle.fill_cache(hb, fmt=fmt)
    # S1: every byte of the cache
    assert np.array_equal(res["cache"].reshape(-1), cache.reshape(-1)), "K cache bytes differ"
    # S2a: q codes, scales, folded weights
    qc, qs = oracle.q_quant(hb.q)
    assert np.array_equal(res["q8"], qc), "q FP8 codes differ"
    assert np.array_equal(res["q_scale"], qs), "q scales differ"
    assert np.array_equal(res["w_folded"], fold_reference(hb.w, qs)), "folded weights differ"
    if rows is None:
        rows = np.arange(hb.num_tokens)
    rows = np.asarray(rows, np.int64)
    if rows.size == 0:
        return res
    ora_topk, scores = oracle.indexer(hb, cache, rows=rows, with_scores=True)
    lens = hb.positions[rows] + 1
    if check_logits:
        for i, t in enumerate(rows):
            n = int(lens[i])
            ok, worst, at = compare.check_scores(res["logits"][t, :n], scores[i, :n])
            assert ok, f"row {t}: score error {worst:.3g}x tolerance at key {at}"
    fails = compare.check_topk(res["topk"][rows], scores, lens, hb.topk)
    assert not fails, f"top-k mismatches in {len(fails)} rows, first {fails[0]}"
    # S5 on the GPU's own ids, looked up in the oracle's table of the row
    for t in rows:
        ids = res["topk"][t]
        table = conversion_table(hb, t)
        want = np.where(ids >= 0, table[np.clip(ids, 0, None)], -1)
        assert np.array_equal(res["phys"][t], want), f"row {t}: physical ids differ"
        assert res["valid"][t] == int((ids >= 0).sum())
    return res


def test_prefill512_full():
    check_batch(synth.prefill512())


def test_decode_batch_scaled():
    check_batch(synth.decode32(scale=0.1))


def test_prefill_chunks_scaled():
    hb = synth.make_batch(2, [], [(700, 700), (333, 333), (129, 129)], 128, name="prefill-small")
    check_batch(hb)


def test_long_decode_scaled():
    check_batch(synth.decode8x128k(scale=0.15, n_reqs=2))


def test_mixed_batch_chunked_prefill():
    # decodes of ragged lengths, a chunked prefill with 300 cached tokens, a fresh prefill
    hb = synth.make_batch(7, [3000, 64, 1, 130, 127, 128, 129], [(500, 200), (129, 129), (70, 3)], 64,
                          spare_blocks=5, bt_pad=2)
    check_batch(hb)


def test_rows_shorter_than_topk():
    hb = synth.make_batch(8, [5, 17, 2048], [(40, 40)], 2048)
    res = check_batch(hb)
    assert (res["topk"][0] == -1).sum() == 2048 - 5


def test_decode_requests_with_two_query_tokens():
    # speculative-decode style: two query tokens per request in the decode segment
    hb = synth.make_batch(9, [], [(900, 2), (300, 2), (77, 2)], 64)
    hb.num_decodes = 3
    check_batch(hb)


def test_identical_keys_every_score_ties():
    # every key of a request identical: one score per row, so the boundary bin
    # holds the whole row (per-row kernel past its candidate buffer; the
    # multi-CTA select past its staged candidates)
    hb = synth.make_batch(13, [9000, 20000], [], 256)
    first = {}
    for i, s in enumerate(hb.ctx_slots):
        r = 0 if i < 8999 else 1
        first.setdefault(r, hb.ctx_k[i].copy())
        hb.ctx_k[i] = first[r]
    for t in range(hb.num_tokens):
        hb.k_new[t] = first[t]
    check_batch(hb)


def test_identical_keys_prefill_rows_tie():
    # a prefill whose keys are all identical: every row's boundary bin holds
    # the whole row, past the per-row kernel's staged candidate buffer
    hb = synth.make_batch(14, [300], [(3000, 3000)], 256)
    kv = hb.k_new[hb.num_decodes].copy()
    hb.ctx_k[:] = kv
    hb.k_new[:] = kv
    check_batch(hb)


def test_empty_batch():
    hb = synth.make_batch(10, [], [], 64)
    db = DeviceBatch(hb)
    q8, _, wf = db.quant_fold()
    out = dsa.indexer_logits_topk(db.batch, q8, wf, db.k_cache, 64)
    assert out.shape == (0, 64)


def test_convert_standalone_bit_exact():
    hb = synth.make_batch(11, [700, 70, 1], [(300, 300)], 64)
    T, k = hb.num_tokens, 256
    lens = hb.positions + 1
    u = synth.uniform01(11, 99, T * k).reshape(T, k)
    logical = np.floor(u * (lens[:, None] + 1)).astype(np.int32) - 1  # ids in [-1, n)
    db = DeviceBatch(hb, fill_context=False)
    lg = torch.from_numpy(logical).to(DEV)
    for stride_rows in (0, 64, 128, 1000):
        phys, valid = dsa.topk_logical_to_physical(lg, db.batch.req_id_per_token, db.batch.block_table,
                                                   block_stride_rows=stride_rows)
        want_p, want_v = oracle.convert(logical, hb.req_id_per_token, hb.block_table, 64, stride_rows)
        assert np.array_equal(phys.cpu().numpy(), want_p)
        assert np.array_equal(valid.cpu().numpy(), want_v)


def test_quantiser_every_bf16_value():
    """Every finite bf16 bit pattern, in rows whose amax spans the whole range."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    vals = (bits << np.uint32(16)).view(np.float32)
    finite = bits[np.isfinite(vals)].astype(np.uint16)
    n_rows = (finite.size + 127) // 128
    k = np.zeros(n_rows * 128, np.uint16)
    k[: finite.size] = finite
    k = k.reshape(n_rows, 128)
    extra = synth.bf16_bits(np.array([[0.0] * 128, [-0.0] * 128, [1e-30] * 128, [448.0] + [1.0] * 127]))
    k = np.concatenate([k, extra])
    slots = np.arange(k.shape[0], dtype=np.int64)
    num_blocks = (k.shape[0] + 63) // 64
    want = oracle.new_cache(num_blocks)
    assert oracle.k_quant_write(k, slots, want) == 0
    cache = torch.zeros((num_blocks, 8448), dtype=torch.uint8, device=DEV)
    from tests.gpu_harness import bf16_tensor
    dsa.indexer_k_quant_write(bf16_tensor(k), torch.from_numpy(slots).to(DEV), cache)
    assert np.array_equal(cache.cpu().numpy(), want)


def test_slot_errors_are_flagged_not_written():
    k = synth.bf16_bits(synth.normal(12, 1, 4 * 128).reshape(4, 128))
    slots = np.array([3, -1, 64 * 2, 5], np.int64)  # -1: padding; 128: past a 2-block cache
    cache = torch.zeros((2, 8448), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    from tests.gpu_harness import bf16_tensor
    dsa.indexer_k_quant_write(bf16_tensor(k), torch.from_numpy(slots).to(DEV), cache, err)
    want = oracle.new_cache(2)
    assert oracle.k_quant_write(k, slots, want) == 1
    assert np.array_equal(cache.cpu().numpy(), want)
    assert dsa.check_device_error(err) == 1


def test_k_quant_write_strided_view_bit_exact():
    # k as the column view kw[:, :128] (row stride 192) of a fused projection
    # output, as [IC] `Indexer.forward` slices it: every cache byte bit-exact
    hb = synth.make_batch(15, [300, 70], [(200, 130)], 64)
    kw_bits = np.concatenate([hb.k_new, synth.bf16_bits(hb.w)], axis=1)
    from tests.gpu_harness import bf16_tensor
    kw = bf16_tensor(kw_bits)
    for fmt in ("fp8", "fp4"):
        cache = dsa.new_k_cache(hb.num_blocks, fmt, device=DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        dsa.indexer_k_quant_write(kw[:, :128], torch.from_numpy(hb.slot_mapping).to(DEV), cache, err)
        want = oracle.new_cache(hb.num_blocks, fmt)
        assert oracle.k_quant_write(hb.k_new, hb.slot_mapping, want) == 0
        assert dsa.check_device_error(err) == 0
        assert np.array_equal(cache.cpu().numpy(), want), fmt


def test_decode_row_longer_than_one_cta_stages():
    # a decode row past 32768 scores takes the select of independent chunk
    # CTAs; the other rows of the batch share its launch
    hb = synth.make_batch(16, [140000, 3000, 2049], [], 2048)
    check_batch(hb)


def test_decode_rows_ragged_lengths_one_cta_per_row():
    # decode rows staged whole by one CTA each, ragged lengths and tails,
    # k from 512 to 2048, rows up to the 32768-score staging limit
    for seed, lens, k in ((17, [1000, 700, 600], 512), (18, [1500, 900], 1024), (19, [5000, 4097, 2100], 1024),
                          (20, [8000, 1100], 1024), (21, [32768, 20000, 7000, 64], 2048)):
        check_batch(synth.make_batch(seed, lens, [], k))


def test_long_decode_rows_every_score_ties():
    # decode rows past 32768 scores whose keys are all identical: the boundary
    # bin holds the whole row, past the resolving CTA's staged candidates
    hb = synth.make_batch(23, [40000, 33000], [], 2048)
    first = {}
    for i in range(hb.ctx_k.shape[0]):
        r = 0 if i < 39999 else 1
        first.setdefault(r, hb.ctx_k[i].copy())
        hb.ctx_k[i] = first[r]
    for t in range(hb.num_tokens):
        hb.k_new[t] = first[t]
    check_batch(hb)


def test_topk_output_rows_not_16_byte_aligned():
    # the per-row top-k writes ids four at a time with 16-byte stores only when
    # the output rows allow it; an output starting 4 bytes into a buffer takes
    # the scalar stores, with the same result
    hb = synth.make_batch(24, [3000, 40], [(600, 600)], 256)
    db = DeviceBatch(hb)
    res = db.run()  # writes this step's K into the cache
    assert res["dev_err"] == 0
    q8, _, wf = db.quant_fold()
    scores = dsa.indexer_logits(db.batch, q8, wf, db.k_cache)
    T, k = hb.num_tokens, hb.topk
    big = torch.full((T * k + 1,), -7, dtype=torch.int32, device=DEV)
    shifted = big[1:].view(T, k)
    assert shifted.data_ptr() % 16 == 4
    dsa.indexer_topk(db.batch, scores, k, topk_out=shifted)
    torch.cuda.synchronize()
    assert int(big[0].item()) == -7  # nothing written before the view
    got = shifted.cpu().numpy()
    rows = np.arange(T)
    _, ora_scores = oracle.indexer(hb, oracle.fill_cache(hb), rows=rows, with_scores=True)
    lens = hb.positions + 1
    fails = compare.check_topk(got, ora_scores, lens, k)
    assert not fails, f"top-k mismatches in {len(fails)} rows, first {fails[0]}"
    short = lens <= k
    assert np.array_equal(got[short], res["topk"][short])  # every key in order, then -1
