"""The allocation-free indexer entry point, dsa_indexer_logits_topk_static.

It serves callers that cannot allocate device memory (plugins handed only an
op's tensors, code that may not call the allocator): its scratch is a static
device array inside the library. Here it is called through the C ABI twice in
a row, on two different batches, and each result is checked against the
allocating entry point dsa_indexer_logits_topk on the same inputs and against
the oracle's fp64 scores, with the top-k tolerance used by the other tests
(ties within 2e-3 of the k-th score may resolve either way). The file is named
to be collected last.
"""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_quant_gb300 as dsa
import oracle
from dsa_sparse_attention_quant_gb300 import binding, synth
from oracle import compare
from tests.gpu_harness import DeviceBatch

pytestmark = pytest.mark.gpu


def _same_topk(a, b, scores, lens, k):
    for t in range(a.shape[0]):
        if np.array_equal(np.sort(a[t]), np.sort(b[t])):
            continue
        n = int(lens[t])
        for ids in (a[t], b[t]):
            ok, msg = compare.check_topk_row(ids, scores[t, :n].astype(np.float64), k)
            assert ok, f"row {t}: {msg}"


def _check(hb):
    db = DeviceBatch(hb)
    q8, _, wf = db.quant_fold()
    want = dsa.indexer_logits_topk(db.batch, q8, wf, db.k_cache, hb.topk, k_new=db.k_new,
                                   slot_mapping=db.slot_mapping, dev_err=db.dev_err)
    got = torch.full_like(want, -7)
    dsa.binding.indexer_logits_topk_static(db.batch, q8, wf, db.k_cache, hb.topk, got, k_new=db.k_new,
                                           slot_mapping=db.slot_mapping, dev_err=db.dev_err)
    scores = dsa.indexer_logits(db.batch, q8, wf, db.k_cache)
    torch.cuda.synchronize()
    assert dsa.check_device_error(db.dev_err) == 0
    got, want = got.cpu().numpy(), want.cpu().numpy()
    lens = hb.positions + 1
    _same_topk(got, want, scores.cpu().numpy(), lens, hb.topk)
    # against the oracle: the static call's cache bytes and its top-k sets
    cache = oracle.fill_cache(hb)
    assert np.array_equal(db.k_cache.cpu().numpy(), cache)
    _, ora_scores = oracle.indexer(hb, cache, rows=np.arange(hb.num_tokens), with_scores=True)
    fails = compare.check_topk(got, ora_scores, lens, hb.topk)
    assert not fails, f"static call vs oracle: {fails[:2]}"


def test_static_entry_point_two_calls_in_a_row():
    _check(synth.decode32(scale=0.25))                              # first call on this device sets up
    _check(synth.make_batch(21, [900, 70], [(400, 260)], 64))       # second call reuses the array


def test_static_entry_point_rejects_oversized_batch():
    hb = synth.make_batch(22, [100], [], 16)
    db = DeviceBatch(hb, fill_context=False)
    b = db.batch
    big = dsa.Batch(b.query_start_loc, b.seq_lens, b.block_table, b.req_id_per_token, b.num_decodes,
                    b.num_blocks, max_seq_len=1 << 24)  # the score row alone needs 64 MiB
    assert dsa.indexer_workspace_size(big, 16) > binding.STATIC_WORKSPACE_BYTES
    q8, _, wf = db.quant_fold()
    out = torch.empty((1, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(dsa.DsaError, match="workspace too small"):
        binding.indexer_logits_topk_static(big, q8, wf, db.k_cache, 16, out)
