"""Inconsistent step metadata on the GPU: flagged in the device error word,
never a fault.

Every index the kernels derive from device inputs is range-checked: the
access is skipped and a DSA_DEVERR_* bit is set (the slot and RoPE-position
bits are covered with the K write and the fused RoPE, the consumer's gather
bit with the gather). Here: a block-table entry past the cache for a visible
page (the score kernel skips that page), a decode request whose length is
shorter than its query (the row gets no keys: -1 ids), and ids the stand-alone
conversion cannot map (a request outside the block table, a page past its
row: -1 and flagged, the block table not read)."""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_quant_gb300 as dsa
from dsa_sparse_attention_quant_gb300 import synth
from tests.gpu_harness import DEV, DeviceBatch

pytestmark = pytest.mark.gpu

BLOCK_RANGE, ID_RANGE, SEQ_RANGE = 2, 4, 16


def test_block_table_entry_past_the_cache_is_flagged():
    hb = synth.make_batch(61, [1000, 300], [], 64)
    assert hb.block_table[0, 1] >= 0  # page 1 of request 0 holds visible keys 64..127
    hb.block_table[0, 1] = hb.num_blocks + 5
    res = DeviceBatch(hb).run()
    assert res["dev_err"] & BLOCK_RANGE, f"device error word {res['dev_err']:#x}"
    # the other request's row is unaffected in shape: k ids, all within its keys
    row = res["topk"][1]
    assert np.all((row >= 0) & (row <= hb.positions[1])) and len(set(row.tolist())) == 64


def test_decode_request_shorter_than_its_query_is_flagged():
    hb = synth.make_batch(62, [500, 700], [], 32)
    hb.seq_lens[0] = 0  # a decode request has one query token: at least one key
    res = DeviceBatch(hb).run()
    assert res["dev_err"] & SEQ_RANGE, f"device error word {res['dev_err']:#x}"
    assert np.all(res["topk"][0] == -1) and np.all(res["phys"][0] == -1) and res["valid"][0] == 0


def test_conversion_of_unmappable_ids_is_flagged():
    block_table = torch.tensor([[4, 7], [2, -1]], dtype=torch.int32, device=DEV)  # 2 requests, 2 pages each
    req = torch.tensor([0, 1, 2, -1], dtype=torch.int32, device=DEV)  # tokens 2 and 3: no such request
    logical = torch.tensor([[0, 65, 130, -1],     # page 2 is past the row (bt_stride 2)
                            [3, 64, -1, 10],      # page 1 of request 1 is a -1 entry
                            [0, 1, 2, 3],
                            [0, -1, -1, -1]], dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    phys, valid = dsa.topk_logical_to_physical(logical, req, block_table, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == ID_RANGE
    want = np.array([[4 * 64 + 0, 7 * 64 + 1, -1, -1],
                     [2 * 64 + 3, -1, -1, 2 * 64 + 10],
                     [-1, -1, -1, -1],
                     [-1, -1, -1, -1]], np.int32)
    assert np.array_equal(phys.cpu().numpy(), want)
    assert valid.cpu().tolist() == [2, 2, 0, 0]


def test_a_pipeline_wait_that_runs_out_reports_a_timeout():
    """The bounded wait every pipeline uses, on a barrier nothing completes:
    the kernel gives up after about a second, sets the timeout bit and
    returns; the context keeps working (a normal batch after it is correct)."""
    import time
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.perf_counter()
    dsa.binding.selftest_wait_timeout(err)
    torch.cuda.synchronize()
    assert int(err.item()) == 8  # DSA_DEVERR_TIMEOUT
    assert 0.5 < time.perf_counter() - t0 < 30.0
    from tests.test_gpu_parity import check_batch
    check_batch(synth.make_batch(63, [300, 90], [(200, 40)], 32))
