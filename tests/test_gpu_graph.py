"""The layer runner captured once in a CUDA graph and replayed on new inputs.

The runner allocates nothing, never synchronises and reads nothing back, and
every kernel parameter (tensor maps included) is captured by value, so a graph
of one call replays on the same buffers whatever they hold. Here the call is
captured on one step's inputs, the buffers are then overwritten with another
step's (same shapes and metadata, other q, w, K), and the replay's top-k must
match the oracle on the new inputs."""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_quant_gb300 as dsa
import oracle
from dsa_sparse_attention_quant_gb300 import synth
from oracle import compare
from tests.gpu_harness import DEV, bf16_tensor

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("split", [False, True])
def test_captured_layer_run_replays_on_new_inputs(split):
    # split: decode rows heavy enough that the runner scores them on a share of
    # the SMs beside the prefill rows, so the capture holds the side stream's
    # fork and join
    shape = ([3000] * 8, [(300, 300)]) if split else ([900, 2500, 64], [(700, 500)])
    first = synth.make_batch(41, *shape, 256, table_seed=40)
    second = synth.make_batch(42, *shape, 256, table_seed=40)  # same metadata and pages, other values
    assert np.array_equal(first.block_table, second.block_table)
    batch = dsa.Batch.from_host(first, DEV)
    q, w, kn = bf16_tensor(first.q), torch.from_numpy(first.w).to(DEV), bf16_tensor(first.k_new)
    slots = torch.from_numpy(first.slot_mapping).to(DEV)
    cache = torch.zeros((first.num_blocks, 8448), dtype=torch.uint8, device=DEV)
    ctx_slots = torch.from_numpy(first.ctx_slots).to(DEV)
    dsa.indexer_k_quant_write(bf16_tensor(first.ctx_k), ctx_slots, cache)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    stack = dsa.LayerStack(batch, "F", [dict(q=q, w=w, k_new=kn, k_cache=cache)], first.topk, slot_mapping=slots,
                           dev_err=err)
    assert (stack.decode_sms() > 0) == split
    stack.run()  # first call on the device outside the capture
    torch.cuda.synchronize()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        stack.run()
    torch.cuda.current_stream().wait_stream(side)

    # the second step's values into the same buffers, then replay
    q.copy_(bf16_tensor(second.q))
    w.copy_(torch.from_numpy(second.w).to(DEV))
    kn.copy_(bf16_tensor(second.k_new))
    cache.zero_()
    dsa.indexer_k_quant_write(bf16_tensor(second.ctx_k), ctx_slots, cache)
    stack.topk_buf.fill_(-7)
    graph.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref_cache = oracle.fill_cache(second)
    assert np.array_equal(cache.cpu().numpy(), ref_cache), "the replay's K write differs"
    rows = np.arange(second.num_tokens)
    _, scores = oracle.indexer(second, ref_cache, rows=rows, with_scores=True)
    fails = compare.check_topk(stack.topk_buf.cpu().numpy(), scores, second.positions + 1, second.topk)
    assert not fails, f"top-k mismatches in {len(fails)} rows, first {fails[0]}"


def test_graphed_layer_stack_first_call_then_replays():
    """LayerStack(graphed=True): the first run() computes the step and captures
    it; the next run() replays the capture on the buffers' new contents."""
    shape = ([700, 3000, 1], [(400, 300)])
    first = synth.make_batch(43, *shape, 128, table_seed=44)
    second = synth.make_batch(45, *shape, 128, table_seed=44)
    batch = dsa.Batch.from_host(first, DEV)
    q, w, kn = bf16_tensor(first.q), torch.from_numpy(first.w).to(DEV), bf16_tensor(first.k_new)
    slots = torch.from_numpy(first.slot_mapping).to(DEV)
    ctx_slots = torch.from_numpy(first.ctx_slots).to(DEV)
    cache = dsa.new_k_cache(first.num_blocks, device=DEV)
    dsa.indexer_k_quant_write(bf16_tensor(first.ctx_k), ctx_slots, cache)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    stack = dsa.LayerStack(batch, "F", [dict(q=q, w=w, k_new=kn, k_cache=cache)], first.topk, slot_mapping=slots,
                           dev_err=err, graphed=True)
    for hb, refill in ((first, False), (second, True)):
        if refill:
            q.copy_(bf16_tensor(hb.q))
            w.copy_(torch.from_numpy(hb.w).to(DEV))
            kn.copy_(bf16_tensor(hb.k_new))
            cache.zero_()
            dsa.indexer_k_quant_write(bf16_tensor(hb.ctx_k), ctx_slots, cache)
            stack.topk_buf.fill_(-7)
        topk, phys, valid = stack.run()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ref_cache = oracle.fill_cache(hb)
        assert np.array_equal(cache.cpu().numpy(), ref_cache)
        _, scores = oracle.indexer(hb, ref_cache, rows=np.arange(hb.num_tokens), with_scores=True)
        assert not compare.check_topk(topk.cpu().numpy(), scores, hb.positions + 1, hb.topk)
        t = topk.cpu().numpy()
        ph, _ = oracle.convert(t, hb.req_id_per_token, hb.block_table)
        assert np.array_equal(phys.cpu().numpy(), ph)
        assert np.array_equal(valid.cpu().numpy(), (t >= 0).sum(axis=1))
    assert stack._graph is not None
