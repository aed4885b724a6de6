"""RoPE of q and K fused into the quantiser, GPU against oracle.

"IndexCache：DeepSeek 稀疏注意力中的跨层索引复用", `Indexer.forward`: the leading
64 dims of every q head and of the shared K row are rotated by
`rotary_emb(positions, q_pe, k_pe)` before the FP8 quantisation. The GPU path
takes un-rotated bf16 rows, positions and a cos/sin table and rotates them on
the way into the quantiser; the oracle rotates the same inputs (`ora_rope`),
then quantises. Codes, scales, folded weights and cache bytes must agree bit
for bit; the scores and top-k of a layer run with the rotation, within the
usual tolerance.
"""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_quant_gb300 as dsa
import oracle
from dsa_sparse_attention_quant_gb300 import synth
from oracle import compare
from tests.gpu_harness import DEV, bf16_tensor
from tests.test_gpu_parity import fold_reference

pytestmark = pytest.mark.gpu


def test_q_rope_quant_fold_bit_exact_with_an_out_of_range_position():
    T, max_pos = 37, 4096
    rng = np.random.default_rng(21)
    q = synth.bf16_bits(rng.standard_normal((T, 64, 128)) * 3.0)
    w = rng.standard_normal((T, 64)).astype(np.float32)
    pos = rng.integers(0, max_pos, T).astype(np.int64)
    pos[5] = max_pos  # outside the table: left unrotated, flagged
    cs = synth.rope_cos_sin(max_pos)
    rot, bad = oracle.rope(q, pos, cs, 64)
    assert bad == 64
    codes, scales = oracle.q_quant(rot)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    q8, qs, wf = dsa.indexer_q_rope_quant_fold(
        bf16_tensor(q), torch.from_numpy(w).to(DEV), torch.from_numpy(pos).to(DEV), torch.from_numpy(cs).to(DEV),
        q_scale=torch.empty((T, 64), dtype=torch.float32, device=DEV), dev_err=err)
    assert np.array_equal(q8.cpu().numpy(), codes)
    assert np.array_equal(qs.cpu().numpy().view(np.uint32), scales.view(np.uint32))
    assert np.array_equal(wf.cpu().numpy().view(np.uint32), fold_reference(w, scales).view(np.uint32))
    assert int(err.item()) == 32  # DSA_DEVERR_POS_RANGE


def test_k_rope_quant_write_bit_exact():
    n, max_pos = 1000, 70000
    rng = np.random.default_rng(22)
    k = synth.bf16_bits(rng.standard_normal((n, 128)) * 2.0)
    pos = rng.integers(0, max_pos, n).astype(np.int64)
    slots = rng.permutation(16 * 64)[:n].astype(np.int64)
    cs = synth.rope_cos_sin(max_pos)
    rot, bad = oracle.rope(k, pos, cs, 1)
    assert bad == 0
    ref = oracle.new_cache(16)
    oracle.k_quant_write(rot, slots, ref)
    cache = torch.zeros((16, 8448), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.indexer_k_rope_quant_write(bf16_tensor(k), torch.from_numpy(pos).to(DEV), torch.from_numpy(cs).to(DEV),
                                   torch.from_numpy(slots).to(DEV), cache, dev_err=err)
    assert int(err.item()) == 0
    assert np.array_equal(cache.cpu().numpy(), ref)


@pytest.mark.parametrize("shape", ["mixed", "prefill"])
def test_layer_run_with_rope_matches_the_oracle(shape):
    if shape == "mixed":
        hb = synth.make_batch(23, [700, 3000, 45], [(900, 600), (300, 300)], 256)
    else:
        hb = synth.make_batch(24, [], [(512, 512)], 128, identity_table=True)
    max_pos = int(hb.seq_lens.max()) + 1
    cs = synth.rope_cos_sin(max_pos)
    ctx_pos = np.concatenate([np.arange(0, s - q, dtype=np.int64)
                              for s, q in zip(hb.seq_lens.tolist(), np.diff(hb.query_start_loc).tolist())])
    # the oracle's inputs: the same rows, rotated by the oracle
    q_rot, b0 = oracle.rope(hb.q, hb.positions, cs, 64)
    k_rot, b1 = oracle.rope(hb.k_new, hb.positions, cs, 1)
    c_rot, b2 = oracle.rope(hb.ctx_k, ctx_pos, cs, 1)
    assert b0 == b1 == b2 == 0
    import dataclasses
    hr = dataclasses.replace(hb, q=q_rot, k_new=k_rot, ctx_k=c_rot)
    ref_cache = oracle.fill_cache(hr)

    # the GPU: un-rotated rows in; context K written by the rotating S1, then one F layer with RoPE
    batch = dsa.Batch.from_host(hb, DEV)
    cache = torch.zeros((hb.num_blocks, 8448), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    cs_t = torch.from_numpy(cs).to(DEV)
    dsa.indexer_k_rope_quant_write(bf16_tensor(hb.ctx_k), torch.from_numpy(ctx_pos).to(DEV), cs_t,
                                   torch.from_numpy(hb.ctx_slots).to(DEV), cache, dev_err=err)
    layers = [dict(q=bf16_tensor(hb.q), w=torch.from_numpy(hb.w).to(DEV), k_new=bf16_tensor(hb.k_new),
                   k_cache=cache)]
    topk, phys, valid = dsa.layer_stack_run(batch, "F", layers, hb.topk,
                                            slot_mapping=torch.from_numpy(hb.slot_mapping).to(DEV), dev_err=err,
                                            positions=torch.from_numpy(hb.positions).to(DEV), rope_cos_sin=cs_t)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(cache.cpu().numpy(), ref_cache), "K cache bytes differ"
    rows = np.arange(hb.num_tokens)
    ora_topk, scores = oracle.indexer(hr, ref_cache, rows=rows, with_scores=True)
    lens = hb.positions + 1
    fails = compare.check_topk(topk.cpu().numpy(), scores, lens, hb.topk)
    assert not fails, f"top-k mismatches in {len(fails)} rows, first {fails[0]}"
