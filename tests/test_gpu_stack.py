"""The IndexCache layer-stack runner against the oracle.

Every F layer (own q, w, new K and K cache) runs the whole path; every layer,
F or S, hands the consumer the buffers of its producer — the nearest F layer
at or before it — and S layers launch nothing.
"""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_quant_gb300 as dsa
import oracle
from dsa_sparse_attention_quant_gb300 import synth
from oracle import compare
from tests.gpu_harness import DEV, bf16_tensor

pytestmark = pytest.mark.gpu


def fused_projection(hb):
    """[IC] `Indexer.forward`'s fused projection output kw, bf16 [T, 128 + 64]:
    the new K rows in columns 0..127 and the head weights, rounded to bf16 (the
    projection's dtype), in columns 128..191. Returns kw and the weights as the
    fp32 values the oracle receives (bf16 converts to fp32 exactly)."""
    w_bits = synth.bf16_bits(hb.w)
    kw_bits = np.concatenate([hb.k_new, w_bits], axis=1)
    return bf16_tensor(kw_bits), synth.bf16_to_f32(w_bits)


def run_stack(n_layers, freq, scale, n_decode, pattern=None, check_rows=None, fmt="fp8", strided=False,
              block_stride_rows=0, work=None, want_split=None):
    fs, prod = dsa.schedule_build(n_layers, True, freq, 2, pattern)
    fs_o, prod_o = oracle.schedule(n_layers, True, freq, 2, pattern)
    assert fs == fs_o and prod == prod_o.tolist()
    hbs = {l: synth.stack_layer(l, scale, n_decode) for l in range(n_layers) if fs[l] == "F"}
    meta = hbs[0]
    for hb in hbs.values():
        assert np.array_equal(hb.block_table, meta.block_table)
    batch = dsa.Batch.from_host(meta, DEV)
    slots = torch.from_numpy(meta.slot_mapping).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    layers = []
    for l in range(n_layers):
        if fs[l] != "F":
            layers.append(None)
            continue
        hb = hbs[l]
        cache = dsa.new_k_cache(hb.num_blocks, fmt, device=DEV)
        dsa.indexer_k_quant_write(bf16_tensor(hb.ctx_k), torch.from_numpy(hb.ctx_slots).to(DEV), cache, err)
        if strided:  # k and w as the column views of one fused projection output
            kw, hb.w = fused_projection(hb)
            assert kw.shape[1] == 192 and kw[:, 128:].stride(0) == 192
            layers.append(dict(q=bf16_tensor(hb.q), w=kw[:, 128:], k_new=kw[:, :128], k_cache=cache, kw=kw))
        else:
            layers.append(dict(q=bf16_tensor(hb.q), w=torch.from_numpy(hb.w).to(DEV), k_new=bf16_tensor(hb.k_new),
                               k_cache=cache))
    T, k = meta.num_tokens, meta.topk
    topk_buf = torch.empty((T, k), dtype=torch.int32, device=DEV)
    phys_buf = torch.empty((T, k), dtype=torch.int32, device=DEV)
    valid_buf = torch.empty(T, dtype=torch.int32, device=DEV)
    seen = []

    def consumer(layer, producer, phys_ptr, valid_ptr):
        assert phys_ptr == phys_buf.data_ptr() and valid_ptr == valid_buf.data_ptr()
        seen.append((layer, producer, phys_buf.clone(), valid_buf.clone(), topk_buf.clone()))

    stack = dsa.LayerStack(batch, fs, layers, k, slot_mapping=slots, topk_buf=topk_buf, phys_buf=phys_buf,
                           valid_buf=valid_buf, consumer=consumer, dev_err=err, block_stride_rows=block_stride_rows,
                           work=work)
    if want_split is not None:  # decode scores on a share of the SMs beside the prefill scores, or not
        assert (stack.decode_sms() > 0) == want_split
    stack.run()
    torch.cuda.synchronize()
    assert dsa.check_device_error(err) == 0
    assert [s[0] for s in seen] == list(range(n_layers))
    assert [s[1] for s in seen] == prod
    snap = {s[0]: s for s in seen}
    for l in range(n_layers):
        p = prod[l]
        assert torch.equal(snap[l][2], snap[p][2]) and torch.equal(snap[l][3], snap[p][3])
    rows = np.arange(T) if check_rows is None else check_rows
    for l, hb in hbs.items():
        cache = oracle.fill_cache(hb, fmt=fmt)
        assert np.array_equal(layers[l]["k_cache"].cpu().numpy(), cache), f"layer {l}: cache bytes"
        _, scores = oracle.indexer(hb, cache, rows=rows, with_scores=True)
        lens = hb.positions[rows] + 1
        topk = snap[l][4].cpu().numpy()[rows]
        fails = compare.check_topk(topk, scores, lens, k)
        assert not fails, f"layer {l}: {fails[:2]}"
        phys = snap[l][2].cpu().numpy()[rows]
        valid = snap[l][3].cpu().numpy()[rows]
        assert np.array_equal(valid, (topk >= 0).sum(axis=1)), f"layer {l}: valid counts"
        for i, t in enumerate(rows):
            n = int(lens[i])
            table, _ = oracle.convert(np.arange(n, dtype=np.int32)[None, :], hb.req_id_per_token[t:t + 1],
                                      hb.block_table, 64, block_stride_rows)
            want = np.where(topk[i] >= 0, table[0][np.clip(topk[i], 0, None)], -1)
            assert np.array_equal(phys[i], want)
    return fs


def test_stack_freq4_scaled():
    # the batch's work is known from its host metadata: decode and prefill
    # scores run side by side on split SMs
    fs = run_stack(9, 4, scale=0.05, n_decode=6, want_split=True)
    assert fs == "FFSSSFSSS"


def test_stack_freq4_scaled_one_after_the_other():
    # no work given: decode scores, then prefill scores, each on the whole GPU
    run_stack(5, 4, scale=0.05, n_decode=6, work=(0, 0), want_split=False)


def test_stack_pattern_scaled():
    run_stack(6, 4, scale=0.03, n_decode=3, pattern="FSFFSS")


def test_stack_fused_projection_views():
    # k_new and w are the column views kw[:, :128] and kw[:, 128:] (bf16, row
    # stride 192) of one fused projection output, as [IC] `Indexer.forward`
    # slices them: cache bytes bit-exact, top-k and ids against the oracle
    run_stack(5, 4, scale=0.05, n_decode=6, strided=True)


def test_stack_block_stride_rows_128():
    # the runner's fused conversion with 128 physical rows per block ([IG]
    # `_convert_once`, BLOCK_STRIDE_ROWS), against the oracle's conversion
    run_stack(5, 4, scale=0.05, n_decode=6, block_stride_rows=128)


def test_stack_fused_projection_views_fp4_stride_1000():
    run_stack(5, 4, scale=0.03, n_decode=3, fmt="fp4", strided=True, block_stride_rows=1000)


def run_layer(hb, want_split, fmt="fp8"):
    """One F layer of ``hb`` through the runner, top-k, physical ids and valid
    counts against the oracle."""
    batch = dsa.Batch.from_host(hb, DEV)
    cache = dsa.new_k_cache(hb.num_blocks, fmt, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    dsa.indexer_k_quant_write(bf16_tensor(hb.ctx_k), torch.from_numpy(hb.ctx_slots).to(DEV), cache, err)
    layers = [dict(q=bf16_tensor(hb.q), w=torch.from_numpy(hb.w).to(DEV), k_new=bf16_tensor(hb.k_new),
                   k_cache=cache)]
    stack = dsa.LayerStack(batch, "F", layers, hb.topk, slot_mapping=torch.from_numpy(hb.slot_mapping).to(DEV),
                           dev_err=err)
    assert (stack.decode_sms() > 0) == want_split
    topk, phys, valid = stack.run()
    torch.cuda.synchronize()
    assert dsa.check_device_error(err) == 0
    ref_cache = oracle.fill_cache(hb, fmt=fmt)
    assert np.array_equal(cache.cpu().numpy(), ref_cache)
    rows = np.arange(hb.num_tokens)
    _, scores = oracle.indexer(hb, ref_cache, rows=rows, with_scores=True)
    lens = hb.positions + 1
    topk = topk.cpu().numpy()
    assert not compare.check_topk(topk, scores, lens, hb.topk)
    phys, valid = phys.cpu().numpy(), valid.cpu().numpy()
    assert np.array_equal(valid, (topk >= 0).sum(axis=1))
    for t in rows:
        table, _ = oracle.convert(np.arange(int(lens[t]), dtype=np.int32)[None, :], hb.req_id_per_token[t:t + 1],
                                  hb.block_table, 64, 0)
        assert np.array_equal(phys[t], np.where(topk[t] >= 0, table[0][np.clip(topk[t], 0, None)], -1))


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
def test_split_layer_with_decode_rows_past_one_cta(fmt):
    # decode rows longer than one CTA stages (chunk CTAs and a resolving CTA
    # per row) on the decode share of the SMs, beside a prefill on the rest
    hb = synth.make_batch(31, [40000, 36000, 35000, 2500], [(600, 600)], 2048)
    run_layer(hb, want_split=True, fmt=fmt)


@pytest.mark.parametrize("work", [None, (0, 0)])
def test_stack_without_consumer(work):
    # no consumer: every F layer after the first starts its prologue as a
    # programmatic dependent of the previous layer's top-k; every cache and the
    # last F layer's ids (left in the buffers) against the oracle
    n_layers, freq = 9, 4
    fs, _ = dsa.schedule_build(n_layers, True, freq, 2)
    hbs = {l: synth.stack_layer(l, 0.05, 6) for l in range(n_layers) if fs[l] == "F"}
    meta = hbs[0]
    batch = dsa.Batch.from_host(meta, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    layers = []
    for l in range(n_layers):
        if fs[l] != "F":
            layers.append(None)
            continue
        hb = hbs[l]
        cache = dsa.new_k_cache(hb.num_blocks, device=DEV)
        dsa.indexer_k_quant_write(bf16_tensor(hb.ctx_k), torch.from_numpy(hb.ctx_slots).to(DEV), cache, err)
        layers.append(dict(q=bf16_tensor(hb.q), w=torch.from_numpy(hb.w).to(DEV), k_new=bf16_tensor(hb.k_new),
                           k_cache=cache))
    stack = dsa.LayerStack(batch, fs, layers, meta.topk, slot_mapping=torch.from_numpy(meta.slot_mapping).to(DEV),
                           dev_err=err, work=work)
    topk, phys, valid = stack.run()
    torch.cuda.synchronize()
    assert dsa.check_device_error(err) == 0
    for l, hb in hbs.items():
        assert np.array_equal(layers[l]["k_cache"].cpu().numpy(), oracle.fill_cache(hb)), f"layer {l}: cache bytes"
    last = max(hbs)
    hb = hbs[last]
    rows = np.arange(hb.num_tokens)
    _, scores = oracle.indexer(hb, oracle.fill_cache(hb), rows=rows, with_scores=True)
    lens = hb.positions + 1
    topk = topk.cpu().numpy()
    assert not compare.check_topk(topk, scores, lens, hb.topk)
    assert np.array_equal(valid.cpu().numpy(), (topk >= 0).sum(axis=1))
