"""The C-ABI library on a machine without a GPU: it loads, exports every symbol
that include/dsaidx.h declares, runs its host-only schedule builder exactly
like the oracle, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_quant_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "dsaidx.h")).read()
    return sorted(set(re.findall(r"DSA_API\s+[\w\s\*]*?\b(dsa_\w+)\s*\(", text)))


def test_header_declares_binding_symbols():
    assert declared_symbols() == sorted(binding.SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = binding.load()
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert lib.dsa_version() == 301
    assert lib.dsa_status_string(0) == b"ok"
    assert b"invalid" in lib.dsa_status_string(1)


@pytest.mark.parametrize("n_layers", [0, 1, 2, 5, 13, 61, 96])
@pytest.mark.parametrize("freq", [1, 2, 3, 4, 7])
@pytest.mark.parametrize("offset", [1, 2, 3])
def test_schedule_matches_oracle(n_layers, freq, offset):
    for use in (False, True):
        want = oracle.schedule(n_layers, use, freq, offset)
        got = binding.schedule_build(n_layers, use, freq, offset)
        assert got[0] == want[0]
        assert got[1] == want[1].tolist()


def test_schedule_patterns_and_rejections():
    for pat in ["F", "FS", "FFSSF", "F" + "S" * 60, "FSFSFSFS"]:
        want = oracle.schedule(len(pat), True, 4, 2, pat)
        got = binding.schedule_build(len(pat), True, 4, 2, pat)
        assert got[0] == want[0] and got[1] == want[1].tolist()
    for kw in [dict(n_layers=3, pattern="FSX"), dict(n_layers=3, pattern="FS"), dict(n_layers=2, pattern="SF"),
               dict(n_layers=4, freq=0), dict(n_layers=4, freq=3, offset=0), dict(n_layers=-1)]:
        args = dict(use_index_cache=True, freq=4, offset=2, pattern=None)
        args.update(kw)
        with pytest.raises(binding.DsaError):
            binding.schedule_build(**args)
        with pytest.raises(ValueError):
            oracle.schedule(**args)


def test_host_validation_without_gpu():
    lib = binding.load()
    P = ctypes.c_void_p
    # negative token count, bad row stride, bad top-k: rejected on the host
    assert lib.dsa_indexer_k_quant_write(P(16), -1, 128, P(16), P(16), 1, None, None) == binding.DSA_EINVAL
    assert lib.dsa_indexer_k_quant_write(P(16), 4, 100, P(16), P(16), 1, None, None) == binding.DSA_EINVAL
    assert lib.dsa_topk_logical_to_physical(P(16), 4, 6, P(16), P(16), 1, 1, 0, P(16), None, None,
                                            None) == binding.DSA_EINVAL
    assert lib.dsa_topk_logical_to_physical(P(16), 4, 8192, P(16), P(16), 1, 1, 0, P(16), None, None,
                                            None) == binding.DSA_EINVAL
    assert lib.dsa_topk_logical_to_physical(P(16), 4, 64, P(16), P(16), -1, 1, 0, P(16), None, None,
                                            None) == binding.DSA_EINVAL  # negative request count
    b = binding.DsaBatchC(1, 2, 1, 1, 10, 1, 1, 16, 16, 16, 16)  # num_decodes > num_reqs
    assert lib.dsa_indexer_workspace_size(ctypes.byref(b), 64) == 0
    # empty batches are no-ops that succeed without a device
    assert lib.dsa_indexer_k_quant_write(None, 0, 128, None, P(16), 1, None, None) == binding.DSA_OK
    empty = binding.DsaBatchC(0, 0, 0, 0, 0, 1, 1, None, None, None, None)
    assert lib.dsa_indexer_logits_topk(ctypes.byref(empty), None, None, None, 64, None, None, 0, None, None,
                                       None, None) == binding.DSA_OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_valid_call_without_gpu_reports_no_device():
    lib = binding.load()
    P = ctypes.c_void_p
    st = lib.dsa_indexer_k_quant_write(P(256), 4, 128, P(256), P(256), 1, None, None)
    assert st == binding.DSA_ENODEV


def test_ue8m0_exponent_rule_equals_division_for_every_bf16_amax():
    # The GPU quantiser takes the ue8m0 scale from amax's exponent bits (e = E - 8,
    # plus one when the significand exceeds 1.75) instead of dividing by 448; for
    # every finite bf16 amax (and the 1e-10 floor) that equals the oracle's rule,
    # RN(amax / 448) rounded up to a power of two.
    b = np.arange(0x0000, 0x7F80, dtype=np.uint32)
    a = np.maximum((b << 16).view(np.float32), np.float32(1e-10))
    ref = np.array([oracle.ue8m0_scale(float(x)) for x in a[::97]], np.float32)
    u = a.view(np.uint32)
    rule = (((u >> 23) - 8 + ((u & 0x7FFFFF) > 0x600000)) << 23).astype(np.uint32).view(np.float32)
    assert np.array_equal(rule[::97].view(np.uint32), ref.view(np.uint32))
    r = (a / np.float32(448.0)).astype(np.float32).view(np.uint32)
    up = np.where((r & 0x7FFFFF) != 0, (r & 0x7F800000) + 0x800000, r).astype(np.uint32)
    assert np.array_equal(rule.view(np.uint32), up)


def test_rope_entry_points_reject_bad_arguments_on_the_host():
    lib = binding.load()
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: every call below fails its host checks first
    k_write = lib.dsa_indexer_k_rope_quant_write
    # no cos/sin table, no positions, empty table, misaligned table
    assert k_write(fake, 4, 128, fake, None, 16, fake, fake, 8, None, None) == binding.DSA_EINVAL
    assert k_write(fake, 4, 128, None, fake, 16, fake, fake, 8, None, None) == binding.DSA_EINVAL
    assert k_write(fake, 4, 128, fake, fake, 0, fake, fake, 8, None, None) == binding.DSA_EINVAL
    assert k_write(fake, 4, 128, fake, P(4100), 16, fake, fake, 8, None, None) == binding.DSA_EINVAL
    assert k_write(fake, 0, 128, fake, fake, 16, fake, fake, 8, None, None) == binding.DSA_OK
    q_fold = lib.dsa_indexer_q_rope_quant_fold
    assert q_fold(fake, fake, 4, fake, None, 16, 0.0, fake, None, fake, None, None) == binding.DSA_EINVAL
    assert q_fold(fake, fake, 4, fake, fake, 0, 0.0, fake, None, fake, None, None) == binding.DSA_EINVAL
    assert q_fold(fake, fake, 0, fake, fake, 16, 0.0, fake, None, fake, None, None) == binding.DSA_OK


def test_fp4_cache_arguments_rejected_on_the_host():
    lib = binding.load()
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: every call below fails its host checks first
    w4 = lib.dsa_indexer_k_quant_write_fp4
    # the FP4 cache must be 32-byte aligned (the packed 4-bit tensor-map type)
    assert w4(fake, 4, 128, None, None, 0, fake, P(4112), 8, None, None) == binding.DSA_EINVAL
    # a cos/sin table needs positions and a positive max_pos
    assert w4(fake, 4, 128, None, fake, 16, fake, fake, 8, None, None) == binding.DSA_EINVAL
    assert w4(fake, 4, 128, fake, fake, 0, fake, fake, 8, None, None) == binding.DSA_EINVAL
    assert w4(fake, 4, 100, None, None, 0, fake, fake, 8, None, None) == binding.DSA_EINVAL
    assert w4(fake, 0, 128, None, None, 0, fake, fake, 8, None, None) == binding.DSA_OK
    # an unknown cache format, and an FP4 cache that is only 16-byte aligned
    bad = binding.DsaBatchC(1, 1, 1, 1, 10, 1, 1, fake, fake, fake, fake, 2)
    assert lib.dsa_indexer_logits_topk(ctypes.byref(bad), fake, fake, fake, 64, fake, fake, 1 << 30, None, None,
                                       None, None) == binding.DSA_EINVAL
    fp4 = binding.DsaBatchC(1, 1, 1, 1, 10, 1, 1, fake, fake, fake, fake, 1)
    assert lib.dsa_indexer_logits_topk(ctypes.byref(fp4), fake, fake, P(4112), 64, fake, fake, 1 << 30, None, None,
                                       None, None) == binding.DSA_EINVAL


def test_cache_format_from_page_size():
    assert binding.cache_format(torch.zeros((3, 8448), dtype=torch.uint8)) == 0
    assert binding.cache_format(torch.zeros((3, 4352), dtype=torch.uint8)) == 1
    assert binding.cache_format(torch.zeros((3, 64, 68), dtype=torch.uint8)) == 1
    with pytest.raises(binding.DsaError):
        binding.cache_format(torch.zeros((3, 4096), dtype=torch.uint8))


def test_fp4_scale_exponent_rule_equals_division_for_every_bf16_amax():
    # The GPU's FP4 scale comes from amax's exponent bits (e = E - 2, plus one
    # when the significand exceeds 1.5) instead of dividing by 6; for every
    # finite bf16 amax (and the 1e-10 floor) that equals the oracle's rule,
    # RN(amax / 6) rounded up to a power of two.
    b = np.arange(0x0000, 0x7F80, dtype=np.uint32)
    a = np.maximum((b << 16).view(np.float32), np.float32(1e-10))
    ref = np.array([oracle.ue8m0_scale_e2m1(float(x)) for x in a[::97]], np.float32)
    u = a.view(np.uint32)
    rule = (((u >> 23) - 2 + ((u & 0x7FFFFF) > 0x400000)) << 23).astype(np.uint32).view(np.float32)
    assert np.array_equal(rule[::97].view(np.uint32), ref.view(np.uint32))
    r = (a / np.float32(6.0)).astype(np.float32).view(np.uint32)
    up = np.where((r & 0x7FFFFF) != 0, (r & 0x7F800000) + 0x800000, r).astype(np.uint32)
    assert np.array_equal(rule.view(np.uint32), up)


def test_cache_format_of_an_empty_cache():
    assert binding.cache_format(torch.zeros((0, 8448), dtype=torch.uint8)) == 0
    assert binding.cache_format(torch.zeros((0, 4352), dtype=torch.uint8)) == 1
    with pytest.raises(binding.DsaError):
        binding.cache_format(torch.zeros(8448, dtype=torch.uint8))


def test_graphed_layer_stack_refuses_a_consumer():
    with pytest.raises(binding.DsaError, match="consumer"):
        binding.LayerStack(None, "F", [None], 4, consumer=lambda *a: None, graphed=True)


def test_layer_inputs_strides_and_weight_dtype_checked_on_the_host():
    """DsaLayerInputs row strides and w dtype: bad values are rejected before
    any launch; the fused projection's views (strides 192, bf16 w) pass the
    host checks (then report no device here)."""
    lib = binding.load()
    b = binding.DsaBatchC(1, 1, 1, 1, 100, 2, 4, 256, 256, 256, 256)
    fs = b"F"

    def run(**kw):
        L = dict(q=256, w=256 + 256, k_new=256, k_cache=256, k_row_stride=0, w_row_stride=0, w_dtype=0)
        L.update(kw)
        arr = (binding.DsaLayerInputsC * 1)(binding.DsaLayerInputsC(**L))
        plan = binding.DsaStackPlanC(1, fs, arr, 64, 0.0, 0, None, None, 0)
        return lib.dsa_layer_stack_run(ctypes.byref(plan), ctypes.byref(b), ctypes.c_void_p(256),
                                       ctypes.c_void_p(256), ctypes.c_void_p(256), None, binding.CONSUMER_FN(),
                                       None, ctypes.c_void_p(256), 1 << 30, None, None)

    for bad in [dict(w_dtype=2), dict(w_dtype=-1), dict(k_row_stride=100), dict(k_row_stride=132),
                dict(k_row_stride=-8), dict(w_row_stride=63), dict(w_row_stride=-1),
                dict(w=256 + 3, w_dtype=1), dict(w=256 + 2, w_dtype=0)]:
        assert run(**bad) == binding.DSA_EINVAL, bad
    if not torch.cuda.is_available():  # on a GPU these placeholder pointers would reach the kernels
        assert run(k_row_stride=192, w_row_stride=192, w=256 + 256, w_dtype=1) == binding.DSA_ENODEV


def test_step_work_from_host_metadata_matches_per_token_sum():
    # decode_keys / prefill_pairs of DsaStackPlan: the keys each token sees
    # (position + 1), summed per segment; here against the synthetic batches'
    # own per-token positions
    from dsa_sparse_attention_quant_gb300 import synth
    for hb in (synth.make_batch(3, [900, 2500, 64], [(700, 500), (40, 3)], 256, with_data=False),
               synth.stack_layer(0, scale=0.05, n_decode=6, with_data=False),
               synth.make_batch(4, [], [(300, 300)], 64, with_data=False)):
        dk, pp = binding.Batch.work_from_host(hb.query_start_loc, hb.seq_lens, hb.num_decodes)
        td = int(hb.query_start_loc[hb.num_decodes])
        keys = hb.positions.astype(np.int64) + 1
        assert dk == int(keys[:td].sum()) and pp == int(keys[td:].sum())


def test_decode_sms_query_needs_a_device():
    if torch.cuda.is_available():
        pytest.skip("checked on the GPU by the stack tests")
    from dsa_sparse_attention_quant_gb300 import synth
    hb = synth.make_batch(3, [900, 2500], [(700, 500)], 256, with_data=False)
    lib = binding.load()
    plan = binding.DsaStackPlanC()
    plan.decode_keys, plan.prefill_pairs = binding.Batch.work_from_host(hb.query_start_loc, hb.seq_lens, hb.num_decodes)
    out = ctypes.c_int32(-1)
    assert lib.dsa_layer_stack_decode_sms(ctypes.byref(plan), None, ctypes.byref(out)) != 0  # no batch
    assert lib.dsa_layer_stack_decode_sms(None, None, ctypes.byref(out)) != 0
