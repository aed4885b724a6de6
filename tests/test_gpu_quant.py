"""Quantiser edge cases on the GPU, bit for bit against the oracle.

The GPU finds each group's power-of-two scale from the exponent bits of amax
(no division); the oracle divides amax by 448 and rounds up to a power of two
("Indexer.forward" and the FP8 indexer-cache snippet of "IndexCache：DeepSeek
稀疏注意力中的跨层索引复用": per-token group FP8 quantisation with ue8m0 scales).
These rows put amax exactly on and next to every scale boundary (448*2^k and
the bf16 values beside it) across the exponent range, plus all-zero rows,
rows below the 1e-10 floor, bf16 subnormals and the largest bf16 values.
"""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_quant_gb300 as dsa
import oracle
from dsa_sparse_attention_quant_gb300 import synth
from tests.gpu_harness import DEV
from tests.test_gpu_parity import fold_reference

pytestmark = pytest.mark.gpu


def edge_rows() -> np.ndarray:
    """bf16 bit patterns [R, 128]: one designated amax per row, the rest smaller."""
    amaxes = []
    for k in range(-132, 121):  # 448 * 2^k spans the normal bf16 range
        for m in (1.0, 1.7421875, 1.75, 1.7578125, 1.9921875):
            e = k + 8
            if -126 <= e <= 127:
                amaxes.append(np.ldexp(m, e))
    rng = np.random.default_rng(7)
    rows = []
    for i, a in enumerate(amaxes):
        x = rng.uniform(-1.0, 1.0, 128) * a * 0.9
        x[i % 128] = a if i % 2 else -a
        rows.append(synth.bf16_bits(x))
    specials = [np.zeros(128), np.full(128, 1e-12), np.full(128, -3e-39),  # zero, below the floor, subnormal
                np.full(128, 3.3895313892515355e38), np.linspace(-1e-10, 1e-10, 128)]
    rows += [synth.bf16_bits(x) for x in specials]
    r = np.stack(rows)
    r[-3, 5] = 0x7F7F  # the largest finite bf16
    return r


def test_k_quant_scale_boundaries_bit_exact():
    k = edge_rows()
    n = k.shape[0]
    blocks = (n + 63) // 64
    slots = np.arange(n, dtype=np.int64)
    ref = oracle.new_cache(blocks)
    oracle.k_quant_write(k, slots, ref)
    cache = torch.zeros((blocks, 8448), dtype=torch.uint8, device=DEV)
    kt = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).to(DEV)
    dsa.indexer_k_quant_write(kt, torch.from_numpy(slots).to(DEV), cache)
    got = cache.cpu().numpy()
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} cache bytes differ"


def test_q_quant_scale_boundaries_bit_exact():
    k = edge_rows()
    T = (k.shape[0] + 63) // 64
    q = np.zeros((T * 64, 128), np.uint16)
    q[: k.shape[0]] = k
    q = q.reshape(T, 64, 128)
    w = np.random.default_rng(8).standard_normal((T, 64)).astype(np.float32)
    codes, scales = oracle.q_quant(q)
    qt = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(DEV)
    q8, qs, wf = dsa.indexer_q_quant_fold(qt, torch.from_numpy(w).to(DEV),
                                          q_scale=torch.empty((T, 64), dtype=torch.float32, device=DEV))
    assert np.array_equal(q8.cpu().numpy(), codes)
    assert np.array_equal(qs.cpu().numpy().view(np.uint32), scales.view(np.uint32))
    assert np.array_equal(wf.cpu().numpy().view(np.uint32), fold_reference(w, scales).view(np.uint32))
