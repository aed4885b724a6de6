"""Parity at the full workload sizes, through the same calls the benchmark
times: every cache byte bit-exact, and scores / top-k / physical ids on every
row the oracle can afford (all rows for the decode workloads, a seeded sample
of rows for the long prefill and the layer stack)."""
import numpy as np
import pytest

import oracle
from dsa_sparse_attention_quant_gb300 import synth
from tests.test_gpu_parity import check_batch
from tests.test_gpu_stack import run_stack

pytestmark = pytest.mark.gpu


def sampled_rows(hb, n_per_req: int, seed: int):
    """First, last and seeded random query rows of every request."""
    rows = []
    qsl = hb.query_start_loc
    for r in range(hb.num_reqs):
        a, b = int(qsl[r]), int(qsl[r + 1])
        if b - a <= n_per_req:
            rows.extend(range(a, b))
            continue
        u = synth.uniform01(seed, 100 + r, n_per_req - 2)
        pick = {a, b - 1} | {a + int(x * (b - a)) for x in u}
        rows.extend(sorted(pick))
    return np.array(sorted(set(rows)), np.int64)


def test_decode32_full():
    check_batch(synth.decode32())


def test_decode8x128k_full():
    check_batch(synth.decode8x128k(), check_logits=True)


def test_prefill4x8k_sampled_rows():
    hb = synth.prefill4x8k()
    check_batch(hb, rows=sampled_rows(hb, 16, 31), check_logits=True)


def test_stack61_layers_full_size_sampled_rows():
    # the 61-layer schedule itself is pinned exactly on the CPU; here the first
    # five layers (F F S S S) run at full per-layer size
    hb0 = synth.stack_layer(0)
    rows = np.concatenate([np.arange(0, 64, 8), sampled_rows(hb0, 24, 47)[sampled_rows(hb0, 24, 47) >= 64]])
    fs = run_stack(5, 4, scale=1.0, n_decode=64, check_rows=rows)
    assert fs == "FFSSS"
    assert oracle.schedule(61, True, 4)[0].count("F") == 16
