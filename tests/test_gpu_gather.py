"""The consumer's gather of the selected rows by physical slot, GPU against oracle.

The sparse MLA of each layer reads, per query token, the KV rows of its
selected keys, by the physical slots the indexer produced. The row format is
not on the pages, so the gather moves bytes; it must equal the oracle's byte
for byte, with zero rows for -1 and for out-of-range ids (flagged)."""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_quant_gb300 as dsa
import oracle
from tests.gpu_harness import DEV

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("row_bytes,stride,k", [(656, 656, 256), (144, 160, 2048), (16, 16, 7)])
def test_gather_rows_bit_exact(row_bytes, stride, k):
    rng = np.random.default_rng(row_bytes + k)
    R, T = 3000, 29
    rows = rng.integers(0, 256, size=(R, stride), dtype=np.uint8)
    phys = rng.integers(-1, R, size=(T, k)).astype(np.int32)
    phys[3, : k // 2] = -1  # a short row's tail
    phys[7, 0] = R          # out of range: zeros, flagged
    ref, bad = oracle.gather_rows(rows, phys, row_bytes)
    assert bad == 1
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = dsa.gather_rows(torch.from_numpy(rows).to(DEV), torch.from_numpy(phys).to(DEV), row_bytes, dev_err=err)
    assert np.array_equal(out.cpu().numpy(), ref)
    assert int(err.item()) == 4  # DSA_DEVERR_ID_RANGE


def test_gather_rows_empty_and_all_padding():
    rows = torch.zeros((4, 32), dtype=torch.uint8, device=DEV)
    out = dsa.gather_rows(rows, torch.zeros((0, 8), dtype=torch.int32, device=DEV), 32)
    assert out.shape == (0, 8, 32)
    phys = torch.full((3, 5), -1, dtype=torch.int32, device=DEV)
    out = dsa.gather_rows(rows + 9, phys, 16)
    assert int(out.sum().item()) == 0
