"""Drives the CUDA path through the binding on a seeded ``synth.Batch`` and
collects results as numpy arrays for comparison with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import dsa_sparse_attention_quant_gb300 as dsa
from dsa_sparse_attention_quant_gb300 import synth

DEV = "cuda"


def bf16_tensor(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


class DeviceBatch:
    """A synth.Batch uploaded to the GPU, with its K cache (FP8 or FP4 pages)
    filled by the CUDA path."""

    def __init__(self, hb: synth.Batch, fill_context: bool = True, fmt: str = "fp8"):
        self.hb = hb
        self.batch = dsa.Batch.from_host(hb, DEV)
        self.q = bf16_tensor(hb.q)
        self.w = torch.from_numpy(hb.w).to(DEV)
        self.k_new = bf16_tensor(hb.k_new)
        self.slot_mapping = torch.from_numpy(hb.slot_mapping).to(DEV)
        self.k_cache = dsa.new_k_cache(hb.num_blocks, fmt, device=DEV)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=DEV)
        if fill_context and hb.ctx_k.shape[0]:
            ctx = bf16_tensor(hb.ctx_k)
            slots = torch.from_numpy(hb.ctx_slots).to(DEV)
            dsa.indexer_k_quant_write(ctx, slots, self.k_cache, self.dev_err)
            del ctx, slots

    def quant_fold(self):
        return dsa.indexer_q_quant_fold(self.q, self.w, q_scale=torch.empty((self.hb.num_tokens, 64),
                                                                            dtype=torch.float32, device=DEV))

    def run(self, with_logits: bool = False):
        """S1 (fused) + S2a + S2b + S3 + S5. Returns a dict of numpy arrays."""
        q8, qs, wf = self.quant_fold()
        out = {"q8": q8, "q_scale": qs, "w_folded": wf}
        topk = dsa.indexer_logits_topk(self.batch, q8, wf, self.k_cache, self.hb.topk, k_new=self.k_new,
                                       slot_mapping=self.slot_mapping, dev_err=self.dev_err)
        out["topk"] = topk
        if with_logits:
            out["logits"] = dsa.indexer_logits(self.batch, q8, wf, self.k_cache, dev_err=self.dev_err)
        phys, valid = dsa.topk_logical_to_physical(topk, self.batch.req_id_per_token, self.batch.block_table,
                                                   dev_err=self.dev_err)
        out["phys"] = phys
        out["valid"] = valid
        torch.cuda.synchronize()
        res = {k: v.cpu().numpy() for k, v in out.items()}
        res["dev_err"] = int(self.dev_err.item())
        res["cache"] = self.k_cache.cpu().numpy()
        return res
