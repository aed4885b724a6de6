"""GB300-native (sm_103a) DSA sparse-attention indexer with IndexCache reuse.

The compute lives in ``libdsaidx.so`` (CUDA kernels behind the C ABI of
``include/dsaidx.h``); ``binding`` is its thin Python face. ``synth`` builds
seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    Batch,
    DsaError,
    LayerStack,
    cache_format,
    check_device_error,
    gather_rows,
    indexer_k_quant_write,
    indexer_k_rope_quant_write,
    indexer_logits,
    indexer_logits_topk,
    indexer_plan,
    indexer_q_quant_fold,
    indexer_q_rope_quant_fold,
    indexer_topk,
    indexer_workspace_size,
    layer_stack_run,
    layer_stack_workspace_size,
    load,
    new_k_cache,
    schedule_build,
    topk_logical_to_physical,
)

__version__ = "0.3.1"
