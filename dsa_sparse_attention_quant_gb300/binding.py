"""ctypes binding of ``libdsaidx.so`` (the C ABI of ``include/dsaidx.h``).

Argument marshalling only: every step of the indexer runs in the library's
CUDA kernels. Torch supplies device memory (outputs and workspaces are
allocated with torch when the caller does not pass them) and the current
CUDA stream. If the library is missing or no sm_103 GPU is present the calls
raise; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import numpy as np

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

DSA_OK, DSA_EINVAL, DSA_ECUDA, DSA_EDEVICE, DSA_ENOSPACE, DSA_ENODEV = range(6)
DEVERR = {
    1: "slot out of range",
    2: "block id out of range",
    4: "top-k id out of range",
    8: "pipeline wait timed out",
    16: "seq_len inconsistent",
}
HEADS, HEAD_DIM, BLOCK_SIZE, PAGE_BYTES = 64, 128, 64, 8448
FP4_PAGE_BYTES = 4352  # 64 slots x (64 E2M1 code bytes + 4 scale bytes)

SYMBOLS = [
    "dsa_status_string", "dsa_version", "dsa_check_device_error",
    "dsa_indexer_k_quant_write", "dsa_indexer_q_quant_fold",
    "dsa_indexer_workspace_size", "dsa_indexer_logits_topk",
    "dsa_indexer_plan", "dsa_indexer_logits", "dsa_indexer_topk",
    "dsa_topk_logical_to_physical", "dsa_schedule_build",
    "dsa_layer_stack_workspace_size", "dsa_layer_stack_run", "dsa_layer_stack_decode_sms",
    "dsa_indexer_logits_topk_static", "dsa_set_launch_events",
    "dsa_indexer_k_rope_quant_write", "dsa_indexer_q_rope_quant_fold", "dsa_gather_rows",
    "dsa_indexer_k_quant_write_fp4", "dsa_selftest_wait_timeout",
]
STATIC_WORKSPACE_BYTES = 32 << 20


class DsaError(RuntimeError):
    pass


class DsaBatchC(ctypes.Structure):
    _fields_ = [
        ("num_reqs", ctypes.c_int32),
        ("num_decodes", ctypes.c_int32),
        ("num_decode_tokens", ctypes.c_int32),
        ("num_tokens", ctypes.c_int32),
        ("max_seq_len", ctypes.c_int32),
        ("bt_stride", ctypes.c_int64),
        ("num_blocks", ctypes.c_int64),
        ("query_start_loc", ctypes.c_void_p),
        ("seq_lens", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("req_id_per_token", ctypes.c_void_p),
        ("k_cache_format", ctypes.c_int32),
    ]


class DsaLayerInputsC(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p),
        ("w", ctypes.c_void_p),
        ("k_new", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p),
        ("k_row_stride", ctypes.c_int64),
        ("w_row_stride", ctypes.c_int64),
        ("w_dtype", ctypes.c_int32),
    ]


CONSUMER_FN = ctypes.CFUNCTYPE(None, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_void_p)


class DsaStackPlanC(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32),
        ("fs", ctypes.c_char_p),
        ("layers", ctypes.POINTER(DsaLayerInputsC)),
        ("topk", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("block_stride_rows", ctypes.c_int32),
        ("positions", ctypes.c_void_p),
        ("rope_cos_sin", ctypes.c_void_p),
        ("rope_max_pos", ctypes.c_int64),
        ("decode_keys", ctypes.c_int64),
        ("prefill_pairs", ctypes.c_int64),
    ]


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libdsaidx.so (building it with nvcc first if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise DsaError(f"{path} is not built")
            _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I32, I64, F32, SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        BP = ctypes.POINTER(DsaBatchC)
        sig = {
            "dsa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "dsa_version": (ctypes.c_int, []),
            "dsa_check_device_error": (ctypes.c_int, [P, P, P]),
            "dsa_indexer_k_quant_write": (ctypes.c_int, [P, I64, I64, P, P, I64, P, P]),
            "dsa_indexer_q_quant_fold": (ctypes.c_int, [P, P, I64, F32, P, P, P, P]),
            "dsa_indexer_workspace_size": (SZ, [BP, I32]),
            "dsa_indexer_logits_topk": (ctypes.c_int, [BP, P, P, P, I32, P, P, SZ, P, P, P, P]),
            "dsa_indexer_plan": (ctypes.c_int, [BP, P, SZ, P, P]),
            "dsa_indexer_logits": (ctypes.c_int, [BP, P, P, P, P, I64, P, SZ, P, P]),
            "dsa_indexer_topk": (ctypes.c_int, [BP, P, I64, I32, P, P, SZ, P]),
            "dsa_topk_logical_to_physical": (ctypes.c_int, [P, I64, I32, P, P, I32, I64, I32, P, P, P, P]),
            "dsa_schedule_build": (ctypes.c_int, [I32, I32, I32, I32, ctypes.c_char_p, P, P]),
            "dsa_layer_stack_workspace_size": (SZ, [BP, I32]),
            "dsa_layer_stack_run": (ctypes.c_int, [ctypes.POINTER(DsaStackPlanC), BP, P, P, P, P, CONSUMER_FN, P, P,
                                                   SZ, P, P]),
            "dsa_indexer_logits_topk_static": (ctypes.c_int, [BP, P, P, P, I32, P, P, P, P, P]),
            "dsa_layer_stack_decode_sms": (ctypes.c_int, [ctypes.POINTER(DsaStackPlanC), BP, P]),
            "dsa_set_launch_events": (ctypes.c_int, [P, I32]),
            "dsa_indexer_k_rope_quant_write": (ctypes.c_int, [P, I64, I64, P, P, I64, P, P, I64, P, P]),
            "dsa_indexer_k_quant_write_fp4": (ctypes.c_int, [P, I64, I64, P, P, I64, P, P, I64, P, P]),
            "dsa_selftest_wait_timeout": (ctypes.c_int, [P, P]),
            "dsa_indexer_q_rope_quant_fold": (ctypes.c_int, [P, P, I64, P, P, I64, F32, P, P, P, P, P]),
            "dsa_gather_rows": (ctypes.c_int, [P, I64, I64, I64, P, I64, I32, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int, what: str) -> None:
    if status != DSA_OK:
        msg = load().dsa_status_string(status).decode()
        raise DsaError(f"{what}: {msg} (status {status})")


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, what):
    if not t.is_cuda:
        raise DsaError(f"{what} must be a CUDA tensor")
    if t.dtype != dtype:
        raise DsaError(f"{what} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise DsaError(f"{what} must be contiguous")


# ---------------------------------------------------------------- batches

class Batch:
    """Device-side step metadata (the C ``DsaBatch``) plus the tensors it points to."""

    def __init__(self, query_start_loc, seq_lens, block_table, req_id_per_token, num_decodes: int,
                 num_blocks: int, max_seq_len: int | None = None, num_decode_tokens: int | None = None):
        for t, n in ((query_start_loc, "query_start_loc"), (seq_lens, "seq_lens"), (block_table, "block_table"),
                     (req_id_per_token, "req_id_per_token")):
            _need(t, torch.int32, n)
        self.query_start_loc = query_start_loc
        self.seq_lens = seq_lens
        self.block_table = block_table
        self.req_id_per_token = req_id_per_token
        self.num_reqs = int(seq_lens.shape[0])
        self.num_tokens = int(req_id_per_token.shape[0])
        self.num_decodes = int(num_decodes)
        self.num_blocks = int(num_blocks)
        if max_seq_len is None:
            max_seq_len = int(seq_lens.max().item()) if self.num_reqs else 1
        self.max_seq_len = int(max_seq_len)
        if num_decode_tokens is None:
            num_decode_tokens = int(query_start_loc[self.num_decodes].item()) if self.num_reqs else 0
        self.num_decode_tokens = int(num_decode_tokens)
        self.work = (0, 0)  # (decode_keys, prefill_pairs) when known on the host; see work_from_host
        self.c = DsaBatchC(self.num_reqs, self.num_decodes, self.num_decode_tokens, self.num_tokens, self.max_seq_len,
                           int(block_table.shape[1]) if block_table.dim() == 2 else 1, self.num_blocks,
                           query_start_loc.data_ptr(), seq_lens.data_ptr(), block_table.data_ptr(),
                           req_id_per_token.data_ptr())

    @staticmethod
    def work_from_host(query_start_loc, seq_lens, num_decodes: int):
        """(decode_keys, prefill_pairs) of a step from host copies of its
        metadata: the sums over the decode and the prefill tokens of the keys
        each token sees (position + 1), as ``DsaStackPlan`` takes them."""
        qsl = np.asarray(query_start_loc, dtype=np.int64)
        sl = np.asarray(seq_lens, dtype=np.int64)
        ql = qsl[1:] - qsl[:-1]
        # a request of ql tokens ending at length sl: its tokens see sl - ql + 1 .. sl keys
        per_req = ql * (sl - ql) + ql * (ql + 1) // 2
        return int(per_req[:num_decodes].sum()), int(per_req[num_decodes:].sum())

    @classmethod
    def from_host(cls, hb, device="cuda"):
        """From a ``synth.Batch`` (numpy metadata) to device tensors."""
        def d(a):
            return torch.from_numpy(a.astype("int32")).to(device)
        b = cls(d(hb.query_start_loc), d(hb.seq_lens), d(hb.block_table), d(hb.req_id_per_token),
                hb.num_decodes, hb.num_blocks, int(hb.seq_lens.max()) if hb.num_reqs else 1,
                int(hb.query_start_loc[hb.num_decodes]) if hb.num_reqs else 0)
        b.work = cls.work_from_host(hb.query_start_loc, hb.seq_lens, hb.num_decodes)
        return b


def selftest_wait_timeout(dev_err, stream=None):
    """Diagnostic: a bounded pipeline wait on a barrier nothing completes; after
    about 1 s it sets DSA_DEVERR_TIMEOUT (8) in ``dev_err`` and returns."""
    _need(dev_err, torch.int32, "dev_err")
    _check(load().dsa_selftest_wait_timeout(_ptr(dev_err), _stream(stream)), "dsa_selftest_wait_timeout")


# ---------------------------------------------------------------- K caches

def new_k_cache(num_blocks: int, fmt: str = "fp8", device=None):
    """A zeroed indexer K cache of ``num_blocks`` pages: FP8 (8448-byte pages) or
    FP4 (4352-byte pages of E2M1 codes)."""
    if fmt not in ("fp8", "fp4"):
        raise DsaError("fmt must be 'fp8' or 'fp4'")
    page = FP4_PAGE_BYTES if fmt == "fp4" else PAGE_BYTES
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    return torch.zeros((int(num_blocks), page), dtype=torch.uint8, device=dev)


def cache_format(k_cache) -> int:
    """DSA_KCACHE_FP8 (0) or DSA_KCACHE_FP4 (1), from the page size of a
    [num_blocks, page_bytes] (or [num_blocks, ...]) uint8 K cache."""
    if k_cache.dtype != torch.uint8:
        raise DsaError(f"k_cache must be torch.uint8, got {k_cache.dtype}")
    if k_cache.dim() < 2:
        raise DsaError("k_cache must be [num_blocks, page bytes] (or [num_blocks, 64, slot bytes])")
    page = math.prod(int(d) for d in k_cache.shape[1:])
    if page == PAGE_BYTES:
        return 0
    if page == FP4_PAGE_BYTES:
        return 1
    raise DsaError(f"k_cache pages of {page} bytes are neither FP8 ({PAGE_BYTES}) nor FP4 ({FP4_PAGE_BYTES})")


def _bind_format(batch, k_cache):
    batch.c.k_cache_format = cache_format(k_cache)


# ---------------------------------------------------------------- entry points

def indexer_k_quant_write(k, slot_mapping, k_cache, dev_err=None, stream=None):
    """S1: quantise bf16 K rows into the cache at their slots, FP8 or FP4 by the
    cache's page size."""
    _need(slot_mapping, torch.int64, "slot_mapping")
    _need(k_cache, torch.uint8, "k_cache")
    fp4 = cache_format(k_cache) == 1
    n = int(slot_mapping.shape[0])
    if n == 0:
        return
    if k.dtype != torch.bfloat16 or not k.is_cuda or k.stride(-1) != 1:
        raise DsaError("k must be a CUDA bf16 tensor with unit inner stride")
    row_stride = int(k.stride(0)) if k.dim() == 2 else HEAD_DIM
    if fp4:
        st = load().dsa_indexer_k_quant_write_fp4(_ptr(k), n, row_stride, None, None, 0, _ptr(slot_mapping),
                                                  _ptr(k_cache), int(k_cache.shape[0]), _ptr(dev_err),
                                                  _stream(stream))
        _check(st, "dsa_indexer_k_quant_write_fp4")
        return
    st = load().dsa_indexer_k_quant_write(_ptr(k), n, row_stride, _ptr(slot_mapping), _ptr(k_cache),
                                          int(k_cache.shape[0]), _ptr(dev_err), _stream(stream))
    _check(st, "dsa_indexer_k_quant_write")


def gather_rows(rows, physical, row_bytes: int, out=None, dev_err=None, stream=None):
    """The consumer's gather: out[t, j] = the first row_bytes bytes of
    rows[physical[t, j]] (uint8 [R, stride]); zero rows for -1."""
    _need(rows, torch.uint8, "rows")
    _need(physical, torch.int32, "physical")
    T, k = physical.shape
    if out is None:
        out = torch.empty((T, k, int(row_bytes)), dtype=torch.uint8, device=physical.device)
    st = load().dsa_gather_rows(_ptr(rows), int(rows.shape[0]), int(row_bytes), int(rows.stride(0)),
                                _ptr(physical), T, k, _ptr(out), _ptr(dev_err), _stream(stream))
    _check(st, "dsa_gather_rows")
    return out


def _rope_table(cos_sin):
    _need(cos_sin, torch.float32, "cos_sin")
    if cos_sin.dim() != 2 or cos_sin.shape[1] != 64:
        raise DsaError("cos_sin must be [max_pos, 64] fp32")
    return int(cos_sin.shape[0])


def indexer_k_rope_quant_write(k, positions, cos_sin, slot_mapping, k_cache, dev_err=None, stream=None):
    """RoPE of k's leading 64 dims (by positions and the cos/sin table), then S1."""
    _need(slot_mapping, torch.int64, "slot_mapping")
    _need(positions, torch.int64, "positions")
    _need(k_cache, torch.uint8, "k_cache")
    fp4 = cache_format(k_cache) == 1
    max_pos = _rope_table(cos_sin)
    n = int(slot_mapping.shape[0])
    if n == 0:
        return
    if k.dtype != torch.bfloat16 or not k.is_cuda or k.stride(-1) != 1:
        raise DsaError("k must be a CUDA bf16 tensor with unit inner stride")
    row_stride = int(k.stride(0)) if k.dim() == 2 else HEAD_DIM
    fn = load().dsa_indexer_k_quant_write_fp4 if fp4 else load().dsa_indexer_k_rope_quant_write
    st = fn(_ptr(k), n, row_stride, _ptr(positions), _ptr(cos_sin), max_pos, _ptr(slot_mapping), _ptr(k_cache),
            int(k_cache.shape[0]), _ptr(dev_err), _stream(stream))
    _check(st, "dsa_indexer_k_quant_write_fp4" if fp4 else "dsa_indexer_k_rope_quant_write")


def indexer_q_rope_quant_fold(q, w, positions, cos_sin, softmax_scale: float = 0.0, q_fp8=None, q_scale=None,
                              w_folded=None, dev_err=None, stream=None):
    """RoPE of every q head's leading 64 dims, then S2a."""
    _need(q, torch.bfloat16, "q")
    _need(w, torch.float32, "w")
    _need(positions, torch.int64, "positions")
    max_pos = _rope_table(cos_sin)
    T = int(q.shape[0])
    if q_fp8 is None:
        q_fp8 = torch.empty((T, HEADS, HEAD_DIM), dtype=torch.uint8, device=q.device)
    if w_folded is None:
        w_folded = torch.empty((T, HEADS), dtype=torch.float32, device=q.device)
    st = load().dsa_indexer_q_rope_quant_fold(_ptr(q), _ptr(w), T, _ptr(positions), _ptr(cos_sin), max_pos,
                                              float(softmax_scale), _ptr(q_fp8), _ptr(q_scale), _ptr(w_folded),
                                              _ptr(dev_err), _stream(stream))
    _check(st, "dsa_indexer_q_rope_quant_fold")
    return q_fp8, q_scale, w_folded


def indexer_q_quant_fold(q, w, softmax_scale: float = 0.0, q_fp8=None, q_scale=None, w_folded=None, stream=None):
    _need(q, torch.bfloat16, "q")
    _need(w, torch.float32, "w")
    T = int(q.shape[0])
    if q_fp8 is None:
        q_fp8 = torch.empty((T, HEADS, HEAD_DIM), dtype=torch.uint8, device=q.device)
    if w_folded is None:
        w_folded = torch.empty((T, HEADS), dtype=torch.float32, device=q.device)
    st = load().dsa_indexer_q_quant_fold(_ptr(q), _ptr(w), T, float(softmax_scale), _ptr(q_fp8), _ptr(q_scale),
                                         _ptr(w_folded), _stream(stream))
    _check(st, "dsa_indexer_q_quant_fold")
    return q_fp8, q_scale, w_folded


def indexer_workspace_size(batch: Batch, topk: int) -> int:
    return int(load().dsa_indexer_workspace_size(ctypes.byref(batch.c), int(topk)))


def _workspace(nbytes: int, device, ws=None):
    if ws is None:
        ws = torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)
    return ws


def indexer_logits_topk(batch: Batch, q_fp8, w_folded, k_cache, topk: int, topk_out=None, ws=None, k_new=None,
                        slot_mapping=None, dev_err=None, stream=None):
    dev = q_fp8.device
    if topk_out is None:
        topk_out = torch.empty((batch.num_tokens, int(topk)), dtype=torch.int32, device=dev)
    nbytes = indexer_workspace_size(batch, topk)
    ws = _workspace(nbytes, dev, ws)
    _bind_format(batch, k_cache)
    st = load().dsa_indexer_logits_topk(ctypes.byref(batch.c), _ptr(q_fp8), _ptr(w_folded), _ptr(k_cache),
                                        int(topk), _ptr(topk_out), _ptr(ws), ws.numel(), _ptr(k_new),
                                        _ptr(slot_mapping), _ptr(dev_err), _stream(stream))
    _check(st, "dsa_indexer_logits_topk")
    return topk_out


def indexer_logits_topk_static(batch: Batch, q_fp8, w_folded, k_cache, topk: int, topk_out, k_new=None,
                               slot_mapping=None, dev_err=None, stream=None):
    """``indexer_logits_topk`` without any allocation: for callers that cannot
    allocate device memory. ``topk_out`` must be passed; the scratch is the
    library's own static device array (DSA_STATIC_WORKSPACE_BYTES), shared by
    all calls, so calls must not overlap on the GPU."""
    _bind_format(batch, k_cache)
    st = load().dsa_indexer_logits_topk_static(ctypes.byref(batch.c), _ptr(q_fp8), _ptr(w_folded), _ptr(k_cache),
                                               int(topk), _ptr(topk_out), _ptr(k_new), _ptr(slot_mapping),
                                               _ptr(dev_err), _stream(stream))
    _check(st, "dsa_indexer_logits_topk_static")
    return topk_out


def indexer_plan(batch: Batch, ws=None, dev_err=None, stream=None):
    """Plan the batch into ``ws`` (allocated if None) and return ``ws``."""
    dev = batch.seq_lens.device
    ws = _workspace(indexer_workspace_size(batch, 4), dev, ws)
    st = load().dsa_indexer_plan(ctypes.byref(batch.c), _ptr(ws), ws.numel(), _ptr(dev_err), _stream(stream))
    _check(st, "dsa_indexer_plan")
    return ws


def indexer_logits(batch: Batch, q_fp8, w_folded, k_cache, logits=None, ws=None, dev_err=None, stream=None):
    """Scores of every causal (token, key) pair; plans into ``ws`` first when ``ws`` is None."""
    dev = q_fp8.device
    ld = (batch.max_seq_len + 3) // 4 * 4
    if logits is None:
        logits = torch.full((batch.num_tokens, ld), float("nan"), dtype=torch.float32, device=dev)
    if ws is None:
        ws = indexer_plan(batch, dev_err=dev_err, stream=stream)
    _bind_format(batch, k_cache)
    st = load().dsa_indexer_logits(ctypes.byref(batch.c), _ptr(q_fp8), _ptr(w_folded), _ptr(k_cache),
                                   _ptr(logits), int(logits.stride(0)), _ptr(ws), ws.numel(), _ptr(dev_err),
                                   _stream(stream))
    _check(st, "dsa_indexer_logits")
    return logits


def indexer_topk(batch: Batch, logits, topk: int, topk_out=None, stream=None):
    if topk_out is None:
        topk_out = torch.empty((batch.num_tokens, int(topk)), dtype=torch.int32, device=logits.device)
    st = load().dsa_indexer_topk(ctypes.byref(batch.c), _ptr(logits), int(logits.stride(0)), int(topk),
                                 _ptr(topk_out), None, 0, _stream(stream))
    _check(st, "dsa_indexer_topk")
    return topk_out


def topk_logical_to_physical(logical, req_id_per_token, block_table, block_stride_rows: int = 0, physical=None,
                             valid_counts=None, with_valid_counts: bool = True, dev_err=None, stream=None):
    _need(logical, torch.int32, "logical")
    T, k = logical.shape
    if physical is None:
        physical = torch.empty_like(logical)
    if valid_counts is None and with_valid_counts:
        valid_counts = torch.empty(T, dtype=torch.int32, device=logical.device)
    st = load().dsa_topk_logical_to_physical(_ptr(logical), int(T), int(k), _ptr(req_id_per_token),
                                             _ptr(block_table), int(block_table.shape[0]),
                                             int(block_table.shape[1]), int(block_stride_rows),
                                             _ptr(physical), _ptr(valid_counts), _ptr(dev_err), _stream(stream))
    _check(st, "dsa_topk_logical_to_physical")
    return physical, valid_counts


def schedule_build(n_layers: int, use_index_cache: bool = True, freq: int = 1, offset: int = 2,
                   pattern: str | None = None):
    """Host-side IndexCache schedule: (fs string, producer list)."""
    fs = ctypes.create_string_buffer(max(int(n_layers), 1))
    prod = (ctypes.c_int32 * max(int(n_layers), 1))()
    st = load().dsa_schedule_build(int(n_layers), int(bool(use_index_cache)), int(freq), int(offset),
                                   None if pattern is None else pattern.encode(), fs, prod)
    _check(st, "dsa_schedule_build")
    return fs.raw[:n_layers].decode(), list(prod[:n_layers])


def set_launch_events(events=()) -> None:
    """Launch timeline: the following fused calls on this thread record these
    torch.cuda.Event objects, one before the first kernel and one after every
    kernel (an empty sequence switches it off)."""
    handles = (ctypes.c_void_p * max(len(events), 1))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    st = load().dsa_set_launch_events(handles, len(events))
    _check(st, "dsa_set_launch_events")


def check_device_error(dev_err, stream=None) -> int:
    out = ctypes.c_uint32(0)
    st = load().dsa_check_device_error(_ptr(dev_err), ctypes.byref(out), _stream(stream))
    if st not in (DSA_OK, DSA_EDEVICE):
        _check(st, "dsa_check_device_error")
    return int(out.value)


def layer_stack_workspace_size(batch: Batch, topk: int) -> int:
    return int(load().dsa_layer_stack_workspace_size(ctypes.byref(batch.c), int(topk)))


def _layer_inputs(L) -> DsaLayerInputsC:
    """The C inputs of an F layer. ``w`` may be fp32 or bf16 and ``w`` and
    ``k_new`` may be row-strided 2-D views (unit inner stride), e.g. the column
    views ``kw[:, :128]`` and ``kw[:, 128:]`` of one fused projection output."""
    q, w, kn = L["q"], L["w"], L.get("k_new")
    _need(q, torch.bfloat16, "q")
    if w.dtype not in (torch.float32, torch.bfloat16) or not w.is_cuda or w.dim() != 2 or w.stride(1) != 1:
        raise DsaError("w must be a CUDA fp32 or bf16 [T, 64] tensor with unit inner stride")
    if kn is not None and (kn.dtype != torch.bfloat16 or not kn.is_cuda or kn.dim() != 2 or kn.stride(1) != 1):
        raise DsaError("k_new must be a CUDA bf16 [T, 128] tensor with unit inner stride")
    return DsaLayerInputsC(q.data_ptr(), w.data_ptr(), kn.data_ptr() if kn is not None else None,
                           L["k_cache"].data_ptr(), int(kn.stride(0)) if kn is not None else 0, int(w.stride(0)),
                           1 if w.dtype == torch.bfloat16 else 0)


class LayerStack:
    """A prepared ``dsa_layer_stack_run``: the C plan, the per-layer input table,
    the output buffers and the workspace are built once; ``run()`` issues the
    call again on the same tensors (whose contents may change between runs).
    ``layers[l]`` is None for 'S' layers, else a dict with tensors ``q``, ``w``,
    ``k_cache`` and optionally ``k_new``. ``consumer(layer, producer, phys_ptr,
    valid_ptr)`` is called per layer. With ``rope_cos_sin`` ([max_pos, 64]
    fp32) and ``positions`` (int64 [T]), q and k_new arrive un-rotated and each
    F layer rotates them (RoPE) on the way into the quantiser.

    ``graphed=True``: the first ``run()`` runs the stack and captures the same
    call into a CUDA graph; later calls replay the graph on the given stream,
    which saves the host work of each call (argument checks, tensor maps,
    launches). The graph reads and writes the same buffers, so a step's new
    inputs go into them before ``run()``; metadata that sizes the launch (the
    batch's lengths) must not change. A graphed stack takes no consumer (a
    host callback would run at capture only).

    ``work`` = (decode_keys, prefill_pairs), the step's keys seen by its decode
    tokens and by its prefill tokens (``Batch.work_from_host``); by default the
    batch's own, known when it was built from host metadata. With both given,
    each F layer scores the decode rows on a share of the SMs beside the
    prefill rows (``DsaStackPlan.decode_keys``); (0, 0) keeps one after the
    other."""

    def __init__(self, batch: Batch, fs: str, layers, topk: int, slot_mapping=None, topk_buf=None, phys_buf=None,
                 valid_buf=None, consumer=None, ws=None, softmax_scale: float = 0.0, block_stride_rows: int = 0,
                 dev_err=None, positions=None, rope_cos_sin=None, graphed: bool = False, work=None):
        if graphed and consumer is not None:
            raise DsaError("a graphed LayerStack takes no consumer: a host callback runs only at capture")
        self._graphed = bool(graphed)
        self._graph = None
        n = len(fs)
        self._arr = (DsaLayerInputsC * max(n, 1))()
        self._keep = [batch, slot_mapping, dev_err, positions, rope_cos_sin]
        fmts = {cache_format(L["k_cache"]) for L in layers if L is not None}
        if len(fmts) > 1:
            raise DsaError("all layers' K caches must have one format")
        if fmts:
            batch.c.k_cache_format = fmts.pop()
        for l, L in enumerate(layers):
            if L is None:
                continue
            self._keep.append(L)
            self._arr[l] = _layer_inputs(L)
        max_pos = 0
        if rope_cos_sin is not None:
            max_pos = _rope_table(rope_cos_sin)
            _need(positions, torch.int64, "positions")
        self._fs = fs.encode()
        decode_keys, prefill_pairs = batch.work if work is None else work
        self._plan = DsaStackPlanC(n, self._fs, self._arr, int(topk), float(softmax_scale), int(block_stride_rows),
                                   _ptr(positions) if rope_cos_sin is not None else None, _ptr(rope_cos_sin),
                                   max_pos, int(decode_keys), int(prefill_pairs))
        dev = torch.device("cuda", torch.cuda.current_device())
        T = batch.num_tokens
        self.topk_buf = topk_buf if topk_buf is not None else torch.empty((T, int(topk)), dtype=torch.int32,
                                                                          device=dev)
        self.phys_buf = phys_buf if phys_buf is not None else torch.empty((T, int(topk)), dtype=torch.int32,
                                                                          device=dev)
        self.valid_buf = valid_buf if valid_buf is not None else torch.empty(T, dtype=torch.int32, device=dev)
        self.ws = _workspace(layer_stack_workspace_size(batch, topk), dev, ws)
        if consumer is not None:
            self._cb = CONSUMER_FN(lambda l, p, ph, va, u: consumer(int(l), int(p), ph, va))
        else:
            self._cb = CONSUMER_FN()
        self._fn = load().dsa_layer_stack_run
        self._args = (ctypes.byref(self._plan), ctypes.byref(batch.c), _ptr(slot_mapping), _ptr(self.topk_buf),
                      _ptr(self.phys_buf), _ptr(self.valid_buf), self._cb, None, _ptr(self.ws), self.ws.numel(),
                      _ptr(dev_err))

    def decode_sms(self) -> int:
        """SMs each F layer gives the decode rows' scores beside the prefill
        rows' (0: one after the other)."""
        out = ctypes.c_int32(0)
        _check(load().dsa_layer_stack_decode_sms(ctypes.byref(self._plan), self._args[1], ctypes.byref(out)),
               "dsa_layer_stack_decode_sms")
        return int(out.value)

    def run(self, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream()
        if self._graph is not None:
            with torch.cuda.stream(s):
                self._graph.replay()
            return self.topk_buf, self.phys_buf, self.valid_buf
        st = self._fn(*self._args, ctypes.c_void_p(s.cuda_stream))
        _check(st, "dsa_layer_stack_run")
        if self._graphed:  # capture the same call (the eager call above did any first-use set-up)
            side = torch.cuda.Stream(device=s.device)
            side.wait_stream(s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                st = self._fn(*self._args, ctypes.c_void_p(side.cuda_stream))
            s.wait_stream(side)
            _check(st, "dsa_layer_stack_run (capture)")
            self._graph = g
        return self.topk_buf, self.phys_buf, self.valid_buf


def layer_stack_run(batch: Batch, fs: str, layers, topk: int, slot_mapping=None, topk_buf=None, phys_buf=None,
                    valid_buf=None, consumer=None, ws=None, softmax_scale: float = 0.0, block_stride_rows: int = 0,
                    dev_err=None, stream=None, positions=None, rope_cos_sin=None, work=None):
    """Run a stack of layers once (see ``LayerStack`` for the arguments)."""
    return LayerStack(batch, fs, layers, topk, slot_mapping, topk_buf, phys_buf, valid_buf, consumer, ws,
                      softmax_scale, block_stride_rows, dev_err, positions, rope_cos_sin, work=work).run(stream)
