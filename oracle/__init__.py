"""CPU oracle of the DSA indexer path — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and
its binding) never imports it and shares no code with it.

The arithmetic lives in ``dsa_oracle.c`` (plain C, fp64 on dequantised
values); this module compiles it on first use with gcc and wraps it with
ctypes over numpy arrays. ``Oracle(lib_path)`` binds another build of the same
source (the tests use this to load deliberately broken copies and check that
the pins catch them).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "dsa_oracle.c")
_SRC = [SOURCE, os.path.join(_HERE, "dsa_oracle.h")]
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libdsa_oracle.so")
_lock = threading.Lock()

HEADS = 64
DIM = 128
BLOCK = 64
PAGE_BYTES = 64 * 132      # FP8 cache page: 64 x 128 B E4M3 K, then 64 fp32 scales
FP4_PAGE_BYTES = 64 * 68   # FP4 cache page: 64 x 64 B E2M1 K (two per byte), then 64 fp32 scales
FMT = {"fp8": 0, "fp4": 1}
GCC_FLAGS = ["-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp",
             "-ffp-contract=off", "-fno-fast-math"]


def compile_source(src: str, out: str) -> str:
    """Compile an oracle source file into a shared library at ``out``."""
    tmp = out + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", *GCC_FLAGS, "-I", _HERE, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``dsa_oracle.c`` if the library is missing or older than its sources."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = force or not os.path.exists(_LIB_PATH) or any(
        os.path.getmtime(s) > os.path.getmtime(_LIB_PATH) for s in _SRC
    )
    if stale:
        compile_source(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I32 = ctypes.c_int
    sig = {
        "ora_e4m3_value": (ctypes.c_double, [ctypes.c_uint8]),
        "ora_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
        "ora_ue8m0_scale": (ctypes.c_float, [ctypes.c_float]),
        "ora_quant_group": (None, [P, I32, P, P]),
        "ora_slot_offsets": (None, [I64, P, P]),
        "ora_slot_offsets_fmt": (None, [I64, I32, P, P]),
        "ora_k_quant_write": (I64, [P, I64, P, P, I64]),
        "ora_k_quant_write_fmt": (I64, [P, I64, P, P, I64, I32]),
        "ora_e2m1_value": (ctypes.c_double, [ctypes.c_uint8]),
        "ora_e2m1_encode": (ctypes.c_uint8, [ctypes.c_float]),
        "ora_ue8m0_scale_e2m1": (ctypes.c_float, [ctypes.c_float]),
        "ora_quant_group_e2m1": (None, [P, I32, P, P]),
        "ora_q_quant": (None, [P, I64, P, P]),
        "ora_rope": (I64, [P, I64, I64, P, P, I64, P]),
        "ora_gather_rows": (I64, [P, I64, I64, I64, P, I64, I32, P]),
        "ora_logits_row": (None, [P, P, P, P, P, I64, P]),
        "ora_logits_row_fmt": (None, [P, P, P, P, I32, P, I64, P]),
        "ora_indexer_fmt": (I64, [P, P, P, I32, P, I64, P, P, P, I64, I32, P, P, I64]),
        "ora_topk_row": (None, [P, I64, I32, P]),
        "ora_indexer": (I64, [P, P, P, P, I64, P, P, P, I64, I32, P, P, I64]),
        "ora_convert": (None, [P, I64, I32, P, P, I64, I32, I32, P, P]),
        "ora_schedule": (I32, [I32, I32, I32, I32, ctypes.c_char_p, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def cache_format(cache: np.ndarray) -> int:
    """0 for an FP8 cache (pages of 8448 B), 1 for an FP4 cache (pages of 4352 B)."""
    assert cache.dtype == np.uint8 and cache.ndim == 2 and cache.flags["C_CONTIGUOUS"]
    if cache.shape[1] == PAGE_BYTES:
        return 0
    if cache.shape[1] == FP4_PAGE_BYTES:
        return 1
    raise ValueError(f"cache pages of {cache.shape[1]} B are neither FP8 ({PAGE_BYTES}) nor FP4 ({FP4_PAGE_BYTES})")


class Oracle:
    """The oracle's entry points over numpy arrays, bound to one compiled library."""

    def __init__(self, lib_path: str | None = None):
        self._lib = _bind(ctypes.CDLL(lib_path or build()))

    # -- E4M3 and the group scale ------------------------------------------
    def e4m3_value(self, code: int) -> float:
        return float(self._lib.ora_e4m3_value(int(code)))

    def e4m3_encode(self, v: float) -> int:
        return int(self._lib.ora_e4m3_encode(float(v)))

    def e4m3_encode_array(self, v) -> np.ndarray:
        flat = _c(v, np.float32).ravel()
        enc = self._lib.ora_e4m3_encode
        out = np.fromiter((enc(float(x)) for x in flat), dtype=np.uint8, count=flat.size)
        return out.reshape(np.shape(v))

    def ue8m0_scale(self, amax: float) -> float:
        return float(self._lib.ora_ue8m0_scale(float(amax)))

    def quant_group(self, x):
        """Quantise one group of fp32 values; returns (codes uint8, scale float)."""
        x = _c(x, np.float32)
        codes = np.zeros(x.shape[0], np.uint8)
        s = np.zeros(1, np.float32)
        self._lib.ora_quant_group(_p(x), int(x.shape[0]), _p(codes), _p(s))
        return codes, float(s[0])

    # -- E2M1 (the FP4 cache's element) --------------------------------------
    def e2m1_value(self, code: int) -> float:
        return float(self._lib.ora_e2m1_value(int(code)))

    def e2m1_encode(self, v: float) -> int:
        return int(self._lib.ora_e2m1_encode(float(v)))

    def ue8m0_scale_e2m1(self, amax: float) -> float:
        return float(self._lib.ora_ue8m0_scale_e2m1(float(amax)))

    def quant_group_e2m1(self, x):
        """Quantise one group of fp32 values to packed E2M1; returns (bytes uint8, scale)."""
        x = _c(x, np.float32)
        assert x.shape[0] % 2 == 0
        packed = np.zeros(x.shape[0] // 2, np.uint8)
        s = np.zeros(1, np.float32)
        self._lib.ora_quant_group_e2m1(_p(x), int(x.shape[0]), _p(packed), _p(s))
        return packed, float(s[0])

    # -- paged cache --------------------------------------------------------
    def slot_offsets(self, slot: int, fmt: str = "fp8"):
        kb = np.zeros(1, np.int64)
        sb = np.zeros(1, np.int64)
        self._lib.ora_slot_offsets_fmt(int(slot), FMT[fmt], _p(kb), _p(sb))
        return int(kb[0]), int(sb[0])

    @staticmethod
    def new_cache(num_blocks: int, fmt: str = "fp8") -> np.ndarray:
        return np.zeros((num_blocks, FP4_PAGE_BYTES if fmt == "fp4" else PAGE_BYTES), np.uint8)

    def k_quant_write(self, k_bf16, slot_mapping, cache: np.ndarray) -> int:
        """Quantise bf16 K rows into ``cache`` in place: uint8 [num_blocks, 8448]
        (FP8) or [num_blocks, 4352] (FP4), told apart by the page size.

        Returns the number of tokens whose slot was beyond the cache."""
        k = _c(k_bf16, np.uint16)
        sm = _c(slot_mapping, np.int64)
        fmt = cache_format(cache)
        return int(self._lib.ora_k_quant_write_fmt(_p(k), int(sm.shape[0]), _p(sm), _p(cache),
                                                   int(cache.shape[0]), fmt))

    def q_quant(self, q_bf16):
        """Quantise q rows of 128 (any leading shape); returns (codes, scales)."""
        q = _c(q_bf16, np.uint16)
        codes = np.zeros(q.shape, np.uint8)
        scales = np.zeros(q.shape[:-1], np.float32)
        self._lib.ora_q_quant(_p(q), q.size // DIM, _p(codes), _p(scales))
        return codes, scales

    def rope(self, x_bf16, positions, cos_sin, rows_per_token: int):
        """Rotate the leading 64 dims of bf16 rows of 128 (any leading shape);
        row r belongs to token r // rows_per_token. Returns (rotated bits, rows
        left unrotated because their position is outside the table)."""
        x = _c(x_bf16, np.uint16)
        pos = _c(positions, np.int64)
        cs = _c(cos_sin, np.float32)
        out = np.empty_like(x)
        bad = self._lib.ora_rope(_p(x), x.size // DIM, int(rows_per_token), _p(pos), _p(cs), int(cs.shape[0]),
                                 _p(out))
        return out, int(bad)

    def gather_rows(self, rows: np.ndarray, physical, row_bytes: int):
        """out[t, j] = the first row_bytes bytes of rows[physical[t, j]] (uint8 [R, stride]),
        zeros for -1 or an out-of-range id; returns (out, out-of-range count)."""
        assert rows.dtype == np.uint8 and rows.ndim == 2 and rows.flags["C_CONTIGUOUS"]
        ph = _c(physical, np.int32)
        T, k = ph.shape
        out = np.full((T, k, row_bytes), 0xA5, np.uint8)  # a row the gather skipped would show
        bad = self._lib.ora_gather_rows(_p(rows), rows.shape[0], int(row_bytes), rows.shape[1], _p(ph), T, k,
                                        _p(out))
        return out, int(bad)

    def fill_cache(self, batch, cache: np.ndarray | None = None, include_new: bool = True, fmt: str = "fp8"):
        """The oracle's own cache for ``batch``: context K, then this step's K."""
        if cache is None:
            cache = self.new_cache(batch.num_blocks, fmt)
        self.k_quant_write(batch.ctx_k, batch.ctx_slots, cache)
        if include_new:
            self.k_quant_write(batch.k_new, batch.slot_mapping, cache)
        return cache

    # -- scores and selection -----------------------------------------------
    def logits_row(self, q_codes, q_scale, w, cache, bt_row, n_keys: int) -> np.ndarray:
        out = np.zeros(max(int(n_keys), 1), np.float64)
        self._lib.ora_logits_row_fmt(
            _p(_c(q_codes, np.uint8)), _p(_c(q_scale, np.float32)), _p(_c(w, np.float32)),
            _p(cache), cache_format(cache), _p(_c(bt_row, np.int32)), int(n_keys), _p(out))
        return out[: int(n_keys)]

    def topk_row(self, scores, k: int) -> np.ndarray:
        sc = _c(scores, np.float64)
        out = np.zeros(int(k), np.int32)
        self._lib.ora_topk_row(_p(sc), int(sc.shape[0]), int(k), _p(out))
        return out

    def indexer(self, batch, cache: np.ndarray, rows=None, with_scores: bool = False):
        """Top-k (and optionally fp64 scores) for the given query rows of ``batch``.

        ``cache`` must already hold every key the rows see. Returns ``topk
        [n_rows, k]`` and, if asked, ``scores [n_rows, max_len]`` (entries past
        a row's length are 0).
        """
        if rows is None:
            rows = np.arange(batch.num_tokens, dtype=np.int64)
        rows = _c(rows, np.int64)
        n = int(rows.shape[0])
        k = int(batch.topk)
        topk = np.zeros((max(n, 1), k), np.int32)
        pos = _c(batch.positions, np.int64)
        ld = int(pos[rows].max() + 1) if (with_scores and n) else 0
        scores = np.zeros((max(n, 1), max(ld, 1)), np.float64) if with_scores else None
        bt = _c(batch.block_table, np.int32)
        rc = self._lib.ora_indexer_fmt(
            _p(_c(batch.q, np.uint16)), _p(_c(batch.w, np.float32)), _p(cache), cache_format(cache),
            _p(bt), int(bt.shape[1]), _p(_c(batch.req_id_per_token, np.int32)), _p(pos),
            _p(rows), n, k, _p(topk), _p(scores), ld)
        if rc != 0:
            raise RuntimeError("oracle indexer: bad arguments")
        topk = topk[:n]
        return (topk, scores[:n]) if with_scores else topk

    # -- conversion and schedule -------------------------------------------
    def convert(self, logical, req_id_per_token, block_table, block_size: int = BLOCK,
                block_stride_rows: int = 0):
        lg = _c(logical, np.int32)
        T, k = lg.shape
        bt = _c(block_table, np.int32)
        phys = np.zeros_like(lg)
        valid = np.zeros(max(T, 1), np.int32)
        self._lib.ora_convert(_p(lg), T, k, _p(_c(req_id_per_token, np.int32)), _p(bt),
                              int(bt.shape[1]), int(block_size), int(block_stride_rows),
                              _p(phys), _p(valid))
        return phys, valid[:T]

    def schedule(self, n_layers: int, use_index_cache: bool = True, freq: int = 1,
                 offset: int = 2, pattern: str | None = None):
        """Returns (fs string, producer int32 array); raises ValueError if invalid."""
        fs = np.zeros(max(n_layers, 1), np.uint8)
        prod = np.zeros(max(n_layers, 1), np.int32)
        rc = self._lib.ora_schedule(int(n_layers), int(bool(use_index_cache)), int(freq),
                                    int(offset), None if pattern is None else pattern.encode(),
                                    _p(fs), _p(prod))
        if rc != 0:
            raise ValueError("invalid IndexCache schedule")
        return bytes(fs[:n_layers]).decode(), prod[:n_layers].copy()


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from this package's ``dsa_oracle.c``."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle()
    return _default


def __getattr__(name):
    # module-level access to the default oracle's entry points: oracle.indexer(...)
    if name.startswith("__"):
        raise AttributeError(name)
    return getattr(get(), name)
