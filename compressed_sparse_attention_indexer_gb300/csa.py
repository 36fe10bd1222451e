"""ctypes binding of libcsa (include/csa.h): argument marshalling only.

Every step of the decode path runs in the CUDA library; this module turns
torch device tensors into the C structs and pointers the entry points take,
and raises on a non-zero return code.  If the library has not been built,
the first call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

CSA_OK, CSA_ERR_INVALID_ARG, CSA_ERR_UNSUPPORTED, CSA_ERR_WORKSPACE = 0, 1, 2, 3
CSA_ERR_CUDA, CSA_ERR_BAD_INDEX, CSA_ERR_TIMEOUT = 4, 5, 6
CSA_DTYPE_F32, CSA_DTYPE_BF16, CSA_DTYPE_FP8_E4M3 = 0, 1, 2
ERROR_NAMES = {0: "CSA_OK", 1: "CSA_ERR_INVALID_ARG", 2: "CSA_ERR_UNSUPPORTED", 3: "CSA_ERR_WORKSPACE",
               4: "CSA_ERR_CUDA", 5: "CSA_ERR_BAD_INDEX", 6: "CSA_ERR_TIMEOUT"}

EXPORTS = ("csa_decode_create", "csa_decode_destroy", "csa_indexer_topk", "csa_sparse_attn",
           "csa_decode_step", "csa_indexer_scores", "csa_topk_select", "csa_check_batch",
           "csa_get_status", "csa_last_error", "csa_last_launch_count", "csa_abi_version",
           "csa_profile_enable", "csa_profile_read", "csa_indexer_topk_static", "csa_cache_writeback",
           "csa_debug_set_wait_polls")
STAGES = ("plan", "indexer", "topk", "attention")


class CsaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


class CConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("heads", "row_dim", "v_dim", "idx_heads", "idx_dim", "ratio", "topk", "win",
                 "hca_ratio", "dtype")] + [
        ("softmax_scale", ctypes.c_float), ("rope_base", ctypes.c_float),
        ("max_batch", ctypes.c_int32), ("max_queries_per_req", ctypes.c_int32),
        ("max_context", ctypes.c_int32), ("idx_dtype", ctypes.c_int32)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64


class CBatch(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("S", ctypes.c_int32), ("ctx_len", _P), ("ctx_len_host", _P),
                ("q", _P), ("q_idx", _P), ("w", _P),
                ("raw_kv", _P), ("raw_off", _P), ("raw_stride", _I64), ("raw_rows", _I64),
                ("cmp_kv", _P), ("cmp_off", _P), ("cmp_stride", _I64), ("cmp_rows", _I64),
                ("idx_k", _P), ("idx_off", _P), ("idx_stride", _I64), ("idx_rows", _I64),
                ("hca_kv", _P), ("hca_off", _P), ("hca_stride", _I64), ("hca_rows", _I64),
                ("idx_scale", _P),
                ("raw_table", _P), ("cmp_table", _P), ("idx_table", _P), ("hca_table", _P),
                ("raw_block", ctypes.c_int32), ("cmp_block", ctypes.c_int32),
                ("idx_block", ctypes.c_int32), ("hca_block", ctypes.c_int32),
                ("table_stride", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def lib(path: str | None = None):
    """Loads libcsa; raises if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or os.environ.get("CSA_LIB") or _build.LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libcsa is not built ({p} missing): run "
                                   "compressed_sparse_attention_indexer_gb300.build.build()")
            L = ctypes.CDLL(p)
            i32, vp = ctypes.c_int32, ctypes.c_void_p
            H = ctypes.c_void_p
            L.csa_decode_create.argtypes = [ctypes.POINTER(CConfig), ctypes.POINTER(H)]
            L.csa_decode_destroy.argtypes = [H]
            L.csa_decode_destroy.restype = None
            L.csa_indexer_topk.argtypes = [H, ctypes.POINTER(CBatch), vp, vp, vp]
            L.csa_sparse_attn.argtypes = [H, ctypes.POINTER(CBatch), vp, vp, vp, vp, vp]
            L.csa_decode_step.argtypes = [H, ctypes.POINTER(CBatch), vp, vp, vp, vp, vp]
            L.csa_indexer_scores.argtypes = [H, ctypes.POINTER(CBatch), vp, ctypes.c_int64, i32, vp]
            L.csa_topk_select.argtypes = [H, i32, vp, ctypes.c_int64, vp, vp, vp, vp]
            L.csa_check_batch.argtypes = [ctypes.POINTER(CConfig), ctypes.POINTER(CBatch)]
            L.csa_get_status.argtypes = [H, vp]
            L.csa_last_error.restype = ctypes.c_char_p
            L.csa_last_launch_count.argtypes = [H]
            L.csa_last_launch_count.restype = i32
            L.csa_abi_version.restype = i32
            L.csa_profile_enable.argtypes = [H, i32]
            L.csa_profile_read.argtypes = [H, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(i32)]
            L.csa_debug_set_wait_polls.argtypes = [H, i32]
            L.csa_indexer_topk_static.argtypes = [ctypes.POINTER(CConfig), ctypes.POINTER(CBatch), vp,
                                                  vp, vp, vp]
            L.csa_cache_writeback.argtypes = [vp, ctypes.c_int64, vp, i32, vp, ctypes.c_int64,
                                              ctypes.c_int64, ctypes.c_int64, vp, vp]
            for name in ("csa_decode_create", "csa_indexer_topk", "csa_sparse_attn", "csa_decode_step",
                         "csa_indexer_scores", "csa_topk_select", "csa_check_batch", "csa_get_status",
                         "csa_profile_enable", "csa_profile_read", "csa_indexer_topk_static",
                         "csa_cache_writeback", "csa_debug_set_wait_polls"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def last_error() -> str:
    return lib().csa_last_error().decode()


def _check(rc: int):
    if rc != CSA_OK:
        raise CsaError(rc, last_error())


def make_config(cfg, max_batch: int, max_queries: int, max_context: int) -> CConfig:
    """C config from a workloads.CsaConfig."""
    return CConfig(heads=cfg.H, row_dim=cfg.D, v_dim=cfg.V, idx_heads=cfg.Hi, idx_dim=cfg.Di,
                   ratio=cfg.ratio, topk=cfg.topk, win=cfg.win, hca_ratio=cfg.hca_ratio,
                   dtype=CSA_DTYPE_BF16 if cfg.dtype == "bf16" else CSA_DTYPE_F32,
                   softmax_scale=cfg.softmax_scale, rope_base=cfg.rope_base,
                   max_batch=max_batch, max_queries_per_req=max_queries, max_context=max_context,
                   idx_dtype=CSA_DTYPE_FP8_E4M3 if getattr(cfg, "idx_dtype", "") == "fp8" else 0)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def make_batch_struct(batch: dict, ctx_len_host=None) -> CBatch:
    """C batch from a dict of device tensors (see workloads.make_batch/to_device).

    ctx_len_host: optional int32 CPU tensor with the same lengths (kept alive by
    the caller while the struct is in use)."""
    def rows(t):
        return 0 if t is None else int(t.shape[0])
    return CBatch(
        B=int(batch["B"]), S=int(batch["S"]), ctx_len=_ptr(batch["ctx_len"]),
        ctx_len_host=_ptr(ctx_len_host),
        q=_ptr(batch["q"]), q_idx=_ptr(batch["q_idx"]), w=_ptr(batch["w"]),
        raw_kv=_ptr(batch["raw_kv"]), raw_off=_ptr(batch.get("raw_off")),
        raw_stride=int(batch["raw_stride"]), raw_rows=rows(batch["raw_kv"]),
        cmp_kv=_ptr(batch["cmp_kv"]), cmp_off=_ptr(batch.get("cmp_off")),
        cmp_stride=int(batch["cmp_stride"]), cmp_rows=rows(batch["cmp_kv"]),
        idx_k=_ptr(batch["idx_k"]), idx_off=_ptr(batch.get("idx_off")),
        idx_stride=int(batch["idx_stride"]), idx_rows=rows(batch["idx_k"]),
        hca_kv=_ptr(batch.get("hca_kv")), hca_off=_ptr(batch.get("hca_off")),
        hca_stride=int(batch.get("hca_stride") or 0), hca_rows=rows(batch.get("hca_kv")),
        idx_scale=_ptr(batch.get("idx_scale")),
        raw_table=_ptr(batch.get("raw_table")), cmp_table=_ptr(batch.get("cmp_table")),
        idx_table=_ptr(batch.get("idx_table")), hca_table=_ptr(batch.get("hca_table")),
        raw_block=int(batch.get("raw_block") or 0), cmp_block=int(batch.get("cmp_block") or 0),
        idx_block=int(batch.get("idx_block") or 0), hca_block=int(batch.get("hca_block") or 0),
        table_stride=int(batch.get("table_stride") or 0))


def check_batch(cconfig: CConfig, cbatch: CBatch) -> int:
    """Host-side validation only (no GPU); returns the C return code."""
    return lib().csa_check_batch(ctypes.byref(cconfig), ctypes.byref(cbatch))


def indexer_topk_static(cconfig: CConfig, cb: CBatch, topk_idx, topk_cnt, status=None, stream=None):
    """Steps (a)+(b) without a handle or any device allocation (scratch in the
    library's static device array; see csa_indexer_topk_static in csa.h)."""
    _check(lib().csa_indexer_topk_static(ctypes.byref(cconfig), ctypes.byref(cb), _ptr(topk_idx),
                                         _ptr(topk_cnt), _ptr(status), _stream(stream)))


def cache_writeback(rows, slot, pool, status=None, stream=None):
    """pool[slot[t]] = rows[t] on the device (see csa_cache_writeback in csa.h).

    rows [n, ...] and pool [pool_rows, ...]: device tensors whose rows are
    contiguous and of the same byte size; slot [n] int64 (negative = skip)."""
    n = int(rows.shape[0])
    row_bytes = rows[0].numel() * rows.element_size() if n else 0
    assert n == 0 or pool[0].numel() * pool.element_size() == row_bytes, "row sizes differ"
    _check(lib().csa_cache_writeback(_ptr(rows), int(rows.stride(0)) * rows.element_size(), _ptr(slot),
                                     n, _ptr(pool), int(pool.stride(0)) * pool.element_size(),
                                     int(pool.shape[0]), int(row_bytes), _ptr(status), _stream(stream)))


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(stream) if not hasattr(stream, "cuda_stream") else stream.cuda_stream


class Decoder:
    """One csa_handle: a fixed layer shape plus its device workspace."""

    def __init__(self, cfg, max_batch: int, max_queries: int, max_context: int):
        self.cfg = cfg
        self.cconfig = make_config(cfg, max_batch, max_queries, max_context)
        h = ctypes.c_void_p()
        _check(lib().csa_decode_create(ctypes.byref(self.cconfig), ctypes.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            lib().csa_decode_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- entry points (tensors must be on the current device) --------------
    def decode_step(self, cb: CBatch, out, lse=None, topk_idx=None, topk_cnt=None, stream=None):
        _check(lib().csa_decode_step(self.handle, ctypes.byref(cb), _ptr(out), _ptr(lse),
                                     _ptr(topk_idx), _ptr(topk_cnt), _stream(stream)))

    def indexer_topk(self, cb: CBatch, topk_idx, topk_cnt, stream=None):
        _check(lib().csa_indexer_topk(self.handle, ctypes.byref(cb), _ptr(topk_idx), _ptr(topk_cnt),
                                      _stream(stream)))

    def sparse_attn(self, cb: CBatch, topk_idx, topk_cnt, out, lse=None, stream=None):
        _check(lib().csa_sparse_attn(self.handle, ctypes.byref(cb), _ptr(topk_idx), _ptr(topk_cnt),
                                     _ptr(out), _ptr(lse), _stream(stream)))

    def indexer_scores(self, cb: CBatch, scores, score_all: bool = True, stream=None):
        _check(lib().csa_indexer_scores(self.handle, ctypes.byref(cb), _ptr(scores),
                                        int(scores.stride(0)), 1 if score_all else 0, _stream(stream)))

    def topk_select(self, scores, n, topk_idx, topk_cnt, stream=None):
        _check(lib().csa_topk_select(self.handle, int(scores.shape[0]), _ptr(scores),
                                     int(scores.stride(0)), _ptr(n), _ptr(topk_idx), _ptr(topk_cnt),
                                     _stream(stream)))

    def status(self, stream=None) -> int:
        """Synchronises and returns (and clears) the device status code."""
        return lib().csa_get_status(self.handle, _stream(stream))

    def last_launch_count(self) -> int:
        return lib().csa_last_launch_count(self.handle)

    def debug_wait_polls(self, polls: int):
        """Test hook: the attention tile kernel's consumer waits give up after
        `polls` polls (0: at once); negative restores the default."""
        _check(lib().csa_debug_set_wait_polls(self.handle, int(polls)))

    def profile(self, enable: bool):
        _check(lib().csa_profile_enable(self.handle, 1 if enable else 0))

    def profile_read(self) -> dict:
        """{stage: (milliseconds, launches)} since the last read."""
        ms = (ctypes.c_float * 4)()
        n = (ctypes.c_int32 * 4)()
        _check(lib().csa_profile_read(self.handle, ms, n))
        return {STAGES[i]: (float(ms[i]), int(n[i])) for i in range(4)}
