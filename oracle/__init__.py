"""CPU oracle for the CSA decode step: plain fp64 C, loaded with ctypes.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The CUDA library never
links or calls it, and it imports nothing from the CUDA package.

The C source (``csa_oracle.c``) follows the method step by step: indexer
score, full-sort Top-K (or the bypass), the gathered rows, one softmax over
their union, inverse RoPE.  See its header for the page citations and the
readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, f"libcsa_oracle_{platform.machine()}.so")
_lib = None
_lock = threading.Lock()

ORC_F32, ORC_BF16, ORC_FP8_E4M3 = 0, 1, 2
FORCE_SCORE = 1


class OrcCfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("H", "D", "V", "Hi", "Di", "ratio", "topk", "win", "hca_ratio", "dtype")] + [
        ("scale", ctypes.c_double), ("rope_base", ctypes.c_double), ("idx_dtype", ctypes.c_int32)]


_P = ctypes.c_void_p


class OrcBatch(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("S", ctypes.c_int32), ("ctx_len", _P),
                ("q", _P), ("q_idx", _P), ("w", _P),
                ("raw", _P), ("raw_off", _P), ("raw_stride", ctypes.c_int64),
                ("cmp", _P), ("cmp_off", _P), ("cmp_stride", ctypes.c_int64),
                ("idx", _P), ("idx_off", _P), ("idx_stride", ctypes.c_int64),
                ("hca", _P), ("hca_off", _P), ("hca_stride", ctypes.c_int64),
                ("idx_scale", _P),
                ("raw_table", _P), ("cmp_table", _P), ("idx_table", _P), ("hca_table", _P),
                ("raw_block", ctypes.c_int32), ("cmp_block", ctypes.c_int32),
                ("idx_block", ctypes.c_int32), ("hca_block", ctypes.c_int32),
                ("table_stride", ctypes.c_int32)]


class OrcQueryInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("pos", "vis", "nwin", "cnt", "vis2", "rows_used")]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math) if needed."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                        "-ffp-contract=off", "-pthread", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            # CSA_ORACLE_LIB lets the mutation tests load a deliberately broken build
            _lib = ctypes.CDLL(os.environ.get("CSA_ORACLE_LIB") or build())
            d = ctypes.POINTER(ctypes.c_double)
            i32 = ctypes.c_int32
            _lib.orc_index_scores.argtypes = [i32, i32, d, d, i32, d, d]
            _lib.orc_topk.argtypes = [d, i32, i32, ctypes.POINTER(i32)]
            _lib.orc_topk.restype = i32
            _lib.orc_attend.argtypes = [i32, i32, i32, ctypes.c_double, d, i32, d, d, d]
            _lib.orc_inverse_rope.argtypes = [i32, i32, i32, ctypes.c_double, ctypes.c_double, d]
            _lib.orc_decode.argtypes = [ctypes.POINTER(OrcCfg), ctypes.POINTER(OrcBatch),
                                        ctypes.POINTER(i32), i32, i32, i32, d, d,
                                        ctypes.POINTER(i32), ctypes.POINTER(OrcQueryInfo)]
            _lib.orc_decode.restype = ctypes.c_int
            _lib.orc_query_scores.argtypes = [ctypes.POINTER(OrcCfg), ctypes.POINTER(OrcBatch),
                                              i32, i32, d]
            _lib.orc_query_scores.restype = i32
            _lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
            _lib.orc_e4m3_to_double.restype = ctypes.c_double
    return _lib


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


# ---------------------------------------------------------------------------
# single steps (fp64 numpy in, fp64 numpy out)

def index_scores(q_idx, w, k_idx) -> np.ndarray:
    """score_j = sum_h w_h * ReLU(q_idx[h] . k_idx[j]); q_idx [Hi,Di], w [Hi], k_idx [n,Di]."""
    qi, wv, k = _f64(q_idx), _f64(w), _f64(k_idx)
    Hi, Di = qi.shape
    n = k.shape[0]
    out = np.zeros(n, np.float64)
    lib().orc_index_scores(Hi, Di, _dp(qi), _dp(wv), n, _dp(k) if n else _dp(np.zeros(1)), _dp(out))
    return out


def topk(scores, K: int) -> np.ndarray:
    """The min(n,K) best indices by (-score, index), ascending."""
    s = _f64(scores)
    idx = np.full(max(K, 1), -1, np.int32)
    c = lib().orc_topk(_dp(s) if s.size else _dp(np.zeros(1)), s.size, K,
                       idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    return idx[:c].copy()


def attend(q, rows, V: int, scale: float):
    """One softmax over `rows` [n,D] for heads q [H,D]; returns (o [H,V], lse [H])."""
    qv, r = _f64(q), _f64(rows).reshape(-1, np.asarray(q).shape[1])
    H, D = qv.shape
    o = np.zeros((H, V), np.float64)
    lse = np.zeros(H, np.float64)
    lib().orc_attend(H, D, V, float(scale), _dp(qv), r.shape[0],
                     _dp(r) if r.size else _dp(np.zeros(1)), _dp(o), _dp(lse))
    return o, lse


def inverse_rope(o, pos: float, R: int, base: float) -> np.ndarray:
    """Inverse RoPE on the last R of the V output dims of o [H,V]; returns a copy."""
    x = _f64(o).copy()
    H, V = x.shape
    lib().orc_inverse_rope(H, V, R, float(pos), float(base), _dp(x))
    return x


# ---------------------------------------------------------------------------
# whole decode step over a host batch

def _storage(t) -> np.ndarray:
    """Raw storage of a CPU tensor/array as a contiguous numpy array (bf16 -> uint16 bits)."""
    import torch
    if isinstance(t, torch.Tensor):
        t = t.detach().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()
    return np.ascontiguousarray(t)


def make_cfg(cfg) -> OrcCfg:
    """From a workload config object (see the workloads module)."""
    return OrcCfg(H=cfg.H, D=cfg.D, V=cfg.V, Hi=cfg.Hi, Di=cfg.Di, ratio=cfg.ratio,
                  topk=cfg.topk, win=cfg.win, hca_ratio=cfg.hca_ratio,
                  dtype=ORC_BF16 if cfg.dtype == "bf16" else ORC_F32,
                  scale=cfg.softmax_scale, rope_base=cfg.rope_base,
                  idx_dtype=ORC_FP8_E4M3 if getattr(cfg, "idx_dtype", "") == "fp8" else 0)


class _HostBatch:
    """Keeps the numpy views alive while the C struct points into them."""

    def __init__(self, batch: dict):
        self.arrs = {}

        def keep(name, dtype=None):
            v = batch.get(name)
            if v is None:
                return None
            a = _storage(v)
            if dtype is not None:
                a = np.ascontiguousarray(a.astype(dtype, copy=False))
            self.arrs[name] = a
            return a.ctypes.data

        self.c = OrcBatch(
            B=int(batch["B"]), S=int(batch["S"]), ctx_len=keep("ctx_len", np.int32),
            q=keep("q"), q_idx=keep("q_idx"), w=keep("w", np.float32),
            raw=keep("raw_kv"), raw_off=keep("raw_off", np.int64), raw_stride=int(batch["raw_stride"]),
            cmp=keep("cmp_kv"), cmp_off=keep("cmp_off", np.int64), cmp_stride=int(batch["cmp_stride"]),
            idx=keep("idx_k"), idx_off=keep("idx_off", np.int64), idx_stride=int(batch["idx_stride"]),
            hca=keep("hca_kv"), hca_off=keep("hca_off", np.int64),
            hca_stride=int(batch.get("hca_stride", 0) or 0),
            idx_scale=keep("idx_scale", np.float32),
            raw_table=keep("raw_table", np.int32), cmp_table=keep("cmp_table", np.int32),
            idx_table=keep("idx_table", np.int32), hca_table=keep("hca_table", np.int32),
            raw_block=int(batch.get("raw_block") or 0), cmp_block=int(batch.get("cmp_block") or 0),
            idx_block=int(batch.get("idx_block") or 0), hca_block=int(batch.get("hca_block") or 0),
            table_stride=int(batch.get("table_stride") or 0))


def decode(cfg, batch: dict, qids=None, nthreads: int | None = None, force_score: bool = False):
    """Runs the oracle over queries `qids` (flattened b*S+s; default all).

    Returns dict: out [nq,H,V] (after inverse RoPE), lse [nq,H], topk_idx [nq,K]
    (ascending, -1 padded), and per-query pos/vis/nwin/cnt/vis2/rows_used.
    """
    hb = _HostBatch(batch)
    c = make_cfg(cfg)
    nq_all = int(batch["B"]) * int(batch["S"])
    q = np.arange(nq_all, dtype=np.int32) if qids is None else np.ascontiguousarray(qids, dtype=np.int32)
    nq = q.size
    out = np.zeros((nq, cfg.H, cfg.V), np.float64)
    lse = np.zeros((nq, cfg.H), np.float64)
    idx = np.full((nq, cfg.topk), -1, np.int32)
    info = (OrcQueryInfo * max(nq, 1))()
    nthreads = nthreads or os.cpu_count() or 1
    rc = lib().orc_decode(ctypes.byref(c), ctypes.byref(hb.c),
                          q.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), nq,
                          FORCE_SCORE if force_score else 0, nthreads, _dp(out), _dp(lse),
                          idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), info)
    if rc == -2:
        raise ValueError("oracle: a row a query needs lies in an unmapped block of a paged pool")
    if rc != 0:
        raise ValueError("oracle: a query has pos < 0 (ctx_len < S)")
    res = {"out": out, "lse": lse, "topk_idx": idx, "qids": q}
    for f in ("pos", "vis", "nwin", "cnt", "vis2", "rows_used"):
        res[f] = np.array([getattr(info[i], f) for i in range(nq)], np.int64)
    return res


def cache_writeback(pool: np.ndarray, rows: np.ndarray, slot) -> tuple[np.ndarray, bool]:
    """The cache update before a step ("Perf: parallelize the DSpark TP-4 SWA
    decode hot tasks", PR description: the KV scatter by slot mapping commits
    every mapping entry): a copy of `pool` in which row slot[t] holds rows[t]
    for every t with 0 <= slot[t] < len(pool), token order.  A negative slot
    is a padding token; a slot past the pool is skipped and reported (the
    returned flag).  Works on raw bytes, so any element type behaves alike."""
    out = np.array(pool, copy=True)
    bad = False
    for t, s in enumerate(np.asarray(slot).tolist()):
        if s < 0:
            continue
        if s >= out.shape[0]:
            bad = True
            continue
        out[s] = rows[t]
    return out, bad


def e4m3_value(byte: int) -> float:
    """The value of one OCP FP8 E4M3 byte (as the indexer-key pool stores it)."""
    return float(lib().orc_e4m3_to_double(int(byte) & 0xFF))


def query_scores(cfg, batch: dict, b: int, s: int) -> np.ndarray:
    """fp64 indexer scores of every visible compressed row of query (b, s)."""
    hb = _HostBatch(batch)
    c = make_cfg(cfg)
    pos = int(_storage(batch["ctx_len"])[b]) - int(batch["S"]) + s
    vis = (pos + 1) // cfg.ratio
    out = np.zeros(max(vis, 1), np.float64)
    n = lib().orc_query_scores(ctypes.byref(c), ctypes.byref(hb.c), b, s, _dp(out))
    if n < 0:
        raise ValueError("oracle: a key row lies in an unmapped block of a paged pool")
    return out[:n]
