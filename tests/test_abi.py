"""The C ABI without a GPU: the library loads, exports every declared symbol,
and its host-side checks return the documented codes before any launch."""
import ctypes
import os
import re

import pytest
import torch

from compressed_sparse_attention_indexer_gb300 import build as csa_build
from compressed_sparse_attention_indexer_gb300 import csa
from compressed_sparse_attention_indexer_gb300.workloads import WORKLOADS, CsaConfig

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    csa_build.build()
    return csa.lib()


def declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "csa.h")).read()
    return sorted(set(re.findall(r"CSA_API\s+[\w\s\*]*?\b(csa_\w+)\s*\(", hdr)))


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), f"{n} declared in csa.h but not exported"
    assert set(names) == set(csa.EXPORTS)
    assert L.csa_abi_version() == 3


def _cfg(**kw):
    base = dict(heads=64, row_dim=576, v_dim=512, idx_heads=64, idx_dim=128, ratio=4, topk=512,
                win=128, hca_ratio=0, dtype=csa.CSA_DTYPE_BF16, softmax_scale=0.0,
                rope_base=10000.0, max_batch=4, max_queries_per_req=1, max_context=8192)
    base.update(kw)
    return csa.CConfig(**base)


def _batch(**kw):
    a = 0x10000  # any 16-byte aligned value: nothing is dereferenced by the checks
    base = dict(B=2, S=1, ctx_len=a, ctx_len_host=None, q=a, q_idx=a, w=a,
                raw_kv=a, raw_off=a, raw_stride=576, raw_rows=10,
                cmp_kv=a, cmp_off=a, cmp_stride=576, cmp_rows=10,
                idx_k=a, idx_off=a, idx_stride=128, idx_rows=10,
                hca_kv=None, hca_off=None, hca_stride=0, hca_rows=0)
    base.update(kw)
    return csa.CBatch(**base)


def check(cfg, b):
    return csa.lib().csa_check_batch(ctypes.byref(cfg), ctypes.byref(b))


def test_valid_batch_passes(L):
    assert check(_cfg(), _batch()) == csa.CSA_OK
    assert check(_cfg(), _batch(B=0)) == csa.CSA_OK   # empty batch: a no-op


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), csa.CSA_ERR_INVALID_ARG),
    (dict(ctx_len=None), csa.CSA_ERR_INVALID_ARG),
    (dict(q_idx=0x10008), csa.CSA_ERR_INVALID_ARG),          # misaligned
    (dict(raw_stride=500), csa.CSA_ERR_INVALID_ARG),          # below row width
    (dict(cmp_stride=580), csa.CSA_ERR_INVALID_ARG),          # 1160 B: not a multiple of 16
    (dict(idx_rows=-1), csa.CSA_ERR_INVALID_ARG),
    (dict(B=5), csa.CSA_ERR_WORKSPACE),                       # above max_batch
    (dict(S=2), csa.CSA_ERR_WORKSPACE),                       # above max_queries_per_req
    (dict(B=-1), csa.CSA_ERR_INVALID_ARG),
    (dict(S=0), csa.CSA_ERR_INVALID_ARG),
])
def test_bad_batch_codes(L, kw, code):
    assert check(_cfg(), _batch(**kw)) == code
    assert csa.last_error()


def test_host_lengths_checked(L):
    lens = (ctypes.c_int32 * 2)(100, 8193)   # 8193 > max_context
    assert check(_cfg(), _batch(ctx_len_host=ctypes.addressof(lens))) == csa.CSA_ERR_WORKSPACE
    lens2 = (ctypes.c_int32 * 2)(100, 0)     # below S
    assert check(_cfg(), _batch(ctx_len_host=ctypes.addressof(lens2))) == csa.CSA_ERR_WORKSPACE
    lens3 = (ctypes.c_int32 * 2)(1, 8192)
    assert check(_cfg(), _batch(ctx_len_host=ctypes.addressof(lens3))) == csa.CSA_OK


def test_hca_pool_required_when_enabled(L):
    assert check(_cfg(hca_ratio=128), _batch()) == csa.CSA_ERR_INVALID_ARG
    assert check(_cfg(hca_ratio=128), _batch(hca_kv=0x10000, hca_off=0x10000, hca_stride=576,
                                             hca_rows=4)) == csa.CSA_OK


@pytest.mark.parametrize("kw,code", [
    (dict(heads=0), csa.CSA_ERR_INVALID_ARG),
    (dict(v_dim=600), csa.CSA_ERR_INVALID_ARG),
    (dict(v_dim=511), csa.CSA_ERR_INVALID_ARG),               # odd rope width
    (dict(dtype=7), csa.CSA_ERR_UNSUPPORTED),
    (dict(topk=0), csa.CSA_ERR_INVALID_ARG),
    (dict(win=0), csa.CSA_ERR_INVALID_ARG),
    (dict(max_context=4 * 40961), csa.CSA_ERR_UNSUPPORTED),   # Top-K keys exceed shared memory
    (dict(rope_base=0.0), csa.CSA_ERR_INVALID_ARG),
])
def test_bad_config_codes(L, kw, code):
    assert check(_cfg(**kw), _batch()) == code


def test_create_rejects_bad_config_without_touching_the_gpu(L):
    h = ctypes.c_void_p()
    cfg = _cfg(heads=0)
    assert L.csa_decode_create(ctypes.byref(cfg), ctypes.byref(h)) == csa.CSA_ERR_INVALID_ARG
    assert h.value is None
    assert L.csa_decode_create(None, ctypes.byref(h)) == csa.CSA_ERR_INVALID_ARG
    # entry points refuse a NULL handle before any CUDA call
    assert L.csa_decode_step(None, None, None, None, None, None, None) == csa.CSA_ERR_INVALID_ARG
    assert L.csa_get_status(None, None) == csa.CSA_ERR_INVALID_ARG
    L.csa_decode_destroy(None)


def test_workload_configs_map_onto_the_abi():
    for name, wl in WORKLOADS.items():
        c = csa.make_config(wl.cfg, 64, 8, 65536)
        assert c.heads == wl.cfg.H and c.row_dim == wl.cfg.D and c.v_dim == wl.cfg.V
        assert abs(c.softmax_scale - wl.cfg.softmax_scale) < 1e-7


def test_product_path_has_no_oracle_dependency():
    # the CUDA package must not import, load or name the oracle
    pkg = os.path.join(ROOT, "compressed_sparse_attention_indexer_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, f
                assert "csa_oracle" not in txt, f


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(csa, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        csa.lib(str(tmp_path / "nope.so"))
    monkeypatch.setattr(csa, "_lib", None)
