"""FP8 E4M3 indexer keys with a per-row fp32 scale (the quantised indexer cache).

The pages pass the indexer cache as a key pool plus a per-row scale pool
("Fix: complete DeepSeek V4 TP CSA decode", PR description); the element
format (OCP FP8 E4M3) is this library's reading.  A key row is
scale[row] * e4m3(bytes) and the score formula is unchanged.

CPU: the host checks of the C ABI (the oracle's pins are in
test_fp8_oracle_pins.py).
GPU: indexer scores, Top-K and outputs against the oracle, at small sizes
with poisoned gap rows and at the full long-context size in the launch
configuration the benchmark times, and the allocation-free entry.
"""
import ctypes
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_indexer_gb300 import build as csa_build
from compressed_sparse_attention_indexer_gb300 import csa
from compressed_sparse_attention_indexer_gb300.workloads import (
    BF16_CFG, WORKLOADS, Workload, make_batch, to_device)
from helpers import TOL_BF16, TOL_LSE_BF16, assert_close, assert_topk_sets

FP8_CFG = replace(BF16_CFG, idx_dtype="fp8")
DEV = "cuda:0"


# ---------------------------------------------------------------------------
# CPU: host checks of the C ABI

def _cfg(**kw):
    base = dict(heads=64, row_dim=576, v_dim=512, idx_heads=64, idx_dim=128, ratio=4, topk=512,
                win=128, hca_ratio=0, dtype=csa.CSA_DTYPE_BF16, softmax_scale=0.0,
                rope_base=10000.0, max_batch=4, max_queries_per_req=1, max_context=8192,
                idx_dtype=csa.CSA_DTYPE_FP8_E4M3)
    base.update(kw)
    return csa.CConfig(**base)


def _batch(**kw):
    a = 0x10000  # any 16-byte aligned value: the host checks dereference nothing
    base = dict(B=2, S=1, ctx_len=a, ctx_len_host=None, q=a, q_idx=a, w=a,
                raw_kv=a, raw_off=a, raw_stride=576, raw_rows=10,
                cmp_kv=a, cmp_off=a, cmp_stride=576, cmp_rows=10,
                idx_k=a, idx_off=a, idx_stride=128, idx_rows=10,
                hca_kv=None, hca_off=None, hca_stride=0, hca_rows=0, idx_scale=a)
    base.update(kw)
    return csa.CBatch(**base)


@pytest.fixture(scope="module")
def L():
    csa_build.build()
    return csa.lib()


def check(cfg, b):
    return csa.lib().csa_check_batch(ctypes.byref(cfg), ctypes.byref(b))


def test_fp8_batch_passes_the_host_checks(L):
    assert check(_cfg(), _batch()) == csa.CSA_OK
    assert check(_cfg(), _batch(idx_stride=144)) == csa.CSA_OK   # 144 bytes: 16-byte multiple


@pytest.mark.parametrize("cfg_kw,batch_kw,code", [
    (dict(dtype=csa.CSA_DTYPE_F32), {}, csa.CSA_ERR_UNSUPPORTED),      # FP8 keys need bf16
    (dict(idx_heads=32), {}, csa.CSA_ERR_UNSUPPORTED),                 # and the 64 x 128 indexer
    (dict(idx_dim=64), {}, csa.CSA_ERR_UNSUPPORTED),
    (dict(idx_dtype=7), {}, csa.CSA_ERR_UNSUPPORTED),                  # no such key format
    ({}, dict(idx_scale=None), csa.CSA_ERR_INVALID_ARG),               # the scales are required
    ({}, dict(idx_scale=0x10004), csa.CSA_ERR_INVALID_ARG),            # misaligned scales
    ({}, dict(idx_stride=136), csa.CSA_ERR_INVALID_ARG),               # 136 bytes: not 16-aligned
    ({}, dict(idx_stride=120), csa.CSA_ERR_INVALID_ARG),               # below the row width
])
def test_fp8_host_check_codes(L, cfg_kw, batch_kw, code):
    assert check(_cfg(**cfg_kw), _batch(**batch_kw)) == code
    assert csa.last_error()


def test_fp8_keys_take_prefill_chunks(L):
    # a request's queries beyond what the tcgen05 indexer holds at once are
    # split into query groups, so FP8 keys take any queries per request
    assert check(_cfg(max_queries_per_req=512), _batch(S=512)) == csa.CSA_OK
    assert check(_cfg(max_queries_per_req=13), _batch(S=13)) == csa.CSA_OK


def test_bf16_keys_ignore_the_scale_pointer(L):
    assert check(_cfg(idx_dtype=0), _batch(idx_scale=None, idx_stride=128)) == csa.CSA_OK


# ---------------------------------------------------------------------------
# GPU parity

def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    csa_build.build()
    oracle.build()
    torch.cuda.set_device(0)


def _run_step(wl, hb, max_context=None, host_lens=False):
    cfg = wl.cfg
    db = to_device(hb, DEV)
    B, S = hb["B"], hb["S"]
    dec = csa.Decoder(cfg, B, S, max_context or max(int(hb["ctx_len"].max()), 4))
    out = torch.full((B, S, cfg.H, cfg.V), float("nan"), dtype=cfg.torch_dtype, device=DEV)
    lse = torch.full((B, S, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
    idx = torch.full((B, S, cfg.topk), -7, dtype=torch.int32, device=DEV)
    cnt = torch.full((B, S), -7, dtype=torch.int32, device=DEV)
    lh = hb["ctx_len"].clone() if host_lens else None
    cb = csa.make_batch_struct(db, lh)
    dec.decode_step(cb, out, lse, idx, cnt)
    st = dec.status()
    nq = B * S
    return dict(dec=dec, db=db, cb=cb, lh=lh, status=st,
                out=out.float().cpu().numpy().reshape(nq, cfg.H, cfg.V),
                lse=lse.cpu().numpy().reshape(nq, cfg.H),
                idx=idx.cpu().numpy().reshape(nq, cfg.topk), cnt=cnt.cpu().numpy().reshape(nq))


def _check(wl, hb, g, ref=None, what=""):
    cfg = wl.cfg
    ref = ref if ref is not None else oracle.decode(cfg, hb)
    assert g["status"] == csa.CSA_OK, csa.last_error()
    S = hb["S"]
    assert_topk_sets(g["idx"], g["cnt"], ref, lambda q: oracle.query_scores(cfg, hb, q // S, q % S),
                     cfg.topk, what)
    assert_close(g["out"], ref["out"], TOL_BF16, what + " out")
    assert_close(g["lse"], ref["lse"], TOL_LSE_BF16, what + " lse")
    return ref


@pytest.mark.gpu
@pytest.mark.parametrize("signs", [False, True])
def test_fp8_indexer_scores_against_oracle(signs):
    # signs: every third row's scale negated and every seventh row's zero, so
    # that the kernel's per-dot-product scaling (a scale that is not
    # positive cannot be moved out of the ReLU) is checked beside the
    # factored one
    _gpu()
    wl = Workload("fp8-scores", FP8_CFG, B=4, S=1, L=1, seed=33)
    hb = make_batch(wl, lens=[8192, 300, 1029, 4097], gap_rows=2)
    if signs:
        sc_ = hb["idx_scale"].clone()
        sc_[::3] = -sc_[::3]
        sc_[::7] = 0.0
        hb["idx_scale"] = sc_
    db = to_device(hb, DEV)
    dec = csa.Decoder(FP8_CFG, 4, 1, 8192)
    ld = 8192 // 4
    scores = torch.full((4, ld), float("nan"), dtype=torch.float32, device=DEV)
    dec.indexer_scores(csa.make_batch_struct(db), scores, score_all=True)
    assert dec.status() == csa.CSA_OK
    sc = scores.cpu().numpy()
    qi = hb["q_idx"].double().numpy()
    w = hb["w"].double().numpy()
    codes = hb["idx_k"].view(torch.float8_e4m3fn).to(torch.float64).numpy()
    scale = hb["idx_scale"].double().numpy()
    for q in range(4):
        ref = oracle.query_scores(FP8_CFG, hb, q, 0)
        n = len(ref)
        got = sc[q, :n]
        assert np.isnan(sc[q, n:]).all(), "entries past vis must stay untouched"
        # error bound of fp32 accumulation: relative to
        # sum_h w_h sum_d |q_hd| |scale_j code_jd|
        off = int(hb["idx_off"][q])
        k = np.abs(codes[off:off + n]) * np.abs(scale[off:off + n])[:, None]
        mag = k @ np.abs(qi[q, 0]).T @ w[q, 0]
        bound = 2e-6 * mag + 1e-30
        assert (np.abs(got - ref) <= bound).all(), \
            f"q{q}: max err {np.abs(got - ref).max():.3e}, ratio {(np.abs(got - ref) / bound).max():.2f}"


@pytest.mark.gpu
@pytest.mark.parametrize("host_lens", [False, True])
def test_fp8_decode_step_small_with_poisoned_gaps(host_lens):
    _gpu()
    # bypass (vis <= K), just above K, ragged tails, several items per request;
    # NaN codes between requests poison any row read out of range
    lens = [1000, 2052, 2049, 9000, 5003, 130, 16384]
    wl = Workload("fp8-small", FP8_CFG, B=len(lens), S=1, L=1, seed=34)
    hb = make_batch(wl, lens=lens, gap_rows=2)
    g = _run_step(wl, hb, max_context=16384, host_lens=host_lens)
    _check(wl, hb, g, what=f"fp8 small host_lens={host_lens}")


@pytest.mark.gpu
def test_fp8_workload_full_size_in_the_benchmarked_configuration():
    _gpu()
    wl = WORKLOADS["long_ragged_b64_fp8idx"]
    hb = make_batch(wl)
    g = _run_step(wl, hb, max_context=65536, host_lens=True)
    ref = _check(wl, hb, g, what="long_ragged_b64_fp8idx")
    g2 = _run_step(wl, hb, max_context=65536, host_lens=False)
    _check(wl, hb, g2, ref=ref, what="long_ragged_b64_fp8idx device lengths")


@pytest.mark.gpu
def test_fp8_allocation_free_entry_matches_the_handle():
    _gpu()
    lens = [8192, 2049, 300, 5000]
    wl = Workload("fp8-static", FP8_CFG, B=len(lens), S=1, L=1, seed=35)
    hb = make_batch(wl, lens=lens, gap_rows=2)
    db = to_device(hb, DEV)
    dec = csa.Decoder(FP8_CFG, len(lens), 1, 8192)
    lh = hb["ctx_len"].clone()
    cb = csa.make_batch_struct(db, lh)
    ref_idx = torch.full((len(lens), 1, 512), -7, dtype=torch.int32, device=DEV)
    ref_cnt = torch.full((len(lens), 1), -7, dtype=torch.int32, device=DEV)
    dec.indexer_topk(cb, ref_idx, ref_cnt)
    assert dec.status() == csa.CSA_OK
    idx = torch.full_like(ref_idx, -9)
    cnt = torch.full_like(ref_cnt, -9)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    csa.indexer_topk_static(dec.cconfig, cb, idx, cnt, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(idx, ref_idx) and torch.equal(cnt, ref_cnt)
