"""Prefill chunks on the indexer: a request of S new tokens, each token scoring
its own causally visible compressed rows.

The pages' prefill runs the same indexer over a chunk of new tokens
(hw-native-sys/pypto-lib "Fix: port the DeepSeek-V4 MoE, hc_pre and prefill
fixes to DSpark"); query s of a request of context length L sits at position
L - S + s and sees floor((L - S + s + 1) / ratio) compressed rows.  A
request whose queries do not fit the indexer kernel at once has its work split
into (query group, key chunk) items: groups of 4 queries on the tcgen05
kernel (bf16 and FP8 keys), of 8 on the warp-MMA kernel.  These tests cross
the group boundaries (S = 10, 13: a ragged last group), mix requests with
no, few and many visible rows, build the work list both on the host (host
lengths) and on the device, and compare every score with the fp64 oracle.
"""
import os
import subprocess
import sys
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_indexer_gb300 import build as csa_build
from compressed_sparse_attention_indexer_gb300 import csa
from compressed_sparse_attention_indexer_gb300.workloads import (
    BF16_CFG, Workload, make_batch, to_device)
from helpers import TOL_BF16, TOL_LSE_BF16, assert_close, assert_topk_sets

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FP8_CFG = replace(BF16_CFG, idx_dtype="fp8")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    csa_build.build()
    oracle.build()
    torch.cuda.set_device(0)


def check_prefill_scores(cfg, S, lens, seed, host_lens):
    """Every score of every query of the batch against the oracle, within the
    fp32 accumulation bound; entries past a query's visible rows untouched."""
    wl = Workload("prefill-scores", cfg, B=len(lens), S=S, L=1, seed=seed)
    hb = make_batch(wl, lens=lens, gap_rows=2)
    db = to_device(hb, DEV)
    B = len(lens)
    mc = max(lens)
    dec = csa.Decoder(cfg, B, S, mc)
    ld = mc // cfg.ratio
    scores = torch.full((B * S, ld), float("nan"), dtype=torch.float32, device=DEV)
    lh = hb["ctx_len"].clone() if host_lens else None
    dec.indexer_scores(csa.make_batch_struct(db, lh), scores, score_all=True)
    assert dec.status() == csa.CSA_OK, csa.last_error()
    sc = scores.cpu().numpy()
    qi = hb["q_idx"].double().numpy()
    w = hb["w"].double().numpy()
    if cfg.idx_dtype == "fp8":
        keys = (hb["idx_k"].view(torch.float8_e4m3fn).to(torch.float64)
                * hb["idx_scale"].double()[:, None]).numpy()
    else:
        keys = hb["idx_k"].double().numpy()
    for q in range(B * S):
        b, s = divmod(q, S)
        ref = oracle.query_scores(cfg, hb, b, s)
        n = len(ref)
        assert n == (lens[b] - S + s + 1) // cfg.ratio
        got = sc[q, :n]
        assert np.isnan(sc[q, n:]).all(), f"q{q}: entries past vis must stay untouched"
        off = int(hb["idx_off"][b])
        mag = np.abs(keys[off:off + n]) @ np.abs(qi[b, s]).T @ w[b, s]
        bound = 2e-6 * mag + 1e-30
        assert (np.abs(got - ref) <= bound).all(), \
            f"q{q}: max err {np.abs(got - ref).max():.3e}, ratio {(np.abs(got - ref) / bound).max():.2f}"


# S = 13: groups 4, 4, 4, 1; L = 13: queries with 0 .. 3 visible rows; the
# longest request spans several key chunks with a ragged last one
@pytest.mark.parametrize("host_lens", [False, True])
def test_bf16_prefill_scores_split_by_query_group(host_lens):
    check_prefill_scores(BF16_CFG, 13, [13, 600, 4109, 2100], seed=71, host_lens=host_lens)


@pytest.mark.parametrize("host_lens", [False, True])
def test_fp8_prefill_scores_split_by_query_group(host_lens):
    # S = 10: groups 4, 4, 2 (above the queries the FP8 kernel holds at once)
    check_prefill_scores(FP8_CFG, 10, [2000, 5003, 10], seed=72, host_lens=host_lens)


def test_bf16_prefill_scores_wide_chunk():
    check_prefill_scores(BF16_CFG, 64, [2305, 64, 9000], seed=73, host_lens=True)


def test_fp8_prefill_decode_step():
    # the whole step with FP8 keys on a 16-token chunk: Top-K sets and outputs
    lens = [3000, 700, 2070]
    S = 16
    wl = Workload("fp8-prefill", FP8_CFG, B=len(lens), S=S, L=1, seed=74)
    hb = make_batch(wl, lens=lens, gap_rows=2)
    db = to_device(hb, DEV)
    B = len(lens)
    cfg = FP8_CFG
    dec = csa.Decoder(cfg, B, S, max(lens))
    out = torch.full((B, S, cfg.H, cfg.V), float("nan"), dtype=cfg.torch_dtype, device=DEV)
    lse = torch.full((B, S, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
    idx = torch.full((B, S, cfg.topk), -7, dtype=torch.int32, device=DEV)
    cnt = torch.full((B, S), -7, dtype=torch.int32, device=DEV)
    lh = hb["ctx_len"].clone()  # the struct holds a raw pointer: keep the tensor alive
    dec.decode_step(csa.make_batch_struct(db, lh), out, lse, idx, cnt)
    assert dec.status() == csa.CSA_OK, csa.last_error()
    ref = oracle.decode(cfg, hb)
    nq = B * S
    assert_topk_sets(idx.cpu().numpy().reshape(nq, -1), cnt.cpu().numpy().reshape(nq), ref,
                     lambda q: oracle.query_scores(cfg, hb, q // S, q % S), cfg.topk, "fp8 prefill")
    assert_close(out.float().cpu().numpy().reshape(nq, cfg.H, cfg.V), ref["out"], TOL_BF16,
                 "fp8 prefill out")
    assert_close(lse.cpu().numpy().reshape(nq, cfg.H), ref["lse"], TOL_LSE_BF16, "fp8 prefill lse")


CHILD = r'''
import sys
sys.path.insert(0, ROOT); sys.path.insert(0, ROOT + "/tests")
import torch
torch.cuda.set_device(0)
from compressed_sparse_attention_indexer_gb300.workloads import BF16_CFG
from test_prefill_indexer import check_prefill_scores
for host in (False, True):
    check_prefill_scores(BF16_CFG, 13, [13, 600, 4109, 2100], seed=71, host_lens=host)
    check_prefill_scores(BF16_CFG, 21, [3000, 21], seed=75, host_lens=host)
print("warp-mma prefill ok")
'''


def test_prefill_scores_on_the_warp_mma_indexer():
    # the warp-MMA kernel's own split (groups of 8; S = 13 and 21: ragged last groups)
    code = "ROOT = %r\n" % ROOT + CHILD
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, CSA_INDEXER="mma"),
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "warp-mma prefill ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
