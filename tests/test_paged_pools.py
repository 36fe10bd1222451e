"""Paged pools: block tables instead of per-request contiguous row ranges.

The pages' cache pools are allocator-mapped ("Fix: complete DeepSeek V4 TP CSA
decode", PR description: pools with allocator-valid, collision-free slot
mappings, comparators that check only mapped rows).  With a block table, row r
of request b lives in pool block table[b, r / block] at offset r % block.

CPU: paging is a layout, so the oracle gives bit-identical results on a
batch and on the same batch paged (several block sizes, FP8 keys, the heavy
stream with several queries per request); a row needed from an unmapped
block is an error; the host checks of the new fields.  GPU: the step on paged
pools against the oracle (unused pool rows are NaN, so a wrong row poisons
the output), with device and host lengths and under the other kernel
selections, and an unmapped block reported through the status word.
"""
import ctypes
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
    BF16_CFG, Workload, make_batch, paginate, to_device)
from helpers import TOL_BF16, TOL_LSE_BF16, assert_close, assert_topk_sets

DEV = "cuda:0"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = {
    # name: (cfg, S, lens, blocks)
    "small_blocks": (BF16_CFG, 1, [700, 5003, 2052, 130], dict(raw=16, cmp=64, idx=128)),
    "fp8_large_blocks": (replace(BF16_CFG, idx_dtype="fp8"), 1, [9000, 300, 2051],
                         dict(raw=128, cmp=256, idx=256)),
    "hca_multitoken": (replace(BF16_CFG, hca_ratio=128), 4, [3000, 1027],
                       dict(raw=32, cmp=32, idx=128, hca=8)),
    "partly_paged": (BF16_CFG, 2, [4100, 600], dict(cmp=48)),
}


def _batch(name, seed=9):
    cfg, S, lens, blocks = CASES[name]
    wl = Workload("paged-" + name, cfg, B=len(lens), S=S, L=1, seed=seed)
    hb = make_batch(wl, lens=lens, gap_rows=1)
    return wl, hb, paginate(hb, blocks, seed=seed + 1)


# ---------------------------------------------------------------------------
# CPU: the oracle

@pytest.mark.parametrize("name", sorted(CASES))
def test_paging_is_a_layout_for_the_oracle(name):
    oracle.build()
    wl, hb, pg = _batch(name)
    a = oracle.decode(wl.cfg, hb)
    b = oracle.decode(wl.cfg, pg)
    assert np.array_equal(a["topk_idx"], b["topk_idx"])
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])
    S = hb["S"]
    for q in range(hb["B"] * S):
        if a["vis"][q] > 0:
            assert np.array_equal(oracle.query_scores(wl.cfg, hb, q // S, q % S),
                                  oracle.query_scores(wl.cfg, pg, q // S, q % S))


def test_a_needed_row_in_an_unmapped_block_is_an_error():
    oracle.build()
    wl, hb, pg = _batch("small_blocks")
    pg["cmp_table"] = pg["cmp_table"].clone()
    pg["cmp_table"][1, 0] = -1
    with pytest.raises(ValueError):
        oracle.decode(wl.cfg, pg)


# ---------------------------------------------------------------------------
# CPU: host checks

@pytest.fixture(scope="module")
def L():
    csa_build.build()
    return csa.lib()


def _cfg():
    return csa.make_config(BF16_CFG, 4, 1, 8192)


def _cbatch(**kw):
    a = 0x10000
    base = dict(B=2, S=1, ctx_len=a, ctx_len_host=None, q=a, q_idx=a, w=a,
                raw_kv=a, raw_off=None, raw_stride=576, raw_rows=10,
                cmp_kv=a, cmp_off=None, cmp_stride=576, cmp_rows=10,
                idx_k=a, idx_off=None, idx_stride=128, idx_rows=10,
                hca_kv=None, hca_off=None, hca_stride=0, hca_rows=0,
                raw_table=a, cmp_table=a, idx_table=a, raw_block=16, cmp_block=64, idx_block=128,
                table_stride=8)
    base.update(kw)
    return csa.CBatch(**base)


def _check(b):
    return csa.lib().csa_check_batch(ctypes.byref(_cfg()), ctypes.byref(b))


def test_paged_batch_passes_without_offsets(L):
    assert _check(_cbatch()) == csa.CSA_OK


@pytest.mark.parametrize("kw", [dict(idx_block=100), dict(idx_block=64), dict(raw_block=0),
                                dict(cmp_block=-3), dict(table_stride=0), dict(cmp_table=0x10002),
                                dict(raw_table=None)])  # raw not paged and raw_off NULL
def test_paged_host_check_codes(L, kw):
    assert _check(_cbatch(**kw)) == csa.CSA_ERR_INVALID_ARG
    assert csa.last_error()


# ---------------------------------------------------------------------------
# GPU parity

def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    csa_build.build()
    oracle.build()
    torch.cuda.set_device(0)


def _run(wl, pg, host_lens):
    cfg = wl.cfg
    db = to_device(pg, DEV)
    B, S = pg["B"], pg["S"]
    dec = csa.Decoder(cfg, B, S, max(int(pg["ctx_len"].max()), 4))
    out = torch.full((B, S, cfg.H, cfg.V), float("nan"), dtype=cfg.torch_dtype, device=DEV)
    lse = torch.full((B, S, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
    idx = torch.full((B, S, cfg.topk), -7, dtype=torch.int32, device=DEV)
    cnt = torch.full((B, S), -7, dtype=torch.int32, device=DEV)
    lh = pg["ctx_len"].clone() if host_lens else None
    dec.decode_step(csa.make_batch_struct(db, lh), out, lse, idx, cnt)
    nq = B * S
    return (dec.status(), out.float().cpu().numpy().reshape(nq, cfg.H, cfg.V),
            lse.cpu().numpy().reshape(nq, cfg.H), idx.cpu().numpy().reshape(nq, cfg.topk),
            cnt.cpu().numpy().reshape(nq))


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("host_lens", [False, True])
def test_paged_step_matches_oracle(name, host_lens):
    _gpu()
    wl, hb, pg = _batch(name)
    ref = oracle.decode(wl.cfg, pg)
    st, out, lse, idx, cnt = _run(wl, pg, host_lens)
    assert st == csa.CSA_OK, csa.last_error()
    S = pg["S"]
    assert_topk_sets(idx, cnt, ref, lambda q: oracle.query_scores(wl.cfg, pg, q // S, q % S),
                     wl.cfg.topk, name)
    assert_close(out, ref["out"], TOL_BF16, name + " out")
    assert_close(lse, ref["lse"], TOL_LSE_BF16, name + " lse")


@pytest.mark.gpu
def test_unmapped_block_is_reported():
    _gpu()
    wl, hb, pg = _batch("small_blocks")
    pg["cmp_table"] = pg["cmp_table"].clone()
    pg["cmp_table"][1, 0] = -1            # compressed rows 0..63 of request 1
    st, *_ = _run(wl, pg, True)
    assert st == csa.CSA_ERR_BAD_INDEX


CHILD = r'''
import sys, numpy as np, torch
sys.path.insert(0, ROOT); sys.path.insert(0, ROOT + "/tests")
import oracle
from test_paged_pools import _batch, _run
from helpers import TOL_BF16, assert_close, assert_topk_sets
from compressed_sparse_attention_indexer_gb300 import csa
for name in ("small_blocks", "hca_multitoken"):
    wl, hb, pg = _batch(name)
    ref = oracle.decode(wl.cfg, pg)
    st, out, lse, idx, cnt = _run(wl, pg, True)
    assert st == csa.CSA_OK, csa.last_error()
    S = pg["S"]
    assert_topk_sets(idx, cnt, ref, lambda q: oracle.query_scores(wl.cfg, pg, q // S, q % S), 512, name)
    assert_close(out, ref["out"], TOL_BF16, name)
print("paged variant ok")
'''


@pytest.mark.gpu
@pytest.mark.parametrize("env", [{"CSA_INDEXER": "mma", "CSA_ATTN": "mma"}])
def test_paged_pools_under_the_warp_mma_kernels(env):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    code = "ROOT = %r\n" % ROOT + CHILD
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, **env), cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "paged variant ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
