"""Oracle pins for FP8 E4M3 indexer keys with a per-row fp32 scale.

The pages pass the indexer cache as a key pool plus a per-row scale pool
("Fix: complete DeepSeek V4 TP CSA decode", PR description); the element
format (OCP FP8 E4M3) is a reading.  A key row is scale[row] * e4m3(bytes)
and the score formula is unchanged.  The decoder is pinned to torch's
float8_e4m3fn cast (a library routine) and to the format's landmark values;
the scaled scoring path is pinned to the bf16 path on keys both can hold
exactly, and to the positive homogeneity of ReLU.
"""
import math
from dataclasses import replace

import numpy as np
import torch

import oracle
from compressed_sparse_attention_indexer_gb300.workloads import BF16_CFG, Workload, make_batch

FP8_CFG = replace(BF16_CFG, idx_dtype="fp8")


def test_e4m3_decoder_matches_torch_float8_on_every_code():
    oracle.build()
    got = np.array([oracle.e4m3_value(v) for v in range(256)])
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()
    # landmarks of the format: 1.0, the largest finite value, the smallest
    # subnormal and normal, signs, the two NaN codes, signed zero
    assert got[0x38] == 1.0 and got[0xB8] == -1.0
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6 and got[0x07] == 7 * 2.0 ** -9
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF]) and nan.sum() == 2
    assert got[0x00] == 0.0 and math.copysign(1.0, got[0x80]) == -1.0


def test_fp8_scoring_equals_the_bf16_path_on_exactly_representable_keys():
    # with power-of-two row scales every dequantised key is a bf16 value, so
    # the FP8 oracle path must give the bf16 path's scores bit for bit
    oracle.build()
    wl = Workload("fp8-vs-bf16", FP8_CFG, B=3, S=2, L=1, seed=31)
    hb8 = make_batch(wl, lens=[3000, 700, 5003], gap_rows=1)
    sc = hb8["idx_scale"]
    p2 = torch.where(torch.isfinite(sc) & (sc > 0), torch.exp2(torch.round(torch.log2(sc))), sc)
    hb8["idx_scale"] = p2.contiguous()
    codes = hb8["idx_k"].view(torch.float8_e4m3fn).to(torch.float64)
    hb16 = dict(hb8)
    hb16["idx_k"] = (codes * p2.double()[:, None]).to(torch.bfloat16).contiguous()
    fin = ~codes.isnan()
    assert torch.equal(hb16["idx_k"].double()[fin], (codes * p2.double()[:, None])[fin])  # exact
    hb16["idx_scale"] = None
    for b in range(3):
        for s in range(2):
            a = oracle.query_scores(FP8_CFG, hb8, b, s)
            r = oracle.query_scores(BF16_CFG, hb16, b, s)
            assert a.shape == r.shape and np.array_equal(a, r), (b, s)
    d8 = oracle.decode(FP8_CFG, hb8, force_score=True)
    d16 = oracle.decode(BF16_CFG, hb16, force_score=True)
    assert np.array_equal(d8["topk_idx"], d16["topk_idx"])
    assert np.array_equal(d8["out"], d16["out"])


def test_scale_multiplies_every_score_of_a_row():
    # doubling one row's scale doubles that row's score (ReLU is positively
    # homogeneous) and leaves the other rows alone
    oracle.build()
    wl = Workload("fp8-scale", FP8_CFG, B=1, S=1, L=1, seed=32)
    hb = make_batch(wl, lens=[4000])
    base = oracle.query_scores(FP8_CFG, hb, 0, 0)
    off = int(hb["idx_off"][0])
    hb2 = dict(hb)
    hb2["idx_scale"] = hb["idx_scale"].clone()
    hb2["idx_scale"][off + 17] *= 2.0
    got = oracle.query_scores(FP8_CFG, hb2, 0, 0)
    assert got[17] == 2.0 * base[17]
    mask = np.ones_like(base, bool)
    mask[17] = False
    assert np.array_equal(got[mask], base[mask])


