"""GPU parity: every step of the CUDA path, through the C ABI, against the CPU oracle.

Same seeded inputs on both sides.  Top-K index sets must match exactly except
for elements whose oracle score is within 1e-6 (relative) of the K-th
oracle score; attention outputs within 2e-2 max-abs / 1e-2 mean-abs of the
fp64 oracle for bf16 inputs and 1e-5 for the fp32 workload.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_indexer_gb300 import build as csa_build
from compressed_sparse_attention_indexer_gb300 import csa
from compressed_sparse_attention_indexer_gb300.workloads import (
    BF16_CFG, CsaConfig, Dists, Workload, WORKLOADS, make_batch, to_device)
from helpers import TOL_BF16, TOL_LSE_BF16, TOL_LSE_F32, assert_close, assert_topk_sets, tol_for

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    csa_build.build()
    oracle.build()
    torch.cuda.set_device(0)


def run_step(wl, hb, max_context=None, host_lens=False):
    cfg = wl.cfg
    db = to_device(hb, DEV)
    B, S = hb["B"], hb["S"]
    mc = max_context or max(int(hb["ctx_len"].max()), 4)
    dec = csa.Decoder(cfg, B, S, mc)
    out = torch.full((B, S, cfg.H, cfg.V), float("nan"), dtype=cfg.torch_dtype, device=DEV)
    lse = torch.full((B, S, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
    idx = torch.full((B, S, cfg.topk), -7, dtype=torch.int32, device=DEV)
    cnt = torch.full((B, S), -7, dtype=torch.int32, device=DEV)
    lens_host = hb["ctx_len"].clone() if host_lens else None
    cb = csa.make_batch_struct(db, lens_host)
    dec.decode_step(cb, out, lse, idx, cnt)
    st = dec.status()
    nq = B * S
    return dict(dec=dec, db=db, cb=cb, status=st, lens_host=lens_host,
                out=out.float().cpu().numpy().reshape(nq, cfg.H, cfg.V),
                lse=lse.cpu().numpy().reshape(nq, cfg.H),
                idx=idx.cpu().numpy().reshape(nq, cfg.topk), cnt=cnt.cpu().numpy().reshape(nq))


def scores_fn(cfg, hb):
    S = hb["S"]
    return lambda q: oracle.query_scores(cfg, hb, q // S, q % S)


def check_against_oracle(wl, hb, g, ref=None, what=""):
    cfg = wl.cfg
    ref = ref if ref is not None else oracle.decode(cfg, hb)
    assert g["status"] == csa.CSA_OK, csa.last_error()
    assert_topk_sets(g["idx"], g["cnt"], ref, scores_fn(cfg, hb), cfg.topk, what)
    assert_close(g["out"], ref["out"], tol_for(cfg), what + " out")
    # bf16 path: the softmax weights are rounded to bf16 before they are
    # summed (the bound is derived beside TOL_LSE_BF16)
    lse_tol = TOL_LSE_F32 if cfg.dtype == "f32" else TOL_LSE_BF16
    assert_close(g["lse"], ref["lse"], lse_tol, what + " lse")
    return ref


# ---------------------------------------------------------------------------
# the named workloads, full size (prefill_b2_t512: a 512-token prefill chunk
# per request, each token with its own visibility and Top-K)

@pytest.mark.parametrize("name", ["tiny_f32", "bypass_b16_l256", "topk_b16_l8192",
                                  "long_ragged_b64", "multitoken_hca_b16_s8", "prefill_b2_t512"])
def test_workload_decode_step(name):
    wl = WORKLOADS[name]
    hb = make_batch(wl)
    g = run_step(wl, hb, max_context=65536 if name == "long_ragged_b64" else None)
    ref = check_against_oracle(wl, hb, g, what=name)
    # the launch configuration bench.py times: lengths known on the host
    # (host-built work lists, no prep kernels)
    gh = run_step(wl, hb, max_context=65536 if name == "long_ragged_b64" else None, host_lens=True)
    check_against_oracle(wl, hb, gh, ref=ref, what=name + " host-lengths")
    # attention alone on the oracle's own selection isolates steps (c)-(d)
    cfg = wl.cfg
    B, S = hb["B"], hb["S"]
    idx = torch.from_numpy(ref["topk_idx"]).to(DEV).view(B, S, cfg.topk)
    cnt = torch.from_numpy(ref["cnt"].astype(np.int32)).to(DEV).view(B, S)
    out = torch.empty(B, S, cfg.H, cfg.V, dtype=cfg.torch_dtype, device=DEV)
    g["dec"].sparse_attn(g["cb"], idx, cnt, out)
    assert g["dec"].status() == csa.CSA_OK
    assert_close(out.float().cpu().numpy().reshape(B * S, cfg.H, cfg.V), ref["out"], tol_for(cfg),
                 name + " sparse_attn")
    # bypass workload: no scoring launch when the host knows every query fits K
    if name == "bypass_b16_l256":
        assert (ref["cnt"] == ref["vis"]).all()


def test_indexer_topk_entry_matches_decode_step():
    wl = WORKLOADS["topk_b16_l8192"]
    hb = make_batch(wl)
    g = run_step(wl, hb)
    B, S = hb["B"], hb["S"]
    idx = torch.empty(B, S, wl.cfg.topk, dtype=torch.int32, device=DEV)
    cnt = torch.empty(B, S, dtype=torch.int32, device=DEV)
    g["dec"].indexer_topk(g["cb"], idx, cnt)
    assert g["dec"].status() == csa.CSA_OK
    np.testing.assert_array_equal(idx.cpu().numpy().reshape(B * S, -1), g["idx"])
    np.testing.assert_array_equal(cnt.cpu().numpy().reshape(-1), g["cnt"])


# ---------------------------------------------------------------------------
# step (a) alone: fp32 scores against fp64

@pytest.mark.parametrize("name,lens", [("topk_b16_l8192", [8192, 300, 1029, 4097]),
                                       ("tiny_f32", None)])
def test_indexer_scores_against_oracle(name, lens):
    wl = WORKLOADS[name]
    cfg = wl.cfg
    hb = make_batch(wl, lens=lens)
    db = to_device(hb, DEV)
    B, S = hb["B"], hb["S"]
    mc = int(hb["ctx_len"].max())
    dec = csa.Decoder(cfg, B, S, mc)
    ld = mc // cfg.ratio
    scores = torch.full((B * S, ld), float("nan"), dtype=torch.float32, device=DEV)
    dec.indexer_scores(csa.make_batch_struct(db), scores, score_all=True)
    assert dec.status() == csa.CSA_OK
    sc = scores.cpu().numpy()
    qi = hb["q_idx"].double().numpy()
    w = hb["w"].double().numpy()
    for q in range(B * S):
        b, s = divmod(q, S)
        ref = oracle.query_scores(cfg, hb, b, s)
        n = len(ref)
        got = sc[q, :n]
        assert np.isnan(sc[q, n:]).all(), "entries past vis must stay untouched"
        # error bound of fp32 accumulation: relative to sum_h w_h sum_d |q_hd k_jd|
        off = int(hb["idx_off"][b])
        k = hb["idx_k"][off:off + n].double().numpy()
        mag = np.abs(k) @ np.abs(qi[b, s]).T @ w[b, s]
        bound = 2e-6 * mag + 1e-30
        assert (np.abs(got - ref) <= bound).all(), \
            f"q{q}: max err {np.abs(got - ref).max():.3e}, ratio {(np.abs(got - ref) / bound).max():.2f}"


# ---------------------------------------------------------------------------
# step (b) alone, bit exact on seeded fp32 scores

def _topk_cases(rng):
    cases = []
    for n in (255, 256, 257, 511, 512, 513, 1023, 1024, 1025, 4096, 16384):
        s = rng.standard_normal(n).astype(np.float32)
        cases.append(("normal", s))
        q = (np.round(rng.standard_normal(n) * 4) / 4).astype(np.float32)    # many exact ties
        cases.append(("ties", q))
        p = rng.uniform(-1, 0, n).astype(np.float32)
        planted = rng.choice(np.arange(n // 2, n), size=min(512, n // 2), replace=False)
        p[planted] = rng.uniform(1, 2, planted.size).astype(np.float32)
        cases.append(("planted_tail", p))
    cases.append(("all_equal", np.full(3000, 2.5, np.float32)))
    z = np.zeros(2000, np.float32)
    z[::2] = -0.0
    z[1500:] = -1.0
    cases.append(("signed_zero", z))
    cases.append(("neg_and_inf", np.concatenate([-np.abs(rng.standard_normal(900)).astype(np.float32),
                                                 np.full(3, -np.inf, np.float32)])))
    cases.append(("narrow_band", (100.0 + rng.standard_normal(16384) * 1e-4).astype(np.float32)))
    # two values: the K-th key is one of > 1024 equal keys (ties by index after
    # the radix passes), once after a higher group and once as the top group
    cases.append(("high_then_equal", np.concatenate([np.full(300, 5.0), np.full(4000, 1.0)]).astype(np.float32)))
    cases.append(("two_values", np.where(rng.random(16384) < 0.5, 1.0, 2.0).astype(np.float32)))
    return cases


def test_topk_select_bit_exact():
    rng = np.random.default_rng(2024)
    cfg = BF16_CFG
    cases = _topk_cases(rng)
    dec = csa.Decoder(cfg, len(cases), 1, 65536)
    ld = 16384
    sc = np.full((len(cases), ld), np.nan, np.float32)
    n = np.zeros(len(cases), np.int32)
    for i, (_, s) in enumerate(cases):
        sc[i, :s.size] = s
        n[i] = s.size
    idx = torch.empty(len(cases), cfg.topk, dtype=torch.int32, device=DEV)
    cnt = torch.empty(len(cases), dtype=torch.int32, device=DEV)
    dec.topk_select(torch.from_numpy(sc).to(DEV), torch.from_numpy(n).to(DEV), idx, cnt)
    assert dec.status() == csa.CSA_OK
    gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
    for i, (name, s) in enumerate(cases):
        ref = oracle.topk(s.astype(np.float64), cfg.topk)
        assert gc[i] == ref.size, name
        assert gi[i, :ref.size].tolist() == ref.tolist(), f"{name} n={s.size}"
        assert (gi[i, ref.size:] == -1).all()


def test_topk_select_bit_exact_short_rows():
    # max_context / ratio <= 2048: the register kernel with two keys per thread
    rng = np.random.default_rng(2026)
    cfg = BF16_CFG
    cases = [(name, s) for name, s in _topk_cases(rng) if s.size <= 2048]
    cases.append(("full_2048_ties", (np.round(rng.standard_normal(2048) * 2) / 2).astype(np.float32)))
    cases.append(("all_equal_2048", np.full(2048, 0.75, np.float32)))
    dec = csa.Decoder(cfg, len(cases), 1, 8192)
    ld = 2048
    sc = np.full((len(cases), ld), np.nan, np.float32)
    n = np.zeros(len(cases), np.int32)
    for i, (_, s) in enumerate(cases):
        sc[i, :s.size] = s
        n[i] = s.size
    idx = torch.empty(len(cases), cfg.topk, dtype=torch.int32, device=DEV)
    cnt = torch.empty(len(cases), dtype=torch.int32, device=DEV)
    dec.topk_select(torch.from_numpy(sc).to(DEV), torch.from_numpy(n).to(DEV), idx, cnt)
    assert dec.status() == csa.CSA_OK
    gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
    for i, (name, s) in enumerate(cases):
        ref = oracle.topk(s.astype(np.float64), cfg.topk)
        assert gc[i] == ref.size, name
        assert gi[i, :ref.size].tolist() == ref.tolist(), f"{name} n={s.size}"
        assert (gi[i, ref.size:] == -1).all()


def test_topk_select_bit_exact_rows_past_16384():
    # max_context / ratio above 16384: the shared-memory Top-K kernel
    rng = np.random.default_rng(2025)
    cfg = BF16_CFG
    cases = []
    for n in (16385, 20000, 32768):
        cases.append(("normal", rng.standard_normal(n).astype(np.float32)))
        cases.append(("ties", (np.round(rng.standard_normal(n) * 4) / 4).astype(np.float32)))
    cases.append(("all_equal", np.full(17000, -3.0, np.float32)))
    dec = csa.Decoder(cfg, len(cases), 1, 131072)
    ld = 32768
    sc = np.full((len(cases), ld), np.nan, np.float32)
    n = np.zeros(len(cases), np.int32)
    for i, (_, s) in enumerate(cases):
        sc[i, :s.size] = s
        n[i] = s.size
    idx = torch.empty(len(cases), cfg.topk, dtype=torch.int32, device=DEV)
    cnt = torch.empty(len(cases), dtype=torch.int32, device=DEV)
    dec.topk_select(torch.from_numpy(sc).to(DEV), torch.from_numpy(n).to(DEV), idx, cnt)
    assert dec.status() == csa.CSA_OK
    gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
    for i, (name, s) in enumerate(cases):
        ref = oracle.topk(s.astype(np.float64), cfg.topk)
        assert gc[i] == ref.size, name
        assert gi[i].tolist() == ref.tolist(), f"{name} n={s.size}"


def _nonfinite_row(rng, n, f_nan, f_ninf=0.0, n_pinf=0):
    s = rng.standard_normal(n).astype(np.float32)
    pos = rng.permutation(n)
    a, b = int(f_nan * n), int((f_nan + f_ninf) * n)
    s[pos[:a]] = np.nan
    s[pos[a:b]] = -np.inf
    s[pos[b:b + n_pinf]] = np.inf
    return s


@pytest.mark.parametrize("max_context,ld,sizes", [(8192, 2048, (2000, 600, 1500, 2048)),
                                                  (65536, 16384, (16384, 700, 5000, 3000)),
                                                  (131072, 32768, (20000, 17000, 18000, 16500))])
def test_topk_select_nonfinite_scores(max_context, ld, sizes):
    # NaN scores rank below every other score (-inf included), +inf above;
    # equal keys (every NaN is one key) go to the lower index.  The oracle
    # takes no NaN, so its input maps -inf and NaN to two values below every
    # finite float, in that order.  Each of the three Top-K kernels (two and
    # sixteen keys per thread in registers, rows in shared memory) on rows
    # with scattered NaN, fewer finite scores than K, only NaN, and -inf / +inf
    # mixed in.
    rng = np.random.default_rng(max_context)
    cfg = BF16_CFG
    n1, n2, n3, n4 = sizes
    cases = [("nan_10pct", _nonfinite_row(rng, n1, 0.10, n_pinf=3)),
             ("finite_below_k", _nonfinite_row(rng, n2, 1.0 - 300.0 / n2)),
             ("all_nan", np.full(n3, np.nan, np.float32)),
             ("nan_and_ninf", _nonfinite_row(rng, n4, 0.45, f_ninf=0.45, n_pinf=5))]
    dec = csa.Decoder(cfg, len(cases), 1, max_context)
    sc = np.full((len(cases), ld), np.nan, np.float32)
    n = np.zeros(len(cases), np.int32)
    for i, (_, s) in enumerate(cases):
        sc[i, :s.size] = s
        n[i] = s.size
    idx = torch.empty(len(cases), cfg.topk, dtype=torch.int32, device=DEV)
    cnt = torch.empty(len(cases), dtype=torch.int32, device=DEV)
    dec.topk_select(torch.from_numpy(sc).to(DEV), torch.from_numpy(n).to(DEV), idx, cnt)
    assert dec.status() == csa.CSA_OK
    gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
    for i, (name, s) in enumerate(cases):
        d = s.astype(np.float64)
        d = np.where(np.isnan(d), -1e301, np.where(np.isneginf(d), -1e300, d))
        ref = oracle.topk(d, cfg.topk)
        assert gc[i] == ref.size, name
        assert gi[i, :ref.size].tolist() == ref.tolist(), f"{name} n={s.size}"


# ---------------------------------------------------------------------------
# edge cases: tiny and ragged lengths, bypass boundary, maximum length, poison

def test_edge_lengths_flagship_shape():
    # vis 0 (empty compressed stream), pos+1 not a multiple of 4, vis = K-1,K,K+1
    # (bypass boundary), 1023..1025, ragged tails, and the maximum 16384
    lens = [1, 2, 3, 4, 5, 130, 2047, 2048, 2051, 2052, 2055, 4095, 4096, 4100, 4103, 65536]
    wl = Workload("edge", BF16_CFG, B=len(lens), S=1, L=1, seed=77)
    hb = make_batch(wl, lens=lens, gap_rows=3)
    g = run_step(wl, hb, max_context=65536, host_lens=True)
    check_against_oracle(wl, hb, g, what="edge")


def test_edge_lengths_without_host_lengths():
    lens = [7, 2049, 3000, 700]
    wl = Workload("edge2", BF16_CFG, B=len(lens), S=1, L=1, seed=78)
    hb = make_batch(wl, lens=lens, gap_rows=2)
    g = run_step(wl, hb, max_context=8192, host_lens=False)
    check_against_oracle(wl, hb, g, what="edge2")


def test_planted_tail_candidates_flagship_shape():
    # key rows aligned with indexer head 0 planted past rows 256 and 1024: the
    # selection must be exactly the planted rows
    wl = Workload("planted", BF16_CFG, B=3, S=1, L=1, seed=91)
    lens = [4 * 1100, 4 * 1500, 4 * 2100]
    hb = make_batch(wl, lens=lens)
    K = BF16_CFG.topk
    rng = np.random.default_rng(5)
    planted_all = []
    for b, L in enumerate(lens):
        vis = L // 4
        qi = hb["q_idx"][b, 0].float()
        qi[:] = qi[0]                           # every indexer head = head 0
        hb["q_idx"][b, 0] = qi.to(torch.bfloat16)
        off = int(hb["idx_off"][b])
        u = qi[0] / qi[0].norm()
        keys = -torch.rand(vis, 1) * u[None, :] * 4
        planted = np.sort(rng.choice(np.arange(300, vis), size=K, replace=False))
        keys[planted] = (1.0 + torch.rand(K, 1)) * u[None, :] * 4
        hb["idx_k"][off:off + vis] = keys.to(torch.bfloat16)
        planted_all.append(planted)
    g = run_step(wl, hb)
    assert g["status"] == csa.CSA_OK
    for b in range(3):
        assert g["idx"][b].tolist() == planted_all[b].tolist()
    check_against_oracle(wl, hb, g, what="planted")


def test_duplicate_keys_tie_to_lower_index():
    wl = Workload("dups", BF16_CFG, B=1, S=1, L=1, seed=92)
    L = 4 * 1000
    hb = make_batch(wl, lens=[L])
    off = int(hb["idx_off"][0])
    hb["idx_k"][off:off + 1000] = hb["idx_k"][off]     # every key identical: all scores tie
    g = run_step(wl, hb)
    assert g["idx"][0].tolist() == list(range(BF16_CFG.topk))
    check_against_oracle(wl, hb, g, what="dups")


def test_multi_token_small():
    cfg = CsaConfig(hca_ratio=128)
    wl = Workload("mt", cfg, B=3, S=8, L=1, seed=93)
    hb = make_batch(wl, lens=[2052, 700, 40000], gap_rows=1)
    g = run_step(wl, hb, max_context=40000, host_lens=True)
    check_against_oracle(wl, hb, g, what="multi-token")


@pytest.mark.parametrize("S", [2, 3, 7])
def test_multi_token_query_groups(S):
    # S queries per request on the tensor-core shape: the tcgen05 indexer
    # scores up to four queries of a request per MMA group (N = 64 per
    # query), so S = 2, 3, 7 give groups of 2, 3 and 4 + 3; requests that
    # bypass scoring, that cross the bypass boundary inside the chunk and
    # that select, both launch forms, against the oracle.
    wl = Workload("mt-groups", BF16_CFG, B=4, S=S, L=1, seed=200 + S)
    hb = make_batch(wl, lens=[2048 + S - 2, 9000, 700, 30001], gap_rows=1)
    ref = None
    for host in (False, True):
        g = run_step(wl, hb, max_context=30001, host_lens=host)
        ref = check_against_oracle(wl, hb, g, ref=ref, what=f"S={S} host={host}")


def test_generic_shapes_simt_path():
    # shapes outside the tensor-core set (bf16 and fp32) run on the SIMT kernels
    for dt in ("bf16", "f32"):
        cfg = CsaConfig(H=6, D=48, V=32, Hi=3, Di=16, ratio=4, topk=5, win=4, hca_ratio=16, dtype=dt)
        wl = Workload("generic", cfg, B=4, S=3, L=1, seed=94)
        hb = make_batch(wl, lens=[3, 9, 40, 131], gap_rows=1)
        g = run_step(wl, hb)
        check_against_oracle(wl, hb, g, what=f"generic-{dt}")


# ---------------------------------------------------------------------------
# value range: KV rows of any bf16 magnitude.  Multiplying every KV row by 2^e
# and q by 2^-e leaves every score q . row unchanged, so the exact output is
# 2^e times the unscaled output.  Every rounding the step makes (fp32
# accumulation, the bf16 segment partials, the bf16 output) commutes with a
# power-of-two scale while values stay inside their type's normal range, so
# the scaled GPU output must be the unscaled GPU output times 2^e bit for bit,
# and within the usual tolerance of the oracle run on the scaled inputs.
# 2^17 puts outputs near 1e5 (past fp16's 65504) and 2^-20 near 1e-7 (below
# fp16's normal range).

def _scaled_rows(hb, e):
    out = dict(hb)
    f = 2.0 ** e
    out["q"] = (hb["q"].float() * (1.0 / f)).to(hb["q"].dtype)
    for k in ("raw_kv", "cmp_kv", "hca_kv"):
        if hb.get(k) is not None:
            out[k] = (hb[k].float() * f).to(hb[k].dtype)
    return out


@pytest.mark.parametrize("name,lens,e", [("topk_b16_l8192", [8192, 5000, 700, 129], 17),
                                         ("topk_b16_l8192", [8192, 5000, 700, 129], -20),
                                         ("multitoken_hca_b16_s8", [32768, 4100], 17),
                                         ("long_ragged_b64", [65536, 1024, 30001], 17)])
def test_value_range_scaled_rows(name, lens, e):
    wl = WORKLOADS[name]
    hb = make_batch(wl, lens=lens)
    hs = _scaled_rows(hb, e)
    # the scaled inputs are exact: q * 2^-e * 2^e and row * 2^e * 2^-e round-trip
    assert torch.equal((hs["q"].float() * 2.0 ** e).to(hb["q"].dtype), hb["q"])
    assert torch.equal((hs["cmp_kv"].float() * 2.0 ** -e).to(hb["cmp_kv"].dtype), hb["cmp_kv"])
    mc = max(lens)
    g = run_step(wl, hb, max_context=mc, host_lens=True)
    gs = run_step(wl, hs, max_context=mc, host_lens=True)
    assert gs["status"] == csa.CSA_OK, csa.last_error()
    assert np.isfinite(gs["out"]).all()
    np.testing.assert_array_equal(gs["out"], g["out"] * 2.0 ** e)
    np.testing.assert_array_equal(gs["lse"], g["lse"])
    np.testing.assert_array_equal(gs["idx"], g["idx"])
    ref = oracle.decode(wl.cfg, hs)
    assert_topk_sets(gs["idx"], gs["cnt"], ref, scores_fn(wl.cfg, hs), wl.cfg.topk, name)
    assert_close(gs["out"] * 2.0 ** -e, ref["out"] * 2.0 ** -e, TOL_BF16, f"{name} 2^{e} out")
    assert_close(gs["lse"], ref["lse"], TOL_LSE_BF16, f"{name} 2^{e} lse")


# ---------------------------------------------------------------------------
# determinism, empty batch, device-side error reporting

def test_bitwise_deterministic():
    wl = WORKLOADS["topk_b16_l8192"]
    hb = make_batch(wl)
    g1 = run_step(wl, hb)
    g2 = run_step(wl, hb)
    np.testing.assert_array_equal(g1["out"], g2["out"])
    np.testing.assert_array_equal(g1["idx"], g2["idx"])
    np.testing.assert_array_equal(g1["lse"], g2["lse"])


def test_many_consecutive_steps_keep_a_clean_status():
    # a few thousand back-to-back steps in the bench's launch configuration
    # (PDL chaining, host lengths): a lost barrier phase or a race between
    # consecutive kernels shows up as CSA_ERR_TIMEOUT or a changed output
    wl = WORKLOADS["long_ragged_b64"]
    hb = make_batch(wl)
    db = to_device(hb, DEV)
    cfg = wl.cfg
    dec = csa.Decoder(cfg, hb["B"], 1, 65536)
    lens_host = hb["ctx_len"].clone()  # kept alive while the struct points at it
    cb = csa.make_batch_struct(db, lens_host)
    out = torch.empty(hb["B"], 1, cfg.H, cfg.V, dtype=cfg.torch_dtype, device=DEV)
    idx = torch.empty(hb["B"], 1, cfg.topk, dtype=torch.int32, device=DEV)
    cnt = torch.empty(hb["B"], 1, dtype=torch.int32, device=DEV)
    dec.decode_step(cb, out, None, idx, cnt)
    first = out.clone()
    for i in range(2000):
        dec.decode_step(cb, out, None, idx, cnt)
        if i % 4 == 3:
            dec.sparse_attn(cb, idx, cnt, out)
    torch.cuda.synchronize()
    assert dec.status() == csa.CSA_OK, csa.last_error()
    assert torch.equal(out, first)


def test_steps_without_indexer_work_between_selecting_steps():
    # The indexer publishes each request's scored items to one of two
    # counter sets and zeroes the other for its next launch; a step whose
    # queries all bypass scoring launches no indexer.  Alternating such steps
    # (with and without host lengths) with selecting ones, with the indexer +
    # Top-K entry (which publishes nothing) in between, every selecting step
    # must reproduce the first one bit for bit with a clean status: a counter
    # set left stale would let Top-K read scores early.
    wl = WORKLOADS["topk_b16_l8192"]
    cfg = wl.cfg
    sel = make_batch(wl, lens=[8192, 5000, 2100, 4097])
    byp = make_batch(wl, lens=[2048, 700, 129, 1])
    ds, db_ = to_device(sel, DEV), to_device(byp, DEV)
    dec = csa.Decoder(cfg, 4, 1, 8192)
    ls, lb = sel["ctx_len"].clone(), byp["ctx_len"].clone()
    structs = [csa.make_batch_struct(ds, ls), csa.make_batch_struct(ds)]
    bstructs = [csa.make_batch_struct(db_, lb), csa.make_batch_struct(db_)]
    out = torch.empty(4, 1, cfg.H, cfg.V, dtype=cfg.torch_dtype, device=DEV)
    idx = torch.empty(4, 1, cfg.topk, dtype=torch.int32, device=DEV)
    cnt = torch.empty(4, 1, dtype=torch.int32, device=DEV)
    dec.decode_step(structs[0], out, None, idx, cnt)
    torch.cuda.synchronize()
    assert dec.status() == csa.CSA_OK, csa.last_error()
    first, first_idx = out.clone(), idx.clone()
    for i in range(12):
        for _ in range(i % 3):
            dec.decode_step(bstructs[i % 2], out, None, idx, cnt)
        if i % 4 == 1:
            dec.indexer_topk(structs[i % 2], idx, cnt)
        out.fill_(float("nan"))
        dec.decode_step(structs[(i // 2) % 2], out, None, idx, cnt)
        torch.cuda.synchronize()
        assert dec.status() == csa.CSA_OK, csa.last_error()
        assert torch.equal(idx, first_idx)
        assert torch.equal(out, first)
    dec.close()


@pytest.mark.parametrize("name,lens,dists,what", [
    ("topk_b16_l8192", [8192, 5000, 2100, 300], Dists(q=16.0), "peaked"),
    ("multitoken_hca_b16_s8", [32768, 9000], Dists(q=16.0), "peaked"),
    ("topk_b16_l8192", [8192, 5000, 2100, 300], Dists(q=0.0), "flat"),
    ("topk_b16_l8192", [8192, 5000, 2100, 300], Dists(w_hi=0.0), "zero_scores")])
def test_softmax_and_score_extremes_against_oracle(name, lens, dists, what):
    # peaked: query heads drawn with standard deviation 16 instead of 1:
    # scores of standard deviation ~16 (raw rows) and ~8 (compressed rows), so
    # a job's maximum often exceeds a segment's reference maximum by more than
    # 8 in log2 units and the accumulated output is rescaled in TMEM, and the
    # softmax is dominated by a few rows.  flat: q = 0, every attention score
    # 0, the output the mean of the rows and lse = ln(rows).  zero_scores:
    # w = 0, every indexer score 0, so the selection is the first K rows
    # (ties to the lower index), checked exactly.  Both launch forms.
    wl = WORKLOADS[name]
    hb = make_batch(wl, lens=lens, dists=dists)
    ref = None
    for host in (False, True):
        g = run_step(wl, hb, host_lens=host)
        ref = check_against_oracle(wl, hb, g, ref=ref, what=f"{name} {what} host={host}")
        if what == "zero_scores":
            np.testing.assert_array_equal(g["idx"], ref["topk_idx"].reshape(g["idx"].shape))


def test_large_k_takes_the_warp_mma_attention():
    # K = 4096 gives a query up to 2 + 64 jobs of 64 rows, more than the
    # tcgen05 merge takes (64): the step's attention then runs on the
    # warp-MMA kernel by itself, with the tcgen05 indexer and the register
    # Top-K (selection of 4096 of up to 10000 rows) before it.  Requests past,
    # below and at the bypass boundary, both launch forms, against the oracle.
    cfg = dataclasses.replace(BF16_CFG, topk=4096)
    wl = Workload("k4096", cfg, B=3, S=1, L=1, seed=4096)
    hb = make_batch(wl, lens=[40000, 16384, 9000])
    ref = None
    for host in (False, True):
        g = run_step(wl, hb, max_context=40960, host_lens=host)
        ref = check_against_oracle(wl, hb, g, ref=ref, what=f"K=4096 host={host}")
        if host:  # indexer, Top-K and one attention launch (not tile + merge)
            assert g["dec"].last_launch_count() == 3
    assert (ref["cnt"] == [4096, 4096, 2250]).all()


def test_long_context_takes_the_shared_memory_topk():
    # max_context 131072: rows of up to 32768 compressed scores, past what the
    # register Top-K holds, so the step selects with the shared-memory kernel
    # (float scores from the indexer, the Top-K blocks still started per
    # request and publishing ready flags to the attention).  Both launch
    # forms, against the oracle.
    wl = WORKLOADS["topk_b16_l8192"]
    hb = make_batch(wl, lens=[131072, 100001, 70000, 5000], seed=131)
    ref = None
    for host in (False, True):
        g = run_step(wl, hb, max_context=131072, host_lens=host)
        ref = check_against_oracle(wl, hb, g, ref=ref, what=f"long context host={host}")
    assert (ref["vis"] == [32768, 25000, 17500, 1250]).all()


def test_counter_sets_after_a_smaller_batch():
    # A publishing launch zeroes the other counter set for the next one.  When
    # a smaller batch comes between two larger ones, the entries past the
    # small batch must be cleared as well: otherwise the third step's Top-K
    # blocks of those requests find the first step's counts already at their
    # target and select from the scores as they stand (the first step's).
    # The third step must equal the same batch run on a fresh handle.
    wl = WORKLOADS["topk_b16_l8192"]
    cfg = wl.cfg
    lens = [8192, 6000, 4097, 8192, 3000, 7000, 2500, 8000]
    big1 = to_device(make_batch(wl, lens=lens, seed=601), DEV)
    small = to_device(make_batch(wl, lens=[8192, 5000], seed=602), DEV)
    big2 = to_device(make_batch(wl, lens=lens, seed=603), DEV)
    lt = torch.tensor(lens, dtype=torch.int32)
    B = len(lens)

    def outputs(bs):
        return (torch.empty(bs, 1, cfg.H, cfg.V, dtype=cfg.torch_dtype, device=DEV),
                torch.empty(bs, 1, cfg.topk, dtype=torch.int32, device=DEV),
                torch.empty(bs, 1, dtype=torch.int32, device=DEV))

    fresh = csa.Decoder(cfg, B, 1, 8192)
    o_ref, i_ref, c_ref = outputs(B)
    fresh.decode_step(csa.make_batch_struct(big2, lt), o_ref, None, i_ref, c_ref)
    torch.cuda.synchronize()
    assert fresh.status() == csa.CSA_OK, csa.last_error()
    fresh.close()

    ls = torch.tensor([8192, 5000], dtype=torch.int32)  # host lengths, alive while used
    dec = csa.Decoder(cfg, B, 1, 8192)
    for rep in range(3):
        o, i, c = outputs(B)
        dec.decode_step(csa.make_batch_struct(big1, lt), o, None, i, c)
        o2, i2, c2 = outputs(2)
        dec.decode_step(csa.make_batch_struct(small, ls), o2, None, i2, c2)
        o, i, c = outputs(B)
        o.fill_(float("nan"))
        dec.decode_step(csa.make_batch_struct(big2, lt), o, None, i, c)
        torch.cuda.synchronize()
        assert dec.status() == csa.CSA_OK, csa.last_error()
        assert torch.equal(i, i_ref), f"repetition {rep}"
        assert torch.equal(c, c_ref)
        assert torch.equal(o, o_ref)
    dec.close()


@pytest.mark.parametrize("name,maxB,max_len", [("topk_b16_l8192", 8, 8192),
                                               ("topk_b16_l8192 fp8", 8, 8192),
                                               ("multitoken_hca_b16_s8", 4, 16384)])
def test_random_batch_sequence_matches_fresh_handles(name, maxB, max_len):
    # Every piece of state that outlives a step (counter sets, ready flags and
    # their epochs, work lists, scores, partials) must not leak into the next
    # one: one handle runs a seeded random sequence of batches of different
    # sizes, lengths and data (one all-bypass), with and without host
    # lengths, and each step must equal that batch run alone on a fresh
    # handle in the same launch form, bit for bit.  (The two forms may differ
    # in the last bits: with host lengths the tile CTAs' job split favours
    # the CTAs that start while Top-K runs, which moves segment boundaries
    # and so the merge's rounding.)  Single-token steps start Top-K per
    # request on the indexer's counters; multi-token steps wait for the
    # indexer grid and add the heavy-compression stream.  "fp8": the same
    # with E4M3 indexer keys and per-row scales.
    wl = WORKLOADS[name.split()[0]]
    if name.endswith("fp8"):
        wl = dataclasses.replace(wl, cfg=dataclasses.replace(wl.cfg, idx_dtype="fp8"))
    cfg = wl.cfg
    S = wl.S
    rng = np.random.default_rng(77)
    bypass_len = cfg.topk * cfg.ratio - S  # every query's vis <= K
    batches = []
    for i in range(6):
        B = int(rng.integers(1, maxB + 1))
        hi = bypass_len if i == 2 else max_len  # batch 2: every query bypasses scoring
        lens = [int(x) for x in rng.integers(S, hi + 1, size=B)]
        batches.append((to_device(make_batch(wl, lens=lens, seed=700 + i), DEV),
                        torch.tensor(lens, dtype=torch.int32)))

    def run(dec, db, lh):
        B = int(db["B"])
        o = torch.full((B, S, cfg.H, cfg.V), float("nan"), dtype=cfg.torch_dtype, device=DEV)
        i = torch.full((B, S, cfg.topk), -7, dtype=torch.int32, device=DEV)
        c = torch.full((B, S), -7, dtype=torch.int32, device=DEV)
        dec.decode_step(csa.make_batch_struct(db, lh), o, None, i, c)
        torch.cuda.synchronize()
        assert dec.status() == csa.CSA_OK, csa.last_error()
        return o, i, c

    ref = {}
    for k, (db, lh) in enumerate(batches):
        for host in (True, False):
            fresh = csa.Decoder(cfg, maxB, S, max_len)
            ref[k, host] = run(fresh, db, lh if host else None)
            fresh.close()
    dec = csa.Decoder(cfg, maxB, S, max_len)
    for step in range(24):
        k = int(rng.integers(0, len(batches)))
        db, lh = batches[k]
        host = step % 3 != 0
        o, i, c = run(dec, db, lh if host else None)
        r = ref[k, host]
        assert torch.equal(i, r[1]), f"step {step}, batch {k}, host lengths {host}"
        assert torch.equal(c, r[2]), f"step {step}, batch {k}, host lengths {host}"
        assert torch.equal(o, r[0]), f"step {step}, batch {k}, host lengths {host}"
    dec.close()


def test_empty_batch_is_a_noop():
    wl = WORKLOADS["bypass_b16_l256"]
    hb = make_batch(wl, lens=[256])
    db = to_device(hb, DEV)
    dec = csa.Decoder(wl.cfg, 4, 1, 256)
    cb = csa.make_batch_struct(db)
    cb.B = 0
    out = torch.zeros(1, dtype=torch.bfloat16, device=DEV)
    dec.decode_step(cb, out)
    assert dec.last_launch_count() == 0 and dec.status() == csa.CSA_OK


def test_device_side_bad_length_and_index_are_reported():
    wl = Workload("bad", BF16_CFG, B=3, S=1, L=1, seed=95)
    hb = make_batch(wl, lens=[3000, 2500, 600])
    db = to_device(hb, DEV)
    dec = csa.Decoder(wl.cfg, 3, 1, 4096)
    # (1) a length beyond max_context in device memory: that query reads
    # nothing and writes zeros; the others are unaffected
    db["ctx_len"][1] = 5000
    out = torch.full((3, 1, 64, 512), 7.0, dtype=torch.bfloat16, device=DEV)
    dec.decode_step(csa.make_batch_struct(db), out)
    assert dec.status() == csa.CSA_ERR_BAD_INDEX
    assert (out[1] == 0).all()
    ref = oracle.decode(wl.cfg, hb, qids=[0, 2])
    assert_close(out[[0, 2]].float().cpu().numpy().reshape(2, 64, 512), ref["out"], TOL_BF16, "bad-len")
    assert dec.status() == csa.CSA_OK   # the status was cleared by the read
    # (2) caller indices out of range in csa_sparse_attn are skipped and reported
    db["ctx_len"][1] = 2500
    idx = torch.full((3, 1, 512), -1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(3, 1, dtype=torch.int32, device=DEV)
    idx[0, 0, :3] = torch.tensor([5, 10**6, 7])
    cnt[0, 0] = 3
    dec.sparse_attn(csa.make_batch_struct(db), idx, cnt, out)
    assert dec.status() == csa.CSA_ERR_BAD_INDEX
    assert torch.isfinite(out.float()).all()
    # (3) a pool offset that points past the pool
    db["cmp_off"][2] = 10**9
    dec.decode_step(csa.make_batch_struct(db), out)
    assert dec.status() == csa.CSA_ERR_BAD_INDEX
    assert torch.isfinite(out.float()).all()


def test_host_errors_leave_outputs_untouched():
    wl = WORKLOADS["bypass_b16_l256"]
    hb = make_batch(wl)
    db = to_device(hb, DEV)
    dec = csa.Decoder(wl.cfg, 16, 1, 256)
    out = torch.full((16, 1, 64, 512), 3.0, dtype=torch.bfloat16, device=DEV)
    cb = csa.make_batch_struct(db)
    cb.B = 17   # above max_batch
    with pytest.raises(csa.CsaError) as e:
        dec.decode_step(cb, out)
    assert e.value.code == csa.CSA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (out == 3.0).all()
