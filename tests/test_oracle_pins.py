"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test states a closed form, an invariant, a textbook/library routine, an
independently written brute force, or a hand-worked example.  Together they
are chosen so that a dropped term, a wrong sign or index, or a transposed
operand anywhere in the oracle fails at least one of them.  No GPU needed.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from compressed_sparse_attention_indexer_gb300.workloads import (
    CsaConfig, Dists, Workload, WORKLOADS, make_batch)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(7)


# --------------------------------------------------------------------------
# indexer score

def test_scores_unit_vector_keys(oracle_mod):
    # k_j = e_{d_j}: q.k_j = q[:, d_j], so score_j = sum_h w_h max(0, q[h, d_j]).
    Hi, Di = 5, 7
    q = rng.standard_normal((Hi, Di))
    w = rng.uniform(0, 1, Hi)
    dsel = [3, 0, 6, 3, 1]
    k = np.zeros((len(dsel), Di))
    for j, d in enumerate(dsel):
        k[j, d] = 1.0
    got = oracle_mod.index_scores(q, w, k)
    for j, d in enumerate(dsel):
        expect = sum(w[h] * max(0.0, q[h, d]) for h in range(Hi))
        assert got[j] == pytest.approx(expect, abs=1e-15)


def test_scores_relu_and_homogeneity(oracle_mod):
    # One head, w = 1: score(alpha*q) = alpha*|q|^2 for alpha > 0, 0 for alpha < 0.
    q = rng.standard_normal((1, 9))
    n2 = float(q[0] @ q[0])
    k = np.stack([2.0 * q[0], -3.0 * q[0], 0.5 * q[0]])
    got = oracle_mod.index_scores(q, np.ones(1), k)
    np.testing.assert_allclose(got, [2.0 * n2, 0.0, 0.5 * n2], rtol=1e-14, atol=1e-14)


def test_scores_linear_in_w_and_row_permutation(oracle_mod):
    Hi, Di, n = 6, 16, 40
    q = rng.standard_normal((Hi, Di))
    k = rng.standard_normal((n, Di))
    w1, w2 = rng.uniform(0, 1, Hi), rng.uniform(0, 1, Hi)
    s1 = oracle_mod.index_scores(q, w1, k)
    s2 = oracle_mod.index_scores(q, w2, k)
    s12 = oracle_mod.index_scores(q, w1 + w2, k)
    np.testing.assert_allclose(s12, s1 + s2, rtol=1e-12, atol=1e-12)
    perm = rng.permutation(n)
    np.testing.assert_array_equal(oracle_mod.index_scores(q, w1, k[perm]), s1[perm])
    # a head with w_h = 0 drops out entirely
    w3 = w1.copy()
    w3[2] = 0.0
    np.testing.assert_allclose(oracle_mod.index_scores(np.delete(q, 2, 0), np.delete(w3, 2), k),
                               oracle_mod.index_scores(q, w3, k), rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# Top-K

def _select_by_repeated_argmax(scores, K):
    """Independent brute force: take the best remaining K times, ties to the lower index."""
    left = list(range(len(scores)))
    out = []
    for _ in range(min(K, len(scores))):
        best = left[0]
        for j in left[1:]:
            if scores[j] > scores[best]:
                best = j
        out.append(best)
        left.remove(best)
    return sorted(out)


def test_topk_against_brute_force_small(oracle_mod):
    for n in range(1, 65):
        # quantised scores so that exact ties are common
        s = np.round(rng.standard_normal(n) * 3) / 2
        for K in sorted({1, 8, max(n - 1, 1), n, n + 5}):
            got = oracle_mod.topk(s, K)
            assert got.tolist() == _select_by_repeated_argmax(s, K), (n, K)


def test_topk_all_equal_takes_lowest_indices(oracle_mod):
    for n, K in [(10, 3), (300, 256), (2048, 512)]:
        assert oracle_mod.topk(np.zeros(n), K).tolist() == list(range(K))


def test_topk_signed_zero_is_a_tie(oracle_mod):
    s = np.array([-0.0, 0.0, -0.0, 0.0, -1.0])
    assert oracle_mod.topk(s, 2).tolist() == [0, 1]
    assert oracle_mod.topk(s[::-1].copy(), 2).tolist() == [1, 2]


@pytest.mark.parametrize("n", [255, 256, 257, 1023, 1024, 1025, 16384])
def test_topk_planted_tail_candidates(oracle_mod, n):
    # the true top candidates sit beyond positions 256 / 1024 (a partially
    # ordered prefix would miss them)
    K = min(64, n)
    s = rng.uniform(-1, 0, n)
    planted = np.sort(rng.choice(np.arange(n // 2, n), size=K, replace=False))
    s[planted] = rng.uniform(1, 2, K)
    assert oracle_mod.topk(s, K).tolist() == planted.tolist()


# --------------------------------------------------------------------------
# attention over a row set

def test_attend_single_row(oracle_mod):
    q = rng.standard_normal((3, 10))
    row = rng.standard_normal((1, 10))
    o, lse = oracle_mod.attend(q, row, 6, 0.3)
    np.testing.assert_array_equal(o, np.broadcast_to(row[0, :6], (3, 6)))
    np.testing.assert_allclose(lse, 0.3 * q @ row[0], rtol=1e-14)


def test_attend_equal_rows_and_zero_query(oracle_mod):
    q = rng.standard_normal((2, 8))
    row = rng.standard_normal(8)
    o, lse = oracle_mod.attend(q, np.tile(row, (5, 1)), 5, 0.7)
    np.testing.assert_allclose(o, np.broadcast_to(row[:5], (2, 5)), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(lse, 0.7 * q @ row + math.log(5), rtol=1e-14)
    rows = rng.standard_normal((9, 8))
    o0, lse0 = oracle_mod.attend(np.zeros((2, 8)), rows, 5, 0.7)
    np.testing.assert_allclose(o0, np.broadcast_to(rows[:, :5].mean(0), (2, 5)), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse0, math.log(9), rtol=1e-14)


def test_attend_matches_torch_sdpa(oracle_mod):
    H, D, V, n = 4, 24, 16, 33
    q = rng.standard_normal((H, D))
    rows = rng.standard_normal((n, D))
    scale = 1 / math.sqrt(D)
    o, lse = oracle_mod.attend(q, rows, V, scale)
    tq = torch.tensor(q)[None, :, None, :]               # [1, H, 1, D]
    tk = torch.tensor(rows)[None, None].expand(1, H, n, D)
    tv = torch.tensor(rows[:, :V])[None, None].expand(1, H, n, V)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)[0, :, 0]
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-13)
    ref_lse = torch.logsumexp(torch.tensor(q) @ torch.tensor(rows).T * scale, dim=1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=1e-13)


def _merge(parts):
    """Log-sum-exp merge of (o, lse) stream partials; empty streams have lse = -inf."""
    lses = np.stack([p[1] for p in parts])
    m = lses.max(0)
    wts = np.exp(lses - m)
    tot = wts.sum(0)
    o = sum(wts[i][:, None] * parts[i][0] for i in range(len(parts))) / tot[:, None]
    return o, m + np.log(tot)


def test_union_softmax_equals_stream_merge_and_merge_is_associative(oracle_mod):
    H, D, V = 3, 12, 8
    q = rng.standard_normal((H, D))
    a, b, c = (rng.standard_normal((n, D)) * s for n, s in [(7, 1.0), (13, 0.5), (4, 2.0)])
    pa, pb, pc = (oracle_mod.attend(q, x, V, 0.4) for x in (a, b, c))
    union = oracle_mod.attend(q, np.concatenate([a, b, c]), V, 0.4)
    merged = _merge([pa, pb, pc])
    np.testing.assert_allclose(merged[0], union[0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(merged[1], union[1], rtol=1e-13)
    left = _merge([_merge([pa, pb]), pc])
    right = _merge([pa, _merge([pb, pc])])
    np.testing.assert_allclose(left[0], right[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(left[1], right[1], rtol=0, atol=1e-12)
    # an empty stream (lse = -inf) leaves the merge unchanged
    empty = oracle_mod.attend(q, np.zeros((0, D)), V, 0.4)
    assert np.all(np.isneginf(empty[1])) and not empty[0].any()
    m2 = _merge([pa, empty])
    np.testing.assert_allclose(m2[0], pa[0], rtol=1e-15, atol=1e-15)


# --------------------------------------------------------------------------
# inverse RoPE

def _rotate_complex(x, pos, R, base, sign):
    """Rotation of interleaved pairs written with complex numbers."""
    V = x.shape[-1]
    z = x[..., V - R::2] + 1j * x[..., V - R + 1::2]
    theta = pos * base ** (-2.0 * np.arange(R // 2) / R)
    z = z * np.exp(sign * 1j * theta)
    y = x.copy()
    y[..., V - R::2] = z.real
    y[..., V - R + 1::2] = z.imag
    return y


def test_inverse_rope_identity_at_pos0(oracle_mod):
    o = rng.standard_normal((3, 20))
    np.testing.assert_array_equal(oracle_mod.inverse_rope(o, 0, 8, 10000.0), o)


@pytest.mark.parametrize("pos", [1, 7, 1234, 65535])
def test_inverse_rope_is_rotation_by_minus_angle(oracle_mod, pos):
    H, V, R = 4, 24, 8
    o = rng.standard_normal((H, V))
    got = oracle_mod.inverse_rope(o, pos, R, 10000.0)
    np.testing.assert_allclose(got, _rotate_complex(o, pos, R, 10000.0, -1), rtol=1e-12, atol=1e-12)
    # untouched value dims, norm per pair preserved, RoPE then inverse is the identity
    np.testing.assert_array_equal(got[:, :V - R], o[:, :V - R])
    n0 = o[:, V - R::2] ** 2 + o[:, V - R + 1::2] ** 2
    n1 = got[:, V - R::2] ** 2 + got[:, V - R + 1::2] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12)
    fwd = _rotate_complex(o, pos, R, 10000.0, +1)
    np.testing.assert_allclose(oracle_mod.inverse_rope(fwd, pos, R, 10000.0), o, rtol=1e-10, atol=1e-11)


def test_inverse_rope_quarter_turn_is_signed_swap(oracle_mod):
    # base chosen so that pair 1 turns by exactly pi/2 at pos = 1: theta_1 = base^(-2/4)
    base = (2 / math.pi) ** 2
    o = np.array([[0.0, 0.0, 3.0, 5.0]])   # V = 4, R = 4: pairs (0,1) angle 1, (2,3) angle pi/2
    got = oracle_mod.inverse_rope(o, 1, 4, base)
    np.testing.assert_allclose(got[0, 2:], [5.0, -3.0], atol=1e-15)


# --------------------------------------------------------------------------
# the whole decode step

def _hand_batch(inp, K):
    cfg = CsaConfig(H=1, D=4, V=2, Hi=1, Di=2, ratio=4, topk=K, win=1, dtype="f32", scale=1.0)
    raw = torch.zeros(8, 4)
    raw[7] = torch.tensor(inp["raw_row_7"])
    b = dict(B=1, S=1, ctx_len=torch.tensor([inp["ctx_len"]], dtype=torch.int32),
             q=torch.tensor(inp["q"], dtype=torch.float32).view(1, 1, 1, 4),
             q_idx=torch.tensor(inp["q_idx"]).view(1, 1, 1, 2), w=torch.tensor(inp["w"]).view(1, 1, 1),
             raw_kv=raw, raw_off=torch.zeros(1, dtype=torch.int64), raw_stride=4,
             cmp_kv=torch.tensor(inp["cmp"]), cmp_off=torch.zeros(1, dtype=torch.int64), cmp_stride=4,
             idx_k=torch.tensor(inp["k_idx"]), idx_off=torch.zeros(1, dtype=torch.int64), idx_stride=2,
             hca_kv=None, hca_off=None, hca_stride=0)
    return cfg, b


def test_hand_worked_example(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_decode.json")))
    for K, key in [(1, "K1"), (2, "K2")]:
        cfg, b = _hand_batch(g["inputs"], K)
        r = oracle_mod.decode(cfg, b, nthreads=1)
        exp = g["expected"][key]
        assert r["topk_idx"][0, :len(exp["topk"])].tolist() == exp["topk"]
        assert int(r["rows_used"][0]) == exp["rows_used"]
        np.testing.assert_allclose(r["out"][0, 0], exp["out"], atol=1e-7)
        assert r["lse"][0, 0] == pytest.approx(exp["lse"], abs=1e-7)


SMALL = CsaConfig(H=4, D=40, V=32, Hi=3, Di=16, ratio=4, topk=6, win=5, dtype="f32")


def _small_wl(cfg=SMALL, S=1, seed=5):
    return Workload("small", cfg, B=1, S=S, L=1, seed=seed)


def test_row_bound_over_many_positions(oracle_mod):
    lens = list(range(1, 60)) + [61, 62, 63, 64, 97, 200]
    wl = _small_wl()
    b = make_batch(wl, lens=lens, gap_rows=1)
    r = oracle_mod.decode(SMALL, b, nthreads=4)
    for i, L in enumerate(lens):
        pos = L - 1
        vis = (pos + 1) // SMALL.ratio
        assert r["rows_used"][i] == min(SMALL.win, pos + 1) + min(vis, SMALL.topk)
        assert r["cnt"][i] == min(vis, SMALL.topk)
        sel = r["topk_idx"][i]
        assert (sel[r["cnt"][i]:] == -1).all()
        assert np.all(np.diff(sel[:r["cnt"][i]]) > 0) and (sel[:r["cnt"][i]] < vis).all()
    assert np.isfinite(r["out"]).all()   # NaN gap rows between requests were never read


def test_bypass_identity(oracle_mod):
    # with vis <= K, scoring everything and keeping min(vis, K) equals the bypass
    lens = [4, 5, 8, 17, 23, 24, 25]            # vis 1..6 with K = 6
    b = make_batch(_small_wl(), lens=lens)
    plain = oracle_mod.decode(SMALL, b, nthreads=2)
    forced = oracle_mod.decode(SMALL, b, nthreads=2, force_score=True)
    np.testing.assert_array_equal(plain["topk_idx"], forced["topk_idx"])
    np.testing.assert_array_equal(plain["out"], forced["out"])
    for i in range(len(lens)):
        assert plain["topk_idx"][i, :plain["cnt"][i]].tolist() == list(range(plain["vis"][i]))


def _dense_reference(cfg, b, bi, s, rows_list):
    """torch SDPA over an explicit row list, then the complex-form inverse rotation."""
    q = b["q"][bi, s].double()
    rows = torch.cat(rows_list).double()
    H, D = q.shape
    n = rows.shape[0]
    o = torch.nn.functional.scaled_dot_product_attention(
        q[None, :, None, :], rows[None, None].expand(1, H, n, D),
        rows[None, None, :, :cfg.V].expand(1, H, n, cfg.V), scale=cfg.softmax_scale)[0, :, 0]
    pos = int(b["ctx_len"][bi]) - b["S"] + s
    return _rotate_complex(o.numpy(), pos, cfg.R, cfg.rope_base, -1)


def test_dense_equivalence_when_window_and_k_cover_everything(oracle_mod):
    # WIN >= pos+1 and K >= vis: the step is dense attention over every raw
    # row [0, pos] and every visible compressed row [0, vis)
    cfg = CsaConfig(H=3, D=24, V=16, Hi=2, Di=8, ratio=4, topk=100, win=64, dtype="f32")
    lens = [1, 3, 4, 9, 30, 64]
    b = make_batch(_small_wl(cfg), lens=lens, raw_keep=64)
    r = oracle_mod.decode(cfg, b, nthreads=2)
    for i, L in enumerate(lens):
        pos = L - 1
        vis = (pos + 1) // 4
        raw_rows = b["raw_kv"][int(b["raw_off"][i]): int(b["raw_off"][i]) + pos + 1]
        cmp_rows = b["cmp_kv"][int(b["cmp_off"][i]): int(b["cmp_off"][i]) + vis]
        ref = _dense_reference(cfg, b, i, 0, [raw_rows, cmp_rows])
        np.testing.assert_allclose(r["out"][i], ref, rtol=1e-10, atol=1e-12)


def test_selected_rows_are_the_planted_ones(oracle_mod):
    # plant key rows aligned with indexer head 0 far in the tail; every other
    # key is anti-aligned, so only the planted rows have positive scores
    cfg = CsaConfig(H=2, D=24, V=16, Hi=2, Di=8, ratio=4, topk=5, win=3, dtype="f32")
    L = 4 * 300
    b = make_batch(_small_wl(cfg), lens=[L])
    qi = b["q_idx"][0, 0]
    qi[1] = qi[0]
    nvis = L // 4
    keys = -torch.rand(nvis, 1) * qi[0][None, :]
    planted = [257, 260, 280, 290, 299]
    for j in planted:
        keys[j] = (1.0 + j / 1000.0) * qi[0]
    off = int(b["idx_off"][0])
    b["idx_k"][off:off + nvis] = keys
    r = oracle_mod.decode(cfg, b, nthreads=1)
    assert r["topk_idx"][0].tolist() == planted
    sc = oracle_mod.query_scores(cfg, b, 0, 0)
    assert (sc[planted] > 0).all() and np.count_nonzero(sc > 0) == len(planted)
    # and the output is dense attention over the window and exactly those rows
    raw0 = int(b["raw_off"][0])
    cmp0 = int(b["cmp_off"][0])
    ref = _dense_reference(cfg, b, 0, 0, [b["raw_kv"][raw0 + L - 3: raw0 + L],
                                          b["cmp_kv"][[cmp0 + j for j in planted]]])
    np.testing.assert_allclose(r["out"][0], ref, rtol=1e-10, atol=1e-12)


def test_duplicated_keys_tie_to_lower_index(oracle_mod):
    cfg = CsaConfig(H=2, D=24, V=16, Hi=2, Di=8, ratio=4, topk=3, win=2, dtype="f32")
    b = make_batch(_small_wl(cfg), lens=[64])
    off = int(b["idx_off"][0])
    qi = b["q_idx"][0, 0]
    b["idx_k"][off:off + 16] = 0.0      # every score 0: one big tie
    best = qi[0].clone()
    for j in (2, 9, 11, 14):
        b["idx_k"][off + j] = best        # four identical best rows
    r = oracle_mod.decode(cfg, b, nthreads=1)
    assert r["topk_idx"][0].tolist() == [2, 9, 11]


def test_multi_token_and_hca_stream(oracle_mod):
    # S queries per request at pos = L - S + s; a third stream holds every
    # visible ratio-r2 row.  Checked against dense SDPA over the row union.
    cfg = CsaConfig(H=2, D=24, V=16, Hi=2, Di=8, ratio=4, topk=4, win=3, hca_ratio=8, dtype="f32")
    wl = Workload("s", cfg, B=2, S=4, L=1, seed=11)
    b = make_batch(wl, lens=[40, 23])
    r = oracle_mod.decode(cfg, b, nthreads=2)
    for q in range(8):
        bi, s = divmod(q, 4)
        L = int(b["ctx_len"][bi])
        pos = L - 4 + s
        vis, vis2 = (pos + 1) // 4, (pos + 1) // 8
        assert r["pos"][q] == pos and r["vis2"][q] == vis2
        assert r["rows_used"][q] == min(3, pos + 1) + min(vis, 4) + vis2
        sel = r["topk_idx"][q, :r["cnt"][q]].tolist()
        sc = oracle_mod.query_scores(cfg, b, bi, s)
        assert sel == _select_by_repeated_argmax(sc, 4)
        raw0, cmp0, h0 = int(b["raw_off"][bi]), int(b["cmp_off"][bi]), int(b["hca_off"][bi])
        rows = [b["raw_kv"][raw0 + pos - min(3, pos + 1) + 1: raw0 + pos + 1],
                b["cmp_kv"][[cmp0 + j for j in sel]], b["hca_kv"][h0:h0 + vis2]]
        np.testing.assert_allclose(r["out"][q], _dense_reference(cfg, b, bi, s, rows), rtol=1e-10, atol=1e-12)


def test_empty_compressed_stream(oracle_mod):
    # pos < ratio - 1: no compressed row is visible; the window alone decides
    cfg = CsaConfig(H=2, D=24, V=16, Hi=2, Di=8, ratio=4, topk=4, win=8, dtype="f32")
    b = make_batch(_small_wl(cfg), lens=[1, 2, 3])
    r = oracle_mod.decode(cfg, b, nthreads=1)
    for i, L in enumerate([1, 2, 3]):
        assert r["vis"][i] == 0 and r["cnt"][i] == 0 and (r["topk_idx"][i] == -1).all()
        raw0 = int(b["raw_off"][i])
        ref = _dense_reference(cfg, b, i, 0, [b["raw_kv"][raw0: raw0 + L]])
        np.testing.assert_allclose(r["out"][i], ref, rtol=1e-10, atol=1e-12)


def test_bf16_storage_is_decoded_exactly(oracle_mod):
    # bf16 inputs: the oracle must read the exact stored values; compare with
    # the same batch upcast to fp32 storage (bf16 -> fp32 is exact)
    cfg16 = CsaConfig(H=2, D=24, V=16, Hi=2, Di=8, ratio=4, topk=4, win=3, dtype="bf16")
    cfg32 = CsaConfig(H=2, D=24, V=16, Hi=2, Di=8, ratio=4, topk=4, win=3, dtype="f32")
    b16 = make_batch(_small_wl(cfg16), lens=[50, 33])
    b32 = {k: (v.float() if isinstance(v, torch.Tensor) and v.dtype == torch.bfloat16 else v)
           for k, v in b16.items()}
    r16 = oracle_mod.decode(cfg16, b16, nthreads=1)
    r32 = oracle_mod.decode(cfg32, b32, nthreads=1)
    np.testing.assert_array_equal(r16["out"], r32["out"])
    np.testing.assert_array_equal(r16["topk_idx"], r32["topk_idx"])


def test_named_workloads_shapes(oracle_mod):
    # the tiny fp32 workload end to end, and visibility counts of the others
    wl = WORKLOADS["tiny_f32"]
    b = make_batch(wl)
    r = oracle_mod.decode(wl.cfg, b, nthreads=1)
    assert r["vis"][0] == 16 and r["cnt"][0] == 8 and r["rows_used"][0] == 16
    assert np.isfinite(r["out"]).all()
    for name, L, vis in [("bypass_b16_l256", 256, 64), ("topk_b16_l8192", 8192, 2048)]:
        assert WORKLOADS[name].L == L and (L - 1 + 1) // WORKLOADS[name].cfg.ratio == vis
