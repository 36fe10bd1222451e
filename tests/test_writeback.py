"""The cache update before a step: csa_cache_writeback scatters each new
token's row into a pool at its slot ("Perf: parallelize the DSpark TP-4 SWA
decode hot tasks", PR description: the KV scatter by slot mapping must commit
every mapping entry, whatever the row count).

CPU: the oracle's definition against properties that fix it (identity
mapping, a permutation and its inverse, padding and out-of-range slots leave
rows alone), and the entry point's host checks.  GPU: bit-exact against the
oracle for bf16 KV rows (16-byte copies), FP8 key rows, fp32 scale rows
(4-byte copies) and an odd row size (byte copies), row counts that are not a
multiple of any tile, padding slots and an out-of-range slot; and the decode
step reading rows that were written this way.
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_indexer_gb300 import build as csa_build
from compressed_sparse_attention_indexer_gb300 import csa

DEV = "cuda:0"


# ---------------------------------------------------------------------------
# CPU: the oracle

def test_identity_mapping_copies_every_row():
    rng = np.random.default_rng(1)
    pool = rng.integers(0, 255, (40, 24), dtype=np.uint8)
    rows = rng.integers(0, 255, (40, 24), dtype=np.uint8)
    out, bad = oracle.cache_writeback(pool, rows, np.arange(40))
    assert not bad and np.array_equal(out, rows)


def test_permutation_then_gather_returns_the_rows():
    rng = np.random.default_rng(2)
    pool = np.zeros((100, 7), np.float32)
    rows = rng.standard_normal((37, 7)).astype(np.float32)
    slot = rng.permutation(100)[:37]
    out, bad = oracle.cache_writeback(pool, rows, slot)
    assert not bad and np.array_equal(out[slot], rows)
    untouched = np.setdiff1d(np.arange(100), slot)
    assert np.array_equal(out[untouched], pool[untouched])


def test_padding_and_out_of_range_slots_leave_the_pool_alone():
    pool = np.arange(30, dtype=np.int32).reshape(10, 3)
    rows = -np.ones((3, 3), np.int32)
    out, bad = oracle.cache_writeback(pool, rows, [-1, 10, 4])
    assert bad
    ref = pool.copy()
    ref[4] = -1
    assert np.array_equal(out, ref)
    out2, bad2 = oracle.cache_writeback(pool, rows, [-1, -5, -1])
    assert not bad2 and np.array_equal(out2, pool)


# ---------------------------------------------------------------------------
# CPU: host checks of the entry point

@pytest.fixture(scope="module")
def L():
    csa_build.build()
    return csa.lib()


def _wb(L, rows=0x10000, rs=256, slot=0x10000, n=4, pool=0x10000, ps=256, prow=10, rb=256):
    return L.csa_cache_writeback(rows, rs, slot, n, pool, ps, prow, rb, None, None)


def test_host_checks(L):
    assert _wb(L, n=0, rows=None, slot=None, pool=None) == csa.CSA_OK      # nothing to do
    assert _wb(L, n=-1) == csa.CSA_ERR_INVALID_ARG
    assert _wb(L, rows=None) == csa.CSA_ERR_INVALID_ARG
    assert _wb(L, slot=None) == csa.CSA_ERR_INVALID_ARG
    assert _wb(L, pool=None) == csa.CSA_ERR_INVALID_ARG
    assert _wb(L, rs=128) == csa.CSA_ERR_INVALID_ARG                        # stride below the row
    assert _wb(L, ps=100) == csa.CSA_ERR_INVALID_ARG
    assert _wb(L, prow=-1) == csa.CSA_ERR_INVALID_ARG
    assert csa.last_error()


# ---------------------------------------------------------------------------
# GPU parity

def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    csa_build.build()
    torch.cuda.set_device(0)


def _case(rows_cpu, pool_cpu, slot_np):
    rows = rows_cpu.to(DEV)
    pool = pool_cpu.to(DEV)
    slot = torch.from_numpy(np.asarray(slot_np, np.int64)).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa.cache_writeback(rows, slot, pool, status)
    torch.cuda.synchronize()
    as_bytes = lambda t: t.contiguous().view(torch.uint8).numpy().reshape(t.shape[0], -1)
    ref, bad = oracle.cache_writeback(as_bytes(pool_cpu), as_bytes(rows_cpu), slot_np)
    got = as_bytes(pool.cpu())
    assert np.array_equal(got, ref)
    assert int(status.item()) == (1 if bad else 0)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,width", [(torch.bfloat16, 576), (torch.uint8, 128),
                                         (torch.float32, 1), (torch.uint8, 6)])
@pytest.mark.parametrize("n", [1, 33, 64, 1000])
def test_writeback_matches_oracle(dtype, width, n):
    _gpu()
    g = torch.Generator().manual_seed(n * 7 + width)
    prow = 3 * n + 5
    if dtype == torch.uint8:
        rows = torch.randint(0, 256, (n, width), generator=g, dtype=torch.uint8)
        pool = torch.randint(0, 256, (prow, width), generator=g, dtype=torch.uint8)
    else:
        rows = torch.randn(n, width, generator=g).to(dtype)
        pool = torch.randn(prow, width, generator=g).to(dtype)
    rng = np.random.default_rng(n + width)
    slot = rng.permutation(prow)[:n].astype(np.int64)
    slot[::7] = -1                   # padding tokens
    _case(rows, pool, slot)
    if n > 2:                        # one slot past the pool
        slot[1] = prow
        _case(rows, pool, slot)


@pytest.mark.gpu
def test_written_rows_are_what_the_step_reads():
    # write only the window rows of a batch into a NaN-filled raw pool by slot
    # mapping (as the cache update before the step does), then decode: the
    # output equals the oracle on the original pool, so the step read exactly
    # the rows written
    _gpu()
    from compressed_sparse_attention_indexer_gb300.workloads import BF16_CFG, Workload, make_batch, to_device
    from helpers import TOL_BF16, assert_close
    lens = [700, 3000, 130]
    S = 2
    wl = Workload("wb", BF16_CFG, B=3, S=S, L=1, seed=77)
    hb = make_batch(wl, lens=lens, gap_rows=1)
    db = to_device(hb, DEV)
    ref = oracle.decode(BF16_CFG, hb)
    rows_needed = []
    for b, L in enumerate(lens):
        lo = max(0, L - S - BF16_CFG.win + 1)
        rows_needed += [int(hb["raw_off"][b]) + r for r in range(lo, L)]
    slot = torch.tensor(rows_needed, dtype=torch.int64, device=DEV)
    src = db["raw_kv"][slot].contiguous()            # the new tokens' rows, in token order
    pool = torch.full_like(db["raw_kv"], float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa.cache_writeback(src, slot, pool, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    db2 = dict(db)
    db2["raw_kv"] = pool
    dec = csa.Decoder(BF16_CFG, 3, S, 4096)
    out = torch.empty(3, S, 64, 512, dtype=torch.bfloat16, device=DEV)
    dec.decode_step(csa.make_batch_struct(db2), out)
    assert dec.status() == csa.CSA_OK
    assert_close(out.float().cpu().numpy().reshape(3 * S, 64, 512), ref["out"], TOL_BF16, "writeback")
