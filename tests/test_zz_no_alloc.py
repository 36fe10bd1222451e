"""The allocation-free indexer + Top-K entry point, csa_indexer_topk_static.

It launches the same kernels as csa_indexer_topk, with its scratch (status
word, work list, score matrix) in the library's static device array instead
of a handle's workspace, so its outputs must equal that entry point's bit for
bit, on consecutive calls that reuse the scratch and with or without host
lengths.  The file is named to be collected after the other test files; each
test here also passes when run alone.
"""
import ctypes

import pytest

from compressed_sparse_attention_indexer_gb300 import csa
from compressed_sparse_attention_indexer_gb300.workloads import BF16_CFG, Workload, make_batch, to_device

DEV = "cuda:0"
SCRATCH_BYTES = 8 << 20


def _fake_batch(B, S):
    a = 0x10000  # any 16-byte aligned value: the host checks dereference nothing
    return csa.CBatch(B=B, S=S, ctx_len=a, ctx_len_host=None, q=a, q_idx=a, w=a,
                      raw_kv=a, raw_off=a, raw_stride=576, raw_rows=10,
                      cmp_kv=a, cmp_off=a, cmp_stride=576, cmp_rows=10,
                      idx_k=a, idx_off=a, idx_stride=128, idx_rows=10,
                      hca_kv=None, hca_off=None, hca_stride=0, hca_rows=0)


def test_oversize_batch_is_rejected_before_any_device_work():
    # 64 x 8 queries x 16384 scores x 4 bytes = 32 MiB of scores > 8 MiB
    cfg = csa.make_config(BF16_CFG, 64, 8, 65536)
    b = _fake_batch(64, 8)
    rc = csa.lib().csa_indexer_topk_static(ctypes.byref(cfg), ctypes.byref(b), 0x10000, 0x10000,
                                           None, None)
    assert rc == csa.CSA_ERR_WORKSPACE
    msg = csa.last_error()
    assert "scratch" in msg and str(SCRATCH_BYTES) in msg and "csa_indexer_topk" in msg


def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from compressed_sparse_attention_indexer_gb300 import build as csa_build
    csa_build.build()
    torch.cuda.set_device(0)
    return torch


@pytest.mark.gpu
@pytest.mark.parametrize("S", [1, 2])
def test_static_entry_matches_indexer_topk_on_consecutive_calls(S):
    torch = _gpu()
    cfg = BF16_CFG
    lens = [8192, 2049, 300, 5000, 3 + S, 6000, 4097, 129]
    B = len(lens)
    wl = Workload("noalloc", cfg, B=B, S=S, L=1, seed=4242 + S)
    hb = make_batch(wl, lens=lens, gap_rows=2)
    db = to_device(hb, DEV)
    dec = csa.Decoder(cfg, B, S, 8192)
    for host_lens in (True, False):
        lh = hb["ctx_len"].clone() if host_lens else None
        cb = csa.make_batch_struct(db, lh)
        ref_idx = torch.full((B, S, cfg.topk), -7, dtype=torch.int32, device=DEV)
        ref_cnt = torch.full((B, S), -7, dtype=torch.int32, device=DEV)
        dec.indexer_topk(cb, ref_idx, ref_cnt)
        assert dec.status() == csa.CSA_OK
        status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
        for call in range(2):
            idx = torch.full((B, S, cfg.topk), -9, dtype=torch.int32, device=DEV)
            cnt = torch.full((B, S), -9, dtype=torch.int32, device=DEV)
            csa.indexer_topk_static(dec.cconfig, cb, idx, cnt, status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0, (host_lens, call)
            assert torch.equal(cnt, ref_cnt), (host_lens, call)
            assert torch.equal(idx, ref_idx), (host_lens, call)


@pytest.mark.gpu
def test_static_entry_reports_a_device_side_bad_length_and_recovers():
    torch = _gpu()
    cfg = BF16_CFG
    wl = Workload("noalloc-bad", cfg, B=3, S=1, L=1, seed=97)
    hb = make_batch(wl, lens=[3000, 2500, 600])
    db = to_device(hb, DEV)
    cc = csa.make_config(cfg, 3, 1, 4096)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    idx = torch.full((3, 1, cfg.topk), -9, dtype=torch.int32, device=DEV)
    cnt = torch.full((3, 1), -9, dtype=torch.int32, device=DEV)
    # a length beyond max_context in device memory: that query is marked bad
    db["ctx_len"][1] = 5000
    csa.indexer_topk_static(cc, csa.make_batch_struct(db), idx, cnt, status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1
    # the next call starts from a cleared status word
    db["ctx_len"][1] = 2500
    csa.indexer_topk_static(cc, csa.make_batch_struct(db), idx, cnt, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.gpu
def test_static_entry_with_an_empty_batch_only_sets_up():
    torch = _gpu()
    cc = csa.make_config(BF16_CFG, 4, 1, 4096)
    b = _fake_batch(0, 1)
    rc = csa.lib().csa_indexer_topk_static(ctypes.byref(cc), ctypes.byref(b), 0x10000, 0x10000,
                                           None, None)
    assert rc == csa.CSA_OK
    torch.cuda.synchronize()
    # with a status word to fill, an empty batch reports a clean status
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream()
    rc = csa.lib().csa_indexer_topk_static(ctypes.byref(cc), ctypes.byref(b), 0x10000, 0x10000,
                                           ctypes.c_void_p(status.data_ptr()),
                                           ctypes.c_void_p(stream.cuda_stream))
    assert rc == csa.CSA_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
