"""The device-side timeout path, driven on purpose and without any fault.

Every wait of the tcgen05 kernels on another thread's progress (an mbarrier
phase) is bounded: when it runs out, the block sets an abort flag that every
role checks, waits for the copies and tensor-core operations it already
started, frees its tensor memory and returns, and the status word records
CSA_ERR_TIMEOUT.  The test hook csa_debug_set_wait_polls(0) makes the
attention tile kernel's consumer waits give up at their first poll, so a step
takes that path whatever the data.  The step must return, csa_get_status must
report CSA_ERR_TIMEOUT, and a normal step afterwards on the same handle must
reproduce, bit for bit, the output of a step run before it.  Nothing here
faults, traps or spins without a bound.  ("Fix: port the DeepSeek-V4 MoE,
hc_pre and prefill fixes to DSpark", PR description: a waiter must not be
able to hold its resources forever.)
"""
import pytest
import torch

from compressed_sparse_attention_indexer_gb300 import build as csa_build
from compressed_sparse_attention_indexer_gb300 import csa
from compressed_sparse_attention_indexer_gb300.workloads import WORKLOADS, make_batch, to_device

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    csa_build.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("host_lens", [True, False])
def test_wait_gives_up_reports_timeout_and_the_next_step_is_clean(host_lens):
    wl = WORKLOADS["topk_b16_l8192"]
    hb = make_batch(wl, lens=[8192, 2100, 700, 129])
    db = to_device(hb, DEV)
    cfg = wl.cfg
    B = hb["B"]
    dec = csa.Decoder(cfg, B, 1, 8192)
    lens_host = hb["ctx_len"].clone() if host_lens else None
    cb = csa.make_batch_struct(db, lens_host)
    out = torch.empty(B, 1, cfg.H, cfg.V, dtype=cfg.torch_dtype, device=DEV)
    idx = torch.empty(B, 1, cfg.topk, dtype=torch.int32, device=DEV)
    cnt = torch.empty(B, 1, dtype=torch.int32, device=DEV)
    dec.decode_step(cb, out, None, idx, cnt)
    assert dec.status() == csa.CSA_OK, csa.last_error()
    first = out.clone()
    for _ in range(3):
        dec.debug_wait_polls(0)
        dec.decode_step(cb, out, None, idx, cnt)
        assert dec.status() == csa.CSA_ERR_TIMEOUT
        dec.sparse_attn(cb, idx, cnt, out)
        assert dec.status() == csa.CSA_ERR_TIMEOUT
        dec.debug_wait_polls(-1)
        out.fill_(float("nan"))
        dec.decode_step(cb, out, None, idx, cnt)
        assert dec.status() == csa.CSA_OK, csa.last_error()
        assert torch.equal(out, first)
    dec.close()
