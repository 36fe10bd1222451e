"""The same parity check under the other kernel selections and launch modes.

CSA_INDEXER=mma selects the warp-MMA indexer (the measured baseline of the
tcgen05 one); CSA_ATTN=mma selects the warp-MMA attention kernel (the
measured baseline of the tcgen05 tile kernel + merge);
CSA_TOPK=radix selects the shared-memory Top-K kernel (the measured baseline
of the register one); CSA_PDL=0 launches without programmatic dependent
launch.  All are read once
per process, so each variant runs in a child process.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, numpy as np, torch
sys.path.insert(0, ROOT); sys.path.insert(0, ROOT + "/tests")
import oracle
from compressed_sparse_attention_indexer_gb300 import csa
from compressed_sparse_attention_indexer_gb300.workloads import BF16_CFG, Workload, make_batch, to_device
from helpers import TOL_BF16, assert_close, assert_topk_sets
cfg = BF16_CFG
for lens, host in (([8192, 2049, 300, 5000, 3], True), ([4100, 7, 2052], False)):
    wl = Workload("v", cfg, B=len(lens), S=1, L=1, seed=321)
    hb = make_batch(wl, lens=lens, gap_rows=2)
    db = to_device(hb, "cuda:0")
    B = hb["B"]
    dec = csa.Decoder(cfg, B, 1, 8192)
    out = torch.empty(B, 1, 64, 512, dtype=torch.bfloat16, device="cuda:0")
    idx = torch.empty(B, 1, 512, dtype=torch.int32, device="cuda:0")
    cnt = torch.empty(B, 1, dtype=torch.int32, device="cuda:0")
    lh = hb["ctx_len"].clone() if host else None
    for _ in range(2):
        dec.decode_step(csa.make_batch_struct(db, lh), out, None, idx, cnt)
    assert dec.status() == csa.CSA_OK, csa.last_error()
    ref = oracle.decode(cfg, hb)
    assert_topk_sets(idx.cpu().numpy().reshape(B, -1), cnt.cpu().numpy().reshape(-1), ref,
                     lambda q: oracle.query_scores(cfg, hb, q, 0), 512, "variant")
    assert_close(out.float().cpu().numpy().reshape(B, 64, 512), ref["out"], TOL_BF16, "variant")
print("variant ok")
'''


@pytest.mark.parametrize("env", [{"CSA_INDEXER": "mma"}, {"CSA_PDL": "0"},
                                 {"CSA_INDEXER": "mma", "CSA_PDL": "0"}, {"CSA_ATTN": "mma"},
                                 {"CSA_ATTN": "mma", "CSA_PDL": "0"}, {"CSA_TOPK": "radix"}])
def test_variant_parity(env):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    code = "ROOT = %r\n" % ROOT + CHILD
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, **env), cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "variant ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]


# FP8 keys under the indexer's other launch shapes: converted items in
# shared memory (CSA_T5_ATMEM=0, two CTAs per SM with one converted item
# each), one CTA per SM (CSA_T5_CTAS=1, converted items in TMEM beside six
# accumulators), and both
CHILD_FP8 = CHILD.replace(
    "cfg = BF16_CFG", "from dataclasses import replace\ncfg = replace(BF16_CFG, idx_dtype=\"fp8\")")


@pytest.mark.parametrize("env", [{"CSA_T5_ATMEM": "0"}, {"CSA_T5_CTAS": "1"},
                                 {"CSA_T5_ATMEM": "0", "CSA_T5_CTAS": "1"}])
def test_fp8_indexer_launch_shapes(env):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    code = "ROOT = %r\n" % ROOT + CHILD_FP8
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, **env), cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "variant ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]


CHILD_SPLIT = r'''
import sys, numpy as np, torch
sys.path.insert(0, ROOT)
from compressed_sparse_attention_indexer_gb300 import csa
from compressed_sparse_attention_indexer_gb300.workloads import WORKLOADS, make_batch, to_device
wl = WORKLOADS["long_ragged_b64"]
hb = make_batch(wl)
db = to_device(hb, "cuda:0")
cfg = wl.cfg
B = hb["B"]
dec = csa.Decoder(cfg, B, 1, 65536)
out = torch.empty(B, 1, cfg.H, cfg.V, dtype=cfg.torch_dtype, device="cuda:0")
idx = torch.empty(B, 1, cfg.topk, dtype=torch.int32, device="cuda:0")
cnt = torch.empty(B, 1, dtype=torch.int32, device="cuda:0")
lh = hb["ctx_len"].clone()  # the struct holds its pointer: keep it alive
cb = csa.make_batch_struct(db, lh)
for _ in range(3):
    dec.decode_step(cb, out, None, idx, cnt)
assert dec.status() == csa.CSA_OK, csa.last_error()
np.savez(OUT, out=out.float().cpu().numpy(), idx=idx.cpu().numpy(), cnt=cnt.cpu().numpy())
print("split ok")
'''


def _split_run(tmp_path, name, env):
    out = str(tmp_path / (name + ".npz"))
    code = "ROOT = %r\nOUT = %r\n" % (ROOT, out) + CHILD_SPLIT
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, **env), cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "split ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
    import numpy as np
    return np.load(out)


@pytest.mark.parametrize("env", [{"CSA_TILE_WEIGHT": "2:1"}, {"CSA_TILE_WEIGHT": "1:1"},
                                 {"CSA_EARLY_SPLIT": "1"}])
def test_job_split_only_regroups_segments(env, tmp_path):
    """The split of the attention job lists over the tile CTAs (weights of the
    CTAs that start beside the Top-K blocks, or the W / C split) only changes
    which jobs share a segment: on the full long-context batch the Top-K
    output is bit-identical to the default split's and the output agrees
    within the bf16 tolerance (the default split is checked against the
    oracle in test_gpu_parity)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from helpers import TOL_BF16, assert_close
    base = _split_run(tmp_path, "default", {})
    var = _split_run(tmp_path, "variant", env)
    assert (base["idx"] == var["idx"]).all() and (base["cnt"] == var["cnt"]).all()
    B = base["out"].shape[0]
    assert_close(var["out"].reshape(B, 64, 512), base["out"].reshape(B, 64, 512), TOL_BF16, "split")
