"""GPU parity of the persistent split grid (one CTA per SM, each working through
several chunks back to back) against the fp64 oracle.

The library runs the bf16 16-heads-per-CTA split persistent when one CTA per
chunk would take several waves.  These small cases force that form (the plan is
checked) and cover what only it has: several items per CTA with their partials
written one tile late, O^T accumulating in alternate tensor-memory buffers,
queries reloaded when a CTA moves to another sequence or head group, ragged
sequence ends inside the stream zeroed before the PV, chunks of one tile, and
poisoned (NaN) tails.  The full-size ragged and long-context workloads run
persistent in tests/test_gpu_parity.py.
"""
import numpy as np
import pytest
import torch

from _parity import compare, run_cuda, run_oracle
from workloads import MlaConfig, make_inputs

pytestmark = pytest.mark.gpu


def cfg_of(B, H, S, **kw):
    return MlaConfig(name=f"persist_b{B}_h{H}_s{S}", dtype="bf16", batch=B, heads=H, s_max=S,
                     hidden=2048, **kw)


def ragged(B, S, seed, edge=(1, 127, 128, 129, 255, 256, 257)):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(1, S + 1, (B,), generator=g, dtype=torch.int32)
    for i, e in enumerate(edge):
        if i < B and e <= S:
            lens[i] = e
    lens[-1] = S
    return lens


def check_persistent(mla, cfg, splits):
    d = mla.dims(cfg.batch, cfg.heads, cfg.s_max, mla.MLA_BF16)
    sp, chunk, persistent = mla.plan(d, splits)
    assert persistent, (sp, chunk)
    assert chunk % 128 == 0
    return sp


@pytest.mark.parametrize("path", ["step", "calls"])
def test_ragged_items_one_tile_chunks(cuda_lib, path):
    """24 sequences x 8 chunks of one tile: 192 one-CTA chunks, persistent."""
    cfg = cfg_of(24, 16, 1024)
    check_persistent(cuda_lib, cfg, 8)
    inp = make_inputs(cfg, seed=501, poison_tail=True, lengths=ragged(24, 1024, 501))
    gpu = run_cuda(inp, num_splits=8, path=path)
    assert gpu["status"] == 0
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


def test_head_groups_change_the_query(cuda_lib):
    """48 heads (three 16-head groups): a CTA's items cross head groups and
    sequences, so its query is reloaded in the middle of its stream."""
    cfg = cfg_of(20, 48, 600)
    check_persistent(cuda_lib, cfg, 4)
    inp = make_inputs(cfg, seed=502, poison_tail=True, lengths=ragged(20, 600, 502))
    gpu = run_cuda(inp, num_splits=4)
    assert gpu["status"] == 0
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


def test_many_short_sequences(cuda_lib):
    """200 sequences of at most 256 rows: items of one tile from many sequences
    per CTA (a query load at almost every item), lengths of 1 and tile edges."""
    cfg = cfg_of(200, 16, 256)
    check_persistent(cuda_lib, cfg, 2)
    inp = make_inputs(cfg, seed=503, poison_tail=True, lengths=ragged(200, 256, 503))
    gpu = run_cuda(inp, num_splits=2)
    assert gpu["status"] == 0
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


def test_long_sequences_many_chunks(cuda_lib):
    """Two sequences of 8192 rows at 128 requested chunks: 64 chunks of one tile
    per sequence, consecutive chunks of one sequence in each CTA."""
    cfg = cfg_of(2, 16, 8192)
    sp = check_persistent(cuda_lib, cfg, 128)
    inp = make_inputs(cfg, seed=504, lengths=torch.tensor([8192, 5000], dtype=torch.int32))
    gpu = run_cuda(inp, num_splits=128)
    assert gpu["status"] == 0 and gpu["splits"] == sp
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


def test_large_scores_rescale_across_items(cuda_lib):
    """Rows scaled x8: the lazy rescale inside an item, and a fresh maximum at
    every item's start."""
    cfg = cfg_of(24, 16, 1024, scaled_row_frac=0.05, scaled_row_gain=8.0)
    check_persistent(cuda_lib, cfg, 8)
    inp = make_inputs(cfg, seed=505, lengths=ragged(24, 1024, 505))
    gpu = run_cuda(inp, num_splits=8)
    assert gpu["status"] == 0
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


def test_repeatable(cuda_lib):
    cfg = cfg_of(24, 16, 1024)
    inp = make_inputs(cfg, seed=506, lengths=ragged(24, 1024, 506))
    a, b = run_cuda(inp, num_splits=8), run_cuda(inp, num_splits=8)
    for k in ("o_c", "lse", "o"):
        np.testing.assert_array_equal(a[k], b[k])
