"""GPU parity of the split kernel's two operand forms at head counts that are a
multiple of 64, against the fp64 oracle.

By default (mla_set_split_parts(0)) a bf16 cache with 64 or 128 heads runs the
64-heads-per-CTA instance, which hands the query and the softmax weights P to
the tensor core as one bf16 part each; mla_set_split_parts(2) restores the
hi + lo parts (32 heads per CTA).  Both must meet the bf16 tolerances on the
V3 head count ("Multi-Head Latent Attention", 3.1: 128 heads) at full size and
on small ragged cases with poisoned tails, tile edges and several chunk
counts.  The two-part form must also hold with rows of large magnitude.
"""
import numpy as np
import pytest
import torch

from _parity import compare, run_cuda, run_oracle
from workloads import V3_BF16_H128_B32_S16384, MlaConfig, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[0, 2], ids=["parts_default", "parts_hilo"])
def parts(request, cuda_lib):
    cuda_lib.set_split_parts(request.param)
    try:
        yield request.param
    finally:
        cuda_lib.set_split_parts(0)


def small(B, H, S, **kw):
    return MlaConfig(name=f"h{H}_b{B}_s{S}", dtype="bf16", batch=B, heads=H, s_max=S,
                     hidden=2048, **kw)


def test_heads_per_cta_follows_the_switch(cuda_lib):
    mla = cuda_lib
    d = lambda H, dt=mla.MLA_BF16: mla.dims(2, H, 256, dt)
    try:
        assert [mla.heads_per_cta(d(H)) for H in (16, 32, 48, 64, 128)] == [16, 32, 16, 64, 64]
        assert mla.heads_per_cta(d(128, mla.MLA_FP8_E4M3)) == 16
        mla.set_split_parts(2)
        assert [mla.heads_per_cta(d(H)) for H in (16, 32, 48, 64, 128)] == [16, 32, 16, 32, 32]
        with pytest.raises(mla.MlaError):
            mla.set_split_parts(1)
    finally:
        mla.set_split_parts(0)


@pytest.mark.parametrize("path", ["step", "calls"])
@pytest.mark.parametrize("H,S,lengths,splits", [
    (64, 300, [1, 129, 300], 0),
    (64, 300, [128, 127, 257], 3),
    (128, 200, [200, 61, 33], 2),
    (128, 520, [520, 384, 5], 1),
    (128, 1100, [1100, 700, 999], 7),
])
def test_small_ragged(parts, path, H, S, lengths, splits):
    cfg = small(len(lengths), H, S)
    inp = make_inputs(cfg, seed=H + S + splits, poison_tail=True,
                      lengths=torch.tensor(lengths, dtype=torch.int32))
    gpu = run_cuda(inp, num_splits=splits, path=path)
    assert gpu["status"] == 0
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


def test_v3heads_full_size(parts):
    inp = make_inputs(V3_BF16_H128_B32_S16384, seed=0)
    gpu = run_cuda(inp)
    assert gpu["status"] == 0
    ref, bs = run_oracle(inp, batches=[0, 13, 31])
    compare(gpu, ref, bs, "bf16")


def test_large_rows_with_two_parts(cuda_lib):
    """5 % of the rows scaled x8 at 128 heads: the hi + lo form stays within the
    bf16 tolerances (scores spread over tens of units)."""
    cuda_lib.set_split_parts(2)
    try:
        cfg = small(3, 128, 2048, scaled_row_frac=0.05, scaled_row_gain=8.0)
        inp = make_inputs(cfg, seed=64, lengths=torch.tensor([2048, 1500, 777], dtype=torch.int32))
        gpu = run_cuda(inp, num_splits=4)
    finally:
        cuda_lib.set_split_parts(0)
    assert gpu["status"] == 0
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


def test_forms_agree_and_repeat(cuda_lib):
    """The two forms compute the same attention (to bf16 rounding), and each is
    repeatable bit for bit."""
    cfg = small(3, 128, 700)
    inp = make_inputs(cfg, seed=65, lengths=torch.tensor([700, 650, 300], dtype=torch.int32))
    runs = {}
    try:
        for p in (0, 2, 0):
            cuda_lib.set_split_parts(p)
            runs.setdefault(p, []).append(run_cuda(inp, num_splits=3))
    finally:
        cuda_lib.set_split_parts(0)
    for k in ("o_c", "lse", "o"):
        np.testing.assert_array_equal(runs[0][0][k], runs[0][1][k])
        a, b = runs[0][0][k], runs[2][0][k]
        assert np.linalg.norm(a - b) <= 5e-3 * np.linalg.norm(b)
