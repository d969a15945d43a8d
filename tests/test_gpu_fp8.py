"""GPU parity of the FP8 (E4M3) latent cache: the decode step through the C ABI
against the fp64 oracle on the same E4M3 values (the oracle decodes the codes
itself), per call and end to end, with the bf16 tolerances; and the cache
append writing E4M3 rows.

Small cases span several 128-row tiles, ragged and poisoned tails and many
chunk counts; the four FP8 workloads run in the bench's launch configuration
with the oracle on every sequence or, for the largest, on sampled ones.
"""
import numpy as np
import pytest
import torch

from _parity import compare, run_cuda, run_oracle
from oracle import mla_oracle as O
from workloads import (FP8, V2LITE_FP8_B4_S65536_LONG, V2LITE_FP8_B8_S4096, V2LITE_FP8_B64_RAGGED,
                       V3_FP8_H128_B32_S16384, MlaConfig, make_append_inputs, make_inputs)

pytestmark = pytest.mark.gpu


def small(B=3, H=16, S=300, **kw):
    return MlaConfig(name=f"small_fp8_b{B}_h{H}_s{S}", dtype="fp8", batch=B, heads=H, s_max=S,
                     hidden=2048, **kw)


@pytest.mark.parametrize("path", ["step", "calls"])
@pytest.mark.parametrize("splits", [0, 1, 2, 7])
def test_small_ragged(cuda_lib, splits, path):
    cfg = small()
    inp = make_inputs(cfg, seed=40 + splits, poison_tail=True,
                      lengths=torch.tensor([1, 130, 300], dtype=torch.int32))
    gpu = run_cuda(inp, num_splits=splits, path=path)
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "fp8")
    assert gpu["status"] == 0


@pytest.mark.parametrize("lengths", [[127, 128, 129], [255, 256, 257], [2, 3, 5], [8, 136, 264]])
def test_tile_edges(cuda_lib, lengths):
    cfg = small()
    inp = make_inputs(cfg, seed=45, poison_tail=True, lengths=torch.tensor(lengths, dtype=torch.int32))
    gpu = run_cuda(inp, num_splits=2)
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "fp8")
    assert gpu["status"] == 0


@pytest.mark.parametrize("H", [32, 128])
def test_head_groups(cuda_lib, H):
    cfg = small(H=H, B=2, S=400)
    inp = make_inputs(cfg, seed=H, lengths=torch.tensor([400, 137], dtype=torch.int32))
    gpu = run_cuda(inp, num_splits=3)
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "fp8")


def test_large_scores_stay_finite(cuda_lib):
    """Rows scaled x8 push scores far from zero: the online softmax must rescale."""
    cfg = small(S=700, B=2, scaled_row_frac=0.05, scaled_row_gain=8.0)
    inp = make_inputs(cfg, seed=46)
    gpu = run_cuda(inp, num_splits=3)
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "fp8")


def test_repeatable(cuda_lib):
    inp = make_inputs(small(), seed=47)
    a, b = run_cuda(inp, 3), run_cuda(inp, 3)
    for k in ("o_c", "lse", "o"):
        np.testing.assert_array_equal(a[k], b[k])


@pytest.mark.parametrize("path", ["step", "calls"])
def test_v2lite_fp8_b8_s4096(cuda_lib, path):
    inp = make_inputs(V2LITE_FP8_B8_S4096, seed=0)
    gpu = run_cuda(inp, path=path)
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "fp8")


def test_v2lite_fp8_b64_ragged(cuda_lib):
    inp = make_inputs(V2LITE_FP8_B64_RAGGED, seed=0, poison_tail=True)
    gpu = run_cuda(inp)
    assert gpu["status"] == 0
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "fp8")


def test_v3heads_fp8_h128_b32_s16384(cuda_lib):
    inp = make_inputs(V3_FP8_H128_B32_S16384, seed=0)
    gpu = run_cuda(inp)
    ref, bs = run_oracle(inp, batches=[0, 17, 31])
    compare(gpu, ref, bs, "fp8")


def test_v2lite_fp8_long_context_128_splits(cuda_lib):
    cfg = V2LITE_FP8_B4_S65536_LONG
    inp = make_inputs(cfg, seed=0)
    gpu = run_cuda(inp, num_splits=cfg.num_splits)
    assert gpu["splits"] >= 128
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "fp8")


@pytest.mark.parametrize("B,hidden", [(8, 2048), (32, 7168), (5, 1152)])
def test_cache_append_e4m3_rows(cuda_lib, B, hidden):
    """The appended row is the oracle's row rounded to E4M3: the code must be the
    nearest-even code of the fp64 value, except where that value lies within
    1e-5 (relative) of a rounding midpoint, where either neighbour is a valid
    rounding of the kernel's fp32 sum.  Every other row is untouched."""
    mla = cuda_lib
    cfg = MlaConfig(name="append_fp8", dtype="fp8", batch=B, heads=16, s_max=24, hidden=hidden)
    inp = make_append_inputs(cfg, seed=48)
    cache0 = torch.randn((B, cfg.s_max, cfg.row), generator=torch.Generator().manual_seed(9)).to(FP8)
    cache = cache0.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = mla.dims(B, cfg.heads, cfg.s_max, mla.MLA_FP8_E4M3)
    mla.cache_append(d, inp.x.cuda(), inp.w_kva.cuda(), inp.positions.cuda(), cache, cfg.rope_base,
                     dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = cache.cpu().view(torch.uint8)
    pos = inp.positions.long()
    exact = O.cache_append_row(inp.x.double().numpy(), inp.w_kva.double().numpy(), pos.numpy(),
                               cfg.d_c, cfg.rope_base)
    want = O.e4m3_round(exact)
    codes = got[torch.arange(B), pos].numpy()
    bad = codes != want
    if bad.any():
        # accept the other neighbour only next to a midpoint
        lo = np.minimum(O.e4m3_to_float64(codes), O.e4m3_to_float64(want))
        hi = np.maximum(O.e4m3_to_float64(codes), O.e4m3_to_float64(want))
        mid = 0.5 * (lo + hi)
        near_mid = np.abs(exact - mid) <= 1e-5 * np.abs(exact)
        adjacent = np.abs(codes.astype(int) - want.astype(int)) == 1
        assert np.all((near_mid & adjacent)[bad]), f"{int(bad.sum())} codes off"
    mask = torch.ones((B, cfg.s_max), dtype=torch.bool)
    mask[torch.arange(B), pos] = False
    assert torch.equal(got[mask], cache0.view(torch.uint8)[mask])
