"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, on the
same seeded inputs, per call (q_abs, q_pe, o_c, lse) and end to end (o).

Small cases span several 32-row tiles, ragged tails and many chunk counts; the
five full-size workloads run in the launch configuration the bench uses (the
library's own chunk choice, or the 128 chunks the long-context workload asks
for), with the oracle on every sequence or, for the largest, on sampled ones.
"""
import numpy as np
import pytest
import torch

from _parity import compare, run_cuda, run_oracle
from workloads import (V2LITE_BF16_B4_S65536_LONG, V2LITE_BF16_B8_S4096, V2LITE_BF16_B64_RAGGED,
                       V2LITE_F32_B1_S64, V3_BF16_H128_B32_S16384, MlaConfig, cache_storage,
                       make_inputs)

pytestmark = pytest.mark.gpu


def small(dtype="bf16", B=3, H=16, S=200, **kw):
    return MlaConfig(name=f"small_{dtype}_b{B}_h{H}_s{S}", dtype=dtype, batch=B, heads=H, s_max=S,
                     hidden=2048, **kw)


# ------------------------------------------------------------------ small cases
@pytest.mark.parametrize("path", ["step", "calls"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("splits", [0, 1, 2, 7])
def test_small_ragged(cuda_lib, dtype, splits, path):
    cfg = small(dtype)
    inp = make_inputs(cfg, seed=splits, poison_tail=True,
                      lengths=torch.tensor([1, 33, 200], dtype=torch.int32))
    gpu = run_cuda(inp, num_splits=splits, path=path)
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, dtype)
    assert gpu["status"] == 0


@pytest.mark.parametrize("lengths", [[32, 64, 96], [31, 63, 95], [2, 3, 5], [190, 199, 200]])
def test_tile_edges(cuda_lib, lengths):
    cfg = small()
    inp = make_inputs(cfg, seed=5, poison_tail=True, lengths=torch.tensor(lengths, dtype=torch.int32))
    gpu = run_cuda(inp, num_splits=3)
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


@pytest.mark.parametrize("path", ["step", "calls"])
@pytest.mark.parametrize("S,lengths", [(384, [384, 300]), (512, [512, 400]), (640, [640, 555])])
def test_tile_count_parity(cuda_lib, S, lengths, path):
    """One chunk of 3, 4 or 5 tiles: the 16-head kernel reads the last tile's O^T
    blocks in place from its stream ring or again from L2 depending on whether
    the tile count is odd or even; the second sequence's last tile is partial."""
    cfg = small(B=2, S=S)
    inp = make_inputs(cfg, seed=S, poison_tail=True, lengths=torch.tensor(lengths, dtype=torch.int32))
    gpu = run_cuda(inp, num_splits=1, path=path)
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")
    assert gpu["status"] == 0


@pytest.mark.parametrize("H", [32, 128])
@pytest.mark.parametrize("path", ["step", "calls"])
def test_head_groups(cuda_lib, H, path):
    cfg = small(H=H, B=2, S=300)
    inp = make_inputs(cfg, seed=H, lengths=torch.tensor([300, 137], dtype=torch.int32))
    gpu = run_cuda(inp, num_splits=4, path=path)
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


def test_batch_tail_in_projections(cuda_lib):
    """B=19: the projections' batch tiles of 16 have a ragged second tile."""
    cfg = small(B=19, S=64)
    inp = make_inputs(cfg, seed=9)
    gpu = run_cuda(inp)
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


def test_large_scores_stay_finite(cuda_lib):
    """Rows scaled x8 push scores far from zero: the online softmax must rescale."""
    cfg = small(S=512, B=2, scaled_row_frac=0.05, scaled_row_gain=8.0)
    inp = make_inputs(cfg, seed=3)
    gpu = run_cuda(inp, num_splits=5)
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


def test_lengths_out_of_range_are_reported(cuda_lib):
    """A length past the capacity is the cache overflow of the KV-cache page: the
    kernels clamp it and raise an error bit; an empty sequence gives o_c = 0."""
    import head_latent_attention_absorbed_gb300 as mla
    cfg = small(S=96)
    inp = make_inputs(cfg, seed=1, lengths=torch.tensor([96, 96, 96], dtype=torch.int32))
    bad = inp.lengths.clone()
    bad[0] = 500          # overflow -> clamped to 96
    bad[2] = 0            # empty
    inp.lengths = bad
    gpu = run_cuda(inp, num_splits=2)
    assert gpu["status"] & mla.MLA_DEV_LENGTH_OUT_OF_RANGE
    inp.lengths = torch.tensor([96, 96, 96], dtype=torch.int32)
    ref, _ = run_oracle(inp, [0, 1])
    compare({k: v for k, v in gpu.items() if k != "status"}, ref, [0, 1], "bf16")
    assert np.all(gpu["o_c"][2] == 0.0) and np.all(np.isneginf(gpu["lse"][2]))


def test_repeatable(cuda_lib):
    cfg = small()
    inp = make_inputs(cfg, seed=2)
    a, b = run_cuda(inp, 3), run_cuda(inp, 3)
    for k in ("q_abs", "o_c", "lse", "o"):
        np.testing.assert_array_equal(a[k], b[k])


# ------------------------------------------------------------------ the five workloads
def test_v2lite_f32_b1_s64(cuda_lib):
    inp = make_inputs(V2LITE_F32_B1_S64, seed=0)
    gpu = run_cuda(inp)
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "f32")


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("path", ["step", "calls"])
def test_v2lite_bf16_b8_s4096(cuda_lib, seed, path):
    inp = make_inputs(V2LITE_BF16_B8_S4096, seed=seed)
    gpu = run_cuda(inp, path=path)
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


def test_v2lite_bf16_b64_ragged(cuda_lib):
    inp = make_inputs(V2LITE_BF16_B64_RAGGED, seed=0, poison_tail=True)
    gpu = run_cuda(inp)
    assert gpu["status"] == 0
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


def test_v3heads_bf16_h128_b32_s16384(cuda_lib):
    inp = make_inputs(V3_BF16_H128_B32_S16384, seed=0)
    gpu = run_cuda(inp)
    ref, bs = run_oracle(inp, batches=[0, 17, 31])
    compare(gpu, ref, bs, "bf16")
    assert np.all(np.isfinite(gpu["o"]))


def test_v2lite_long_context_128_splits(cuda_lib):
    cfg = V2LITE_BF16_B4_S65536_LONG
    inp = make_inputs(cfg, seed=0)
    gpu = run_cuda(inp, num_splits=cfg.num_splits)
    assert gpu["splits"] >= 128
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "f32"])
def test_captured_step_from_host_memory(cuda_lib, dtype):
    """DecodeStep.capture: a CUDA graph of mla_decode_step whose kernels read the
    step's inputs from pinned host memory and write o there; two replays with
    different host inputs both equal the device-resident eager path bit for bit
    and match the oracle."""
    mla = cuda_lib
    cfg = small(dtype=dtype, B=3, S=300)
    base = make_inputs(cfg, seed=21, poison_tail=True,
                       lengths=torch.tensor([300, 45, 129], dtype=torch.int32))
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, cache_storage(cfg),
                          rope_base=cfg.rope_base, softmax_scale=cfg.softmax_scale)
    cache, w_uk, w_uv = base.cache.cuda(), base.w_uk.cuda(), base.w_uv.cuda()
    hs = step.capture(cache, w_uk, w_uv)
    hs.lengths.copy_(base.lengths)
    hs.positions.copy_(base.positions)
    for seed in (22, 23):
        other = make_inputs(cfg, seed=seed)            # new queries; same cache and weights
        hs.q_nope.copy_(other.q_nope)
        hs.q_rope.copy_(other.q_rope)
        hs.replay()
        torch.cuda.synchronize()
        got = hs.out.double().numpy().copy()
        eager = step.run(other.q_nope.cuda(), other.q_rope.cuda(), cache, base.lengths.cuda(),
                         base.positions.cuda(), w_uk, w_uv)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got, eager.double().cpu().numpy())
        inp = make_inputs(cfg, seed=21, poison_tail=True, lengths=base.lengths)
        inp.q_nope, inp.q_rope = other.q_nope, other.q_rope
        ref, bs = run_oracle(inp)
        from _parity import assert_close
        assert_close("o", got[bs], ref["o"], dtype)
    assert int(step.status.item()) == 0



@pytest.mark.parametrize("dtype,B,H", [("bf16", 70, 16), ("bf16", 5, 128), ("fp8", 67, 32)])
def test_host_memory_step_many_rows_and_heads(cuda_lib, dtype, B, H):
    """The host-memory absorb (one CTA per head, up to 64 query rows per pass):
    more than one pass of rows, a partial last 16-row tile, 128 heads.  A replay
    equals the device-resident eager step bit for bit and matches the oracle."""
    mla = cuda_lib
    cfg = small(dtype=dtype, B=B, H=H, S=160)
    g = torch.Generator().manual_seed(B + H)
    lengths = torch.randint(1, 161, (B,), generator=g, dtype=torch.int32)
    lengths[0] = 160
    inp = make_inputs(cfg, seed=31, poison_tail=True, lengths=lengths)
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, cache_storage(cfg),
                          rope_base=cfg.rope_base, softmax_scale=cfg.softmax_scale)
    cache, w_uk, w_uv = inp.cache.cuda(), inp.w_uk.cuda(), inp.w_uv.cuda()
    hs = step.capture(cache, w_uk, w_uv)
    hs.q_nope.copy_(inp.q_nope)
    hs.q_rope.copy_(inp.q_rope)
    hs.lengths.copy_(inp.lengths)
    hs.positions.copy_(inp.positions)
    hs.out.fill_(float("nan"))
    hs.launch()
    torch.cuda.synchronize()
    got = hs.out.double().numpy().copy()
    q_abs = step.q_abs.double().cpu().numpy()
    eager = step.run(inp.q_nope.cuda(), inp.q_rope.cuda(), cache, inp.lengths.cuda(),
                     inp.positions.cuda(), w_uk, w_uv)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(q_abs, step.q_abs.double().cpu().numpy())
    np.testing.assert_array_equal(got, eager.double().cpu().numpy())
    assert int(step.status.item()) == 0
    ref, bs = run_oracle(inp, batches=[0, 1, B // 2, B - 1])
    from _parity import assert_close
    assert_close("q_abs", q_abs[bs], ref["q_abs"], dtype)
    assert_close("o", got[bs], ref["o"], dtype)


def test_pageable_host_memory_is_refused(cuda_lib):
    """mla_decode_step accepts page-locked host buffers for its inputs and output
    but refuses pageable ones before anything is enqueued."""
    import ctypes
    mla = cuda_lib
    cfg = small(B=2, S=64)
    inp = make_inputs(cfg, seed=24)
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, torch.bfloat16)
    pageable = inp.q_nope.clone()                      # ordinary host memory
    assert not pageable.is_pinned()
    with pytest.raises(ValueError):
        step.run(pageable, inp.q_rope.cuda(), inp.cache.cuda(), inp.lengths.cuda(),
                 inp.positions.cuda(), inp.w_uk.cuda(), inp.w_uv.cuda())
    lib = mla.load()
    d = step.dims
    dev = lambda t: t.cuda()
    qr, cache, ln, ps = dev(inp.q_rope), dev(inp.cache), dev(inp.lengths), dev(inp.positions)
    wuk, wuv = dev(inp.w_uk), dev(inp.w_uv)
    st = lib.mla_decode_step(ctypes.byref(d), pageable.data_ptr(), qr.data_ptr(), wuk.data_ptr(),
                             ps.data_ptr(), 10000.0, cache.data_ptr(), ln.data_ptr(),
                             float(step.scale), 0, wuv.data_ptr(), step.workspace.data_ptr(),
                             step.workspace.numel(), step.q_abs.data_ptr(), step.q_pe.data_ptr(),
                             step.o_c.data_ptr(), None, step.out.data_ptr(), None,
                             torch.cuda.current_stream().cuda_stream)
    assert st == 1                                     # MLA_ERR_INVALID_ARG
    assert b"q_nope" in lib.mla_last_error_message()
