"""GPU parity of multi-token decode (q_len new tokens per sequence, causal within
the block): mla_absorb_q over B * q_len query rows, mla_decode_attn_multi,
mla_out_proj, against the fp64 oracle's decode_multi_token on the same seeded
inputs, for the bf16, fp32 and FP8 caches."""
import numpy as np
import pytest
import torch

from _parity import assert_close
from oracle import mla_oracle as O
from workloads import (V2LITE_BF16_B8_S4096_Q4, V2LITE_FP8_B8_S4096_Q4, MlaConfig, cache_storage,
                       make_inputs)

pytestmark = pytest.mark.gpu


def run_cuda(inp, num_splits=0):
    import head_latent_attention_absorbed_gb300 as mla
    cfg = inp.cfg
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, cache_storage(cfg), q_len=cfg.q_len,
                          num_splits_requested=num_splits, rope_base=cfg.rope_base,
                          softmax_scale=cfg.softmax_scale)
    d = lambda t: t.cuda().contiguous()
    step.run(d(inp.q_nope), d(inp.q_rope), d(inp.cache), d(inp.lengths), d(inp.positions),
             d(inp.w_uk), d(inp.w_uv))
    torch.cuda.synchronize()
    T = cfg.q_len
    f = lambda t: t.detach().cpu().double().numpy()
    shp = lambda a: a.reshape((cfg.batch, T) + a.shape[1:])
    return dict(q_abs=shp(f(step.q_abs)), q_pe=shp(f(step.q_pe)), o_c=shp(f(step.o_c)),
                lse=shp(f(step.lse)), o=shp(f(step.out)), status=int(step.status.item()))


def run_oracle(inp, batches=None):
    cfg = inp.cfg
    T = cfg.q_len
    bs = list(range(cfg.batch)) if batches is None else list(batches)
    out = {k: [] for k in ("q_abs", "q_pe", "o_c", "lse", "o")}
    for b in bs:
        n = int(inp.lengths[b])
        if inp.cache.dtype == torch.float8_e4m3fn:
            cache = O.e4m3_to_float64(inp.cache[b:b + 1, :n].view(torch.uint8).numpy())
        else:
            cache = inp.cache[b:b + 1, :n].double().numpy()
        qn = inp.q_nope[b * T:(b + 1) * T].double().numpy()[None]
        qr = inp.q_rope[b * T:(b + 1) * T].double().numpy()[None]
        r = O.decode_multi_token(qn, qr, inp.w_uk.double().numpy(), inp.w_uv.double().numpy(),
                                 cache, np.array([n]), T, cfg.softmax_scale, cfg.rope_base)
        for k in out:
            out[k].append(r[k][0])
    return {k: np.stack(v) for k, v in out.items()}, bs


def compare(gpu, ref, bs, dtype):
    for k in ("q_abs", "q_pe", "o_c", "lse", "o"):
        assert_close(k, gpu[k][bs], ref[k], dtype)


def small(dtype, q_len, B=3, S=300, H=16):
    return MlaConfig(name=f"mtp_{dtype}_q{q_len}", dtype=dtype, batch=B, heads=H, s_max=S,
                     hidden=2048, q_len=q_len)


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "f32"])
@pytest.mark.parametrize("q_len", [2, 4])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_small_multi_token(cuda_lib, dtype, q_len, splits):
    cfg = small(dtype, q_len)
    inp = make_inputs(cfg, seed=60 + q_len, poison_tail=True,
                      lengths=torch.tensor([q_len, 129, 300], dtype=torch.int32))
    gpu = run_cuda(inp, splits)
    assert gpu["status"] == 0
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, dtype)


def test_q_len_one_is_ordinary_decode(cuda_lib):
    """q_len = 1 through mla_decode_attn_multi equals mla_decode_attn bit for bit."""
    import head_latent_attention_absorbed_gb300 as mla
    cfg = small("bf16", 1)
    inp = make_inputs(cfg, seed=63, lengths=torch.tensor([17, 200, 300], dtype=torch.int32))
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, torch.bfloat16, num_splits_requested=3)
    d = lambda t: t.cuda().contiguous()
    step.run_calls(d(inp.q_nope), d(inp.q_rope), d(inp.cache), d(inp.lengths), d(inp.positions),
                   d(inp.w_uk), d(inp.w_uv))
    o_c = torch.empty_like(step.o_c)
    mla.decode_attn_multi(step.dims, 1, step.q_abs, step.q_pe, d(inp.cache), d(inp.lengths), o_c,
                          step.workspace, step.scale, 3)
    torch.cuda.synchronize()
    assert torch.equal(o_c, step.o_c)


def test_short_sequence_is_reported(cuda_lib):
    """A sequence shorter than q_len cannot hold the step's tokens: error bit."""
    import head_latent_attention_absorbed_gb300 as mla
    cfg = small("bf16", 4, B=2, S=64)
    inp = make_inputs(cfg, seed=64, lengths=torch.tensor([3, 64], dtype=torch.int32))
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, torch.bfloat16, q_len=4)
    d = lambda t: t.cuda().contiguous()
    step.run(d(inp.q_nope), d(inp.q_rope), d(inp.cache), d(inp.lengths), d(inp.positions),
             d(inp.w_uk), d(inp.w_uv))
    torch.cuda.synchronize()
    assert int(step.status.item()) & mla.MLA_DEV_LENGTH_OUT_OF_RANGE


@pytest.mark.parametrize("cfg", [V2LITE_BF16_B8_S4096_Q4, V2LITE_FP8_B8_S4096_Q4],
                         ids=["bf16", "fp8"])
def test_bench_shape_four_tokens(cuda_lib, cfg):
    inp = make_inputs(cfg, seed=0)
    gpu = run_cuda(inp)
    assert gpu["status"] == 0
    ref, bs = run_oracle(inp, batches=[0, 5])
    compare(gpu, ref, bs, cfg.dtype)


@pytest.mark.parametrize("H,q_len,parts", [(32, 4, 0), (32, 2, 0), (128, 2, 0), (48, 2, 0),
                                           (48, 4, 0), (64, 3, 0), (128, 3, 0), (128, 2, 2)])
def test_multi_token_head_groups(cuda_lib, H, q_len, parts):
    """Several head groups with several tokens: 32-head CTAs (hi + lo parts), paired
    tokens at 48 heads, and at 64 and 128 heads the 64-head one-part CTAs (parts 0)
    or the 32-head hi + lo ones (parts 2); each token masks its own later rows."""
    cfg = small("bf16", q_len, B=2, S=300, H=H)
    inp = make_inputs(cfg, seed=70 + H + q_len, poison_tail=True,
                      lengths=torch.tensor([130, 300], dtype=torch.int32))
    cuda_lib.set_split_parts(parts)
    try:
        gpu = run_cuda(inp, 0)
    finally:
        cuda_lib.set_split_parts(0)
    assert gpu["status"] == 0
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_separate_calls_multi_token(cuda_lib, dtype):
    """The three calls (absorb over B*q_len rows, mla_decode_attn_multi, out_proj)
    match the oracle as the one-call step does."""
    import head_latent_attention_absorbed_gb300 as mla
    cfg = small(dtype, 4)
    inp = make_inputs(cfg, seed=90, poison_tail=True,
                      lengths=torch.tensor([4, 129, 300], dtype=torch.int32))
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, cache_storage(cfg), q_len=4)
    d = lambda t: t.cuda().contiguous()
    step.run_calls(d(inp.q_nope), d(inp.q_rope), d(inp.cache), d(inp.lengths), d(inp.positions),
                   d(inp.w_uk), d(inp.w_uv))
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    f = lambda t: t.detach().cpu().double().numpy().reshape((cfg.batch, 4) + tuple(t.shape[1:]))
    gpu = dict(q_abs=f(step.q_abs), q_pe=f(step.q_pe), o_c=f(step.o_c), lse=f(step.lse),
               o=f(step.out))
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_captured_multi_token_step_from_host_memory(cuda_lib, dtype):
    """DecodeStep.capture with four tokens: the kernels read the pinned host inputs
    and write o in place; a replay and a direct launch equal the device-resident
    eager step bit for bit."""
    import numpy as np
    import head_latent_attention_absorbed_gb300 as mla
    cfg = small(dtype, 4)
    inp = make_inputs(cfg, seed=91, poison_tail=True,
                      lengths=torch.tensor([4, 129, 300], dtype=torch.int32))
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, cache_storage(cfg), q_len=4)
    cache, w_uk, w_uv = inp.cache.cuda(), inp.w_uk.cuda(), inp.w_uv.cuda()
    hs = step.capture(cache, w_uk, w_uv)
    hs.q_nope.copy_(inp.q_nope)
    hs.q_rope.copy_(inp.q_rope)
    hs.lengths.copy_(inp.lengths)
    hs.positions.copy_(inp.positions)
    hs.replay()
    torch.cuda.synchronize()
    got = hs.out.double().numpy().copy()
    hs.out.fill_(float("nan"))
    hs.launch()                     # the same step as one direct call
    torch.cuda.synchronize()
    launched = hs.out.double().numpy().copy()
    eager = step.run(inp.q_nope.cuda(), inp.q_rope.cuda(), cache, inp.lengths.cuda(),
                     inp.positions.cuda(), w_uk, w_uv)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got, eager.double().cpu().numpy())
    np.testing.assert_array_equal(launched, got)
    assert int(step.status.item()) == 0


def test_odd_token_count_persistent(cuda_lib):
    """Three tokens per sequence (not paired) on 40 sequences: 120 query groups x
    4 chunks run as the persistent split grid."""
    import head_latent_attention_absorbed_gb300 as mla
    cfg = small("bf16", 3, B=40, S=512)
    d = mla.dims(cfg.batch, cfg.heads, cfg.s_max, mla.MLA_BF16)
    assert mla.plan(mla.query_dims(d, 3), 4)[2]
    g = torch.Generator().manual_seed(61)
    lens = torch.randint(3, 513, (40,), generator=g, dtype=torch.int32)
    lens[0], lens[1] = 3, 129
    inp = make_inputs(cfg, seed=61, poison_tail=True, lengths=lens)
    gpu = run_cuda(inp, 4)
    assert gpu["status"] == 0
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")

