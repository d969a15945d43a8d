"""GPU parity of the two steps around the decode path, through the C ABI, against
the fp64 oracle on the same seeded inputs:

- mla_cache_append: the new token's cache row (fused kv_a_proj down-projection,
  RoPE on its key part at the token's position), written at that position;
- mla_wo_proj: the output projection W^O on the concatenated head outputs.
"""
import numpy as np
import pytest
import torch

from _parity import assert_close, run_oracle
from oracle import mla_oracle as O
from workloads import (MlaConfig, make_append_inputs, make_inputs, make_wo_inputs,
                       V2LITE_BF16_B8_S4096, V3_BF16_H128_B32_S16384, V2LITE_F32_B1_S64)

pytestmark = pytest.mark.gpu


def cfg_of(base, **kw):
    d = dict(name=base.name + "_next", dtype=base.dtype, batch=base.batch, heads=base.heads,
             s_max=base.s_max, hidden=base.hidden)
    d.update(kw)
    return MlaConfig(**d)


def _dt(cfg):
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


@pytest.mark.parametrize("cfg", [
    cfg_of(V2LITE_BF16_B8_S4096, s_max=64),
    cfg_of(V3_BF16_H128_B32_S16384, s_max=64),
    cfg_of(V2LITE_BF16_B8_S4096, batch=19, s_max=40),
    cfg_of(V2LITE_BF16_B8_S4096, batch=5, s_max=24, hidden=1152),
    cfg_of(V2LITE_BF16_B8_S4096, batch=70, s_max=8),
    cfg_of(V2LITE_F32_B1_S64),
], ids=["v2lite_bf16", "v3_bf16", "v2lite_bf16_b19", "hidden1152_b5", "b70", "v2lite_f32"])
def test_cache_append_rows(cuda_lib, cfg):
    mla = cuda_lib
    inp = make_append_inputs(cfg, seed=31)
    dt = _dt(cfg)
    cache0 = torch.randn((cfg.batch, cfg.s_max, cfg.row), generator=torch.Generator().manual_seed(7)).to(dt)
    cache = cache0.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = mla.dims(cfg.batch, cfg.heads, cfg.s_max, mla.dtype_code(dt))
    mla.cache_append(d, inp.x.cuda(), inp.w_kva.cuda(), inp.positions.cuda(), cache, cfg.rope_base,
                     dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = cache.cpu()
    pos = inp.positions.long()
    ref = O.cache_append_row(inp.x.double().numpy(), inp.w_kva.double().numpy(), pos.numpy(),
                             cfg.d_c, cfg.rope_base)
    rows = got[torch.arange(cfg.batch), pos].double().numpy()
    assert_close("appended row", rows, ref, cfg.dtype)
    # every other row is untouched, bit for bit
    mask = torch.ones((cfg.batch, cfg.s_max), dtype=torch.bool)
    mask[torch.arange(cfg.batch), pos] = False
    assert torch.equal(got[mask], cache0[mask])


def test_cache_append_out_of_range_position(cuda_lib):
    mla = cuda_lib
    cfg = cfg_of(V2LITE_BF16_B8_S4096, batch=3, s_max=16)
    inp = make_append_inputs(cfg, seed=32)
    pos = torch.tensor([2, 16, -1], dtype=torch.int32)       # two positions out of range
    cache0 = torch.zeros((cfg.batch, cfg.s_max, cfg.row), dtype=torch.bfloat16)
    cache = cache0.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d = mla.dims(cfg.batch, cfg.heads, cfg.s_max, mla.MLA_BF16)
    mla.cache_append(d, inp.x.cuda(), inp.w_kva.cuda(), pos.cuda(), cache, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & mla.MLA_DEV_LENGTH_OUT_OF_RANGE
    got = cache.cpu()
    assert torch.count_nonzero(got[1]) == 0 and torch.count_nonzero(got[2]) == 0
    ref = O.cache_append_row(inp.x.double().numpy()[:1], inp.w_kva.double().numpy(), [2],
                             cfg.d_c, cfg.rope_base)
    assert_close("in-range row", got[0, 2:3].double().numpy(), ref, "bf16")


def test_append_then_decode(cuda_lib):
    """A token appended at position len_b is attended by the next decode step: the
    step over lengths len_b + 1 matches the oracle on the oracle's appended cache."""
    mla = cuda_lib
    cfg = MlaConfig(name="append_decode", dtype="bf16", batch=4, heads=16, s_max=300,
                    hidden=2048)
    lens = torch.tensor([5, 130, 256, 299], dtype=torch.int32)   # rows already cached
    base = make_inputs(cfg, seed=33, lengths=lens + 1)
    app = make_append_inputs(cfg, seed=34)
    cache = base.cache.cuda()
    d = mla.dims(cfg.batch, cfg.heads, cfg.s_max, mla.MLA_BF16)
    mla.cache_append(d, app.x.cuda(), app.w_kva.cuda(), lens.cuda(), cache, cfg.rope_base)
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, torch.bfloat16,
                          rope_base=cfg.rope_base, softmax_scale=cfg.softmax_scale)
    out = step.run(base.q_nope.cuda(), base.q_rope.cuda(), cache, (lens + 1).cuda(),
                   lens.cuda(), base.w_uk.cuda(), base.w_uv.cuda())
    torch.cuda.synchronize()
    # oracle: the same cache with the oracle's appended rows (rounded to bf16 like the cache)
    rows = O.cache_append_row(app.x.double().numpy(), app.w_kva.double().numpy(), lens.numpy(),
                              cfg.d_c, cfg.rope_base)
    base.cache[torch.arange(cfg.batch), lens.long()] = torch.from_numpy(rows).to(torch.bfloat16)
    ref, bs = run_oracle(base)
    assert_close("o", out.double().cpu().numpy()[bs], ref["o"], "bf16")


@pytest.mark.parametrize("cfg", [
    cfg_of(V2LITE_BF16_B8_S4096),
    cfg_of(V3_BF16_H128_B32_S16384),
    cfg_of(V2LITE_BF16_B8_S4096, batch=19),
    cfg_of(V2LITE_BF16_B8_S4096, batch=70, hidden=1160),
    cfg_of(V2LITE_F32_B1_S64),
], ids=["v2lite_bf16", "v3_bf16", "v2lite_bf16_b19", "b70_hidden1160", "v2lite_f32"])
def test_wo_proj(cuda_lib, cfg):
    mla = cuda_lib
    inp = make_wo_inputs(cfg, seed=35)
    d = mla.dims(cfg.batch, cfg.heads, cfg.s_max, mla.dtype_code(_dt(cfg)))
    y = torch.empty((cfg.batch, cfg.hidden), dtype=torch.float32, device="cuda")
    mla.wo_proj(d, inp.o.cuda(), inp.w_o.cuda(), y)
    torch.cuda.synchronize()
    ref = O.output_projection(inp.o.double().numpy(), inp.w_o.double().numpy())
    assert_close("y", y.double().cpu().numpy(), ref, cfg.dtype)
