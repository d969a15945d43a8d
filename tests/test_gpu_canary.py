"""Out-of-bounds writes, caught without a sanitizer: every output buffer (and the
workspace) of every call sits between guard regions filled with a sentinel bit
pattern, and every input is compared bit for bit after the call.  A kernel that
writes one element past its output, or into an input, fails here."""
import pytest
import torch

from workloads import (MlaConfig, cache_storage, make_append_inputs, make_inputs,
                       make_materialized_inputs, make_wo_inputs)

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side (a multiple of 256, so alignment is kept)
SENTINEL = 0xA5


def guarded(shape, dtype):
    """(view, whole): a CUDA tensor of ``shape`` inside a buffer with GUARD sentinel
    bytes before and after it."""
    n = 1
    for x in shape:
        n *= x
    nbytes = n * torch.tensor([], dtype=dtype).element_size()
    whole = torch.full((GUARD + nbytes + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
    view = whole[GUARD:GUARD + nbytes].view(dtype).view(shape)
    return view, whole


def guards_intact(whole, what):
    head, tail = whole[:GUARD], whole[-GUARD:]
    assert bool((head == SENTINEL).all()), f"{what}: written before its start"
    assert bool((tail == SENTINEL).all()), f"{what}: written past its end"


def small(dtype, B=3, S=300, H=16, hidden=2048, q_len=1):
    return MlaConfig(name=f"canary_{dtype}", dtype=dtype, batch=B, heads=H, s_max=S,
                     hidden=hidden, q_len=q_len)


@pytest.mark.parametrize("dtype,H,q_len,B", [("bf16", 16, 1, 3), ("fp8", 16, 1, 3),
                                             ("f32", 16, 1, 3), ("bf16", 32, 1, 3),
                                             ("bf16", 16, 4, 3), ("fp8", 16, 2, 3),
                                             ("bf16", 16, 1, 60), ("bf16", 16, 3, 20),
                                             ("bf16", 128, 1, 3), ("bf16", 64, 3, 3)])
@pytest.mark.parametrize("splits", [0, 3])
def test_decode_calls_stay_in_bounds(cuda_lib, dtype, H, q_len, B, splits):
    """B = 60 (three chunks) and 20 x 3 tokens run the persistent split grid; 64
    and 128 heads the 64-head, one-part CTAs."""
    mla = cuda_lib
    cfg = small(dtype, B=B, S=300, H=H, q_len=q_len)
    lens = torch.tensor([300, 129, max(q_len, 17)] * (B // 3), dtype=torch.int32)
    inp = make_inputs(cfg, seed=80, lengths=lens)
    d = mla.dims(cfg.batch, cfg.heads, cfg.s_max, mla.dtype_code(cache_storage(cfg)))
    qd = mla.query_dims(d, q_len)
    R = cfg.batch * q_len
    dev = lambda t: t.cuda().contiguous()
    ins = {k: dev(getattr(inp, k)) for k in ("q_nope", "q_rope", "cache", "lengths", "positions",
                                              "w_uk", "w_uv")}
    before = {k: v.clone() for k, v in ins.items()}
    q_abs, g_qa = guarded((R, H, 512), torch.float32)
    q_pe, g_qp = guarded((R, H, 64), torch.float32)
    o_c, g_oc = guarded((R, H, 512), torch.float32)
    lse, g_lse = guarded((R, H), torch.float32)
    out, g_out = guarded((R, H, 128), torch.float32)
    ws, g_ws = guarded((mla.multi_workspace_bytes(d, q_len, splits),), torch.uint8)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = cfg.softmax_scale
    if q_len == 1:
        mla.decode_step(d, ins["q_nope"], ins["q_rope"], ins["w_uk"], ins["positions"],
                        ins["cache"], ins["lengths"], ins["w_uv"], ws, q_abs, q_pe, o_c, out,
                        scale, cfg.rope_base, splits, lse, status)
        torch.cuda.synchronize()
        for g, what in ((g_qa, "q_abs"), (g_qp, "q_pe"), (g_oc, "o_c"), (g_lse, "lse"),
                        (g_out, "out"), (g_ws, "workspace")):
            guards_intact(g, f"mla_decode_step {what}")
    # the separate calls (the multi-token call for several tokens)
    mla.absorb_q(qd, ins["q_nope"], ins["q_rope"], ins["w_uk"], ins["positions"], q_abs, q_pe,
                 cfg.rope_base)
    if q_len == 1:
        mla.decode_attn(d, q_abs, q_pe, ins["cache"], ins["lengths"], o_c, ws, scale, splits,
                        lse, status)
    else:
        mla.decode_attn_multi(d, q_len, q_abs, q_pe, ins["cache"], ins["lengths"], o_c, ws,
                              scale, splits, lse, status)
    mla.out_proj(qd, o_c, ins["w_uv"], out)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for g, what in ((g_qa, "q_abs"), (g_qp, "q_pe"), (g_oc, "o_c"), (g_lse, "lse"),
                    (g_out, "out"), (g_ws, "workspace")):
        guards_intact(g, what)
    for k, v in ins.items():
        assert torch.equal(v.view(torch.uint8) if v.dtype == torch.float8_e4m3fn else v,
                           before[k].view(torch.uint8) if v.dtype == torch.float8_e4m3fn
                           else before[k]), f"input {k} was written"


@pytest.mark.parametrize("dtype,B,hidden", [("bf16", 19, 2048), ("fp8", 5, 1152), ("f32", 3, 256)])
def test_projection_calls_stay_in_bounds(cuda_lib, dtype, B, hidden):
    """Cache append writes exactly one row per sequence; W^O and the materialised
    calls write only their outputs."""
    mla = cuda_lib
    cfg = small(dtype, B=B, S=24, hidden=hidden)
    d = mla.dims(cfg.batch, cfg.heads, cfg.s_max, mla.dtype_code(cache_storage(cfg)))
    wdt = torch.float32 if dtype == "f32" else torch.bfloat16
    ap = make_append_inputs(cfg, seed=81)
    cache, g_cache = guarded((B, cfg.s_max, 576), cache_storage(cfg))
    cache.view(torch.uint8).fill_(0)
    x, w_kva, pos = ap.x.cuda(), ap.w_kva.cuda(), ap.positions.cuda()
    x0, w0 = x.clone(), w_kva.clone()
    mla.cache_append(d, x, w_kva, pos, cache, cfg.rope_base)
    torch.cuda.synchronize()
    guards_intact(g_cache, "cache")
    assert torch.equal(x, x0) and torch.equal(w_kva, w0)
    untouched = torch.ones((B, cfg.s_max), dtype=torch.bool, device="cuda")
    untouched[torch.arange(B, device="cuda"), pos.long()] = False
    assert bool((cache.view(torch.uint8)[untouched] == 0).all()), "a row other than the new one"

    wo = make_wo_inputs(cfg, seed=82)
    o, w_o = wo.o.cuda(), wo.w_o.cuda()
    y, g_y = guarded((B, hidden), torch.float32)
    mla.wo_proj(d, o, w_o, y)

    m = make_materialized_inputs(cfg, seed=83)
    H = cfg.heads
    w_kq, g_kq = guarded((H * 512, hidden), wdt)
    w_ov, g_ov = guarded((hidden, H * 512), wdt)
    mla.materialize_wkq(d, m.w_q_nope.cuda(), m.base.w_uk.cuda(), w_kq)
    mla.materialize_wov(d, m.w_o.cuda(), m.base.w_uv.cuda(), w_ov)
    q_abs, g_qa = guarded((B, H, 512), torch.float32)
    q_pe, g_qp = guarded((B, H, 64), torch.float32)
    mla.absorb_q_materialized(d, m.x.cuda(), w_kq, m.base.q_rope.cuda(), m.base.positions.cuda(),
                              q_abs, q_pe, cfg.rope_base)
    o_c = torch.randn((B, H, 512), device="cuda")
    y2, g_y2 = guarded((B, hidden), torch.float32)
    mla.ov_proj(d, o_c, w_ov, y2)
    torch.cuda.synchronize()
    for g, what in ((g_y, "W^O y"), (g_kq, "W^KQ"), (g_ov, "W^OV"), (g_qa, "q_abs"),
                    (g_qp, "q_pe"), (g_y2, "W^OV y")):
        guards_intact(g, what)
