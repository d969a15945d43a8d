"""GPU parity of the bench's own launch configuration: many decode steps in a row
with no synchronisation between them.

The bench captures K consecutive mla_decode_step calls in one CUDA graph.  The
kernels are launched with programmatic dependent launch, so step k+1's absorb
(its W_UK fetch and cache prefetch) and the set-up of its split overlap step k's
tail, and every step shares one workspace and one q_abs / q_pe.  A cross-step
hazard (a split writing partials that the previous tail has not read yet, an
absorb overwriting q_abs before the previous split has loaded it) would leave
every single-step test green.  Here each step of such a graph gets its own
inputs (its own cache, weights and queries, as the bench's rotating layer copies)
and its own o_c, lse and o, and every step is compared with the fp64 oracle.

The same holds for the e2e path: several captured host-memory steps
(DecodeStep.capture) replayed, or launched directly, back to back at the
bench's size.
"""
import numpy as np
import pytest
import torch

from _parity import assert_close, run_oracle
from workloads import V2LITE_BF16_B8_S4096, V2LITE_FP8_B8_S4096, cache_storage, make_inputs

pytestmark = pytest.mark.gpu

STEPS = 6


def _layer_inputs(cfg, n, seed0):
    """n independent draws of the workload: each step reads its own layer."""
    return [make_inputs(cfg, seed=seed0 + k) for k in range(n)]


@pytest.mark.parametrize("cfg", [V2LITE_BF16_B8_S4096, V2LITE_FP8_B8_S4096],
                         ids=lambda c: c.name)
def test_graph_of_consecutive_steps(cuda_lib, cfg):
    mla = cuda_lib
    dev = "cuda"
    layers = _layer_inputs(cfg, STEPS, 300)
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, cache_storage(cfg), device=dev,
                          rope_base=cfg.rope_base, softmax_scale=cfg.softmax_scale)
    d = step.dims
    B, H = cfg.batch, cfg.heads
    put = lambda t: t.to(dev).contiguous()
    ins = [dict(qn=put(x.q_nope), qr=put(x.q_rope), cache=put(x.cache), wuk=put(x.w_uk),
                wuv=put(x.w_uv), lengths=put(x.lengths), pos=put(x.positions)) for x in layers]
    outs = [dict(o_c=torch.full((B, H, 512), float("nan"), device=dev),
                 lse=torch.full((B, H), float("nan"), device=dev),
                 o=torch.full((B, H, 128), float("nan"), device=dev)) for _ in range(STEPS)]

    def one(k):
        i, o = ins[k], outs[k]
        mla.decode_step(d, i["qn"], i["qr"], i["wuk"], i["pos"], i["cache"], i["lengths"],
                        i["wuv"], step.workspace, step.q_abs, step.q_pe, o["o_c"], o["o"],
                        step.scale, step.rope_base, 0, o["lse"], step.status)

    for k in range(STEPS):          # eager warm-up (module load, kernel attributes)
        one(k)
    torch.cuda.synchronize()
    for o in outs:
        for t in o.values():
            t.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
        for k in range(STEPS):
            one(k)
    g.replay()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    for k in range(STEPS):
        ref, bs = run_oracle(layers[k])
        got = {n: t.double().cpu().numpy() for n, t in outs[k].items()}
        assert_close(f"step {k} o_c", got["o_c"][bs], ref["o_c"], cfg.dtype)
        assert_close(f"step {k} lse", got["lse"][bs], ref["lse"], cfg.dtype)
        assert_close(f"step {k} o", got["o"][bs], ref["o"], cfg.dtype)


def test_bench_graph_form(cuda_lib):
    """The bench's graph as it is: DecodeStep.run (every step writes the same
    o_c, lse and o) over rotating copies of one layer; the last step's outputs
    equal the oracle's."""
    mla = cuda_lib
    cfg = V2LITE_BF16_B8_S4096
    inp = make_inputs(cfg, seed=0)
    L = 4
    caches = [inp.cache.cuda() for _ in range(L)]
    wuk = [inp.w_uk.cuda() for _ in range(L)]
    wuv = [inp.w_uv.cuda() for _ in range(L)]
    qn, qr = inp.q_nope.cuda(), inp.q_rope.cuda()
    lengths, pos = inp.lengths.cuda(), inp.positions.cuda()
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, torch.bfloat16,
                          rope_base=cfg.rope_base, softmax_scale=cfg.softmax_scale)
    run = lambda k: step.run(qn, qr, caches[k % L], lengths, pos, wuk[k % L], wuv[k % L])
    for k in range(3):
        run(k)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
        for k in range(40):
            run(k)
    step.out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    ref, bs = run_oracle(inp)
    assert_close("o_c", step.o_c.double().cpu().numpy()[bs], ref["o_c"], "bf16")
    assert_close("lse", step.lse.double().cpu().numpy()[bs], ref["lse"], "bf16")
    assert_close("o", step.out.double().cpu().numpy()[bs], ref["o"], "bf16")


def test_host_steps_back_to_back_at_bench_size(cuda_lib):
    """The e2e leg's path: steps captured from host memory (queries staged by the
    absorb's shared-memory variant at full size), four layers replayed back to
    back with no synchronisation; each step's o, written to its own pinned host
    buffer, equals the oracle's."""
    mla = cuda_lib
    cfg = V2LITE_BF16_B8_S4096
    layers = _layer_inputs(cfg, 4, 400)
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, torch.bfloat16,
                          rope_base=cfg.rope_base, softmax_scale=cfg.softmax_scale)
    hosts = []
    for x in layers:
        hs = step.capture(x.cache.cuda(), x.w_uk.cuda(), x.w_uv.cuda())
        hs.q_nope.copy_(x.q_nope)
        hs.q_rope.copy_(x.q_rope)
        hs.lengths.copy_(x.lengths)
        hs.positions.copy_(x.positions)
        hs.out.fill_(float("nan"))
        hosts.append(hs)
    for hs in hosts:
        hs.replay()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    for k, (hs, x) in enumerate(zip(hosts, layers)):
        ref, bs = run_oracle(x)
        assert_close(f"layer {k} o", hs.out.double().numpy()[bs], ref["o"], "bf16")
    ref, bs = run_oracle(layers[-1])
    assert_close("last o_c", step.o_c.double().cpu().numpy()[bs], ref["o_c"], "bf16")


@pytest.mark.parametrize("cfg", [V2LITE_BF16_B8_S4096, V2LITE_FP8_B8_S4096], ids=lambda c: c.dtype)
def test_host_steps_launched_directly(cuda_lib, cfg):
    """HostStep.launch (the direct call, arguments converted at capture) computes
    what replay computes, bit for bit, and back-to-back launches over four layers
    (each step's absorb overlapping the previous step's tail) equal the oracle."""
    mla = cuda_lib
    layers = _layer_inputs(cfg, 4, 410)
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, cache_storage(cfg),
                          rope_base=cfg.rope_base, softmax_scale=cfg.softmax_scale)
    hosts = []
    for x in layers:
        hs = step.capture(x.cache.cuda(), x.w_uk.cuda(), x.w_uv.cuda())
        hs.q_nope.copy_(x.q_nope)
        hs.q_rope.copy_(x.q_rope)
        hs.lengths.copy_(x.lengths)
        hs.positions.copy_(x.positions)
        hosts.append(hs)
    hosts[0].replay()
    torch.cuda.synchronize()
    replayed = hosts[0].out.clone()
    for hs in hosts:
        hs.out.fill_(float("nan"))
    for _ in range(2):
        for hs in hosts:
            hs.launch()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    assert torch.equal(hosts[0].out, replayed)
    for k, (hs, x) in enumerate(zip(hosts, layers)):
        ref, bs = run_oracle(x)
        assert_close(f"layer {k} o", hs.out.double().numpy()[bs], ref["o"], cfg.dtype)


def test_plain_launches_equal_overlapped(cuda_lib):
    """The bench's plain-launch timing mode (programmatic launch off) computes the
    same step bit for bit as the default overlapped launches."""
    mla = cuda_lib
    cfg = V2LITE_BF16_B8_S4096
    inp = make_inputs(cfg, seed=5)
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, torch.bfloat16,
                          rope_base=cfg.rope_base, softmax_scale=cfg.softmax_scale)
    args = [t.cuda() for t in (inp.q_nope, inp.q_rope, inp.cache, inp.lengths, inp.positions,
                               inp.w_uk, inp.w_uv)]
    outs = []
    for overlap in (True, False, True):
        mla.set_launch_overlap(overlap)
        try:
            step.run(*args)
            torch.cuda.synchronize()
        finally:
            mla.set_launch_overlap(True)
        outs.append([t.clone() for t in (step.q_abs, step.o_c, step.lse, step.out)])
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    for a, b in zip(outs[0], outs[2]):
        assert torch.equal(a, b)
