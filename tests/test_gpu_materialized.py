"""GPU parity of the materialised absorption ("Multi-Head Latent Attention" 3.3,
eq. 3.3.3 and 3.5): the weight transforms mla_materialize_wkq / _wov, and the step
mla_absorb_q_materialized -> mla_decode_attn -> mla_ov_proj, through the C ABI,
against the fp64 oracle on the same seeded inputs.

The oracle forms W^KQ and W^OV in fp64 and stores them in the weight type the way
a model would (a cast to bf16, nearest even); the GPU forms them with fp32 sums
and rounds once.  The two may differ by one unit in the last place where a sum
lands next to a rounding boundary; the step's outputs are compared at the usual
tolerances.
"""
import numpy as np
import pytest
import torch

from _parity import assert_close
from oracle import mla_oracle as O
from workloads import (MlaConfig, V2LITE_BF16_B8_S4096, V2LITE_F32_B1_S64, cache_storage,
                       make_materialized_inputs)

pytestmark = pytest.mark.gpu


def _wdt(cfg):
    return torch.float32 if cfg.dtype == "f32" else torch.bfloat16


def _stored(w64, cfg):
    """An fp64 oracle matrix as the model keeps it: cast once to the weight type."""
    return torch.from_numpy(w64).to(_wdt(cfg))


def _dims(mla, cfg):
    return mla.dims(cfg.batch, cfg.heads, cfg.s_max, mla.dtype_code(cache_storage(cfg)))


def _check_materialized(got, ref64, absprod, cfg, what):
    """GPU matrix against the fp64 product.  An fp32 sum of K = 128 products is off
    by at most K 2^-24 sum_k |a_k b_k| (``absprod``); on top of that a bf16 result
    may sit one unit away from the rounded product.  bf16 results must also equal
    the rounded product almost everywhere."""
    g = got.double().numpy()
    acc = 128 * 2.0 ** -24 * absprod
    if cfg.dtype == "f32":
        bad = np.abs(g - ref64) > acc + 2.0 ** -24 * np.abs(ref64)
        assert not np.any(bad), f"{what}: {int(bad.sum())} values beyond the fp32 bound"
        return
    r = _stored(ref64, cfg).double().numpy()
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(r), 1e-30))) - 7)
    bad = np.abs(g - r) > ulp + acc
    assert not np.any(bad), f"{what}: {int(bad.sum())} values beyond one bf16 unit + fp32 bound"
    frac = float(np.mean(g != r))
    assert frac <= 1e-3, f"{what}: {frac:.2e} of the values differ from the rounded product"


@pytest.mark.parametrize("dtype,H,hidden", [("bf16", 16, 2048), ("f32", 16, 256),
                                            ("bf16", 128, 7168)],
                         ids=["v2lite_bf16", "f32", "v3_bf16"])
def test_materialized_weights(cuda_lib, dtype, H, hidden):
    mla = cuda_lib
    cfg = MlaConfig(name="mat_w", dtype=dtype, batch=1, heads=H, s_max=8, hidden=hidden)
    m = make_materialized_inputs(cfg, seed=50)
    d = _dims(mla, cfg)
    wkq = torch.empty((H * 512, hidden), dtype=_wdt(cfg), device="cuda")
    wov = torch.empty((hidden, H * 512), dtype=_wdt(cfg), device="cuda")
    mla.materialize_wkq(d, m.w_q_nope.cuda(), m.base.w_uk.cuda(), wkq)
    mla.materialize_wov(d, m.w_o.cuda(), m.base.w_uv.cuda(), wov)
    torch.cuda.synchronize()
    heads = range(H) if H <= 16 else (0, 77, H - 1)   # the oracle checks sampled heads at V3 size
    wq, wuk = m.w_q_nope.double().numpy(), m.base.w_uk.double().numpy()
    wo, wuv = m.w_o.double().numpy(), m.base.w_uv.double().numpy()
    for h in heads:
        kq_h = O.materialize_wkq(wq[h:h + 1], wuk[h:h + 1])[0]
        kq_abs = O.materialize_wkq(np.abs(wq[h:h + 1]), np.abs(wuk[h:h + 1]))[0]
        _check_materialized(wkq[h * 512:(h + 1) * 512].cpu(), kq_h, kq_abs, cfg, f"W^KQ head {h}")
        ov_h = O.materialize_wov(wo[:, h * 128:(h + 1) * 128], wuv[h:h + 1])
        ov_abs = O.materialize_wov(np.abs(wo[:, h * 128:(h + 1) * 128]), np.abs(wuv[h:h + 1]))
        _check_materialized(wov[:, h * 512:(h + 1) * 512].cpu(), ov_h, ov_abs, cfg,
                            f"W^OV head {h}")


def _run_step(mla, cfg, m, splits=0):
    """materialise on the GPU, then absorb_q_materialized -> decode_attn -> ov_proj."""
    d = _dims(mla, cfg)
    B, H = cfg.batch, cfg.heads
    dev = lambda t: t.cuda().contiguous()
    wkq = torch.empty((H * 512, cfg.hidden), dtype=_wdt(cfg), device="cuda")
    wov = torch.empty((cfg.hidden, H * 512), dtype=_wdt(cfg), device="cuda")
    mla.materialize_wkq(d, dev(m.w_q_nope), dev(m.base.w_uk), wkq)
    mla.materialize_wov(d, dev(m.w_o), dev(m.base.w_uv), wov)
    q_abs = torch.empty((B, H, 512), dtype=torch.float32, device="cuda")
    q_pe = torch.empty((B, H, 64), dtype=torch.float32, device="cuda")
    o_c = torch.empty((B, H, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    y = torch.empty((B, cfg.hidden), dtype=torch.float32, device="cuda")
    ws = torch.empty((mla.workspace_bytes(d, splits),), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.absorb_q_materialized(d, dev(m.x), wkq, dev(m.base.q_rope), dev(m.base.positions), q_abs,
                              q_pe, cfg.rope_base)
    mla.decode_attn(d, q_abs, q_pe, dev(m.base.cache), dev(m.base.lengths), o_c, ws,
                    cfg.softmax_scale, splits, lse, status)
    mla.ov_proj(d, o_c, wov, y)
    torch.cuda.synchronize()
    f = lambda t: t.cpu().double().numpy()
    return dict(q_abs=f(q_abs), q_pe=f(q_pe), o_c=f(o_c), lse=f(lse), y=f(y),
                status=int(status.item()))


def _oracle_step(cfg, m, batches):
    wkq = _stored(O.materialize_wkq(m.w_q_nope.double().numpy(), m.base.w_uk.double().numpy()),
                  cfg).double().numpy()
    wov = _stored(O.materialize_wov(m.w_o.double().numpy(), m.base.w_uv.double().numpy()),
                  cfg).double().numpy()
    out = {k: [] for k in ("q_abs", "q_pe", "o_c", "lse", "y")}
    for b in batches:
        a = m.base.as_float64_numpy(b)
        if a["cache"] is None:
            a["cache"] = O.e4m3_to_float64(a["cache_e4m3"])
        n = int(a["lengths"][0])
        r = O.decode_materialized(m.x[b:b + 1].double().numpy(), a["q_rope"], wkq, wov,
                                  a["cache"][:, :n], a["lengths"], a["positions"],
                                  cfg.softmax_scale, cfg.rope_base)
        for k in out:
            out[k].append(r[k][0])
    return {k: np.stack(v) for k, v in out.items()}


def small(dtype, B=3, S=300, H=16, hidden=2048):
    return MlaConfig(name=f"mat_{dtype}", dtype=dtype, batch=B, heads=H, s_max=S, hidden=hidden)


@pytest.mark.parametrize("cfg,lengths,splits", [
    (small("bf16"), [300, 129, 1], 0),
    (small("bf16"), [300, 129, 1], 3),
    (small("fp8"), [300, 17, 256], 0),
    (small("f32", B=2, S=64, hidden=256), [64, 5], 0),
    (small("bf16", B=2, S=64, H=128, hidden=1024), [64, 40], 0),
], ids=["bf16", "bf16_3splits", "fp8", "f32", "v3_heads"])
def test_materialized_step_small(cuda_lib, cfg, lengths, splits):
    m = make_materialized_inputs(cfg, seed=51, poison_tail=True,
                                 lengths=torch.tensor(lengths, dtype=torch.int32))
    gpu = _run_step(cuda_lib, cfg, m, splits)
    assert gpu["status"] == 0
    bs = list(range(cfg.batch))
    ref = _oracle_step(cfg, m, bs)
    for k in ("q_abs", "q_pe", "o_c", "lse", "y"):
        assert_close(k, gpu[k][bs], ref[k], cfg.dtype)


def test_materialized_step_bench_shape(cuda_lib):
    """The bench workload's shapes (B 8, 4096 rows, V2-Lite), sequences 0 and 5."""
    cfg = V2LITE_BF16_B8_S4096
    m = make_materialized_inputs(cfg, seed=0)
    gpu = _run_step(cuda_lib, cfg, m)
    assert gpu["status"] == 0
    bs = [0, 5]
    ref = _oracle_step(cfg, m, bs)
    for k in ("q_abs", "q_pe", "o_c", "lse", "y"):
        assert_close(k, gpu[k][bs], ref[k], cfg.dtype)


def test_materialized_f32_workload(cuda_lib):
    cfg = V2LITE_F32_B1_S64
    m = make_materialized_inputs(cfg, seed=2)
    gpu = _run_step(cuda_lib, cfg, m)
    ref = _oracle_step(cfg, m, [0])
    for k in ("q_abs", "q_pe", "o_c", "lse", "y"):
        assert_close(k, gpu[k][[0]], ref[k], cfg.dtype)
