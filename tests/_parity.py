"""Helpers of the GPU parity tests: run the CUDA path through the C ABI on seeded
inputs, run the fp64 oracle on the same bits, and compare."""
from __future__ import annotations

import numpy as np
import torch

from oracle import mla_oracle as O
from workloads import (TOL_BF16_MAX_ABS, TOL_BF16_REL_L2, TOL_F32_MAX_ABS, MlaInputs,
                       cache_storage)


def run_cuda(inp: MlaInputs, num_splits: int = 0, device: str = "cuda", path: str = "step"):
    """One decode step through the C ABI: ``path`` "step" is mla_decode_step (one call,
    fused combine + W_UV for bf16), "calls" the three calls mla_absorb_q,
    mla_decode_attn, mla_out_proj.  Returns fp64 numpy arrays."""
    import head_latent_attention_absorbed_gb300 as mla
    cfg = inp.cfg
    dt = cache_storage(cfg)   # the cache's type names the library dtype
    step = mla.DecodeStep(cfg.batch, cfg.heads, cfg.s_max, dt, device=device,
                          num_splits_requested=num_splits, rope_base=cfg.rope_base,
                          softmax_scale=cfg.softmax_scale)
    dev = lambda t: t.to(device).contiguous()
    run = step.run if path == "step" else step.run_calls
    run(dev(inp.q_nope), dev(inp.q_rope), dev(inp.cache), dev(inp.lengths),
        dev(inp.positions), dev(inp.w_uk), dev(inp.w_uv))
    torch.cuda.synchronize()
    f = lambda t: t.detach().to("cpu", torch.float64).numpy()
    return dict(q_abs=f(step.q_abs), q_pe=f(step.q_pe), o_c=f(step.o_c), lse=f(step.lse),
                o=f(step.out), status=int(step.status.item()), splits=step.splits)


def run_oracle(inp: MlaInputs, batches=None):
    """Oracle outputs for the listed sequences (all by default), one at a time."""
    cfg = inp.cfg
    batches = list(range(cfg.batch)) if batches is None else list(batches)
    res = {k: [] for k in ("q_abs", "q_pe", "o_c", "lse", "o")}
    for b in batches:
        a = inp.as_float64_numpy(b)
        if a["cache"] is None:   # FP8 cache: the oracle decodes the E4M3 codes
            a["cache"] = O.e4m3_to_float64(a["cache_e4m3"])
        n = int(a["lengths"][0])
        a["cache"] = a["cache"][:, :n]
        r = O.decode_absorbed(a["q_nope"], a["q_rope"], a["w_uk"], a["w_uv"], a["cache"],
                              a["lengths"], a["positions"], cfg.softmax_scale, cfg.rope_base)
        for k in res:
            res[k].append(r[k][0])
    return {k: np.stack(v) for k, v in res.items()}, batches


def rel_l2(x, ref):
    return float(np.linalg.norm((x - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))


def max_abs(x, ref):
    return float(np.max(np.abs(x - ref)))


def assert_close(name: str, x, ref, dtype: str):
    assert np.all(np.isfinite(x)), f"{name}: non-finite values"
    ma = max_abs(x, ref)
    if dtype == "f32":
        assert ma <= TOL_F32_MAX_ABS, f"{name}: max abs {ma:.3e} > {TOL_F32_MAX_ABS}"
    else:
        rl = rel_l2(x, ref)
        assert ma <= TOL_BF16_MAX_ABS, f"{name}: max abs {ma:.3e} > {TOL_BF16_MAX_ABS}"
        assert rl <= TOL_BF16_REL_L2, f"{name}: rel L2 {rl:.3e} > {TOL_BF16_REL_L2}"
    return ma


def compare(gpu, ref, batches, dtype: str):
    """Per-call parity: absorb (q_abs, q_pe), attention (o_c, lse), output o."""
    out = {}
    for k in ("q_abs", "q_pe", "o_c", "lse", "o"):
        out[k] = assert_close(k, gpu[k][batches], ref[k], dtype)
    return out
