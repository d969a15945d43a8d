"""mla_decode_attn_noalloc: the decode attention for hosts that cannot allocate
device memory (an engine whose own pool owns all of it, or a loop where cudaMalloc
would synchronise the device).  It keeps its chunk partials in a fixed array inside
the library instead of a caller-supplied workspace.

Checked through the C ABI against mla_decode_attn on the same inputs, on two calls
in a row with different inputs and chunk counts, so a second call that saw the first
call's leftovers in the shared array would show.  Both calls run the same kernels
with the same chunking on the same inputs, so their results must be equal bit for
bit.  With an FP8 cache the scratch also holds the query's E4M3 image after the
partials, which the size check counts.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from workloads import (V2LITE_BF16_B8_S4096, V2LITE_FP8_B8_S4096, MlaConfig, cache_storage,
                       make_inputs)

pytestmark = pytest.mark.gpu


def _decode_both(mla, inp, num_splits):
    """o_c and lse from mla_decode_attn (caller workspace) and from the fixed-scratch call."""
    cfg = inp.cfg
    dt = cache_storage(cfg)   # the cache's type names the library dtype
    dev = "cuda"
    B, H = cfg.batch, cfg.heads
    d = mla.dims(B, H, cfg.s_max, mla.dtype_code(dt))
    q_abs = torch.empty(B, H, 512, dtype=torch.float32, device=dev)
    q_pe = torch.empty(B, H, 64, dtype=torch.float32, device=dev)
    mla.absorb_q(d, inp.q_nope.to(dev), inp.q_rope.to(dev), inp.w_uk.to(dev),
                 inp.positions.to(dev), q_abs, q_pe, rope_base=cfg.rope_base)
    cache, lengths = inp.cache.to(dev).contiguous(), inp.lengths.to(dev)
    ws = torch.empty(mla.workspace_bytes(d, num_splits), dtype=torch.uint8, device=dev)
    out = {}
    for name in ("workspace", "noalloc"):
        o_c = torch.full((B, H, 512), float("nan"), dtype=torch.float32, device=dev)
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        if name == "workspace":
            mla.decode_attn(d, q_abs, q_pe, cache, lengths, o_c, ws, cfg.softmax_scale,
                            num_splits, lse=lse, dev_status=status)
        else:
            mla.decode_attn_noalloc(d, q_abs, q_pe, cache, lengths, o_c, cfg.softmax_scale,
                                    num_splits, lse=lse, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        out[name] = (o_c.double().cpu().numpy(), lse.double().cpu().numpy())
    return out


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_noalloc_matches_workspace_call_twice(cuda_lib, dtype):
    mla = cuda_lib
    # first call: the 8 x 4096-row decode workload, library's chunk choice
    first = make_inputs(V2LITE_BF16_B8_S4096 if dtype == "bf16" else V2LITE_FP8_B8_S4096,
                        seed=11)
    # second call: other inputs, a ragged batch and fewer chunks, so a partial that
    # the second call failed to write would still hold the first call's value
    cfg2 = MlaConfig(name=f"noalloc_ragged_{dtype}_b5_s1000", dtype=dtype, batch=5, heads=16,
                     s_max=1000, hidden=2048)
    second = make_inputs(cfg2, seed=12, poison_tail=True,
                         lengths=torch.tensor([1, 129, 1000, 640, 77], dtype=torch.int32))
    for inp, splits in ((first, 0), (second, 3)):
        r = _decode_both(mla, inp, splits)
        for k, name in ((0, "o_c"), (1, "lse")):
            got, want = r["noalloc"][k], r["workspace"][k]
            assert np.all(np.isfinite(got)), f"{name}: non-finite values"
            assert np.array_equal(got, want), \
                f"{name}: max abs difference {np.max(np.abs(got - want)):.3e}, equality expected"


def test_noalloc_rejects_partials_beyond_the_fixed_size(cuda_lib):
    mla = cuda_lib
    lib = mla.load()
    limit = 16 << 20
    d = mla.dims(64, 128, 65536, mla.MLA_BF16)
    assert mla.workspace_bytes(d, 64) > limit
    buf = torch.zeros(1024, dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p(buf.data_ptr())
    code = lib.mla_decode_attn_noalloc(ctypes.byref(d), p, p, p, p, 0.07, 64, p, None, None, None)
    assert code == 3                                   # MLA_ERR_WORKSPACE, nothing launched
    assert b"scratch" in lib.mla_last_error_message()
    torch.cuda.synchronize()
