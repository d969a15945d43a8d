"""The split kernel's bounded waits, made to run out on purpose without a fault.

A test hook (mla_test_set_split_hooks) shortens every bounded wait of the bf16
split kernel to a few milliseconds and lets its HBM ring issue only the first
tile of each chunk.  With chunks of four tiles, the score, softmax and PV roles
then wait for boxes that are never requested; nothing is in flight when their
waits run out.  The kernel must return on its own, report
MLA_DEV_PIPELINE_TIMEOUT in the status word, write no partial, and leave the
context usable: the next call with the hooks reset matches the oracle.
(A wait that runs out is the kernel-side form of the overflow-returns-an-error
rule of "Transformer and KV Cache Basics".)
"""
import numpy as np
import pytest
import torch

from _parity import assert_close, run_oracle
from workloads import MlaConfig, make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H", [16, 32, 64])
def test_bounded_waits_run_out_and_report(cuda_lib, H):
    mla = cuda_lib
    lib = mla.load()
    cfg = MlaConfig(name=f"timeout_b2_h{H}_s512", dtype="bf16", batch=2, heads=H, s_max=512,
                    hidden=2048)
    inp = make_inputs(cfg, seed=77, lengths=torch.tensor([512, 512], dtype=torch.int32))
    dev = "cuda"
    d = mla.dims(cfg.batch, H, cfg.s_max, mla.MLA_BF16)
    q_abs = torch.empty(cfg.batch, H, 512, dtype=torch.float32, device=dev)
    q_pe = torch.empty(cfg.batch, H, 64, dtype=torch.float32, device=dev)
    mla.absorb_q(d, inp.q_nope.to(dev), inp.q_rope.to(dev), inp.w_uk.to(dev),
                 inp.positions.to(dev), q_abs, q_pe, rope_base=cfg.rope_base)
    cache, lengths = inp.cache.to(dev), inp.lengths.to(dev)
    ws = torch.full((mla.workspace_bytes(d, 1),), 0x7F, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    try:
        lib.mla_test_set_split_hooks(5_000_000, 1)     # 5 ms waits; one tile of four
        mla.decode_split(d, q_abs, q_pe, cache, lengths, ws, cfg.softmax_scale, 1, status)
    finally:
        lib.mla_test_set_split_hooks(0, 0)
    torch.cuda.synchronize()                           # the kernel returned by itself
    assert int(status.item()) & mla.MLA_DEV_PIPELINE_TIMEOUT
    assert bool(torch.all(ws == 0x7F)), "a timed-out CTA wrote partials"

    # The context is still usable and the hooks are off again.
    status.zero_()
    o_c = torch.empty(cfg.batch, H, 512, dtype=torch.float32, device=dev)
    lse = torch.empty(cfg.batch, H, dtype=torch.float32, device=dev)
    mla.decode_attn(d, q_abs, q_pe, cache, lengths, o_c, ws, cfg.softmax_scale, 1, lse=lse,
                    dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, bs = run_oracle(inp)
    assert_close("o_c", o_c.double().cpu().numpy()[bs], ref["o_c"], "bf16")
    assert_close("lse", lse.double().cpu().numpy()[bs], ref["lse"], "bf16")
    assert np.all(np.isfinite(o_c.cpu().numpy()))


def test_bounded_waits_run_out_in_a_persistent_grid(cuda_lib):
    """The same on the persistent grid (several chunks per CTA): CTAs whose
    stream holds more than one tile time out and report; the next call with the
    hooks reset matches the oracle."""
    mla = cuda_lib
    lib = mla.load()
    cfg = MlaConfig(name="timeout_persist_b200_s256", dtype="bf16", batch=200, heads=16,
                    s_max=256, hidden=2048)
    inp = make_inputs(cfg, seed=78)
    dev = "cuda"
    d = mla.dims(cfg.batch, 16, cfg.s_max, mla.MLA_BF16)
    assert mla.plan(d, 2)[2]                           # persistent
    q_abs = torch.empty(cfg.batch, 16, 512, dtype=torch.float32, device=dev)
    q_pe = torch.empty(cfg.batch, 16, 64, dtype=torch.float32, device=dev)
    mla.absorb_q(d, inp.q_nope.to(dev), inp.q_rope.to(dev), inp.w_uk.to(dev),
                 inp.positions.to(dev), q_abs, q_pe, rope_base=cfg.rope_base)
    cache, lengths = inp.cache.to(dev), inp.lengths.to(dev)
    ws = torch.empty((mla.workspace_bytes(d, 2),), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    try:
        lib.mla_test_set_split_hooks(5_000_000, 1)
        mla.decode_split(d, q_abs, q_pe, cache, lengths, ws, cfg.softmax_scale, 2, status)
    finally:
        lib.mla_test_set_split_hooks(0, 0)
    torch.cuda.synchronize()
    assert int(status.item()) & mla.MLA_DEV_PIPELINE_TIMEOUT
    status.zero_()
    o_c = torch.empty(cfg.batch, 16, 512, dtype=torch.float32, device=dev)
    lse = torch.empty(cfg.batch, 16, dtype=torch.float32, device=dev)
    mla.decode_attn(d, q_abs, q_pe, cache, lengths, o_c, ws, cfg.softmax_scale, 2, lse=lse,
                    dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, bs = run_oracle(inp, batches=[0, 77, 199])
    assert_close("o_c", o_c.double().cpu().numpy()[bs], ref["o_c"], "bf16")
    assert_close("lse", lse.double().cpu().numpy()[bs], ref["lse"], "bf16")

