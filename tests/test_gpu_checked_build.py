"""The checked build (-DMLA_CHECK): the decode kernels test every index they can
compute before the access and report MLA_DEV_BOUNDS instead of touching memory
outside a buffer.  The small parity cases and the bench workload run through
that library (built here beside the default one); the results must still match
the oracle, and neither the calls' status words nor the library's bounds word
may carry the bit.
"""
import ctypes

import pytest
import torch

from _parity import compare, run_cuda, run_oracle
from workloads import V2LITE_BF16_B8_S4096, MlaConfig, make_inputs

pytestmark = pytest.mark.gpu


class _Ptr:
    """A one-int32 device buffer at a raw address, for torch."""

    def __init__(self, ptr):
        self.__cuda_array_interface__ = {"shape": (1,), "typestr": "<i4", "data": (ptr, False),
                                         "version": 3}


@pytest.fixture(scope="module")
def checked(cuda_lib):
    from head_latent_attention_absorbed_gb300 import _binding, build
    path = build.build(check=True)
    lib = _binding.load(path)
    assert lib.mla_built_with_checks() == 1
    saved = _binding._lib
    _binding._lib = lib          # every binding call goes to the checked library
    word = ctypes.c_void_p()
    assert lib.mla_debug_bounds_word(ctypes.byref(word)) == 0
    flags = torch.as_tensor(_Ptr(word.value), device="cuda")
    try:
        yield lib, flags
    finally:
        _binding._lib = saved


def small(B, H, S, **kw):
    return MlaConfig(name=f"checked_b{B}_h{H}_s{S}", dtype="bf16", batch=B, heads=H, s_max=S,
                     hidden=2048, **kw)


CASES = [   # (config, lengths, chunks requested, operand parts: 0 default, 2 hi + lo)
    (small(3, 16, 300), [1, 129, 300], 0, 0),
    (small(3, 16, 300), [7, 255, 300], 3, 0),
    (small(2, 32, 300), [300, 137], 4, 0),
    (small(2, 128, 200), [200, 61], 2, 0),   # 64 heads per CTA, one part
    (small(2, 128, 200), [200, 61], 2, 2),   # 32 heads per CTA, hi + lo
    (small(3, 64, 520), [520, 385, 1], 1, 0),
    (small(24, 16, 1024), None, 8, 0),       # persistent grid
    (small(20, 48, 600), None, 4, 0),        # persistent, head groups
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_small_cases_under_index_checks(checked, case):
    from head_latent_attention_absorbed_gb300 import _binding
    lib, flags = checked
    cfg, lengths, splits, parts = CASES[case]
    flags.zero_()
    lens = torch.tensor(lengths, dtype=torch.int32) if lengths else None
    inp = make_inputs(cfg, seed=90 + case, poison_tail=True, lengths=lens)
    _binding.set_split_parts(parts)
    try:
        gpu = run_cuda(inp, num_splits=splits)
    finally:
        _binding.set_split_parts(0)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0, "an index check failed"
    assert gpu["status"] == 0
    ref, bs = run_oracle(inp)
    compare(gpu, ref, bs, "bf16")


def test_bench_workload_under_index_checks(checked):
    lib, flags = checked
    flags.zero_()
    inp = make_inputs(V2LITE_BF16_B8_S4096, seed=3)
    gpu = run_cuda(inp)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0 and gpu["status"] == 0
    ref, bs = run_oracle(inp, batches=[0, 7])
    compare(gpu, ref, bs, "bf16")


def test_default_build_has_no_checks(cuda_lib):
    from head_latent_attention_absorbed_gb300 import _binding
    assert _binding.load(_binding.LIB_PATH).mla_built_with_checks() == 0
