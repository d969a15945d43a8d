"""The C-ABI library builds, loads, exports every symbol its header declares, and
rejects bad arguments on the host before launching anything (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def lib():
    from head_latent_attention_absorbed_gb300 import build as b
    path = b.build()
    import head_latent_attention_absorbed_gb300 as mla
    return mla, mla.load(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("mla_absorb_q", "mla_decode_attn", "mla_out_proj"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    mla, so = lib
    names = declared_functions()
    out = subprocess.run(["nm", "-D", "--defined-only", mla.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for n in names:
        assert n in exported, n
        assert hasattr(so, n)
    assert set(mla.EXPORTED) <= set(names)


def test_status_strings(lib):
    _, so = lib
    so.mla_status_string.restype = ctypes.c_char_p
    assert so.mla_status_string(0) == b"MLA_OK"
    assert so.mla_status_string(3) == b"MLA_ERR_WORKSPACE"


def _d(mla, **kw):
    base = dict(batch=2, heads=16, s_max=100, dtype=mla.MLA_BF16)
    base.update(kw)
    return mla.dims(base["batch"], base["heads"], base["s_max"], base["dtype"])


def test_host_validation(lib):
    mla, so = lib
    P = ctypes.c_void_p
    good = 0x10000
    d = _d(mla)
    # NULL pointer
    assert so.mla_decode_attn(ctypes.byref(d), None, P(good), P(good), P(good), 0.1, 0, P(good),
                              1 << 30, P(good), None, None, None) == 1
    # misaligned cache
    assert so.mla_decode_attn(ctypes.byref(d), P(good), P(good), P(good + 2), P(good), 0.1, 0,
                              P(good), 1 << 30, P(good), None, None, None) == 1
    # workspace too small
    assert so.mla_decode_attn(ctypes.byref(d), P(good), P(good), P(good), P(good), 0.1, 0,
                              P(good), 16, P(good), None, None, None) == 3
    assert b"workspace" in so.mla_last_error_message()
    # unsupported sizes
    bad = _d(mla, heads=15)
    assert so.mla_decode_attn(ctypes.byref(bad), P(good), P(good), P(good), P(good), 0.1, 0,
                              P(good), 1 << 30, P(good), None, None, None) == 2
    bad = mla.dims(2, 16, 100, mla.MLA_BF16, d_c=256)
    assert so.mla_absorb_q(ctypes.byref(bad), P(good), P(good), P(good), P(good), 1e4, P(good),
                           P(good), None) == 2
    bad = mla.dims(0, 16, 100, mla.MLA_BF16)
    assert so.mla_out_proj(ctypes.byref(bad), P(good), P(good), P(good), None) == 1
    # negative split request, non-positive scale, bad rope base
    assert so.mla_decode_attn(ctypes.byref(d), P(good), P(good), P(good), P(good), 0.1, -1,
                              P(good), 1 << 30, P(good), None, None, None) == 1
    assert so.mla_decode_attn(ctypes.byref(d), P(good), P(good), P(good), P(good), 0.0, 0,
                              P(good), 1 << 30, P(good), None, None, None) == 1
    assert so.mla_absorb_q(ctypes.byref(d), P(good), P(good), P(good), P(good), -1.0, P(good),
                           P(good), None) == 1


def test_split_planning(lib):
    mla, _ = lib
    # explicit requests: chunks are multiples of 8 rows
    d = mla.dims(4, 16, 65536, mla.MLA_BF16)
    assert mla.num_splits(d, 128) == 128
    assert mla.num_splits(mla.dims(1, 16, 256, mla.MLA_F32), 7) == 7    # 40-row chunks
    assert mla.num_splits(mla.dims(1, 16, 20, mla.MLA_F32), 7) == 3     # 8-row chunks: 8, 8, 4
    assert mla.num_splits(mla.dims(1, 16, 300, mla.MLA_F32), 3) == 3    # ceil(300/3)=100 -> 104-row chunks
    assert mla.num_splits(mla.dims(1, 16, 1, mla.MLA_F32), 5) == 1
    # workspace grows with splits: B*splits*H*(512+1) floats (256-byte aligned pieces)
    n = 4 * 128 * 16
    ws = mla.workspace_bytes(d, 128)
    assert ws >= n * 513 * 4 and ws < n * 513 * 4 + 512
    # automatic choice is a valid split count
    for (B, H, S) in [(8, 16, 4096), (64, 16, 8192), (32, 128, 16384), (1, 16, 64)]:
        s = mla.num_splits(mla.dims(B, H, S, mla.MLA_BF16), 0)
        assert 1 <= s <= (S + 7) // 8


def test_host_validation_of_later_calls(lib):
    """Argument errors of the multi-token and materialised calls come back as a
    status before anything is launched (no GPU needed)."""
    mla, so = lib
    P = ctypes.c_void_p
    good = 0x10000
    d = _d(mla)
    # multi-token: q_len must be >= 1; the workspace is sized for B * q_len query rows
    assert so.mla_decode_attn_multi(ctypes.byref(d), 0, P(good), P(good), P(good), P(good), 0.1,
                                    0, P(good), 1 << 30, P(good), None, None, None) == 1
    need = mla.multi_workspace_bytes(d, 4, 0)
    assert need > mla.workspace_bytes(d, 0)
    assert mla.multi_workspace_bytes(d, 1, 0) == mla.workspace_bytes(d, 0)
    assert mla.multi_num_splits(d, 1, 0) == mla.num_splits(d, 0)
    assert so.mla_decode_attn_multi(ctypes.byref(d), 4, P(good), P(good), P(good), P(good), 0.1,
                                    0, P(good), need - 1, P(good), None, None, None) == 3
    assert so.mla_decode_attn_multi(ctypes.byref(d), 4, P(good), P(good), P(good), None, 0.1,
                                    0, P(good), need, P(good), None, None, None) == 1
    # materialised form: d_in a multiple of 64, d_out a multiple of 8, no NULLs
    assert so.mla_absorb_q_materialized(ctypes.byref(d), 100, P(good), P(good), P(good), P(good),
                                        1e4, P(good), P(good), None) == 2
    assert so.mla_absorb_q_materialized(ctypes.byref(d), 128, None, P(good), P(good), P(good),
                                        1e4, P(good), P(good), None) == 1
    assert so.mla_ov_proj(ctypes.byref(d), 2044, P(good), P(good), P(good), None) == 2
    assert so.mla_ov_proj(ctypes.byref(d), 2048, P(good), None, P(good), None) == 1
    assert so.mla_materialize_wkq(ctypes.byref(d), 0, P(good), P(good), P(good), None) == 1
    assert so.mla_materialize_wov(ctypes.byref(d), 2048, P(good), P(good), P(good + 4), None) == 1


def test_planner_prefers_whole_tiles(lib):
    """bf16 and FP8 chunks are costed in whole 128-row tiles: 8 sequences of 4096
    rows take 16 chunks of 256 rows (one wave on 148 or 152 SMs), not 18-19
    chunks whose last tile is partial; the fp32 kernel, which has no tiles, is
    planned on rows."""
    mla, _ = lib
    for dt in (mla.MLA_BF16, mla.MLA_FP8_E4M3):
        assert mla.num_splits(mla.dims(8, 16, 4096, dt), 0) == 16
    s32 = mla.num_splits(mla.dims(8, 16, 4096, mla.MLA_F32), 0)
    assert 1 <= s32 <= 512


def test_multi_token_planning_counts_paired_ctas(lib):
    """With a bf16 cache, 16 heads and an even q_len, two tokens share a CTA, so
    the multi-token planner fills the GPU with more chunks than the unpaired one
    would; its workspace covers every (sequence, token, head, chunk) partial."""
    mla, _ = lib
    d = mla.dims(8, 16, 4096, mla.MLA_BF16)
    paired = mla.multi_num_splits(d, 4, 0)
    unpaired = mla.num_splits(mla.query_dims(d, 4), 0)
    assert paired > unpaired
    assert mla.multi_workspace_bytes(d, 4, 0) == mla.workspace_bytes(mla.query_dims(d, 4), paired)
    # odd q_len, FP8 and 32-head caches are not paired
    for dd, q in ((d, 3), (mla.dims(8, 16, 4096, mla.MLA_FP8_E4M3), 4),
                  (mla.dims(8, 32, 4096, mla.MLA_BF16), 4)):
        assert mla.multi_num_splits(dd, q, 0) == mla.num_splits(mla.query_dims(dd, q), 0)


def test_split_parts_switch(lib):
    """Heads per split CTA under mla_set_split_parts (host logic, no GPU): one
    bf16 part and 64 heads per CTA at multiples of 64 heads by default, hi + lo
    parts (32 or 16 heads) when asked; other values are refused."""
    mla, so = lib
    hp = lambda H, dt=mla.MLA_BF16: so.mla_decode_heads_per_cta(ctypes.byref(mla.dims(2, H, 256, dt)))
    try:
        assert [hp(H) for H in (16, 32, 48, 64, 128, 192)] == [16, 32, 16, 64, 64, 64]
        assert hp(128, mla.MLA_FP8_E4M3) == 16 and hp(128, mla.MLA_F32) == 1
        assert so.mla_set_split_parts(1) == 1 and so.mla_set_split_parts(-3) == 1
        assert hp(128) == 64                               # a refused value changes nothing
        assert so.mla_set_split_parts(2) == 0
        assert [hp(H) for H in (16, 32, 48, 64, 128)] == [16, 32, 16, 32, 32]
        # the planner counts the CTAs of the form in force
        d = mla.dims(32, 128, 16384, mla.MLA_BF16)
        assert mla.num_splits(d, 0) >= 1
    finally:
        so.mla_set_split_parts(0)
    assert so.mla_decode_heads_per_cta(ctypes.byref(mla.dims(0, 16, 64, mla.MLA_BF16))) == 0
