"""Plain fp64 CPU oracle for one MLA decode step (naive and weight-absorbed).

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import or run this module.  It shares no code
with the CUDA library and imports nothing from it.  It is slow on purpose:
every function is the plain definition written out with NumPy in float64, with
no blocking, fusion or reordering beyond what the definition states.

Sources (web pages, cited by title and section):

* "Multi-Head Latent Attention" (Lior Sinai), section 2.1 "KV Caching / Theory":
  decoding with a cache gives exactly the last column of full attention.
* same page, section 3.1 "C cache": K and V are recovered from the cached
  latent C^KV by W^UK and W^UV.
* same page, section 3.3 "Absorption" and eq. 3.3.3: the per-head score
  C^KV^T (W^UK^T q) and the output W^UV (C^KV z) need no decompressed K or V.
* same page, section 3.6 "Decoupled RoPE": scores add a RoPE part
  k^R . q^R, k^R is shared by all heads, and the sum is scaled by
  1/sqrt(d_h + d_R).
* same page, section 3.7 "Code": RoPE as a complex multiply of adjacent pairs
  by cos + i sin of (position * theta_i), theta_i = base^(-2i/dim), positions
  counted from 0.
* "Deepseek V2 Lite Inference Engine in C", MLA notes: the fused row order
  (kv_lora, k_rope) of kv_a_proj, and kv_b_proj's per-head interleaved
  [k_nope ; v] row blocks, which the naive form below rebuilds.
* "Transformer and KV Cache Basics", Engineering item 4: masked positions get
  -inf before the softmax.

Every function here is pinned by ``tests/test_oracle_pins.py`` against facts
that the pages and mathematics fix (closed forms, brute force, invariants).

Array conventions (row-major, per sequence b):
  cache[b, t, :d_c]  = c_kv row of token t;  cache[b, t, d_c:] = k_rope row (already rotated)
  q_nope[b, h, :d_nope], q_rope[b, h, :d_rope]
  w_uk[h, d, c]  (W^UK of head h, d_nope x d_c)   w_uv[h, e, c]  (W^UV of head h, d_v x d_c)
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------------------- RoPE
def rope_theta(d_rope: int, base: float) -> np.ndarray:
    """theta_i = base^(-(2i)/d_rope), i = 0 .. d_rope/2 - 1 (Multi-Head Latent Attention, 3.7)."""
    if d_rope % 2:
        raise ValueError("RoPE needs an even width")
    i = np.arange(d_rope // 2, dtype=np.float64)
    return np.float64(base) ** (-(2.0 * i) / d_rope)


def apply_rope(x: np.ndarray, pos, base: float) -> np.ndarray:
    """Rotate adjacent pairs (x[2i], x[2i+1]) as the complex number x[2i] + i x[2i+1]
    by exp(i * pos * theta_i) (Multi-Head Latent Attention, 3.7).

    x: [..., d_rope]; pos: scalar or an array broadcastable to x.shape[:-1].
    """
    x = np.asarray(x, dtype=np.float64)
    theta = rope_theta(x.shape[-1], base)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * (np.cos(ang) + 1j * np.sin(ang))
    out = np.empty_like(x)
    out[..., 0::2] = z.real
    out[..., 1::2] = z.imag
    return out


# ----------------------------------------------------------------------------- absorbed form
def absorb_q(q_nope: np.ndarray, w_uk: np.ndarray) -> np.ndarray:
    """q_abs[b,h,c] = sum_d q_nope[b,h,d] * w_uk[h,d,c]: the query contracted with W^UK
    before it meets the cache (Multi-Head Latent Attention, 3.3; the right-to-left
    order of the einsum quoted there)."""
    return np.einsum("bhd,hdc->bhc", q_nope, w_uk)


def softmax_stats(s: np.ndarray):
    """Exact softmax over the last axis: returns (p, lse) with lse = log sum exp(s)."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = np.sum(e, axis=-1, keepdims=True)
    return e / z, (m + np.log(z))[..., 0]


def decode_absorbed(q_nope, q_rope, w_uk, w_uv, cache, lengths, positions,
                    scale: float, base: float):
    """One decode step in weight-absorbed form, exact softmax, no splits.

    Returns a dict of fp64 arrays: q_abs [B,H,d_c], q_pe [B,H,d_rope],
    o_c [B,H,d_c] (latent output), lse [B,H] (natural log of the softmax
    normaliser of the scaled scores), o [B,H,d_v], and p (list over b of [H,S_b]).
    """
    B, H, _ = q_nope.shape
    d_c = w_uk.shape[2]
    q_abs = absorb_q(q_nope, w_uk)
    q_pe = apply_rope(q_rope, np.asarray(positions)[:, None], base)
    o_c = np.zeros((B, H, d_c))
    lse = np.full((B, H), -np.inf)
    o = np.zeros((B, H, w_uv.shape[1]))
    ps = []
    for b in range(B):
        n = int(lengths[b])
        if n <= 0:
            raise ValueError("a sequence with no cached rows has no softmax")
        c = cache[b, :n, :d_c]          # [S_b, d_c]
        kr = cache[b, :n, d_c:]         # [S_b, d_rope]
        s = scale * (q_abs[b] @ c.T + q_pe[b] @ kr.T)     # [H, S_b]
        p, lse[b] = softmax_stats(s)
        o_c[b] = p @ c                                     # latent output, d_c per head
        o[b] = np.einsum("hec,hc->he", w_uv, o_c[b])        # W^UV applied after attention
        ps.append(p)
    return dict(q_abs=q_abs, q_pe=q_pe, o_c=o_c, lse=lse, o=o, p=ps)


# ----------------------------------------------------------------------------- naive form
def kv_b_proj_from(w_uk: np.ndarray, w_uv: np.ndarray) -> np.ndarray:
    """Fused up-projection with per-head interleaved row blocks [k_nope(h); v(h)]
    ("Deepseek V2 Lite Inference Engine in C", MLA notes): shape [H*(d_nope+d_v), d_c]."""
    H, d_nope, d_c = w_uk.shape
    d_v = w_uv.shape[1]
    w = np.empty((H, d_nope + d_v, d_c))
    w[:, :d_nope] = w_uk
    w[:, d_nope:] = w_uv
    return w.reshape(H * (d_nope + d_v), d_c)


def decode_naive(q_nope, q_rope, w_uk, w_uv, cache, lengths, positions,
                 scale: float, base: float):
    """One decode step without absorption: decompress every cached row into per-head
    K and V through kv_b_proj, then standard multi-head attention with the decoupled
    RoPE part concatenated (Multi-Head Latent Attention, 3.1 and 3.7; "Deepseek V2
    Lite Inference Engine in C", "Use original weights").

    Returns dict(o [B,H,d_v], p list of [H,S_b]).
    """
    B, H, d_nope = q_nope.shape
    d_c = w_uk.shape[2]
    d_v = w_uv.shape[1]
    kvb = kv_b_proj_from(w_uk, w_uv)
    q_pe = apply_rope(q_rope, np.asarray(positions)[:, None], base)
    o = np.zeros((B, H, d_v))
    ps = []
    for b in range(B):
        n = int(lengths[b])
        c = cache[b, :n, :d_c]
        kr = cache[b, :n, d_c:]
        kv = (c @ kvb.T).reshape(n, H, d_nope + d_v)       # [S, H, 256]
        k_nope, v = kv[..., :d_nope], kv[..., d_nope:]
        Q = np.concatenate([q_nope[b], q_pe[b]], axis=-1)   # [H, 192]
        K = np.concatenate([k_nope, np.broadcast_to(kr[:, None, :], (n, H, kr.shape[1]))],
                           axis=-1)                          # [S, H, 192], k_rope shared
        s = scale * np.einsum("hk,thk->ht", Q, K)
        p, _ = softmax_stats(s)
        o[b] = np.einsum("ht,the->he", p, v)
        ps.append(p)
    return dict(o=o, p=ps)


def causal_attention_naive(q_nope_seq, q_rope_seq, w_uk, w_uv, cache_seq, scale, base):
    """Full causal self-attention over one sequence of S tokens, every query row i
    rotated at position i, future keys masked with -inf ("Transformer and KV Cache
    Basics", item 4; Multi-Head Latent Attention, 2.1).  q_*_seq: [S,H,*];
    cache_seq: [S,row].  Returns outputs [S,H,d_v]."""
    S, H, d_nope = q_nope_seq.shape
    d_c = w_uk.shape[2]
    d_v = w_uv.shape[1]
    kvb = kv_b_proj_from(w_uk, w_uv)
    c, kr = cache_seq[:, :d_c], cache_seq[:, d_c:]
    kv = (c @ kvb.T).reshape(S, H, d_nope + d_v)
    k_nope, v = kv[..., :d_nope], kv[..., d_nope:]
    q_pe = apply_rope(q_rope_seq, np.arange(S)[:, None], base)
    Q = np.concatenate([q_nope_seq, q_pe], axis=-1)                       # [S,H,192]
    K = np.concatenate([k_nope, np.broadcast_to(kr[:, None, :], (S, H, kr.shape[1]))], -1)
    s = scale * np.einsum("ihk,jhk->hij", Q, K)                           # [H, S_q, S_k]
    future = np.arange(S)[:, None] < np.arange(S)[None, :]
    s = np.where(future[None], -np.inf, s)
    p, _ = softmax_stats(s)
    return np.einsum("hij,jhe->ihe", p, v)


# ----------------------------------------------------------------------------- multi-token decode
def decode_multi_token(q_nope, q_rope, w_uk, w_uv, cache, lengths, q_len: int,
                       scale: float, base: float):
    """Decode of q_len new tokens per sequence in one step (speculative or
    multi-token decoding), weight-absorbed, exact softmax.

    "Transformer and KV Cache Basics", Thinking item 4 (mask design): prefill and
    decode are treated alike; the cache already holds the new tokens, so with
    k_len cached rows the q_len queries sit at positions k_len - q_len .. k_len - 1
    and a key is masked when its position is past the query's (the small upper
    right triangle of the score matrix).  Each query is rotated at its own
    position (Multi-Head Latent Attention, 3.7).

    q_nope: [B, q_len, H, d_nope]; q_rope: [B, q_len, H, d_rope]; lengths: [B] (k_len).
    Returns dict(q_abs, q_pe, o_c, lse, o) with leading dims [B, q_len].
    """
    q_nope = np.asarray(q_nope, dtype=np.float64)
    B, T, H, _ = q_nope.shape
    if T != q_len:
        raise ValueError("q_nope's second axis is the token axis of length q_len")
    d_c = w_uk.shape[2]
    lengths = np.asarray(lengths)
    if np.any(lengths < q_len):
        raise ValueError("every sequence must already cache its q_len new tokens")
    query_pos = lengths[:, None] - q_len + np.arange(q_len)[None, :]            # [B, T]
    q_abs = absorb_q(q_nope.reshape(B * T, H, -1), w_uk).reshape(B, T, H, d_c)
    q_pe = apply_rope(q_rope, query_pos[..., None], base)                       # [B, T, H, d_R]
    o_c = np.zeros((B, T, H, d_c))
    lse = np.zeros((B, T, H))
    o = np.zeros((B, T, H, w_uv.shape[1]))
    for b in range(B):
        n = int(lengths[b])
        c, kr = cache[b, :n, :d_c], cache[b, :n, d_c:]
        s = scale * (np.einsum("thc,sc->ths", q_abs[b], c) + np.einsum("thr,sr->ths", q_pe[b], kr))
        future = query_pos[b][:, None] < np.arange(n)[None, :]                  # [T, n]
        s = np.where(future[:, None, :], -np.inf, s)
        p, lse[b] = softmax_stats(s)
        o_c[b] = np.einsum("ths,sc->thc", p, c)
        o[b] = np.einsum("hec,thc->the", w_uv, o_c[b])
    return dict(q_abs=q_abs, q_pe=q_pe, o_c=o_c, lse=lse, o=o)


# ----------------------------------------------------------------------------- split-KV combine
def split_decode_combine(q_abs, q_pe, cache_b, n: int, scale: float, chunk: int):
    """Split-KV for one sequence: per chunk j of `chunk` rows compute the chunk's
    normalised latent output o_j and lse_j, then merge with
    L = log sum_j exp(lse_j), o_c = sum_j exp(lse_j - L) o_j.  An exact rewrite of
    the softmax over all rows (used to check the combine arithmetic).
    q_abs [H,d_c], q_pe [H,d_rope], cache_b [S,row].  Returns (o_c [H,d_c], lse [H])."""
    d_c = q_abs.shape[1]
    os_, ls_ = [], []
    for t0 in range(0, n, chunk):
        t1 = min(n, t0 + chunk)
        c, kr = cache_b[t0:t1, :d_c], cache_b[t0:t1, d_c:]
        s = scale * (q_abs @ c.T + q_pe @ kr.T)
        p, l = softmax_stats(s)
        os_.append(p @ c)
        ls_.append(l)
    lse = np.stack(ls_)                       # [J, H]
    L = np.max(lse, axis=0) + np.log(np.sum(np.exp(lse - np.max(lse, axis=0)), axis=0))
    w = np.exp(lse - L)                       # [J, H]
    o_c = np.einsum("jh,jhc->hc", w, np.stack(os_))
    return o_c, L


# ----------------------------------------------------------------------------- around the path
def cache_append_row(x: np.ndarray, w_kva: np.ndarray, pos, d_c: int, base: float) -> np.ndarray:
    """The cache row of one new token per sequence.

    "Deepseek V2 Lite Inference Engine in C", MLA notes: one fused down-projection
    kv_a_proj [d_c + d_rope, hidden] maps the token's hidden state to
    (kv_lora, k_rope).  "Multi-Head Latent Attention" 3.5: the latent part is
    what the cache stores; 3.7: the RoPE key is rotated at the token's position
    before it is cached (the decode then uses it as stored).

    x: [B, hidden]; w_kva: [d_c + d_rope, hidden]; pos: [B].  Returns [B, d_c + d_rope]:
    [x . w_kva[:d_c]^T  ||  RoPE(x . w_kva[d_c:]^T, pos)].
    """
    y = np.asarray(x, dtype=np.float64) @ np.asarray(w_kva, dtype=np.float64).T
    out = y.copy()
    out[:, d_c:] = apply_rope(y[:, d_c:], np.asarray(pos), base)
    return out


def output_projection(o: np.ndarray, w_o: np.ndarray) -> np.ndarray:
    """The attention layer's output: the heads' value outputs concatenated and
    multiplied by W^O ("Multi-Head Latent Attention", eq. 3.3.3: W^O applied to the
    concatenated per-head outputs).

    o: [B, H, d_v]; w_o: [hidden, H * d_v].  Returns [B, hidden].
    """
    o = np.asarray(o, dtype=np.float64)
    return o.reshape(o.shape[0], -1) @ np.asarray(w_o, dtype=np.float64).T


# ----------------------------------------------------------------------------- materialised absorption
def materialize_wkq(w_q_nope: np.ndarray, w_uk: np.ndarray) -> np.ndarray:
    """W^KQ_h = (W^UK_h)^T W^UQ_h for every head h: the absorption's query-side
    product written out once as a matrix ("Multi-Head Latent Attention", 3.3: the
    dimensional analysis gives W^KQ one d_c-row slice per head; 3.5 forms it by a
    batched product of W^UK transposed with W^UQ; "Deepseek V2 Lite Inference Engine
    in C", MLA notes: the materialised WukWq of shape (16, 2048, 512)).

    w_q_nope: [H, d_nope, d_in], the rows of the query projection whose output meets
    the latent keys (q_nope = w_q_nope[h] x); w_uk: [H, d_nope, d_c].
    Returns [H, d_c, d_in]: q_abs[b, h, :] = W^KQ[h] x_b.
    """
    w_q_nope = np.asarray(w_q_nope, dtype=np.float64)
    w_uk = np.asarray(w_uk, dtype=np.float64)
    H, d_nope, d_c = w_uk.shape
    out = np.empty((H, d_c, w_q_nope.shape[2]))
    for h in range(H):
        out[h] = w_uk[h].T @ w_q_nope[h]
    return out


def materialize_wov(w_o: np.ndarray, w_uv: np.ndarray) -> np.ndarray:
    """W^OV = W^O W^UV with the head dimension kept ("Multi-Head Latent Attention",
    eq. 3.3.3, Y = W^O V Z = W^OV C^KV Z; 3.5 reshapes W^O to (d_out, d_h, H) and
    multiplies each head's block by W^UV of that head): column block h of W^OV
    (d_c wide) is W^O's column block h (d_v wide) times W^UV_h.

    w_o: [d_out, H * d_v]; w_uv: [H, d_v, d_c].  Returns [d_out, H * d_c].
    """
    w_o = np.asarray(w_o, dtype=np.float64)
    w_uv = np.asarray(w_uv, dtype=np.float64)
    H, d_v, d_c = w_uv.shape
    out = np.empty((w_o.shape[0], H * d_c))
    for h in range(H):
        out[:, h * d_c:(h + 1) * d_c] = w_o[:, h * d_v:(h + 1) * d_v] @ w_uv[h]
    return out


def decode_materialized(x, q_rope, w_kq, w_ov, cache, lengths, positions,
                        scale: float, base: float):
    """One decode step in the materialised absorbed form: the absorbed query is
    W^KQ x (no q_nope in between), the latent attention is that of the absorbed
    form (3.3, 3.6), and the layer output is W^OV applied to the heads' latent
    outputs concatenated (eq. 3.3.3).

    x: [B, d_in]; q_rope: [B, H, d_rope]; w_kq: [H, d_c, d_in]; w_ov: [d_out, H*d_c].
    Returns dict(q_abs [B,H,d_c], q_pe [B,H,d_rope], o_c [B,H,d_c], lse [B,H],
    y [B, d_out]).
    """
    x = np.asarray(x, dtype=np.float64)
    w_kq = np.asarray(w_kq, dtype=np.float64)
    H, d_c, _ = w_kq.shape
    B = x.shape[0]
    q_abs = np.einsum("hci,bi->bhc", w_kq, x)
    q_pe = apply_rope(q_rope, np.asarray(positions)[:, None], base)
    o_c = np.zeros((B, H, d_c))
    lse = np.full((B, H), -np.inf)
    for b in range(B):
        n = int(lengths[b])
        if n <= 0:
            raise ValueError("a sequence with no cached rows has no softmax")
        c, kr = cache[b, :n, :d_c], cache[b, :n, d_c:]
        s = scale * (q_abs[b] @ c.T + q_pe[b] @ kr.T)
        p, lse[b] = softmax_stats(s)
        o_c[b] = p @ c
    y = o_c.reshape(B, H * d_c) @ np.asarray(w_ov, dtype=np.float64).T
    return dict(q_abs=q_abs, q_pe=q_pe, o_c=o_c, lse=lse, y=y)


# ----------------------------------------------------------------------------- FP8 cache elements
def e4m3_to_float64(codes) -> np.ndarray:
    """Values of FP8 E4M3 codes ("Multi-Head Latent Attention" 3.1: a cached element
    takes one to four bytes, FP8 to FP32).

    The E4M3 format used for caches (finite-only): bit 7 the sign, bits 6-3 the
    exponent with bias 7, bits 2-0 the mantissa.  Exponent field 0 holds the
    subnormals (m / 8) 2^-6; otherwise the value is (1 + m / 8) 2^(e - 7).  The one
    pattern with all exponent and mantissa bits set is NaN (there are no
    infinities), so the largest magnitude is 1.75 * 2^8 = 448.
    """
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where((c & 0x80) != 0, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    return np.where((e == 15) & (m == 7), np.nan, sign * mag)


def e4m3_round(x) -> np.ndarray:
    """E4M3 code of the value nearest to x (uint8), ties to the code whose last
    mantissa bit is 0, magnitudes past 448 saturated to 448, NaN to NaN: the
    rounding of a value into an FP8 cache.  Written as the definition: the
    nearest of the 254 finite E4M3 values, by exhaustive comparison.
    """
    x = np.asarray(x, dtype=np.float64)
    codes = np.array([c for c in range(256) if not np.isnan(e4m3_to_float64(c))], dtype=np.int64)
    vals = e4m3_to_float64(codes)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    for i, v in enumerate(flat):
        if np.isnan(v):
            out[i] = 0x7F
            continue
        v = min(max(v, -448.0), 448.0)
        d = np.abs(vals - v)
        near = codes[d == d.min()]
        if len(near) > 1:
            even = near[(near & 1) == 0]
            near = even if len(even) else near
        # zero keeps the sign of x
        if vals[np.searchsorted(codes, near[0])] == 0.0:
            out[i] = 0x80 if np.signbit(v) else 0x00
        else:
            out[i] = near[0]
    return out.reshape(x.shape)
