"""Host logic of bench.py that needs no GPU: the BLAS thread query of the CPU
baseline, and the oracle check of the last timed step (it must pass on the
oracle's own outputs and fail on a perturbed copy)."""
import numpy as np

import bench
from oracle import mla_oracle as O
from workloads import V2LITE_F32_B1_S64, make_inputs


def test_blas_threads_reads_a_count():
    lib, n = bench.blas_threads()
    assert lib is None or (isinstance(n, int) and n >= 1)


def test_oracle_check_accepts_exact_and_rejects_perturbed():
    cfg = V2LITE_F32_B1_S64
    a = make_inputs(cfg, seed=0).as_float64_numpy()
    r = O.decode_absorbed(a["q_nope"], a["q_rope"], a["w_uk"], a["w_uv"], a["cache"],
                          a["lengths"], a["positions"], cfg.softmax_scale, cfg.rope_base)
    out = {k: r[k].copy() for k in ("o", "o_c", "lse")}
    assert bench.oracle_check(cfg, out, seed=0)["ok"]
    out["o_c"][0, 3, 7] += 1e-3
    res = bench.oracle_check(cfg, out, seed=0)
    assert not res["ok"] and res["o_c"]["max_abs"] > 9e-4
