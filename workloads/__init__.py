"""Seeded synthetic MLA decode workloads shared by the tests, the smoke check and the bench.

Holds sizes and random draws only; no arithmetic of the method lives here.
"""
from .configs import (ALL_CONFIGS, BY_NAME, FP8_CONFIGS, MULTI_TOKEN_CONFIGS, MlaConfig,
                      TOL_BF16_MAX_ABS, V2LITE_BF16_B8_S4096_Q4, V2LITE_FP8_B8_S4096_Q4,
                      TOL_BF16_REL_L2, TOL_F32_MAX_ABS, V2LITE_BF16_B4_S65536_LONG,
                      V2LITE_BF16_B8_S4096, V2LITE_BF16_B64_RAGGED, V2LITE_F32_B1_S64,
                      V2LITE_FP8_B4_S65536_LONG, V2LITE_FP8_B8_S4096, V2LITE_FP8_B64_RAGGED,
                      V3_BF16_H128_B32_S16384, V3_FP8_H128_B32_S16384)
from .generate import (FP8, AppendInputs, MaterializedInputs, MlaInputs, OutProjInputs,
                       cache_storage, make_append_inputs, make_inputs, make_materialized_inputs,
                       make_wo_inputs)

__all__ = [
    "ALL_CONFIGS", "BY_NAME", "FP8_CONFIGS", "MULTI_TOKEN_CONFIGS", "V2LITE_BF16_B8_S4096_Q4",
    "V2LITE_FP8_B8_S4096_Q4", "MlaConfig", "MlaInputs", "make_inputs",
    "AppendInputs", "make_append_inputs", "OutProjInputs", "make_wo_inputs", "FP8",
    "MaterializedInputs", "make_materialized_inputs",
    "cache_storage", "TOL_BF16_MAX_ABS", "TOL_BF16_REL_L2", "TOL_F32_MAX_ABS",
    "V2LITE_F32_B1_S64", "V2LITE_BF16_B8_S4096", "V2LITE_BF16_B64_RAGGED",
    "V3_BF16_H128_B32_S16384", "V2LITE_BF16_B4_S65536_LONG", "V2LITE_FP8_B8_S4096",
    "V2LITE_FP8_B64_RAGGED", "V3_FP8_H128_B32_S16384", "V2LITE_FP8_B4_S65536_LONG",
]
