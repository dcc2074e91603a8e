"""The decode-step model and byte accounting reproduce the figures printed on
"When quantization pays -- and when it does not" (all modelled H100 numbers)."""
import json
import os

import pytest

from weight_only_int4_gemm_gb300 import model

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "decode_step_model.json")))
I, P = G["inputs"], G["printed"]
# Streamed weights of Llama-3-8B from its linear shapes (32 decoder layers of
# qkv 4096->6144, o 4096->4096, gate_up 4096->28672, down 14336->4096, plus the
# 4096->128256 lm_head); the page prints this as 7.50 B.
LAYER = 4096 * 6144 + 4096 * 4096 + 4096 * 28672 + 14336 * 4096
W_EXACT = 32 * LAYER + 4096 * 128256
# The page's own arithmetic uses the rounded W = 7.50e9 (e.g. 7.50 x 0.5156 /
# 3.35 = 1.15 ms), so the model is evaluated with that value.
W = I["W_params"]
BETA = I["beta_bytes_per_s"]
BF16 = model.Scheme(I["b_w_bf16"], I["P_bf16_flops"])
FP8 = model.Scheme(I["b_w_8bit"], I["P_fp8_flops"])
INT4 = model.Scheme(I["b_w_int4_g128"], I["P_bf16_flops"], c=I["c_int4"], issue_rate=I["D_lanes_per_s"])


def test_streamed_weight_count():
    assert W_EXACT == 7_504_658_432
    assert round(W_EXACT / 1e9, 2) == I["W_params"] / 1e9
    assert round(W_EXACT * 2 / 1e9, 2) == P["bf16_bytes_GB"]


def test_effective_bytes_per_weight():
    assert model.BYTES_PER_WEIGHT_SYM * 8 == I["effective_bits_int4_g128"]
    assert round(model.BYTES_PER_WEIGHT_SYM, 4) == I["b_w_int4_g128"]


def test_memory_floors():
    assert round(model.memory_floor(W, BETA, BF16) * 1e3, 2) == P["bf16_floor_ms"]
    assert round(model.memory_floor(W, BETA, FP8) * 1e3, 2) == P["int8_floor_ms"]
    assert round(model.memory_floor(W, BETA, INT4) * 1e3, 2) == P["int4_floor_ms"]


def test_slopes_and_tax():
    assert round(model.mma_slope(W, BF16) * 1e6, 2) == P["bf16_slope_us_per_B"]
    assert round(model.mma_slope(W, FP8) * 1e6, 2) == P["fp8_slope_us_per_B"]
    assert round(model.dequant_tax(W, INT4) * 1e3, 2) == P["dequant_tax_ms"]


def test_regime_boundaries():
    # W4A16 math line meets its own memory floor
    b47 = model.batch_where_math_reaches(model.memory_floor(W, BETA, INT4), W, INT4)
    assert round(b47) == P["B_w4a16_advantage_decays"]
    # ridge with free dequant
    free = model.Scheme(INT4.bytes_per_weight, INT4.tensor_peak)
    m_star = model.batch_where_math_reaches(model.memory_floor(W, BETA, free), W, free)
    assert round(m_star) == P["M_star_free_dequant"]
    assert model.ridge_batch(BETA, INT4.tensor_peak, INT4.bytes_per_weight) == pytest.approx(m_star)
    # bf16 ridge
    b_star = model.batch_where_math_reaches(model.memory_floor(W, BETA, BF16), W, BF16)
    assert round(b_star) == P["B_star_bf16_ridge"]
    # W4A16 math line crosses bf16's memory floor
    b266 = model.batch_where_math_reaches(model.memory_floor(W, BETA, BF16), W, INT4)
    assert round(b266) == P["B_w4a16_stops_paying"]
    # ... and the 8-bit memory floor
    b118 = model.batch_where_math_reaches(model.memory_floor(W, BETA, FP8), W, INT4)
    assert round(b118) == P["B_threshold_int4_vs_8bit_floor"]


def test_deployment_b_at_480():
    # These three figures agree with the unrounded W (with W = 7.50e9 the
    # W4A16 step is 7.725 ms, which prints as 7.72).
    t_fp8 = model.step_time(W_EXACT, 480, BETA, FP8)
    t_bf16 = model.step_time(W_EXACT, 480, BETA, BF16)
    t_int4 = model.step_time(W_EXACT, 480, BETA, INT4)
    assert round(t_fp8 * 1e3, 2) == P["B480_fp8_ms"]
    assert round(t_bf16 * 1e3, 2) == P["B480_bf16_ms"]
    assert round(t_int4 * 1e3, 2) == P["B480_w4a16_ms"]
    assert round((t_int4 - t_bf16) / t_bf16 * 100) == P["B480_tax_share_percent"]


def test_deployment_a_at_3():
    assert round(model.step_time(W, 3, BETA, INT4) * 1e3, 2) == P["int4_floor_ms"]
    assert round(model.step_time(W, 3, BETA, BF16) * 1e3, 2) == P["bf16_floor_ms"]


def test_linear_byte_and_flop_accounting():
    # K*N/2 codes + K/128*N bf16 scales + x + y
    assert model.linear_bytes(1, 4096, 4096) == 8388608 + 262144 + 8192 + 8192
    assert model.linear_bytes(1, 4096, 4096, zero_points=True) == 8388608 + 262144 + 65536 + 8192 + 8192
    assert model.linear_flops(16, 4096, 28672) == 2 * 16 * 4096 * 28672
    # at B = 0 the weight stream alone is 4.125 / 4.15625 bits per weight
    assert (model.linear_bytes(0, 8192, 8192) * 8) / (8192 * 8192) == 4.125
    assert (model.linear_bytes(0, 8192, 8192, True) * 8) / (8192 * 8192) == 4.15625
