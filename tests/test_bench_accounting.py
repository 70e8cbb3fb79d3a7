"""bench.py's roofline numerators (CPU): the algorithmic bytes and flops it divides by each measured
time, restated from their definitions (the method's operand sizes and its chunkwise product count),
so that a drift in either fails here."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

D, C = 128, 64  # head dims and chunk of the measured workloads
BF16, FP32 = 2, 4


def test_prefill_bytes_and_flops_per_token_head():
    # q, k, v in bf16, g in fp32, beta in fp32, out in bf16
    assert bench.PREFILL_BYTES_PER_TOKEN_HEAD == 3 * D * BF16 + D * FP32 + FP32 + D * BF16 == 1540
    # five C x d products per token (A, M, T.V, T.K^, M.U) and three d x d (W S, Q^ S, K_^T U)
    assert bench.PREFILL_FLOPS_PER_TOKEN_HEAD == 2 * (5 * C * D + 3 * D * D) == 180224
    assert bench.PREFILL_BYTES_PER_TOKEN_HEAD * 8192 * 32 == 403701760  # the bench's prefill workload


def test_prefill_bytes_for_other_head_sizes():
    # the same operands at dk = dv = d; the 128-dim figure is the constant above
    for d in (64, 128):
        assert bench.prefill_bytes_per_token_head(d, d) == 3 * d * BF16 + d * FP32 + FP32 + d * BF16
    assert bench.prefill_bytes_per_token_head(128, 128) == bench.PREFILL_BYTES_PER_TOKEN_HEAD
    assert bench.prefill_bytes_per_token_head(64, 64) == 772
    assert bench.prefill_bytes_per_token_head(64, 64) * 8192 * 32 + 32 * 64 * 64 * FP32 == 202899456  # with hT


def test_decode_and_verify_bytes():
    state = D * D * FP32
    assert bench.DECODE_STATE_BYTES == 2 * state  # read and written once
    io = 3 * D * BF16 + D * FP32 + FP32 + D * BF16 + D * BF16  # q, k, v, g, beta, gate, out
    assert bench.DECODE_IO_BYTES_PER_TOKEN_HEAD == io == 1796
    assert (2 * state + io) * 256 * 32 == 1088454656  # one decode step of the bench workload (1.088 GB)
    assert (state + 4 * io) * 256 * 32 == 595722240  # verify: state read once, four tokens of I/O


def test_backward_flop_count_per_chunk_head():
    # 14 C x C x d products, 8 C x d x d and 2 C^3 (X^T dX X^T)
    assert bench.BWD_FLOPS_PER_CHUNK_HEAD == 2 * (14 * C * C * D + 8 * C * D * D + 2 * C ** 3)
    assert bench.BWD_FLOPS_PER_CHUNK_HEAD * (8192 // C) * 32 == 133143986176
