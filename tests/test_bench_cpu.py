"""The bench's algorithmic work per step (the roofline numerators), without a
GPU: prefill FLOPs counted from the visible (query, key) pairs of the
bottom-right causal mask, decode bytes from the INT4 row size, against
hand-computed values for the measured workloads."""

import bench


def test_prefill_flops_by_hand():
    # causal 8192 x 8192: pairs 8192 * 8193 / 2 per head, 2 * 32 heads, 4 * 128 flops each
    assert bench.prefill_flops(2, 32, 8192, 8192, 128, True) == 4.0 * 128 * 64 * (8192 * 8193 // 2)
    assert bench.prefill_flops(2, 32, 8192, 8192, 128, True) == 1099645845504.0
    assert bench.prefill_flops(1, 1, 3, 5, 64, False) == 4.0 * 64 * 15
    # chunked causal, bottom-right: query i of 2 sees keys j <= i + 3 of 5 -> 4 + 5 pairs
    assert bench.prefill_flops(1, 1, 2, 5, 64, True) == 4.0 * 64 * 9
    assert bench.prefill_flops(1, 1, 1, 7, 64, True) == 4.0 * 64 * 7   # one query sees every key


def test_decode_bytes_by_hand():
    # one (token, kv-head) row: D/2 + D/2 code bytes + 2 + 2 scale bytes = 132 at D = 128
    assert bench.workload_config("gqa_decode")["kv_bytes_per_step"] == 8 * 8 * 4096 * 132 == 34603008
    assert bench.workload_config("long_decode")["kv_bytes_per_step"] == 8 * 131072 * 132 == 138412032
    cfg = bench.workload_config("causal_prefill")
    assert cfg["flops_per_step"] == 1099645845504.0 and cfg["causal"] is True
