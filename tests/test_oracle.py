"""The CPU oracle against its pins (no GPU)."""

from oracle import attention as A
from oracle import blocks as B
from oracle import paging as P
from tests import pins


def test_address_example():
    pins.check_address_example(P.translate, P.blocks_needed, P.tail_waste)


def test_translate_matches_enumeration():
    pins.check_translate_enumeration(P.translate)


def test_utilization_and_waste():
    pins.check_utilization(P.paged_utilization, P.reserved_utilization,
                           P.mean_tail_waste, P.allocated_slots)


def test_kv_bytes_opt13b():
    pins.check_kv_bytes(P.kv_bytes_per_token)


def test_cow_demo():
    pins.check_cow_demo(B.BlockPool)


def test_fork_workload():
    pins.check_fork_workload(B.BlockPool)


def test_pool_vs_contiguous_lists():
    pins.check_pool_vs_contiguous(B.BlockPool, P.allocated_slots)


def test_write():
    pins.check_write(A.write_tokens)


def test_copy():
    pins.check_copy(A.copy_blocks)


def test_attention_bruteforce():
    pins.check_bruteforce(A.attention)


def test_attention_contiguous_torch():
    pins.check_contiguous_torch(A.attention)


def test_attention_special_cases():
    pins.check_special_cases(A.attention)


def test_attention_gqa_mapping():
    pins.check_gqa_mapping(A.attention)


def test_attention_relabel_invariance():
    pins.check_relabel_invariance(A.attention)


def test_attention_invalid_rows():
    pins.check_invalid_rows(A.attention)


def test_split_merge():
    pins.check_split_merge(A.attention, A.partition_stats, A.merge_partitions)


def test_bf16_widening():
    pins.check_bf16(A.to_f64)


def test_oracle_bruteforce_helper_agrees():
    # The package's own pure-Python helper matches the test's brute force.
    q, kp, vp, tables, lens, b = pins.tiny_case(11)
    keys = [[float(x) for x in r] for r in pins.contiguous_rows(kp, tables[0], lens[0], b, 1)]
    vals = [[float(x) for x in r] for r in pins.contiguous_rows(vp, tables[0], lens[0], b, 1)]
    qr = [float(x) for x in q[0, 1]]
    assert A.attention_bruteforce(qr, keys, vals, 0.3) == pins.brute(qr, keys, vals, 0.3)


def test_swap():
    pins.check_swap(A.swap_blocks, A.copy_blocks)


def test_prefill():
    pins.check_prefill(A.prefill_attention, A.attention)


def test_e4m3():
    pins.check_e4m3(A.e4m3_encode, A.e4m3_decode)


def test_fp8_write_and_attention():
    pins.check_fp8_write_and_attention(A.write_tokens_fp8, A.dequantize_pool, A.attention,
                                       A.e4m3_encode)


def test_fp8_prefill():
    pins.check_fp8_prefill(A.prefill_attention, A.attention, A.dequantize_pool)
