"""Planted mistakes in copies of the oracle must fail the pins (no GPU).

Each case edits one line of an oracle function's source (a dropped term, a
wrong index, a swapped operand), compiles the edited copy in a private
namespace, and runs the pin that should catch it.  The real oracle modules
are never modified.
"""

import inspect
import textwrap

import pytest

from oracle import attention as A
from oracle import blocks as B
from oracle import paging as P
from tests import pins


def mutant(obj, old, new, **overrides):
    src = textwrap.dedent(inspect.getsource(obj))
    assert old in src, "mutation anchor not found: %r" % old
    ns = dict(inspect.getmodule(obj).__dict__)
    ns.update(overrides)
    exec(compile(src.replace(old, new, 1), "<mutant>", "exec"), ns)
    return ns[obj.__name__]


def fails(check, *args):
    with pytest.raises((AssertionError, IndexError)):
        check(*args)


def test_offset_off_by_one():
    fails(pins.check_translate_enumeration, mutant(P.translate, "offset = t % b", "offset = (t + 1) % b"))


def test_wrong_table_entry():
    fails(pins.check_translate_enumeration,
          mutant(P.translate, "physical = table[logical]", "physical = table[logical - 1]"))


def test_floor_instead_of_ceil():
    bad = mutant(P.blocks_needed, "-(-num_tokens // b)", "num_tokens // b")
    fails(pins.check_address_example, P.translate, bad, P.tail_waste)


def test_waste_sign():
    bad = mutant(P.mean_tail_waste, "tail_waste(t, b)", "(t % b)")
    fails(pins.check_utilization, P.paged_utilization, P.reserved_utilization, bad, P.allocated_slots)


def test_kv_bytes_missing_factor():
    fails(pins.check_kv_bytes, mutant(P.kv_bytes_per_token, "2 * num_layers", "num_layers"))


def test_attention_missing_scale():
    fails(pins.check_bruteforce, mutant(A.attention, "z = scale * (keys @", "z = (keys @"))


def test_attention_values_swapped_for_keys():
    fails(pins.check_bruteforce, mutant(A.attention, "(w @ vals) / w.sum()", "(w @ keys) / w.sum()"))


def test_attention_short_by_one():
    fails(pins.check_bruteforce,
          mutant(A.attention, "length = int(seq_lens[s])", "length = max(1, int(seq_lens[s]) - 1)"))


def test_attention_gather_offset():
    bad_gather = mutant(A.gather_rows, "t % b, :]", "(t + 1) % b, :]")
    fails(pins.check_bruteforce, mutant(A.attention, "group = n_heads", "group = n_heads",
                                        gather_rows=bad_gather))


def test_attention_head_grouping():
    fails(pins.check_gqa_mapping,
          mutant(A.attention, "range(kvh * group, (kvh + 1) * group)", "range(kvh, n_heads, kv_heads)"))


def test_write_swapped_divmod():
    fails(pins.check_write, mutant(A.write_tokens, "blk, off = slot // b, slot % b", "blk, off = slot % b, slot // b"))


def test_copy_direction():
    fails(pins.check_copy, mutant(A.copy_blocks, "k_out[dst] = k_out[src]", "k_out[src] = k_out[dst]"))


def test_bf16_shift():
    fails(pins.check_bf16, mutant(A.to_f64, "<< np.uint32(16)", "<< np.uint32(15)"))


def test_merge_without_rescale():
    fails(pins.check_split_merge, A.attention, A.partition_stats,
          mutant(A.merge_partitions, "c = np.exp(m - big) * np.asarray", "c = np.asarray"))


def test_append_without_copy_on_write():
    fails(pins.check_cow_demo,
          mutant(B.BlockPool, "shared = not full and self.holders_of_tail(tail) > 1", "shared = False"))


def test_copy_on_write_without_the_copy():
    fails(pins.check_cow_demo, mutant(B.BlockPool, "self._duplicate(tail, mine)", "pass"))


def test_tail_fill_off_by_one_block():
    bad = mutant(B.BlockPool, "(len(self.tables[name]) - 1) * self.width",
                 "len(self.tables[name]) * self.width")
    fails(pins.check_pool_vs_contiguous, bad, P.allocated_slots)


def test_release_ignores_sharing():
    bad = mutant(B.BlockPool, "if blk not in still_held:", "if True:")
    fails(pins.check_pool_vs_contiguous, bad, P.allocated_slots)


def test_swap_direction():
    bad = mutant(A.swap_blocks, 'if direction == "out":', 'if direction == "in":')
    with pytest.raises((AssertionError, IndexError, ValueError)):
        pins.check_swap(bad, A.copy_blocks)


def test_prefill_not_causal():
    bad = mutant(A.prefill_attention, "visible = first + i + 1", "visible = length")
    fails(pins.check_prefill, bad, A.attention)


def test_prefill_off_by_one_position():
    bad = mutant(A.prefill_attention, "visible = first + i + 1", "visible = first + i")
    with pytest.raises((AssertionError, IndexError, ValueError)):
        pins.check_prefill(bad, A.attention)


def test_e4m3_ties_away_from_even():
    bad = mutant(A.e4m3_encode, "np.where(lo % 2 == 0, lo, hi)", "hi")
    fails(pins.check_e4m3, bad, A.e4m3_decode)


def test_e4m3_wrong_bias():
    bad = mutant(A.e4m3_decode, "2.0 ** (exp - 7.0)", "2.0 ** (exp - 8.0)")
    fails(pins.check_e4m3, A.e4m3_encode, bad)


def test_fp8_prefill_value_scale_on_keys():
    bad = mutant(A.prefill_attention, "keys = keys * float(k_scale[kvh])",
                 "keys = keys * float(v_scale[kvh])")
    fails(pins.check_fp8_prefill, bad, A.attention, A.dequantize_pool)


def test_fp8_prefill_missing_value_scale():
    bad = mutant(A.prefill_attention, "vals = vals * float(v_scale[kvh])", "vals = vals")
    fails(pins.check_fp8_prefill, bad, A.attention, A.dequantize_pool)
