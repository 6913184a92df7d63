"""Address translation and allocation accounting of a paged KV cache (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

[vLLM-TGI] = "Inside vLLM and TGI: Paging, Versioned Schedulers and
Operations"; [VM-LLM] = "vLLM and PagedAttention: Virtual Memory for LLM
Serving" (transcript); [CB-PA] = "Continuous Batching & PagedAttention: vLLM
Memory Management Architecture".

All arithmetic is exact Python integer arithmetic; ratios are returned as
``fractions.Fraction`` so tests can compare them with the pages' rounded
figures without any floating-point doubt.
"""

from fractions import Fraction


def translate(t, b, table):
    """Map a zero-based logical token position to its physical location.

    [vLLM-TGI] "Block addresses and fragmentation arithmetic": a position t
    in a sequence with block width b lies in logical block t // b at offset
    t % b, and the physical block is the table entry for that logical block.
    [VM-LLM] (paging paragraph) and [CB-PA] "Core PagedAttention Mechanics"
    describe the same mapping.

    The flat "slot" is ``physical * b + offset``: the index of the token's
    row if the pool is viewed as one array of ``num_blocks * b`` rows.  The
    pages have no name for it; it is the quantity the KV write consumes.

    Returns ``(logical_block, offset, physical_block, slot)``.
    """
    if t < 0 or b < 1:
        raise ValueError("position must be >= 0 and block width >= 1")
    logical = t // b
    offset = t % b
    if logical >= len(table):
        raise IndexError("position %d lies beyond the table (%d blocks)" % (t, len(table)))
    physical = table[logical]
    return logical, offset, physical, physical * b + offset


def slot_to_block(slot, b):
    """Invert a flat slot into ``(physical_block, offset)`` (divmod by b)."""
    return slot // b, slot % b


def blocks_needed(num_tokens, b):
    """Blocks a sequence of ``num_tokens`` tokens occupies: ceil(n / b).

    [vLLM-TGI] "Block addresses and fragmentation arithmetic" (a 50-token
    request at b=16 uses four blocks; token 65 needs a fifth) and the
    admission step of "Exact CPU block manager and copy-on-write".
    """
    if num_tokens < 0 or b < 1:
        raise ValueError("num_tokens must be >= 0 and b >= 1")
    return -(-num_tokens // b)


def allocated_slots(lengths, b):
    """Total slots held by live sequences: sum over i of b * ceil(T_i / b).

    [vLLM-TGI] "Block addresses and fragmentation arithmetic".
    """
    return sum(b * blocks_needed(t, b) for t in lengths)


def tail_waste(num_tokens, b):
    """Unused slots in a sequence's last block: (-T) mod b, in [0, b-1].

    [vLLM-TGI] "Block addresses and fragmentation arithmetic".
    """
    return (-num_tokens) % b


def paged_utilization(lengths, b):
    """Aggregate payload utilization sum(T_i) / sum(b * ceil(T_i / b)).

    [vLLM-TGI] "Block addresses and fragmentation arithmetic" asks which of
    three ratios is meant; the aggregate (ratio of sums, equal to the ratio
    of the sample means) is the one its own allocator exercise computes.
    """
    used = sum(lengths)
    return Fraction(used, allocated_slots(lengths, b))


def reserved_utilization(lengths, reserve):
    """Used fraction when every request reserves ``reserve`` slots.

    [vLLM-TGI] "Block addresses and fragmentation arithmetic": the
    max-reservation allocator holds N * T_max slots.
    """
    if any(t > reserve for t in lengths):
        raise ValueError("a length exceeds the reservation")
    return Fraction(sum(lengths), reserve * len(lengths))


def mean_tail_waste(lengths, b):
    """Mean of (-T_i) mod b over the sample, as an exact fraction."""
    return Fraction(sum(tail_waste(t, b) for t in lengths), len(lengths))


def kv_bytes_per_token(num_layers, hidden_size, elem_bytes):
    """Bytes of keys plus values one token holds across all layers.

    [VM-LLM] (sizing paragraph): one OPT-13B token needs about 800 KB of KV
    data in FP16.  Each layer stores one key and one value vector of the
    model's hidden width, so the total is 2 * layers * hidden * bytes.
    """
    return 2 * num_layers * hidden_size * elem_bytes
