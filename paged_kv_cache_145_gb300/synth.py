"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module holds no step of the method: no address translation, no block
counting, no attention arithmetic.  It only names the workloads and draws
their random parts -- sequence lengths, the order in which physical block
ids are handed out, and N(0, 1) tensors -- from fixed seeds, so that the
CUDA path and the CPU oracle can be fed identical inputs.

Workload shapes follow the pages: OPT-13B (40 heads of 128 = 5120 hidden,
FP16) from the sizing paragraph of "vLLM and PagedAttention: Virtual Memory
for LLM Serving"; lengths uniform over the integers 200..2000 from the
capacity exercise of "Inside vLLM and TGI: Paging, Versioned Schedulers and
Operations" ("Block addresses and fragmentation arithmetic"); 16-token blocks
from both.  The Llama-3-8B-shaped GQA, parallel-sampling and long-context
workloads extend those shapes to grouped heads, forks and long contexts.
"""

import numpy as np
import torch

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
               "e4m3": torch.float8_e4m3fn}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}

# name -> shape of one decode step.  Lengths are cached tokens *before* the
# step; the step writes one token per sequence at position T_i and attends
# over T_i + 1 positions.
CONFIGS = {
    "tiny": dict(
        index=0, heads=4, kv_heads=4, head_dim=64, dtype="f32", block_size=16,
        lengths=[50, 20, 65, 1], pool_blocks=32,
        about="1 layer, 4 heads (MHA), head_dim 64, fp32, block 16, pool of 32 "
              "permuted blocks, 4 sequences of lengths {50, 20, 65, 1}"),
    "opt13b": dict(
        index=1, heads=40, kv_heads=40, head_dim=128, dtype="f16", block_size=16,
        layers=40, batch=64, len_lo=200, len_hi=2000, slack=0.10,
        about="OPT-13B-shaped decode: 40 heads MHA, head_dim 128, fp16, block 16, "
              "batch 64, context lengths U{200..2000}, shuffled pool = need + 10%"),
    "gqa": dict(
        index=2, heads=32, kv_heads=8, head_dim=128, dtype="bf16", block_size=16,
        layers=32, batch=256, len_lo=200, len_hi=2000, slack=0.10,
        about="Llama-3-8B-shaped GQA decode: 32 query / 8 KV heads, head_dim 128, "
              "bf16, block 16, batch 256, context lengths U{200..2000}"),
    "fork": dict(
        index=3, heads=32, kv_heads=8, head_dim=128, dtype="bf16", block_size=16,
        layers=32, groups=16, forks=8, prompt=1031, slack=0.10,
        about="parallel sampling: 16 groups x 8 forks sharing a 1031-token prompt "
              "(last block partial), GQA 32/8, head_dim 128, bf16, block 16"),
    "prefill": dict(
        index=5, heads=32, kv_heads=8, head_dim=128, dtype="bf16", block_size=16,
        batch=8, prefix=0, chunk=2048, slack=0.10,
        about="paged prefill: 8 prompts of 2048 tokens (no cached prefix), GQA 32/8, "
              "head_dim 128, bf16, block 16, causal"),
    "chunked": dict(
        index=6, heads=32, kv_heads=8, head_dim=128, dtype="bf16", block_size=16,
        batch=8, prefix=4096, chunk=512, slack=0.10,
        about="chunked prefill: 8 sequences with 4096 cached positions and a 512-token "
              "chunk, GQA 32/8, head_dim 128, bf16, block 16, causal"),
    "long": dict(
        index=4, heads=32, kv_heads=8, head_dim=128, dtype="bf16", block_size=16,
        layers=32, batch=8, len_lo=16384, len_hi=32768, slack=0.10, partition_size=512,
        about="long-context split-K: GQA 32/8, head_dim 128, bf16, batch 8, "
              "context lengths U{16384..32768}, 512-token partitions"),
}


def seed_of(name, stream=0):
    """Seed of one random stream of a workload (config index * 1000 + 17)."""
    return CONFIGS[name]["index"] * 1000 + 17 + 101 * stream


def lengths(name, batch=None):
    """Cached lengths before the step, as int64 (seeded, uniform integers)."""
    cfg = CONFIGS[name]
    if "lengths" in cfg:
        return np.asarray(cfg["lengths"], dtype=np.int64)
    n = cfg["batch"] if batch is None else batch
    rng = np.random.default_rng(seed_of(name, 1))
    return rng.integers(cfg["len_lo"], cfg["len_hi"] + 1, size=n).astype(np.int64)


def free_order(seed, num_blocks):
    """A seeded permutation of the physical block ids 0..num_blocks-1."""
    return np.random.default_rng(seed).permutation(num_blocks).astype(np.int64)


def pool_with_slack(blocks_in_use, slack):
    """Pool size: the blocks in use plus a fractional reserve, rounded up."""
    return int(np.ceil(blocks_in_use * (1.0 + slack)))


def normal(seed, shape, dtype, device="cpu"):
    """N(0, 1) values drawn in float32 from a seeded generator, then cast.

    ``device="cpu"`` draws on the host; ``"cuda"`` draws with the device's
    generator (fast for multi-GB pools; values differ from the host's).
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    x = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    return x.to(TORCH_DTYPE[dtype])


def random_codes(seed, shape, device="cpu"):
    """Seeded random bytes for an 8-bit E4M3 pool, avoiding the two bytes
    that encode NaN (0x7F, 0xFF)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    mag = torch.randint(0, 0x7F, shape, generator=gen, device=device, dtype=torch.int32)
    sign = torch.randint(0, 2, shape, generator=gen, device=device, dtype=torch.int32) * 0x80
    return (mag | sign).to(torch.uint8).view(torch.float8_e4m3fn)


def storage_numpy(t, dtype):
    """Host NumPy copy of a tensor in its stored form (bf16 as uint16 bits,
    E4M3 as uint8 codes)."""
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    if dtype == "e4m3":
        return t.view(torch.uint8).numpy()
    return t.numpy()
