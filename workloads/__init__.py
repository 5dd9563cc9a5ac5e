"""Seeded synthetic inputs shaped like the pages' workloads.

This module is shared by the tests, the bench and the oracle-driven checks.  It
holds NONE of the method's arithmetic: no slot numbers, no block-table lookups,
no attention.  It only produces

* the shape parameters of each workload;
* an allocator *trace*: the sequence of block-manager operations (new
  sequence, append n tokens, fork, release) that builds the workload's block
  tables, plus the initial order of the free list;
* seeded random tensors (queries, new keys/values, pool contents).

Whoever replays a trace (the product allocator or the oracle model) computes
the tables itself; ``replay`` below only dispatches operations by name.

Workloads (shapes from the pages' problem statement and the chat example on
the n4n.ai page; seeds are 152 + index):

0 ``tiny``   4 sequences, context 40/17/100/5, 8 heads = 8 KV heads, head_dim
             64, block 16, pool 64 blocks drawn from a seeded permutation.
1 ``7b``     batch 64, 32 heads = 32 KV heads, head_dim 128, block 16, context
             uniform integers in [50, 900], pool 1.25x the blocks needed,
             shuffled free list.
2 ``chat``   batch 128, prompt U{100..2000} + generation U{50..500}; requests
             arrive one per step and allocate their prompt, every active request
             appends one token per step, and 64 transient requests (same length
             laws) arrive at random steps, run U{1..gen} steps and are released,
             so freed blocks are reused mid-run; pool 1.25x the peak need,
             shuffled.
3 ``gqa``    batch 256, 32 query heads, 8 KV heads, head_dim 128, block 32,
             context log-uniform in [256, 4096], pool 1.25x, shuffled.
4 ``prefix`` 128 sequences fork one 500-token prefix (32 blocks of 16, the last
             holding 4 tokens), then append private suffixes U{50..500} one
             token per step in ascending sequence order; the first step makes
             127 copy-on-write copies of the shared tail block.

In every workload the decode step appends one token to each batch sequence:
``context_len`` counts that token, which ``reshape_and_cache`` writes before
attention runs.  A trace therefore appends ``context_len - 1`` tokens.
"""

from dataclasses import dataclass, field
import math

import numpy as np

NAMES = ["tiny", "7b", "chat", "gqa", "prefix"]
BASE_SEED = 152


@dataclass
class Workload:
    name: str
    index: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    free_order: np.ndarray           # initial free list (a permutation of the pool)
    ops: list                        # trace before the decode step
    batch: list                      # decode batch: seq ids, in batch order
    context_lens: list               # context length of each batch seq after the decode append
    scale: float
    seed: int
    marks: dict = field(default_factory=dict)   # name -> op index (phase boundaries)

    @property
    def num_seqs(self):
        return len(self.batch)

    @property
    def group(self):
        return self.num_heads // self.num_kv_heads

    def max_blocks_per_seq(self):
        return -(-max(self.context_lens) // self.block_size)

    def kv_read_bytes(self):
        """K and V bytes one decode step must read (fp16)."""
        return 2 * sum(self.context_lens) * self.num_kv_heads * self.head_dim * 2

    def describe(self):
        return (f"{self.name}: N={self.num_seqs} H={self.num_heads} Hkv={self.num_kv_heads} "
                f"D={self.head_dim} bs={self.block_size} NB={self.num_blocks} "
                f"ctx[min={min(self.context_lens)} mean={np.mean(self.context_lens):.0f} "
                f"max={max(self.context_lens)}]")


def _ceil_div(a, b):
    return -(-int(a) // int(b))


def _simple(name, index, lens, heads, kv_heads, head_dim, block_size, pool=None, base=BASE_SEED):
    """Independent sequences appended one after another, in index order."""
    rng = np.random.default_rng(base + index)
    lens = [int(x) for x in lens]
    if pool is None:
        pool = math.ceil(1.25 * sum(_ceil_div(n, block_size) for n in lens))
    free_order = rng.permutation(pool).astype(np.int32)
    ops = []
    for s, n in enumerate(lens):
        ops.append(("new",))
        if n - 1 > 0:
            ops.append(("append", s, n - 1))
    return Workload(name, index, heads, kv_heads, head_dim, block_size, pool,
                    free_order, ops, list(range(len(lens))), lens,
                    1.0 / math.sqrt(head_dim), base + index)


def tiny(block_size=16, base=BASE_SEED):
    pool = 64 if block_size == 16 else None
    return _simple("tiny", 0, [40, 17, 100, 5], 8, 8, 64, block_size, pool=pool, base=base)


def decode_7b(num_seqs=64, block_size=16, base=BASE_SEED):
    rng = np.random.default_rng(base + 1)
    lens = rng.integers(50, 901, size=max(64, num_seqs))[:num_seqs]
    return _simple("7b", 1, lens, 32, 32, 128, block_size, base=base)


def gqa(num_seqs=256, block_size=32, base=BASE_SEED):
    rng = np.random.default_rng(base + 3)
    u = rng.uniform(math.log(256), math.log(4097), size=256)[:num_seqs]
    lens = np.clip(np.floor(np.exp(u)).astype(np.int64), 256, 4096)
    return _simple("gqa", 3, lens, 32, 8, 128, block_size, base=base)


def chat(num_main=128, num_transient=64, block_size=16, base=BASE_SEED):
    """Arrival-order allocation with interleaved frees (see module docstring).

    Step k: (1) main request k (k < num_main) arrives and appends its prompt;
    transients whose arrival step is k do the same; (2) every request that
    arrived before step k and still has tokens to generate appends one token,
    in sequence-id order; (3) transients that have run their length are
    released.  Main requests stop after gen - 1 generated tokens; the decode
    step appends the last one.
    """
    rng = np.random.default_rng(base + 2)
    prompt = rng.integers(100, 2001, size=128)[:num_main]
    gen = rng.integers(50, 501, size=128)[:num_main]
    t_prompt = rng.integers(100, 2001, size=64)[:num_transient]
    t_gen = rng.integers(50, 501, size=64)[:num_transient]
    t_run = rng.integers(1, t_gen + 1)          # U{1..gen} steps before release
    t_arrive = np.sort(rng.integers(0, 2 * max(num_main, 1), size=64)[:num_transient])

    ops = []
    seq_of_main, seq_of_tr = {}, {}
    todo = {}          # seq -> tokens still to append one per step
    tokens = {}        # seq -> current length (for pool sizing only)
    transient_seqs = set()
    next_seq = 0
    peak_blocks = 0
    k = 0
    while True:
        arrivals = []
        if k < num_main:
            arrivals.append(("main", k))
        for j in np.nonzero(t_arrive == k)[0]:
            arrivals.append(("tr", int(j)))
        old_active = sorted(s for s, left in todo.items() if left > 0)
        for kind, i in arrivals:
            seq = next_seq
            next_seq += 1
            ops.append(("new",))
            n = int(prompt[i] if kind == "main" else t_prompt[i])
            ops.append(("append", seq, n))
            tokens[seq] = n
            if kind == "main":
                seq_of_main[i] = seq
                todo[seq] = int(gen[i]) - 1
            else:
                seq_of_tr[i] = seq
                todo[seq] = int(t_run[i])
                transient_seqs.add(seq)
        for seq in old_active:
            ops.append(("append", seq, 1))
            tokens[seq] += 1
            todo[seq] -= 1
        peak_blocks = max(peak_blocks, sum(_ceil_div(n, block_size) for n in tokens.values()))
        for seq in sorted(transient_seqs):
            if todo[seq] == 0:
                ops.append(("release", seq))
                transient_seqs.discard(seq)
                del todo[seq]
                del tokens[seq]
        k += 1
        arrivals_left = k < num_main or bool(np.any(t_arrive >= k))
        if not arrivals_left and not transient_seqs and all(v == 0 for v in todo.values()):
            break
    batch = [seq_of_main[i] for i in range(num_main)]
    lens = [int(prompt[i] + gen[i]) for i in range(num_main)]
    final_blocks = sum(_ceil_div(n, block_size) for n in lens)
    pool = math.ceil(1.25 * max(peak_blocks, final_blocks))
    free_order = rng.permutation(pool).astype(np.int32)
    return Workload("chat", 2, 32, 32, 128, block_size, pool, free_order, ops,
                    batch, lens, 1.0 / math.sqrt(128), base + 2)


def prefix(num_seqs=128, prefix_len=500, block_size=16, base=BASE_SEED):
    """One prefix forked num_seqs - 1 times, then private suffixes."""
    rng = np.random.default_rng(base + 4)
    suffix = rng.integers(50, 501, size=128)[:num_seqs]
    ops = [("new",), ("append", 0, prefix_len)]
    for _ in range(num_seqs - 1):
        ops.append(("fork", 0))
    marks = {"divergence": len(ops)}
    for k in range(1, int(suffix.max())):
        for s in range(num_seqs):
            if int(suffix[s]) - 1 >= k:
                ops.append(("append", s, 1))
        if k == 1:
            marks["after_divergence"] = len(ops)
    lens = [prefix_len + int(x) for x in suffix]
    shared_full = prefix_len // block_size
    private = sum(_ceil_div(n, block_size) - shared_full for n in lens)
    pool = math.ceil(1.25 * (_ceil_div(prefix_len, block_size) + private))
    free_order = rng.permutation(pool).astype(np.int32)
    return Workload("prefix", 4, 32, 32, 128, block_size, pool, free_order, ops,
                    list(range(num_seqs)), lens, 1.0 / math.sqrt(128),
                    base + 4, marks)


def make(name, **kw):
    """The named workload; keyword arguments go to its generator (sizes,
    block_size, and base: the seed its draws derive from, BASE_SEED unless
    given)."""
    return {"tiny": tiny, "7b": decode_7b, "chat": chat, "gqa": gqa,
            "prefix": prefix}[name](**kw)


def replay(allocator, ops, start=0, stop=None):
    """Apply trace ops[start:stop] to an allocator object.

    The allocator needs new_seq(), append_tokens(seq, n) -> (slots, cows),
    fork(seq) and release(seq).  Returns the list of per-op results.
    """
    results = []
    for op in ops[start:stop]:
        kind = op[0]
        if kind == "new":
            results.append(allocator.new_seq())
        elif kind == "append":
            results.append(allocator.append_tokens(op[1], op[2]))
        elif kind == "fork":
            results.append(allocator.fork(op[1]))
        elif kind == "release":
            results.append(allocator.release(op[1]))
        else:
            raise ValueError(f"unknown op {op!r}")
    return results


# ---------------------------------------------------------------------------
# Seeded tensors.  torch is imported lazily so that the trace helpers above
# stay importable without it.

def _gen(device, seed):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_fp16(shape, seed, device="cpu"):
    """N(0, 1) samples rounded to fp16, from torch's generator on ``device``."""
    import torch
    return torch.randn(tuple(shape), generator=_gen(device, seed), device=device,
                       dtype=torch.float32).to(torch.float16)


def normal_fp16_large(shape, seed, device="cpu", chunk_rows=1024):
    """Like normal_fp16 for pools of several GB: filled row-chunk by row-chunk."""
    import torch
    out = torch.empty(tuple(shape), dtype=torch.float16, device=device)
    g = _gen(device, seed)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        out[r0:r1] = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g,
                                 device=device, dtype=torch.float32).to(torch.float16)
    return out


def tensors(wl, device="cpu", with_pool=True):
    """Seeded value tensors of a workload.

    Returns a dict with query [N][H][D], key/value (the decode step's new
    token) [N][H_kv][D] and, if with_pool, key_cache/value_cache
    [NB][H_kv][bs][D], all fp16 on ``device``.
    """
    n, h, hkv, d = wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim
    base = wl.seed * 1000
    out = {
        "query": normal_fp16((n, h, d), base + 1, device),
        "key": normal_fp16((n, hkv, d), base + 2, device),
        "value": normal_fp16((n, hkv, d), base + 3, device),
    }
    if with_pool:
        shape = (wl.num_blocks, hkv, wl.block_size, d)
        out["key_cache"] = normal_fp16_large(shape, base + 4, device)
        out["value_cache"] = normal_fp16_large(shape, base + 5, device)
    return out
