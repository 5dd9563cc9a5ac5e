"""The oracle's pins catch plausible mistakes (CPU only).

Each mutant below plants one mistake in the oracle -- a dropped term, a wrong
index, a transposed operand, a wrong free-list end, a missed reference count
-- and the oracle's pin tests (test_oracle_attention.py,
test_oracle_block_manager.py, test_oracle_swap.py) are run against it in a
fresh interpreter.  Every mutant must make at least one pin fail; the
unmutated oracle must pass them all.  Mutants live only here and only patch
the oracle modules in the child process.

Run by hand: python tests/test_oracle_mutants.py <mutant>
"""

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIN_FILES = ["tests/test_oracle_attention.py", "tests/test_oracle_block_manager.py", "tests/test_oracle_swap.py"]


# -- attention ---------------------------------------------------------------

def _attention_mutants():
    import numpy as np

    from oracle import attention as A

    def ignore_table(table_row, t, block_size):          # reads logical block t // bs
        return t // block_size, t % block_size

    def offset_plus_one(table_row, t, block_size):
        return int(table_row[t // block_size]), (t + 1) % block_size

    def head(keys, values, q, x):
        w = np.exp(x - x.max())
        return (w @ values) / w.sum()

    def no_scale(q, keys, values, scale):
        q, keys, values = (np.asarray(a, np.float64) for a in (q, keys, values))
        return np.zeros(q.shape[0]) if keys.shape[0] == 0 else head(keys, values, q, keys @ q)

    def negated_scores(q, keys, values, scale):
        q, keys, values = (np.asarray(a, np.float64) for a in (q, keys, values))
        return np.zeros(q.shape[0]) if keys.shape[0] == 0 else head(keys, values, q, -scale * (keys @ q))

    def unnormalised(q, keys, values, scale):
        q, keys, values = (np.asarray(a, np.float64) for a in (q, keys, values))
        if keys.shape[0] == 0:
            return np.zeros(q.shape[0])
        x = scale * (keys @ q)
        return np.exp(x - x.max()) @ values

    gather = A.gather_sequence

    def drop_last_token(cache, table_row, context_len, block_size):
        return gather(cache, table_row, max(0, context_len - 1), block_size)

    def token_major_layout(cache, table_row, context_len, block_size):
        nb, hkv, bs, d = cache.shape                      # reads it as [NB][bs][Hkv][D]
        flat = np.ascontiguousarray(cache).reshape(nb, bs, hkv, d)
        out = np.empty((context_len, hkv, d))
        for t in range(context_len):
            blk, off = A.token_location(table_row, t, block_size)
            out[t] = flat[blk, off].astype(np.float64)
        return out

    def gqa_modulo(query_seq, key_cache, value_cache, table_row, context_len, scale):
        h, hkv = query_seq.shape[0], key_cache.shape[1]
        keys = A.gather_sequence(key_cache, table_row, context_len, key_cache.shape[2])
        values = A.gather_sequence(value_cache, table_row, context_len, key_cache.shape[2])
        out = np.zeros((h, query_seq.shape[1]))
        for i in range(h):
            out[i] = A.attention_one_head(query_seq[i], keys[:, i % hkv], values[:, i % hkv], scale)
        return out

    return {
        "ignore_table": (A, "token_location", ignore_table),
        "offset_plus_one": (A, "token_location", offset_plus_one),
        "no_scale": (A, "attention_one_head", no_scale),
        "negated_scores": (A, "attention_one_head", negated_scores),
        "unnormalised": (A, "attention_one_head", unnormalised),
        "drop_last_token": (A, "gather_sequence", drop_last_token),
        "token_major_layout": (A, "gather_sequence", token_major_layout),
        "gqa_modulo": (A, "paged_decode_attention_one", gqa_modulo),
    }


# -- cache ops ---------------------------------------------------------------

def _cache_op_mutants():
    from oracle import cache_ops as C

    def block_offset_swapped(slot, block_size):
        return slot % block_size, slot // block_size

    def copy_keys_only(key_cache, value_cache, pairs):
        for src, dst in pairs:
            key_cache[int(dst)] = key_cache[int(src)]

    def negative_slots_written(key, value, key_cache, value_cache, slot_mapping):
        bs = key_cache.shape[2]
        for t in range(key.shape[0]):
            blk, off = divmod(int(slot_mapping[t]), bs)   # -1 lands in the last block
            key_cache[blk, :, off, :] = key[t]
            value_cache[blk, :, off, :] = value[t]

    return {
        "block_offset_swapped": (C, "slot_location", block_offset_swapped),
        "copy_keys_only": (C, "copy_blocks", copy_keys_only),
        "negative_slots_written": (C, "reshape_and_cache", negative_slots_written),
    }


# -- memory accounting -----------------------------------------------------------

def _accounting_mutants():
    from oracle import accounting as M

    def blocks_floor(n_tokens, block_size):
        return int(n_tokens) // int(block_size)

    def kv_bytes_keys_only(num_layers, num_kv_heads, head_dim, bytes_per_elem):
        return num_layers * num_kv_heads * head_dim * bytes_per_elem

    def waste_as_use(lengths, block_size):
        return sum(int(n) for n in lengths) / M.paged_slots(lengths, block_size)

    return {
        "blocks_floor": (M, "blocks_for_tokens", blocks_floor),
        "kv_bytes_keys_only": (M, "kv_bytes_per_token", kv_bytes_keys_only),
        "waste_as_use": (M, "paged_waste_fraction", waste_as_use),
    }


# -- block manager -------------------------------------------------------------

def _block_manager_mutants():
    from oracle.block_manager import BlockManagerModel as M

    def lifo_take(self):
        blk = self.free.pop()
        self.refs[blk] = 1
        self.fill[blk] = 0
        return blk

    fork = M.fork

    def fork_without_refs(self, parent):
        child = fork(self, parent)
        for blk in self.tables[child]:
            self.refs[blk] -= 1
        return child

    release = M.release

    def release_to_front(self, seq):
        pool = self.host_free if seq in self.swapped else self.free
        freed = release(self, seq)
        for blk in freed:
            pool.remove(blk)
        pool.extendleft(freed)
        return freed

    append = M.append_token

    def cow_when_full(self, seq):
        table = self.tables.get(seq)
        if table and self.fill[table[-1]] == self.block_size and self.refs[table[-1]] > 1 and self.free:
            old = table[-1]                              # copies a full shared block before moving on
            new = self._take_free_block()
            self.fill[new] = self.fill[old]
            self.refs[old] -= 1
            table[-1] = new
        return append(self, seq)

    def cow_loses_fill(self, seq):
        table = self.tables.get(seq)
        shared = bool(table) and self.fill[table[-1]] < self.block_size and self.refs[table[-1]] > 1
        slot, cow = append(self, seq)
        if shared and cow is not None:                   # the copy starts empty instead of at the fill
            new = cow[1]
            self.fill[new] = 1
            slot = new * self.block_size
        return slot, cow

    move = M._move

    def swap_counts_one(self, seqs, want_swapped, src, dst):
        pairs = move(self, seqs, want_swapped, src, dst)
        for _, new in pairs:
            dst[0][new] = 1
        return pairs

    return {
        "free_list_lifo": (M, "_take_free_block", lifo_take),
        "fork_without_refs": (M, "fork", fork_without_refs),
        "release_to_front": (M, "release", release_to_front),
        "cow_when_full": (M, "append_token", cow_when_full),
        "cow_loses_fill": (M, "append_token", cow_loses_fill),
        "swap_counts_one": (M, "_move", swap_counts_one),
    }


MUTANTS = ["ignore_table", "offset_plus_one", "no_scale", "negated_scores", "unnormalised", "drop_last_token",
           "token_major_layout", "gqa_modulo", "block_offset_swapped", "copy_keys_only", "negative_slots_written",
           "free_list_lifo", "fork_without_refs", "release_to_front", "cow_when_full", "cow_loses_fill",
           "swap_counts_one", "blocks_floor", "kv_bytes_keys_only", "waste_as_use"]


def _install(name):
    table = {**_attention_mutants(), **_cache_op_mutants(), **_accounting_mutants(), **_block_manager_mutants()}
    assert sorted(table) == sorted(MUTANTS)
    owner, attr, fn = table[name]
    setattr(owner, attr, fn)


@pytest.fixture(scope="module")
def pin_runs():
    """Exit code and output of the pin run for every mutant and for none;
    the children run side by side (each is independent)."""
    from concurrent.futures import ThreadPoolExecutor
    env = dict(os.environ, OMP_NUM_THREADS="1", MKL_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1")

    def run(m):
        r = subprocess.run([sys.executable, os.path.abspath(__file__), m], cwd=ROOT, env=env, text=True,
                           stdout=subprocess.PIPE, stderr=subprocess.STDOUT, timeout=600)
        return m, (r.returncode, r.stdout[-3000:])

    with ThreadPoolExecutor(max_workers=max(2, os.cpu_count() or 2)) as pool:
        return dict(pool.map(run, ["none"] + MUTANTS))


def test_unmutated_oracle_passes_its_pins(pin_runs):
    rc, text = pin_runs["none"]
    assert rc == 0, text


@pytest.mark.parametrize("mutant", MUTANTS)
def test_pins_catch_mutant(pin_runs, mutant):
    rc, text = pin_runs[mutant]
    # 1 = some test failed (not a collection, usage or internal error)
    assert rc == 1, f"mutant {mutant} survived the pins (exit {rc})\n" + text


if __name__ == "__main__":
    sys.path.insert(0, ROOT)
    if sys.argv[1] != "none":
        _install(sys.argv[1])
    sys.exit(pytest.main(["-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu", *PIN_FILES]))
