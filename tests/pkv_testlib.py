"""Shared helpers of the GPU tests: build a workload's state on both sides.

The CUDA side gets its tables from the product block manager (libpkv); the
oracle side gets its own from the oracle model; the two are first checked to
be identical.  Value tensors come from the seeded generators in workloads/.
"""

import numpy as np
import torch

import workloads as W
from oracle import attention as OA
from oracle import cache_ops as OC
from oracle.block_manager import BlockManagerModel

TOL = 2e-3   # max abs error of fp16 output vs the fp64 oracle


class Case:
    """A workload at its decode step, on the GPU and in the oracle."""

    def __init__(self, wl, device="cuda", poison=True, pool_on_host=False):
        import paged_kv_cache_152_gb300 as pkv
        self.wl = wl
        mb = wl.max_blocks_per_seq()
        self.mb = mb
        # product path: the C++ block manager
        alloc = pkv.BlockAllocator(wl.num_blocks, wl.block_size, wl.free_order)
        W.replay(alloc, wl.ops)
        slots, pairs = alloc.append_batch(wl.batch)
        tables, lens = alloc.export(wl.batch, mb)
        self.alloc = alloc
        # oracle path: the model
        model = BlockManagerModel(wl.num_blocks, wl.block_size, wl.free_order)
        W.replay(model, wl.ops)
        exp = [model.append_token(s) for s in wl.batch]
        mt, ml = model.export(wl.batch, mb)
        assert tables.tolist() == mt and lens.tolist() == ml, "block tables differ"
        assert slots.tolist() == [e[0] for e in exp]
        assert len(pairs) == 0 and all(e[1] is None for e in exp)
        self.o_tables = np.array(mt, dtype=np.int64)
        self.o_lens = np.array(ml, dtype=np.int64)
        self.o_slots = np.array([e[0] for e in exp], dtype=np.int64)

        t = W.tensors(wl, device)
        if poison:
            mask = OC.valid_slot_mask(self.o_tables, self.o_lens, wl.num_blocks, wl.block_size)
            bad = torch.from_numpy(~mask).to(device)          # [NB][bs]
            bad = bad[:, None, :, None].expand_as(t["key_cache"])
            t["key_cache"].masked_fill_(bad, float("nan"))
            t["value_cache"].masked_fill_(bad, float("nan"))
        self.t = t
        self.tables = torch.from_numpy(tables).to(device)
        self.lens = torch.from_numpy(lens).to(device)
        self.slots = torch.from_numpy(slots.astype(np.int64)).to(device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.out = torch.full((wl.num_seqs, wl.num_heads, wl.head_dim), float("nan"),
                              dtype=torch.float16, device=device)
        # oracle copies of everything it reads (taken before any GPU write)
        self.o_query = t["query"].cpu().numpy()
        self.o_key = t["key"].cpu().numpy()
        self.o_value = t["value"].cpu().numpy()
        self.o_kc = t["key_cache"].cpu().numpy()
        self.o_vc = t["value_cache"].cpu().numpy()

    # -- product calls ---------------------------------------------------------
    def write_new_tokens(self):
        import paged_kv_cache_152_gb300 as pkv
        pkv.reshape_and_cache(self.t["key"], self.t["value"], self.t["key_cache"], self.t["value_cache"],
                              self.slots, status=self.status)

    def decode(self, num_ctas=0, out=None):
        import paged_kv_cache_152_gb300 as pkv
        out = self.out if out is None else out
        pkv.paged_attention_decode(out, self.t["query"], self.t["key_cache"], self.t["value_cache"],
                                   self.tables, self.lens, self.wl.scale, num_ctas=num_ctas,
                                   status=self.status)
        return out

    # -- oracle ----------------------------------------------------------------
    def oracle_write_new_tokens(self):
        OC.reshape_and_cache(self.o_key, self.o_value, self.o_kc, self.o_vc, self.o_slots)

    def oracle_decode(self, seqs=None):
        return OA.paged_decode_attention(self.o_query, self.o_kc, self.o_vc, self.o_tables, self.o_lens,
                                         self.wl.scale, seqs=seqs)


def bits16(x):
    """fp16 tensor/array -> int16 numpy view, for bit-exact comparisons."""
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x).view(np.int16)


def max_abs_err(gpu_out, ref, seqs=None):
    g = gpu_out.float().cpu().numpy().astype(np.float64)
    rows = range(g.shape[0]) if seqs is None else seqs
    return max(float(np.max(np.abs(g[s] - ref[s]))) for s in rows)
