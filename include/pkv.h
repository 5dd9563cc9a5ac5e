/*
 * pkv.h -- C ABI of the paged KV cache library (libpkv.so).
 *
 * The library implements the data-parallel hot path of PagedAttention for one
 * GPU (sm_103a):
 *
 *   pkv_paged_attention_decode  single-query decode attention that reads the
 *                               KV cache through per-sequence block tables;
 *   pkv_paged_attention_decode_append
 *                               the same, writing each sequence's new token
 *                               in the same launch;
 *   pkv_decode_plan_*           a decode call validated once and launched (or
 *                               run as a whole serving step) many times;
 *   pkv_reshape_and_cache       the slot-mapped write of new tokens' K/V;
 *   pkv_copy_blocks             the whole-block copy behind copy-on-write;
 *   pkv_swap_blocks             block copies between device and page-locked
 *                               host pools (swap out / in);
 *   *_layers                    the cache ops over every layer's pool in one
 *                               launch;
 *   pkv_alloc_* / pkv_seq_* ... the host block manager that hands out blocks,
 *                               counts references, forks and copies on write,
 *                               swaps sequences out and in, exports the block
 *                               tables, and checkpoints its state.
 *
 * Sources (cited by page title and section):
 *   [P1] "Paged Attention: OS-Inspired Memory Management for KV Caches",
 *        modernaiengineering.com, lesson 13.6;
 *   [P2] "What is PagedAttention and how does it manage KV cache?", n4n.ai;
 *   [P3] worksonmygpu.com, deep-dive post "PagedAttention (vLLM)".
 *
 * Conventions for every call:
 *   - Every entry point returns an int status (pkv_status below).  A call that
 *     fails leaves every host-side object exactly as it was.
 *   - Device pointers are BORROWED: the caller owns and allocates all device
 *     memory (KV pools, tables, outputs, workspace).  The library never
 *     allocates device memory itself.
 *   - Kernels are launched asynchronously on the caller's stream (NULL = the
 *     legacy default stream).  Argument errors are detected on the host before
 *     any launch.  Errors that depend on device data (a slot or table entry
 *     outside the pool, a device wait that gave up) are written to the
 *     caller's int32 device status word: the first error wins (0 -> code), the
 *     word is never cleared by the library, and a NULL status pointer means
 *     "do not report".  Kernels never trap: after a device error the affected
 *     outputs are unspecified but the CUDA context stays usable.
 *   - Cache layout (chosen here; [P2] "How PagedAttention works" only fixes
 *     that tokens are contiguous inside a block): key_cache and value_cache
 *     are separate fp16 tensors [num_blocks][num_kv_heads][block_size][head_dim],
 *     row-major.  Token `off` of physical block `b`, KV head `h`, element `i`
 *     sits at element ((b*num_kv_heads + h)*block_size + off)*head_dim + i.
 *   - A slot names one token position of the pool: slot = b*block_size + off
 *     ([P1] paged_vs_contiguous.py example: token 37 -> logical block 2,
 *     offset 5).
 *   - Base pointers of the caches, query, key, value and out must be 16-byte
 *     aligned (torch allocations are 256-byte aligned).
 *   - Calls launch on the calling thread's current CUDA device, which must be
 *     the one that holds their device pointers.  Several devices in one process
 *     are fine (each decode kernel's dynamic shared-memory limit is raised per
 *     device); a plan, like any call, runs on the device it was created on.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; declared here so that this header
 * needs no CUDA header. */
typedef struct CUstream_st *pkv_stream_t;

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,     /* bad pointer, size, shape or id (host check) */
    PKV_ERR_OUT_OF_BLOCKS = 2,   /* block manager: free list cannot satisfy the call */
    PKV_ERR_CUDA = 3,            /* a CUDA runtime call failed (launch, attribute) */
    PKV_ERR_DEVICE_TIMEOUT = 4,  /* device: a bounded wait gave up (status word only) */
    PKV_ERR_OUT_OF_RANGE = 5,    /* device: slot / table entry / context outside the pool or table */
    PKV_ERR_NOT_FOUND = 6,       /* block manager: unknown or released sequence id */
    PKV_ERR_UNSUPPORTED = 7,     /* shape not compiled into this build (head_dim, block_size, group) */
    PKV_ERR_SWAPPED = 8          /* block manager: the sequence is swapped out (or, for a swap in, resident) */
} pkv_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *pkv_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int pkv_version(void);

/* ------------------------------------------------------------------------ */
/* Decode attention                                                          */
/* ------------------------------------------------------------------------ */

/*
 * pkv_paged_attention_decode
 *
 * [P1] "How PagedAttention works", step 4: each decode step walks the block
 * table, loads each block's keys and values and computes attention exactly as
 * if they were contiguous.  For every sequence s and query head h, with
 * L = context_lens[s], kvh = h / (num_heads / num_kv_heads) (consecutive
 * query-head groups share a KV head), and token t stored in physical block
 * block_tables[s][t / block_size] at offset t % block_size:
 *
 *     out[s][h] = sum_t softmax_t(scale * q[s][h] . K[t][kvh]) * V[t][kvh]
 *
 * computed in fp32 (online softmax, fp32 accumulation) and rounded to fp16 to
 * nearest even.  L == 0 gives an all-zero row.  Entries of a table row past
 * ceil(L / block_size) are never read (they may hold -1).
 *
 * Arguments (all device pointers unless noted):
 *   out          fp16 [num_seqs][num_heads][head_dim]           (written)
 *   query        fp16 [num_seqs][num_heads][head_dim]
 *   key_cache    fp16 [num_blocks][num_kv_heads][block_size][head_dim]
 *   value_cache  same shape as key_cache
 *   block_tables int32 [num_seqs][max_blocks_per_seq], row-major
 *   context_lens int32 [num_seqs]
 *   scale        softmax scale (host value), usually 1/sqrt(head_dim)
 *   num_ctas     persistent grid size; 0 = one full wave (SM count x CTAs
 *                per SM).  A small batch leaves some of them idle (every
 *                worker warp gets at least 4 chunks of 16 rows; while the
 *                (sequence, KV head) segments are short, no more CTAs work
 *                than there are segments).  Any value >= 1 gives the same
 *                result within rounding; 1 makes every sequence a single
 *                pass.
 *   workspace    device scratch of at least pkv_decode_workspace_size(...)
 *                bytes for the same (num_seqs, num_heads, num_kv_heads,
 *                head_dim, block_size, num_ctas); 256-byte aligned.  It
 *                carries state from call to call (an epoch word that every
 *                call advances, and completion counters that each call
 *                prepares for the next), so keep one workspace per stream of
 *                calls; what it holds on first use does not matter (zeroed
 *                or not), nor does a call that gave up, and a launch recorded
 *                once and replayed (a CUDA graph) works.  It must not be used
 *                by another call that runs at the same time.
 *   dev_status   int32 device status word (nullable), see conventions.
 *   stream       CUDA stream.
 *
 * Supported: head_dim in {64, 128}; block_size in {8, 16, 32, 64, 128};
 * num_heads / num_kv_heads in {1, 2, 4, 8}; 1 <= num_seqs <= 4096;
 * num_blocks * num_kv_heads * block_size < 2^31 (the cache rows the tensor
 * copies address: up to 512 GB per cache at head_dim 128, 256 GB at 64) and
 * max_blocks_per_seq * block_size <= 2^30, else PKV_ERR_INVALID_ARG.
 * A context longer than max_blocks_per_seq*block_size, or a table entry
 * outside [0, num_blocks), sets PKV_ERR_OUT_OF_RANGE in dev_status; such a
 * context is clamped to its table and such an entry reads block 0.
 * Launches one kernel on `stream`, with programmatic dependent launch: it may
 * start while the preceding kernel in the stream finishes, and reads
 * context_lens and block_tables before it waits for that kernel (everything
 * else — the caches, query, workspace, out — only after).  So context_lens
 * and block_tables must not be written by a kernel that signals its
 * dependents early (griddepcontrol.launch_dependents /
 * cudaTriggerProgrammaticLaunchCompletion) before it writes them; memory
 * copies, ordinary kernels and this library's kernels never do.
 */
int pkv_paged_attention_decode(void *out, const void *query,
                               const void *key_cache, const void *value_cache,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens,
                               int num_seqs, int num_heads, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks,
                               float scale, int num_ctas,
                               void *workspace, size_t workspace_bytes,
                               int32_t *dev_status, pkv_stream_t stream);

/*
 * pkv_paged_attention_decode_append
 *
 * One decode step in one launch: what pkv_reshape_and_cache of each
 * sequence's new token followed by pkv_paged_attention_decode computes ([P1]
 * "How PagedAttention works", steps 2-4: write the token into the next slot
 * of the last block, then attend over the whole table).  For every sequence s
 * with L = context_lens[s] > 0, the new token is position L-1: key[s] and
 * value[s] ([num_kv_heads][head_dim] each) are written to that position's
 * slot (block block_tables[s][(L-1)/block_size], offset (L-1)%block_size) of
 * key_cache / value_cache, and attention covers positions 0..L-1 with them.
 * No slot mapping is needed: the slot follows from the table.  Outputs and
 * cache contents are identical to the two-call sequence.  Copy-on-write
 * copies (pkv_copy_blocks) must still run before it.
 *
 *   key, value   fp16 [num_seqs][num_kv_heads][head_dim] (device)
 *   key_cache, value_cache  written at the new tokens' slots (device)
 * Other arguments, workspace, errors and launch ordering (which inputs are
 * read before the wait for the preceding kernel) as pkv_paged_attention_decode.
 */
int pkv_paged_attention_decode_append(void *out, const void *query,
                                      const void *key, const void *value,
                                      void *key_cache, void *value_cache,
                                      const int32_t *block_tables, int max_blocks_per_seq,
                                      const int32_t *context_lens,
                                      int num_seqs, int num_heads, int num_kv_heads,
                                      int head_dim, int block_size, int num_blocks,
                                      float scale, int num_ctas,
                                      void *workspace, size_t workspace_bytes,
                                      int32_t *dev_status, pkv_stream_t stream);

/*
 * Decode plans: validate once, launch many times.
 *
 * A serving loop calls the decode with the same buffers every step; only
 * their contents (queries, new tokens, tables, lengths) change.
 * pkv_decode_plan_create checks the arguments, picks the kernel and grid and
 * encodes the caches' TMA descriptors once; pkv_decode_plan_launch then
 * launches exactly what pkv_paged_attention_decode_append (key/value
 * non-NULL) or pkv_paged_attention_decode (both NULL) would, with no host
 * work but the launch.  Same results, errors and device status as those
 * calls.  The plan borrows every pointer: the buffers must outlive it, and
 * must not be moved or freed while it is in use.  A plan is read-only after
 * creation (launches from several host threads are fine; on one workspace
 * they must be stream-ordered, as for the direct calls).
 *
 * A plan's out may also be page-locked host memory mapped into the device's
 * address space (cudaHostAlloc / cudaMallocHost memory on a system with
 * unified addressing, or memory registered with cudaHostRegisterMapped).
 * The kernel then writes each output row over the CPU-GPU link as soon as it
 * is final, so a serving step needs no copy of the output back
 * (pkv_decode_plan_step with host_out == NULL); the host reads out once the
 * stream has passed the launch.  pkv_decode_plan_create checks where out
 * lives (cudaPointerGetAttributes): device memory of the current device,
 * managed memory or mapped host memory; anything else (pageable host memory,
 * another device's memory) is PKV_ERR_INVALID_ARG, a failed query
 * PKV_ERR_CUDA.  The direct calls take device or managed memory only.
 */
typedef struct pkv_decode_plan pkv_decode_plan_t;
int pkv_decode_plan_create(void *out, const void *query, const void *key, const void *value,
                           void *key_cache, void *value_cache,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *context_lens,
                           int num_seqs, int num_heads, int num_kv_heads,
                           int head_dim, int block_size, int num_blocks,
                           float scale, int num_ctas,
                           void *workspace, size_t workspace_bytes,
                           int32_t *dev_status, pkv_decode_plan_t **plan);
int pkv_decode_plan_launch(const pkv_decode_plan_t *plan, pkv_stream_t stream);

/*
 * pkv_decode_plan_step: one serving step in one call, all on `stream`:
 * in_bytes from host_in to dev_in (the step's inputs -- queries, new K/V,
 * tables, lengths -- staged in one region that the plan's device pointers
 * lie in), then the plan's launch, then the plan's output (fp16
 * [num_seqs][num_heads][head_dim]) to host_out.  in_bytes == 0 skips the
 * first copy and host_out == NULL the last.  host_in / host_out should be
 * page-locked for the copies to be asynchronous.  The caller synchronises the
 * stream before reading host_out or reusing host_in.  PKV_ERR_INVALID_ARG for
 * a NULL plan or a missing pointer; PKV_ERR_CUDA when a copy or the launch
 * fails to enqueue (nothing after it is enqueued).
 */
int pkv_decode_plan_step(const pkv_decode_plan_t *plan, void *dev_in, const void *host_in, size_t in_bytes,
                         void *host_out, pkv_stream_t stream);

/*
 * pkv_decode_plan_step_mapped: one serving step whose inputs the kernel reads
 * straight from page-locked host memory, with no copy in: every input pointer
 * of the plan (query, key, value, block_tables, context_lens, shared_blocks)
 * that lies in [dev_base, dev_base + in_bytes) is read at the same offset of
 * host_in, over the CPU-GPU link; the others as created.  dev_base is only an
 * address here (the region the plan was created on): it is neither read nor
 * written.  The queries and new K/V rows are copied by the kernel's lanes 16
 * bytes at a time, a few chunks ahead of their use, and the lengths and
 * tables are read in its prologue.  Then the output goes to host_out as in
 * pkv_decode_plan_step (NULL: none; a plan whose out is mapped host memory
 * needs none).  Same results, bit for bit, as staging host_in into dev_base
 * and launching.
 *
 *   host_in  page-locked host memory mapped for the current device
 *            (cudaHostAlloc / cudaMallocHost with unified addressing, or
 *            cudaHostRegisterMapped), in_bytes long, holding the inputs at
 *            their offsets in the plan's region; query, key and value
 *            16-byte aligned.  The caller must not write it until the
 *            stream has passed the launch.
 * PKV_ERR_INVALID_ARG for a NULL plan, in_bytes == 0, host_in that is not
 * such memory (cudaPointerGetAttributes), a misaligned input, or an input
 * that starts inside the region but runs past its end (nothing is
 * enqueued); PKV_ERR_UNSUPPORTED if the library was built without the
 * kernels that read host inputs; PKV_ERR_CUDA when the launch or the copy
 * out fails to enqueue.
 */
int pkv_decode_plan_step_mapped(const pkv_decode_plan_t *plan, const void *dev_base, const void *host_in,
                                size_t in_bytes, void *host_out, pkv_stream_t stream);
void pkv_decode_plan_destroy(pkv_decode_plan_t *plan);

/*
 * Decode attention with prefix sharing.
 *
 * [P1] "Memory sharing across requests" and [P2] "How PagedAttention works"
 * (prefix sharing): sequences forked from one prompt read the same physical
 * blocks for it.  These calls compute exactly what
 * pkv_paged_attention_decode_append (key/value non-NULL) or
 * pkv_paged_attention_decode (both NULL) compute, and take one more input:
 *
 *   shared_blocks  int32 [num_seqs] (device): for s >= 1, how many leading
 *                  logical blocks sequence s has in common with sequence
 *                  s - 1 (same physical block at the same logical index);
 *                  entry 0 is ignored.  pkv_export_shared_prefix computes it.
 *                  It must not claim more than the tables hold in common
 *                  (the shared blocks are read through the first sequence's
 *                  table); smaller values are always correct, and all zeros
 *                  is the plain decode.
 *
 * Up to 8 consecutive sequences that share blocks form a group; the group's
 * shared full blocks (never the block of a member's last token) are read
 * once for all of them, with the members' queries as the rows of one
 * tensor-core tile, then each member's own blocks with only its row live.
 * Results are run-to-run deterministic for a fixed grid and agree with the
 * plain decode within rounding (not bit for bit).  On a batch without
 * sharing the plain calls are faster (the grouped kernel keeps 8 rows per
 * segment): pass the hints where forks share blocks.  The grouped kernel serves group 1
 * (num_heads == num_kv_heads), block sizes 16 to 128 and up to 1024
 * sequences; other calls run the plain kernel (shared_blocks is then not
 * read).  The workspace is pkv_decode_workspace_size_shared(...) bytes, and
 * otherwise follows the rules of pkv_paged_attention_decode.  A NULL
 * shared_blocks with num_seqs > 0 is PKV_ERR_INVALID_ARG.
 */
int pkv_paged_attention_decode_shared(void *out, const void *query, const void *key,
                                      const void *value, void *key_cache, void *value_cache,
                                      const int32_t *block_tables, int max_blocks_per_seq,
                                      const int32_t *context_lens, const int32_t *shared_blocks,
                                      int num_seqs, int num_heads, int num_kv_heads,
                                      int head_dim, int block_size, int num_blocks,
                                      float scale, int num_ctas,
                                      void *workspace, size_t workspace_bytes,
                                      int32_t *dev_status, pkv_stream_t stream);
int pkv_decode_plan_create_shared(void *out, const void *query, const void *key, const void *value,
                                  void *key_cache, void *value_cache,
                                  const int32_t *block_tables, int max_blocks_per_seq,
                                  const int32_t *context_lens, const int32_t *shared_blocks,
                                  int num_seqs, int num_heads, int num_kv_heads,
                                  int head_dim, int block_size, int num_blocks,
                                  float scale, int num_ctas,
                                  void *workspace, size_t workspace_bytes,
                                  int32_t *dev_status, pkv_decode_plan_t **plan);
size_t pkv_decode_workspace_size_shared(int num_seqs, int num_heads, int num_kv_heads,
                                        int head_dim, int block_size, int num_ctas);

/* Bytes of workspace pkv_paged_attention_decode needs (host call; queries the
 * current device's SM count when num_ctas == 0).  Returns 0 for unsupported
 * shapes. */
size_t pkv_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                 int head_dim, int block_size, int num_ctas);

/* The grid size num_ctas == 0 resolves to on the current device for this
 * shape (host call), or 0 for unsupported shapes. */
int pkv_decode_default_ctas(int num_heads, int num_kv_heads, int head_dim,
                            int block_size);

/*
 * pkv_paged_attention_decode_noalloc
 *
 * The pages have no counterpart to this entry point: it exists for callers
 * that cannot allocate device memory themselves.  Typical ones are a serving
 * engine or framework that has already handed nearly all of the GPU's memory
 * to its own KV pool and caching allocator (a separate cudaMalloc would fail,
 * or fragment memory the engine budgets to the byte), a plug-in that the host
 * application gives no allocation rights, and hot loops that cannot afford
 * cudaMalloc/cudaFree, which may synchronise the whole device.
 *
 * It computes exactly what pkv_paged_attention_decode computes, with the same
 * arguments minus workspace / workspace_bytes.  Its scratch is a fixed array
 * of PKV_DECODE_NOALLOC_SCRATCH_BYTES (16 MiB) that lives inside the library
 * as a static device variable: every GPU that loads the library holds those
 * 16 MiB until the process exits.  The call itself allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Limit: the scratch a call needs is pkv_decode_workspace_size(num_seqs,
 * num_heads, num_kv_heads, head_dim, block_size, num_ctas); a call that needs
 * more than PKV_DECODE_NOALLOC_SCRATCH_BYTES returns PKV_ERR_INVALID_ARG and
 * launches nothing.  The need grows with num_seqs * num_kv_heads (16 bytes
 * each) and with the grid.  At the default grid of one CTA per SM on a
 * 152-SM GB300 the call fits while num_seqs * num_kv_heads is at most:
 *
 *                 group 1    group 2    group 4    group 8
 *   head_dim 64   1,003,408    958,272    867,984    687,408
 *   head_dim 128    959,632    870,720    692,880    337,200
 *
 * (so at num_seqs = 4096, group 8, head_dim 128, num_kv_heads may be at most
 * 82).  A larger num_ctas leaves less room.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and keeps it; make that
 * first call before any stream capture.  A failed look-up returns
 * PKV_ERR_CUDA.  Devices with ordinals 0 to 63 are served; a call with a
 * higher ordinal current returns PKV_ERR_UNSUPPORTED.
 *
 * Sharing: all calls in the process share the one array, and it keeps what
 * the last call left in it.  Nothing needs clearing between calls: partial
 * results are rewritten before they are read, and the completion counters
 * are tagged with an epoch that every call advances, so leftovers of an
 * earlier call (even one that failed) are never taken for the current one.
 * Two calls whose kernels
 * overlap on the GPU (different streams, or different host threads) race on
 * the array and give wrong results: serialise them, for example on one
 * stream.  Other errors and the device status word behave as for
 * pkv_paged_attention_decode.
 */
#define PKV_DECODE_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int pkv_paged_attention_decode_noalloc(void *out, const void *query,
                                       const void *key_cache, const void *value_cache,
                                       const int32_t *block_tables, int max_blocks_per_seq,
                                       const int32_t *context_lens,
                                       int num_seqs, int num_heads, int num_kv_heads,
                                       int head_dim, int block_size, int num_blocks,
                                       float scale, int num_ctas,
                                       int32_t *dev_status, pkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Cache writes                                                              */
/* ------------------------------------------------------------------------ */

/*
 * pkv_reshape_and_cache
 *
 * [P1] "How PagedAttention works", steps 2-3: a new token goes into the next
 * slot of its sequence's last block.  For t in [0, num_tokens): if
 * slot_mapping[t] >= 0, copy key[t][h][:] and value[t][h][:] (every KV head h)
 * to slot slot_mapping[t] of key_cache / value_cache.  A negative slot is
 * skipped.  Bit-exact copies.
 *
 *   key, value    fp16 [num_tokens][num_kv_heads][head_dim] (device)
 *   key_cache, value_cache   pool, layout above (device, written)
 *   slot_mapping  int64 [num_tokens] (device)
 *   dev_status    a slot >= num_blocks*block_size sets PKV_ERR_OUT_OF_RANGE
 *                 and that token is not written.
 * head_dim must be a multiple of 8.  num_tokens == 0 launches nothing.
 * Two tokens with the same slot race (the caller's block manager never
 * produces that).
 */
int pkv_reshape_and_cache(const void *key, const void *value,
                          void *key_cache, void *value_cache,
                          const int64_t *slot_mapping, int num_tokens,
                          int num_kv_heads, int head_dim, int block_size,
                          int num_blocks, int32_t *dev_status,
                          pkv_stream_t stream);

/*
 * pkv_copy_blocks
 *
 * [P1] "Memory sharing across requests": copy-on-write copies a shared block
 * to a fresh block before the writer's token goes in.  For each pair
 * (src, dst) = block_pairs[2*i], block_pairs[2*i+1], copy the block_bytes
 * bytes of physical block src over block dst, in key_cache and in
 * value_cache.  Bit-exact.  Must run before the pkv_reshape_and_cache that
 * writes the copying sequence's token.
 *
 *   block_pairs  int64 [num_pairs][2] (device)
 *   block_bytes  bytes of one physical block in one cache
 *                (num_kv_heads*block_size*head_dim*2 for fp16); multiple of 16
 *   dev_status   a pair outside [0, num_blocks) sets PKV_ERR_OUT_OF_RANGE and
 *                is skipped.
 * The destinations must be pairwise distinct and no destination may also be
 * a source in the same call (pkv_validate_block_pairs checks this on a host
 * copy).  num_pairs == 0 launches nothing.
 */
int pkv_copy_blocks(void *key_cache, void *value_cache,
                    const int64_t *block_pairs, int num_pairs,
                    size_t block_bytes, int num_blocks,
                    int32_t *dev_status, pkv_stream_t stream);

/*
 * Multi-layer cache ops.  [P2] "How PagedAttention works": a block holds its
 * tokens for all layers and heads, so one slot mapping (and one list of
 * copy-on-write pairs) serves every layer.  These do, in ONE launch, what
 * num_layers calls of pkv_reshape_and_cache / pkv_copy_blocks would do, one
 * per layer, with every layer's pool shaped alike.
 *
 *   keys, values            HOST arrays [num_layers] of device pointers, each
 *                           fp16 [num_tokens][num_kv_heads][head_dim]
 *   key_caches, value_caches HOST arrays [num_layers] of device pointers to
 *                           each layer's pool (layout above)
 *   slot_mapping, block_pairs, dev_status: device, as for the one-layer calls
 * 1 <= num_layers <= PKV_MAX_LAYERS.  The pointer arrays are copied into the
 * kernel's parameters; nothing is allocated.  Same errors as the one-layer
 * calls; a NULL or misaligned pointer in an array is PKV_ERR_INVALID_ARG.
 */
#define PKV_MAX_LAYERS 128
int pkv_reshape_and_cache_layers(const void *const *keys, const void *const *values,
                                 void *const *key_caches, void *const *value_caches,
                                 int num_layers, const int64_t *slot_mapping,
                                 int num_tokens, int num_kv_heads, int head_dim,
                                 int block_size, int num_blocks, int32_t *dev_status,
                                 pkv_stream_t stream);
int pkv_copy_blocks_layers(void *const *key_caches, void *const *value_caches,
                           int num_layers, const int64_t *block_pairs, int num_pairs,
                           size_t block_bytes, int num_blocks, int32_t *dev_status,
                           pkv_stream_t stream);

/*
 * pkv_swap_blocks
 *
 * [P2] "Why it matters for KV cache", "Swapping and preemption": blocks are
 * evicted to CPU memory when GPU memory runs short and fetched back when the
 * request resumes ([P1] "Common misconceptions": a technique separate from
 * paging itself).  For each pair (src, dst) = block_pairs[2*i],
 * block_pairs[2*i+1], copy the block_bytes bytes of block src of the SOURCE
 * pool over block dst of the DESTINATION pool, in the key and the value
 * pools.  Bit-exact.  Both pools have the cache layout above (block-major,
 * block_bytes per block); one of them is normally page-locked host memory,
 * which the kernel reads or writes directly over the CPU-GPU link (no copy
 * engine, one launch for any number of scattered blocks).
 *
 *   src_key, src_value    source pools: device memory of the current device
 *                         or page-locked host memory (cudaHostAlloc,
 *                         cudaHostRegister); src_num_blocks blocks each
 *   dst_key, dst_value    destination pools, same rules; dst_num_blocks
 *   block_pairs           int64 [num_pairs][2] (device-accessible): (source
 *                         block, destination block), e.g. the pairs of
 *                         pkv_swap_out (device -> host) or pkv_swap_in
 *                         (host -> device)
 *   block_bytes           bytes of one block in one cache; multiple of 16
 *   dev_status            a pair outside either pool sets
 *                         PKV_ERR_OUT_OF_RANGE and is skipped
 * Pageable (unregistered) host memory, or another device's memory, is
 * PKV_ERR_INVALID_ARG before anything is launched (the pointer attributes are
 * queried on the host; on a machine without a GPU that query fails with
 * PKV_ERR_CUDA).  Destination blocks must be pairwise distinct and must not
 * overlap the source blocks of the same call.  num_pairs == 0 launches
 * nothing.
 */
int pkv_swap_blocks(const void *src_key, const void *src_value,
                    void *dst_key, void *dst_value,
                    const int64_t *block_pairs, int num_pairs, size_t block_bytes,
                    int src_num_blocks, int dst_num_blocks,
                    int32_t *dev_status, pkv_stream_t stream);

/* pkv_swap_blocks for every layer in one launch: HOST arrays [num_layers] of
 * pool pointers (each under the rules above), one pair list for all layers
 * (a block id spans all layers).  1 <= num_layers <= PKV_MAX_LAYERS. */
int pkv_swap_blocks_layers(const void *const *src_keys, const void *const *src_values,
                           void *const *dst_keys, void *const *dst_values, int num_layers,
                           const int64_t *block_pairs, int num_pairs, size_t block_bytes,
                           int src_num_blocks, int dst_num_blocks,
                           int32_t *dev_status, pkv_stream_t stream);

/* Host check of a pair list for pkv_copy_blocks: ids in range, destinations
 * distinct, no destination also a source.  PKV_OK or PKV_ERR_INVALID_ARG. */
int pkv_validate_block_pairs(const int64_t *host_pairs, int num_pairs,
                             int num_blocks);

/* ------------------------------------------------------------------------ */
/* Block manager (host)                                                      */
/* ------------------------------------------------------------------------ */

/*
 * A pool of num_blocks physical blocks of block_size token slots each
 * ([P1] "What PagedAttention is"; [P2] "How PagedAttention works": a global
 * pool handed out block by block).
 *
 * Rules ([P1] "How PagedAttention works", "Memory sharing across requests",
 * practice block manager and its exercises):
 *   - The free list is FIFO: blocks are taken from the front and released
 *     blocks are put at the back, in table order.  initial_free_order (host,
 *     nullable) gives the starting order (a permutation of 0..num_blocks-1);
 *     NULL means 0, 1, 2, ...
 *   - Every block has a reference count (sequences using it) and a fill
 *     (token slots written).
 *   - Appending a token: if the sequence has no block or its last block is
 *     full, a fresh block is taken; else if the last block is shared
 *     (count > 1) it is copied on write: a fresh block takes the old block's
 *     fill, the table points at it, the old block's count drops by one, and
 *     the pair (old, new) is returned for pkv_copy_blocks.  Then the token
 *     takes the next slot of the last block.
 *   - Fork: the child's table is a copy of the parent's (partial last block
 *     included); every block's count rises by one.  No device work.
 *   - Release: every block's count drops by one; blocks reaching zero go back
 *     to the free list.  No device work.
 *   - Sequence ids are handed out 0, 1, 2, ... and never reused.
 * An operation that needs more free blocks than there are returns
 * PKV_ERR_OUT_OF_BLOCKS and changes nothing.  The object is not thread-safe.
 *
 * Swapping ([P2] "Why it matters for KV cache", "Swapping and preemption";
 * [P1] "Common misconceptions").  An optional second pool of host blocks
 * (pkv_alloc_host_pool) with its own FIFO free list, counts and fills:
 *   - Swap out of a group of distinct resident sequences: every distinct
 *     device block the group holds gets one host block, in order of first
 *     appearance (sequences in the given order, each table in logical order),
 *     with count = the group members holding it and the block's fill.  The
 *     device block's count drops by that many; at zero it returns to the
 *     device free list (same order).  The tables then name host blocks.
 *   - Swap in: the mirror image, host blocks -> fresh device blocks.
 *   - Sharing inside a group survives the round trip; sharing with sequences
 *     outside it does not (each keeps its own copy).
 *   - A swapped-out sequence can be released (its host blocks go back to the
 *     host free list) or swapped in; append, fork, export and swap out return
 *     PKV_ERR_SWAPPED.
 *   - Each call returns the (source, destination) pairs whose data
 *     pkv_swap_blocks must move, in allocation order, before the blocks are
 *     used.  Out of blocks in the destination pool: PKV_ERR_OUT_OF_BLOCKS,
 *     nothing changed.
 */
typedef struct pkv_alloc pkv_alloc_t;

int pkv_alloc_create(int num_blocks, int block_size,
                     const int32_t *initial_free_order, pkv_alloc_t **out);
void pkv_alloc_destroy(pkv_alloc_t *a);

int pkv_seq_new(pkv_alloc_t *a, int *seq_id);

/* Append one token.  *slot_out = its slot; cow_pair_out = {src, dst} of a
 * copy-on-write, or {-1, -1}.  cow_pair_out may be NULL only if the caller
 * knows no copy can happen. */
int pkv_append_token(pkv_alloc_t *a, int seq, int64_t *slot_out,
                     int32_t cow_pair_out[2]);

/* Append n tokens to one sequence, all or nothing.  slots_out [n] (nullable)
 * receives their slots.  At most one copy-on-write can happen (the first
 * token's); cow_pair_out [2] (nullable) receives it, *n_cow (nullable) is 0
 * or 1. */
int pkv_append_tokens(pkv_alloc_t *a, int seq, int n, int64_t *slots_out,
                      int32_t *cow_pair_out, int *n_cow);

/* One decode step's appends: one token to each of the n DISTINCT sequences
 * seqs[0..n), in that order, all or nothing.  slots_out [n]; cow_pairs_out
 * [n][2] receives the copy-on-write pairs in order, *n_cow their count. */
int pkv_append_batch(pkv_alloc_t *a, const int32_t *seqs, int n,
                     int64_t *slots_out, int32_t *cow_pairs_out, int *n_cow);

int pkv_fork(pkv_alloc_t *a, int parent, int *child);

/* Release a sequence; *n_freed (nullable) = blocks returned to the free list. */
int pkv_release(pkv_alloc_t *a, int seq, int *n_freed);

/* Block tables and context lengths of n sequences, for the decode call.
 * tables [n][max_blocks_per_seq] row-major, padded with -1; ctx_lens [n]
 * (nullable).  A table longer than max_blocks_per_seq is an
 * PKV_ERR_INVALID_ARG (nothing written). */
int pkv_export_tables(const pkv_alloc_t *a, const int32_t *seqs, int n,
                      int32_t *tables, int max_blocks_per_seq,
                      int32_t *ctx_lens);

/* Prefix sharing of a batch, for pkv_paged_attention_decode_shared: for i in
 * [1, n), shared_out[i] = the number of leading logical blocks of sequence
 * seqs[i] whose physical block is the one of seqs[i-1] at the same logical
 * index (the blocks a fork shares with its parent until copy-on-write);
 * shared_out[0] = 0.  Same errors as pkv_export_tables (nothing written). */
int pkv_export_shared_prefix(const pkv_alloc_t *a, const int32_t *seqs, int n,
                             int32_t *shared_out);

int pkv_seq_length(const pkv_alloc_t *a, int seq, int *num_tokens);
int pkv_seq_num_blocks(const pkv_alloc_t *a, int seq, int *num_blocks);
int pkv_seq_table(const pkv_alloc_t *a, int seq, int32_t *table, int cap,
                  int *num_blocks);
int pkv_block_refcount(const pkv_alloc_t *a, int block, int *refs);
int pkv_block_fill(const pkv_alloc_t *a, int block, int *fill);
int pkv_num_free(const pkv_alloc_t *a, int *num_free);
/* The free list, front first: out [cap]; *n = its length. */
int pkv_free_list(const pkv_alloc_t *a, int32_t *out, int cap, int *n);

/* Give the manager a host pool of num_host_blocks blocks; host_free_order
 * (nullable) as for pkv_alloc_create.  Allowed while no host block is in use
 * (replaces the previous host pool). */
int pkv_alloc_host_pool(pkv_alloc_t *a, int num_host_blocks,
                        const int32_t *host_free_order);
/* Swap out / in n distinct sequences seqs[0..n).  pairs_out [cap][2] receives
 * the (source, destination) pairs, *n_pairs their count; cap must be at least
 * the total table length of the group (else PKV_ERR_INVALID_ARG, nothing
 * changed). */
int pkv_swap_out(pkv_alloc_t *a, const int32_t *seqs, int n, int32_t *pairs_out,
                 int cap, int *n_pairs);
int pkv_swap_in(pkv_alloc_t *a, const int32_t *seqs, int n, int32_t *pairs_out,
                int cap, int *n_pairs);
int pkv_seq_swapped(const pkv_alloc_t *a, int seq, int *swapped);
int pkv_host_block_refcount(const pkv_alloc_t *a, int block, int *refs);
int pkv_host_block_fill(const pkv_alloc_t *a, int block, int *fill);
int pkv_num_free_host(const pkv_alloc_t *a, int *num_free);
int pkv_host_free_list(const pkv_alloc_t *a, int32_t *out, int cap, int *n);

/*
 * Checkpoint of the block manager: its whole state as a byte blob, and an
 * object rebuilt from one.  The KV contents are the caller's device (or
 * pinned host) memory and are not part of it; a blob restores the tables
 * that index them.
 *
 * pkv_alloc_save: *bytes (required) receives the blob's size.  buf == NULL
 *   asks for the size only (PKV_OK).  Otherwise cap must be >= that size
 *   (else PKV_ERR_INVALID_ARG, nothing written) and the blob is written to
 *   buf (host memory, caller-owned).
 * pkv_alloc_load: builds a new object from `bytes` bytes at buf and stores
 *   it in *out (destroy it with pkv_alloc_destroy).  The restored object is
 *   indistinguishable from the saved one: same free-list orders, counts,
 *   fills, sequence ids (the next new id included), swap states and tables,
 *   so every later call gives the same results on both.
 *
 * Blob format (version 1), every field a little-endian int32 unless noted:
 *   magic 0x41564B50 ("PKVA" in memory), version, num_blocks, block_size,
 *   num_host_blocks, number of sequence ids handed out (M);
 *   device free list: its length F, then F block ids in FIFO order;
 *   device fills: num_blocks entries;
 *   host free list: length, then ids in FIFO order; host fills:
 *   num_host_blocks entries;
 *   M sequence records: flags (bit 0 alive, bit 1 swapped out), table
 *   length L, then L block ids (host block ids when swapped out).
 * Reference counts are not stored: they are the number of table entries
 * naming each block.  A blob is accepted only if it is a state the rules
 * above can reach: fields in range, every block either free (count 0, fill
 * 0, listed once) or held, every block but a table's last one full, a last
 * block holding 1..block_size tokens, no table or swap flag on a released
 * id, and no bytes left over.  Anything else returns PKV_ERR_INVALID_ARG
 * and leaves *out untouched.
 */
int pkv_alloc_save(const pkv_alloc_t *a, void *buf, size_t cap, size_t *bytes);
int pkv_alloc_load(const void *buf, size_t bytes, pkv_alloc_t **out);

/* ------------------------------------------------------------------------ */
/* Self-test                                                                 */
/* ------------------------------------------------------------------------ */

/*
 * Launches one CTA that waits, with the same bounded mbarrier wait the decode
 * kernel uses, on a barrier that nothing ever completes, giving up after
 * limit_ns nanoseconds.  The kernel then writes PKV_ERR_DEVICE_TIMEOUT to
 * dev_status and returns normally.  Lets a test check the give-up path
 * without a hang.  limit_ns must be in [1e3, 1e9].
 */
int pkv_selftest_wait_timeout(int32_t *dev_status, uint64_t limit_ns,
                              pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
