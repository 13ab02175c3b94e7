/*
 * pagedkv.h - C ABI of libpagedkv.so: paged KV-cache data movement on one GB300 (sm_103a).
 *
 * The library moves paged KV-cache bytes the way a prefill/decode-disaggregated
 * vLLM deployment does on each GPU:
 *   1. kv_slot_mapping + kv_reshape_and_cache   write new tokens' K/V into the paged
 *                                               per-layer caches;
 *   2. kv_build_xfer_list                       flatten per-request block lists into
 *                                               maximal contiguous block runs;
 *   3. kv_pack_blocks                           gather those runs into one contiguous
 *                                               staging buffer (the sender's payload);
 *   4. kv_unpack_blocks                         scatter a staging buffer into the
 *                                               receiver's own block ids, optionally
 *                                               with another block size or a head slice.
 * The network transfer between machines is not part of this library.
 *
 * Conventions for every entry point
 *  - Pointers named "device" are caller-owned CUDA device memory; the library never
 *    allocates, frees or keeps them.  Host arrays (kv_cache_desc.base, the new_kv
 *    pointer table) are read during the call only.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and never synchronises, except kv_get_last_error.
 *  - Kernels of a few waves or less are launched with programmatic stream serialisation
 *    allowed, so their CTAs may be scheduled while the previous kernel on `stream` still runs;
 *    each waits for that kernel to complete before its first memory access, so the data sees
 *    plain stream order.  Launches that fill the GPU for longer (pack and unpack with tail
 *    CTAs, row writes of more than two waves) are plain stream-ordered launches.
 *  - The first call of an entry point on a device sets up per-device state (launch
 *    attributes, occupancy, symbol addresses; the first kv_wait_signal loads every kernel):
 *    make it outside a stream capture.  Calls after it can be captured into CUDA graphs.
 *  - That per-device state (the error word's address, the static builder scratch's address,
 *    occupancy figures) is kept for the life of the process and is not looked up again: it does
 *    not survive cudaDeviceReset or a reset of the device's primary context.  A process that
 *    resets a device must not call this library on that device afterwards.
 *  - Payload bytes are opaque: rows are moved as 16-byte vectors and never converted,
 *    so NaN payloads, infinities and -0 arrive bit-exact.
 *  - Argument errors the host can see are returned at once and nothing is launched.
 *    Data-dependent errors (an id or slot outside the cache, a list inconsistent with
 *    its offsets) skip only the offending write and set a bit in a sticky per-device
 *    error word, read and cleared with kv_get_last_error.
 *  - Base addresses, strides, row and slice sizes and staging pointers must be multiples
 *    of 16 bytes (KV_ERR_ALIGN otherwise).
 *
 * Sources (the vLLM PD-disaggregation pages this library restates):
 *  [S] drawing "vllm v1 调度逻辑 和 distributed 分布式原理": "batch tensor 组装" (the slot
 *      formula), "Paged kv cache" (16 slots per block), the per-layer tensor panel (one
 *      tensor per layer, one block_table for all layers) and the two layer shapes.
 *  [N] page "0. vllm 如何使用 nccl 传输 kv cache", sections 2.3 (transfer flow) and 2.4
 *      (extract_kv_from_layer / inject_kv_into_layer).
 *  [F] page "5. flagcx connector design & dev & test", section 1.2 (the xfer_list, flattened
 *      over layers, contiguous groups and requests).
 *  [M] page "vLLM PD 分离 源码级机制", sections 4.1 (receiver metadata: base addresses,
 *      block lengths, local block ids) and 4.2 (_build_transfer_params, _send_blocks).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Entry points are the only symbols libpagedkv.so exports. */
#if defined(__GNUC__)
#define KV_API __attribute__((visibility("default")))
#else
#define KV_API
#endif

typedef struct CUstream_st *kv_stream_t; /* identical to cudaStream_t */

/* Status codes returned by every entry point. */
enum {
    KV_OK = 0,
    KV_ERR_INVALID_ARG = 1, /* null pointer, negative size, inconsistent descriptor */
    KV_ERR_ALIGN = 2,       /* an address, stride or size is not a multiple of 16 bytes */
    KV_ERR_RANGE = 3,       /* a size does not fit: slice beyond the row, staging too small */
    KV_ERR_CUDA = 4,        /* a CUDA runtime call failed (see kv_last_cuda_error) */
    KV_ERR_TIMEOUT = 5,     /* a bounded device wait gave up */
    KV_ERR_UNSUPPORTED = 6  /* outside the implemented limits (documented per call) */
};

/* Bits of the sticky device error word (kv_get_last_error). */
#define KV_DERR_TABLE     0x01 /* slot_mapping: request, position or table entry invalid (slot -1 written) */
#define KV_DERR_SLOT      0x02 /* reshape_and_cache: slot beyond num_blocks * block_size (row skipped) */
#define KV_DERR_BLOCK     0x04 /* pack/unpack: a run names a block outside the cache (run skipped) */
#define KV_DERR_LIST      0x08 /* xfer builder: req_offsets[0] != 0 or req_offsets[n_reqs] != n_blocks */
#define KV_DERR_CAPACITY  0x10 /* more runs than run_capacity (extra runs not written / not copied) */
#define KV_DERR_STAGE     0x20 /* a run's staging range lies outside the staging buffer (run skipped) */
#define KV_DERR_DST_TABLE 0x40 /* unpack remap: a request's destination list is too short (rows skipped) */
#define KV_DERR_TIMEOUT   0x80 /* a bounded device wait gave up */

/*
 * Geometry of one paged cache [S][M].  A cache is n_tensors device tensors of equal
 * geometry (one per layer, or one K and one V tensor per layer).  Row (t, b, p, o) -
 * tensor t, block b, plane p (0 = K, 1 = V when a tensor holds both), slot o - starts at
 *     base[t] + b * block_stride + p * plane_stride + o * token_stride
 * and holds row_bytes bytes (heads * head_dim * element size).  Examples:
 *     separate K/V [num_blocks, bs, H, D]:  n_planes 1, block_stride bs*row, token_stride row
 *     blocks-first [num_blocks, 2, bs, H, D]: n_planes 2, plane_stride bs*row, block_stride 2*bs*row
 *     kv-first     [2, num_blocks, bs, H, D]: n_planes 2, plane_stride num_blocks*bs*row
 *     MLA latent   [num_blocks, bs, 576]:    n_planes 1, row 1152
 * base is a HOST array of n_tensors device addresses; it is read during the call only.
 */
typedef struct {
    int32_t n_tensors;
    int32_t block_size;   /* token slots per block (> 0) */
    int32_t n_planes;     /* 1 or 2 */
    int32_t row_bytes;    /* bytes of one token row of one plane */
    int64_t num_blocks;   /* blocks per tensor */
    int64_t block_stride; /* bytes */
    int64_t plane_stride; /* bytes (ignored when n_planes == 1) */
    int64_t token_stride; /* bytes */
    const uint64_t *base; /* host array [n_tensors] of device addresses */
} kv_cache_desc;

/*
 * Layout of a staging buffer [N][F].  Staged entry (t, i, p, o) - tensor t, entry i of
 * the flattened block list (requests in order, each request's blocks in list order),
 * plane p, slot o of the source block size - is slice_bytes bytes at
 *     ((((t * n_blocks + i) * n_planes + p) * block_size) + o) * slice_bytes.
 * For a whole-row slice this is layer[block_ids] per (request, tensor) concatenated,
 * i.e. the tensor the NCCL connector sends per "request_id#layer_name" [N].
 */
typedef struct {
    int64_t n_blocks;    /* N: entries in the flattened source block list */
    int32_t n_tensors;
    int32_t n_planes;
    int32_t block_size;  /* SOURCE block size */
    int32_t slice_bytes; /* bytes per staged row (multiple of 16) */
} kv_stage_desc;

/* One contiguous group [F][M]: n_blocks consecutive source ids starting at src_block,
 * landing on consecutive destination ids starting at dst_block (-1 when the list had no
 * destination ids), occupying staging entries stage_block .. stage_block + n_blocks - 1.
 * 24 bytes, 8-byte aligned. */
typedef struct {
    int32_t req;
    int32_t src_block;
    int32_t dst_block;
    int32_t n_blocks;
    int64_t stage_block;
} kv_xfer_run;

/* Library version string, e.g. "pagedkv 0.1.0 sm_103a". */
KV_API const char *kv_version(void);

/* Human-readable name of a status code. */
KV_API const char *kv_status_string(int status);

/* The last CUDA runtime error seen by a call that returned KV_ERR_CUDA (cudaError_t value). */
KV_API int kv_last_cuda_error(void);

/*
 * kv_slot_mapping [S "batch tensor 组装"]:
 *     slot_out[i] = block_table[token_req[i] * bt_row_stride + token_pos[i] / block_size] * block_size
 *                   + token_pos[i] % block_size
 * block_table: device int32 [n_reqs, max_blocks_per_req] with row stride bt_row_stride
 * (elements); token_req, token_pos: device int32 [n_tokens]; slot_out: device int64
 * [n_tokens].  A token whose request is outside [0, n_reqs), whose position is negative
 * or beyond max_blocks_per_req * block_size, or whose table entry is negative gets
 * slot -1 and sets KV_DERR_TABLE.  n_tokens == 0 launches nothing.
 */
KV_API int kv_slot_mapping(const int32_t *block_table, int32_t n_reqs, int32_t max_blocks_per_req,
                    int64_t bt_row_stride, const int32_t *token_req, const int32_t *token_pos,
                    int64_t n_tokens, int32_t block_size, int64_t *slot_out, kv_stream_t stream);

/*
 * kv_reshape_and_cache [S "Paged kv cache", M section 6 timeline (prefill writes the KV cache into local GPU memory)]:
 * for every cache tensor t, plane p and token i with slot[i] >= 0,
 *     row (t, slot[i] / block_size, p, slot[i] % block_size) <- new_kv[t * n_planes + p] + i * new_token_stride
 * All tensors of the descriptor (e.g. every layer of a decode step) are written by one
 * launch per 128 tensors.  new_kv: HOST array of n_tensors * n_planes device addresses,
 * each of [n_tokens] rows of cache->row_bytes bytes, new_token_stride bytes apart.
 * slot: device int64 [n_tokens]; slot < 0 is a padding token and is skipped; a slot at
 * or beyond num_blocks * block_size sets KV_DERR_SLOT and is skipped.  Two tokens with
 * the same slot race (undefined which row lands).  Limits: num_blocks * block_size
 * < 2^31 and n_tokens * n_planes * row_bytes / 16 < 2^31 (KV_ERR_UNSUPPORTED).
 */
KV_API int kv_reshape_and_cache(const kv_cache_desc *cache, const uint64_t *new_kv, int64_t new_token_stride,
                         const int64_t *slot, int64_t n_tokens, kv_stream_t stream);

/*
 * kv_write_tokens [S "batch tensor 组装", "Paged kv cache"]: kv_slot_mapping and
 * kv_reshape_and_cache in one call.  Each token's slot is looked up in the block table inside
 * the row-copy kernel (block_size = cache->block_size), one launch per 128 tensors, and
 * written to slot_out when it is given.  A row shape whose n_planes * row_bytes / 16 chunks
 * need more than 16 CTAs of 256 threads to span a whole number of tokens (e.g. 17 or 25
 * chunks) takes a kernel without the pipelined lookup; with slot_out given it then runs as
 * the two calls.  Arguments as for the two calls; slot_out (device
 * int64 [n_tokens], may be NULL) receives the slots, -1 for invalid tokens, exactly as
 * kv_slot_mapping writes them.  An invalid token sets KV_DERR_TABLE and writes nothing; a slot
 * beyond the cache sets KV_DERR_SLOT.  Limits as for kv_reshape_and_cache.
 */
KV_API int kv_write_tokens(const kv_cache_desc *cache, const uint64_t *new_kv, int64_t new_token_stride,
                           const int32_t *block_table, int32_t n_reqs, int32_t max_blocks_per_req,
                           int64_t bt_row_stride, const int32_t *token_req, const int32_t *token_pos,
                           int64_t n_tokens, int64_t *slot_out, kv_stream_t stream);

/* Device workspace bytes kv_build_xfer_list needs for a list of n_blocks entries. */
KV_API int kv_xfer_workspace_bytes(int64_t n_blocks, int64_t *bytes_out);

/*
 * kv_build_xfer_list [F section 1.2, M section 4.2]: flattens per-request block lists
 * into runs, in request order then list order.  Entry i starts a new run when it is
 * the first entry of its request, when src_ids[i] != src_ids[i-1] + 1, when dst_ids
 * is given and dst_ids[i] != dst_ids[i-1] + 1, or when the open run already holds
 * max_run_blocks blocks (max_run_blocks > 0; 0 = uncapped).  Ids keep their list
 * order; nothing is sorted.
 * req_offsets: device int32 [n_reqs + 1] (CSR: request r owns entries
 * [req_offsets[r], req_offsets[r+1]), req_offsets[0] = 0, req_offsets[n_reqs] =
 * n_blocks); src_ids, dst_ids: device int32 [n_blocks], dst_ids may be NULL.
 * Output: runs (device, run_capacity records) and *n_runs (device int32, the total
 * number of runs, even when it exceeds run_capacity, in which case KV_DERR_CAPACITY is
 * set and only the first run_capacity runs are written; n_blocks runs always suffice).
 * workspace: device scratch of kv_xfer_workspace_bytes(n_blocks) bytes, 16-byte
 * aligned, zeroed by this call on `stream`; calls sharing a workspace must be ordered.
 * Lists of up to 5120 entries are built by one CTA that leaves the workspace untouched
 * (it must still be passed and large enough).
 * Limit: n_blocks < 2^31 - 2^12.
 */
KV_API int kv_build_xfer_list(const int32_t *req_offsets, int32_t n_reqs, const int32_t *src_ids,
                       const int32_t *dst_ids, int64_t n_blocks, int32_t max_run_blocks,
                       kv_xfer_run *runs, int64_t run_capacity, int32_t *n_runs,
                       void *workspace, int64_t workspace_bytes, kv_stream_t stream);

/*
 * kv_build_xfer_list_static - the pages have no counterpart to this entry point.
 * It is kv_build_xfer_list with the same arguments and results, except that it needs no
 * workspace: its look-back scratch is a fixed array of KV_XFER_STATIC_SCRATCH_BYTES
 * (64 KiB) inside libpagedkv.so, held by every GPU that loads the library until the
 * process exits.  It is for callers that cannot allocate device memory at the moment
 * they build a transfer list: a transport's progress thread, where cudaMalloc and
 * cudaFree may synchronise the device and stall the model's stream, or a serving
 * process whose KV-cache pool already reserved nearly all free device memory, where
 * even a small allocation can fail.  Nothing here calls cudaMalloc, cudaFree or any
 * allocating routine; the caller still passes the inputs and the runs / n_runs outputs.
 *  - n_blocks above KV_XFER_STATIC_MAX_BLOCKS is rejected with KV_ERR_RANGE before
 *    anything is queued.
 *  - The first call on each device looks up the array's device address with
 *    cudaGetSymbolAddress (with that device current) and caches it; make that first call
 *    before any stream capture.
 *  - Every call clears the part of the array it uses on `stream` before its kernel runs.
 *    All calls on a device share the one array, so calls that overlap on the GPU (on
 *    different streams without ordering) race and produce garbage; order them.
 */
#define KV_XFER_STATIC_SCRATCH_BYTES 65536
#define KV_XFER_STATIC_MAX_BLOCKS 4177920 /* 2040 tiles of 2048 entries: (65536 - 256) / 32 */
KV_API int kv_build_xfer_list_static(const int32_t *req_offsets, int32_t n_reqs, const int32_t *src_ids,
                                     const int32_t *dst_ids, int64_t n_blocks, int32_t max_run_blocks,
                                     kv_xfer_run *runs, int64_t run_capacity, int32_t *n_runs,
                                     kv_stream_t stream);

/*
 * kv_clip_block_lists [M section 3.1: request_finished sends get_sw_clipped_blocks(block_ids)]:
 * the sliding-window clip of per-request block lists, applied before kv_build_xfer_list.  The
 * function's body is not on the page; reading: a layer attending to the last `window` tokens
 * needs, of request r with n_tokens[r] tokens, only its list entries
 *     q = max(0, n_tokens[r] - window) / block_size  ..  ceil(n_tokens[r] / block_size) - 1
 * (never past the request's list); window <= 0 keeps every entry that holds a token.
 * req_offsets (n_reqs + 1), ids (n_ids), n_tokens (n_reqs): device int32.  Writes the kept
 * entries, in order, to out_ids (device, out_capacity >= n_ids) with CSR out_offsets
 * (device int32, n_reqs + 1).  The kept count is out_offsets[n_reqs]; a caller that knows
 * n_tokens and the list lengths on the host can compute it without reading the device.
 * Clip a destination list that is aligned entry-by-entry with the source list with the same
 * arguments to keep the two aligned.  Inconsistent offsets or negative token counts set
 * KV_DERR_LIST; no write ever leaves out_ids.  Limit: n_ids < 2^31.
 */
KV_API int kv_clip_block_lists(const int32_t *req_offsets, int32_t n_reqs, const int32_t *ids, int64_t n_ids,
                               const int32_t *n_tokens, int32_t window, int32_t block_size,
                               int32_t *out_offsets, int32_t *out_ids, int64_t out_capacity, kv_stream_t stream);

/*
 * kv_block_hashes [S: the hash-table labels h0 = hash(seed, [t0..t1]), h1 = hash(h0, [t2..t3]), ...
 * keying cached_block_hash_to_block]: the prefix hash chain over every request's FULL token
 * blocks, h_i = H(h_(i-1), tokens of block i) with h_(-1) = seed, so requests sharing a prefix
 * share its hashes.  The pages do not name H; this library reads it as FNV-1a 64 (basis
 * 0xcbf29ce484222325, prime 0x100000001b3) over h_(i-1) as 8 little-endian bytes followed by the
 * block's token ids as 4 little-endian bytes each.  A partial last block is not hashed.
 * tok_offsets (n_reqs + 1) is the CSR of each request's token ids in tokens (device int32).
 * Writes the hashes, in order, to out_hashes (device uint64, 8-byte aligned, out_capacity >=
 * n_tokens / block_size) with CSR out_offsets (device int32, n_reqs + 1).  Inconsistent
 * offsets set KV_DERR_LIST and no write leaves out_hashes.  Limit: n_tokens < 2^31.
 * workspace: NULL, or device scratch of at least 2 KiB per slot (n_tokens / block_size slots),
 * 16-byte aligned; kv_block_hashes_workspace_bytes(n_tokens, block_size) gives the full size,
 * 2 KiB + 4 bytes per slot rounded up to 16.  Calls sharing a workspace must be ordered.
 *  - With a workspace, every block's hash is split by a property of FNV-1a (the xor of a byte
 *    changes only the state's low byte, so the rest of a step is linear): each block's token
 *    contribution is tabulated for all 256 possible low bytes of the state after the parent,
 *    in parallel, and one warp per request then walks its chain doing, per block, the
 *    low-byte chain of the parent's 8 bytes, a table lookup and a sum.  With the full size,
 *    the tables and the walks run in one cooperative launch (walkers on SMs of their own read
 *    each table once it is published) when the walk is the longer part, as for a few long
 *    prompts; otherwise, or with a workspace of the tables alone, a table kernel runs first.
 *    A wait that runs out (2 s) sets KV_DERR_TIMEOUT.
 *  - Without one, one thread per request runs the plain byte chain (about 5x slower for
 *    16-token blocks).  Every path gives the same hashes.
 */
KV_API int kv_block_hashes_workspace_bytes(int64_t n_tokens, int32_t block_size, int64_t *bytes_out);
KV_API int kv_block_hashes(const int32_t *tok_offsets, int32_t n_reqs, const int32_t *tokens, int64_t n_tokens,
                           int32_t block_size, uint64_t seed, int32_t *out_offsets, uint64_t *out_hashes,
                           int64_t out_capacity, void *workspace, int64_t workspace_bytes, kv_stream_t stream);

/*
 * kv_pack_blocks [N section 2.4 extract_kv_from_layer, F section 1.2]: for every
 * tensor t and run of `runs`, copies rows (t, src_block + m, p, o) - byte slice
 * [src_slice_off, src_slice_off + stage->slice_bytes) of each row - to the staging
 * entries (t, stage_block + m, p, o) of the layout in kv_stage_desc.
 * stage->n_tensors, n_planes and block_size must equal the cache's.  runs/n_runs are
 * device memory as written by kv_build_xfer_list; at most run_capacity runs are read
 * (KV_DERR_CAPACITY if *n_runs is larger).  max_run_blocks is the cap the runs were
 * built with (0 if uncapped): runs are split into pieces of at most 16 KiB for the
 * warps by it; a longer run is still copied whole.  stage_buf: device memory, or pinned
 * host memory (cudaHostAlloc / cudaHostRegister) when the payload is to be spilled to the
 * host as the NCCL page's receiver does past its buffer threshold [N section 2.3]; the
 * copy then runs over the host link.  Unregistered host memory is KV_ERR_INVALID_ARG.
 * stage_bytes bytes, at least
 * n_tensors * n_blocks * n_planes * block_size * slice_bytes.  A run outside the cache
 * (KV_DERR_BLOCK) or the staging range (KV_DERR_STAGE) is skipped.
 */
KV_API int kv_pack_blocks(const kv_cache_desc *src, int32_t src_slice_off, const kv_stage_desc *stage,
                   const kv_xfer_run *runs, const int32_t *n_runs, int64_t run_capacity,
                   int32_t max_run_blocks, void *stage_buf, int64_t stage_bytes, kv_stream_t stream);

/*
 * kv_unpack_blocks [N section 2.3 step 14 (kv_cache_layer[block_ids] = tensor),
 * M sections 4.1-4.2 (receiver block ids, TP heterogeneity)]: the inverse of pack, into
 * the receiver's cache `dst`, writing each staged row slice at byte dst_slice_off of the
 * destination row (stage->slice_bytes bytes).
 *  - Whole-block mode (dst_ids == NULL): staged block stage_block + m of each run goes to
 *    destination block dst_block + m (runs built with destination ids).  Needs
 *    stage->block_size == dst->block_size.
 *  - Remap mode (dst_ids != NULL): staged token j of request r (j counts the slots of r's
 *    staged blocks in order) goes to slot j % dst->block_size of block
 *    dst_ids[dst_req_offsets[r] + j / dst->block_size].  src_req_offsets is the CSR the
 *    runs were built from; dst_req_offsets/dst_ids the receiver's per-request block
 *    lists (device int32, n_reqs + 1 and any length).  A request whose destination list
 *    is too short sets KV_DERR_DST_TABLE and its uncovered rows are skipped.
 * max_run_blocks, stage_buf: as for kv_pack_blocks (pinned host staging is read over the
 * host link).
 * stage->n_tensors and n_planes must equal dst's.  Destination ids must be distinct:
 * two staged rows aimed at one destination row race.  A call with nothing staged
 * (stage->n_blocks == 0) returns KV_OK before the mode is looked at, so an empty
 * destination list passed as a null dst_ids is fine.
 */
KV_API int kv_unpack_blocks(const kv_cache_desc *dst, int32_t dst_slice_off, const kv_stage_desc *stage,
                     const kv_xfer_run *runs, const int32_t *n_runs, int64_t run_capacity,
                     int32_t max_run_blocks, const void *stage_buf, int64_t stage_bytes,
                     const int32_t *src_req_offsets, const int32_t *dst_req_offsets,
                     const int32_t *dst_ids, int32_t n_reqs, kv_stream_t stream);

/*
 * Transfer-completion signal [F section 1.2]: the receiver's per-pair signal counter.
 * The sender's last put of a transfer adds 1; the receiver waits until the counter reaches
 * the largest value it expects, which covers every transfer before it.  16 bytes of device
 * memory, 16-byte aligned, zeroed once by the caller and then only touched by these calls.
 */
typedef struct {
    uint64_t value;    /* monotonic counter */
    uint32_t arrived;  /* internal: CTAs of the current signalled call that have finished */
    uint32_t reserved;
} kv_signal;

/*
 * kv_unpack_blocks_signal [N section 2.3 step 14, F section 1.2]: kv_unpack_blocks, and once
 * every row of this call has landed in dst (all tensors), signal->value += add with release
 * semantics at GPU scope - done by the last CTA of the copy kernel, so no extra launch is
 * needed (a call with nothing to copy posts the increment with a one-thread kernel).
 * Signalled calls sharing a signal must be ordered (one stream, or events).
 */
KV_API int kv_unpack_blocks_signal(const kv_cache_desc *dst, int32_t dst_slice_off, const kv_stage_desc *stage,
                                   const kv_xfer_run *runs, const int32_t *n_runs, int64_t run_capacity,
                                   int32_t max_run_blocks, const void *stage_buf, int64_t stage_bytes,
                                   const int32_t *src_req_offsets, const int32_t *dst_req_offsets,
                                   const int32_t *dst_ids, int32_t n_reqs, kv_signal *signal, uint64_t add,
                                   kv_stream_t stream);

/*
 * kv_wait_signal [F section 1.2, flagcxWaitSignal: the receiver polls the signal counter on the GPU until it reaches the expected value]:
 * queues on `stream` a one-thread kernel that polls signal->value (acquire loads) until it
 * is >= expected, so work queued after it on `stream` starts only then.  The wait is
 * bounded: after timeout_us microseconds (1 .. 60,000,000; otherwise KV_ERR_RANGE) it gives
 * up, writes KV_ERR_TIMEOUT to *status_out (device int32, may be NULL) and sets
 * KV_DERR_TIMEOUT; on success it writes KV_OK.  The context stays usable either way.
 * While it polls, the work that sets the counter runs on another stream, and its kernels must
 * already be loaded: CUDA loads a kernel's code lazily, on first use, and that load may
 * synchronise the context, which would hold the producer's launch until this wait ends.  The
 * first call on a device (outside a stream capture) loads every kernel of this library
 * before it queues the poll; load your own producer kernels first (run them once, or set
 * CUDA_MODULE_LOADING=EAGER).  The
 * kernels queued after the wait on `stream` are scheduled only once it ends, so they cannot
 * take the SM space the producer needs.
 */
KV_API int kv_wait_signal(const kv_signal *signal, uint64_t expected, uint32_t timeout_us, int32_t *status_out,
                          kv_stream_t stream);

/*
 * kv_get_last_error: copies the current device's sticky error word (KV_DERR_* bits) to
 * *host_out after the work queued on `stream` so far, clears it when clear != 0, and
 * SYNCHRONISES `stream`.  Work on other streams is not waited for.
 */
KV_API int kv_get_last_error(int32_t *host_out, int32_t clear, kv_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDKV_H */
