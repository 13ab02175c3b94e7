/*
 * CPU oracle for the paged KV-cache data path.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously correct statement
 * of what the GPU path computes.  Only the test-suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or helper with the CUDA library, and it imports nothing from it.
 *
 * Every step is integer index arithmetic plus byte copies: payload bytes are
 * opaque (bf16 bit patterns, NaN and -0 included) and are moved with memcpy.
 *
 * Sources (vLLM prefill/decode disaggregation pages):
 *  [S] drawing "vllm v1 调度逻辑 和 distributed 分布式原理":
 *      "batch tensor 组装"  slot_mapping[flat_token_i] =
 *          block_table[req_i, position_i // block_size] * block_size + position_i % block_size
 *      "Paged kv cache"      block B3 holds tokens t0..t15 in slots 0..15, K/V per slot
 *      per-layer panel       one tensor per layer (layer_0 .. layer_47), blocks contiguous
 *                            inside a layer, one block_table read by every layer
 *      last two labels       layer shapes (num_blocks, 2, bs, H, D) and (2, num_blocks, bs, H, D)
 *  [N] page "0. vllm 如何使用 nccl 传输 kv cache", section 2.4 (extract_kv_from_layer:
 *      layer[block_ids, ...] / layer[:, block_ids, ...]) and the transfer-flow step 14
 *      and consumer loop (kv_cache_layer[block_ids] = tensor)
 *  [F] page "5. flagcx connector design & dev & test", section 1.2: the sender flattens
 *      its work into an xfer_list over layers, contiguous groups and requests
 *  [M] page "vLLM PD 分离 源码级机制", section 4.2: per-layer, per-block source and
 *      destination addresses; _send_blocks issues (src_ptrs, dst_ptrs, lengths)
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - staging order: tensor, then request (given order), then block (list order),
 *    then plane (K, V), then token slot; every entry is one row slice.  For a
 *    blocks-first or single-plane layer this is exactly layer[block_ids] per
 *    (request, tensor) [N]; for kv-first the plane loop sits inside the block.
 *  - a "contiguous group" [F] is a maximal run of consecutive source ids (and of
 *    consecutive destination ids when those are given) inside one request, capped
 *    at max_run_blocks blocks (0 = no cap).
 *  - slot < 0 marks a padding token and is skipped.
 *  - a request's staged tokens are all slots of its listed source blocks; on a
 *    receiver with another block size, staged token j of request r lands in slot
 *    j % dst_bs of the (j / dst_bs)-th block of r's destination list.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t   n_tensors;
    uint8_t **base;          /* host address of each tensor */
    int64_t   num_blocks;
    int32_t   block_size;    /* token slots per block */
    int32_t   n_planes;      /* 1 (a K-only, V-only or latent tensor) or 2 (K and V planes) */
    int64_t   block_stride;  /* bytes from block b to block b+1 */
    int64_t   plane_stride;  /* bytes from the K plane to the V plane */
    int64_t   token_stride;  /* bytes from slot o to slot o+1 */
    int32_t   row_bytes;     /* bytes of one token row of one plane */
} ora_cache;

/* Address of the row of (tensor t, block, plane, slot offset). */
static uint8_t *row_addr(const ora_cache *c, int32_t t, int64_t block, int32_t plane, int64_t offset)
{
    return c->base[t] + block * c->block_stride + (int64_t)plane * c->plane_stride
         + offset * c->token_stride;
}

/* ---- slot_mapping [S] -------------------------------------------------------
 * block_table is [n_reqs, max_blocks] with row stride row_stride (elements).
 * A token whose request, position or table entry is invalid gets slot -1.
 * Returns the number of such tokens. */
int64_t ora_slot_mapping(const int32_t *block_table, int32_t n_reqs, int32_t max_blocks,
                         int64_t row_stride, const int32_t *token_req, const int32_t *token_pos,
                         int64_t n_tokens, int32_t block_size, int64_t *slot)
{
    int64_t bad = 0;
    for (int64_t i = 0; i < n_tokens; i++) {
        int32_t req = token_req[i];
        int32_t position = token_pos[i];
        if (req < 0 || req >= n_reqs || position < 0 || position / block_size >= max_blocks) {
            slot[i] = -1;
            bad++;
            continue;
        }
        int32_t block = block_table[(int64_t)req * row_stride + position / block_size];
        if (block < 0) {
            slot[i] = -1;
            bad++;
            continue;
        }
        slot[i] = (int64_t)block * block_size + position % block_size;
    }
    return bad;
}

static int cmp_i64(const void *a, const void *b)
{
    int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return (x > y) - (x < y);
}

/* ---- reshape_and_cache [S] ----------------------------------------------------
 * For every tensor t, plane p and token i with slot[i] >= 0:
 *   row (t, slot / bs, p, slot % bs) <- src[t * n_planes + p] + i * src_token_stride
 * src holds n_tensors * n_planes host addresses of [n_tokens, row_bytes] arrays.
 * Returns the number of tokens whose block lies outside the cache (those rows are
 * not written), or -1 (nothing written) when two tokens name the same slot. */
int64_t ora_reshape_and_cache(const ora_cache *c, uint8_t *const *src, int64_t src_token_stride,
                              const int64_t *slot, int64_t n_tokens)
{
    /* duplicates would make the result depend on write order: reject them */
    int64_t *sorted = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_tokens > 0 ? n_tokens : 1));
    int64_t m = 0;
    for (int64_t i = 0; i < n_tokens; i++)
        if (slot[i] >= 0) sorted[m++] = slot[i];
    qsort(sorted, (size_t)m, sizeof(int64_t), cmp_i64);
    for (int64_t i = 1; i < m; i++)
        if (sorted[i] == sorted[i - 1]) { free(sorted); return -1; }
    free(sorted);

    int64_t bad = 0;
    for (int64_t i = 0; i < n_tokens; i++) {
        if (slot[i] < 0) continue;                       /* padding token */
        int64_t block = slot[i] / c->block_size;
        int64_t offset = slot[i] % c->block_size;
        if (block >= c->num_blocks) { bad++; continue; }
        for (int32_t t = 0; t < c->n_tensors; t++)
            for (int32_t p = 0; p < c->n_planes; p++)
                memcpy(row_addr(c, t, block, p, offset),
                       src[(int64_t)t * c->n_planes + p] + i * src_token_stride,
                       (size_t)c->row_bytes);
    }
    return bad;
}

/* Request lists are CSR: request r owns list entries [req_offsets[r], req_offsets[r+1]). */
static int csr_ok(const int32_t *req_offsets, int32_t n_reqs, int64_t n_entries)
{
    if (n_reqs < 0 || req_offsets[0] != 0 || req_offsets[n_reqs] != n_entries) return 0;
    for (int32_t r = 0; r < n_reqs; r++)
        if (req_offsets[r + 1] < req_offsets[r]) return 0;
    return 1;
}

/* ---- xfer_list [F][M] -----------------------------------------------------------
 * Walks requests in order and blocks in list order.  Entry i starts a new run when
 * it is the first entry of its request, when src_ids[i] != src_ids[i-1] + 1, when
 * dst_ids is given and dst_ids[i] != dst_ids[i-1] + 1, or when the current run
 * already holds max_run_blocks blocks (max_run_blocks > 0).  Otherwise it extends
 * the current run.  A run records (request, first src id, first dst id or -1,
 * length, list position of its first entry).
 * Returns the number of runs; -1 if the CSR offsets are inconsistent; -2 if there
 * are more runs than capacity (the first capacity runs are written). */
int64_t ora_build_xfer_list(const int32_t *req_offsets, int32_t n_reqs,
                            const int32_t *src_ids, const int32_t *dst_ids, int64_t n_blocks,
                            int32_t max_run_blocks,
                            int32_t *run_req, int32_t *run_src, int32_t *run_dst,
                            int32_t *run_len, int64_t *run_stage, int64_t capacity)
{
    if (!csr_ok(req_offsets, n_reqs, n_blocks)) return -1;
    int64_t n_runs = 0;
    int64_t cur = -1;        /* index of the open run */
    int32_t cur_len = 0;
    for (int32_t r = 0; r < n_reqs; r++) {
        for (int64_t i = req_offsets[r]; i < req_offsets[r + 1]; i++) {
            int fresh = (i == req_offsets[r])
                     || (src_ids[i] != src_ids[i - 1] + 1)
                     || (dst_ids != NULL && dst_ids[i] != dst_ids[i - 1] + 1)
                     || (max_run_blocks > 0 && cur_len == max_run_blocks);
            if (fresh) {
                cur = n_runs++;
                cur_len = 1;
                if (cur < capacity) {
                    run_req[cur] = r;
                    run_src[cur] = src_ids[i];
                    run_dst[cur] = dst_ids != NULL ? dst_ids[i] : -1;
                    run_len[cur] = 1;
                    run_stage[cur] = i;
                }
            } else {
                cur_len++;
                if (cur < capacity) run_len[cur] = cur_len;
            }
        }
    }
    return n_runs > capacity ? -2 : n_runs;
}

/* ---- pack [N][F] ------------------------------------------------------------------
 * stage <- for each tensor t, request r, listed block (list order), plane p, slot o:
 *            the slice_bytes bytes at slice_off inside row (t, block, p, o).
 * Returns 0; -1 (nothing written) if the CSR is inconsistent, an id is outside the
 * cache or the slice does not fit in a row. */
int64_t ora_pack(const ora_cache *src, int32_t slice_off, int32_t slice_bytes,
                 const int32_t *req_offsets, int32_t n_reqs, const int32_t *src_ids,
                 int64_t n_blocks, uint8_t *stage)
{
    if (!csr_ok(req_offsets, n_reqs, n_blocks)) return -1;
    if (slice_off < 0 || slice_bytes <= 0 || slice_off + slice_bytes > src->row_bytes) return -1;
    for (int64_t i = 0; i < n_blocks; i++)
        if (src_ids[i] < 0 || src_ids[i] >= src->num_blocks) return -1;

    uint8_t *out = stage;
    for (int32_t t = 0; t < src->n_tensors; t++)
        for (int32_t r = 0; r < n_reqs; r++)
            for (int64_t i = req_offsets[r]; i < req_offsets[r + 1]; i++)
                for (int32_t p = 0; p < src->n_planes; p++)
                    for (int32_t o = 0; o < src->block_size; o++) {
                        memcpy(out, row_addr(src, t, src_ids[i], p, o) + slice_off, (size_t)slice_bytes);
                        out += slice_bytes;
                    }
    return 0;
}

/* ---- unpack [N][M] ----------------------------------------------------------------
 * Reads the staging buffer in the order pack wrote it (source geometry: src_block_size
 * slots and n_planes planes per staged block, slice_bytes per row).  Staged token j
 * of request r (j counts the slots of r's staged blocks in order) goes to slot
 * j % dst->block_size of block dst_ids[dst_req_offsets[r] + j / dst->block_size],
 * at byte dst_slice_off of the row.
 * Returns 0; -1 (nothing written) if a list is inconsistent, the geometry does not
 * fit, a request's destination list is too short, a destination id is outside the
 * cache, or two staged tokens would land in the same destination block. */
int64_t ora_unpack(const ora_cache *dst, int32_t dst_slice_off, int32_t slice_bytes,
                   int32_t src_block_size, int32_t n_planes,
                   const int32_t *req_offsets, int32_t n_reqs, int64_t n_blocks,
                   const int32_t *dst_req_offsets, const int32_t *dst_ids, int64_t n_dst_ids,
                   const uint8_t *stage)
{
    if (!csr_ok(req_offsets, n_reqs, n_blocks) || !csr_ok(dst_req_offsets, n_reqs, n_dst_ids)) return -1;
    if (n_planes != dst->n_planes || src_block_size <= 0) return -1;
    if (dst_slice_off < 0 || slice_bytes <= 0 || dst_slice_off + slice_bytes > dst->row_bytes) return -1;

    /* every destination block that receives a token, for the duplicate check */
    int64_t *used = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_dst_ids > 0 ? n_dst_ids : 1));
    int64_t n_used = 0;
    for (int32_t r = 0; r < n_reqs; r++) {
        int64_t tokens = (int64_t)(req_offsets[r + 1] - req_offsets[r]) * src_block_size;
        int64_t need = (tokens + dst->block_size - 1) / dst->block_size;
        if (need > dst_req_offsets[r + 1] - dst_req_offsets[r]) { free(used); return -1; }
        for (int64_t q = 0; q < need; q++) {
            int32_t b = dst_ids[dst_req_offsets[r] + q];
            if (b < 0 || b >= dst->num_blocks) { free(used); return -1; }
            used[n_used++] = b;
        }
    }
    qsort(used, (size_t)n_used, sizeof(int64_t), cmp_i64);
    for (int64_t k = 1; k < n_used; k++)
        if (used[k] == used[k - 1]) { free(used); return -1; }
    free(used);

    const uint8_t *in = stage;
    for (int32_t t = 0; t < dst->n_tensors; t++)
        for (int32_t r = 0; r < n_reqs; r++)
            for (int64_t q = 0; q < req_offsets[r + 1] - req_offsets[r]; q++)
                for (int32_t p = 0; p < n_planes; p++)
                    for (int32_t o = 0; o < src_block_size; o++) {
                        int64_t j = q * src_block_size + o;      /* staged token of request r */
                        int32_t block = dst_ids[dst_req_offsets[r] + j / dst->block_size];
                        memcpy(row_addr(dst, t, block, p, j % dst->block_size) + dst_slice_off,
                               in, (size_t)slice_bytes);
                        in += slice_bytes;
                    }
    return 0;
}

/* ---- sliding-window clip [M section 3.1] -------------------------------------------
 * request_finished hands the sender get_sw_clipped_blocks(block_ids); the function's body
 * is not on the page.  Reading: a layer whose attention sees only the last `window`
 * tokens needs, of a request with n = n_tokens[r] tokens, only the blocks that hold tokens
 * max(0, n - window) .. n - 1, i.e. list entries
 *     q = max(0, n - window) / block_size  ..  ceil(n / block_size) - 1
 * (never past the request's list).  window <= 0 keeps every block that holds a token.
 * The kept entries go, in order, to out_ids with CSR out_offsets[n_reqs + 1].
 * Returns the number of kept entries; -1 if the CSR is inconsistent, block_size <= 0 or
 * a token count is negative. */
int64_t ora_clip_block_lists(const int32_t *req_offsets, int32_t n_reqs, const int32_t *ids, int64_t n_ids,
                             const int32_t *n_tokens, int32_t window, int32_t block_size,
                             int32_t *out_offsets, int32_t *out_ids)
{
    if (!csr_ok(req_offsets, n_reqs, n_ids) || block_size <= 0) return -1;
    int64_t k = 0;
    out_offsets[0] = 0;
    for (int32_t r = 0; r < n_reqs; r++) {
        int64_t n = n_tokens[r];
        if (n < 0) return -1;
        int64_t first_token = (window > 0 && n > window) ? n - window : 0;
        int64_t first = first_token / block_size;
        int64_t end = (n + block_size - 1) / block_size;
        int64_t len = req_offsets[r + 1] - req_offsets[r];
        if (end > len) end = len;
        for (int64_t q = first; q < end; q++) out_ids[k++] = ids[req_offsets[r] + q];
        out_offsets[r + 1] = (int32_t)k;
    }
    return k;
}

/* ---- prefix hash chain over token blocks [S] --------------------------------------
 * The drawing's hash table ("cached_block_hash_to_block") keys every full block by a chain:
 *     h0 = hash(seed, [t0 .. t(bs-1)]),  h_i = hash(h_(i-1), [tokens of block i])
 * The pages do not name the hash.  Reading: FNV-1a 64 (offset basis 0xcbf29ce484222325,
 * prime 0x100000001b3, each byte xored in, then multiplied) over the parent hash as 8
 * little-endian bytes followed by the block's token ids as 4 little-endian bytes each.
 * Only full blocks are hashed (a partial last block is not cacheable yet). */
uint64_t ora_fnv1a64(const uint8_t *data, int64_t len)
{
    uint64_t h = 0xcbf29ce484222325ull;
    for (int64_t i = 0; i < len; i++) {
        h ^= data[i];
        h *= 0x100000001b3ull;
    }
    return h;
}

/* tok_offsets [n_reqs + 1] is the CSR of each request's token ids in tokens.  Writes the
 * hashes of every request's full blocks, in order, to out_hashes with CSR out_offsets
 * [n_reqs + 1].  Returns the number of hashes, or -1 if the CSR is inconsistent or
 * block_size <= 0. */
int64_t ora_block_hashes(const int32_t *tok_offsets, int32_t n_reqs, const int32_t *tokens, int64_t n_tokens,
                         int32_t block_size, uint64_t seed, int32_t *out_offsets, uint64_t *out_hashes)
{
    if (!csr_ok(tok_offsets, n_reqs, n_tokens) || block_size <= 0) return -1;
    uint8_t *buf = (uint8_t *)malloc(8 + 4 * (size_t)block_size);
    int64_t k = 0;
    out_offsets[0] = 0;
    for (int32_t r = 0; r < n_reqs; r++) {
        int64_t n = tok_offsets[r + 1] - tok_offsets[r];
        uint64_t parent = seed;
        for (int64_t b = 0; b < n / block_size; b++) {
            for (int j = 0; j < 8; j++) buf[j] = (uint8_t)(parent >> (8 * j));
            for (int32_t t = 0; t < block_size; t++) {
                uint32_t id = (uint32_t)tokens[tok_offsets[r] + b * block_size + t];
                for (int j = 0; j < 4; j++) buf[8 + 4 * t + j] = (uint8_t)(id >> (8 * j));
            }
            parent = ora_fnv1a64(buf, 8 + 4 * (int64_t)block_size);
            out_hashes[k++] = parent;
        }
        out_offsets[r + 1] = (int32_t)k;
    }
    free(buf);
    return k;
}
