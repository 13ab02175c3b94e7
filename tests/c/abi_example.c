/* A plain C11 caller of libpagedkv.so: the header alone is enough to drive the path.
 * It builds a tiny cache, writes two new tokens through slot_mapping + reshape_and_cache,
 * lists two requests' blocks, builds the xfer_list, packs into a staging buffer, unpacks into
 * a second cache at other block ids, and checks the bytes.  It then hashes two token lists
 * with and without a workspace and checks the first hash against FNV-1a computed here. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime.h>

#include "pagedkv.h"

#define NB 8       /* blocks */
#define BS 4       /* slots per block */
#define ROW 32     /* bytes per token row */
#define BLK (BS * ROW)

#define CHECK(x)                                                            \
    do {                                                                    \
        int s_ = (x);                                                       \
        if (s_ != KV_OK) {                                                  \
            fprintf(stderr, "%s -> %s\n", #x, kv_status_string(s_));        \
            return 1;                                                       \
        }                                                                   \
    } while (0)

int main(void)
{
    uint8_t host[NB * BLK], back[NB * BLK];
    for (int i = 0; i < NB * BLK; i++) host[i] = (uint8_t)(i * 7 + 3);
    const int32_t offsets[3] = {0, 2, 3}; /* request 0: blocks 5, 6; request 1: block 1 */
    const int32_t src_ids[3] = {5, 6, 1};
    const int32_t dst_ids[3] = {2, 3, 7};

    void *src = 0, *dst = 0, *stage = 0, *ws = 0, *d_off = 0, *d_src = 0, *d_dst = 0, *d_runs = 0, *d_n = 0;
    int64_t ws_bytes = 0;
    CHECK(kv_xfer_workspace_bytes(3, &ws_bytes));
    if (cudaMalloc(&src, NB * BLK) || cudaMalloc(&dst, NB * BLK) || cudaMalloc(&stage, 3 * BLK) ||
        cudaMalloc(&ws, (size_t)ws_bytes) || cudaMalloc(&d_off, sizeof offsets) || cudaMalloc(&d_src, sizeof src_ids) ||
        cudaMalloc(&d_dst, sizeof dst_ids) || cudaMalloc(&d_runs, 3 * sizeof(kv_xfer_run)) ||
        cudaMalloc(&d_n, sizeof(int32_t)))
        return 2;
    cudaMemcpy(src, host, sizeof host, cudaMemcpyHostToDevice);
    cudaMemset(dst, 0, NB * BLK);
    cudaMemcpy(d_off, offsets, sizeof offsets, cudaMemcpyHostToDevice);
    cudaMemcpy(d_src, src_ids, sizeof src_ids, cudaMemcpyHostToDevice);
    cudaMemcpy(d_dst, dst_ids, sizeof dst_ids, cudaMemcpyHostToDevice);

    uint64_t src_base[1] = {(uint64_t)(uintptr_t)src}, dst_base[1] = {(uint64_t)(uintptr_t)dst};
    kv_cache_desc sc = {1, BS, 1, ROW, NB, BLK, BLK, ROW, src_base};
    kv_cache_desc dc = {1, BS, 1, ROW, NB, BLK, BLK, ROW, dst_base};
    kv_stage_desc sd = {3, 1, 1, BS, ROW};

    /* two new tokens: request 0 position 5 (its second block, id 6, slot 1), request 1 position 2 */
    const int32_t table[4] = {5, 6, 1, -1};
    const int32_t tok_req[2] = {0, 1}, tok_pos[2] = {5, 2};
    uint8_t rows[2 * ROW];
    for (int i = 0; i < 2 * ROW; i++) rows[i] = (uint8_t)(200 + i);
    void *d_table = 0, *d_treq = 0, *d_tpos = 0, *d_slot = 0, *d_rows = 0;
    if (cudaMalloc(&d_table, sizeof table) || cudaMalloc(&d_treq, sizeof tok_req) || cudaMalloc(&d_tpos, sizeof tok_pos) ||
        cudaMalloc(&d_slot, 2 * sizeof(int64_t)) || cudaMalloc(&d_rows, sizeof rows))
        return 2;
    cudaMemcpy(d_table, table, sizeof table, cudaMemcpyHostToDevice);
    cudaMemcpy(d_treq, tok_req, sizeof tok_req, cudaMemcpyHostToDevice);
    cudaMemcpy(d_tpos, tok_pos, sizeof tok_pos, cudaMemcpyHostToDevice);
    cudaMemcpy(d_rows, rows, sizeof rows, cudaMemcpyHostToDevice);
    CHECK(kv_slot_mapping(d_table, 2, 2, 2, d_treq, d_tpos, 2, BS, d_slot, 0));
    const uint64_t new_kv[1] = {(uint64_t)(uintptr_t)d_rows};
    CHECK(kv_reshape_and_cache(&sc, new_kv, ROW, d_slot, 2, 0));
    int64_t slots[2] = {0, 0};
    cudaMemcpy(slots, d_slot, sizeof slots, cudaMemcpyDeviceToHost);
    if (slots[0] != 6 * BS + 1 || slots[1] != 1 * BS + 2) {
        fprintf(stderr, "slots %lld %lld\n", (long long)slots[0], (long long)slots[1]);
        return 6;
    }
    memcpy(host + slots[0] * ROW, rows, ROW); /* the host copy now holds the written rows too */
    memcpy(host + slots[1] * ROW, rows + ROW, ROW);

    CHECK(kv_build_xfer_list(d_off, 2, d_src, d_dst, 3, 2, d_runs, 3, d_n, ws, ws_bytes, 0));
    CHECK(kv_pack_blocks(&sc, 0, &sd, d_runs, d_n, 3, 2, stage, 3 * BLK, 0));
    CHECK(kv_unpack_blocks(&dc, 0, &sd, d_runs, d_n, 3, 2, stage, 3 * BLK, 0, 0, 0, 0, 0));
    int32_t err = -1, n_runs = -1;
    CHECK(kv_get_last_error(&err, 1, 0));
    cudaMemcpy(&n_runs, d_n, sizeof n_runs, cudaMemcpyDeviceToHost);
    cudaMemcpy(back, dst, sizeof back, cudaMemcpyDeviceToHost);
    if (err != 0 || n_runs != 2) { /* runs: (5,6)->(2,3) and 1->7 */
        fprintf(stderr, "err %d runs %d\n", err, n_runs);
        return 3;
    }
    for (int i = 0; i < 3; i++)
        if (memcmp(back + dst_ids[i] * BLK, host + src_ids[i] * BLK, BLK) != 0) return 4;
    for (int b = 0; b < NB; b++)
        if (b != 2 && b != 3 && b != 7)
            for (int k = 0; k < BLK; k++)
                if (back[b * BLK + k] != 0) return 5;

    /* prefix hashes: request 0 has 9 tokens (2 full blocks of 4), request 1 has 4 (1 block) */
    const int32_t h_off[3] = {0, 9, 13};
    int32_t h_tok[13];
    for (int i = 0; i < 13; i++) h_tok[i] = 1000 + 37 * i;
    void *d_hoff = 0, *d_htok = 0, *d_hout_off = 0, *d_h1 = 0, *d_h2 = 0, *d_hws = 0;
    int64_t hws_bytes = 0;
    CHECK(kv_block_hashes_workspace_bytes(13, BS, &hws_bytes));
    if (cudaMalloc(&d_hoff, sizeof h_off) || cudaMalloc(&d_htok, sizeof h_tok) || cudaMalloc(&d_hout_off, sizeof h_off) ||
        cudaMalloc(&d_h1, 3 * sizeof(uint64_t)) || cudaMalloc(&d_h2, 3 * sizeof(uint64_t)) ||
        cudaMalloc(&d_hws, (size_t)hws_bytes))
        return 2;
    cudaMemcpy(d_hoff, h_off, sizeof h_off, cudaMemcpyHostToDevice);
    cudaMemcpy(d_htok, h_tok, sizeof h_tok, cudaMemcpyHostToDevice);
    CHECK(kv_block_hashes(d_hoff, 2, d_htok, 13, BS, 81, d_hout_off, d_h1, 3, d_hws, hws_bytes, 0));
    CHECK(kv_block_hashes(d_hoff, 2, d_htok, 13, BS, 81, d_hout_off, d_h2, 3, 0, 0, 0));
    uint64_t h1[3], h2[3];
    int32_t hout_off[3];
    cudaMemcpy(h1, d_h1, sizeof h1, cudaMemcpyDeviceToHost);
    cudaMemcpy(h2, d_h2, sizeof h2, cudaMemcpyDeviceToHost);
    cudaMemcpy(hout_off, d_hout_off, sizeof hout_off, cudaMemcpyDeviceToHost);
    if (hout_off[0] != 0 || hout_off[1] != 2 || hout_off[2] != 3 || memcmp(h1, h2, sizeof h1) != 0) return 7;
    /* FNV-1a 64 over the seed's 8 little-endian bytes, then the block's 4 tokens' 4 bytes each */
    uint64_t h = 0xcbf29ce484222325ull;
    for (int k = 0; k < 8; k++) h = (h ^ ((81ull >> (8 * k)) & 0xffu)) * 0x100000001b3ull;
    for (int t = 0; t < BS; t++)
        for (int k = 0; k < 4; k++) h = (h ^ (((uint32_t)h_tok[t] >> (8 * k)) & 0xffu)) * 0x100000001b3ull;
    if (h1[0] != h) return 8;
    CHECK(kv_get_last_error(&err, 1, 0));
    if (err != 0) return 9;
    printf("c abi ok: %s\n", kv_version());
    return 0;
}
