/* A plain C11 caller of libpagedkv.so: the header alone is enough to drive the path.
 * It builds a tiny cache, lists two requests' blocks, builds the xfer_list, packs into a
 * staging buffer, unpacks into a second cache at other block ids, and checks the bytes. */
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
    printf("c abi ok: %s\n", kv_version());
    return 0;
}
