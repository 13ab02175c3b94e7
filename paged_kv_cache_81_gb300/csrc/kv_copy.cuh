// Shared between the copy engines of kv_pack_blocks / kv_unpack_blocks (not part of the ABI).
#pragma once

#include "kv_common.cuh"

namespace pkv {

// Cache-side address modes of a copy (the staging side is always linear):
//   MERGED  a run of blocks is one contiguous span
//   SPANS   every (block, plane) is a contiguous span of block_size rows; blocks and planes are
//           strided (kv-first layers, padded blocks)
//   ROWS    row by row: a head slice or a strided token dimension
//   REMAP   unpack onto another block size / another block list (token granular)
enum CopyMode { MERGED = 0, SPANS = 1, ROWS = 2, REMAP = 3 };

struct CopyParams {
    const kv_xfer_run *runs;
    const int32_t *n_runs;
    int64_t run_capacity;
    uint8_t *stage;
    int64_t stage_tensor_bytes;  // n_stage_blocks * stage_block_bytes
    int64_t stage_block_bytes;   // planes * bs * slice
    int64_t n_stage_blocks;
    int64_t num_blocks;  // cache blocks per tensor
    int64_t block_stride;
    int64_t plane_stride;
    int64_t token_stride;
    int32_t row_off;  // byte offset of the slice inside a cache row
    int32_t n_tensors;
    int32_t tensor_begin;
    int32_t max_pieces;
    int32_t resident;           // CTAs of the grid's persistent part
    int32_t tail_div;           // the grid's tail CTAs take items / tail_div of the items (0: no tail)
    uint32_t chunks_per_block;  // staged block / 16
    FastDiv div_cpr;            // chunks per staged row
    FastDiv div_bs;             // staged (source) block size
    FastDiv div_rpb;            // staged rows per block = planes * bs
    FastDiv div_cpb;            // chunks per staged block
    FastDiv div_cps;            // chunks per (block, plane) span = bs * slice / 16
    FastDiv div_dbs;            // destination block size (REMAP)
    const int32_t *src_req_offsets;
    const int32_t *dst_req_offsets;
    const int32_t *dst_ids;
    int32_t n_reqs;
    int *err;
    kv_signal *signal;    // when set: the last CTA to finish adds signal_add to signal->value
    uint64_t signal_add;
    uint64_t base[kMaxTensorsPerLaunch];
};

// End of a copy kernel when a completion signal is requested (every thread of the CTA calls
// it after its last copy): the CTA's writes are fenced, the CTA is counted on
// signal->arrived, and the last CTA of the grid resets the count and publishes
// signal->value += add with release semantics.
__device__ __forceinline__ void signal_on_exit(const CopyParams &p)
{
    if (p.signal == nullptr) return;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned prev = atomicAdd(&p.signal->arrived, 1u);
        if (prev == gridDim.x - 1) {
            p.signal->arrived = 0;
            __threadfence();
            asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(&p.signal->value), "l"(p.signal_add)
                         : "memory");
        }
    }
}

// Launches the TMA bulk-copy engine for a MERGED or SPANS copy (kv_bulk.cu).
int launch_bulk_copy(const CopyParams &p, int mode, bool pack, const DeviceInfo &dev, cudaStream_t s);

}  // namespace pkv
