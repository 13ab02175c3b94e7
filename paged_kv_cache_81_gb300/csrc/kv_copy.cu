// kv_pack_blocks / kv_unpack_blocks: the gather into, and scatter out of, the staging buffer.
//
// Gather semantics: page "0. vllm 如何使用 nccl 传输 kv cache", section 2.4
// (extract_kv_from_layer: layer[block_ids] / layer[:, block_ids]); scatter semantics: the
// same page, section 2.3 step 14 (kv_cache_layer[block_ids] = tensor); per-layer,
// per-block addressing with a head slice for TP heterogeneity: page "vLLM PD 分离 源码级
// 机制", section 4.2 (_build_transfer_params).
//
// Work decomposition: an item is one piece (at most kPieceChunks 16-byte chunks) of one
// (tensor, run).  Items are numbered piece-major, then tensor, then run, so consecutive warps
// write adjacent staging ranges and no warp keeps drawing empty pieces.  The grid has two parts:
//  - `resident` persistent CTAs (every CTA the SMs hold at once) walk the first 7/8 of the
//    items with a warp stride, so the warps in flight work on one dense window of items;
//  - tail CTAs, queued behind them, take the last 1/8 in chunks of kTailItemsPerWarp items per
//    warp; the block scheduler places each on whichever SM frees up first.
// Some SMs scatter rows measurably slower than others (on GB300 four groups of about ten SMs
// took ~10% longer over the same static share of an unpack), so a purely static split waits for
// them; the tail lets the faster SMs finish the work instead.  An eighth for the tail and a
// quarter measured the same on the page-shaped, kv-first and asymmetric presets; with no tail
// and purely hardware-scheduled CTAs (each a contiguous range of items) unpack ran as fast but
// pack of whole 8 KiB blocks lost 3%, its staging writes spread over many small ranges.  A copy
// with fewer than kTailMinItemsPerWarp items per warp has no tail.  Inside a CTA the warps draw their
// items from a shared-memory ticket, so a warp that is ahead takes the next item of its CTA.
// Inside a piece each lane keeps kUnroll 16-byte loads in flight before storing them.
//
// Address modes of the cache side (the staging side is always linear):
//   MERGED  a run is one contiguous span (dense blocks, block_stride == staged block bytes)
//   SPANS   each (block, plane) is contiguous; blocks and planes are strided (kv-first layers)
//   ROWS    row by row: a head slice or a strided token dimension
//   REMAP   unpack onto another block size / another block list (token granular)
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kv_copy.cuh"

namespace {

using pkv::CopyParams;
using pkv::FastDiv;
using pkv::MERGED;
using pkv::SPANS;
using pkv::ROWS;
using pkv::REMAP;

#ifndef PKV_COPY_UNROLL
#define PKV_COPY_UNROLL 8  // 16-byte loads each lane keeps in flight
#endif
#ifndef PKV_COPY_MIN_CTAS
#define PKV_COPY_MIN_CTAS 1  // launch-bounds hint: resident CTAs per SM the register budget must allow
#endif
#ifndef PKV_ROWS_MIN_CTAS
#define PKV_ROWS_MIN_CTAS 1  // the same hint for the ROWS and REMAP modes (more index arithmetic per chunk)
#endif
#ifndef PKV_COPY_TAIL_DIV
#define PKV_COPY_TAIL_DIV 8  // 1 / (the share of the items left to the tail CTAs)
#endif
#ifndef PKV_COPY_TAIL_ITEMS
#define PKV_COPY_TAIL_ITEMS 2  // items per warp of one tail CTA
#endif

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = PKV_COPY_UNROLL;
constexpr uint32_t kPieceChunks = 1024;  // 16 KiB
constexpr int64_t kTailDiv = PKV_COPY_TAIL_DIV;  // the tail CTAs take items / kTailDiv of the items
constexpr int kTailItemsPerWarp = PKV_COPY_TAIL_ITEMS;  // a tail CTA's chunk: kWarps * this many items
constexpr int kMaxTailCtasPerResident = 8;       // more tail chunks than this are strided over
// A copy of fewer than this many items per warp of the persistent part has no tail: its time is
// launch and latency, and a second round of CTAs would only add to it.
constexpr int64_t kTailMinItemsPerWarp = 8;

template <int MODE, bool PACK>
__global__ void __launch_bounds__(kThreads, MODE >= pkv::ROWS ? PKV_ROWS_MIN_CTAS : PKV_COPY_MIN_CTAS)
    copy_runs_kernel(const __grid_constant__ CopyParams p)
{
    pkv::grid_dep_entry();  // before any global memory access
    const int lane = threadIdx.x & 31;
    const unsigned wib = threadIdx.x >> 5;  // warp in the CTA
    __shared__ unsigned s_ticket;           // the CTA's next item ticket
    if (threadIdx.x == 0) s_ticket = kWarps;  // tickets 0 .. kWarps-1 are the warps' first items
    __syncthreads();
    int64_t nr = *p.n_runs;
    if (nr > p.run_capacity) {
        if (blockIdx.x == 0 && threadIdx.x == 0) pkv::set_error(p.err, KV_DERR_CAPACITY);
        nr = p.run_capacity;
    }
    if (nr < 0) nr = 0;
    // Items are numbered piece-major: (piece, tensor, run).  Every run has a piece 0, so the
    // first n_tensors * nr items are all non-empty and spread evenly over the warps.
    const int64_t per_piece = nr * p.n_tensors;
    const int64_t items = per_piece * p.max_pieces;

    // Ticket i of this CTA -> item.  Persistent CTA b: round i / kWarps of the warp-stride walk
    // over [0, n_static), slot b * kWarps + i % kWarps.  Tail CTA b (b >= resident): item i %
    // chunk of chunk (b - resident) + (i / chunk) * n_tail_ctas of [n_static, items).  Both are
    // increasing in i, so the first item past the end ends the warp's walk.
    const int64_t quantum = (int64_t)kWarps * p.resident;
    const int64_t n_static = p.tail_div > 0 ? (items - items / p.tail_div) / quantum * quantum : items;
    const bool tail = (int64_t)blockIdx.x >= p.resident;
    const int64_t chunk = (int64_t)kWarps * kTailItemsPerWarp;
    const int64_t n_tail_ctas = (int64_t)gridDim.x - p.resident;
    const int64_t slot = tail ? (int64_t)blockIdx.x - p.resident : (int64_t)blockIdx.x * kWarps;
    const int64_t item_end = tail ? items : n_static;
    auto item_of = [&](unsigned i) -> int64_t {
        if (tail) return n_static + ((int64_t)(i / chunk) * n_tail_ctas + slot) * chunk + i % chunk;
        return (int64_t)(i / kWarps) * quantum + slot + i % kWarps;
    };
    auto next_ticket = [&]() -> unsigned {
        unsigned t = 0;
        if (lane == 0) t = atomicAdd(&s_ticket, 1u);
        return __shfl_sync(0xffffffffu, t, 0);
    };

    int64_t item = item_of(wib);
    kv_xfer_run next;
    if (item < item_end) next = p.runs[item % per_piece % nr];
    while (item < item_end) {
        const int64_t cur = item;
        const kv_xfer_run run = next;
        item = item_of(next_ticket());
        if (item < item_end) next = p.runs[item % per_piece % nr];  // prefetch: overlaps the copy below
        const int32_t piece = (int32_t)(cur / per_piece);
        const int64_t rest = cur - (int64_t)piece * per_piece;
        const int32_t t = (int32_t)(rest / nr);

        const uint64_t item_chunks64 = (uint64_t)(int64_t)run.n_blocks * p.chunks_per_block;
        const uint64_t c_begin = (uint64_t)piece * kPieceChunks;
        if (run.n_blocks <= 0 || c_begin >= item_chunks64) continue;
        const bool first_piece = piece == 0;
        if (run.stage_block < 0 || run.stage_block + run.n_blocks > p.n_stage_blocks ||
            item_chunks64 >= (1ull << 32)) {
            if (first_piece && lane == 0) pkv::set_error(p.err, KV_DERR_STAGE);
            continue;
        }
        const uint32_t item_chunks = (uint32_t)item_chunks64;
        const uint32_t c_end =
            piece == p.max_pieces - 1 ? item_chunks : (uint32_t)std::min<uint64_t>(c_begin + kPieceChunks, item_chunks);

        int64_t blk = 0;  // first cache block of the run (MERGED / SPANS / ROWS)
        int32_t j0 = 0, dn = 0;  // REMAP: first staged token of the run in its request; dst list length
        const int32_t *dl = nullptr;
        if (MODE == REMAP) {
            const int32_t r = run.req;
            if (r < 0 || r >= p.n_reqs) {
                if (first_piece && lane == 0) pkv::set_error(p.err, KV_DERR_DST_TABLE);
                continue;
            }
            const int32_t s0 = p.src_req_offsets[r];
            const int32_t d0 = p.dst_req_offsets[r];
            dn = (int32_t)max((int64_t)-1, min((int64_t)INT32_MAX, (int64_t)p.dst_req_offsets[r + 1] - d0));
            if (run.stage_block < s0 || dn < 0 || d0 < 0) {  // offsets that do not match the runs
                if (first_piece && lane == 0) pkv::set_error(p.err, KV_DERR_DST_TABLE);
                continue;
            }
            j0 = (int32_t)((run.stage_block - s0) * (int64_t)p.div_bs.d);
            dl = p.dst_ids + d0;
        } else {
            blk = PACK ? run.src_block : run.dst_block;
            if (blk < 0 || blk + run.n_blocks > p.num_blocks) {
                if (first_piece && lane == 0) pkv::set_error(p.err, KV_DERR_BLOCK);
                continue;
            }
        }

        uint8_t *const cache_t = reinterpret_cast<uint8_t *>(p.base[t]);
        uint8_t *const stage_item = p.stage + (int64_t)(p.tensor_begin + t) * p.stage_tensor_bytes +
                                    run.stage_block * p.stage_block_bytes;

        for (uint32_t c0 = (uint32_t)c_begin + lane; c0 < c_end; c0 += 32 * kUnroll) {
            uint4 v[kUnroll];
            uint8_t *dst[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; u++) {
                dst[u] = nullptr;
                const uint32_t c = c0 + 32u * u;
                if (c >= c_end) continue;
                uint8_t *cache_addr;
                if (MODE == MERGED) {
                    cache_addr = cache_t + blk * p.block_stride + (int64_t)c * 16;
                } else if (MODE == SPANS) {
                    const uint32_t m = pkv::fdiv(c, p.div_cpb);
                    const uint32_t w = c - m * p.div_cpb.d;
                    const uint32_t plane = pkv::fdiv(w, p.div_cps);
                    const uint32_t o = w - plane * p.div_cps.d;
                    cache_addr = cache_t + (blk + m) * p.block_stride + (int64_t)plane * p.plane_stride +
                                 (int64_t)o * 16;
                } else {
                    const uint32_t row = pkv::fdiv(c, p.div_cpr);
                    const uint32_t q = c - row * p.div_cpr.d;
                    const uint32_t m = pkv::fdiv(row, p.div_rpb);
                    const uint32_t rr = row - m * p.div_rpb.d;
                    const uint32_t plane = pkv::fdiv(rr, p.div_bs);
                    const uint32_t o = rr - plane * p.div_bs.d;
                    if (MODE == ROWS) {
                        cache_addr = cache_t + (blk + m) * p.block_stride + (int64_t)plane * p.plane_stride +
                                     (int64_t)o * p.token_stride + p.row_off + (int64_t)q * 16;
                    } else {  // REMAP: staged token j of the request -> destination slot
                        const uint32_t j = (uint32_t)j0 + m * p.div_bs.d + o;
                        const uint32_t dq = pkv::fdiv(j, p.div_dbs);
                        if (dq >= (uint32_t)dn) {
                            pkv::set_error(p.err, KV_DERR_DST_TABLE);
                            continue;
                        }
                        const int32_t db = dl[dq];
                        if (db < 0 || db >= p.num_blocks) {
                            pkv::set_error(p.err, KV_DERR_BLOCK);
                            continue;
                        }
                        const uint32_t doff = j - dq * p.div_dbs.d;
                        cache_addr = cache_t + (int64_t)db * p.block_stride + (int64_t)plane * p.plane_stride +
                                     (int64_t)doff * p.token_stride + p.row_off + (int64_t)q * 16;
                    }
                }
                uint8_t *stage_addr = stage_item + (int64_t)c * 16;
                if (PACK) {
                    v[u] = pkv::ld_once(cache_addr);
                    dst[u] = stage_addr;
                } else {
                    v[u] = pkv::ld_once(stage_addr);
                    dst[u] = cache_addr;
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; u++)
                if (dst[u] != nullptr) pkv::st_stream(dst[u], v[u]);
        }
    }
    pkv::signal_on_exit(p);
}

using KernelFn = void (*)(CopyParams);

KernelFn pick(int mode, bool pack)
{
    switch (mode * 2 + (pack ? 1 : 0)) {
    case MERGED * 2 + 1: return copy_runs_kernel<MERGED, true>;
    case MERGED * 2: return copy_runs_kernel<MERGED, false>;
    case SPANS * 2 + 1: return copy_runs_kernel<SPANS, true>;
    case SPANS * 2: return copy_runs_kernel<SPANS, false>;
    case ROWS * 2 + 1: return copy_runs_kernel<ROWS, true>;
    case ROWS * 2: return copy_runs_kernel<ROWS, false>;
    default: return copy_runs_kernel<REMAP, false>;
    }
}

// Resident CTAs per SM of each kernel variant, per device (computed once).
int resident_ctas(int device, int mode, bool pack)
{
    static std::mutex mu;
    static int cache[64][4][2];
    std::lock_guard<std::mutex> lock(mu);
    int &slot = cache[device & 63][mode][pack ? 1 : 0];
    if (slot == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, pick(mode, pack), kThreads, 0) != cudaSuccess || n <= 0)
            n = 1;
        slot = n;
    }
    return slot;
}

// Copy engine for contiguous spans (whole runs, or one span per (block, plane)).  With both
// engines on the persistent-plus-tail work split, the TMA bulk-copy engine (kv_bulk.cu) moves
// spans of 4 KiB and more faster than the register-staged warp engine above (GB/s, pack /
// unpack, full presets: 8 KiB blocks 6836 / 6854 against 6564 / 6788; kv-first 4 KiB planes
// 6823 / 6835 against 6737 / 6761; 32 KiB blocks 6933 / 6929).  Smaller spans keep the warp
// engine.  PAGEDKV_COPY_ENGINE=lsu|bulk (read once) forces one engine for measurements.
bool bulk_engine(int64_t block_bytes)
{
    static const int forced = [] {
        const char *e = std::getenv("PAGEDKV_COPY_ENGINE");
        if (e == nullptr) return 0;
        if (std::strcmp(e, "bulk") == 0) return 1;
        if (std::strcmp(e, "lsu") == 0) return 2;
        return 0;
    }();
    if (forced) return forced == 1;
    return block_bytes >= 4 * 1024;
}

// The staging buffer may be device memory or pinned host memory (cudaHostAlloc /
// cudaHostRegister), the spill target of a receiver whose device memory is short.  Host
// memory is addressed through its device mapping; unregistered host memory is refused.
int staging_address(uint8_t *buf, uint8_t **dev_addr, bool *is_host)
{
    *is_host = false;
    *dev_addr = buf;
    if (buf == nullptr) return KV_OK;
    cudaPointerAttributes a{};
    const cudaError_t e = cudaPointerGetAttributes(&a, buf);
    if (e != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of an unknown pointer
        return KV_ERR_INVALID_ARG;
    }
    if (a.type == cudaMemoryTypeUnregistered) return KV_ERR_INVALID_ARG;
    if (a.type == cudaMemoryTypeHost) {
        if (a.devicePointer == nullptr) return KV_ERR_INVALID_ARG;
        *is_host = true;
        *dev_addr = static_cast<uint8_t *>(a.devicePointer);
    }
    return KV_OK;
}

// Address mode of the cache side: MERGED when a run of blocks is one span, SPANS when every
// (block, plane) is a span of block_size whole rows, ROWS otherwise.
int cache_mode(const kv_cache_desc *c, int32_t row_off, int32_t slice)
{
    if (row_off != 0 || slice != c->row_bytes || c->token_stride != c->row_bytes) return ROWS;
    const int64_t span = (int64_t)c->block_size * c->row_bytes;
    const bool dense_block = c->n_planes == 1 || c->plane_stride == span;
    return dense_block && c->block_stride == c->n_planes * span ? MERGED : SPANS;
}

int launch(const kv_cache_desc *cache, const kv_stage_desc *stage, int mode, bool pack, int32_t row_off,
           const kv_xfer_run *runs, const int32_t *n_runs, int64_t run_capacity, uint8_t *stage_buf,
           int32_t max_run_blocks, int32_t dst_block_size, const int32_t *src_req_offsets,
           const int32_t *dst_req_offsets, const int32_t *dst_ids, int32_t n_reqs, kv_signal *signal,
           uint64_t signal_add, cudaStream_t s)
{
    const pkv::DeviceInfo *dev = pkv::current_device();
    if (dev == nullptr) return KV_ERR_CUDA;
    const int64_t stage_block_bytes = (int64_t)stage->n_planes * stage->block_size * stage->slice_bytes;
    const int64_t cpb = stage_block_bytes / 16;
    if (cpb >= (1ll << 31)) return KV_ERR_UNSUPPORTED;
    bool host_stage = false;
    int st = staging_address(stage_buf, &stage_buf, &host_stage);
    if (st != KV_OK) return st;

    CopyParams p{};
    p.runs = runs;
    p.n_runs = n_runs;
    p.run_capacity = run_capacity;
    p.stage = stage_buf;
    p.stage_block_bytes = stage_block_bytes;
    p.stage_tensor_bytes = stage->n_blocks * stage_block_bytes;
    p.n_stage_blocks = stage->n_blocks;
    p.num_blocks = cache->num_blocks;
    p.block_stride = cache->block_stride;
    p.plane_stride = cache->plane_stride;
    p.token_stride = cache->token_stride;
    p.row_off = row_off;
    p.chunks_per_block = (uint32_t)cpb;
    p.div_cpr = pkv::make_fastdiv((uint32_t)(stage->slice_bytes / 16));
    p.div_bs = pkv::make_fastdiv((uint32_t)stage->block_size);
    p.div_rpb = pkv::make_fastdiv((uint32_t)(stage->n_planes * stage->block_size));
    p.div_cpb = pkv::make_fastdiv((uint32_t)cpb);
    p.div_cps = pkv::make_fastdiv((uint32_t)(cpb / stage->n_planes));
    p.div_dbs = pkv::make_fastdiv((uint32_t)std::max(1, dst_block_size));
    p.src_req_offsets = src_req_offsets;
    p.dst_req_offsets = dst_req_offsets;
    p.dst_ids = dst_ids;
    p.n_reqs = n_reqs;
    p.err = dev->err_word;
    const int64_t run_chunks = (int64_t)std::max(1, max_run_blocks) * cpb;
    p.max_pieces = max_run_blocks > 0 ? (int32_t)std::min<int64_t>((run_chunks + kPieceChunks - 1) / kPieceChunks, 1 << 20) : 1;

    // staging in host memory goes over the host link with the warp engine's 16-byte accesses
    const int64_t piece = mode == MERGED ? stage_block_bytes : stage_block_bytes / stage->n_planes;
    // a remap whose staged blocks land whole inside destination blocks, on rows the slice fills,
    // is one span per staged (block, plane)
    const bool remap_spans = mode == REMAP && row_off == 0 && cache->row_bytes == stage->slice_bytes &&
                             cache->token_stride == stage->slice_bytes && dst_block_size % stage->block_size == 0;
    const bool bulk = !host_stage && (mode == MERGED || mode == SPANS || remap_spans) && bulk_engine(piece);
    const KernelFn fn = pick(mode, pack);
    int grid = 0;
    bool with_tail = false;
    if (!bulk) {
        // persistent CTAs, plus enough tail CTAs for the largest tail the device-side run count
        // allows (a tail CTA whose chunk lies past the items exits at once)
        p.resident = dev->num_sms * resident_ctas(dev->device, mode, pack);
        const int64_t items_max = (int64_t)std::min<int64_t>(run_capacity, stage->n_blocks) * p.max_pieces *
                                  std::min(pkv::kMaxTensorsPerLaunch, cache->n_tensors);
        const int64_t quantum = (int64_t)kWarps * p.resident;
        const int64_t chunk = (int64_t)kWarps * kTailItemsPerWarp;
        with_tail = kTailDiv > 0 && items_max >= kTailMinItemsPerWarp * quantum;
        p.tail_div = with_tail ? (int32_t)kTailDiv : 0;
        const int64_t tail_ctas = (items_max / std::max<int64_t>(1, kTailDiv) + quantum + chunk - 1) / chunk;
        grid = p.resident + (with_tail ? (int)std::max<int64_t>(1, std::min<int64_t>(tail_ctas, (int64_t)kMaxTailCtasPerResident * p.resident)) : 0);
    }
    for (int32_t t0 = 0; t0 < cache->n_tensors; t0 += pkv::kMaxTensorsPerLaunch) {
        const int32_t nt = std::min(pkv::kMaxTensorsPerLaunch, cache->n_tensors - t0);
        p.n_tensors = nt;
        p.tensor_begin = t0;
        const bool last = t0 + pkv::kMaxTensorsPerLaunch >= cache->n_tensors;
        p.signal = last ? signal : nullptr;
        p.signal_add = signal_add;
        for (int32_t t = 0; t < nt; t++) p.base[t] = cache->base[t0 + t];
        if (bulk) {
            st = pkv::launch_bulk_copy(p, mode, pack, *dev, s);
        } else {
            pkv::launch_as(!with_tail, fn, grid, kThreads, 0, s, p);  // tail CTAs: a plain launch
            st = pkv::cuda_status(cudaGetLastError());
        }
        if (st != KV_OK) return st;
    }
    return KV_OK;
}

int check_stage(const kv_stage_desc *stage, const void *buf, int64_t stage_bytes)
{
    if (stage == nullptr || stage->n_blocks < 0 || stage->n_tensors < 0 || stage->block_size <= 0 ||
        (stage->n_planes != 1 && stage->n_planes != 2) || stage->slice_bytes <= 0 || stage_bytes < 0)
        return KV_ERR_INVALID_ARG;
    if (!pkv::aligned16((int64_t)stage->slice_bytes)) return KV_ERR_ALIGN;
    int64_t need = stage->n_blocks;  // staged bytes; a size past int64 is refused, not wrapped
    const int64_t factors[4] = {stage->n_tensors, stage->n_planes, stage->block_size, stage->slice_bytes};
    for (const int64_t f : factors)
        if (__builtin_mul_overflow(need, f, &need)) return KV_ERR_RANGE;
    if (need > 0 && buf == nullptr) return KV_ERR_INVALID_ARG;
    if (!pkv::aligned16(buf)) return KV_ERR_ALIGN;
    if (stage_bytes < need) return KV_ERR_RANGE;
    return KV_OK;
}

}  // namespace

int pkv::preload_copy_kernels()
{
    return pkv::load_kernels(copy_runs_kernel<MERGED, true>, copy_runs_kernel<MERGED, false>,
                             copy_runs_kernel<SPANS, true>, copy_runs_kernel<SPANS, false>, copy_runs_kernel<ROWS, true>,
                             copy_runs_kernel<ROWS, false>, copy_runs_kernel<REMAP, false>);
}

extern "C" {

int kv_pack_blocks(const kv_cache_desc *src, int32_t src_slice_off, const kv_stage_desc *stage,
                      const kv_xfer_run *runs, const int32_t *n_runs, int64_t run_capacity,
                      int32_t max_run_blocks, void *stage_buf, int64_t stage_bytes, kv_stream_t stream)
{
    int st = pkv::check_cache(src);
    if (st != KV_OK) return st;
    st = check_stage(stage, stage_buf, stage_bytes);
    if (st != KV_OK) return st;
    if (stage->n_tensors != src->n_tensors || stage->n_planes != src->n_planes ||
        stage->block_size != src->block_size || run_capacity < 0 || max_run_blocks < 0)
        return KV_ERR_INVALID_ARG;
    if (src_slice_off < 0 || src_slice_off + (int64_t)stage->slice_bytes > src->row_bytes) return KV_ERR_RANGE;
    if (!pkv::aligned16((int64_t)src_slice_off)) return KV_ERR_ALIGN;
    if (src->n_tensors == 0 || stage->n_blocks == 0 || run_capacity == 0) return KV_OK;
    if (runs == nullptr || n_runs == nullptr) return KV_ERR_INVALID_ARG;
    const int mode = cache_mode(src, src_slice_off, stage->slice_bytes);
    return launch(src, stage, mode, true, src_slice_off, runs, n_runs, run_capacity, (uint8_t *)stage_buf,
                  max_run_blocks, 0, nullptr, nullptr, nullptr, 0, nullptr, 0, (cudaStream_t)stream);
}

int kv_unpack_blocks_signal(const kv_cache_desc *dst, int32_t dst_slice_off, const kv_stage_desc *stage,
                        const kv_xfer_run *runs, const int32_t *n_runs, int64_t run_capacity,
                        int32_t max_run_blocks, const void *stage_buf, int64_t stage_bytes,
                        const int32_t *src_req_offsets, const int32_t *dst_req_offsets,
                        const int32_t *dst_ids, int32_t n_reqs, kv_signal *signal, uint64_t add,
                        kv_stream_t stream)
{
    if (signal != nullptr && ((uintptr_t)signal & 15u) != 0) return KV_ERR_ALIGN;
    int st = pkv::check_cache(dst);
    if (st != KV_OK) return st;
    st = check_stage(stage, stage_buf, stage_bytes);
    if (st != KV_OK) return st;
    if (stage->n_tensors != dst->n_tensors || stage->n_planes != dst->n_planes || run_capacity < 0 ||
        max_run_blocks < 0)
        return KV_ERR_INVALID_ARG;
    if (dst_slice_off < 0 || dst_slice_off + (int64_t)stage->slice_bytes > dst->row_bytes) return KV_ERR_RANGE;
    if (!pkv::aligned16((int64_t)dst_slice_off)) return KV_ERR_ALIGN;
    // Nothing staged: nothing to copy in either mode.  (An empty destination list may then
    // arrive as a null dst_ids, which would otherwise read as whole-block mode.)
    if (dst->n_tensors == 0 || stage->n_blocks == 0 || run_capacity == 0)
        return signal != nullptr ? pkv::post_signal(signal, add, (cudaStream_t)stream) : KV_OK;
    const bool remap = dst_ids != nullptr;
    if (remap && (src_req_offsets == nullptr || dst_req_offsets == nullptr || n_reqs < 0))
        return KV_ERR_INVALID_ARG;
    if (!remap && stage->block_size != dst->block_size) return KV_ERR_INVALID_ARG;
    if (runs == nullptr || n_runs == nullptr) return KV_ERR_INVALID_ARG;
    int mode = REMAP;
    if (!remap) mode = cache_mode(dst, dst_slice_off, stage->slice_bytes);
    return launch(dst, stage, mode, false, dst_slice_off, runs, n_runs, run_capacity,
                  (uint8_t *)const_cast<void *>(stage_buf), max_run_blocks, dst->block_size, src_req_offsets,
                  dst_req_offsets, dst_ids, n_reqs, signal, add, (cudaStream_t)stream);
}

int kv_unpack_blocks(const kv_cache_desc *dst, int32_t dst_slice_off, const kv_stage_desc *stage,
                     const kv_xfer_run *runs, const int32_t *n_runs, int64_t run_capacity,
                     int32_t max_run_blocks, const void *stage_buf, int64_t stage_bytes,
                     const int32_t *src_req_offsets, const int32_t *dst_req_offsets,
                     const int32_t *dst_ids, int32_t n_reqs, kv_stream_t stream)
{
    return kv_unpack_blocks_signal(dst, dst_slice_off, stage, runs, n_runs, run_capacity, max_run_blocks, stage_buf,
                                   stage_bytes, src_req_offsets, dst_req_offsets, dst_ids, n_reqs, nullptr, 0, stream);
}

}  // extern "C"
