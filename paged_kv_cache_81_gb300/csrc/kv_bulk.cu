// TMA bulk-copy engine for kv_pack_blocks / kv_unpack_blocks when the cache side is made of
// contiguous spans: whole runs (MERGED), one span per (block, plane) (SPANS), or, for an unpack
// onto a block size that is a multiple of the staged one, one span per staged (block, plane) at
// its destination block's rows (REMAP).
//
// Each run of the xfer_list (page "5. flagcx connector design & dev & test", section 1.2:
// one transfer per contiguous group) becomes one or more bulk copies of at most kStage
// bytes: global -> shared memory with cp.async.bulk (completion counted on an mbarrier),
// then shared memory -> global with cp.async.bulk (bulk-group completion).  The copy
// itself is done by the SM's TMA unit; no register ever holds payload.
//
// Work split as in the warp engine (kv_copy.cu): the persistent CTAs (one per SM) walk the first
// items - items / kTailDiv items with a pipe stride; tail CTAs queued behind them take the rest in
// chunks of kTailItemsPerPipe items per pipe, each placed on whichever SM frees up first, so SMs
// that copy more slowly than others do not hold up the end of the launch.  Whole runs of 32-72 KiB
// are coarser items than the warp engine's, and a third left to the tail measured best here
// (Mid pack / unpack and MLA pack, GB/s: an eighth 6535 / 6521 and 6785; a quarter 6580 / 6631
// and 6970, with some launches as slow as with an eighth; a third 6923 / 6917 and 6968; a half
// 6915 / 6908 and 6955).  Copies with fewer than kTailMinItemsPerPipe items per pipe have no tail.
//
// One issuing lane per warp ("pipe") owns a ring of kSlots shared-memory slots.  A pipe
// keeps up to kSlots - 1 loads in flight: before it loads into a slot it stores the oldest
// loaded slot, then waits until all but the newest store have finished reading shared
// memory, which frees the slot the new load takes.  The other lanes of the warp fetch the
// next 32 run records while the issuing lane works through the current 32.
// Every mbarrier wait is bounded (2 s of globaltimer); a timeout sets KV_DERR_TIMEOUT,
// stops issuing, waits (bounded again) for the loads in flight and returns.
#include <algorithm>
#include <mutex>

#include "kv_async.cuh"
#include "kv_copy.cuh"

#ifndef PKV_BULK_STAGE_BYTES
#define PKV_BULK_STAGE_BYTES 8192
#endif
#ifndef PKV_BULK_SLOTS
#define PKV_BULK_SLOTS 3
#endif
#ifndef PKV_BULK_PIPES
#define PKV_BULK_PIPES 8
#endif
#ifndef PKV_BULK_TAIL_ITEMS
#define PKV_BULK_TAIL_ITEMS 2  // items per pipe of one tail CTA
#endif
#ifndef PKV_BULK_TAIL_DIV
#define PKV_BULK_TAIL_DIV 3  // 1 / (the share of the items left to the tail CTAs); 0: no tail CTAs
#endif

namespace {

using pkv::CopyParams;

constexpr uint32_t kStage = PKV_BULK_STAGE_BYTES;  // bytes per slot (multiple of 16)
constexpr int kSlots = PKV_BULK_SLOTS;
constexpr int kPipes = PKV_BULK_PIPES;  // warps (pipes) per CTA
constexpr int kBatch = 32;             // run records fetched per warp round
constexpr int64_t kTailDiv = PKV_BULK_TAIL_DIV;
constexpr int kTailItemsPerPipe = PKV_BULK_TAIL_ITEMS;
constexpr int kMaxTailCtasPerResident = 8;  // more tail chunks than this are strided over
constexpr int64_t kTailMinItemsPerPipe = 8;  // fewer items per pipe: no tail (latency-bound copies)
static_assert(kStage % 16 == 0 && kSlots >= 3, "bulk engine shape");

struct PipeState {  // per pipe, in shared memory after the slot data
    uint64_t bar[kSlots];
    uint64_t dst[kSlots];
    uint32_t bytes[kSlots];
    kv_xfer_run rec[kBatch];
};

constexpr size_t kSmemBytes = (size_t)kPipes * kSlots * kStage + (size_t)kPipes * sizeof(PipeState);

using pkv::mbar_arrive_expect_tx;
using pkv::mbar_init;
using pkv::mbar_wait;
using pkv::smem_addr;

#ifndef PKV_BULK_EVICT_FIRST
#define PKV_BULK_EVICT_FIRST 0  // L2 evict-first policy on: 0 none, 1 all bulk copies, 2 unpack's stores, 3 all stores, 4 all loads
#endif

// L2 policy for data read or written once: evict first (what st.global.cs asks for on the
// warp engine's stores), so a copy's lines do not displace the next kernel's.
__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_load(uint32_t dst_smem, const void *src, uint32_t bytes, uint32_t bar)
{
#if PKV_BULK_EVICT_FIRST == 1 || PKV_BULK_EVICT_FIRST == 4
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst_smem),
        "l"(src), "r"(bytes), "r"(bar), "l"(evict_first_policy())
        : "memory");
#else
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst_smem),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
#endif
}

template <bool PACK>
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src_smem, uint32_t bytes)
{
#if PKV_BULK_EVICT_FIRST == 1 || PKV_BULK_EVICT_FIRST == 3
    constexpr bool kHint = true;
#elif PKV_BULK_EVICT_FIRST == 2
    constexpr bool kHint = !PACK;
#else
    constexpr bool kHint = false;
#endif
    if (kHint)
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
                     "r"(src_smem), "r"(bytes), "l"(evict_first_policy())
                     : "memory");
    else
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src_smem),
                     "r"(bytes)
                     : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// The issuing lane's view of one pipe (of a pack when PACK, else of an unpack).
template <bool PACK>
struct Pipe {
    uint32_t data;  // shared address of slot 0
    PipeState *st;
    uint32_t head = 0;  // next op to store
    uint32_t tail = 0;  // next op to load
    bool failed = false;
    int *err;

    __device__ uint32_t bar(int s) const { return smem_addr(&st->bar[s]); }

    __device__ void store_oldest()
    {
        const int s = (int)(head % kSlots);
        if (!mbar_wait(bar(s), (head / kSlots) & 1u)) {
            failed = true;
            pkv::set_error(err, KV_DERR_TIMEOUT);
            return;
        }
        bulk_store<PACK>(reinterpret_cast<void *>(st->dst[s]), data + (uint32_t)s * kStage, st->bytes[s]);
        bulk_commit();
        head++;
    }

    __device__ void push(const uint8_t *src, uint8_t *dst, uint32_t bytes)
    {
        if (failed) return;
        if (tail - head == kSlots - 1) {
            store_oldest();
            if (failed) return;
            bulk_wait_read_1();  // every store but the newest has read its slot
        }
        const int s = (int)(tail % kSlots);
        st->dst[s] = reinterpret_cast<uint64_t>(dst);
        st->bytes[s] = bytes;
        mbar_arrive_expect_tx(bar(s), bytes);
        bulk_load(data + (uint32_t)s * kStage, src, bytes, bar(s));
        tail++;
    }

    __device__ void span(const uint8_t *src, uint8_t *dst, int64_t bytes)
    {
        for (int64_t off = 0; off < bytes; off += kStage)
            push(src + off, dst + off, (uint32_t)std::min<int64_t>(kStage, bytes - off));
    }

    __device__ void drain()
    {
        while (!failed && head != tail) store_oldest();
        if (failed) {  // let the loads still in flight land before shared memory goes away
            for (uint32_t i = head; i != tail; i++) mbar_wait(bar((int)(i % kSlots)), (i / kSlots) & 1u);
        }
        bulk_wait_all();
    }
};

// MODE: MERGED (a run is one span), SPANS (a span per (block, plane)) or REMAP (unpack onto another
// block size: a span per (staged block, plane), landing at the rows of the staged block's first
// token in its destination block; used when the destination's block size is a multiple of the
// staged one and the slice fills the destination's dense rows, so a staged block never straddles
// destination blocks).
template <int MODE, bool PACK>
__global__ void __launch_bounds__(kPipes * 32, 1) bulk_copy_kernel(const __grid_constant__ CopyParams p)
{
    pkv::grid_dep_entry();  // before any global memory access
    extern __shared__ __align__(1024) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    PipeState *st = reinterpret_cast<PipeState *>(smem + (size_t)kPipes * kSlots * kStage) + w;

    Pipe<PACK> pipe;
    pipe.data = smem_addr(smem + (size_t)w * kSlots * kStage);
    pipe.st = st;
    pipe.err = p.err;
    if (lane == 0) {
        for (int s = 0; s < kSlots; s++) mbar_init(pipe.bar(s), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();

    int64_t nr = *p.n_runs;
    if (nr > p.run_capacity) {
        if (blockIdx.x == 0 && threadIdx.x == 0) pkv::set_error(p.err, KV_DERR_CAPACITY);
        nr = p.run_capacity;
    }
    if (nr < 0) nr = 0;
    const int64_t items = nr * p.n_tensors;  // item = tensor * nr + run, tensor-major
    // This pipe's k-th item (increasing in k).  Persistent CTA b: g + k * P over [0, n_static),
    // g = b * kPipes + w, P = resident * kPipes.  Tail CTA b (b >= resident): item w + (k %
    // kTailItemsPerPipe) * kPipes of chunk (b - resident) + (k / kTailItemsPerPipe) * n_tail_ctas
    // of [n_static, items).
    const int64_t P = (int64_t)p.resident * kPipes;
    const int64_t n_static = p.tail_div > 0 ? (items - items / p.tail_div) / P * P : items;
    const bool tail = (int64_t)blockIdx.x >= p.resident;
    const int64_t chunk = (int64_t)kPipes * kTailItemsPerPipe;
    const int64_t n_tail_ctas = (int64_t)gridDim.x - p.resident;
    const int64_t g = tail ? (int64_t)blockIdx.x - p.resident : (int64_t)blockIdx.x * kPipes + w;
    const int64_t item_end = tail ? items : n_static;
    auto item_of = [&](int64_t k) -> int64_t {
        if (tail)
            return n_static + ((k / kTailItemsPerPipe) * n_tail_ctas + g) * chunk + w + (k % kTailItemsPerPipe) * kPipes;
        return g + k * P;
    };
    const int64_t block_bytes = p.stage_block_bytes;
    const int64_t span_bytes = (int64_t)p.div_cps.d * 16;  // one (block, plane) span

    kv_xfer_run next{};
    {
        const int64_t it = item_of(lane);
        if (it < item_end) next = p.runs[it % nr];
    }
    for (int64_t round = 0; item_of(round * kBatch) < item_end; round++) {
        st->rec[lane] = next;
        __syncwarp();
        {
            const int64_t it = item_of((round + 1) * kBatch + lane);  // prefetch the next round
            if (it < item_end) next = p.runs[it % nr];
        }
        if (lane == 0 && !pipe.failed) {
            int32_t cached_req = -1, s0 = 0, d0 = 0, dn = 0;  // REMAP: the last request's lists
            for (int i = 0; i < kBatch; i++) {
                const int64_t item = item_of(round * kBatch + i);
                if (item >= item_end) break;
                const int32_t t = (int32_t)(item / nr);
                const kv_xfer_run run = st->rec[i];
                if (run.n_blocks <= 0) continue;
                if (run.stage_block < 0 || run.stage_block + run.n_blocks > p.n_stage_blocks) {
                    pkv::set_error(p.err, KV_DERR_STAGE);
                    continue;
                }
                if (MODE == pkv::REMAP) {
                    const int32_t r = run.req;
                    if (r < 0 || r >= p.n_reqs) {
                        pkv::set_error(p.err, KV_DERR_DST_TABLE);
                        continue;
                    }
                    if (r != cached_req) {
                        cached_req = r;
                        s0 = p.src_req_offsets[r];
                        d0 = p.dst_req_offsets[r];
                        dn = (int32_t)max((int64_t)-1, min((int64_t)INT32_MAX, (int64_t)p.dst_req_offsets[r + 1] - d0));
                    }
                    if (run.stage_block < s0 || dn < 0 || d0 < 0) {  // offsets that do not match the runs
                        pkv::set_error(p.err, KV_DERR_DST_TABLE);
                        continue;
                    }
                    uint8_t *const cache_t = reinterpret_cast<uint8_t *>(p.base[t]);
                    const int64_t planes = block_bytes / span_bytes;
                    for (int32_t m = 0; m < run.n_blocks; m++) {
                        const int64_t j = (run.stage_block - s0 + m) * (int64_t)p.div_bs.d;  // its first token
                        const int64_t dq = j / p.div_dbs.d;
                        if (dq >= dn) {
                            pkv::set_error(p.err, KV_DERR_DST_TABLE);
                            continue;
                        }
                        const int32_t db = p.dst_ids[d0 + dq];
                        if (db < 0 || db >= p.num_blocks) {
                            pkv::set_error(p.err, KV_DERR_BLOCK);
                            continue;
                        }
                        uint8_t *const dst = cache_t + (int64_t)db * p.block_stride + (j - dq * p.div_dbs.d) * p.token_stride;
                        const uint8_t *const src = p.stage + (int64_t)(p.tensor_begin + t) * p.stage_tensor_bytes +
                                                   (run.stage_block + m) * block_bytes;
                        for (int64_t pl = 0; pl < planes; pl++)
                            pipe.span(src + pl * span_bytes, dst + pl * p.plane_stride, span_bytes);
                    }
                    continue;
                }
                const int64_t blk = PACK ? run.src_block : run.dst_block;
                if (blk < 0 || blk + run.n_blocks > p.num_blocks) {
                    pkv::set_error(p.err, KV_DERR_BLOCK);
                    continue;
                }
                uint8_t *const cache = reinterpret_cast<uint8_t *>(p.base[t]) + blk * p.block_stride;
                uint8_t *const stage =
                    p.stage + (int64_t)(p.tensor_begin + t) * p.stage_tensor_bytes + run.stage_block * block_bytes;
                if (MODE == pkv::MERGED) {
                    const int64_t bytes = (int64_t)run.n_blocks * block_bytes;
                    if (PACK) pipe.span(cache, stage, bytes);
                    else pipe.span(stage, cache, bytes);
                } else {
                    const int64_t planes = block_bytes / span_bytes;
                    for (int32_t m = 0; m < run.n_blocks; m++) {
                        for (int64_t pl = 0; pl < planes; pl++) {
                            uint8_t *c = cache + (int64_t)m * p.block_stride + pl * p.plane_stride;
                            uint8_t *sg = stage + (int64_t)m * block_bytes + pl * span_bytes;
                            if (PACK) pipe.span(c, sg, span_bytes);
                            else pipe.span(sg, c, span_bytes);
                        }
                    }
                }
            }
        }
        __syncwarp();
    }
    if (lane == 0) {
        pipe.drain();
        // the bulk stores were written by the async proxy: order them before the signal
        asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    __syncwarp();
    pkv::signal_on_exit(p);
}

using BulkFn = void (*)(CopyParams);

BulkFn pick(int mode, bool pack)
{
    if (mode == pkv::MERGED) return pack ? bulk_copy_kernel<pkv::MERGED, true> : bulk_copy_kernel<pkv::MERGED, false>;
    if (mode == pkv::REMAP) return bulk_copy_kernel<pkv::REMAP, false>;
    return pack ? bulk_copy_kernel<pkv::SPANS, true> : bulk_copy_kernel<pkv::SPANS, false>;
}

}  // namespace

namespace pkv {

int preload_bulk_kernels()
{
    return load_kernels(bulk_copy_kernel<pkv::MERGED, true>, bulk_copy_kernel<pkv::MERGED, false>,
                        bulk_copy_kernel<pkv::SPANS, true>, bulk_copy_kernel<pkv::SPANS, false>,
                        bulk_copy_kernel<pkv::REMAP, false>);
}

int launch_bulk_copy(const CopyParams &params, int mode, bool pack, const DeviceInfo &dev, cudaStream_t s)
{
    CopyParams p = params;
    static std::mutex mu;
    static bool configured[64][3][2];
    static int per_sm[64][3][2];
    const BulkFn fn = pick(mode, pack);
    const int m = mode == MERGED ? 1 : mode == REMAP ? 2 : 0, d = pack ? 1 : 0, di = dev.device & 63;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!configured[di][m][d]) {
            int st = cuda_status(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes));
            if (st != KV_OK) return st;
            int n = 0;
            st = cuda_status(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kPipes * 32, kSmemBytes));
            if (st != KV_OK) return st;
            per_sm[di][m][d] = std::max(1, n);
            configured[di][m][d] = true;
        }
    }
    // persistent CTAs, plus enough tail CTAs for the largest tail the device-side run count allows
    p.resident = dev.num_sms * per_sm[di][m][d];
    int64_t tail_ctas = 0;
    const int64_t items_max = std::min<int64_t>(p.run_capacity, p.n_stage_blocks) * p.n_tensors;
    const int64_t quantum = (int64_t)kPipes * p.resident;
    p.tail_div = 0;
    if (kTailDiv > 0 && items_max >= kTailMinItemsPerPipe * quantum) {
        const int64_t chunk = (int64_t)kPipes * kTailItemsPerPipe;
        p.tail_div = (int32_t)kTailDiv;
        tail_ctas = std::max<int64_t>(1, std::min<int64_t>((items_max / std::max<int64_t>(1, kTailDiv) + quantum + chunk - 1) / chunk,
                                                           (int64_t)kMaxTailCtasPerResident * p.resident));
    }
    pkv::launch_as(tail_ctas == 0, fn, p.resident + (int)tail_ctas, kPipes * 32, kSmemBytes, s, p);  // tail: plain
    return cuda_status(cudaGetLastError());
}

}  // namespace pkv
