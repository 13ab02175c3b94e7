// kv_build_xfer_list: flattening per-request block lists into maximal contiguous runs.
//
// The sender's xfer_list, flattened over layers, contiguous groups and requests (page "5. flagcx
// connector design & dev & test", section 1.2) needs, per request, the runs of
// consecutive block ids; each run is one (source, destination, length) triple (page
// "vLLM PD 分离 源码级机制", section 4.2, _send_blocks).  The layer factor is applied by
// the copy kernels, which walk (tensor x run).
//
// Single pass over tiles of 2048 list entries, one CTA per tile, tiles taken in launch
// order from a counter.  Entry i is a natural run start when it opens its request or
// breaks id contiguity; the cap adds a start wherever (i - s) % cap == 0 for the
// natural start s of i's run.  A tile's contribution therefore depends on the
// natural start open at its left edge, which the look-back carries:
//   aggregate of [a, b):  first and last natural start in it, and the run starts in
//                         [first natural start, b) (all decidable inside the range);
//   prefix at b:          last natural start before b and the number of run starts before b.
// The cap's starts in a stretch [a, b) with no natural start, continuing a run opened at
// s < a, are counted in closed form: floor((b-1-s)/cap) - floor((a-1-s)/cap).
//
// A list of at most one single-CTA tile (5120 entries) takes a second kernel instead: one
// CTA of 1024 threads, no look-back and no scratch, its run records staged in shared memory
// and written out contiguously.
#include <algorithm>
#include <mutex>

#include "kv_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kItems = 8;
constexpr int kTile = kThreads * kItems;
constexpr int kWarps = kThreads / 32;
constexpr int64_t kHeaderBytes = 256;
constexpr int kOffsetCache = 1024;  // request offsets kept in shared memory when n_reqs + 1 fits
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s bound on any look-back wait

struct TileRecord {  // 32 bytes per tile in the workspace
    int32_t flag;    // 0 empty, 1 aggregate published, 2 inclusive prefix published
    int32_t first_nat;
    int32_t last_nat;
    int32_t cnt;
    int32_t pre_s;
    int32_t pre_cnt;
    int32_t pad[2];
};

struct Agg {
    int32_t first_nat;  // -1: no natural start in the range
    int32_t last_nat;
    int32_t cnt;  // run starts in [first_nat, end)
};

struct Pre {
    int32_t s;    // last natural start before the position
    int32_t cnt;  // run starts before the position
};

__device__ __forceinline__ int32_t cap_starts(int32_t s, int32_t a, int32_t b, int32_t cap)
{
    if (cap <= 0 || b <= a) return 0;
    return (b - 1 - s) / cap - (a - 1 - s) / cap;
}

// Prefix at b from the prefix at a and the aggregate of [a, b).
__device__ __forceinline__ Pre apply(const Agg &g, int32_t a, int32_t b, const Pre &p, int32_t cap)
{
    if (g.first_nat < 0) return Pre{p.s, p.cnt + cap_starts(p.s, a, b, cap)};
    return Pre{g.last_nat, p.cnt + cap_starts(p.s, a, g.first_nat, cap) + g.cnt};
}

// Aggregate of [a, b) from A over [a, m) and B over [m, b).
__device__ __forceinline__ Agg combine(const Agg &A, const Agg &B, int32_t m, int32_t b, int32_t cap)
{
    if (B.first_nat < 0) {
        if (A.first_nat < 0) return A;
        return Agg{A.first_nat, A.last_nat, A.cnt + cap_starts(A.last_nat, m, b, cap)};
    }
    if (A.first_nat < 0) return B;
    return Agg{A.first_nat, B.last_nat, A.cnt + cap_starts(A.last_nat, m, B.first_nat, cap) + B.cnt};
}

__device__ __forceinline__ int32_t ld_acquire(const int32_t *p)
{
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(int32_t *p, int32_t v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

struct Max {
    __device__ int32_t operator()(int32_t a, int32_t b) const { return a > b ? a : b; }
};
struct Min {
    __device__ int32_t operator()(int32_t a, int32_t b) const { return a < b ? a : b; }
};
struct Sum {
    __device__ int32_t operator()(int32_t a, int32_t b) const { return a + b; }
};

// Exclusive block-wide scan of one value per thread over NW warps; *total gets the reduction.
template <int NW = kWarps, typename Op>
__device__ int32_t block_exclusive(int32_t v, int32_t identity, Op op, int32_t *sh, int32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl = op(incl, y);
    }
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    // every warp scans the NW warp totals itself (one shared load and five shuffles)
    int32_t w_incl = lane < NW ? sh[lane] : identity;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, w_incl, d);
        if (lane >= d) w_incl = op(w_incl, y);
    }
    const int32_t all = __shfl_sync(0xffffffffu, w_incl, 31);
    int32_t before = __shfl_sync(0xffffffffu, w_incl, warp > 0 ? warp - 1 : 0);
    if (warp == 0) before = identity;
    __syncthreads();
    int32_t excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = identity;
    *total = all;
    return op(before, excl);
}

struct XferParams {
    const int32_t *req_offsets;
    const int32_t *src;
    const int32_t *dst;  // may be null
    kv_xfer_run *runs;
    int32_t *n_runs;
    uint32_t *counter;
    TileRecord *tiles;
    int *err;
    int64_t capacity;
    int32_t n_reqs;
    int32_t n;
    int32_t cap;
};

// Place of an entry d entries after its run's natural start: d % cap, or d without a cap.
__device__ __forceinline__ int32_t phase_of(int32_t d, int32_t cap) { return cap > 0 ? d % cap : d; }
__device__ __forceinline__ int32_t next_phase(int32_t ph, int32_t cap)
{
    return (cap > 0 && ph + 1 == cap) ? 0 : ph + 1;
}

// First half of a tile: stage the tile's ids (one halo entry each side) and, when few, the
// request offsets in shared memory with coalesced loads; then mark, for this thread's ITEMS
// entries from i0 and the entry after them, which are natural run starts (request start, or
// a break in src or dst id contiguity; past the list counts as a start), with each entry's
// request.  Ends with the block synchronised.
template <int ITEMS, int NT>
__device__ __forceinline__ void stage_and_mark(const XferParams &p, int32_t tile_start, int32_t *sh_src,
                                               int32_t *sh_dst, int32_t *sh_off, bool (&nat)[ITEMS + 1],
                                               int32_t (&req)[ITEMS])
{
    constexpr int kT = ITEMS * NT;
    constexpr int kPer = (kT + 2 + NT - 1) / NT;  // staged ids per thread
    const int tid = threadIdx.x;
    // every load is issued before the first shared store: read-only global loads cannot alias
    // the shared arrays, so they overlap instead of each waiting out the previous store
    int32_t vs[kPer], vd[kPer];
#pragma unroll
    for (int u = 0; u < kPer; u++) {
        const int k = tid + u * NT;
        const int32_t i = tile_start - 1 + k;
        const bool in = k < kT + 2 && i >= 0 && i < p.n;
        vs[u] = in ? __ldg(p.src + i) : 0;
        vd[u] = in && p.dst ? __ldg(p.dst + i) : 0;
    }
    const bool off_cached = p.n_reqs + 1 <= kOffsetCache;
    constexpr int kOffPer = (kOffsetCache + NT - 1) / NT;
    int32_t vo[kOffPer];
    if (off_cached) {
#pragma unroll
        for (int u = 0; u < kOffPer; u++) {
            const int k = tid + u * NT;
            vo[u] = k <= p.n_reqs ? __ldg(p.req_offsets + k) : 0;
        }
    }
#pragma unroll
    for (int u = 0; u < kPer; u++) {
        const int k = tid + u * NT;
        if (k < kT + 2) {
            sh_src[k] = vs[u];
            if (p.dst) sh_dst[k] = vd[u];
        }
    }
    if (off_cached) {
#pragma unroll
        for (int u = 0; u < kOffPer; u++) {
            const int k = tid + u * NT;
            if (k <= p.n_reqs) sh_off[k] = vo[u];
        }
    }
    __syncthreads();
    auto offset = [&](int32_t k) { return off_cached ? sh_off[k] : p.req_offsets[k]; };

    const int32_t i0 = tile_start + tid * ITEMS;
    if (i0 >= p.n) {
#pragma unroll
        for (int k = 0; k <= ITEMS; k++) nat[k] = true;
#pragma unroll
        for (int k = 0; k < ITEMS; k++) req[k] = 0;
        return;
    }
    int32_t lo = 0, hi = p.n_reqs - 1;  // last request whose first entry is <= i0
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (offset(mid) <= i0) lo = mid;
        else hi = mid - 1;
    }
    int32_t r = lo;
    int32_t begin = offset(r), end = offset(r + 1);
    const int32_t base = i0 - tile_start + 1;  // index of entry i0 in the staged ids
    int32_t prev_s = sh_src[base - 1];
    int32_t prev_d = p.dst ? sh_dst[base - 1] : 0;
#pragma unroll
    for (int k = 0; k <= ITEMS; k++) {
        const int32_t i = i0 + k;
        if (i >= p.n) {
            nat[k] = true;  // past the list: closes the last run
            if (k < ITEMS) req[k] = r;
            continue;
        }
        while (i >= end && r < p.n_reqs - 1) {
            r++;
            begin = end;
            end = offset(r + 1);
        }
        const int32_t sv = sh_src[base + k];
        const int32_t dv = p.dst ? sh_dst[base + k] : 0;
        nat[k] = (i == begin) || (sv != prev_s + 1) || (p.dst != nullptr && dv != prev_d + 1);
        if (k < ITEMS) req[k] = r;
        prev_s = sv;
        prev_d = dv;
    }
}

// Second half of a tile: with s0, the natural start open at this thread's first entry i0, and
// cnt0, the runs started before the tile, number every run start and write each run's record
// at its last entry (the entry whose successor starts a run).  Returns the run starts in the
// tile.  An entry whose run start is unknown (s0 < 0) sets `unknown_err`.
template <int ITEMS = kItems, int NW = kWarps>
__device__ __forceinline__ int32_t resolve_and_write(const XferParams &p, const bool (&nat)[ITEMS + 1],
                                                     const int32_t (&req)[ITEMS], int32_t i0, int32_t tile_start,
                                                     int32_t tile_end, int32_t s0, int32_t cnt0,
                                                     const int32_t *sh_src, const int32_t *sh_dst, int32_t *sh_scan,
                                                     int unknown_err, kv_xfer_run *sh_rec = nullptr)
{
    int32_t ph[ITEMS];  // (i - s) % cap for each entry's natural start s
    bool start[ITEMS];
    bool known = s0 >= 0;
    int32_t mine = 0;
    {
        int32_t q = known ? phase_of(i0 - s0, p.cap) : 0;
#pragma unroll
        for (int k = 0; k < ITEMS; k++) {
            const int32_t i = i0 + k;
            if (i < tile_end && nat[k]) q = 0;
            ph[k] = q;
            start[k] = i < tile_end && (nat[k] || (p.cap > 0 && q == 0));
            mine += start[k] ? 1 : 0;
            q = next_phase(q, p.cap);
        }
    }
    int32_t total;
    const int32_t before = block_exclusive<NW>(mine, 0, Sum(), sh_scan, &total);
    int32_t run = cnt0 + before - 1;  // index of the run holding the current entry
#pragma unroll
    for (int k = 0; k < ITEMS; k++) {
        const int32_t i = i0 + k;
        if (i >= tile_end) break;
        if (start[k]) run++;
        if (nat[k]) known = true;
        if (!(nat[k + 1] || (p.cap > 0 && ph[k] + 1 == p.cap))) continue;
        const int32_t first = i - ph[k];
        if (!known || first < 0) {
            pkv::set_error(p.err, unknown_err);
            continue;
        }
        if ((int64_t)run >= p.capacity || run < 0) {
            pkv::set_error(p.err, KV_DERR_CAPACITY);
            continue;
        }
        kv_xfer_run out;
        out.req = req[k];
        const bool staged = first >= tile_start - 1;
        out.src_block = staged ? sh_src[first - tile_start + 1] : p.src[first];
        out.dst_block = p.dst ? (staged ? sh_dst[first - tile_start + 1] : p.dst[first]) : -1;
        out.n_blocks = ph[k] + 1;
        out.stage_block = first;
        if (sh_rec != nullptr) sh_rec[run - cnt0] = out;  // the caller copies the tile's records out
        else p.runs[run] = out;
    }
    return total;
}

__global__ void __launch_bounds__(kThreads) build_xfer_kernel(const __grid_constant__ XferParams p)
{
    pkv::grid_dep_entry();  // before any global memory access
    __shared__ int32_t sh_scan[kWarps];
    __shared__ int32_t sh_tile;
    __shared__ Pre sh_pre;

    const int tid = threadIdx.x;
    if (tid == 0) sh_tile = (int32_t)atomicAdd(p.counter, 1u);
    __syncthreads();
    const int32_t tile = sh_tile;
    const int32_t tile_start = tile * kTile;
    const int32_t tile_end = min(tile_start + kTile, p.n);
    const int32_t i0 = tile_start + tid * kItems;

    const bool checker = tile == 0 && tid == 0;  // validates the offsets' ends, loads issued early
    const int32_t o_first = checker ? __ldg(p.req_offsets) : 0;
    const int32_t o_last = checker ? __ldg(p.req_offsets + p.n_reqs) : p.n;

    __shared__ int32_t sh_src[kTile + 2];
    __shared__ int32_t sh_dst[kTile + 2];
    __shared__ int32_t sh_off[kOffsetCache];
    bool nat[kItems + 1];
    int32_t req[kItems];
    stage_and_mark<kItems, kThreads>(p, tile_start, sh_src, sh_dst, sh_off, nat, req);
    if (o_first != 0 || o_last != p.n) pkv::set_error(p.err, KV_DERR_LIST);

    // ---- tile aggregate from what is decidable locally ----
    int32_t my_last = -1, my_first = 0x7fffffff;
#pragma unroll
    for (int k = 0; k < kItems; k++) {
        const int32_t i = i0 + k;
        if (i < tile_end && nat[k]) {
            my_last = i;
            my_first = min(my_first, i);
        }
    }
    int32_t tile_last;
    const int32_t s_before = block_exclusive(my_last, -1, Max(), sh_scan, &tile_last);
    int32_t tile_first;
    block_exclusive(my_first, 0x7fffffff, Min(), sh_scan, &tile_first);

    // Run starts decidable before the look-back: those after a natural start seen in this tile.
    // ph is the entry's place in its cap piece, (i - s) % cap (or i - s without a cap), kept by
    // incrementing: one division per thread instead of one per entry.
    int32_t known = 0;
    {
        int32_t s = s_before;
        int32_t ph = s >= 0 ? phase_of(i0 - s, p.cap) : 0;
#pragma unroll
        for (int k = 0; k < kItems; k++) {
            const int32_t i = i0 + k;
            if (i < tile_end && nat[k]) {
                s = i;
                ph = 0;
            }
            if (i < tile_end && s >= 0 && (nat[k] || (p.cap > 0 && ph == 0))) known++;
            ph = next_phase(ph, p.cap);
        }
    }
    int32_t tile_cnt;
    block_exclusive(known, 0, Sum(), sh_scan, &tile_cnt);

    // ---- publish, look back, publish the inclusive prefix ----
    // Warp 0 looks back 32 predecessor tiles at a time: lane l reads tile j - l.  The nearest
    // lane holding an inclusive prefix (a tile before the list counts, with prefix {-1, 0})
    // bounds the window; every tile between it and this one must have published its
    // aggregate, else the window is read again (bounded wait).  The aggregates are then
    // folded nearest first, and the prefix applied.  Every lane computes the same values.
    if (tid < 32) {
        const int lane = tid;
        const Agg agg{tile_first == 0x7fffffff ? -1 : tile_first, tile_last, tile_cnt};
        TileRecord *rec = p.tiles + tile;
        Pre excl{-1, 0};
        if (tile > 0) {
            if (lane == 0) {
                rec->first_nat = agg.first_nat;
                rec->last_nat = agg.last_nat;
                rec->cnt = agg.cnt;
                st_release(&rec->flag, 1);
            }
            Agg suffix{-1, -1, 0};  // aggregate of [(j + 1) * kTile, tile_start)
            int32_t j = tile - 1;    // nearest tile not yet folded in
            const unsigned long long t_begin = global_ns();
            unsigned ns = 32;
            while (true) {
                const int32_t jj = j - lane;
                int32_t f = 2;
                Pre pj{-1, 0};
                Agg aj{-1, -1, 0};
                if (jj >= 0) {
                    const TileRecord *pr = p.tiles + jj;
                    f = ld_acquire(&pr->flag);
                    if (f == 2) pj = Pre{__ldcg(&pr->pre_s), __ldcg(&pr->pre_cnt)};
                    else if (f == 1) aj = Agg{__ldcg(&pr->first_nat), __ldcg(&pr->last_nat), __ldcg(&pr->cnt)};
                }
                const unsigned pre_mask = __ballot_sync(0xffffffffu, f == 2);
                const int p_lane = pre_mask ? __ffs(pre_mask) - 1 : 32;
                const unsigned before = p_lane >= 32 ? 0xffffffffu : (1u << p_lane) - 1u;
                if (__ballot_sync(0xffffffffu, f == 0) & before) {
                    const int expired = __shfl_sync(0xffffffffu, lane == 0 ? (int)(global_ns() - t_begin > kWaitLimitNs) : 0, 0);
                    if (expired) {
                        if (lane == 0) pkv::set_error(p.err, KV_DERR_TIMEOUT);
                        break;  // give up: prefix left at {-1, 0}
                    }
                    __nanosleep(ns);
                    ns = min(ns * 2u, 1024u);
                    continue;
                }
                for (int k = 0; k < p_lane; k++) {  // tiles j, j - 1, ..., j - p_lane + 1
                    const Agg ak{__shfl_sync(0xffffffffu, aj.first_nat, k), __shfl_sync(0xffffffffu, aj.last_nat, k),
                                 __shfl_sync(0xffffffffu, aj.cnt, k)};
                    suffix = combine(ak, suffix, (j - k + 1) * kTile, tile_start, p.cap);
                }
                if (p_lane < 32) {
                    const Pre pp{__shfl_sync(0xffffffffu, pj.s, p_lane), __shfl_sync(0xffffffffu, pj.cnt, p_lane)};
                    excl = apply(suffix, (j - p_lane + 1) * kTile, tile_start, pp, p.cap);
                    break;
                }
                j -= 32;
            }
        }
        if (lane == 0) {
            const Pre incl = apply(agg, tile_start, tile_end, excl, p.cap);
            rec->pre_s = incl.s;
            rec->pre_cnt = incl.cnt;
            st_release(&rec->flag, 2);
            sh_pre = excl;
            if (tile_end == p.n) {
                *p.n_runs = incl.cnt;
                if ((int64_t)incl.cnt > p.capacity) pkv::set_error(p.err, KV_DERR_CAPACITY);
            }
        }
    }
    __syncthreads();
    const Pre excl = sh_pre;

    // ---- resolve every entry, number the runs, write each run at its last entry ----
    const int32_t s0 = s_before >= 0 ? s_before : excl.s;  // -1 only after a look-back timeout
    resolve_and_write(p, nat, req, i0, tile_start, tile_end, s0, excl.cnt, sh_src, sh_dst, sh_scan,
                      KV_DERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// Single-CTA builder for lists that fit one tile of NT * kSItems entries: the look-back kernel
// without the look-back, so it needs neither the scratch nor its zeroing.  A short list
// (a decode-side request, a few prompts) is then one launch.  Longer lists go to the
// look-back kernel: one CTA walking several tiles in turn is slower than one CTA per tile.
// The run records go through NT * kSItems * 24 bytes of dynamic shared memory (see below).
// Lists of up to kSSmallTile entries (one request's blocks, say) take a 128-thread instance,
// which needs 15 KB of records instead of 123 KB and fits beside other work on any SM.
// ---------------------------------------------------------------------------
#ifndef PKV_XFER_SINGLE_ITEMS
#define PKV_XFER_SINGLE_ITEMS 5
#endif
#ifndef PKV_XFER_SMALL_THREADS
#define PKV_XFER_SMALL_THREADS 128  // 0: every single-tile list takes the 1024-thread instance
#endif
constexpr int kSThreads = 1024;
constexpr int kSItems = PKV_XFER_SINGLE_ITEMS;
constexpr int kSTile = kSThreads * kSItems;
constexpr int kSSmallThreads = PKV_XFER_SMALL_THREADS > 0 ? PKV_XFER_SMALL_THREADS : 32;
constexpr int kSSmallTile = PKV_XFER_SMALL_THREADS > 0 ? kSSmallThreads * kSItems : 0;

template <int NT>
__global__ void __launch_bounds__(NT) build_xfer_single_kernel(const __grid_constant__ XferParams p)
{
    pkv::grid_dep_entry();  // before any global memory access
    constexpr int kTileN = NT * kSItems;
    constexpr int kNW = NT / 32;
    __shared__ int32_t sh_src[kTileN + 2];
    __shared__ int32_t sh_dst[kTileN + 2];
    __shared__ int32_t sh_off[kOffsetCache];
    __shared__ int32_t sh_scan[kNW];

    const int tid = threadIdx.x;
    const int32_t o_first = tid == 0 ? __ldg(p.req_offsets) : 0;  // the offsets' ends, checked below
    const int32_t o_last = tid == 0 ? __ldg(p.req_offsets + p.n_reqs) : p.n;
    bool nat[kSItems + 1];
    int32_t req[kSItems];
    stage_and_mark<kSItems, NT>(p, 0, sh_src, sh_dst, sh_off, nat, req);
    if (o_first != 0 || o_last != p.n) pkv::set_error(p.err, KV_DERR_LIST);
    const int32_t i0 = tid * kSItems;
    int32_t my_last = -1;
#pragma unroll
    for (int k = 0; k < kSItems; k++)
        if (i0 + k < p.n && nat[k]) my_last = i0 + k;
    int32_t unused;
    // natural start open at i0; -1 only when the offsets do not start at 0
    const int32_t s0 = block_exclusive<kNW>(my_last, -1, Max(), sh_scan, &unused);
    // records go to shared memory first: one thread's runs are consecutive records, so direct
    // stores from a thread's items scatter over a whole warp's range of sectors
    extern __shared__ __align__(16) kv_xfer_run sh_rec[];  // kTileN records
    const int32_t cnt = resolve_and_write<kSItems, kNW>(p, nat, req, i0, 0, p.n, s0, 0, sh_src, sh_dst, sh_scan,
                                                        KV_DERR_LIST, sh_rec);
    __syncthreads();
    const int64_t n_out = min((int64_t)cnt, p.capacity);  // records past the capacity are not written
    const unsigned long long *src64 = reinterpret_cast<const unsigned long long *>(sh_rec);
    unsigned long long *dst64 = reinterpret_cast<unsigned long long *>(p.runs);
    for (int64_t w = tid; w < n_out * 3; w += NT) dst64[w] = src64[w];
    if (tid == 0) {
        *p.n_runs = cnt;
        if ((int64_t)cnt > p.capacity) pkv::set_error(p.err, KV_DERR_CAPACITY);
    }
}

constexpr int kSingleRecordBytes = kSTile * (int)sizeof(kv_xfer_run);
constexpr int kSmallRecordBytes = kSSmallTile * (int)sizeof(kv_xfer_run);
static_assert(kSmallRecordBytes <= 48 * 1024, "the small builder's records must fit the default dynamic smem");

// Launches the single-CTA builder for lists of one tile (the scratch is not touched), else zeroes the look-back scratch (tile counter and tile records: `need` bytes
// at `scratch`) and launches one CTA per tile.
int launch_builder(const int32_t *req_offsets, int32_t n_reqs, const int32_t *src_ids, const int32_t *dst_ids,
                   int64_t n_blocks, int32_t max_run_blocks, kv_xfer_run *runs, int64_t run_capacity,
                   int32_t *n_runs, void *scratch, int64_t need, const pkv::DeviceInfo &dev, cudaStream_t s)
{
    XferParams p{};
    p.req_offsets = req_offsets;
    p.src = src_ids;
    p.dst = dst_ids;
    p.runs = runs;
    p.n_runs = n_runs;
    p.err = dev.err_word;
    p.capacity = run_capacity;
    p.n_reqs = n_reqs;
    p.n = (int32_t)n_blocks;
    p.cap = max_run_blocks;
    if (n_blocks <= kSSmallTile) {
        pkv::launch(build_xfer_single_kernel<kSSmallThreads>, 1, kSSmallThreads, kSmallRecordBytes, s, p);
        return pkv::cuda_status(cudaGetLastError());
    }
    if (n_blocks <= kSTile) {
        static std::mutex mu;
        static bool configured[64];
        {
            std::lock_guard<std::mutex> lock(mu);
            if (!configured[dev.device & 63]) {
                const int st = pkv::cuda_status(cudaFuncSetAttribute(
                    build_xfer_single_kernel<kSThreads>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSingleRecordBytes));
                if (st != KV_OK) return st;
                configured[dev.device & 63] = true;
            }
        }
        pkv::launch(build_xfer_single_kernel<kSThreads>, 1, kSThreads, kSingleRecordBytes, s, p);
        return pkv::cuda_status(cudaGetLastError());
    }
    const int st = pkv::cuda_status(cudaMemsetAsync(scratch, 0, (size_t)need, s));
    if (st != KV_OK) return st;
    p.counter = reinterpret_cast<uint32_t *>(scratch);
    p.tiles = reinterpret_cast<TileRecord *>(reinterpret_cast<uint8_t *>(scratch) + kHeaderBytes);
    const int tiles = (int)((n_blocks + kTile - 1) / kTile);
    // A plain stream-ordered launch: the scratch memset just before it is not a kernel that
    // the entry wait would cover.
    build_xfer_kernel<<<tiles, kThreads, 0, s>>>(p);
    return pkv::cuda_status(cudaGetLastError());
}

}  // namespace

int pkv::preload_xfer_kernels()
{
    return pkv::load_kernels(build_xfer_single_kernel<kSSmallThreads>, build_xfer_single_kernel<kSThreads>,
                             build_xfer_kernel);
}

extern "C" {

int kv_xfer_workspace_bytes(int64_t n_blocks, int64_t *bytes_out)
{
    if (bytes_out == nullptr || n_blocks < 0) return KV_ERR_INVALID_ARG;
    const int64_t tiles = std::max<int64_t>(1, (n_blocks + kTile - 1) / kTile);
    *bytes_out = kHeaderBytes + tiles * (int64_t)sizeof(TileRecord);
    return KV_OK;
}

int kv_build_xfer_list(const int32_t *req_offsets, int32_t n_reqs, const int32_t *src_ids,
                       const int32_t *dst_ids, int64_t n_blocks, int32_t max_run_blocks,
                       kv_xfer_run *runs, int64_t run_capacity, int32_t *n_runs,
                       void *workspace, int64_t workspace_bytes, kv_stream_t stream)
{
    if (n_reqs < 0 || n_blocks < 0 || max_run_blocks < 0 || run_capacity < 0 || n_runs == nullptr ||
        req_offsets == nullptr)
        return KV_ERR_INVALID_ARG;
    if (n_blocks >= (1ll << 31) - kTile) return KV_ERR_UNSUPPORTED;
    if (n_blocks > 0 && (n_reqs == 0 || src_ids == nullptr || (run_capacity > 0 && runs == nullptr)))
        return KV_ERR_INVALID_ARG;
    const cudaStream_t s = (cudaStream_t)stream;
    if (n_blocks == 0) return pkv::cuda_status(cudaMemsetAsync(n_runs, 0, sizeof(int32_t), s));
    int64_t need = 0;
    kv_xfer_workspace_bytes(n_blocks, &need);
    if (workspace == nullptr) return KV_ERR_INVALID_ARG;
    if (!pkv::aligned16(workspace)) return KV_ERR_ALIGN;
    if (workspace_bytes < need) return KV_ERR_RANGE;
    if (((uintptr_t)runs & 7u) != 0) return KV_ERR_ALIGN;
    const pkv::DeviceInfo *dev = pkv::current_device();
    if (dev == nullptr) return KV_ERR_CUDA;
    return launch_builder(req_offsets, n_reqs, src_ids, dst_ids, n_blocks, max_run_blocks, runs, run_capacity,
                          n_runs, workspace, need, *dev, s);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// kv_build_xfer_list_static: the builder above with its look-back scratch in a fixed
// array inside this library instead of a workspace the caller allocates.
// ---------------------------------------------------------------------------
namespace {

constexpr int64_t kStaticScratchBytes = KV_XFER_STATIC_SCRATCH_BYTES;
static_assert(kHeaderBytes + ((KV_XFER_STATIC_MAX_BLOCKS + kTile - 1) / kTile) * (int64_t)sizeof(TileRecord) <=
                  kStaticScratchBytes,
              "KV_XFER_STATIC_MAX_BLOCKS does not fit the static scratch");
static_assert(kHeaderBytes + ((KV_XFER_STATIC_MAX_BLOCKS + kTile) / kTile) * (int64_t)sizeof(TileRecord) >
                  kStaticScratchBytes,
              "KV_XFER_STATIC_MAX_BLOCKS is not the largest list the static scratch holds");

// One copy per device that loads this library, kept until the process exits.  Every
// kv_build_xfer_list_static call on that device uses it.
static __device__ __align__(256) uint8_t g_xfer_static_scratch[kStaticScratchBytes];

constexpr int kMaxStaticDevices = 64;
std::mutex g_static_mutex;
void *g_static_scratch_addr[kMaxStaticDevices];

// Device address of the scratch array on the current device.  In host code the array's
// name stands for a host-side shadow, so the address is looked up once per device (with
// that device current) and cached.
int static_scratch_address(int device, void **out)
{
    if (device < 0 || device >= kMaxStaticDevices) return KV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (g_static_scratch_addr[device] == nullptr) {
        void *p = nullptr;
        const int st = pkv::cuda_status(cudaGetSymbolAddress(&p, g_xfer_static_scratch));
        if (st != KV_OK) return st;
        g_static_scratch_addr[device] = p;
    }
    *out = g_static_scratch_addr[device];
    return KV_OK;
}

}  // namespace

extern "C" int kv_build_xfer_list_static(const int32_t *req_offsets, int32_t n_reqs, const int32_t *src_ids,
                                         const int32_t *dst_ids, int64_t n_blocks, int32_t max_run_blocks,
                                         kv_xfer_run *runs, int64_t run_capacity, int32_t *n_runs,
                                         kv_stream_t stream)
{
    if (n_reqs < 0 || n_blocks < 0 || max_run_blocks < 0 || run_capacity < 0 || n_runs == nullptr ||
        req_offsets == nullptr)
        return KV_ERR_INVALID_ARG;
    if (n_blocks > KV_XFER_STATIC_MAX_BLOCKS) return KV_ERR_RANGE;
    if (n_blocks > 0 && (n_reqs == 0 || src_ids == nullptr || (run_capacity > 0 && runs == nullptr)))
        return KV_ERR_INVALID_ARG;
    if (((uintptr_t)runs & 7u) != 0) return KV_ERR_ALIGN;
    const cudaStream_t s = (cudaStream_t)stream;
    if (n_blocks == 0) return pkv::cuda_status(cudaMemsetAsync(n_runs, 0, sizeof(int32_t), s));
    const pkv::DeviceInfo *dev = pkv::current_device();
    if (dev == nullptr) return KV_ERR_CUDA;
    void *scratch = nullptr;
    int st = static_scratch_address(dev->device, &scratch);
    if (st != KV_OK) return st;

    int64_t need = 0;
    kv_xfer_workspace_bytes(n_blocks, &need);
    return launch_builder(req_offsets, n_reqs, src_ids, dst_ids, n_blocks, max_run_blocks, runs, run_capacity,
                          n_runs, scratch, need, *dev, s);
}
