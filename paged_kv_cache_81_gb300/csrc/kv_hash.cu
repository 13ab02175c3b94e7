// kv_block_hashes: the prefix hash chain over full token blocks.
//
// Drawing "vllm v1 调度逻辑 和 distributed 分布式原理", the hash-table labels: every full block is
// keyed by h0 = hash(seed, [t0 .. t(bs-1)]) and h_i = hash(h_(i-1), [tokens of block i]), so
// equal prefixes give equal keys (cached_block_hash_to_block).  The pages do not name the hash;
// the reading implemented here is FNV-1a 64 over the parent hash as 8 little-endian bytes
// followed by the block's token ids as 4 little-endian bytes each.  Only full blocks are hashed.
//
// FNV-1a is byte-serial and each block starts from its parent's hash, so a request's chain is
// sequential.  With a workspace, each block's hash is split by a property of FNV-1a: the xor of
// a byte only changes the state's low byte c, so a step is h' = P (h + d) with d = (c ^ b) - c
// in [-255, 255], and c itself evolves alone: c' = ((c ^ b) * P) mod 256.  Over a block's n
// token bytes, from the state S reached after the parent's 8 bytes,
//     H = P^n S + D[S mod 256],   D[c] = sum_k P^(n-k) d_k  (the d_k of the chain started at c),
// and D depends only on the block's tokens.  Tables of D for every block and all 256 values of
// c are filled in parallel; a walk per request then needs, per block, the low-byte chain of
// the parent's 8 bytes, one shared-memory lookup and a sum.  Two ways to run it:
//  - tables, then the walk: a table kernel over the whole GPU (its CTA 0 also scans the
//    full-block counts into the output offsets), then per request a CTA whose producer warp
//    copies the tables into a shared-memory ring and whose walker warp runs the chain;
//  - both in one cooperative launch, when the walk is the longer part: walkers on SMs of their
//    own read each table once its flag is set by the CTAs computing them.
// Without a workspace, one CTA scans the counts and one thread per request runs the plain chain.
#include <algorithm>
#include <mutex>

#include "kv_async.cuh"
#include "kv_common.cuh"

#ifndef PKV_HASH_PDL
#define PKV_HASH_PDL 1  // 0: plain stream-ordered launches for every hash kernel
#endif
// After the table kernel, the walk runs one small CTA per request, and each request's chain of
// dependent blocks sets the call's time.  Launched early (programmatic dependent launch), an
// earlier single-warp walk's few CTAs were placed while the table kernel's last wave still held
// the SMs, on the few with room, and took 182 us instead of 100 us on 8 requests of 576 blocks;
// launched plainly they spread over idle SMs.  With a ring of 66 or 98 KiB per CTA, launching
// it early measured the same as plainly (84.3 vs 84.4 and 80.1 vs 80.3 us per call).
#ifndef PKV_HASH_WALK_PDL
#define PKV_HASH_WALK_PDL 0
#endif
constexpr bool kHashPdl = PKV_HASH_PDL;

namespace {

constexpr int kScanThreads = 1024;
constexpr uint64_t kFnvBasis = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;
static_assert(kFnvPrime == (1ull << 40) + 0x1b3u, "fnv_step multiplies by 2^40 + 0x1b3");

// FNV-1a state as two 32-bit halves.  One step h = (h ^ byte) * P with P = 2^40 + 0x1b3:
// modulo 2^64, h * 2^40 only moves the low half up by 8 bits into the high half, and h * 0x1b3
// is one 32x32->64 product of the low half plus a 32-bit product of the high half.  The low
// half's chain (xor, one wide multiply) is the critical path of the plain chain.
struct Fnv {
    uint32_t lo, hi;
};

__device__ __forceinline__ Fnv fnv_step(Fnv h, uint32_t byte)
{
    const uint32_t l = h.lo ^ byte;
    const uint64_t w = (uint64_t)l * 0x1b3u;
    return Fnv{(uint32_t)w, (uint32_t)(w >> 32) + h.hi * 0x1b3u + (l << 8)};
}

// The n low bytes of v, least significant first.
template <int N>
__device__ __forceinline__ Fnv fnv_bytes(Fnv h, uint64_t v)
{
#pragma unroll
    for (int j = 0; j < N; j++) h = fnv_step(h, (uint32_t)(v >> (8 * j)) & 0xffu);
    return h;
}

__device__ __forceinline__ uint64_t fnv_value(Fnv h) { return ((uint64_t)h.hi << 32) | h.lo; }

// State after the parent hash, the first 8 bytes of every block's input.
__device__ __forceinline__ Fnv fnv_block_start(uint64_t parent)
{
    return fnv_bytes<8>(Fnv{(uint32_t)kFnvBasis, (uint32_t)(kFnvBasis >> 32)}, parent);
}

// The full-block count of every request scanned into CSR offsets (global or shared memory) by
// one CTA of THREADS threads; with err, also flags offsets that do not describe n_tokens tokens.
template <int THREADS>
__device__ void count_blocks(const int32_t *__restrict__ off, int32_t n_reqs, int32_t n_tokens, int32_t bs,
                             int32_t *out_off, int *err)
{
    __shared__ int32_t warp_sum[THREADS / 32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        carry = 0;
        if (err != nullptr && (off[0] != 0 || off[n_reqs] != n_tokens)) pkv::set_error(err, KV_DERR_LIST);
    }
    __syncthreads();
    for (int32_t base = 0; base < n_reqs; base += THREADS) {
        const int32_t r = base + tid;
        int32_t cnt = 0;
        if (r < n_reqs) {
            const int64_t n = (int64_t)off[r + 1] - off[r];  // 64-bit: offsets may be anything
            if (n < 0 && err != nullptr) pkv::set_error(err, KV_DERR_LIST);
            cnt = n > 0 ? (int32_t)(n / bs) : 0;
        }
        int32_t incl = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += y;
        }
        if (lane == 31) warp_sum[warp] = incl;
        __syncthreads();
        int32_t before = 0, total = 0;
        for (int w = 0; w < THREADS / 32; w++) {
            if (w < warp) before += warp_sum[w];
            total += warp_sum[w];
        }
        if (r < n_reqs) out_off[r] = carry + before + incl - cnt;
        __syncthreads();
        if (tid == 0) carry += total;
        __syncthreads();
    }
    if (tid == 0) out_off[n_reqs] = carry;
}

__global__ void __launch_bounds__(kScanThreads) hash_count_kernel(const int32_t *__restrict__ off, int32_t n_reqs,
                                                                  int32_t n_tokens, int32_t bs, int32_t *out_off,
                                                                  int *err)
{
    pkv::grid_dep_entry();  // before any global memory access
    count_blocks<kScanThreads>(off, n_reqs, n_tokens, bs, out_off, err);
}

// Request r's span, block count and first hash index; false (and, with err, KV_DERR_LIST where
// the output range is at fault) when r is skipped.
__device__ __forceinline__ bool request_blocks(const int32_t *off, int32_t r, int32_t n_tokens, int32_t bs,
                                               const int32_t *out_off, int64_t limit, int *err, int32_t *begin,
                                               int32_t *k, int64_t *at)
{
    *begin = off[r];
    const int64_t n = (int64_t)off[r + 1] - *begin;  // 64-bit: offsets may be anything
    if (n <= 0 || *begin < 0 || *begin + n > n_tokens) return false;
    *k = (int32_t)(n / bs);
    *at = out_off[r];
    if (*at < 0 || *at + *k > limit) {
        if (err != nullptr) pkv::set_error(err, KV_DERR_LIST);
        return false;
    }
    return *k > 0;
}

// ---- without a workspace: one thread walks each request's bytes ----
constexpr int kChainThreads = 128;
#ifndef PKV_HASH_CHAIN_GROUP
#define PKV_HASH_CHAIN_GROUP 16  // token loads in flight ahead of the chain (1, 4, 16 measured; 16 best)
#endif

__global__ void __launch_bounds__(kChainThreads) hash_chain_kernel(const int32_t *__restrict__ off, int32_t n_reqs,
                                                                   const int32_t *__restrict__ tokens,
                                                                   int32_t n_tokens, int32_t bs, uint64_t seed,
                                                                   const int32_t *__restrict__ out_off,
                                                                   uint64_t *__restrict__ out, int64_t out_capacity,
                                                                   int *err)
{
    pkv::grid_dep_entry();  // before any global memory access
    for (int32_t r = blockIdx.x * blockDim.x + threadIdx.x; r < n_reqs; r += gridDim.x * blockDim.x) {
        int32_t begin, k;
        int64_t at;
        if (!request_blocks(off, r, n_tokens, bs, out_off, out_capacity, err, &begin, &k, &at)) continue;
        uint64_t parent = seed;
        const int32_t *t = tokens + begin;
        for (int32_t b = 0; b < k; b++) {
            Fnv h = fnv_block_start(parent);
            const int32_t *tb = t + (int64_t)b * bs;
            int32_t j = 0;
            // token loads issued a group at a time, ahead of the bytes entering the chain
            for (; j + PKV_HASH_CHAIN_GROUP <= bs; j += PKV_HASH_CHAIN_GROUP) {
                uint32_t v[PKV_HASH_CHAIN_GROUP];
#pragma unroll
                for (int q = 0; q < PKV_HASH_CHAIN_GROUP; q++) v[q] = (uint32_t)__ldg(tb + j + q);
#pragma unroll
                for (int q = 0; q < PKV_HASH_CHAIN_GROUP; q++) h = fnv_bytes<4>(h, v[q]);
            }
            for (; j < bs; j++) h = fnv_bytes<4>(h, (uint32_t)__ldg(tb + j));
            parent = fnv_value(h);
            out[at + b] = parent;
        }
    }
}

// ---- with a workspace: tables of D, then the walk ----
constexpr int kTableThreads = 256;  // one thread per table entry
constexpr int kTableChunk = 512;    // tokens per Horner chunk
constexpr int kTableUnits = 5;      // 3-token units whose loads are issued ahead of their bytes
constexpr int kOffCache = 1024;     // request offsets a table CTA keeps in shared memory
constexpr int kFusedScanMaxReqs = 4096;  // up to this many requests, table CTA 0 also scans the counts
constexpr uint32_t kTableBytes = 256 * sizeof(uint64_t);
#ifndef PKV_HASH_SEG
#define PKV_HASH_SEG 16  // tables per bulk copy of the walk
#endif
#ifndef PKV_HASH_SEGS
#define PKV_HASH_SEGS 4  // segments in the walk's shared-memory ring
#endif
constexpr int kSeg = PKV_HASH_SEG;
constexpr int kSegs = PKV_HASH_SEGS;
static_assert(kSeg >= 1 && kSeg <= 32 && kSegs >= 2, "walk ring shape");
constexpr uint32_t kWalkSmem = (uint32_t)(kSegs * kSeg + 1) * kTableBytes;  // + room to align the ring to 2 KiB

// 64-bit arithmetic modulo 2^64 for the table weights.
__host__ __device__ constexpr uint64_t pow_mod_2_64(uint64_t base, uint64_t e)
{
    uint64_t r = 1;
    while (e) {
        if (e & 1) r *= base;
        base *= base;
        e >>= 1;
    }
    return r;
}
__host__ __device__ constexpr uint64_t inverse_mod_2_64(uint64_t odd)
{
    uint64_t x = odd;  // correct to 3 bits; each Newton step doubles that
    for (int i = 0; i < 5; i++) x *= 2 - odd * x;
    return x;
}
constexpr uint64_t kPrimeInvPow256 = pow_mod_2_64(inverse_mod_2_64(kFnvPrime), kTableThreads);
static_assert(kFnvPrime * inverse_mod_2_64(kFnvPrime) == 1, "P is odd, so invertible modulo 2^64");

// A weight W split for two 32-bit multiply-adds per byte: lo_s is W's low word read as signed,
// hi = W's high word plus bit 31 of the low word, so that for any 32-bit signed d
//     d * W = d * lo_s + 2^32 * (d * hi)   (mod 2^64).
struct SplitWeight {
    int32_t lo_s;
    uint32_t hi;
};
__host__ __device__ constexpr SplitWeight split_weight(uint64_t w)
{
    return SplitWeight{(int32_t)(uint32_t)w, (uint32_t)(w >> 32) + ((uint32_t)w >> 31)};
}
__device__ __forceinline__ uint64_t join_weight(SplitWeight s)
{
    const uint32_t lo = (uint32_t)s.lo_s;
    return ((uint64_t)(s.hi - (lo >> 31)) << 32) | lo;
}

// Table layout.  Blocks are keyed by their slot, floor(first token / block size): a request's
// blocks then have consecutive slots, and no two blocks share one (request r's blocks end at
// or before off[r + 1], where the next request's first slot begins), so the tables fit in
// n_tokens / block size slots with no need for the output offsets.  Slot i's table holds, at
// entry x, D[(x * P) mod 256]: the entry for the state's low byte before the last multiply of
// the parent bytes, which saves the walk that multiply.
//
// D = sum_k P^(n-k) d_k is a weighted sum over the block's bytes in chunks of at most
// kTableChunk tokens, joined by Horner (D <- D * P^(chunk bytes) + chunk sum).  The weights
// P^(M - i), M = min(n, 4 kTableChunk), sit in shared memory; a chunk of m bytes uses the last m
// of them.  Per byte: a byte extract and xor and the chain's multiply; per three bytes, two
// 32-bit multiply-adds that give the group's sum from chain values, and the group's 64-bit
// multiply-add (a signed 32x32->64 and two 32-bit multiply-adds).  Tokens are read straight from
// global memory (the same address across the threads of a table), so a table needs no barrier.
constexpr int kTableChunkBytes = 4 * kTableChunk;

// The weights P^(M - i), i < M, into sh_w by the CTA's first 256 threads (a barrier must follow):
// thread tid takes i = tid, tid + 256, ..., stepping by P^-256.
__device__ __forceinline__ void fill_weights(SplitWeight *sh_w, int32_t M, int tid)
{
    if (tid < kTableThreads && tid < M) {
        uint64_t w = pow_mod_2_64(kFnvPrime, (uint64_t)(M - tid));
        for (int32_t i = tid; i < M; i += kTableThreads) {
            sh_w[i] = split_weight(w);  // P^(M - i)
            w *= kPrimeInvPow256;       // P^(M - i - 256)
        }
    }
}

// D for the block of bs tokens at tp and the starting low byte c0.
__device__ __forceinline__ uint64_t table_entry(const int32_t *__restrict__ tp, int32_t bs, uint32_t c0,
                                                const SplitWeight *sh_w, int32_t M)
{
    uint32_t c = c0;
    uint64_t D = 0;
    for (int32_t j0 = 0; j0 < bs; j0 += kTableChunk) {
        const int32_t m = min(kTableChunk, bs - j0);
        const SplitWeight *w = sh_w + (M - 4 * m);
        int64_t acc = 0;
        uint32_t acc_hi = 0;
        // c keeps the product's high bits: x and c then share all but their low byte, so
        // x - c is still the low bytes' difference, and x's low byte alone sets c's next one.
        // One token at a time (the last bs mod 3 tokens of a chunk):
        auto token = [&](uint32_t v, int32_t q) {
            // a token's 4 weights are 32 contiguous bytes (w + 4q is 32-byte aligned: chunks
            // start at a multiple of 4 weights): two 16-byte loads
            const uint4 w01 = *reinterpret_cast<const uint4 *>(w + 4 * q);
            const uint4 w23 = *reinterpret_cast<const uint4 *>(w + 4 * q + 2);
            const uint32_t wl[4] = {w01.x, w01.z, w23.x, w23.z}, wh[4] = {w01.y, w01.w, w23.y, w23.w};
#pragma unroll
            for (int byte = 0; byte < 4; byte++) {
                const uint32_t x = c ^ ((v >> (8 * byte)) & 0xffu);
                const int32_t d = (int32_t)x - (int32_t)c;
                acc += (int64_t)d * (int32_t)wl[byte];
                acc_hi += (uint32_t)d * wh[byte];
                c = x * 0x1b3u;
            }
        };
        // Three tokens (12 bytes) at a time, their bytes in groups of three sharing the last
        // byte's weight: W_j d_j + W_(j+1) d_(j+1) + W_(j+2) d_(j+2) = W_(j+2) v with
        // v = P^2 d_j + P d_(j+1) + d_(j+2), and modulo 2^64, P^2 = 870 * 2^40 + 189225, so
        // v = L + 2^40 Hh with L = 189225 d_j + 435 d_(j+1) + d_(j+2) (|L| < 2^26) and
        // Hh = 870 d_j + d_(j+1).  The chain keeps c' = 435 x exactly (mod 2^32), so these sums
        // telescope to chain values: L = x_(j+2) - 435^2 c_j and Hh = x_(j+1) + c_(j+1) - 870 c_j
        // (mod 2^32; L read as signed is exact).  One 64-bit multiply-add per three bytes.
        auto tokens3 = [&](uint32_t v0, uint32_t v1, uint32_t v2, int32_t q3) {
#pragma unroll
            for (int g = 0; g < 4; g++) {
                uint32_t cs[3], xs[3];
#pragma unroll
                for (int j = 0; j < 3; j++) {
                    const int i = 3 * g + j;
                    const uint32_t v = i < 4 ? v0 : (i < 8 ? v1 : v2);
                    cs[j] = c;
                    xs[j] = c ^ ((v >> (8 * (i & 3))) & 0xffu);
                    c = xs[j] * 0x1b3u;
                }
                const int32_t L = (int32_t)(xs[2] - 189225u * cs[0]);
                const uint32_t Hh = xs[1] + cs[1] - 870u * cs[0];
                const SplitWeight wt = w[4 * q3 + 3 * g + 2];
                acc += (int64_t)L * wt.lo_s;
                acc_hi += (uint32_t)L * wt.hi + ((Hh * (uint32_t)wt.lo_s) << 8);
            }
        };
        int32_t q = 0;
        for (; q + 3 * kTableUnits <= m; q += 3 * kTableUnits) {
            uint32_t v[3 * kTableUnits];
#pragma unroll
            for (int g = 0; g < 3 * kTableUnits; g++) v[g] = (uint32_t)__ldg(tp + j0 + q + g);
#pragma unroll
            for (int u = 0; u < kTableUnits; u++) tokens3(v[3 * u], v[3 * u + 1], v[3 * u + 2], q + 3 * u);
        }
        for (; q + 3 <= m; q += 3)
            tokens3((uint32_t)__ldg(tp + j0 + q), (uint32_t)__ldg(tp + j0 + q + 1), (uint32_t)__ldg(tp + j0 + q + 2), q);
        for (; q < m; q++) token((uint32_t)__ldg(tp + j0 + q), q);
        D = D * join_weight(w[0]) + (uint64_t)acc + ((uint64_t)acc_hi << 32);
    }
    return D;
}

// The table kernel: slot i, i = blockIdx.x, + gridDim.x, ...; the block (if any) that starts in
// tokens [i * bs, (i + 1) * bs) belongs to the request holding token (i + 1) * bs - 1.  When scan
// is set, CTA 0 first writes the output offsets.
__global__ void __launch_bounds__(kTableThreads) hash_table_kernel(const int32_t *__restrict__ off, int32_t n_reqs,
                                                                   const int32_t *__restrict__ tokens,
                                                                   int32_t n_tokens, int32_t bs, int32_t *out_off,
                                                                   uint64_t *__restrict__ table, int32_t n_slots,
                                                                   pkv::FastDiv div_bs, bool scan, int *err)
{
    pkv::grid_dep_entry();  // before any global memory access
    __shared__ __align__(16) SplitWeight sh_w[kTableChunkBytes];
    __shared__ int32_t sh_off[kOffCache + 1];
    if (scan && blockIdx.x == 0) count_blocks<kTableThreads>(off, n_reqs, n_tokens, bs, out_off, err);
    const int tid = threadIdx.x;
    const bool cached = n_reqs <= kOffCache;
    if (cached)
        for (int i = tid; i <= n_reqs; i += kTableThreads) sh_off[i] = off[i];
    const int32_t M = min(4 * bs, kTableChunkBytes);
    fill_weights(sh_w, M, tid);
    __syncthreads();
    const uint32_t c0 = ((uint32_t)tid * 0xb3u) & 0xffu;  // this thread's low byte of the state
    for (int32_t i = blockIdx.x; i < n_slots; i += gridDim.x) {
        const int64_t t = (int64_t)i * bs;
        const int64_t last = t + bs - 1;
        int32_t lo = 0, hi = n_reqs - 1;  // the last request r with off[r] <= last
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if ((cached ? sh_off[mid] : off[mid]) <= last) lo = mid;
            else hi = mid - 1;
        }
        const int64_t o = cached ? sh_off[lo] : off[lo];
        const int64_t o1 = cached ? sh_off[lo + 1] : off[lo + 1];
        if (o > last) continue;  // (offsets out of order)
        // the one token of the window at a block boundary of r: o + floor((last - o) / bs) * bs
        const int64_t first = o + (int64_t)pkv::fdiv((uint32_t)(last - o), div_bs) * bs;
        if (first + bs > o1 || first + bs > n_tokens) continue;  // no block starts here
        table[(int64_t)i * 256 + tid] = table_entry(tokens + first, bs, c0, sh_w, M);
    }
}

// The walk's constants for n token bytes per block: the hash of a block is
//     H = K0 + sum_{k<8} W_k e_k + T[x]
// with K0 = P^(n+8) basis, W_k = P^(n+8-k), e_k the k-th parent byte's low-byte difference
// (the state is P^8 basis + sum_k P^(8-k) e_k after the parent bytes, and the tokens then
// multiply it by P^n) and T the slot's table at x, the low byte before the last multiply.
struct WalkConsts {
    uint64_t k0;
    SplitWeight w[8];
};

using pkv::kWaitLimitNs;
using pkv::mbar_init;
using pkv::mbar_wait;
using pkv::now_ns;
using pkv::smem_addr;

__device__ __forceinline__ int32_t ld_flag(const int32_t *p)
{
    int32_t v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// One block of the walk from parent h; tab is the shared address of the block's table (2 KiB
// aligned).  The critical path is the low-byte chain of the parent's bytes (an xor and a
// multiply per byte), the table load and an add; the rest of H is summed beside it.  The
// chain's value keeps the product's high bits, which the xor with a byte leaves alone, so
// x - c is exact.  The last multiply uses 8 P, putting the low byte at bits 3..10 where it is
// the table entry's byte offset.
__device__ __forceinline__ uint64_t walk_block(uint64_t h, const WalkConsts &wc, uint32_t tab)
{
    const uint32_t lo = (uint32_t)h, hi = (uint32_t)(h >> 32);
    uint32_t c = (uint32_t)kFnvBasis;
    int32_t e[8];
#pragma unroll
    for (int k = 0; k < 7; k++) {
        const uint32_t x = c ^ (((k < 4 ? lo : hi) >> (8 * (k & 3))) & 0xffu);
        e[k] = (int32_t)(x - c);
        c = x * (k < 6 ? 0x1b3u : 8u * 0x1b3u);
    }
    const uint32_t p7 = (hi >> 21) & 0x7f8u;  // the last parent byte, times 8
    e[7] = (int32_t)((c ^ p7) - c) >> 3;
    const uint32_t addr = (c & 0x7f8u) ^ (p7 | tab);  // tab + 8 * (the low byte after the xor)
    uint64_t t;
    asm volatile("ld.shared.u64 %0, [%1];" : "=l"(t) : "r"(addr));
    int64_t acc = (int64_t)wc.k0;
    uint32_t acc_hi = 0;
#pragma unroll
    for (int k = 0; k < 8; k++) {
        acc += (int64_t)e[k] * wc.w[k].lo_s;
        acc_hi += (uint32_t)e[k] * wc.w[k].hi;
    }
    return (uint64_t)acc + ((uint64_t)acc_hi << 32) + t;
}

// The walk of requests r0, r0 + r_step, ... by two warps of a CTA.  The tables of a request go
// through a ring of kSegs segments of kSeg tables in shared memory (ring: its 2 KiB aligned
// shared address), one bulk copy (cp.async.bulk) per segment.  Warp 1, the producer, issues the
// copies up to kSegs segments ahead: it waits for the segment's slot to be released (mbarrier
// empty[slot]), and with FLAGS (the tables still being written by other CTAs) until the flags of
// all its tables are set, after which an acquire fence and a proxy fence make the tables visible
// to the bulk copy; completion is counted on mbarrier full[slot].  Warp 0, the walker, waits
// for full[slot], walks the segment's blocks (every lane runs the same chain, lane 0 stores each
// hash; a full segment has no bound check per block) and releases the slot.  The fences and
// flag polls thus stay off the walker, and both warps go through the same sequence of
// (request, segment), numbered G across requests: slot G % kSegs, use G / kSegs.  A wait that
// runs out (2 s) sets KV_DERR_TIMEOUT and ends that warp's walk; the producer then waits,
// bounded again, for its copies still in flight.
template <bool FLAGS>
__device__ void walk_requests(int32_t r0, int32_t r_step, const int32_t *__restrict__ off, int32_t n_reqs,
                              int32_t n_tokens, int32_t bs, uint64_t seed, const WalkConsts &wc, const int32_t *at_of,
                              int64_t limit, const uint64_t *__restrict__ table, const int32_t *flags,
                              uint64_t *__restrict__ out, int *err, uint32_t ring, const uint64_t *full,
                              const uint64_t *empty)
{
    const int lane = threadIdx.x & 31;
    const bool producer = (threadIdx.x >> 5) == 1;
    uint32_t G = 0;  // segments of this CTA so far
    for (int32_t r = r0; r < n_reqs; r += r_step) {
        int32_t begin, k;
        int64_t at;
        if (!request_blocks(off, r, n_tokens, bs, at_of, limit, producer ? nullptr : err, &begin, &k, &at)) continue;
        const int32_t slot0 = begin / bs;
        const int32_t nseg = (k + kSeg - 1) / kSeg;
        if (producer) {
            for (int32_t s = 0; s < nseg; s++, G++) {
                const uint32_t slot = G % kSegs, use = G / kSegs;
                bool ok = use == 0 || __all_sync(0xffffffffu, mbar_wait(smem_addr(&empty[slot]), (use - 1) & 1u));
                if (ok && FLAGS) {
                    const int32_t j = s * kSeg + lane;
                    const bool mine = lane < kSeg && j < k;
                    const unsigned long long t0 = now_ns();
                    while (!__all_sync(0xffffffffu, !mine || ld_flag(flags + slot0 + j) != 0))
                        if (__shfl_sync(0xffffffffu, now_ns() - t0 > kWaitLimitNs, 0)) {
                            ok = false;
                            break;
                        }
                    if (ok) {
                        asm volatile("fence.acq_rel.gpu;" ::: "memory");
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                    }
                }
                if (!ok) {  // let the copies still in flight land before shared memory goes away
                    if (lane == 0) pkv::set_error(err, KV_DERR_TIMEOUT);
                    for (uint32_t g = G > kSegs ? G - kSegs : 0; g < G; g++)
                        mbar_wait(smem_addr(&full[g % kSegs]), (g / kSegs) & 1u);
                    return;
                }
                const uint32_t bytes = (uint32_t)min(kSeg, k - s * kSeg) * kTableBytes;
                asm volatile(  // issued by lane 0 (predicated, no branch)
                    "{\n\t.reg .pred p;\n\t"
                    "setp.eq.u32 p, %0, 0;\n\t"
                    "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%1], %2;\n\t"
                    "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%3], [%4], %2, [%1];\n\t"
                    "}" ::"r"(lane),
                    "r"(smem_addr(&full[slot])), "r"(bytes), "r"(ring + slot * (uint32_t)(kSeg * kTableBytes)),
                    "l"(table + ((int64_t)slot0 + (int64_t)s * kSeg) * 256)
                    : "memory");
            }
            continue;
        }
        uint64_t h = seed;
        for (int32_t s = 0; s < nseg; s++, G++) {
            const uint32_t slot = G % kSegs, use = G / kSegs;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&full[slot]), use & 1u))) {
                if (lane == 0) pkv::set_error(err, KV_DERR_TIMEOUT);
                return;
            }
            const uint32_t seg = ring + slot * (uint32_t)(kSeg * kTableBytes);
            const int32_t j0 = s * kSeg;
            if (j0 + kSeg <= k) {  // a full segment: no bound per block
#pragma unroll
                for (int q = 0; q < kSeg; q++) {
                    h = walk_block(h, wc, seg + (uint32_t)q * kTableBytes);
                    if (lane == 0) out[at + j0 + q] = h;
                }
            } else {
#pragma unroll 1
                for (int q = 0; j0 + q < k; q++) {
                    h = walk_block(h, wc, seg + (uint32_t)q * kTableBytes);
                    if (lane == 0) out[at + j0 + q] = h;
                }
            }
            __syncwarp();  // every lane has read the segment before it is released
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "setp.eq.u32 p, %0, 0;\n\t"
                "@p mbarrier.arrive.shared::cta.b64 _, [%1];\n\t}" ::"r"(lane),
                "r"(smem_addr(&empty[slot]))
                : "memory");
        }
    }
}

// The ring's 2 KiB aligned shared address and its barriers' initialisation (by thread 0, then a
// CTA barrier over the walk's two warps).
__device__ __forceinline__ uint32_t walk_ring_setup(const uint8_t *walk_smem, uint64_t *full, uint64_t *empty)
{
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSegs; s++) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("bar.sync 1, 64;" ::: "memory");
    return (smem_addr(walk_smem) + kTableBytes - 1) & ~(kTableBytes - 1);
}

// The walk after the table kernel: a CTA of two warps per request.
constexpr int kWalkThreads = 64;

__global__ void __launch_bounds__(kWalkThreads) hash_walk_kernel(const int32_t *__restrict__ off, int32_t n_reqs,
                                                                 int32_t n_tokens, int32_t bs, uint64_t seed,
                                                                 const __grid_constant__ WalkConsts wc,
                                                                 const int32_t *__restrict__ out_off,
                                                                 const uint64_t *__restrict__ table, int64_t limit,
                                                                 uint64_t *__restrict__ out, int *err)
{
    pkv::grid_dep_entry();  // before any global memory access
    extern __shared__ __align__(16) uint8_t walk_smem[];
    __shared__ __align__(8) uint64_t full[kSegs], empty[kSegs];
    const uint32_t ring = walk_ring_setup(walk_smem, full, empty);
    walk_requests<false>(blockIdx.x, gridDim.x, off, n_reqs, n_tokens, bs, seed, wc, out_off, limit, table, nullptr,
                         out, err, ring, full, empty);
}

// ---- the table kernel and the walk in one cooperative launch ----
// One CTA per SM (its shared memory holds a whole walk ring).  CTAs below n_walk walk request
// blockIdx.x, + n_walk, ... on their own SMs with a walker and a producer warp (they first scan
// the counts themselves, and CTA 0 writes the output offsets).  The other CTAs compute tables, a group of 256 threads per
// table, in block-position order (block 0 of every request, then block 1, ...) so the walks
// find their tables ready; a group publishes a table's flag once it has computed its next one,
// so the release fence finds the table's stores long done.  The flags (one int per slot, after
// the tables in the workspace) are cleared before the launch.
constexpr int kFusedThreads = 1024;
constexpr int kFusedGroups = kFusedThreads / kTableThreads;

__device__ __forceinline__ void group_sync(int g)
{
    asm volatile("bar.sync %0, %1;" ::"r"(g + 1), "n"(kTableThreads) : "memory");
}

__device__ __forceinline__ void publish(int32_t *flag)
{
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(flag), "r"(1) : "memory");
}

__global__ void __launch_bounds__(kFusedThreads, 1) hash_fused_kernel(
    const int32_t *__restrict__ off, int32_t n_reqs, const int32_t *__restrict__ tokens, int32_t n_tokens,
    int32_t bs, pkv::FastDiv div_bs, uint64_t seed, const __grid_constant__ WalkConsts wc, int32_t *out_off,
    uint64_t *__restrict__ table, int32_t *flags, int32_t n_walk, int64_t limit, uint64_t *__restrict__ out, int *err)
{
    pkv::grid_dep_entry();  // before any global memory access
    extern __shared__ __align__(16) uint8_t walk_smem[];
    __shared__ __align__(16) SplitWeight sh_w[kTableChunkBytes];
    __shared__ int32_t sh_off[kOffCache + 1];
    __shared__ __align__(8) uint64_t full[kSegs], empty[kSegs];
    __shared__ int32_t sh_max_k;
    const int tid = threadIdx.x;
    if ((int32_t)blockIdx.x < n_walk) {
        // sh_off serves as this CTA's copy of the output offsets
        count_blocks<kFusedThreads>(off, n_reqs, n_tokens, bs, sh_off, blockIdx.x == 0 ? err : nullptr);
        __syncthreads();
        if (blockIdx.x == 0)
            for (int i = tid; i <= n_reqs; i += kFusedThreads) out_off[i] = sh_off[i];
        if (tid >= kWalkThreads) return;
        const uint32_t ring = walk_ring_setup(walk_smem, full, empty);
        walk_requests<true>(blockIdx.x, n_walk, off, n_reqs, n_tokens, bs, seed, wc, sh_off, limit, table, flags, out,
                            err, ring, full, empty);
        return;
    }
    for (int i = tid; i <= n_reqs; i += kFusedThreads) sh_off[i] = off[i];
    const int32_t M = min(4 * bs, kTableChunkBytes);
    fill_weights(sh_w, M, tid);
    if (tid == 0) sh_max_k = 0;
    __syncthreads();
    for (int r = tid; r < n_reqs; r += kFusedThreads) {  // the most full blocks of any request
        const int32_t o = sh_off[r];
        const int64_t n = (int64_t)sh_off[r + 1] - o;  // the same test as the walks' request_blocks
        if (n > 0 && o >= 0 && o + n <= n_tokens) atomicMax(&sh_max_k, (int32_t)pkv::fdiv((uint32_t)n, div_bs));
    }
    __syncthreads();
    const int g = tid / kTableThreads, ti = tid % kTableThreads;
    const uint32_t c0 = ((uint32_t)ti * 0xb3u) & 0xffu;
    // this group's items: (block b, request r) = w, w + W, ... of b * n_reqs + r
    const int64_t W = (int64_t)(gridDim.x - n_walk) * kFusedGroups;
    const int64_t n_items = (int64_t)n_reqs * sh_max_k;
    const int64_t w0 = (int64_t)(blockIdx.x - n_walk) * kFusedGroups + g;
    int64_t b = w0 / n_reqs;
    int32_t r = (int32_t)(w0 % n_reqs);
    const int64_t step_b = W / n_reqs;
    const int32_t step_r = (int32_t)(W % n_reqs);
    int32_t prev = -1;  // the slot computed last, not yet published
    bool first = true;
    for (int64_t item = w0; item < n_items; item += W) {
        const int32_t o = sh_off[r];
        const int64_t n = (int64_t)sh_off[r + 1] - o;
        const int64_t kr = (n > 0 && o >= 0 && o + n <= n_tokens) ? pkv::fdiv((uint32_t)n, div_bs) : 0;
        if (b < kr) {
            const int32_t slot = (int32_t)(pkv::fdiv((uint32_t)o, div_bs) + b);
            const uint64_t D = table_entry(tokens + o + b * bs, bs, c0, sh_w, M);
            group_sync(g);  // the group's stores of the previous table are all issued
            if (ti == 0 && prev >= 0) publish(flags + prev);
            table[(int64_t)slot * 256 + ti] = D;
            prev = slot;
            if (first) {  // the walks are waiting for the first tables: publish this one at once
                group_sync(g);
                if (ti == 0) publish(flags + slot);
                prev = -1;
                first = false;
            }
        }
        b += step_b;
        r += step_r;
        if (r >= n_reqs) {
            r -= n_reqs;
            b++;
        }
    }
    group_sync(g);
    if (ti == 0 && prev >= 0) publish(flags + prev);
}

}  // namespace

int pkv::preload_hash_kernels()
{
    return pkv::load_kernels(hash_count_kernel, hash_chain_kernel, hash_table_kernel, hash_walk_kernel,
                             hash_fused_kernel);
}

namespace {

// Workspace: the tables (2 KiB per slot), then one flag per slot for the fused launch.
int64_t tables_bytes(int64_t n_slots) { return n_slots * (int64_t)kTableBytes; }
int64_t fused_workspace_bytes(int64_t n_slots)
{
    return (tables_bytes(n_slots) + n_slots * (int64_t)sizeof(int32_t) + 15) & ~(int64_t)15;
}

// Per device, once: both walk kernels may use a whole ring of shared memory, and whether the
// fused launch can run (cooperative launches supported, one CTA fits on an SM).
int prepare_device(const pkv::DeviceInfo *dev, bool *fused_ok)
{
    static std::mutex mu;
    static bool done[64], ok[64];
    std::lock_guard<std::mutex> lock(mu);
    const int d = dev->device & 63;
    if (!done[d]) {
        int st = pkv::cuda_status(
            cudaFuncSetAttribute(hash_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWalkSmem));
        if (st == KV_OK)
            st = pkv::cuda_status(
                cudaFuncSetAttribute(hash_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWalkSmem));
        int coop = 0, per_sm = 0;
        if (st == KV_OK) st = pkv::cuda_status(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev->device));
        if (st == KV_OK)
            st = pkv::cuda_status(
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, hash_fused_kernel, kFusedThreads, kWalkSmem));
        if (st != KV_OK) return st;
        ok[d] = coop != 0 && per_sm >= 1;
        done[d] = true;
    }
    *fused_ok = ok[d];
    return KV_OK;
}

// Whether the fused launch pays.  Its walkers take n_reqs SMs from the tables.  On GB300 the tables
// cost about 0.064 us x SM per token and the walk about 0.08 us per block of the longest request,
// which holds at least n_slots / n_reqs blocks; the fused launch is taken when the tables' loss,
// T_tables * n_reqs / (S - n_reqs), stays under half the walk:
//     bs * 0.064 * n_reqs^2 < 0.5 * 0.08 * S * (S - n_reqs),  i.e.  8 bs n_reqs^2 < 5 S (S - n_reqs).
// (8 prompts of 576 blocks of 16 tokens: fused; 32 requests of 64-token blocks: tables then walk.)
bool fused_pays(int32_t bs, int32_t n_reqs, int num_sms)
{
    if (n_reqs > num_sms / 4) return false;
    return 8ll * bs * n_reqs * n_reqs < 5ll * num_sms * (num_sms - n_reqs);
}

}  // namespace

extern "C" int kv_block_hashes_workspace_bytes(int64_t n_tokens, int32_t block_size, int64_t *bytes_out)
{
    if (bytes_out == nullptr || n_tokens < 0 || block_size <= 0) return KV_ERR_INVALID_ARG;
    *bytes_out = fused_workspace_bytes(n_tokens / block_size);
    return KV_OK;
}

extern "C" int kv_block_hashes(const int32_t *tok_offsets, int32_t n_reqs, const int32_t *tokens, int64_t n_tokens,
                               int32_t block_size, uint64_t seed, int32_t *out_offsets, uint64_t *out_hashes,
                               int64_t out_capacity, void *workspace, int64_t workspace_bytes, kv_stream_t stream)
{
    if (n_reqs < 0 || n_tokens < 0 || block_size <= 0 || out_capacity < 0 || tok_offsets == nullptr ||
        out_offsets == nullptr || workspace_bytes < 0)
        return KV_ERR_INVALID_ARG;
    if (n_tokens >= (1ll << 31)) return KV_ERR_UNSUPPORTED;
    if (n_tokens > 0 && (tokens == nullptr || n_reqs == 0)) return KV_ERR_INVALID_ARG;
    if (out_capacity < n_tokens / block_size) return KV_ERR_RANGE;
    if (out_capacity > 0 && out_hashes == nullptr) return KV_ERR_INVALID_ARG;
    if (((uintptr_t)out_hashes & 7u) != 0) return KV_ERR_ALIGN;
    const int32_t n_slots = (int32_t)(n_tokens / block_size);  // out_capacity >= n_slots (checked above)
    if (workspace != nullptr) {
        if (!pkv::aligned16(workspace)) return KV_ERR_ALIGN;
        if (workspace_bytes < tables_bytes(n_slots)) return KV_ERR_RANGE;
    }
    const pkv::DeviceInfo *dev = pkv::current_device();
    if (dev == nullptr) return KV_ERR_CUDA;
    const cudaStream_t s = (cudaStream_t)stream;
    if (n_reqs == 0) return pkv::cuda_status(cudaMemsetAsync(out_offsets, 0, sizeof(int32_t), s));
    const bool table_path = workspace != nullptr && n_slots > 0;
    bool fused_ok = false;
    int st = KV_OK;
    if (table_path) {
        st = prepare_device(dev, &fused_ok);
        if (st != KV_OK) return st;
    }
    const bool fused = table_path && fused_ok && workspace_bytes >= fused_workspace_bytes(n_slots) &&
                       n_reqs <= kOffCache && fused_pays(block_size, n_reqs, dev->num_sms);
    const bool fused_scan = table_path && n_reqs <= kFusedScanMaxReqs;  // the two-kernel path's table CTA 0 scans
    if (!table_path || !fused_scan) {
        pkv::launch<kHashPdl>(hash_count_kernel, 1, kScanThreads, 0, s, tok_offsets, n_reqs, (int32_t)n_tokens,
                              block_size, out_offsets, dev->err_word);
        st = pkv::cuda_status(cudaGetLastError());
        if (st != KV_OK) return st;
    }
    if (workspace == nullptr) {
        const int blocks = std::max(1, std::min((n_reqs + kChainThreads - 1) / kChainThreads, dev->num_sms * 4));
        pkv::launch<kHashPdl>(hash_chain_kernel, blocks, kChainThreads, 0, s, tok_offsets, n_reqs, tokens,
                              (int32_t)n_tokens, block_size, seed, out_offsets, out_hashes, out_capacity,
                              dev->err_word);
        return pkv::cuda_status(cudaGetLastError());
    }
    if (n_slots == 0) return KV_OK;
    uint64_t *table = reinterpret_cast<uint64_t *>(workspace);
    const pkv::FastDiv div_bs = pkv::make_fastdiv((uint32_t)block_size);
    WalkConsts wc{};
    const uint64_t n8 = 4ull * (uint64_t)block_size + 8;  // bytes hashed per block
    wc.k0 = pow_mod_2_64(kFnvPrime, n8) * kFnvBasis;
    for (int k = 0; k < 8; k++) wc.w[k] = split_weight(pow_mod_2_64(kFnvPrime, n8 - (uint64_t)k));
    if (fused) {
        int32_t *flags = reinterpret_cast<int32_t *>(reinterpret_cast<uint8_t *>(workspace) + tables_bytes(n_slots));
        st = pkv::cuda_status(cudaMemsetAsync(flags, 0, (size_t)n_slots * sizeof(int32_t), s));
        if (st != KV_OK) return st;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)dev->num_sms);
        cfg.blockDim = dim3(kFusedThreads);
        cfg.dynamicSmemBytes = kWalkSmem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, hash_fused_kernel, tok_offsets, n_reqs, tokens,
                                                 (int32_t)n_tokens, block_size, div_bs, seed, wc, out_offsets, table,
                                                 flags, n_reqs, out_capacity, out_hashes, dev->err_word);
        if (e != cudaErrorCooperativeLaunchTooLarge) return pkv::cuda_status(e);
        // not all SMs are free (another context holds some): tables, then the walk (fused implies
        // n_reqs <= kFusedScanMaxReqs, so the table kernel writes the output offsets)
        (void)cudaGetLastError();
    }
    const int table_blocks = std::min(n_slots, dev->num_sms * 8);
    pkv::launch<kHashPdl>(hash_table_kernel, table_blocks, kTableThreads, 0, s, tok_offsets, n_reqs, tokens,
                          (int32_t)n_tokens, block_size, out_offsets, table, n_slots, div_bs, fused_scan,
                          dev->err_word);
    st = pkv::cuda_status(cudaGetLastError());
    if (st != KV_OK) return st;
    const int walk_blocks = std::min(n_reqs, dev->num_sms * 16);
    pkv::launch<kHashPdl && PKV_HASH_WALK_PDL>(hash_walk_kernel, walk_blocks, kWalkThreads, kWalkSmem, s, tok_offsets, n_reqs,
                                               (int32_t)n_tokens, block_size, seed, wc, out_offsets, table,
                                               out_capacity, out_hashes, dev->err_word);
    return pkv::cuda_status(cudaGetLastError());
}
