// kv_block_hashes: the prefix hash chain over full token blocks.
//
// Drawing "vllm v1 调度逻辑 和 distributed 分布式原理", the hash-table labels: every full block is
// keyed by h0 = hash(seed, [t0 .. t(bs-1)]) and h_i = hash(h_(i-1), [tokens of block i]), so
// equal prefixes give equal keys (cached_block_hash_to_block).  The pages do not name the hash;
// the reading implemented here is FNV-1a 64 over the parent hash as 8 little-endian bytes
// followed by the block's token ids as 4 little-endian bytes each.  Only full blocks are hashed.
//
// FNV-1a is byte-serial and each block starts from its parent's hash, so a request's chain is
// sequential.  One CTA first scans the full-block counts into the output CSR offsets.  Then,
// with a workspace, two kernels split each block's hash by a property of FNV-1a: the xor of a
// byte only changes the state's low byte c, so a step is h' = P (h + d) with d = (c ^ b) - c
// in [-255, 255], and c itself evolves alone: c' = ((c ^ b) * P) mod 256.  Over a block's n
// token bytes, from the state S reached after the parent's 8 bytes,
//     H = P^n S + D[S mod 256],   D[c] = sum_k P^(n-k) d_k  (the d_k of the chain started at c),
// and D depends only on the block's tokens.  The table kernel fills D for every block and all
// 256 values of c at once, spread over the whole GPU; the walker then needs, per block, only
// parent's 8 byte steps, one shared-memory lookup and a multiply-add.  Without a workspace one
// thread per request runs the plain byte chain.
#include <algorithm>
#include <mutex>

#include "kv_common.cuh"

#ifndef PKV_HASH_W128
#define PKV_HASH_W128 1  // 0: the table kernel loads each byte's weight on its own
#endif
#ifndef PKV_HASH_PDL
#define PKV_HASH_PDL 1  // 0: plain stream-ordered launches for every hash kernel
#endif
// The walk runs one single-warp CTA per request, and each request's chain of dependent blocks
// sets the call's time.  Launched early (programmatic dependent launch), those few CTAs are
// placed while the table kernel's last wave still holds the SMs, on the few with room, and the
// walk took 182 us instead of 100 us on 8 requests of 576 blocks; launched plainly they spread
// over idle SMs.
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
// half's chain (xor, one wide multiply) is the critical path of the whole hash.
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

__global__ void __launch_bounds__(kScanThreads) hash_count_kernel(const int32_t *__restrict__ off, int32_t n_reqs,
                                                                  int32_t n_tokens, int32_t bs, int32_t *out_off,
                                                                  int *err)
{
    pkv::grid_dep_entry();  // before any global memory access
    __shared__ int32_t warp_sum[kScanThreads / 32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        carry = 0;
        if (off[0] != 0 || off[n_reqs] != n_tokens) pkv::set_error(err, KV_DERR_LIST);
    }
    __syncthreads();
    for (int32_t base = 0; base < n_reqs; base += kScanThreads) {
        const int32_t r = base + tid;
        int32_t cnt = 0;
        if (r < n_reqs) {
            const int32_t n = off[r + 1] - off[r];
            if (n < 0) pkv::set_error(err, KV_DERR_LIST);
            cnt = n > 0 ? n / bs : 0;
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
        for (int w = 0; w < kScanThreads / 32; w++) {
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

// Request r's span, block count and first hash index; false (and KV_DERR_LIST where the output
// range is at fault) when r is skipped.
__device__ __forceinline__ bool request_blocks(const int32_t *off, int32_t r, int32_t n_tokens, int32_t bs,
                                               const int32_t *out_off, int64_t limit, int *err, int32_t *begin,
                                               int32_t *k, int64_t *at)
{
    *begin = off[r];
    const int32_t n = off[r + 1] - *begin;
    if (n <= 0 || *begin < 0 || *begin + n > n_tokens) return false;
    *k = n / bs;
    *at = out_off[r];
    if (*at < 0 || *at + *k > limit) {
        pkv::set_error(err, KV_DERR_LIST);
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
constexpr int kTableThreads = 256;  // one thread per starting low byte c
constexpr int kTableChunk = 512;    // tokens staged in shared memory at a time
#ifndef PKV_HASH_RING
#define PKV_HASH_RING 8
#endif
#ifndef PKV_HASH_BATCH
#define PKV_HASH_BATCH 4
#endif
constexpr int kRing = PKV_HASH_RING;  // tables in flight per walking warp

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
__device__ __forceinline__ SplitWeight split_weight(uint64_t w)
{
    const uint32_t lo = (uint32_t)w;
    return SplitWeight{(int32_t)lo, (uint32_t)(w >> 32) + (lo >> 31)};
}
__device__ __forceinline__ uint64_t join_weight(SplitWeight s)
{
    const uint32_t lo = (uint32_t)s.lo_s;
    return ((uint64_t)(s.hi - (lo >> 31)) << 32) | lo;
}

// Block g's table: D[c] for c = threadIdx.x.  Blocks are numbered by their hash index; a CTA
// takes blocks g = blockIdx.x, + gridDim.x, ... below min(hash count, limit).
// D = sum_k P^(n-k) d_k is taken as a weighted sum over the block's bytes in chunks of at most
// kTableChunkBytes, joined by Horner (D <- D * P^(chunk bytes) + chunk sum).  The weights
// P^(M - i), M = min(n, kTableChunkBytes), are computed once per CTA into shared memory; a
// chunk of m bytes uses the last m of them.  Per byte: a byte extract and xor, one
// subtraction, a signed 32x32->64 multiply-add, a 32-bit multiply-add, and the chain's multiply.
constexpr int kTableChunkBytes = 4 * kTableChunk;

__global__ void __launch_bounds__(kTableThreads) hash_table_kernel(const int32_t *__restrict__ off, int32_t n_reqs,
                                                                   const int32_t *__restrict__ tokens,
                                                                   int32_t n_tokens, int32_t bs,
                                                                   const int32_t *__restrict__ out_off,
                                                                   uint64_t *__restrict__ table, int64_t limit)
{
    pkv::grid_dep_entry();  // before any global memory access
    __shared__ uint32_t sh_tok[kTableChunk];
    __shared__ __align__(16) SplitWeight sh_w[kTableChunkBytes];
    const int64_t n_hash = min((int64_t)out_off[n_reqs], limit);
    const uint32_t c0 = threadIdx.x;
    const int32_t nb = 4 * bs;  // token bytes per block
    const int32_t M = min(nb, kTableChunkBytes);
    if ((int32_t)c0 < M) {
        uint64_t w = pow_mod_2_64(kFnvPrime, (uint64_t)(M - (int32_t)c0));
        for (int32_t i = c0; i < M; i += kTableThreads) {
            sh_w[i] = split_weight(w);  // P^(M - i)
            w *= kPrimeInvPow256;       // P^(M - i - 256)
        }
    }
    for (int64_t g = blockIdx.x; g < n_hash; g += gridDim.x) {
        int32_t lo = 0, hi = n_reqs - 1;  // the request holding hash g: last r with out_off[r] <= g
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (out_off[mid] <= g) lo = mid;
            else hi = mid - 1;
        }
        const int32_t begin = off[lo];
        const int64_t first = (int64_t)begin + (g - out_off[lo]) * (int64_t)bs;  // the block's first token
        const bool ok = begin >= 0 && first >= 0 && first + bs <= n_tokens && off[lo + 1] - begin >= 0;
        uint32_t c = c0;
        uint64_t D = 0;
        for (int32_t j0 = 0; j0 < bs; j0 += kTableChunk) {
            const int32_t m = min(kTableChunk, bs - j0);
            const SplitWeight *w = sh_w + (M - 4 * m);
            __syncthreads();  // the previous chunk has been read (and, the first time, the weights written)
            for (int q = threadIdx.x; q < m; q += kTableThreads) sh_tok[q] = ok ? (uint32_t)tokens[first + j0 + q] : 0u;
            __syncthreads();
            int64_t acc = 0;
            uint32_t acc_hi = 0;
            // c keeps the product's high bits: x and c then share all but their low byte, so
            // x - c is still the low bytes' difference, and x's low byte alone sets c's next one.
#pragma unroll 2
            for (int q = 0; q < m; q++) {
                const uint32_t v = sh_tok[q];
#if PKV_HASH_W128
                // a token's 4 weights are 32 contiguous bytes (w + 4q is 32-byte aligned: chunks
                // start at a multiple of 4 weights): two 16-byte loads instead of four 8-byte ones
                const uint4 w01 = *reinterpret_cast<const uint4 *>(w + 4 * q);
                const uint4 w23 = *reinterpret_cast<const uint4 *>(w + 4 * q + 2);
                const uint32_t wl[4] = {w01.x, w01.z, w23.x, w23.z}, wh[4] = {w01.y, w01.w, w23.y, w23.w};
#endif
#pragma unroll
                for (int byte = 0; byte < 4; byte++) {
                    const uint32_t x = c ^ ((v >> (8 * byte)) & 0xffu);
                    const int32_t d = (int32_t)x - (int32_t)c;
#if PKV_HASH_W128
                    acc += (int64_t)d * (int32_t)wl[byte];
                    acc_hi += (uint32_t)d * wh[byte];
#else
                    const SplitWeight wk = w[4 * q + byte];
                    acc += (int64_t)d * wk.lo_s;
                    acc_hi += (uint32_t)d * wk.hi;
#endif
                    c = x * 0x1b3u;
                }
            }
            D = D * join_weight(w[0]) + (uint64_t)acc + ((uint64_t)acc_hi << 32);
        }
        table[g * 256 + c0] = D;
    }
}

__device__ __forceinline__ void cp_async16(uint32_t smem, const void *gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// One warp per request (one warp per CTA).  The warp keeps the tables of the next kRing blocks
// in flight in a shared-memory ring (cp.async, 64 bytes per lane per table, kBatch tables per
// commit group) while every lane runs the same serial chain; the table entry is a broadcast
// shared load.
constexpr int kBatch = PKV_HASH_BATCH;
static_assert(kRing % kBatch == 0, "the ring holds whole groups");

__global__ void __launch_bounds__(32) hash_walk_kernel(const int32_t *__restrict__ off, int32_t n_reqs,
                                                       int32_t n_tokens, int32_t bs, uint64_t seed, uint64_t p_pow_n,
                                                       const int32_t *__restrict__ out_off,
                                                       const uint64_t *__restrict__ table, int64_t limit,
                                                       uint64_t *__restrict__ out, int *err)
{
    pkv::grid_dep_entry();  // before any global memory access
    constexpr int kGroups = kRing / kBatch;  // commit groups in flight
    extern __shared__ __align__(16) uint64_t ring_mem[];  // kRing tables of 256 entries
    uint64_t(*ring)[256] = reinterpret_cast<uint64_t(*)[256]>(ring_mem);
    const int lane = threadIdx.x;
    const uint32_t ring_base = (uint32_t)__cvta_generic_to_shared(ring_mem);
    for (int32_t r = blockIdx.x; r < n_reqs; r += gridDim.x) {
        int32_t begin, k;
        int64_t at;
        if (!request_blocks(off, r, n_tokens, bs, out_off, limit, err, &begin, &k, &at)) continue;
        const uint64_t *tab = table + at * 256;
        auto fetch = [&](int32_t j0) {  // tables j0 .. j0 + kBatch - 1 into their ring slots, one group
#pragma unroll
            for (int q = 0; q < kBatch; q++) {
                const int32_t j = j0 + q;
                if (j < k) {
                    const char *src = reinterpret_cast<const char *>(tab + (int64_t)j * 256) + lane * 64;
                    const uint32_t dst = ring_base + (uint32_t)((j % kRing) * 2048 + lane * 64);
#pragma unroll
                    for (int w = 0; w < 4; w++) cp_async16(dst + w * 16, src + w * 16);
                }
            }
            cp_async_commit();
        };
#pragma unroll
        for (int g = 0; g < kGroups; g++) fetch(g * kBatch);
        uint64_t parent = seed;
        for (int32_t j0 = 0; j0 < k; j0 += kBatch) {
            cp_async_wait<kGroups - 1>();  // this lane's copies of tables j0 .. j0 + kBatch - 1 have landed
            __syncwarp();                  // and every other lane's
#pragma unroll
            for (int q = 0; q < kBatch; q++) {
                const int32_t j = j0 + q;
                if (j >= k) break;
                const Fnv S = fnv_block_start(parent);
                parent = p_pow_n * fnv_value(S) + ring[j % kRing][S.lo & 0xffu];
                if (lane == 0) out[at + j] = parent;
            }
            __syncwarp();  // the group's slots are read by all lanes before they are refilled
            fetch(j0 + kRing);
        }
        cp_async_wait<0>();
        __syncwarp();
    }
}

}  // namespace

int pkv::preload_hash_kernels()
{
    return pkv::load_kernels(hash_count_kernel, hash_chain_kernel, hash_table_kernel, hash_walk_kernel);
}

extern "C" int kv_block_hashes_workspace_bytes(int64_t n_tokens, int32_t block_size, int64_t *bytes_out)
{
    if (bytes_out == nullptr || n_tokens < 0 || block_size <= 0) return KV_ERR_INVALID_ARG;
    *bytes_out = (n_tokens / block_size) * 256 * (int64_t)sizeof(uint64_t);
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
    int64_t need = 0;
    kv_block_hashes_workspace_bytes(n_tokens, block_size, &need);
    if (workspace != nullptr) {
        if (!pkv::aligned16(workspace)) return KV_ERR_ALIGN;
        if (workspace_bytes < need) return KV_ERR_RANGE;
    }
    const pkv::DeviceInfo *dev = pkv::current_device();
    if (dev == nullptr) return KV_ERR_CUDA;
    const cudaStream_t s = (cudaStream_t)stream;
    if (n_reqs == 0) return pkv::cuda_status(cudaMemsetAsync(out_offsets, 0, sizeof(int32_t), s));
    pkv::launch<kHashPdl>(hash_count_kernel, 1, kScanThreads, 0, s, tok_offsets, n_reqs, (int32_t)n_tokens, block_size,
                          out_offsets, dev->err_word);
    int st = pkv::cuda_status(cudaGetLastError());
    if (st != KV_OK) return st;
    if (workspace == nullptr) {
        const int blocks = std::max(1, std::min((n_reqs + kChainThreads - 1) / kChainThreads, dev->num_sms * 4));
        pkv::launch<kHashPdl>(hash_chain_kernel, blocks, kChainThreads, 0, s, tok_offsets, n_reqs, tokens,
                              (int32_t)n_tokens, block_size, seed, out_offsets, out_hashes, out_capacity,
                              dev->err_word);
        return pkv::cuda_status(cudaGetLastError());
    }
    // hashes beyond n_tokens / block_size only arise from inconsistent offsets (flagged by the count)
    const int64_t limit = std::min<int64_t>(out_capacity, n_tokens / block_size);
    if (limit == 0) return KV_OK;
    uint64_t *table = reinterpret_cast<uint64_t *>(workspace);
    const int table_blocks = (int)std::min<int64_t>(limit, (int64_t)dev->num_sms * 8);
    pkv::launch<kHashPdl>(hash_table_kernel, table_blocks, kTableThreads, 0, s, tok_offsets, n_reqs, tokens,
                          (int32_t)n_tokens, block_size, out_offsets, table, limit);
    st = pkv::cuda_status(cudaGetLastError());
    if (st != KV_OK) return st;
    const uint64_t p_pow_n = pow_mod_2_64(kFnvPrime, 4ull * (uint64_t)block_size);
    constexpr int kRingBytes = kRing * 256 * (int)sizeof(uint64_t);
    static std::mutex mu;
    static bool configured[64];
    {
        std::lock_guard<std::mutex> lock(mu);
        if (kRingBytes > 48 * 1024 && !configured[dev->device & 63]) {
            st = pkv::cuda_status(
                cudaFuncSetAttribute(hash_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes));
            if (st != KV_OK) return st;
            configured[dev->device & 63] = true;
        }
    }
    const int walk_blocks = std::min(n_reqs, dev->num_sms * 16);
    pkv::launch<kHashPdl && PKV_HASH_WALK_PDL>(hash_walk_kernel, walk_blocks, 32, kRingBytes, s, tok_offsets, n_reqs,
                                               (int32_t)n_tokens, block_size, seed, p_pow_n, out_offsets, table, limit,
                                               out_hashes, dev->err_word);
    return pkv::cuda_status(cudaGetLastError());
}
