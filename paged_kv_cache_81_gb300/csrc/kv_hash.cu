// kv_block_hashes: the prefix hash chain over full token blocks.
//
// Drawing "vllm v1 调度逻辑 和 distributed 分布式原理", the hash-table labels: every full block is
// keyed by h0 = hash(seed, [t0 .. t(bs-1)]) and h_i = hash(h_(i-1), [tokens of block i]), so
// equal prefixes give equal keys (cached_block_hash_to_block).  The pages do not name the hash;
// the reading implemented here is FNV-1a 64 over the parent hash as 8 little-endian bytes
// followed by the block's token ids as 4 little-endian bytes each.  Only full blocks are hashed.
//
// FNV-1a is byte-serial and each block starts from its parent's hash, so a request's chain is
// sequential; the parallelism is across requests (one thread each).  One CTA first scans the
// full-block counts into the output CSR offsets.
#include <algorithm>

#include "kv_common.cuh"

namespace {

constexpr int kScanThreads = 1024;
constexpr uint64_t kFnvBasis = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

__device__ __forceinline__ uint64_t fnv_bytes(uint64_t h, uint64_t v, int n)
{
#pragma unroll
    for (int j = 0; j < 8; j++) {
        if (j < n) {
            h ^= (v >> (8 * j)) & 0xffu;
            h *= kFnvPrime;
        }
    }
    return h;
}

__global__ void __launch_bounds__(kScanThreads) hash_count_kernel(const int32_t *__restrict__ off, int32_t n_reqs,
                                                                  int32_t n_tokens, int32_t bs, int32_t *out_off,
                                                                  int *err)
{
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

__global__ void __launch_bounds__(128) hash_chain_kernel(const int32_t *__restrict__ off, int32_t n_reqs,
                                                         const int32_t *__restrict__ tokens, int32_t n_tokens,
                                                         int32_t bs, uint64_t seed,
                                                         const int32_t *__restrict__ out_off,
                                                         uint64_t *__restrict__ out, int64_t out_capacity, int *err)
{
    for (int32_t r = blockIdx.x * blockDim.x + threadIdx.x; r < n_reqs; r += gridDim.x * blockDim.x) {
        const int32_t begin = off[r];
        const int32_t n = off[r + 1] - begin;
        if (n <= 0 || begin < 0 || begin + n > n_tokens) continue;
        const int32_t k = n / bs;
        const int64_t at = out_off[r];
        if (at < 0 || at + k > out_capacity) {
            pkv::set_error(err, KV_DERR_LIST);
            continue;
        }
        uint64_t parent = seed;
        const int32_t *t = tokens + begin;
        for (int32_t b = 0; b < k; b++) {
            uint64_t h = fnv_bytes(kFnvBasis, parent, 8);
            for (int32_t j = 0; j < bs; j++) h = fnv_bytes(h, (uint32_t)t[(int64_t)b * bs + j], 4);
            out[at + b] = h;
            parent = h;
        }
    }
}

}  // namespace

extern "C" int kv_block_hashes(const int32_t *tok_offsets, int32_t n_reqs, const int32_t *tokens, int64_t n_tokens,
                               int32_t block_size, uint64_t seed, int32_t *out_offsets, uint64_t *out_hashes,
                               int64_t out_capacity, kv_stream_t stream)
{
    if (n_reqs < 0 || n_tokens < 0 || block_size <= 0 || out_capacity < 0 || tok_offsets == nullptr ||
        out_offsets == nullptr)
        return KV_ERR_INVALID_ARG;
    if (n_tokens >= (1ll << 31)) return KV_ERR_UNSUPPORTED;
    if (n_tokens > 0 && (tokens == nullptr || n_reqs == 0)) return KV_ERR_INVALID_ARG;
    if (out_capacity < n_tokens / block_size) return KV_ERR_RANGE;
    if (out_capacity > 0 && out_hashes == nullptr) return KV_ERR_INVALID_ARG;
    if (((uintptr_t)out_hashes & 7u) != 0) return KV_ERR_ALIGN;
    const pkv::DeviceInfo *dev = pkv::current_device();
    if (dev == nullptr) return KV_ERR_CUDA;
    const cudaStream_t s = (cudaStream_t)stream;
    if (n_reqs == 0) return pkv::cuda_status(cudaMemsetAsync(out_offsets, 0, sizeof(int32_t), s));
    hash_count_kernel<<<1, kScanThreads, 0, s>>>(tok_offsets, n_reqs, (int32_t)n_tokens, block_size, out_offsets,
                                                  dev->err_word);
    int st = pkv::cuda_status(cudaGetLastError());
    if (st != KV_OK) return st;
    const int threads = 128;
    const int blocks = std::max(1, std::min((n_reqs + threads - 1) / threads, dev->num_sms * 4));
    hash_chain_kernel<<<blocks, threads, 0, s>>>(tok_offsets, n_reqs, tokens, (int32_t)n_tokens, block_size, seed,
                                                 out_offsets, out_hashes, out_capacity, dev->err_word);
    return pkv::cuda_status(cudaGetLastError());
}
