// kv_clip_block_lists: the sliding-window clip of per-request block lists.
//
// Page "vLLM PD 分离 源码级机制", section 3.1: when a request finishes on the prefill side,
// its blocks are queued for sending as get_sw_clipped_blocks(block_ids).  The function's
// body is not on the page; the reading implemented here: a layer whose attention sees only
// the last `window` tokens needs, of a request with n tokens, only the list entries
//     q = max(0, n - window) / block_size  ..  ceil(n / block_size) - 1
// (never past the request's list); window <= 0 keeps every block that holds a token.
//
// Two launches: one CTA scans the kept counts of all requests into the output CSR
// offsets; then a grid-stride kernel moves every kept entry to its place.
#include <algorithm>

#include "kv_common.cuh"

namespace {

constexpr int kScanThreads = 1024;

__device__ __forceinline__ void kept_range(int64_t n, int32_t window, int32_t bs, int32_t len, int32_t *first,
                                           int32_t *end)
{
    const int64_t first_token = (window > 0 && n > window) ? n - window : 0;
    int64_t e = (n + bs - 1) / bs;
    if (e > len) e = len;
    int64_t f = first_token / bs;
    if (f > e) f = e;
    *first = (int32_t)f;
    *end = (int32_t)e;
}

__global__ void __launch_bounds__(kScanThreads) clip_count_kernel(const int32_t *__restrict__ off, int32_t n_reqs,
                                                                  int32_t n_ids, const int32_t *__restrict__ n_tokens,
                                                                  int32_t window, int32_t bs, int32_t *out_off, int *err)
{
    pkv::grid_dep_entry();  // before any global memory access
    __shared__ int32_t warp_sum[kScanThreads / 32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        carry = 0;
        if (off[0] != 0 || off[n_reqs] != n_ids) pkv::set_error(err, KV_DERR_LIST);
    }
    __syncthreads();
    for (int32_t base = 0; base < n_reqs; base += kScanThreads) {
        const int32_t r = base + tid;
        int32_t cnt = 0;
        if (r < n_reqs) {
            int64_t n = n_tokens[r];
            int64_t len64 = (int64_t)off[r + 1] - off[r];  // 64-bit: offsets may be anything
            if (n < 0 || len64 < 0) {
                pkv::set_error(err, KV_DERR_LIST);
                n = n < 0 ? 0 : n;
                len64 = len64 < 0 ? 0 : len64;
            }
            const int32_t len = (int32_t)(len64 > INT32_MAX ? INT32_MAX : len64);
            int32_t f, e;
            kept_range(n, window, bs, len, &f, &e);
            cnt = e - f;
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

__global__ void __launch_bounds__(256) clip_copy_kernel(const int32_t *__restrict__ off, int32_t n_reqs,
                                                        const int32_t *__restrict__ ids, int32_t n_ids,
                                                        const int32_t *__restrict__ n_tokens, int32_t window,
                                                        int32_t bs, const int32_t *__restrict__ out_off,
                                                        int32_t *__restrict__ out_ids, int64_t out_capacity, int *err)
{
    pkv::grid_dep_entry();  // before any global memory access
    const int32_t step = gridDim.x * blockDim.x;
    for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n_ids; i += step) {
        int32_t lo = 0, hi = n_reqs - 1;  // last request whose first entry is <= i
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (off[mid] <= i) lo = mid;
            else hi = mid - 1;
        }
        const int32_t r = lo;
        const int64_t q = (int64_t)i - off[r];
        const int64_t len64 = (int64_t)off[r + 1] - off[r];  // 64-bit: offsets may be anything
        if (q < 0 || len64 <= 0) continue;
        const int32_t len = (int32_t)(len64 > INT32_MAX ? INT32_MAX : len64);
        const int64_t n = n_tokens[r] < 0 ? 0 : n_tokens[r];
        int32_t f, e;
        kept_range(n, window, bs, len, &f, &e);
        if (q < f || q >= e) continue;
        const int64_t at = (int64_t)out_off[r] + (q - f);
        if (at < 0 || at >= out_capacity) {
            pkv::set_error(err, KV_DERR_LIST);
            continue;
        }
        out_ids[at] = ids[i];
    }
}

}  // namespace

int pkv::preload_clip_kernels() { return pkv::load_kernels(clip_count_kernel, clip_copy_kernel); }

extern "C" int kv_clip_block_lists(const int32_t *req_offsets, int32_t n_reqs, const int32_t *ids, int64_t n_ids,
                                   const int32_t *n_tokens, int32_t window, int32_t block_size,
                                   int32_t *out_offsets, int32_t *out_ids, int64_t out_capacity,
                                   kv_stream_t stream)
{
    if (n_reqs < 0 || n_ids < 0 || block_size <= 0 || out_capacity < 0 || req_offsets == nullptr ||
        out_offsets == nullptr)
        return KV_ERR_INVALID_ARG;
    if (n_ids >= (1ll << 31)) return KV_ERR_UNSUPPORTED;
    if (n_reqs > 0 && n_tokens == nullptr) return KV_ERR_INVALID_ARG;
    if (n_ids > 0 && (ids == nullptr || out_ids == nullptr || n_reqs == 0)) return KV_ERR_INVALID_ARG;
    if (out_capacity < n_ids) return KV_ERR_RANGE;
    const pkv::DeviceInfo *dev = pkv::current_device();
    if (dev == nullptr) return KV_ERR_CUDA;
    const cudaStream_t s = (cudaStream_t)stream;
    if (n_reqs == 0) return pkv::cuda_status(cudaMemsetAsync(out_offsets, 0, sizeof(int32_t), s));
    pkv::launch(clip_count_kernel, 1, kScanThreads, 0, s, req_offsets, n_reqs, (int32_t)n_ids, n_tokens, window,
                block_size, out_offsets, dev->err_word);
    int st = pkv::cuda_status(cudaGetLastError());
    if (st != KV_OK || n_ids == 0) return st;
    const int threads = 256;
    const int blocks = (int)std::min<int64_t>((n_ids + threads - 1) / threads, (int64_t)dev->num_sms * 8);
    pkv::launch(clip_copy_kernel, blocks, threads, 0, s, req_offsets, n_reqs, ids, (int32_t)n_ids, n_tokens, window,
                block_size, out_offsets, out_ids, out_capacity, dev->err_word);
    return pkv::cuda_status(cudaGetLastError());
}
