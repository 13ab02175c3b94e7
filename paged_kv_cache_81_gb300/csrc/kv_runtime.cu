// Runtime state of libpagedkv: per-device info, the sticky device error word,
// status strings and kv_get_last_error.
#include <atomic>
#include <mutex>

#include "kv_common.cuh"

namespace {

// One sticky error word per device (each device that loads the module gets its own copy).
__device__ int g_kv_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
pkv::DeviceInfo g_info[kMaxDevices];
bool g_ready[kMaxDevices];
std::atomic<int> g_last_cuda_error{0};

}  // namespace

namespace pkv {

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return KV_OK;
    g_last_cuda_error.store((int)e);
    return KV_ERR_CUDA;
}

const DeviceInfo *current_device()
{
    int dev = 0;
    if (cuda_status(cudaGetDevice(&dev)) != KV_OK) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_ready[dev]) {
        DeviceInfo info{dev, 0, nullptr};
        if (cuda_status(cudaDeviceGetAttribute(&info.num_sms, cudaDevAttrMultiProcessorCount, dev)) != KV_OK)
            return nullptr;
        void *p = nullptr;
        if (cuda_status(cudaGetSymbolAddress(&p, g_kv_error_word)) != KV_OK) return nullptr;
        info.err_word = (int *)p;
        g_info[dev] = info;
        g_ready[dev] = true;
    }
    return &g_info[dev];
}

int check_cache(const kv_cache_desc *c)
{
    if (c == nullptr || c->n_tensors < 0 || c->block_size <= 0 || c->num_blocks < 0 ||
        (c->n_planes != 1 && c->n_planes != 2) || c->row_bytes <= 0 || c->block_stride < 0 ||
        c->plane_stride < 0 || c->token_stride < 0)
        return KV_ERR_INVALID_ARG;
    if (c->n_tensors > 0 && c->base == nullptr) return KV_ERR_INVALID_ARG;
    if (!aligned16((int64_t)c->row_bytes) || !aligned16(c->block_stride) || !aligned16(c->token_stride) ||
        (c->n_planes == 2 && !aligned16(c->plane_stride)))
        return KV_ERR_ALIGN;
    // every row's byte offset, block * block_stride + plane * plane_stride + slot * token_stride
    // + row_bytes, must fit in int64 (the kernels compute it so)
    int64_t span = 0, part = 0;
    if (__builtin_mul_overflow(c->num_blocks, c->block_stride, &span) ||
        __builtin_mul_overflow((int64_t)c->block_size, c->token_stride, &part) || __builtin_add_overflow(span, part, &span) ||
        __builtin_add_overflow(span, c->n_planes == 2 ? c->plane_stride : (int64_t)0, &span) ||
        __builtin_add_overflow(span, (int64_t)c->row_bytes, &span))
        return KV_ERR_RANGE;
    for (int32_t t = 0; t < c->n_tensors; t++) {
        if (c->base[t] == 0) return KV_ERR_INVALID_ARG;
        if (c->base[t] & 15u) return KV_ERR_ALIGN;
    }
    return KV_OK;
}

int preload_all_kernels(const DeviceInfo &dev)
{
    static std::mutex mu;
    static bool done[kMaxDevices];
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev.device]) return KV_OK;
    for (int (*load)() : {preload_write_kernels, preload_xfer_kernels, preload_copy_kernels, preload_bulk_kernels,
                          preload_clip_kernels, preload_hash_kernels, preload_signal_kernels}) {
        const int st = load();
        if (st != KV_OK) return st;
    }
    done[dev.device] = true;
    return KV_OK;
}

}  // namespace pkv

extern "C" {

const char *kv_version(void) { return "pagedkv 0.1.0 sm_103a"; }

const char *kv_status_string(int status)
{
    switch (status) {
    case KV_OK: return "KV_OK";
    case KV_ERR_INVALID_ARG: return "KV_ERR_INVALID_ARG";
    case KV_ERR_ALIGN: return "KV_ERR_ALIGN";
    case KV_ERR_RANGE: return "KV_ERR_RANGE";
    case KV_ERR_CUDA: return "KV_ERR_CUDA";
    case KV_ERR_TIMEOUT: return "KV_ERR_TIMEOUT";
    case KV_ERR_UNSUPPORTED: return "KV_ERR_UNSUPPORTED";
    default: return "KV_ERR_UNKNOWN";
    }
}

int kv_last_cuda_error(void) { return g_last_cuda_error.load(); }

int kv_get_last_error(int32_t *host_out, int32_t clear, kv_stream_t stream)
{
    if (host_out == nullptr) return KV_ERR_INVALID_ARG;
    const pkv::DeviceInfo *d = pkv::current_device();
    if (d == nullptr) return KV_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    int st = pkv::cuda_status(cudaMemcpyAsync(host_out, d->err_word, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    if (st != KV_OK) return st;
    if (clear) {
        st = pkv::cuda_status(cudaMemsetAsync(d->err_word, 0, sizeof(int32_t), s));
        if (st != KV_OK) return st;
    }
    return pkv::cuda_status(cudaStreamSynchronize(s));
}

}  // extern "C"
