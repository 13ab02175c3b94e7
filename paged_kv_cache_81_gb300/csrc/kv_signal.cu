// Transfer-completion signals: the receiver's side of the FlagCX connector's protocol
// (page "5. flagcx connector design & dev & test", section 1.2): the sender adds 1 to a
// per-pair signal counter with its last put of a transfer (sig_val = 1 on the last xfer),
// and the receiver waits, on the GPU, until the counter reaches the largest value it
// expects (a GPU-side poll of the signal buffer) before its forward pass goes on.
// Here kv_unpack_blocks_signal posts the increment when the last row of a scatter has
// landed, and kv_wait_signal is the bounded device-side wait.
#include "kv_common.cuh"

namespace {

constexpr uint64_t kMaxTimeoutUs = 60ull * 1000 * 1000;  // the pages' longest wait, 60 s (the proxy's ready event)

__device__ __forceinline__ unsigned long long now_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__global__ void post_signal_kernel(kv_signal *signal, uint64_t add)
{
    pkv::grid_dep_entry();  // before any global memory access
    __threadfence();
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(&signal->value), "l"(add) : "memory");
}

// One thread polls the counter with acquire loads and an exponential sleep; it gives up after
// timeout_ns of globaltimer time.  It never waits on anything without a limit.
__global__ void wait_signal_kernel(const kv_signal *signal, uint64_t expected, uint64_t timeout_ns, int32_t *status,
                                   int *err)
{
    // The entry wait only: the kernels queued after this one must not be scheduled while it polls,
    // or a persistent copy grid among them could take the SM space of the work on another stream
    // that sets the counter, and the wait would run out.
    pkv::grid_dep_wait();
    const unsigned long long t0 = now_ns();
    unsigned ns = 64;
    while (true) {
        if (ld_acquire_u64(&signal->value) >= expected) {
            if (status) *status = KV_OK;
            return;
        }
        if (now_ns() - t0 > timeout_ns) {
            if (status) *status = KV_ERR_TIMEOUT;
            pkv::set_error(err, KV_DERR_TIMEOUT);
            return;
        }
        __nanosleep(ns);
        ns = ns < 8192 ? ns * 2 : ns;
    }
}

}  // namespace

namespace pkv {

int preload_signal_kernels() { return load_kernels(post_signal_kernel, wait_signal_kernel); }

int post_signal(kv_signal *signal, uint64_t add, cudaStream_t s)
{
    pkv::launch(post_signal_kernel, 1, 1, 0, s, signal, add);
    return cuda_status(cudaGetLastError());
}

}  // namespace pkv

extern "C" int kv_wait_signal(const kv_signal *signal, uint64_t expected, uint32_t timeout_us, int32_t *status_out,
                              kv_stream_t stream)
{
    if (signal == nullptr) return KV_ERR_INVALID_ARG;
    if (((uintptr_t)signal & 15u) != 0 || ((uintptr_t)status_out & 3u) != 0) return KV_ERR_ALIGN;
    if (timeout_us == 0 || timeout_us > kMaxTimeoutUs) return KV_ERR_RANGE;
    const pkv::DeviceInfo *dev = pkv::current_device();
    if (dev == nullptr) return KV_ERR_CUDA;
    // every kernel of the library is loaded before the poll starts (see preload_all_kernels)
    const int st = pkv::preload_all_kernels(*dev);
    if (st != KV_OK) return st;
    pkv::launch(wait_signal_kernel, 1, 1, 0, (cudaStream_t)stream, signal, expected, (uint64_t)timeout_us * 1000ull,
                status_out, dev->err_word);
    return pkv::cuda_status(cudaGetLastError());
}
