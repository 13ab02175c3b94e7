// Internal helpers shared by the libpagedkv translation units (not part of the ABI).
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "pagedkv.h"

namespace pkv {

// Cache tensors whose base addresses one launch carries in its parameter block.
constexpr int kMaxTensorsPerLaunch = 128;

// ---------------------------------------------------------------------------
// Unsigned 32-bit division by a runtime-invariant divisor with a multiply and a
// shift (Granlund & Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994, section 4): for 1 <= d < 2^31 and l = ceil(log2 d),
// m = floor(2^32 * (2^l - d) / d) + 1 and q = (mulhi(n, m) + n) >> l for every
// 32-bit n.  The sum is formed in 64 bits so it cannot overflow.
// ---------------------------------------------------------------------------
struct FastDiv {
    uint32_t d;
    uint32_t m;
    uint32_t l;
};

inline FastDiv make_fastdiv(uint32_t d)
{
    FastDiv f{d, 0u, 0u};
    while ((1ull << f.l) < d) f.l++;
    f.m = (uint32_t)(((1ull << 32) * ((1ull << f.l) - d)) / d + 1);
    return f;
}

__host__ __device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f)
{
#ifdef __CUDA_ARCH__
    uint32_t hi = __umulhi(n, f.m);
#else
    uint32_t hi = (uint32_t)(((uint64_t)n * f.m) >> 32);
#endif
    return (uint32_t)(((uint64_t)hi + n) >> f.l);
}

// ---------------------------------------------------------------------------
// 16-byte global accesses.  Cache rows are read once (no L1 allocation); staging
// and cache writes are streaming (evict-first) stores.
// ---------------------------------------------------------------------------
#ifndef PKV_LD_NO_ALLOCATE
#define PKV_LD_NO_ALLOCATE 1  // 0: read-only loads that may allocate in L1
#endif
#ifndef PKV_ST_STREAMING
#define PKV_ST_STREAMING 1  // 0: plain write-back stores
#endif

__device__ __forceinline__ uint4 ld_once(const void *p)
{
    uint4 v;
#if PKV_LD_NO_ALLOCATE
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
#else
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
#endif
    return v;
}

__device__ __forceinline__ void st_stream(void *p, const uint4 &v)
{
#if PKV_ST_STREAMING
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
#else
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
#endif
}

__device__ __forceinline__ void set_error(int *err, int bits)
{
    atomicOr(err, bits);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched with programmatic
// stream serialisation allowed, so its CTAs may be scheduled while the previous kernel on the
// stream is still running.  Each kernel therefore calls grid_dep_entry() before its first
// global memory access: griddepcontrol.wait returns once every prerequisite grid has completed
// and its memory operations are visible (at once when there is none), which keeps plain stream
// order for the data; only launch and CTA setup overlap the previous kernel.  The kernel then
// allows its own dependents to be scheduled (they take effect once all its CTAs have started).
// A kernel that waits for work on another stream calls grid_dep_wait() alone: its dependents
// are then scheduled only when it ends, so they cannot hold the SM space that work needs.
// ---------------------------------------------------------------------------
#ifndef PKV_PDL
#define PKV_PDL 1  // 0: plain stream-ordered launches
#endif

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void grid_dep_entry()
{
    grid_dep_wait();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// cudaLaunchKernelEx with programmatic stream serialisation when PKV_PDL is on and pdl is true,
// else a plain stream-ordered launch.
//
// Which launches take it: only the ones that the previous kernel's tail cannot be starved by.
// A kernel launched this way may have its CTAs placed as soon as every CTA of the previous
// kernel has started; they then wait, holding SM space, until that kernel completes.  For a
// kernel of a few waves or less that only hides launch latency (the 61-layer decode write:
// 6.1 instead of 6.8 us back to back).  But the copy engines end with tail CTAs that the
// hardware places as SMs free up, and a multi-wave row write keeps placing CTAs until its
// end: a GPU-filling successor launched early took those SMs, and the page-shaped step issued
// with no event between its calls ran 1.664 ms against 1.611 ms with every launch plain.  So
// copies with tail CTAs and row writes of more than two waves launch plainly (launch_as(false)).
template <typename... KArgs, typename... Args>
cudaError_t launch_as(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                      Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = PKV_PDL && pdl;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// launch<true> (the default): programmatic dependent launch; launch<false>: plain.
template <bool Pdl = true, typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                   Args &&...args)
{
    return launch_as(Pdl, kernel, grid, block, smem, stream, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// Host-side runtime state (kv_runtime.cu).
// ---------------------------------------------------------------------------
struct DeviceInfo {
    int device;
    int num_sms;
    int *err_word;  // device address of this device's sticky error word
};

// Info of the current device, created on first use; nullptr after a CUDA error
// (the error is recorded for kv_last_cuda_error).
const DeviceInfo *current_device();

// Records a CUDA error and returns KV_ERR_CUDA, or KV_OK for cudaSuccess.
int cuda_status(cudaError_t e);

inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
inline bool aligned16(int64_t v) { return (v & 15) == 0; }

// Adds `add` to signal->value on `stream` (one thread, release semantics) - used when a
// signalled call has no copy to make (kv_signal.cu).
int post_signal(kv_signal *signal, uint64_t add, cudaStream_t s);

// Validates a cache descriptor; checks the tensor base addresses too.
int check_cache(const kv_cache_desc *c);

// Kernel preloading.  CUDA loads a kernel's code lazily, on first use, and loading may
// synchronise the context; a launch that loads a kernel while another stream runs a kernel
// that polls (kv_wait_signal) would then wait for that poll to end.  cudaFuncGetAttributes
// loads a kernel, so each source file lists its kernels here, and kv_wait_signal loads them
// all (once per device) before it queues its polling kernel.
template <typename... Fns>
int load_kernels(Fns... fns)
{
    cudaFuncAttributes attr;
    for (const void *f : {reinterpret_cast<const void *>(fns)...}) {
        const cudaError_t e = cudaFuncGetAttributes(&attr, f);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return KV_OK;
}
int preload_write_kernels();   // kv_write.cu
int preload_xfer_kernels();    // kv_xfer.cu
int preload_copy_kernels();    // kv_copy.cu
int preload_bulk_kernels();    // kv_bulk.cu
int preload_clip_kernels();    // kv_clip.cu
int preload_hash_kernels();    // kv_hash.cu
int preload_signal_kernels();  // kv_signal.cu
// All of the above, once per device (kv_runtime.cu).
int preload_all_kernels(const DeviceInfo &dev);

}  // namespace pkv
