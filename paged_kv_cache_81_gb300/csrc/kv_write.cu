// kv_slot_mapping and kv_reshape_and_cache: writing new tokens' K/V into the paged cache.
//
// Slot formula: drawing "vllm v1 调度逻辑 和 distributed 分布式原理", label "batch tensor 组装";
// block = slots 0..15 of K/V rows: label "Paged kv cache"; one block_table serves every
// layer: label "总的就是 all kv cache".
#include <algorithm>
#include <climits>
#include <numeric>

#include "kv_common.cuh"

namespace {

using pkv::FastDiv;

__global__ void __launch_bounds__(256) slot_mapping_kernel(const int32_t *__restrict__ table, int32_t n_reqs,
                                                           int32_t max_blocks, int64_t row_stride,
                                                           const int32_t *__restrict__ token_req,
                                                           const int32_t *__restrict__ token_pos, int64_t n_tokens,
                                                           int32_t block_size, int64_t *__restrict__ slot,
                                                           int *err)
{
    pkv::grid_dep_entry();  // before any global memory access
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_tokens; i += step) {
        const int32_t req = token_req[i];
        const int32_t pos = token_pos[i];
        int64_t s = -1;
        if (req >= 0 && req < n_reqs && pos >= 0) {
            const int32_t q = pos / block_size;  // logical block of the position
            if (q < max_blocks) {
                const int32_t block = table[(int64_t)req * row_stride + q];
                if (block >= 0) s = (int64_t)block * block_size + (pos - q * block_size);
            }
        }
        if (s < 0) pkv::set_error(err, KV_DERR_TABLE);
        slot[i] = s;
    }
}

// One launch writes up to kMaxTensorsPerLaunch cache tensors (blockIdx.y = tensor).
// Work is the flat index over (token, plane, 16-byte chunk of the row); consecutive
// threads cover consecutive chunks of one row, so every row is read and written as
// whole coalesced segments.
struct ReshapeParams {
    const int64_t *slot;  // slots of the tokens (reshape_and_cache), or null when FUSED
    // FUSED (kv_write_tokens): each token's slot is looked up in the block table here
    const int32_t *table;
    const int32_t *token_req;
    const int32_t *token_pos;
    int64_t *slot_out;  // optional: the looked-up slots are also written here (first launch only)
    int64_t table_row_stride;
    int32_t n_reqs;
    int32_t max_blocks;
    int64_t src_token_stride;
    int64_t block_stride;
    int64_t plane_stride;
    int64_t token_stride;
    uint32_t total;      // n_tokens * n_planes * chunks_per_row
    uint32_t slot_limit; // num_blocks * block_size
    FastDiv div_cpr;     // chunks per row
    FastDiv div_planes;
    FastDiv div_bs;
    FastDiv div_tokens;
    int32_t n_planes;
    uint32_t n_tokens;
    uint32_t tok_step;   // reshape_rows_kernel: the grid stride in tokens
    int *err;
    uint64_t dst[pkv::kMaxTensorsPerLaunch];
    uint64_t src[pkv::kMaxTensorsPerLaunch * 2];
};

#ifndef PKV_RESHAPE_UNROLL
#define PKV_RESHAPE_UNROLL 4  // 16-byte loads each thread keeps in flight
#endif
#ifndef PKV_RESHAPE_MIN_CTAS
#define PKV_RESHAPE_MIN_CTAS 6  // launch-bounds hint: resident CTAs per SM the register budget must allow
#endif
#ifndef PKV_RESHAPE_LOADS_FIRST
#define PKV_RESHAPE_LOADS_FIRST 1  // 0: resolve each row's slot before issuing its load
#endif
#ifndef PKV_RESHAPE_PLANE_MAJOR
#define PKV_RESHAPE_PLANE_MAJOR 0  // 1: order work (plane, token, chunk) instead of (token, plane, chunk)
#endif
constexpr int kReshapeUnroll = PKV_RESHAPE_UNROLL;
#ifndef PKV_RESHAPE_ROWS
#define PKV_RESHAPE_ROWS 1  // 0: every row write takes the general kernel
#endif
#ifndef PKV_WRITE_SPLIT_ITERATIONS
#define PKV_WRITE_SPLIT_ITERATIONS 0  // kv_write_tokens with slot_out: grid-stride passes per thread above which it splits
#endif
constexpr int64_t kWriteSplitIterations = PKV_WRITE_SPLIT_ITERATIONS;

// The slot of token `tok`: the block table's entry for the token's logical block times the
// block size plus the offset in the block, or -1 for an invalid token.
__device__ __forceinline__ int64_t table_slot(const ReshapeParams &p, uint32_t tok)
{
    const int32_t req = p.token_req[tok];
    const int32_t pos = p.token_pos[tok];
    if (req < 0 || req >= p.n_reqs || pos < 0) return -1;
    const uint32_t q = pkv::fdiv((uint32_t)pos, p.div_bs);
    if (q >= (uint32_t)p.max_blocks) return -1;
    const int32_t block = p.table[(int64_t)req * p.table_row_stride + q];
    if (block < 0) return -1;
    return (int64_t)block * p.div_bs.d + ((uint32_t)pos - q * p.div_bs.d);
}

template <bool FUSED>
__global__ void __launch_bounds__(256, PKV_RESHAPE_MIN_CTAS)
    reshape_and_cache_kernel(const __grid_constant__ ReshapeParams p)
{
    pkv::grid_dep_entry();  // before any global memory access
    const int t = blockIdx.y;
    uint8_t *const dst = reinterpret_cast<uint8_t *>(p.dst[t]);
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t base = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; base < p.total;
         base += stride * kReshapeUnroll) {
        uint4 v[kReshapeUnroll];
        uint32_t tok[kReshapeUnroll], plane[kReshapeUnroll], chunk[kReshapeUnroll];
        // The row loads do not depend on the slot (only the store address does): issue them
        // all first, then resolve the slots while they are in flight.
#pragma unroll
        for (int u = 0; u < kReshapeUnroll; u++) {
            const uint64_t idx = base + (uint64_t)u * stride;
            tok[u] = 0xffffffffu;
            if (idx >= p.total) continue;
            const uint32_t row = pkv::fdiv((uint32_t)idx, p.div_cpr);
            chunk[u] = (uint32_t)idx - row * p.div_cpr.d;
#if PKV_RESHAPE_PLANE_MAJOR
            // rows ordered (plane, token): neighbouring threads take neighbouring tokens of one plane
            plane[u] = pkv::fdiv(row, p.div_tokens);
            tok[u] = row - plane[u] * p.div_tokens.d;
#else
            tok[u] = pkv::fdiv(row, p.div_planes);
            plane[u] = row - tok[u] * p.div_planes.d;
#endif
#if PKV_RESHAPE_LOADS_FIRST
            const uint8_t *src = reinterpret_cast<const uint8_t *>(p.src[t * p.n_planes + plane[u]]);
            v[u] = pkv::ld_once(src + (int64_t)tok[u] * p.src_token_stride + (int64_t)chunk[u] * 16);
#endif
        }
#pragma unroll
        for (int u = 0; u < kReshapeUnroll; u++) {
            if (tok[u] == 0xffffffffu) continue;
            int64_t s;
            if (FUSED) {
                s = table_slot(p, tok[u]);
                const bool first = t == 0 && plane[u] == 0 && chunk[u] == 0;  // one thread per token reports
                if (first && p.slot_out != nullptr) p.slot_out[tok[u]] = s;
                if (s < 0) {
                    if (first) pkv::set_error(p.err, KV_DERR_TABLE);
                    continue;
                }
            } else {
                s = p.slot[tok[u]];
                if (s < 0) continue;  // padding token
            }
            if (s >= (int64_t)p.slot_limit) {
                pkv::set_error(p.err, KV_DERR_SLOT);
                continue;
            }
#if !PKV_RESHAPE_LOADS_FIRST
            const uint8_t *src = reinterpret_cast<const uint8_t *>(p.src[t * p.n_planes + plane[u]]);
            v[u] = pkv::ld_once(src + (int64_t)tok[u] * p.src_token_stride + (int64_t)chunk[u] * 16);
#endif
            const uint32_t block = pkv::fdiv((uint32_t)s, p.div_bs);
            const uint32_t off = (uint32_t)s - block * p.div_bs.d;
            pkv::st_stream(dst + (int64_t)block * p.block_stride + (int64_t)plane[u] * p.plane_stride +
                               (int64_t)off * p.token_stride + (int64_t)chunk[u] * 16,
                           v[u]);
        }
    }
}

// The row write when the grid stride is a whole number of tokens (a multiple of planes x
// chunks per row): then every row a thread takes has the thread's first plane and chunk and
// the rows' tokens are tok_step apart, so the coordinates are computed once per thread and
// each row costs one address step.  Each pass issues its row loads, then all their slot
// lookups, then the stores: a load placed after a store cannot be moved above it (the compiler
// must assume they may alias), so interleaving them would make each row's lookup (two
// dependent loads when FUSED) wait for the previous row's store.
template <bool FUSED>
__global__ void __launch_bounds__(256, PKV_RESHAPE_MIN_CTAS)
    reshape_rows_kernel(const __grid_constant__ ReshapeParams p)
{
    pkv::grid_dep_entry();  // before any global memory access
    constexpr int64_t kNoRow = INT64_MIN;  // past the last token
    const int t = blockIdx.y;
    const uint32_t first = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t row0 = pkv::fdiv(first, p.div_cpr);
    const uint32_t chunk = first - row0 * p.div_cpr.d;
    const uint32_t tok0 = pkv::fdiv(row0, p.div_planes);  // >= n_tokens when first is past the work
    const uint32_t plane = row0 - tok0 * p.div_planes.d;
    const uint8_t *const src = reinterpret_cast<const uint8_t *>(p.src[t * p.n_planes + plane]) + chunk * 16;
    uint8_t *const dst = reinterpret_cast<uint8_t *>(p.dst[t]) + (int64_t)plane * p.plane_stride + chunk * 16;
    const bool reporter = FUSED && t == 0 && plane == 0 && chunk == 0;  // one thread per token reports
    for (uint32_t tok = tok0; tok < p.n_tokens; tok += p.tok_step * kReshapeUnroll) {
        uint4 v[kReshapeUnroll];
        int64_t s[kReshapeUnroll];
#pragma unroll
        for (int u = 0; u < kReshapeUnroll; u++) {
            const uint32_t tk = tok + u * p.tok_step;
            if (tk < p.n_tokens) v[u] = pkv::ld_once(src + (int64_t)tk * p.src_token_stride);
        }
#pragma unroll
        for (int u = 0; u < kReshapeUnroll; u++) {
            const uint32_t tk = tok + u * p.tok_step;
            s[u] = kNoRow;
            if (tk < p.n_tokens) s[u] = FUSED ? table_slot(p, tk) : p.slot[tk];
        }
#pragma unroll
        for (int u = 0; u < kReshapeUnroll; u++) {
            if (s[u] == kNoRow) continue;
            if (FUSED) {
                if (reporter && p.slot_out != nullptr) p.slot_out[tok + u * p.tok_step] = s[u];
                if (s[u] < 0) {
                    if (reporter) pkv::set_error(p.err, KV_DERR_TABLE);
                    continue;
                }
            } else if (s[u] < 0) {
                continue;  // padding token
            }
            if (s[u] >= (int64_t)p.slot_limit) {
                pkv::set_error(p.err, KV_DERR_SLOT);
                continue;
            }
            const uint32_t block = pkv::fdiv((uint32_t)s[u], p.div_bs);
            const uint32_t off = (uint32_t)s[u] - block * p.div_bs.d;
            pkv::st_stream(dst + (int64_t)block * p.block_stride + (int64_t)off * p.token_stride, v[u]);
        }
    }
}

// Argument checks of a row write (kv_reshape_and_cache, kv_write_tokens).  KV_OK with
// *nothing = true when there is nothing to launch.
int validate_rows(const kv_cache_desc *cache, const uint64_t *new_kv, int64_t new_token_stride, int64_t n_tokens,
                  bool *nothing)
{
    *nothing = false;
    int st = pkv::check_cache(cache);
    if (st != KV_OK) return st;
    if (n_tokens < 0 || new_token_stride < 0) return KV_ERR_INVALID_ARG;
    if (n_tokens == 0 || cache->n_tensors == 0) {
        *nothing = true;
        return KV_OK;
    }
    if (new_kv == nullptr) return KV_ERR_INVALID_ARG;
    if (!pkv::aligned16(new_token_stride)) return KV_ERR_ALIGN;
    if (new_token_stride < cache->row_bytes) return KV_ERR_RANGE;
    for (int64_t k = 0; k < (int64_t)cache->n_tensors * cache->n_planes; k++) {
        if (new_kv[k] == 0) return KV_ERR_INVALID_ARG;
        if (new_kv[k] & 15u) return KV_ERR_ALIGN;
    }
    const int64_t slot_limit = cache->num_blocks * (int64_t)cache->block_size;
    const int64_t cpr = cache->row_bytes / 16;
    const int64_t total = n_tokens * cache->n_planes * cpr;
    if (slot_limit >= (1ll << 31) || total >= (1ll << 31) || cpr >= (1ll << 31)) return KV_ERR_UNSUPPORTED;
    return KV_OK;
}

constexpr int kRowThreads = 256;
constexpr int64_t kMaxRowGroup = 16;

// CTAs per tensor of a row-write launch: enough for the work, at most about four waves of
// 8 resident CTAs per SM over the nt tensors of the launch.
void row_grid(const kv_cache_desc *cache, int64_t n_tokens, int32_t nt, const pkv::DeviceInfo &dev, int64_t *need,
              int64_t *cap)
{
    const int64_t total = n_tokens * cache->n_planes * (cache->row_bytes / 16);
    *need = (total + (int64_t)kRowThreads * kReshapeUnroll - 1) / ((int64_t)kRowThreads * kReshapeUnroll);
    *cap = std::max<int64_t>(1, ((int64_t)dev.num_sms * 8 * 4 + nt - 1) / nt);
}

// Launches shared by kv_reshape_and_cache and kv_write_tokens (arguments already validated).
template <bool FUSED>
int launch_rows(const kv_cache_desc *cache, const uint64_t *new_kv, int64_t new_token_stride, int64_t n_tokens,
                ReshapeParams p, cudaStream_t stream)
{
    bool nothing = false;
    int st = validate_rows(cache, new_kv, new_token_stride, n_tokens, &nothing);
    if (st != KV_OK || nothing) return st;
    const int64_t slot_limit = cache->num_blocks * (int64_t)cache->block_size;
    const int64_t cpr = cache->row_bytes / 16;
    const int64_t total = n_tokens * cache->n_planes * cpr;
    const pkv::DeviceInfo *dev = pkv::current_device();
    if (dev == nullptr) return KV_ERR_CUDA;

    p.src_token_stride = new_token_stride;
    p.block_stride = cache->block_stride;
    p.plane_stride = cache->plane_stride;
    p.token_stride = cache->token_stride;
    p.total = (uint32_t)total;
    p.slot_limit = (uint32_t)slot_limit;
    p.div_cpr = pkv::make_fastdiv((uint32_t)cpr);
    p.div_planes = pkv::make_fastdiv((uint32_t)cache->n_planes);
    p.div_bs = pkv::make_fastdiv((uint32_t)cache->block_size);
    p.div_tokens = pkv::make_fastdiv((uint32_t)n_tokens);
    p.n_planes = cache->n_planes;
    p.n_tokens = (uint32_t)n_tokens;
    p.err = dev->err_word;
    // CTAs a grid stride must be a multiple of to cover whole tokens (planes x chunks per row
    // divides 256 x CTAs); above kMaxRowGroup the general kernel runs instead.
    const int64_t row_group = cache->n_planes * cpr / std::gcd<int64_t>(kRowThreads, cache->n_planes * cpr);

    int64_t *slot_out = p.slot_out;
    for (int32_t t0 = 0; t0 < cache->n_tensors; t0 += pkv::kMaxTensorsPerLaunch) {
        const int32_t nt = std::min(pkv::kMaxTensorsPerLaunch, cache->n_tensors - t0);
        for (int32_t t = 0; t < nt; t++) {
            p.dst[t] = cache->base[t0 + t];
            for (int32_t pl = 0; pl < cache->n_planes; pl++)
                p.src[t * cache->n_planes + pl] = new_kv[(int64_t)(t0 + t) * cache->n_planes + pl];
        }
        p.slot_out = t0 == 0 ? slot_out : nullptr;
        int64_t per_tensor_ctas, cap;
        row_grid(cache, n_tokens, nt, *dev, &per_tensor_ctas, &cap);
        int64_t ctas = std::min(per_tensor_ctas, cap);
        if (PKV_RESHAPE_ROWS && row_group <= kMaxRowGroup) {
            ctas = (ctas + row_group - 1) / row_group * row_group;
            p.tok_step = (uint32_t)(ctas * kRowThreads / (cache->n_planes * cpr));
            pkv::launch(reshape_rows_kernel<FUSED>, dim3((unsigned)ctas, (unsigned)nt), kRowThreads, 0, stream, p);
        } else {
            pkv::launch(reshape_and_cache_kernel<FUSED>, dim3((unsigned)ctas, (unsigned)nt), kRowThreads, 0, stream, p);
        }
        st = pkv::cuda_status(cudaGetLastError());
        if (st != KV_OK) return st;
    }
    return KV_OK;
}

}  // namespace

int pkv::preload_write_kernels()
{
    return pkv::load_kernels(slot_mapping_kernel, reshape_and_cache_kernel<true>, reshape_and_cache_kernel<false>,
                             reshape_rows_kernel<true>, reshape_rows_kernel<false>);
}

extern "C" {

int kv_slot_mapping(const int32_t *block_table, int32_t n_reqs, int32_t max_blocks_per_req,
                    int64_t bt_row_stride, const int32_t *token_req, const int32_t *token_pos,
                    int64_t n_tokens, int32_t block_size, int64_t *slot_out, kv_stream_t stream)
{
    if (n_tokens < 0 || n_reqs < 0 || max_blocks_per_req < 0 || block_size <= 0 || bt_row_stride < 0)
        return KV_ERR_INVALID_ARG;
    if (n_tokens == 0) return KV_OK;
    if (token_req == nullptr || token_pos == nullptr || slot_out == nullptr ||
        (n_reqs > 0 && max_blocks_per_req > 0 && block_table == nullptr))
        return KV_ERR_INVALID_ARG;
    if (n_reqs > 0 && bt_row_stride < max_blocks_per_req) return KV_ERR_INVALID_ARG;
    const pkv::DeviceInfo *dev = pkv::current_device();
    if (dev == nullptr) return KV_ERR_CUDA;
    const int threads = 256;
    const int64_t need = (n_tokens + threads - 1) / threads;
    const int blocks = (int)std::min<int64_t>(need, (int64_t)dev->num_sms * 16);
    pkv::launch(slot_mapping_kernel, blocks, threads, 0, (cudaStream_t)stream, block_table, n_reqs, max_blocks_per_req,
                bt_row_stride, token_req, token_pos, n_tokens, block_size, slot_out, dev->err_word);
    return pkv::cuda_status(cudaGetLastError());
}

int kv_reshape_and_cache(const kv_cache_desc *cache, const uint64_t *new_kv, int64_t new_token_stride,
                         const int64_t *slot, int64_t n_tokens, kv_stream_t stream)
{
    if (n_tokens > 0 && slot == nullptr) return KV_ERR_INVALID_ARG;
    ReshapeParams p{};
    p.slot = slot;
    return launch_rows<false>(cache, new_kv, new_token_stride, n_tokens, p, (cudaStream_t)stream);
}

int kv_write_tokens(const kv_cache_desc *cache, const uint64_t *new_kv, int64_t new_token_stride,
                    const int32_t *block_table, int32_t n_reqs, int32_t max_blocks_per_req, int64_t bt_row_stride,
                    const int32_t *token_req, const int32_t *token_pos, int64_t n_tokens, int64_t *slot_out,
                    kv_stream_t stream)
{
    if (n_reqs < 0 || max_blocks_per_req < 0 || bt_row_stride < 0) return KV_ERR_INVALID_ARG;
    if (n_tokens > 0 && (token_req == nullptr || token_pos == nullptr ||
                         (n_reqs > 0 && max_blocks_per_req > 0 && block_table == nullptr)))
        return KV_ERR_INVALID_ARG;
    if (n_reqs > 0 && bt_row_stride < max_blocks_per_req) return KV_ERR_INVALID_ARG;
    // In the fused kernel every pass of a thread waits on the table lookup's two dependent
    // loads.  With slot_out given, the batch runs as slot_mapping into slot_out followed by the
    // plain row copy instead: the same results, and the row copy's launch overlaps slot_mapping
    // (programmatic dependent launch), so it is faster for a decode write too.
    bool nothing = false;
    int st = validate_rows(cache, new_kv, new_token_stride, n_tokens, &nothing);
    if (st != KV_OK || nothing) return st;
    if (slot_out != nullptr) {
        const pkv::DeviceInfo *dev = pkv::current_device();
        if (dev == nullptr) return KV_ERR_CUDA;
        int64_t need, cap;
        row_grid(cache, n_tokens, std::min(pkv::kMaxTensorsPerLaunch, cache->n_tensors), *dev, &need, &cap);
        if (need > kWriteSplitIterations * cap) {
            st = kv_slot_mapping(block_table, n_reqs, max_blocks_per_req, bt_row_stride, token_req, token_pos,
                                 n_tokens, cache->block_size, slot_out, stream);
            if (st != KV_OK) return st;
            return kv_reshape_and_cache(cache, new_kv, new_token_stride, slot_out, n_tokens, stream);
        }
    }
    ReshapeParams p{};
    p.table = block_table;
    p.token_req = token_req;
    p.token_pos = token_pos;
    p.slot_out = slot_out;
    p.table_row_stride = bt_row_stride;
    p.n_reqs = n_reqs;
    p.max_blocks = max_blocks_per_req;
    return launch_rows<true>(cache, new_kv, new_token_stride, n_tokens, p, (cudaStream_t)stream);
}

}  // extern "C"
