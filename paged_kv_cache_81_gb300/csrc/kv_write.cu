// kv_slot_mapping, kv_reshape_and_cache and kv_write_tokens: writing new tokens' K/V into the
// paged cache.
//
// Slot formula: drawing "vllm v1 调度逻辑 和 distributed 分布式原理", label "batch tensor 组装";
// block = slots 0..15 of K/V rows: label "Paged kv cache"; one block_table serves every
// layer: the per-layer tensor panel (layer_0 .. layer_47).
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
    int64_t *slot_out;  // optional, fused token-strided kernel: the looked-up slots (first launch only)
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
#ifndef PKV_RESHAPE_FUSED_MIN_CTAS
#define PKV_RESHAPE_FUSED_MIN_CTAS 4  // the same hint for the fused row write (more state per row in flight)
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
// loads, then the stores: a load placed after a store cannot be moved above it (the compiler
// must assume they may alias), so interleaving them would make each row's slot load wait for
// the previous row's store.
struct RowCoords {
    const uint8_t *src;  // the thread's chunk of token 0's row
    uint8_t *dst;        // the thread's chunk of the row at slot 0 of block 0
    uint32_t tok0;       // the thread's first token (>= n_tokens when the thread has no work)
    bool reporter;       // tensor 0, plane 0, chunk 0: the one thread per token that reports
};

__device__ __forceinline__ RowCoords row_coords(const ReshapeParams &p)
{
    const int t = blockIdx.y;
    const uint32_t first = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t row0 = pkv::fdiv(first, p.div_cpr);
    const uint32_t chunk = first - row0 * p.div_cpr.d;
    const uint32_t tok0 = pkv::fdiv(row0, p.div_planes);
    const uint32_t plane = row0 - tok0 * p.div_planes.d;
    return RowCoords{reinterpret_cast<const uint8_t *>(p.src[t * p.n_planes + plane]) + chunk * 16,
                     reinterpret_cast<uint8_t *>(p.dst[t]) + (int64_t)plane * p.plane_stride + chunk * 16, tok0,
                     t == 0 && plane == 0 && chunk == 0};
}

__global__ void __launch_bounds__(256, PKV_RESHAPE_MIN_CTAS) reshape_rows_kernel(const __grid_constant__ ReshapeParams p)
{
    pkv::grid_dep_entry();  // before any global memory access
    constexpr int64_t kNoRow = INT64_MIN;  // past the last token
    const RowCoords rc = row_coords(p);
    for (uint32_t tok = rc.tok0; tok < p.n_tokens; tok += p.tok_step * kReshapeUnroll) {
        uint4 v[kReshapeUnroll];
        int64_t s[kReshapeUnroll];
#pragma unroll
        for (int u = 0; u < kReshapeUnroll; u++) {
            const uint32_t tk = tok + u * p.tok_step;
            if (tk < p.n_tokens) v[u] = pkv::ld_once(rc.src + (int64_t)tk * p.src_token_stride);
        }
#pragma unroll
        for (int u = 0; u < kReshapeUnroll; u++) {
            const uint32_t tk = tok + u * p.tok_step;
            s[u] = tk < p.n_tokens ? p.slot[tk] : kNoRow;
        }
#pragma unroll
        for (int u = 0; u < kReshapeUnroll; u++) {
            if (s[u] < 0) continue;  // padding token, or past the last token
            if (s[u] >= (int64_t)p.slot_limit) {
                pkv::set_error(p.err, KV_DERR_SLOT);
                continue;
            }
            const uint32_t block = pkv::fdiv((uint32_t)s[u], p.div_bs);
            const uint32_t off = (uint32_t)s[u] - block * p.div_bs.d;
            pkv::st_stream(rc.dst + (int64_t)block * p.block_stride + (int64_t)off * p.token_stride, v[u]);
        }
    }
}

// The same row write with each token's slot looked up in the block table (kv_write_tokens).
// A slot takes two dependent loads: the token's request and position, then its table entry.
// The first pair for the next pass is loaded during this pass, so a pass issues its row loads
// and its table loads together and waits about one round trip, as the plain row write does.
// The state this keeps in flight needs 64 registers: 4 CTAs per SM.
__global__ void __launch_bounds__(256, PKV_RESHAPE_FUSED_MIN_CTAS)
    reshape_rows_fused_kernel(const __grid_constant__ ReshapeParams p)
{
    pkv::grid_dep_entry();  // before any global memory access
    const RowCoords rc = row_coords(p);
    const uint32_t bs = p.div_bs.d;
    int32_t rq[kReshapeUnroll], ps[kReshapeUnroll];  // this pass's tokens' request and position
#pragma unroll
    for (int u = 0; u < kReshapeUnroll; u++) {
        const uint32_t tk = rc.tok0 + u * p.tok_step;
        rq[u] = tk < p.n_tokens ? p.token_req[tk] : -1;
        ps[u] = tk < p.n_tokens ? p.token_pos[tk] : 0;
    }
    for (uint32_t tok = rc.tok0; tok < p.n_tokens; tok += p.tok_step * kReshapeUnroll) {
        uint4 v[kReshapeUnroll];
        int32_t blk[kReshapeUnroll];  // table entry, or -1: the token has no slot
        uint32_t off[kReshapeUnroll];
#pragma unroll
        for (int u = 0; u < kReshapeUnroll; u++) {
            const uint32_t tk = tok + u * p.tok_step;
            if (tk < p.n_tokens) v[u] = pkv::ld_once(rc.src + (int64_t)tk * p.src_token_stride);
        }
#pragma unroll
        for (int u = 0; u < kReshapeUnroll; u++) {
            blk[u] = -1;
            off[u] = 0;
            if (rq[u] >= 0 && rq[u] < p.n_reqs && ps[u] >= 0) {
                const uint32_t q = pkv::fdiv((uint32_t)ps[u], p.div_bs);
                if (q < (uint32_t)p.max_blocks) {
                    blk[u] = p.table[(int64_t)rq[u] * p.table_row_stride + q];
                    off[u] = (uint32_t)ps[u] - q * bs;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kReshapeUnroll; u++) {  // the next pass's requests and positions
            const uint32_t tk = tok + (kReshapeUnroll + u) * p.tok_step;
            rq[u] = tk < p.n_tokens ? p.token_req[tk] : -1;
            ps[u] = tk < p.n_tokens ? p.token_pos[tk] : 0;
        }
#pragma unroll
        for (int u = 0; u < kReshapeUnroll; u++) {
            const uint32_t tk = tok + u * p.tok_step;
            if (tk >= p.n_tokens) continue;
            if (rc.reporter && p.slot_out != nullptr) p.slot_out[tk] = blk[u] < 0 ? -1 : (int64_t)blk[u] * bs + off[u];
            if (blk[u] < 0) {
                if (rc.reporter) pkv::set_error(p.err, KV_DERR_TABLE);
                continue;
            }
            if ((int64_t)blk[u] * bs + off[u] >= (int64_t)p.slot_limit) {
                pkv::set_error(p.err, KV_DERR_SLOT);
                continue;
            }
            pkv::st_stream(rc.dst + (int64_t)blk[u] * p.block_stride + (int64_t)off[u] * p.token_stride, v[u]);
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

// CTAs a grid stride must be a multiple of to cover whole tokens (planes x chunks per row
// divides 256 x CTAs), or 0 when that is above kMaxRowGroup and the general kernel runs.
int64_t row_group_ctas(const kv_cache_desc *cache)
{
    const int64_t per_token = cache->n_planes * (int64_t)(cache->row_bytes / 16);
    const int64_t g = per_token / std::gcd<int64_t>(kRowThreads, per_token);
    return PKV_RESHAPE_ROWS && g <= kMaxRowGroup ? g : 0;
}

#ifndef PKV_RESHAPE_WAVES
#define PKV_RESHAPE_WAVES 64  // the row-write grid's cap, in waves of 8 CTAs per SM
#endif

// CTAs per tensor of a row-write launch: enough for the work, at most about PKV_RESHAPE_WAVES
// waves of 8 resident CTAs per SM over the nt tensors of the launch.
void row_grid(const kv_cache_desc *cache, int64_t n_tokens, int32_t nt, const pkv::DeviceInfo &dev, int64_t *need,
              int64_t *cap)
{
    const int64_t total = n_tokens * cache->n_planes * (cache->row_bytes / 16);
    *need = (total + (int64_t)kRowThreads * kReshapeUnroll - 1) / ((int64_t)kRowThreads * kReshapeUnroll);
    *cap = std::max<int64_t>(1, ((int64_t)dev.num_sms * 8 * PKV_RESHAPE_WAVES + nt - 1) / nt);
}

// A row write of at most two waves (of 8 CTAs per SM) takes programmatic dependent launch; a
// larger one launches plainly (kv_common.cuh, launch_as).
inline bool pdl_rows(int64_t ctas, const pkv::DeviceInfo &dev) { return ctas <= 2ll * dev.num_sms * 8; }

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
    const int64_t row_group = row_group_ctas(cache);

    for (int32_t t0 = 0; t0 < cache->n_tensors; t0 += pkv::kMaxTensorsPerLaunch) {
        const int32_t nt = std::min(pkv::kMaxTensorsPerLaunch, cache->n_tensors - t0);
        if (t0 > 0) p.slot_out = nullptr;  // every launch covers the same tokens
        for (int32_t t = 0; t < nt; t++) {
            p.dst[t] = cache->base[t0 + t];
            for (int32_t pl = 0; pl < cache->n_planes; pl++)
                p.src[t * cache->n_planes + pl] = new_kv[(int64_t)(t0 + t) * cache->n_planes + pl];
        }
        int64_t per_tensor_ctas, cap;
        row_grid(cache, n_tokens, nt, *dev, &per_tensor_ctas, &cap);
        int64_t ctas = std::min(per_tensor_ctas, cap);
        if (row_group > 0) {
            ctas = (ctas + row_group - 1) / row_group * row_group;
            if (FUSED) {
                // A write that one wave of the fused kernel covers in two passes per thread runs
                // as that wave: the second pass's lookups are loaded before the first pass ends,
                // which beats a second, partial wave (61-layer decode: 5.0 instead of 5.4 us).
                const int64_t wave = (int64_t)dev->num_sms * PKV_RESHAPE_FUSED_MIN_CTAS / nt / row_group * row_group;
                if (wave >= row_group && ctas > wave && ctas <= 2 * wave) ctas = wave;
            }
            p.tok_step = (uint32_t)(ctas * kRowThreads / (cache->n_planes * cpr));
            pkv::launch_as(pdl_rows(ctas * nt, *dev), FUSED ? reshape_rows_fused_kernel : reshape_rows_kernel,
                           dim3((unsigned)ctas, (unsigned)nt), kRowThreads, 0, stream, p);
        } else {
            pkv::launch_as(pdl_rows(ctas * nt, *dev), reshape_and_cache_kernel<FUSED>, dim3((unsigned)ctas, (unsigned)nt),
                           kRowThreads, 0, stream, p);
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
                             reshape_rows_kernel, reshape_rows_fused_kernel);
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
    // The row copy looks each token's slot up in the block table (and reports it in slot_out).
    // A row shape that takes the general kernel, whose lookup is not pipelined, runs as
    // slot_mapping followed by the plain row copy when slot_out can hold the slots.
    bool nothing = false;
    int st = validate_rows(cache, new_kv, new_token_stride, n_tokens, &nothing);
    if (st != KV_OK || nothing) return st;
    if (slot_out != nullptr && row_group_ctas(cache) == 0) {
        st = kv_slot_mapping(block_table, n_reqs, max_blocks_per_req, bt_row_stride, token_req, token_pos, n_tokens,
                             cache->block_size, slot_out, stream);
        if (st != KV_OK) return st;
        return kv_reshape_and_cache(cache, new_kv, new_token_stride, slot_out, n_tokens, stream);
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
