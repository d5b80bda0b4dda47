// Step a2: sort (token, expert) pairs into block-padded per-expert spans.
//
// Restates ferrum-kernels 0.7.7 src/backend/cuda/moe.rs, moe_align_block_size
// (+ the _pair_ids variant) and moe_build_pairs_by_token: a counting sort by
// expert, each span padded to a block_size multiple with a sentinel, one
// expert id per block, the padded prefix expert_offsets and the inverse
// pair -> row map. The page runs one 256-thread block sized for about a
// thousand pairs; here the pairs are split in chunks so that 131072 pairs
// spread over the whole GPU, and the result stays deterministic: a pair's row
// is fixed by counts, never by the order atomics land in.
//
//   1. count_rank: each warp walks 256 consecutive pairs in 8 steps of 32 and
//      gives every pair its stable rank among same-expert pairs of the warp
//      (__match_any_sync + popcount of lower lanes + a per-warp running count);
//      the block then turns the per-warp counts into per-warp bases and
//      writes the chunk's per-expert totals.
//   2. scan (one block): per expert, the exclusive prefix over chunks, the
//      padded span, the prefix over experts, expert_ids, sentinels, the tail.
//   3. scatter: row = base[chunk][expert] + rank in chunk.
// Batches of at most one chunk (2048 pairs) run all three steps in a single
// block instead, with the ranks kept in registers.
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kPairsPerWarp = 256;
constexpr int kChunk = kWarps * kPairsPerWarp;  // pairs per block of count_rank
constexpr int kSteps = kPairsPerWarp / 32;

inline int n_chunks(int P) { return (P + kChunk - 1) / kChunk; }

__global__ void __launch_bounds__(32 * kWarps)
align_count_rank_kernel(const int32_t* __restrict__ ids, int P, int E, int32_t* __restrict__ chunk_counts,
                        int32_t* __restrict__ rank_in_chunk, int32_t* err) {
    pdl_wait();
    __shared__ int cnt[kWarps][MOE_MAX_EXPERTS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kWarps * MOE_MAX_EXPERTS; i += blockDim.x) (&cnt[0][0])[i] = 0;
    __syncthreads();

    const int base = blockIdx.x * kChunk + warp * kPairsPerWarp;
    const unsigned lt_mask = (1u << lane) - 1u;
    int my_id[kSteps], my_rank[kSteps];
#pragma unroll
    for (int s = 0; s < kSteps; ++s) {
        const int p = base + s * 32 + lane;
        int id = -1;
        if (p < P) {
            id = ids[p];
            if (id < 0 || id >= E) {
                set_err(err, MOE_DEV_ERR_EXPERT_ID);
                id = -1;
            }
        }
        const unsigned peers = __match_any_sync(0xffffffffu, id);
        const int rank = __popc(peers & lt_mask);
        int before = 0;
        if (id >= 0) before = cnt[warp][id];
        __syncwarp();
        if (id >= 0 && rank == 0) cnt[warp][id] = before + __popc(peers);
        __syncwarp();
        my_id[s] = id;
        my_rank[s] = before + rank;
    }
    __syncthreads();
    // per expert: exclusive prefix over the warps of this chunk
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const int c = cnt[w][e];
            cnt[w][e] = run;
            run += c;
        }
        chunk_counts[static_cast<size_t>(blockIdx.x) * E + e] = run;
    }
    __syncthreads();
#pragma unroll
    for (int s = 0; s < kSteps; ++s) {
        const int p = base + s * 32 + lane;
        if (p < P) rank_in_chunk[p] = my_id[s] >= 0 ? cnt[warp][my_id[s]] + my_rank[s] : -1;
    }
}

__global__ void __launch_bounds__(MOE_MAX_EXPERTS)
align_scan_kernel(int P, int E, int bs, int max_padded, int nchunks, int32_t* __restrict__ chunk_counts,
                  int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                  int32_t* __restrict__ offsets, int32_t* __restrict__ total_post_pad, int32_t* err) {
    pdl_wait();
    __shared__ int s_span[MOE_MAX_EXPERTS];
    __shared__ int s_total;
    const int e = threadIdx.x;
    int count = 0;
    if (e < E) {
        for (int b = 0; b < nchunks; ++b) {
            int32_t* c = chunk_counts + static_cast<size_t>(b) * E + e;
            const int v = *c;
            *c = count;
            count += v;
        }
    }
    const int span = (count + bs - 1) / bs * bs;
    s_span[e] = (e < E) ? span : 0;
    __syncthreads();
    // exclusive prefix over experts (Hillis-Steele on 256 entries)
    for (int d = 1; d < MOE_MAX_EXPERTS; d <<= 1) {
        const int add = (e >= d) ? s_span[e - d] : 0;
        __syncthreads();
        s_span[e] += add;
        __syncthreads();
    }
    const int off = s_span[e] - ((e < E) ? span : 0);  // inclusive -> exclusive
    if (e == MOE_MAX_EXPERTS - 1) s_total = s_span[e];
    __syncthreads();
    const int total = s_total;
    if (total > max_padded) {  // cannot happen when max_padded >= the capacity bound
        if (e == 0) set_err(err, MOE_DEV_ERR_CAPACITY);
        return;
    }
    if (e < E) {
        offsets[e] = off;
        for (int b = 0; b < nchunks; ++b) chunk_counts[static_cast<size_t>(b) * E + e] += off;
        for (int blk = off / bs; blk < (off + span) / bs; ++blk) expert_ids[blk] = e;
        for (int r = off + count; r < off + span; ++r) sorted_ids[r] = P;
    }
    if (e == 0) {
        offsets[E] = total;
        total_post_pad[0] = total;
    }
    for (int r = total + e; r < max_padded; r += blockDim.x) sorted_ids[r] = P;
    for (int blk = total / bs + e; blk < max_padded / bs; blk += blockDim.x) expert_ids[blk] = -1;
}

__global__ void align_scatter_kernel(const int32_t* __restrict__ ids, int P, int E,
                                     const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ rank_in_chunk,
                                     int32_t* __restrict__ sorted_ids, int32_t* __restrict__ pair_to_row) {
    pdl_wait();
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= P) return;
    const int id = ids[p];
    if (id < 0 || id >= E) {
        pair_to_row[p] = -1;
        return;
    }
    const int row = chunk_base[static_cast<size_t>(p / kChunk) * E + id] + rank_in_chunk[p];
    sorted_ids[row] = p;
    pair_to_row[p] = row;
}

// Small batches (P <= kChunk): the three steps in one block, ranks kept in
// registers, no workspace. Same ordering rules, so the same result.
__global__ void __launch_bounds__(32 * kWarps)
align_single_block_kernel(const int32_t* __restrict__ ids, int P, int E, int bs, int max_padded,
                          int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                          int32_t* __restrict__ offsets, int32_t* __restrict__ total_post_pad,
                          int32_t* __restrict__ pair_to_row, int32_t* err) {
    pdl_wait();
    __shared__ int cnt[kWarps][MOE_MAX_EXPERTS];
    __shared__ int s_span[MOE_MAX_EXPERTS];
    __shared__ int s_off[MOE_MAX_EXPERTS];
    __shared__ int s_total;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, e = threadIdx.x;
    for (int i = threadIdx.x; i < kWarps * MOE_MAX_EXPERTS; i += blockDim.x) (&cnt[0][0])[i] = 0;
    __syncthreads();
    // 1. stable rank of every pair among same-expert pairs of its warp
    const int base = warp * kPairsPerWarp;
    const unsigned lt_mask = (1u << lane) - 1u;
    int my_id[kSteps], my_rank[kSteps];
#pragma unroll
    for (int st = 0; st < kSteps; ++st) {
        const int p = base + st * 32 + lane;
        int id = -1;
        if (p < P) {
            id = ids[p];
            if (id < 0 || id >= E) {
                set_err(err, MOE_DEV_ERR_EXPERT_ID);
                id = -1;
            }
        }
        const unsigned peers = __match_any_sync(0xffffffffu, id);
        const int rank = __popc(peers & lt_mask);
        int before = 0;
        if (id >= 0) before = cnt[warp][id];
        __syncwarp();
        if (id >= 0 && rank == 0) cnt[warp][id] = before + __popc(peers);
        __syncwarp();
        my_id[st] = id;
        my_rank[st] = before + rank;
    }
    __syncthreads();
    // 2. per expert: warp bases, count, padded span; prefix over experts
    int count = 0;
    if (e < E) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const int c = cnt[w][e];
            cnt[w][e] = count;
            count += c;
        }
    }
    const int span = (count + bs - 1) / bs * bs;
    s_span[e] = (e < E) ? span : 0;
    __syncthreads();
    for (int d = 1; d < MOE_MAX_EXPERTS; d <<= 1) {
        const int add = (e >= d) ? s_span[e - d] : 0;
        __syncthreads();
        s_span[e] += add;
        __syncthreads();
    }
    const int off = s_span[e] - ((e < E) ? span : 0);
    s_off[e] = off;
    if (e == MOE_MAX_EXPERTS - 1) s_total = s_span[e];
    __syncthreads();
    const int total = s_total;
    if (total > max_padded) {  // cannot happen when max_padded >= the capacity bound
        if (e == 0) set_err(err, MOE_DEV_ERR_CAPACITY);
        return;
    }
    if (e < E) {
        offsets[e] = off;
        for (int blk = off / bs; blk < (off + span) / bs; ++blk) expert_ids[blk] = e;
        for (int r = off + count; r < off + span; ++r) sorted_ids[r] = P;
    }
    if (e == 0) {
        offsets[E] = total;
        total_post_pad[0] = total;
    }
    for (int r = total + e; r < max_padded; r += blockDim.x) sorted_ids[r] = P;
    for (int blk = total / bs + e; blk < max_padded / bs; blk += blockDim.x) expert_ids[blk] = -1;
    // 3. scatter
#pragma unroll
    for (int st = 0; st < kSteps; ++st) {
        const int p = base + st * 32 + lane;
        if (p < P) {
            const int id = my_id[st];
            if (id >= 0) {
                const int row = s_off[id] + cnt[warp][id] + my_rank[st];
                sorted_ids[row] = p;
                pair_to_row[p] = row;
            } else {
                pair_to_row[p] = -1;
            }
        }
    }
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_align_workspace_size(int32_t P, int32_t E) {
    if (P < 0 || E < 1) return 0;
    const size_t chunks = static_cast<size_t>(moe::n_chunks(P));
    const size_t a = (chunks * E * sizeof(int32_t) + 255) / 256 * 256;
    return a + static_cast<size_t>(P) * sizeof(int32_t) + 256;
}

extern "C" int moe_align_block_size(const int32_t* topk_ids, int32_t P, int32_t E, int32_t block_size,
                                    int32_t max_padded, int32_t* sorted_token_ids, int32_t* expert_ids,
                                    int32_t* expert_offsets, int32_t* total_tokens_post_pad, int32_t* pair_to_row,
                                    int32_t* err_word, void* workspace, size_t workspace_bytes, void* stream) {
    MOE_REQUIRE(E >= 1 && E <= MOE_MAX_EXPERTS,
                "moe_align_block_size: num_experts=%d exceeds compile-time MAX_NUM_EXPERTS=%d (or is < 1)", E,
                MOE_MAX_EXPERTS);
    MOE_REQUIRE(block_size >= 1, "moe_align_block_size: block_size=%d must be positive", block_size);
    MOE_REQUIRE(P >= 0, "moe_align_block_size: P=%d is negative", P);
    const int64_t cap = moe_align_capacity(P, E, block_size);
    MOE_REQUIRE(max_padded >= cap && max_padded % block_size == 0,
                "moe_align_block_size: max_padded=%d must be a multiple of block_size=%d and >= capacity %lld",
                max_padded, block_size, (long long)cap);
    MOE_REQUIRE(sorted_token_ids && expert_ids && expert_offsets && total_tokens_post_pad,
                "moe_align_block_size: NULL output");
    MOE_REQUIRE(P == 0 || (topk_ids && pair_to_row), "moe_align_block_size: NULL topk_ids / pair_to_row");
    const size_t need = moe_align_workspace_size(P, E);
    MOE_REQUIRE(workspace && workspace_bytes >= need && moe::aligned16(workspace),
                "moe_align_block_size: workspace of %zu bytes (16-byte aligned) required, got %zu", need,
                workspace_bytes);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int nchunks = moe::n_chunks(P);
    int32_t* chunk_counts = static_cast<int32_t*>(workspace);
    int32_t* rank_in_chunk = reinterpret_cast<int32_t*>(
        static_cast<char*>(workspace) + (static_cast<size_t>(nchunks) * E * sizeof(int32_t) + 255) / 256 * 256);
    int launches = 0;
    if (nchunks <= 1) {
        moe::launch_pdl(moe::align_single_block_kernel, 1, 32 * moe::kWarps, 0, st, topk_ids, P, E, block_size, max_padded,
                                                                      sorted_token_ids, expert_ids, expert_offsets,
                                                                      total_tokens_post_pad, pair_to_row, err_word);
        ++launches;
    } else {
        moe::launch_pdl(moe::align_count_rank_kernel, nchunks, 32 * moe::kWarps, 0, st, topk_ids, P, E, chunk_counts,
                                                                          rank_in_chunk, err_word);
        moe::launch_pdl(moe::align_scan_kernel, 1, MOE_MAX_EXPERTS, 0, st, P, E, block_size, max_padded, nchunks, chunk_counts,
                                                             sorted_token_ids, expert_ids, expert_offsets,
                                                             total_tokens_post_pad, err_word);
        moe::launch_pdl(moe::align_scatter_kernel, (P + 255) / 256, 256, 0, st, topk_ids, P, E, chunk_counts, rank_in_chunk,
                                                                  sorted_token_ids, pair_to_row);
        launches += 3;
    }
    moe::count_launch(launches);
    return moe::check_launch("moe_align_block_size");
}

// ---------------------------------------------------------------------------
// Fixed-scratch variant for callers that cannot allocate device memory.
//
// Some callers of this library have no way to allocate device memory for the
// align workspace: an application whose framework has taken the whole device
// memory budget into its own pool and hands out no allocator, or a
// latency-critical caller that must not make an allocation call (which can
// synchronise the device) on its hot path. For them,
// moe_align_block_size_noalloc runs the same three align kernels with their
// scratch in the fixed array below instead of a caller-provided workspace.
//
// The array is sized for MOE_ALIGN_NOALLOC_MAX_PAIRS pairs and up to
// MOE_MAX_EXPERTS experts (about 1.1 MiB). Every GPU that loads this library
// holds it until the process exits. All calls on a device share it and it
// keeps the previous call's contents; the kernels overwrite every word they
// read in the same call, so nothing needs clearing. Two calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on
// the array and may produce wrong results.
// ---------------------------------------------------------------------------

namespace {
constexpr size_t kNoAllocChunks =
    (static_cast<size_t>(MOE_ALIGN_NOALLOC_MAX_PAIRS) + moe::kChunk - 1) / moe::kChunk;
constexpr size_t kNoAllocScratchBytes =
    (kNoAllocChunks * MOE_MAX_EXPERTS * sizeof(int32_t) + 255) / 256 * 256 +
    static_cast<size_t>(MOE_ALIGN_NOALLOC_MAX_PAIRS) * sizeof(int32_t) + 256;
}  // namespace

static __device__ __align__(256) uint8_t g_align_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_noalloc_mu;
// device address of the array per device ordinal, with the context it was
// looked up in: a context destroyed and made again (cudaDeviceReset) reloads
// the module, so the address is looked up again for the new context
struct NoAllocSlot {
    CUcontext ctx;
    void* ptr;
};
NoAllocSlot g_noalloc[256] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

// Looked up with the device current, once per device and context: in host
// code the array's name is only a host-side stand-in, never a device address.
int noalloc_scratch(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return moe::fail(MOE_ERR_CUDA, "moe_align_block_size_noalloc: cudaGetDevice: %s",
                                           cudaGetErrorString(e));
    if (dev < 0 || dev >= 256) return moe::fail(MOE_ERR_UNSUPPORTED, "moe_align_block_size_noalloc: device %d", dev);
    CtxGetCurrentFn get = ctx_get_current();
    if (!get) return moe::fail(MOE_ERR_CUDA, "moe_align_block_size_noalloc: cuCtxGetCurrent is unavailable");
    CUcontext ctx = nullptr;  // NULL until the runtime has made the device's context current
    if (get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (ctx == nullptr || g_noalloc[dev].ptr == nullptr || g_noalloc[dev].ctx != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_align_noalloc_scratch);  // makes the context current if needed
        if (e != cudaSuccess || p == nullptr)
            return moe::fail(MOE_ERR_CUDA, "moe_align_block_size_noalloc: cudaGetSymbolAddress: %s",
                             cudaGetErrorString(e));
        if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr)
            return moe::fail(MOE_ERR_CUDA, "moe_align_block_size_noalloc: cannot read the current context");
        g_noalloc[dev] = NoAllocSlot{ctx, p};
    }
    *out = g_noalloc[dev].ptr;
    return MOE_OK;
}
}  // namespace

extern "C" int moe_align_block_size_noalloc(const int32_t* topk_ids, int32_t P, int32_t E, int32_t block_size,
                                            int32_t max_padded, int32_t* sorted_token_ids, int32_t* expert_ids,
                                            int32_t* expert_offsets, int32_t* total_tokens_post_pad,
                                            int32_t* pair_to_row, int32_t* err_word, void* stream) {
    MOE_REQUIRE(P >= 0 && P <= MOE_ALIGN_NOALLOC_MAX_PAIRS,
                "moe_align_block_size_noalloc: P=%d pairs is outside [0, %d], the size of the fixed scratch; "
                "use moe_align_block_size with a workspace",
                P, MOE_ALIGN_NOALLOC_MAX_PAIRS);
    MOE_REQUIRE(E >= 1 && E <= MOE_MAX_EXPERTS, "moe_align_block_size_noalloc: num_experts=%d outside [1, %d]", E,
                MOE_MAX_EXPERTS);
    void* scratch = nullptr;
    const int rc = noalloc_scratch(&scratch);
    if (rc != MOE_OK) return rc;
    return moe_align_block_size(topk_ids, P, E, block_size, max_padded, sorted_token_ids, expert_ids, expert_offsets,
                                total_tokens_post_pad, pair_to_row, err_word, scratch, kNoAllocScratchBytes, stream);
}
