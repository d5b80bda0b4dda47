// Step a5: the device-side grouped LoRA fold on sorted expert rows.
//
// Restates spark_model/layers/ops/moe_lora_grouped.rs, moe_lora_grouped_down
// and MoeExpertRoute: a shrink (xa = bf16(x . A_e^T)) and an expand + fold
// (base += scale_e * fp32(bf16(xa . B_e^T))) over one window [row_offset,
// row_end) of the sorted rows, with expert spans read from expert_offsets on
// the device. The page sizes a static worst-case grid (ceil(window/64) x
// n_experts) whose tiles mostly return at once; here a persistent grid walks
// only the non-empty 64-row tiles of span intersect window, listed in shared
// memory from expert_offsets at kernel start.
//
// The work is HBM-bound (rank 16: 2 x rank FLOPs per element of base read and
// written), so both kernels are shaped for coalesced 16-byte / 8-byte access:
//   shrink: a warp per row, lanes split k_in in 16-byte chunks, A_e staged in
//           shared memory, rank partial sums reduced across the warp;
//   expand: each thread owns 64 / rank-capacity consecutive output columns
//           and keeps their B_e rows in registers, walking the tile's rows.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kRowTile = 64;
constexpr int kShrinkWarps = 8;
constexpr int kExpandThreads = 256;

struct LoraTiles {
    int n_tiles;
    int tstart[MOE_MAX_EXPERTS + 1];
    int lo[MOE_MAX_EXPERTS];
};

// rows of expert e inside the window: [max(off[e], row_offset), min(off[e+1], row_end))
__device__ void build_lora_tiles(LoraTiles& s, const int32_t* offsets, int n_experts, uint32_t row_offset,
                                 uint32_t row_end, const uint64_t* a_table) {
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        const int per = (n_experts + 31) / 32;
        int cnt[8];
        int loc = 0;
        for (int j = 0; j < per && j < 8; ++j) {
            const int e = lane * per + j;
            int c = 0;
            if (e < n_experts) {
                const int lo = max(offsets[e], static_cast<int>(row_offset));
                const int hi = min(offsets[e + 1], static_cast<int>(row_end));
                s.lo[e] = lo;
                if (hi > lo && a_table[e] != 0) c = (hi - lo + kRowTile - 1) / kRowTile;
            }
            cnt[j] = c;
            loc += c;
        }
        int inc = loc;
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, inc, d);
            if (lane >= d) inc += o;
        }
        int run = inc - loc;
        for (int j = 0; j < per && j < 8; ++j) {
            const int e = lane * per + j;
            if (e < n_experts) {
                s.tstart[e] = run;
                run += cnt[j];
            }
        }
        if (lane == 31) {
            s.n_tiles = inc;
            s.tstart[n_experts] = inc;
        }
    }
    __syncthreads();
}

__device__ __forceinline__ int lora_tile_expert(const LoraTiles& s, int n_experts, int tile) {
    int lo = 0, hi = n_experts - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.tstart[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// returns the x row of sorted row r, or -1 when the row folds nothing
__device__ __forceinline__ int lora_row_source(int r, const int32_t* sorted_ids, const int32_t* row_adapter, int P,
                                               int top_k, uint32_t x_gather, int32_t* err) {
    const int p = sorted_ids[r];
    if (p == P) return -1;
    if (p < 0 || p > P) {
        set_err(err, MOE_DEV_ERR_PAIR_ID);
        return -1;
    }
    const int tok = p / top_k;
    if (row_adapter && row_adapter[tok] < 0) return -1;
    return x_gather ? tok : r;
}

__global__ void __launch_bounds__(32 * kShrinkWarps)
lora_shrink_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ offsets,
                   const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ row_adapter,
                   const uint64_t* __restrict__ a_table, __nv_bfloat16* __restrict__ xa, int n_experts, int max_rank,
                   int k_in, uint32_t x_gather, uint32_t row_offset, uint32_t row_end, int P, int top_k,
                   int32_t* err) {
    pdl_wait();
    extern __shared__ __align__(16) uint8_t smem[];
    LoraTiles& s = *reinterpret_cast<LoraTiles*>(smem);
    __nv_bfloat16* sA = reinterpret_cast<__nv_bfloat16*>(smem + ((sizeof(LoraTiles) + 15) / 16) * 16);
    build_lora_tiles(s, offsets, n_experts, row_offset, row_end, a_table);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunks = k_in / 8;
    int cur_e = -1;
    for (int tile = blockIdx.x; tile < s.n_tiles; tile += gridDim.x) {
        const int e = lora_tile_expert(s, n_experts, tile);
        if (e != cur_e) {  // stage A_e [max_rank, k_in] (block-uniform)
            __syncthreads();
            const uint4* src = reinterpret_cast<const uint4*>(a_table[e]);
            for (int i = threadIdx.x; i < max_rank * chunks; i += blockDim.x)
                reinterpret_cast<uint4*>(sA)[i] = __ldg(src + i);
            __syncthreads();
            cur_e = e;
        }
        const int r0 = s.lo[e] + (tile - s.tstart[e]) * kRowTile;
        const int hi = min(offsets[e + 1], static_cast<int>(row_end));
        for (int rr = warp; rr < kRowTile; rr += kShrinkWarps) {
            const int r = r0 + rr;
            if (r >= hi) break;
            const int src_row = lora_row_source(r, sorted_ids, row_adapter, P, top_k, x_gather, err);
            if (src_row < 0) continue;
            const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(src_row) * k_in);
            for (int j0 = 0; j0 < max_rank; j0 += 16) {
                float acc[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
                for (int c = lane; c < chunks; c += 32) {
                    const uint4 xv = __ldg(xr + c);
                    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (j0 + j < max_rank) {
                            const uint4 av = reinterpret_cast<const uint4*>(sA)[(j0 + j) * chunks + c];
                            const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float2 a2 = Act<MOE_ACT_BF16>::unpack2(aw[q]);
                                const float2 x2 = Act<MOE_ACT_BF16>::unpack2(xw[q]);
                                acc[j] = fmaf(x2.x, a2.x, acc[j]);
                                acc[j] = fmaf(x2.y, a2.y, acc[j]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < 16; ++j)
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], off);
                if (lane < 16 && j0 + lane < max_rank) {
                    float v = 0.0f;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (j == lane) v = acc[j];
                    xa[static_cast<size_t>(r - row_offset) * max_rank + j0 + lane] = __float2bfloat16_rn(v);
                }
            }
        }
    }
}

// RCAP: rank capacity of this instantiation; CPC: output columns per thread,
// chosen so a thread holds RCAP * CPC = 64 B_e values in registers.
template <int RCAP>
__global__ void __launch_bounds__(kExpandThreads)
lora_expand_fold_kernel(const __nv_bfloat16* __restrict__ xa, const int32_t* __restrict__ offsets,
                        const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ row_adapter,
                        const uint64_t* __restrict__ b_table, const float* __restrict__ scale_table,
                        __nv_bfloat16* __restrict__ base, int n_experts, int n_out, int max_rank, uint32_t row_offset,
                        uint32_t row_end, int P, int top_k, const uint64_t* __restrict__ a_table) {
    pdl_wait();
    constexpr int CPC = 64 / RCAP;
    __shared__ LoraTiles s;
    __shared__ int s_src[kRowTile];
    __shared__ __align__(16) float s_xa[kRowTile][RCAP];
    build_lora_tiles(s, offsets, n_experts, row_offset, row_end, a_table);
    for (int tile = blockIdx.x; tile < s.n_tiles; tile += gridDim.x) {
        const int e = lora_tile_expert(s, n_experts, tile);
        const int r0 = s.lo[e] + (tile - s.tstart[e]) * kRowTile;
        const int hi = min(offsets[e + 1], static_cast<int>(row_end));
        const int nrows = min(kRowTile, hi - r0);
        __syncthreads();  // previous tile done with s_src / s_xa
        for (int i = threadIdx.x; i < nrows; i += blockDim.x)
            s_src[i] = lora_row_source(r0 + i, sorted_ids, row_adapter, P, top_k, 0, nullptr);
        __syncthreads();
        for (int i = threadIdx.x; i < nrows * RCAP; i += blockDim.x) {
            const int rr = i / RCAP, j = i - rr * RCAP;
            s_xa[rr][j] = (s_src[rr] >= 0 && j < max_rank)
                              ? __bfloat162float(xa[static_cast<size_t>(r0 + rr - row_offset) * max_rank + j])
                              : 0.0f;
        }
        __syncthreads();
        const float sc = scale_table[e];
        const __nv_bfloat16* B = reinterpret_cast<const __nv_bfloat16*>(b_table[e]);
        for (int n0 = threadIdx.x * CPC; n0 < n_out; n0 += blockDim.x * CPC) {
            float bw[CPC][RCAP];
#pragma unroll
            for (int i = 0; i < CPC; ++i)
#pragma unroll
                for (int j = 0; j < RCAP; ++j)
                    bw[i][j] = (j < max_rank) ? __bfloat162float(B[static_cast<size_t>(n0 + i) * max_rank + j]) : 0.0f;
            for (int rr = 0; rr < nrows; ++rr) {
                if (s_src[rr] < 0) continue;
                __nv_bfloat16* yrow = base + static_cast<size_t>(r0 + rr) * n_out + n0;
#pragma unroll
                for (int i = 0; i < CPC; ++i) {
                    float acc = 0.0f;
#pragma unroll
                    for (int j = 0; j < RCAP; ++j) acc = fmaf(s_xa[rr][j], bw[i][j], acc);
                    const float d = __bfloat162float(__float2bfloat16_rn(acc));  // bf16 delta
                    const float y = __bfloat162float(yrow[i]);
                    yrow[i] = __float2bfloat16_rn(__fadd_rn(y, __fmul_rn(sc, d)));
                }
            }
        }
    }
}

// ---- decode gather fold: slot-major rows --------------------------------------
//
// Restates [lora] moe_lora_gather_bgmv: row s = t * top_k + j of the flat
// (token, slot) rows takes its expert from indices[s] and its adapt decision
// from row_adapter[s / top_k]; no expert sort. Decode batches have few rows,
// so a block serves one row: its eight warps split the rank for the shrink,
// then its threads split the output columns for the expand.

// the expert row s folds with, or -1 when it folds nothing
__device__ __forceinline__ int gather_row_expert(uint32_t s, const uint32_t* indices, const int32_t* row_adapter,
                                                 const uint64_t* a_table, uint32_t n_experts, uint32_t top_k) {
    const uint32_t e = indices[s];
    if (e >= n_experts || a_table[e] == 0) return -1;
    if (row_adapter && row_adapter[s / top_k] < 0) return -1;
    return static_cast<int>(e);
}

// One block per row s, shrink and expand in one launch (the page uses two):
//   xa[s, j] = bf16(x_row . A_e[j]), warp w taking j = w, w + 8, ...;
//   base[s, n] = bf16(f32(base[s, n]) + f32(scale_e * bf16(xa[s] . B_e[n]))),
//   each thread taking CPC = 64 / RCAP consecutive columns per pass
//   (RCAP: rank capacity of the instantiation).
// The shrink's sums meet in shared memory, so the expand needs no second
// launch and no global round trip of xa.
template <int RCAP>
__global__ void __launch_bounds__(32 * kShrinkWarps)
lora_gather_fold_kernel(const __nv_bfloat16* __restrict__ x, const uint32_t* __restrict__ indices,
                        const int32_t* __restrict__ row_adapter, const uint64_t* __restrict__ a_table,
                        const uint64_t* __restrict__ b_table, const float* __restrict__ scale_table,
                        __nv_bfloat16* __restrict__ xa, __nv_bfloat16* __restrict__ base, uint32_t n_experts,
                        int k_in, int n_out, int max_rank, uint32_t top_k, uint32_t x_gather) {
    pdl_wait();
    constexpr int CPC = 64 / RCAP;
    __shared__ float s_xa[RCAP];
    const uint32_t s = blockIdx.x;
    const int e = gather_row_expert(s, indices, row_adapter, a_table, n_experts, top_k);
    if (e < 0) return;  // block-uniform
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x < RCAP) s_xa[threadIdx.x] = 0.0f;  // ranks past max_rank stay 0
    __syncthreads();
    {
        const int chunks = k_in / 8;
        const size_t src = x_gather ? s / top_k : s;
        const uint4* xr = reinterpret_cast<const uint4*>(x + src * k_in);
        const uint4* A = reinterpret_cast<const uint4*>(a_table[e]);
        constexpr int JW = (RCAP + kShrinkWarps - 1) / kShrinkWarps;  // outputs per warp at most
        float acc[JW];
#pragma unroll
        for (int i = 0; i < JW; ++i) acc[i] = 0.0f;
        for (int c = lane; c < chunks; c += 32) {
            const uint4 xv = __ldg(xr + c);
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int i = 0; i < JW; ++i) {
                const int j = warp + i * kShrinkWarps;
                if (j < max_rank) {
                    const uint4 av = __ldg(A + static_cast<size_t>(j) * chunks + c);
                    const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 a2 = Act<MOE_ACT_BF16>::unpack2(aw[q]);
                        const float2 x2 = Act<MOE_ACT_BF16>::unpack2(xw[q]);
                        acc[i] = fmaf(x2.x, a2.x, acc[i]);
                        acc[i] = fmaf(x2.y, a2.y, acc[i]);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < JW; ++i) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], off);
            const int j = warp + i * kShrinkWarps;
            if (lane == 0 && j < max_rank) {
                const __nv_bfloat16 v = __float2bfloat16_rn(acc[i]);  // bf16 xa
                xa[static_cast<size_t>(s) * max_rank + j] = v;
                s_xa[j] = __bfloat162float(v);
            }
        }
    }
    __syncthreads();
    const __nv_bfloat16* Bbase = reinterpret_cast<const __nv_bfloat16*>(b_table[e]);
    const float sc = scale_table[e];
    for (int n0 = threadIdx.x * CPC; n0 < n_out; n0 += blockDim.x * CPC) {
        // this thread's CPC rows of B_e: CPC * max_rank consecutive values
        const __nv_bfloat16* B = Bbase + static_cast<size_t>(n0) * max_rank;
        float bw[CPC][RCAP];
        if (max_rank == RCAP) {  // 64 values = 128 aligned bytes: eight 16-byte loads
#pragma unroll
            for (int v = 0; v < CPC * RCAP / 8; ++v) {
                const uint4 q = __ldg(reinterpret_cast<const uint4*>(B) + v);
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float2 f = Act<MOE_ACT_BF16>::unpack2(w[h]);
                    const int k0 = v * 8 + 2 * h;
                    bw[k0 / RCAP][k0 % RCAP] = f.x;
                    bw[(k0 + 1) / RCAP][(k0 + 1) % RCAP] = f.y;
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < CPC; ++i)
#pragma unroll
                for (int j = 0; j < RCAP; ++j)
                    bw[i][j] = j < max_rank ? __bfloat162float(B[i * max_rank + j]) : 0.0f;
        }
        __nv_bfloat16* yrow = base + static_cast<size_t>(s) * n_out + n0;
#pragma unroll
        for (int i = 0; i < CPC; ++i) {
            float acc = 0.0f;
#pragma unroll
            for (int j = 0; j < RCAP; ++j) acc = fmaf(s_xa[j], bw[i][j], acc);
            const float d = __bfloat162float(__float2bfloat16_rn(acc));  // bf16 delta
            const float y = __bfloat162float(yrow[i]);
            yrow[i] = __float2bfloat16_rn(__fadd_rn(y, __fmul_rn(sc, d)));
        }
    }
}

}  // namespace
}  // namespace moe

extern "C" int moe_lora_grouped_down(const MoeExpertRoute* route, const void* x, void* base_out,
                                     const int32_t* expert_offsets, const int32_t* sorted_token_ids,
                                     const int32_t* row_adapter, void* xa, uint32_t row_offset, uint32_t row_end,
                                     uint32_t x_gather, int32_t num_tokens, int32_t top_k, void* stream) {
    const char* who = "moe_lora_grouped_down";
    MOE_REQUIRE(route != nullptr, "%s: NULL route", who);
    MOE_REQUIRE(route->n_experts >= 1 && route->n_experts <= MOE_MAX_EXPERTS, "%s: n_experts=%u outside [1, %d]",
                who, route->n_experts, MOE_MAX_EXPERTS);
    MOE_REQUIRE(route->max_rank >= 1 && route->max_rank <= MOE_MAX_LORA_RANK, "%s: max_rank=%u outside [1, %d]",
                who, route->max_rank, MOE_MAX_LORA_RANK);
    MOE_REQUIRE(route->k_in > 0 && route->k_in % 8 == 0, "%s: k_in=%u must be a positive multiple of 8", who,
                route->k_in);
    MOE_REQUIRE(route->n_out > 0 && route->n_out % 4 == 0, "%s: n_out=%u must be a positive multiple of 4", who,
                route->n_out);
    MOE_REQUIRE(row_offset <= row_end && row_end <= 0x7fffffffu, "%s: bad window [%u, %u)", who, row_offset,
                row_end);
    MOE_REQUIRE(x_gather <= 1, "%s: x_gather=%u must be 0 or 1", who, x_gather);
    MOE_REQUIRE(num_tokens >= 0 && top_k >= 1, "%s: bad num_tokens=%d / top_k=%d", who, num_tokens, top_k);
    if (row_end == row_offset) return MOE_OK;
    MOE_REQUIRE(route->a_table && route->b_table && route->scale_table && x && base_out && expert_offsets &&
                    sorted_token_ids && xa,
                "%s: NULL pointer", who);
    MOE_REQUIRE(moe::aligned16(x), "%s: x must be 16-byte aligned", who);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int P = num_tokens * top_k;
    const int sms = moe::sm_count();
    if (sms <= 0) return moe::fail(MOE_ERR_CUDA, "%s: cannot query the SM count", who);
    const int window = static_cast<int>(row_end - row_offset);
    const int max_tiles = (window + moe::kRowTile - 1) / moe::kRowTile + static_cast<int>(route->n_experts);
    const int grid = max_tiles < sms * 2 ? max_tiles : sms * 2;

    const size_t shrink_smem = ((sizeof(moe::LoraTiles) + 15) / 16) * 16 +
                               static_cast<size_t>(route->max_rank) * route->k_in * 2;
    MOE_REQUIRE(shrink_smem <= 200 * 1024, "%s: max_rank * k_in too large for shared memory", who);
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        int rc = moe::set_smem_limit(reinterpret_cast<const void*>(moe::lora_shrink_kernel), 200 * 1024);
        if (rc != MOE_OK) return rc;
        configured_for = dev;
    }
    moe::launch_pdl(moe::lora_shrink_kernel, grid, 32 * moe::kShrinkWarps, shrink_smem, st,
        static_cast<const __nv_bfloat16*>(x), expert_offsets, sorted_token_ids, row_adapter, route->a_table,
        static_cast<__nv_bfloat16*>(xa), route->n_experts, route->max_rank, route->k_in, x_gather, row_offset,
        row_end, P, top_k, nullptr);
    moe::count_launch();
    int rc = moe::check_launch("moe_lora_grouped_down (shrink)");
    if (rc != MOE_OK) return rc;
    const auto* xa_p = static_cast<const __nv_bfloat16*>(xa);
    auto* base_p = static_cast<__nv_bfloat16*>(base_out);
    if (route->max_rank <= 16)
        moe::launch_pdl(moe::lora_expand_fold_kernel<16>, grid, moe::kExpandThreads, 0, st,
            xa_p, expert_offsets, sorted_token_ids, row_adapter, route->b_table, route->scale_table, base_p,
            route->n_experts, route->n_out, route->max_rank, row_offset, row_end, P, top_k, route->a_table);
    else if (route->max_rank <= 32)
        moe::launch_pdl(moe::lora_expand_fold_kernel<32>, grid, moe::kExpandThreads, 0, st,
            xa_p, expert_offsets, sorted_token_ids, row_adapter, route->b_table, route->scale_table, base_p,
            route->n_experts, route->n_out, route->max_rank, row_offset, row_end, P, top_k, route->a_table);
    else
        moe::launch_pdl(moe::lora_expand_fold_kernel<64>, grid, moe::kExpandThreads, 0, st,
            xa_p, expert_offsets, sorted_token_ids, row_adapter, route->b_table, route->scale_table, base_p,
            route->n_experts, route->n_out, route->max_rank, row_offset, row_end, P, top_k, route->a_table);
    moe::count_launch();
    return moe::check_launch("moe_lora_grouped_down (expand)");
}

extern "C" int moe_lora_gather_bgmv(const MoeExpertRoute* route, const void* x, void* base_out,
                                    const uint32_t* indices, const int32_t* row_adapter, void* xa, uint32_t n_slots,
                                    uint32_t top_k, uint32_t x_gather, void* stream) {
    const char* who = "moe_lora_gather_bgmv";
    MOE_REQUIRE(route != nullptr, "%s: NULL route", who);
    MOE_REQUIRE(route->n_experts >= 1 && route->n_experts <= MOE_MAX_EXPERTS, "%s: n_experts=%u outside [1, %d]",
                who, route->n_experts, MOE_MAX_EXPERTS);
    MOE_REQUIRE(route->max_rank >= 1 && route->max_rank <= MOE_MAX_LORA_RANK, "%s: max_rank=%u outside [1, %d]",
                who, route->max_rank, MOE_MAX_LORA_RANK);
    MOE_REQUIRE(route->k_in > 0 && route->k_in % 8 == 0, "%s: k_in=%u must be a positive multiple of 8", who,
                route->k_in);
    MOE_REQUIRE(route->n_out > 0 && route->n_out % 4 == 0, "%s: n_out=%u must be a positive multiple of 4", who,
                route->n_out);
    MOE_REQUIRE(x_gather <= 1, "%s: x_gather=%u must be 0 or 1", who, x_gather);
    MOE_REQUIRE(top_k >= 1, "%s: top_k must be positive", who);
    MOE_REQUIRE(n_slots <= 0x7fffffffu, "%s: n_slots=%u too large", who, n_slots);
    if (n_slots == 0) return MOE_OK;
    MOE_REQUIRE(route->a_table && route->b_table && route->scale_table && x && base_out && indices && xa,
                "%s: NULL pointer", who);
    MOE_REQUIRE(moe::aligned16(x), "%s: x must be 16-byte aligned", who);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const auto* xp = static_cast<const __nv_bfloat16*>(x);
    auto* xa_p = static_cast<__nv_bfloat16*>(xa);
    auto* base_p = static_cast<__nv_bfloat16*>(base_out);
    const int k_in = static_cast<int>(route->k_in), n_out = static_cast<int>(route->n_out),
              rank = static_cast<int>(route->max_rank);
    const dim3 grid(n_slots), block(32 * moe::kShrinkWarps);
    if (rank <= 16)
        moe::launch_pdl(moe::lora_gather_fold_kernel<16>, grid, block, 0, st, xp, indices, row_adapter,
                        route->a_table, route->b_table, route->scale_table, xa_p, base_p, route->n_experts, k_in,
                        n_out, rank, top_k, x_gather);
    else if (rank <= 32)
        moe::launch_pdl(moe::lora_gather_fold_kernel<32>, grid, block, 0, st, xp, indices, row_adapter,
                        route->a_table, route->b_table, route->scale_table, xa_p, base_p, route->n_experts, k_in,
                        n_out, rank, top_k, x_gather);
    else
        moe::launch_pdl(moe::lora_gather_fold_kernel<64>, grid, block, 0, st, xp, indices, row_adapter,
                        route->a_table, route->b_table, route->scale_table, xa_p, base_p, route->n_experts, k_in,
                        n_out, rank, top_k, x_gather);
    moe::count_launch();
    return moe::check_launch("moe_lora_gather_bgmv");
}
