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

constexpr int kRowTile = 64;       // rows per expand tile
constexpr int kColChunk = 512;     // output columns per expand tile (each block walks one chunk)
constexpr int kShrinkTile = 64;    // rows per shrink tile: four 16-row blocks
constexpr int kShrinkWarps = 8;
constexpr int kExpandThreads = 256;

struct LoraTiles {
    int n_tiles;
    int tstart[MOE_MAX_EXPERTS + 1];
    int lo[MOE_MAX_EXPERTS];
};

// rows of expert e inside the window: [max(off[e], row_offset), min(off[e+1], row_end)).
// Every thread of the block first computes the tile counts of its experts
// (all loads issued together), then warp 0 scans them.
__device__ void build_lora_tiles(LoraTiles& s, const int32_t* offsets, int n_experts, uint32_t row_offset,
                                 uint32_t row_end, const uint64_t* a_table, int row_tile) {
    for (int e = threadIdx.x; e < n_experts; e += blockDim.x) {
        const int lo = max(offsets[e], static_cast<int>(row_offset));
        const int hi = min(offsets[e + 1], static_cast<int>(row_end));
        s.lo[e] = lo;
        s.tstart[e] = (hi > lo && a_table[e] != 0) ? (hi - lo + row_tile - 1) / row_tile : 0;  // counts for now
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        const int per = (n_experts + 31) / 32;  // <= 8
        int loc = 0;
        for (int j = 0; j < per; ++j) {
            const int e = lane * per + j;
            if (e < n_experts) loc += s.tstart[e];
        }
        int inc = loc;
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, inc, d);
            if (lane >= d) inc += o;
        }
        int run = inc - loc;
        for (int j = 0; j < per; ++j) {
            const int e = lane * per + j;
            if (e < n_experts) {
                const int c = s.tstart[e];
                s.tstart[e] = run;
                run += c;
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

// One warp-level tensor-core product D[16 x 8] += A[16 x 16] * B[16 x 8]
// (bf16 inputs, f32 accumulation): a = four bf16 pairs of A (rows g, g + 8;
// k = 2t, 2t + 1 and 2t + 8, 2t + 9), b = two pairs of B (k = 2t, 2t + 1 and
// 2t + 8, 2t + 9; column g), d = D[g][2t], D[g][2t + 1], D[g + 8][2t],
// D[g + 8][2t + 1], with g = lane / 4 and t = lane % 4.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// xa = bf16(xrow . A_e^T) for the rows of 64-row tiles: a contraction of
// k_in (768 in the workloads) into max_rank sums, run as warp-level
// tensor-core products (bf16 in, f32 accumulation). Warp task (m, n) covers
// 16 rows x 8 ranks over the whole contraction: its x fragments come straight
// from global memory (rows that fold nothing, or lie past the span, read as
// zeros), its A_e fragments from shared memory (staged by cp.async when the
// block's expert changes). Each sum is rounded once to bf16.
__global__ void __launch_bounds__(32 * kShrinkWarps, 3)
lora_shrink_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ offsets,
                   const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ row_adapter,
                   const uint64_t* __restrict__ a_table, __nv_bfloat16* __restrict__ xa, int n_experts, int max_rank,
                   int k_in, uint32_t x_gather, uint32_t row_offset, uint32_t row_end, int P, int top_k,
                   int32_t* err) {
    pdl_wait();
    extern __shared__ __align__(16) uint8_t smem[];
    LoraTiles& s = *reinterpret_cast<LoraTiles*>(smem);
    __shared__ int s_src[kShrinkTile];
    const uint32_t* sA = reinterpret_cast<const uint32_t*>(smem + ((sizeof(LoraTiles) + 15) / 16) * 16);
    build_lora_tiles(s, offsets, n_experts, row_offset, row_end, a_table, kShrinkTile);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int kw = k_in / 2;                 // bf16 pairs per row
    const int ksteps = (k_in + 15) / 16;     // a last step past k_in reads zeros
    const int nblocks = (max_rank + 7) / 8;  // 8-rank blocks
    int cur_e = -1;
    for (int tile = blockIdx.x; tile < s.n_tiles; tile += gridDim.x) {
        const int e = lora_tile_expert(s, n_experts, tile);
        const int r0 = s.lo[e] + (tile - s.tstart[e]) * kShrinkTile;
        const int hi = min(offsets[e + 1], static_cast<int>(row_end));
        __syncthreads();  // the previous tile is done with s_src and A_e
        for (int i = threadIdx.x; i < kShrinkTile; i += blockDim.x)
            s_src[i] = r0 + i < hi ? lora_row_source(r0 + i, sorted_ids, row_adapter, P, top_k, x_gather, err) : -1;
        if (e != cur_e) {  // stage A_e [max_rank, k_in] (block-uniform)
            const uint4* src = reinterpret_cast<const uint4*>(a_table[e]);
            for (int i = threadIdx.x; i < max_rank * (k_in / 8); i += blockDim.x)
                cp_async16(reinterpret_cast<uint4*>(const_cast<uint32_t*>(sA)) + i, src + i);
            cp_async_commit();
            cp_async_wait_all();
            cur_e = e;
        }
        __syncthreads();
        for (int task = warp; task < 4 * nblocks; task += kShrinkWarps) {
            const int mb = task & 3, nb = task >> 2;
            const int rl = 16 * mb + g, rh = rl + 8;  // this lane's two tile rows
            const int sl = s_src[rl], sh = s_src[rh];
            if (__all_sync(0xffffffffu, sl < 0 && sh < 0)) continue;  // no row of the block folds
            const uint32_t* xl = reinterpret_cast<const uint32_t*>(x + static_cast<size_t>(sl < 0 ? 0 : sl) * k_in);
            const uint32_t* xh = reinterpret_cast<const uint32_t*>(x + static_cast<size_t>(sh < 0 ? 0 : sh) * k_in);
            const int j = 8 * nb + g;  // this lane's rank (the MMA's n index)
            const uint32_t* ar = sA + static_cast<size_t>(j < max_rank ? j : 0) * kw;
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
            for (int ks = 0; ks < ksteps; ++ks) {
                const int p0 = 8 * ks + t, p1 = p0 + 4;  // pair indices of k = 16 ks + 2t and + 8
                uint32_t a[4], b[2];
                a[0] = (sl >= 0 && p0 < kw) ? __ldg(xl + p0) : 0u;
                a[1] = (sh >= 0 && p0 < kw) ? __ldg(xh + p0) : 0u;
                a[2] = (sl >= 0 && p1 < kw) ? __ldg(xl + p1) : 0u;
                a[3] = (sh >= 0 && p1 < kw) ? __ldg(xh + p1) : 0u;
                b[0] = (j < max_rank && p0 < kw) ? ar[p0] : 0u;
                b[1] = (j < max_rank && p1 < kw) ? ar[p1] : 0u;
                mma_bf16_16816(d, a, b);
            }
            // d: (row rl; ranks 8 nb + 2t, + 1) and (row rh; same ranks)
            const int jr = 8 * nb + 2 * t;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int rr = h ? rh : rl;
                if ((h ? sh : sl) < 0) continue;
                __nv_bfloat16* dst = xa + static_cast<size_t>(r0 + rr - row_offset) * max_rank + jr;
                if (jr < max_rank) dst[0] = __float2bfloat16_rn(d[2 * h]);
                if (jr + 1 < max_rank) dst[1] = __float2bfloat16_rn(d[2 * h + 1]);
            }
        }
    }
}

// Two fused multiply-adds on a pair of f32 values in one instruction:
// d.x = fma(a.x, b.x, c.x), d.y = fma(a.y, b.y, c.y), each rounded once.
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long f32x2_pack(float lo, float hi) {
    return (static_cast<unsigned long long>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}

// Packed storage of N consecutive bf16 values (N = 4, 2 or 1): one load or
// store moves a thread's columns of a row.
template <int N> struct BfPack;
template <> struct BfPack<4> {
    using V = uint2;
    static __device__ __forceinline__ float get(const V& v, int i) {
        const uint32_t w = (i < 2) ? v.x : v.y;
        return __uint_as_float((i & 1) ? (w & 0xffff0000u) : (w << 16));
    }
    static __device__ __forceinline__ void set(V& v, int i, __nv_bfloat16 b) {
        const uint32_t u = __bfloat16_as_ushort(b);
        uint32_t& w = (i < 2) ? v.x : v.y;
        w = (i & 1) ? ((w & 0x0000ffffu) | (u << 16)) : ((w & 0xffff0000u) | u);
    }
};
template <> struct BfPack<2> {
    using V = uint32_t;
    static __device__ __forceinline__ float get(const V& v, int i) {
        return __uint_as_float(i ? (v & 0xffff0000u) : (v << 16));
    }
    static __device__ __forceinline__ void set(V& v, int i, __nv_bfloat16 b) {
        const uint32_t u = __bfloat16_as_ushort(b);
        v = i ? ((v & 0x0000ffffu) | (u << 16)) : ((v & 0xffff0000u) | u);
    }
};
template <> struct BfPack<1> {
    using V = unsigned short;
    static __device__ __forceinline__ float get(const V& v, int) { return __uint_as_float(static_cast<uint32_t>(v) << 16); }
    static __device__ __forceinline__ void set(V& v, int, __nv_bfloat16 b) { v = __bfloat16_as_ushort(b); }
};

// RCAP: rank capacity of this instantiation (16, 32 or 64: one to four
// k16 steps). A block takes one work tile: 64 rows of an expert's span
// (inside the window) times a chunk of 512 output columns. It copies the
// tile's base values into shared memory with cp.async (64 KB in flight at
// once) while it stages the rows' xa (bf16, as stored) and which rows fold.
// The rank-RCAP product delta = xa . B_e^T is a K = RCAP contraction: warp w
// computes it for all 64 rows and columns [64 w, 64 w + 64) of the chunk
// with warp-level tensor-core products (16 rows x 8 columns each, f32
// accumulation; a tcgen05 tile of 128 rows would need TMEM and shared-memory
// descriptors for a contraction of 16, and the kernel is bound by the base
// values' read and write anyway), then rounds each sum to bf16, folds it into
// the staged base value and stores the pair of columns to global memory.
template <int RCAP>
__global__ void __launch_bounds__(kExpandThreads, RCAP <= 16 ? 3 : 2)
lora_expand_fold_kernel(const __nv_bfloat16* __restrict__ xa, const int32_t* __restrict__ offsets,
                        const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ row_adapter,
                        const uint64_t* __restrict__ b_table, const float* __restrict__ scale_table,
                        __nv_bfloat16* __restrict__ base, int n_experts, int n_out, int max_rank, uint32_t row_offset,
                        uint32_t row_end, int P, int top_k, const uint64_t* __restrict__ a_table) {
    pdl_wait();
    constexpr int KS = RCAP / 16;  // k16 steps
    extern __shared__ __align__(16) uint8_t lsm[];
    LoraTiles& s = *reinterpret_cast<LoraTiles*>(lsm);
    size_t off = (sizeof(LoraTiles) + 15) / 16 * 16;
    int* s_src = reinterpret_cast<int*>(lsm + off);
    off += kRowTile * sizeof(int);
    uint32_t* s_xa = reinterpret_cast<uint32_t*>(lsm + off);  // [kRowTile][RCAP / 2] bf16 pairs
    off += static_cast<size_t>(kRowTile) * RCAP * 2;
    uint32_t* s_y = reinterpret_cast<uint32_t*>(lsm + off);   // [kRowTile][kColChunk / 2] bf16 pairs
    build_lora_tiles(s, offsets, n_experts, row_offset, row_end, a_table, kRowTile);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int n_chunks = (n_out + kColChunk - 1) / kColChunk;
    for (int wt = blockIdx.x; wt < s.n_tiles * n_chunks; wt += gridDim.x) {
        const int tile = wt / n_chunks, chunk = wt - tile * n_chunks;
        const int e = lora_tile_expert(s, n_experts, tile);
        const int r0 = s.lo[e] + (tile - s.tstart[e]) * kRowTile;
        const int hi = min(offsets[e + 1], static_cast<int>(row_end));
        const int nrows = min(kRowTile, hi - r0);
        const int c0 = chunk * kColChunk;
        const int ncols = min(kColChunk, n_out - c0);  // a multiple of 4
        __syncthreads();  // the previous tile is done with the shared buffers
        // 1. the tile's base values: 8-byte copies, every one in flight at once
        {
            const int per_row = ncols / 4;
            for (int i = threadIdx.x; i < nrows * per_row; i += blockDim.x) {
                const int rr = i / per_row, q = i - rr * per_row;
                asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(s_y + rr * (kColChunk / 2) + 2 * q)),
                             "l"(base + static_cast<size_t>(r0 + rr) * n_out + c0 + 4 * q)
                             : "memory");
            }
            cp_async_commit();
        }
        // 2. meanwhile: which rows fold and their xa (zero for rows that do not fold,
        // for rows past the tile and for ranks past max_rank)
        for (int i = threadIdx.x; i < kRowTile; i += blockDim.x)
            s_src[i] = i < nrows ? lora_row_source(r0 + i, sorted_ids, row_adapter, P, top_k, 0, nullptr) : -1;
        __syncthreads();
        for (int i = threadIdx.x; i < kRowTile * (RCAP / 2); i += blockDim.x) {
            const int rr = i / (RCAP / 2), jp = i - rr * (RCAP / 2);
            uint32_t v = 0u;
            if (s_src[rr] >= 0) {
                const __nv_bfloat16* src = xa + static_cast<size_t>(r0 + rr - row_offset) * max_rank;
                const uint32_t lo = 2 * jp < max_rank ? __bfloat16_as_ushort(src[2 * jp]) : 0u;
                const uint32_t hi2 = 2 * jp + 1 < max_rank ? __bfloat16_as_ushort(src[2 * jp + 1]) : 0u;
                v = lo | (hi2 << 16);
            }
            s_xa[rr * (RCAP / 2) + jp] = v;
        }
        const float sc = scale_table[e];
        const __nv_bfloat16* B = reinterpret_cast<const __nv_bfloat16*>(b_table[e]);
        cp_async_wait_all();
        __syncthreads();
        // 3. xa fragments of the four 16-row blocks, held for the whole chunk
        uint32_t af[4][KS][4];
#pragma unroll
        for (int mb = 0; mb < 4; ++mb)
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const uint32_t* r_lo = s_xa + (16 * mb + g) * (RCAP / 2) + 8 * ks + t;
                const uint32_t* r_hi = r_lo + 8 * (RCAP / 2);
                af[mb][ks][0] = r_lo[0];
                af[mb][ks][1] = r_hi[0];
                af[mb][ks][2] = r_lo[4];
                af[mb][ks][3] = r_hi[4];
            }
        // 4. this warp's columns [64 w, 64 w + 64) of the chunk, 8 at a time; the B_e
        // fragments of all eight blocks are loaded first (one round trip to L2)
        uint32_t bfa[8][KS][2];
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
            const int n = c0 + 64 * warp + 8 * nb + g;  // this lane's column of B (the MMA's n index)
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                // pairs (k = 16 ks + 2t, +1) and (+8, +9) of B_e row n; zero past the chunk or max_rank
                uint32_t b0 = 0u, b1 = 0u;
                if (64 * warp + 8 * nb + g < ncols) {
                    const __nv_bfloat16* brow = B + static_cast<size_t>(n) * max_rank;
                    const int k0 = 16 * ks + 2 * t, k1 = k0 + 8;
                    b0 = (k0 < max_rank ? __bfloat16_as_ushort(brow[k0]) : 0u) |
                         ((k0 + 1 < max_rank ? static_cast<uint32_t>(__bfloat16_as_ushort(brow[k0 + 1])) : 0u) << 16);
                    b1 = (k1 < max_rank ? __bfloat16_as_ushort(brow[k1]) : 0u) |
                         ((k1 + 1 < max_rank ? static_cast<uint32_t>(__bfloat16_as_ushort(brow[k1 + 1])) : 0u) << 16);
                }
                bfa[nb][ks][0] = b0;
                bfa[nb][ks][1] = b1;
            }
        }
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
            const int cl0 = 64 * warp + 8 * nb;  // first chunk column of the block
            if (cl0 >= ncols) break;             // warp-uniform
            const uint32_t (&bf)[KS][2] = bfa[nb];
#pragma unroll
            for (int mb = 0; mb < 4; ++mb) {
                float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) mma_bf16_16816(d, af[mb][ks], bf[ks]);
                // d: rows 16 mb + g (d0, d1) and 16 mb + g + 8 (d2, d3), columns cl0 + 2t, + 1
                const int cl = cl0 + 2 * t;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int rr = 16 * mb + g + 8 * h;
                    if (rr >= nrows || s_src[rr] < 0 || cl >= ncols) continue;
                    const uint32_t yv = s_y[rr * (kColChunk / 2) + cl / 2];
                    const float d0 = __bfloat162float(__float2bfloat16_rn(d[2 * h]));      // bf16 delta
                    const float d1 = __bfloat162float(__float2bfloat16_rn(d[2 * h + 1]));
                    const float y0 = __uint_as_float(yv << 16), y1 = __uint_as_float(yv & 0xffff0000u);
                    const uint32_t o0 = __bfloat16_as_ushort(__float2bfloat16_rn(__fadd_rn(y0, __fmul_rn(sc, d0))));
                    const uint32_t o1 = __bfloat16_as_ushort(__float2bfloat16_rn(__fadd_rn(y1, __fmul_rn(sc, d1))));
                    *reinterpret_cast<uint32_t*>(base + static_cast<size_t>(r0 + rr) * n_out + c0 + cl) =
                        o0 | (o1 << 16);
                }
            }
        }
    }
}

// dynamic shared memory of an expand instantiation
template <int RCAP>
size_t lora_expand_smem() {
    return (sizeof(LoraTiles) + 15) / 16 * 16 + kRowTile * sizeof(int) + static_cast<size_t>(kRowTile) * RCAP * 2 +
           static_cast<size_t>(kRowTile) * kColChunk * 2;
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
    MOE_REQUIRE((reinterpret_cast<uintptr_t>(base_out) & 7) == 0, "%s: base_out must be 8-byte aligned", who);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int P = num_tokens * top_k;
    const int sms = moe::sm_count();
    if (sms <= 0) return moe::fail(MOE_ERR_CUDA, "%s: cannot query the SM count", who);
    const int window = static_cast<int>(row_end - row_offset);
    const int n_chunks = (static_cast<int>(route->n_out) + moe::kColChunk - 1) / moe::kColChunk;
    const long max_tiles = static_cast<long>((window + moe::kRowTile - 1) / moe::kRowTile + route->n_experts) * n_chunks;
    const int grid = static_cast<int>(max_tiles < sms * 4 ? max_tiles : sms * 4);
    const int s_tiles = (window + moe::kShrinkTile - 1) / moe::kShrinkTile + static_cast<int>(route->n_experts);
    const int s_grid = s_tiles < sms * 4 ? s_tiles : sms * 4;

    const size_t shrink_smem = ((sizeof(moe::LoraTiles) + 15) / 16) * 16 +
                               static_cast<size_t>(route->max_rank) * route->k_in * 2;
    MOE_REQUIRE(shrink_smem <= 200 * 1024, "%s: max_rank * k_in too large for shared memory", who);
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        int rc = moe::set_smem_limit(reinterpret_cast<const void*>(moe::lora_shrink_kernel), 200 * 1024);
        if (rc == MOE_OK)
            rc = moe::set_smem_limit(reinterpret_cast<const void*>(moe::lora_expand_fold_kernel<16>),
                                     static_cast<int>(moe::lora_expand_smem<16>()));
        if (rc == MOE_OK)
            rc = moe::set_smem_limit(reinterpret_cast<const void*>(moe::lora_expand_fold_kernel<32>),
                                     static_cast<int>(moe::lora_expand_smem<32>()));
        if (rc == MOE_OK)
            rc = moe::set_smem_limit(reinterpret_cast<const void*>(moe::lora_expand_fold_kernel<64>),
                                     static_cast<int>(moe::lora_expand_smem<64>()));
        if (rc != MOE_OK) return rc;
        configured_for = dev;
    }
    moe::launch_pdl(moe::lora_shrink_kernel, s_grid, 32 * moe::kShrinkWarps, shrink_smem, st,
        static_cast<const __nv_bfloat16*>(x), expert_offsets, sorted_token_ids, row_adapter, route->a_table,
        static_cast<__nv_bfloat16*>(xa), route->n_experts, route->max_rank, route->k_in, x_gather, row_offset,
        row_end, P, top_k, nullptr);
    moe::count_launch();
    int rc = moe::check_launch("moe_lora_grouped_down (shrink)");
    if (rc != MOE_OK) return rc;
    const auto* xa_p = static_cast<const __nv_bfloat16*>(xa);
    auto* base_p = static_cast<__nv_bfloat16*>(base_out);
    if (route->max_rank <= 16)
        moe::launch_pdl(moe::lora_expand_fold_kernel<16>, grid, moe::kExpandThreads, moe::lora_expand_smem<16>(), st,
            xa_p, expert_offsets, sorted_token_ids, row_adapter, route->b_table, route->scale_table, base_p,
            route->n_experts, route->n_out, route->max_rank, row_offset, row_end, P, top_k, route->a_table);
    else if (route->max_rank <= 32)
        moe::launch_pdl(moe::lora_expand_fold_kernel<32>, grid, moe::kExpandThreads, moe::lora_expand_smem<32>(), st,
            xa_p, expert_offsets, sorted_token_ids, row_adapter, route->b_table, route->scale_table, base_p,
            route->n_experts, route->n_out, route->max_rank, row_offset, row_end, P, top_k, route->a_table);
    else
        moe::launch_pdl(moe::lora_expand_fold_kernel<64>, grid, moe::kExpandThreads, moe::lora_expand_smem<64>(), st,
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
