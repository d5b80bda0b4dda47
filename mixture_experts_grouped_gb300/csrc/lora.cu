// Step a5: the device-side grouped LoRA fold on sorted expert rows.
//
// Restates spark_model/layers/ops/moe_lora_grouped.rs, moe_lora_grouped_down
// and MoeExpertRoute: a shrink (xa = bf16(x . A_e^T)) and an expand + fold
// (base += scale_e * fp32(bf16(xa . B_e^T))) over one window [row_offset,
// row_end) of the sorted rows, with expert spans read from expert_offsets on
// the device. The page sizes a static worst-case grid (ceil(window/64) x
// n_experts) whose tiles mostly return at once; here a persistent grid walks
// only the non-empty row tiles of span intersect window, listed in shared
// memory from expert_offsets at kernel start.
//
// The work is HBM-bound (rank 16: 2 x rank FLOPs per element of base read and
// written), so both kernels keep many copies in flight through cp.async rings
// in shared memory and run their small contractions on warp-level tensor-core
// products:
//   shrink: 64-row tiles, the contraction streamed in 128-column stages (x rows
//           and A_e rows side by side), ldmatrix fragments;
//   expand: contiguous ranges of (32-row tile, 256-column) units per block,
//           three units in flight, folded in shared memory and written back
//           with full-width stores.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kShrinkRows = 64;               // rows per shrink tile: four 16-row blocks
constexpr int kShrinkK = 128;                 // contraction columns per shrink stage
constexpr int kShrinkPitch = kShrinkK + 8;    // bf16 per staged row: 272 bytes, rows 4 banks apart
constexpr int kShrinkStages = 4;
constexpr int kShrinkWarps = 8;
constexpr int kExRows = 32;                   // rows per expand tile
constexpr int kExCols = 256;                  // output columns per expand unit
constexpr int kExStages = 4;
constexpr int kExThreads = 256;

struct LoraTiles {
    int n_tiles;
    int tstart[MOE_MAX_EXPERTS + 1];
    int lo[MOE_MAX_EXPERTS];
    int hi[MOE_MAX_EXPERTS];
    uint64_t ptr[MOE_MAX_EXPERTS];  // the expert's A_e (shrink) or B_e (expand)
    float scale[MOE_MAX_EXPERTS];   // scale_e (expand)
};
constexpr int kTilesBytes = (sizeof(LoraTiles) + 15) / 16 * 16;

// rows of expert e inside the window: [max(off[e], row_offset), min(off[e+1], row_end)).
// Every thread of the block first computes the tile counts of its experts
// (all loads issued together) and caches their table pointer and scale (so
// the tile loops read no table from global memory), then warp 0 scans the
// counts.
__device__ void build_lora_tiles(LoraTiles& s, const int32_t* offsets, int n_experts, uint32_t row_offset,
                                 uint32_t row_end, const uint64_t* a_table, int row_tile,
                                 const uint64_t* ptr_table, const float* scale_table) {
    for (int e = threadIdx.x; e < n_experts; e += blockDim.x) {
        const int lo = max(offsets[e], static_cast<int>(row_offset));
        const int hi = min(offsets[e + 1], static_cast<int>(row_end));
        s.lo[e] = lo;
        s.hi[e] = hi;
        s.ptr[e] = ptr_table[e];
        s.scale[e] = scale_table ? scale_table[e] : 0.0f;
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

// the x row of sorted row r holding pair p, or -1 when the row folds nothing
__device__ __forceinline__ int lora_source_of_pair(int r, int p, const int32_t* row_adapter, int P, int top_k,
                                                   uint32_t x_gather, int32_t* err) {
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
// tensor-core products (bf16 in, f32 accumulation, ldmatrix fragments).
// The contraction streams through a ring of kShrinkStages shared-memory
// stages of 128 columns each, filled by cp.async: a stage holds the tile's 64
// x rows and the expert's 8 * ceil(max_rank / 8) A_e rows for those columns
// (rows that fold nothing, rows past the span and columns past k_in arrive as
// zeros). Every thread copies pieces of one x row, so a block keeps three
// stages (about 65 KB at rank 16) in flight while its warps multiply the
// fourth: the work is a read of x at HBM speed, not a chain of dependent
// loads. The ring runs across the block's tiles, so the next tile's first
// stages load while the current one finishes. Warp task (m, n) covers 16 rows
// x 8 ranks; each sum is rounded once to bf16 when the tile's last stage is
// done.
__global__ void __launch_bounds__(32 * kShrinkWarps, 2)
lora_shrink_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ offsets,
                   const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ row_adapter,
                   const uint64_t* __restrict__ a_table, __nv_bfloat16* __restrict__ xa, int n_experts, int max_rank,
                   int k_in, uint32_t x_gather, uint32_t row_offset, uint32_t row_end, int P, int top_k,
                   int32_t* err) {
    pdl_wait();
    extern __shared__ __align__(16) uint8_t smem[];
    LoraTiles& s = *reinterpret_cast<LoraTiles*>(smem);
    uint8_t* s_ok = smem + kTilesBytes;  // [stage][row]: the row folds
    __nv_bfloat16* stg = reinterpret_cast<__nv_bfloat16*>(smem + kTilesBytes + kShrinkStages * kShrinkRows);
    const int nb = (max_rank + 7) / 8;                            // 8-rank blocks
    const int stage_elems = (kShrinkRows + 8 * nb) * kShrinkPitch;  // x rows, then A_e rows
    build_lora_tiles(s, offsets, n_experts, row_offset, row_end, a_table, kShrinkRows, a_table, nullptr);
    const int kch = (k_in + kShrinkK - 1) / kShrinkK;  // stages per tile
    const int my_tiles = s.n_tiles > static_cast<int>(blockIdx.x)
                             ? (s.n_tiles - static_cast<int>(blockIdx.x) + gridDim.x - 1) / gridDim.x
                             : 0;
    const int items = my_tiles * kch;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int xr = tid >> 2;  // the x row this thread copies (four threads per row)
    int src = -1, src_tl = -1;
    const __nv_bfloat16* zero_src = x;  // a valid address for the zero-filling copies
    // pair id at this thread's row of a local tile (-1 past the span): loaded one
    // tile ahead, so that starting a tile waits on no global load
    auto row_pair = [&](int tl) -> int {
        const int tile = static_cast<int>(blockIdx.x) + tl * static_cast<int>(gridDim.x);
        if (tile >= s.n_tiles) return -1;
        const int e = lora_tile_expert(s, n_experts, tile);
        const int r = s.lo[e] + (tile - s.tstart[e]) * kShrinkRows + xr;
        return r < s.hi[e] ? sorted_ids[r] : -1;
    };
    int p_pre = items > 0 ? row_pair(0) : -1;

    auto issue = [&](int item) {
        const int tl = item / kch, kc = item - tl * kch;
        const int tile = static_cast<int>(blockIdx.x) + tl * static_cast<int>(gridDim.x);
        const int e = lora_tile_expert(s, n_experts, tile);
        const int r0 = s.lo[e] + (tile - s.tstart[e]) * kShrinkRows;
        if (tl != src_tl) {
            src_tl = tl;
            src = r0 + xr < s.hi[e] ? lora_source_of_pair(r0 + xr, p_pre, row_adapter, P, top_k, x_gather, err) : -1;
            if (tl + 1 < my_tiles) p_pre = row_pair(tl + 1);
        }
        const int stage = item % kShrinkStages;
        __nv_bfloat16* sb = stg + stage * stage_elems;
        const int k0 = kc * kShrinkK;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int p = (tid & 3) + 4 * q, k = k0 + 8 * p;
            const bool full = src >= 0 && k < k_in;
            cp_async16_zfill(sb + xr * kShrinkPitch + 8 * p,
                             full ? x + static_cast<size_t>(src) * k_in + k : zero_src, full);
        }
        const __nv_bfloat16* A = reinterpret_cast<const __nv_bfloat16*>(s.ptr[e]);
        for (int i = tid; i < 8 * nb * (kShrinkK / 8); i += blockDim.x) {
            const int j = i / (kShrinkK / 8), p = i - j * (kShrinkK / 8), k = k0 + 8 * p;
            const bool full = j < max_rank && k < k_in;
            cp_async16_zfill(sb + (kShrinkRows + j) * kShrinkPitch + 8 * p,
                             full ? A + static_cast<size_t>(j) * k_in + k : zero_src, full);
        }
        if ((tid & 3) == 0) s_ok[stage * kShrinkRows + xr] = src >= 0;
    };

    float acc[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.0f;
    const int ntasks = 4 * nb;  // (16-row block, 8-rank block) pairs, at most 32: four per warp
    // ldmatrix row addresses of this lane inside a stage (bytes): x rows for
    // the four 8x8 pieces of a 16x16 A fragment, A_e rows for the two of B
    const uint32_t a_lane = ((lane & 7) + 8 * ((lane >> 3) & 1)) * kShrinkPitch * 2 + 16 * (lane >> 4);
    const uint32_t b_lane = (kShrinkRows + (lane & 7)) * kShrinkPitch * 2 + 16 * ((lane >> 3) & 1);

    for (int i = 0; i < kShrinkStages - 1; ++i) {
        if (i < items) issue(i);
        cp_async_commit();
    }
    for (int it = 0; it < items; ++it) {
        cp_async_wait_group<kShrinkStages - 2>();  // this thread's copies of item `it` landed
        __syncthreads();                          // everyone's; and item it - 1 is consumed
        if (it + kShrinkStages - 1 < items) issue(it + kShrinkStages - 1);
        cp_async_commit();
        const int tl = it / kch, kc = it - tl * kch, stage = it % kShrinkStages;
        const uint32_t sbase = smem_u32(stg + stage * stage_elems);
        const int ksteps = (min(kShrinkK, k_in - kc * kShrinkK) + 15) / 16;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int task = warp + kShrinkWarps * q;
            if (task >= ntasks) break;  // warp-uniform
            const int mb = task & 3, nbk = task >> 2;
            const uint32_t aa = sbase + a_lane + 16 * mb * kShrinkPitch * 2;
            const uint32_t ba = sbase + b_lane + 8 * nbk * kShrinkPitch * 2;
            for (int ks = 0; ks < ksteps; ++ks) {
                uint32_t a[4], b[2];
                ldmatrix_x4(a, aa + 32 * ks);
                ldmatrix_x2(b, ba + 32 * ks);
                mma_bf16_16816(acc[q], a, b);
            }
        }
        if (kc == kch - 1) {  // the tile's contraction is complete: round and store
            const int tile = static_cast<int>(blockIdx.x) + tl * static_cast<int>(gridDim.x);
            const int e = lora_tile_expert(s, n_experts, tile);
            const int r0 = s.lo[e] + (tile - s.tstart[e]) * kShrinkRows;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int task = warp + kShrinkWarps * q;
                if (task >= ntasks) break;
                const int mb = task & 3, nbk = task >> 2;
                const int jr = 8 * nbk + 2 * t;  // d: rows 16 mb + g (d0, d1), + 8 (d2, d3); ranks jr, jr + 1
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = 16 * mb + g + 8 * h;
                    if (!s_ok[stage * kShrinkRows + row]) continue;
                    __nv_bfloat16* dst = xa + static_cast<size_t>(r0 + row - static_cast<int>(row_offset)) * max_rank + jr;
                    if (jr < max_rank) dst[0] = __float2bfloat16_rn(acc[q][2 * h]);
                    if (jr + 1 < max_rank) dst[1] = __float2bfloat16_rn(acc[q][2 * h + 1]);
                }
                acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.0f;
            }
        }
    }
}

// dynamic shared memory of the shrink for a rank
inline size_t lora_shrink_smem(int max_rank) {
    const int nb = (max_rank + 7) / 8;
    return kTilesBytes + kShrinkStages * kShrinkRows +
           static_cast<size_t>(kShrinkStages) * (kShrinkRows + 8 * nb) * kShrinkPitch * 2;
}

// Two f32 operations on a pair of f32 values in one instruction, each
// rounded to nearest on its own: (a.x op b.x, a.y op b.y).
__device__ __forceinline__ unsigned long long f32x2_mul(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f32x2_add(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// a bf16 pair (low half first) as an f32 pair, exactly
__device__ __forceinline__ unsigned long long bf16x2_to_f32x2(uint32_t v) {
    return (static_cast<unsigned long long>(v & 0xffff0000u) << 32) | static_cast<unsigned long long>(v << 16);
}
// an f32 pair rounded to a bf16 pair (round to nearest even, low half first)
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&b);
}

// Position of one work unit of the expand in the block's range: chunk c,
// tile (of the window's tile list) and its expert e. Units run tile first
// within a chunk, so stepping to the next unit moves the expert forward by
// at most a few entries of the tile list instead of searching it.
struct ExCursor {
    int c, tile, e;
};

// RCAP: rank capacity of this instantiation (16, 32 or 64: one to four k16
// steps). The block takes a contiguous range of work units (a 32-row tile of
// an expert's span inside the window x 256 output columns; units ordered
// column chunk first, so consecutive units mostly share the expert and its
// B_e columns) and streams them through a ring of kExStages shared-memory
// stages filled by cp.async, three units ahead of the one it folds:
//   issue   the unit's base rows that fold (16-byte pieces, or 8-byte ones
//           when n_out % 8 != 0), the tile's xa rows, and the B_e columns of
//           the unit when they differ from the previous unit's (a ring of
//           kExStages B buffers, one per change, so that a buffer is refilled
//           only after every unit that reads it is done);
//   compute the rank-RCAP product delta = xa . B_e^T with warp-level
//           tensor-core products (warp w: columns [32 w, 32 w + 32), both
//           16-row blocks), round each sum to bf16 and fold it into the
//           staged base value (f32 multiply, f32 add, bf16; two columns per
//           instruction) in place;
//   store   the folded rows back with full-width 16-byte stores.
// No step waits on a global load of its own: the expert's B_e address and
// scale come from the tile list in shared memory, and the pair ids that
// decide which rows fold are loaded one unit ahead. The fold runs straight
// through all eight 16 x 8 blocks of the warp (rows past the tile and
// columns past n_out compute stale values that are never stored), so that
// their shared-memory round trips overlap. The stage rows are 512 bytes with
// their 16-byte pieces XOR-swizzled by the row, so that the fragment-ordered
// reads of the compute step hit 32 banks.
template <int RCAP>
__global__ void __launch_bounds__(kExThreads, RCAP <= 16 ? 2 : 1)
lora_expand_fold_kernel(const __nv_bfloat16* __restrict__ xa, const int32_t* __restrict__ offsets,
                        const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ row_adapter,
                        const uint64_t* __restrict__ b_table, const float* __restrict__ scale_table,
                        __nv_bfloat16* __restrict__ base, int n_experts, int n_out, int max_rank, uint32_t row_offset,
                        uint32_t row_end, int P, int top_k, const uint64_t* __restrict__ a_table, uint32_t vec16) {
    pdl_wait();
    constexpr int KS = RCAP / 16;                   // k16 steps
    constexpr int kRowBytes = kExCols * 2;          // 512: one staged row
    constexpr int kStageBytes = kExRows * kRowBytes;
    constexpr int kBElems = kExCols * RCAP;         // one B buffer
    constexpr int kXaElems = kExRows * RCAP;        // one stage's xa rows
    extern __shared__ __align__(16) uint8_t lsm[];
    LoraTiles& s = *reinterpret_cast<LoraTiles*>(lsm);
    int* s_bbuf = reinterpret_cast<int*>(lsm + kTilesBytes);  // B buffer of each stage
    uint8_t* sy = lsm + kTilesBytes + 16;
    __nv_bfloat16* sbuf = reinterpret_cast<__nv_bfloat16*>(sy + kExStages * kStageBytes);
    __nv_bfloat16* sxa = sbuf + kExStages * kBElems;  // [stage][row][max_rank]
    build_lora_tiles(s, offsets, n_experts, row_offset, row_end, a_table, kExRows, b_table, scale_table);
    const int n_chunks = (n_out + kExCols - 1) / kExCols;
    const int n_tiles = s.n_tiles;
    const long long U = static_cast<long long>(n_tiles) * n_chunks;
    const int u0 = static_cast<int>(U * blockIdx.x / gridDim.x);
    const int n_my = static_cast<int>(U * (blockIdx.x + 1) / gridDim.x) - u0;
    if (n_my <= 0) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int rr = tid >> 3, l8 = tid & 7;  // copy role: row rr, pieces l8 + 8 q
    const bool even_rank = (max_rank & 1) == 0;  // rank pairs start on 4-byte boundaries
    const bool xa_pairs = even_rank && (reinterpret_cast<uintptr_t>(xa) & 3u) == 0;

    auto advance = [&](ExCursor& q) {
        if (++q.tile == n_tiles) {
            q.tile = 0;
            ++q.c;
            q.e = 0;
        }
        while (s.tstart[q.e + 1] <= q.tile) ++q.e;  // tstart[n_experts] = n_tiles ends it
    };
    ExCursor cur_issue, cur_next, cur_fold;  // units j + kExStages - 1, the one after it, and j
    cur_issue.c = u0 / n_tiles;
    cur_issue.tile = u0 - cur_issue.c * n_tiles;
    cur_issue.e = lora_tile_expert(s, n_experts, cur_issue.tile);
    cur_fold = cur_issue;
    cur_next = cur_issue;
    struct Unit { int e, r0, nrows, c0, ncols; };
    auto unit = [&](const ExCursor& q) {
        Unit d;
        d.e = q.e;
        d.r0 = s.lo[q.e] + (q.tile - s.tstart[q.e]) * kExRows;
        d.nrows = min(kExRows, s.hi[q.e] - d.r0);
        d.c0 = q.c * kExCols;
        d.ncols = min(kExCols, n_out - d.c0);  // a multiple of 4
        return d;
    };
    // byte offset of 16-byte piece ch of staged row r
    auto piece = [](int r, int ch) { return r * kRowBytes + ((ch ^ (r & 7)) << 4); };
    // pair id at this thread's row of a unit, -1 past the tile
    auto row_pair = [&](const ExCursor& q) -> int {
        const Unit d = unit(q);
        return rr < d.nrows ? sorted_ids[d.r0 + rr] : -1;
    };

    uint32_t okbits = 0;   // bit st: this thread's row of the unit in stage st folds
    int bkey = -1, bver = -1;
    int p_pre = row_pair(cur_next);
    advance(cur_next);
    auto issue = [&](int j) {  // unit j = cur_issue
        const Unit d = unit(cur_issue);
        const int stage = j % kExStages;
        const int key = d.e * n_chunks + cur_issue.c;
        if (key != bkey) {  // the unit's B_e columns [c0, c0 + ncols) x max_rank: one contiguous span
            bkey = key;
            ++bver;
            const uint8_t* src = reinterpret_cast<const uint8_t*>(s.ptr[d.e]) + static_cast<size_t>(d.c0) * max_rank * 2;
            uint8_t* dst = reinterpret_cast<uint8_t*>(sbuf + (bver % kExStages) * kBElems);
            const int bytes = d.ncols * max_rank * 2;  // a multiple of 8
            for (int i = tid; i < (bytes >> 4); i += blockDim.x) cp_async16(dst + 16 * i, src + 16 * i);
            if ((bytes & 15) && tid == 0) cp_async8(dst + (bytes & ~15), src + (bytes & ~15));
        }
        if (tid == 0) s_bbuf[stage] = bver % kExStages;
        {  // the tile's xa rows, as stored: nrows * max_rank contiguous values
            __nv_bfloat16* dst = sxa + stage * kXaElems;
            const __nv_bfloat16* src = xa + static_cast<size_t>(d.r0 - static_cast<int>(row_offset)) * max_rank;
            const int n = d.nrows * max_rank;
            if (xa_pairs) {
                for (int i = tid; i < n / 2; i += blockDim.x) cp_async4(dst + 2 * i, src + 2 * i);
            } else {
                for (int i = tid; i < n; i += blockDim.x) dst[i] = src[i];
            }
        }
        const int p = p_pre;
        const bool ok = p >= 0 && p < P && (row_adapter == nullptr || row_adapter[p / top_k] >= 0);
        okbits = ok ? (okbits | (1u << stage)) : (okbits & ~(1u << stage));
        if (j + 1 < n_my) {  // the next unit's pair id, used one issue later
            p_pre = row_pair(cur_next);
            advance(cur_next);
        }
        advance(cur_issue);
        if (!ok) return;
        const __nv_bfloat16* grow = base + static_cast<size_t>(d.r0 + rr) * n_out + d.c0;
        uint8_t* srow = sy + stage * kStageBytes;
        if (vec16) {
#pragma unroll
            for (int q = 0; q < kExCols / 64; ++q) {
                const int ch = l8 + 8 * q;
                if (8 * ch < d.ncols) cp_async16(srow + piece(rr, ch), grow + 8 * ch);
            }
        } else {
#pragma unroll
            for (int q = 0; q < kExCols / 32; ++q) {
                const int pc = l8 + 8 * q;  // 8-byte piece
                if (4 * pc < d.ncols) cp_async8(srow + piece(rr, pc >> 1) + 8 * (pc & 1), grow + 4 * pc);
            }
        }
    };
    // the bf16 pair (k, k + 1) at element offset i of a shared array; zero past max_rank
    auto pair_at = [&](const __nv_bfloat16* a, int i, int k) -> uint32_t {
        if (k >= max_rank) return 0u;
        if (even_rank) return *reinterpret_cast<const uint32_t*>(a + i);
        const uint32_t lo = __bfloat16_as_ushort(a[i]);
        const uint32_t hi = k + 1 < max_rank ? static_cast<uint32_t>(__bfloat16_as_ushort(a[i + 1])) : 0u;
        return lo | (hi << 16);
    };

    for (int i = 0; i < kExStages - 1; ++i) {
        if (i < n_my) issue(i);
        cp_async_commit();
    }
    for (int j = 0; j < n_my; ++j) {
        const int stage = j % kExStages;
        cp_async_wait_group<kExStages - 2>();
        __syncthreads();  // unit j has landed; unit j - 1 is stored
        if (j + kExStages - 1 < n_my) issue(j + kExStages - 1);
        cp_async_commit();
        const Unit d = unit(cur_fold);
        advance(cur_fold);
        const int cw = 32 * warp;  // this warp's first column of the unit
        if (cw < d.ncols) {
            const float sc = s.scale[d.e];
            const unsigned long long sc2 =
                (static_cast<unsigned long long>(__float_as_uint(sc)) << 32) | __float_as_uint(sc);
            const __nv_bfloat16* bb = sbuf + s_bbuf[stage] * kBElems;
            const __nv_bfloat16* xs = sxa + stage * kXaElems;
            // xa fragments of both 16-row blocks (rows past the tile hold stale values
            // that only reach rows that are not stored)
            uint32_t af[2][KS][4];
#pragma unroll
            for (int mb = 0; mb < 2; ++mb)
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const int rl = 16 * mb + g, k0 = 16 * ks + 2 * t;
                    af[mb][ks][0] = pair_at(xs, rl * max_rank + k0, k0);
                    af[mb][ks][1] = pair_at(xs, (rl + 8) * max_rank + k0, k0);
                    af[mb][ks][2] = pair_at(xs, rl * max_rank + k0 + 8, k0 + 8);
                    af[mb][ks][3] = pair_at(xs, (rl + 8) * max_rank + k0 + 8, k0 + 8);
                }
            // B fragments of this warp's four 8-column blocks (columns past n_out read
            // stale buffer values that only reach columns that are not stored)
            uint32_t bfr[4][KS][2];
#pragma unroll
            for (int nbk = 0; nbk < 4; ++nbk) {
                const int n = cw + 8 * nbk + g;  // this lane's column of B (the MMA's n index)
#pragma unroll
                for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int k = 16 * ks + 2 * t + 8 * h;
                        bfr[nbk][ks][h] = pair_at(bb, n * max_rank + k, k);
                    }
            }
            uint8_t* srow = sy + stage * kStageBytes;
#pragma unroll
            for (int mb = 0; mb < 2; ++mb)
#pragma unroll
                for (int nbk = 0; nbk < 4; ++nbk) {
                    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) mma_bf16_16816(acc, af[mb][ks], bfr[nbk][ks]);
                    // acc: rows 16 mb + g (acc0, acc1) and + 8 (acc2, acc3); columns cw + 8 nbk + 2t, + 1
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int row = 16 * mb + g + 8 * h;
                        uint32_t* yp = reinterpret_cast<uint32_t*>(srow + piece(row, (cw >> 3) + nbk) + 4 * t);
                        const unsigned long long dl = bf16x2_to_f32x2(f32x2_to_bf16x2(acc[2 * h], acc[2 * h + 1]));
                        const unsigned long long o = f32x2_add(bf16x2_to_f32x2(*yp), f32x2_mul(sc2, dl));
                        *yp = f32x2_to_bf16x2(__uint_as_float(static_cast<uint32_t>(o)),
                                              __uint_as_float(static_cast<uint32_t>(o >> 32)));
                    }
                }
        }
        __syncthreads();  // the unit is folded in shared memory
        if ((okbits >> stage) & 1u) {
            __nv_bfloat16* grow = base + static_cast<size_t>(d.r0 + rr) * n_out + d.c0;
            const uint8_t* srow = sy + stage * kStageBytes;
            if (vec16) {
#pragma unroll
                for (int q = 0; q < kExCols / 64; ++q) {
                    const int ch = l8 + 8 * q;
                    if (8 * ch < d.ncols)
                        *reinterpret_cast<uint4*>(grow + 8 * ch) = *reinterpret_cast<const uint4*>(srow + piece(rr, ch));
                }
            } else {
#pragma unroll
                for (int q = 0; q < kExCols / 32; ++q) {
                    const int pc = l8 + 8 * q;
                    if (4 * pc < d.ncols)
                        *reinterpret_cast<uint2*>(grow + 4 * pc) =
                            *reinterpret_cast<const uint2*>(srow + piece(rr, pc >> 1) + 8 * (pc & 1));
                }
            }
        }
    }
}

// dynamic shared memory of an expand instantiation
template <int RCAP>
constexpr size_t lora_expand_smem() {
    return kTilesBytes + 16 + static_cast<size_t>(kExStages) * kExRows * kExCols * 2 +
           static_cast<size_t>(kExStages) * kExCols * RCAP * 2 + static_cast<size_t>(kExStages) * kExRows * RCAP * 2;
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

// ---- decode gather fold grouped by expert -----------------------------------------
//
// The same fold with each block serving one expert: block (e, c) takes expert
// e and output columns [COLS c, COLS (c + 1)). It finds the expert's rows by
// scanning indices (an ordered compaction, kGSeg slots at a time), computes
// their xa with A_e staged in shared memory, and folds its column chunk of
// each row with the chunk's B_e rows held in registers. A_e and B_e are then
// read once per block rather than once per row: at 512 rows over 128
// experts, about 4 rows share each expert's 88 KB of A_e and B_e. Every
// block of an expert recomputes the rows' xa (its column chunks need all of
// it); the blocks of chunk 0 store it.
constexpr int kGThreads = 256;
constexpr int kGSeg = 2048;      // slots scanned per compaction segment
constexpr int kGBatch = 32;      // rows per shrink / fold batch
constexpr int kGAElems = 12288;  // A_e values staged at once (24 KB): kGAElems / RCAP columns of k

template <int RCAP>
struct GatherGroup {
    static constexpr int CPT = RCAP <= 32 ? 2 : 1;  // output columns per thread
    static constexpr int COLS = kGThreads * CPT;    // output columns per block
    static constexpr int KC = kGAElems / RCAP;      // k columns of A_e per stage (a multiple of 8)
};

// The slot counts the grouped kernel takes. Below kGMinSlots the row-per-block
// kernel is faster (measured at rank 16, 128 experts: 512 rows 9.0 us against
// 15.8; 4096 rows 52.2 us against 45.4, where re-reading A_e and B_e per row
// makes the row-per-block kernel L2-bound); above kGMaxSlots each block would
// scan too many expert ids.
constexpr uint32_t kGMinSlots = 2048;
constexpr uint32_t kGMaxSlots = 16384;

template <int RCAP>
__global__ void __launch_bounds__(kGThreads, RCAP <= 16 ? 2 : 1)
lora_gather_grouped_kernel(const __nv_bfloat16* __restrict__ x, const uint32_t* __restrict__ indices,
                           const int32_t* __restrict__ row_adapter, const uint64_t* __restrict__ a_table,
                           const uint64_t* __restrict__ b_table, const float* __restrict__ scale_table,
                           __nv_bfloat16* __restrict__ xa, __nv_bfloat16* __restrict__ base, uint32_t n_experts,
                           int k_in, int n_out, int max_rank, uint32_t n_slots, uint32_t top_k, uint32_t x_gather) {
    pdl_wait();
    using G = GatherGroup<RCAP>;
    constexpr int CPT = G::CPT, KC = G::KC;
    constexpr int UNR = RCAP <= 32 ? 4 : 1;  // x pieces of a row in flight per lane (registers allowing)
    const int n_chunks = (n_out + G::COLS - 1) / G::COLS;
    const uint32_t e = blockIdx.x / n_chunks;
    const int chunk = static_cast<int>(blockIdx.x - e * n_chunks);
    if (e >= n_experts) return;
    const uint64_t aptr = a_table[e];
    if (aptr == 0) return;  // block-uniform: the expert has no adapter
    __shared__ int s_rows[kGSeg];
    __shared__ int s_wcnt[2][kGThreads / 32];
    __shared__ float s_acc[kGBatch][RCAP];
    __shared__ __align__(16) __nv_bfloat16 s_a[kGAElems];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const __nv_bfloat16* A = reinterpret_cast<const __nv_bfloat16*>(aptr);
    const __nv_bfloat16* B = reinterpret_cast<const __nv_bfloat16*>(b_table[e]);
    const float sc = scale_table[e];
    const int c0 = chunk * G::COLS + tid * CPT;  // this thread's first output column
    float bw[CPT][RCAP];  // B_e rows of this thread's columns (zero past n_out or max_rank)
#pragma unroll
    for (int i = 0; i < CPT; ++i)
#pragma unroll
        for (int j = 0; j < RCAP; ++j)
            bw[i][j] = (c0 + i < n_out && j < max_rank) ? __bfloat162float(B[static_cast<size_t>(c0 + i) * max_rank + j])
                                                        : 0.0f;

    for (uint32_t seg = 0; seg < n_slots; seg += kGSeg) {
        // 1. this segment's rows of expert e, in slot order: every thread loads the
        // expert ids of its slots at once, then warp ballots compact them
        constexpr int PER = kGSeg / kGThreads;
        const int rounds = static_cast<int>((min(static_cast<uint32_t>(kGSeg), n_slots - seg) + kGThreads - 1) / kGThreads);
        bool mine[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const uint32_t s = seg + q * kGThreads + tid;
            mine[q] = q < rounds && s < n_slots && indices[s] == e;
        }
        if (row_adapter != nullptr) {
#pragma unroll
            for (int q = 0; q < PER; ++q)
                if (mine[q]) mine[q] = row_adapter[(seg + q * kGThreads + tid) / top_k] >= 0;
        }
        int cnt = 0;
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            if (q >= rounds) break;  // block-uniform
            const unsigned bal = __ballot_sync(0xffffffffu, mine[q]);
            if (lane == 0) s_wcnt[q & 1][warp] = __popc(bal);
            __syncthreads();  // (the other buffer of s_wcnt is the one the next round writes)
            int before = cnt, total = cnt;
#pragma unroll
            for (int w = 0; w < kGThreads / 32; ++w) {
                if (w < warp) before += s_wcnt[q & 1][w];
                total += s_wcnt[q & 1][w];
            }
            if (mine[q]) s_rows[before + __popc(bal & ((1u << lane) - 1u))] = static_cast<int>(seg + q * kGThreads + tid);
            cnt = total;
        }
        __syncthreads();  // s_rows complete
        // 2. the rows in batches: shrink, then fold this block's columns
        for (int b0 = 0; b0 < cnt; b0 += kGBatch) {
            const int nb = min(kGBatch, cnt - b0);
            for (int i = tid; i < kGBatch * RCAP; i += kGThreads) s_acc[i / RCAP][i % RCAP] = 0.0f;
            for (int k0 = 0; k0 < k_in; k0 += KC) {
                const int kc = min(KC, k_in - k0);  // a multiple of 8
                __syncthreads();                    // s_a is free, s_acc is zeroed
                for (int i = tid; i < RCAP * (kc / 8); i += kGThreads) {
                    const int j = i / (kc / 8), p = i - j * (kc / 8);
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (j < max_rank) v = __ldg(reinterpret_cast<const uint4*>(A + static_cast<size_t>(j) * k_in + k0) + p);
                    *reinterpret_cast<uint4*>(s_a + j * kc + 8 * p) = v;
                }
                __syncthreads();
                // warp w: rows b0 + w, + 8, ...; lanes split the chunk in 8-value pieces
                for (int i = warp; i < nb; i += kGThreads / 32) {
                    const uint32_t s = static_cast<uint32_t>(s_rows[b0 + i]);
                    const __nv_bfloat16* xr = x + static_cast<size_t>(x_gather ? s / top_k : s) * k_in + k0;
                    float acc[RCAP];
#pragma unroll
                    for (int j = 0; j < RCAP; ++j) acc[j] = 0.0f;
#pragma unroll UNR
                    for (int c = lane; c < kc / 8; c += 32) {
                        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(xr) + c);
                        const float2 x0 = Act<MOE_ACT_BF16>::unpack2(xv.x), x1 = Act<MOE_ACT_BF16>::unpack2(xv.y),
                                     x2 = Act<MOE_ACT_BF16>::unpack2(xv.z), x3 = Act<MOE_ACT_BF16>::unpack2(xv.w);
#pragma unroll
                        for (int j = 0; j < RCAP; ++j) {
                            const uint4 av = *reinterpret_cast<const uint4*>(s_a + j * kc + 8 * c);
                            const float2 a0 = Act<MOE_ACT_BF16>::unpack2(av.x), a1 = Act<MOE_ACT_BF16>::unpack2(av.y),
                                         a2 = Act<MOE_ACT_BF16>::unpack2(av.z), a3 = Act<MOE_ACT_BF16>::unpack2(av.w);
                            float t = acc[j];
                            t = fmaf(x0.x, a0.x, t); t = fmaf(x0.y, a0.y, t);
                            t = fmaf(x1.x, a1.x, t); t = fmaf(x1.y, a1.y, t);
                            t = fmaf(x2.x, a2.x, t); t = fmaf(x2.y, a2.y, t);
                            t = fmaf(x3.x, a3.x, t); t = fmaf(x3.y, a3.y, t);
                            acc[j] = t;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < RCAP; ++j) {
                        float v = acc[j];
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                        if (lane == 0) s_acc[i][j] += v;  // only this warp touches row i
                    }
                }
            }
            __syncthreads();  // every partial sum is in s_acc
            // xa = bf16 of the sums (ranks past max_rank are zero); chunk 0 stores it
            for (int i = tid; i < nb * RCAP; i += kGThreads) {
                const int r = i / RCAP, j = i - r * RCAP;
                const __nv_bfloat16 v = __float2bfloat16_rn(s_acc[r][j]);
                s_acc[r][j] = __bfloat162float(v);
                if (chunk == 0 && j < max_rank) xa[static_cast<size_t>(s_rows[b0 + r]) * max_rank + j] = v;
            }
            __syncthreads();
            // fold: eight rows at a time, their base values loaded together
            constexpr int RG = 8;
            for (int g0 = 0; g0 < nb; g0 += RG) {
                float yv[RG][CPT];
#pragma unroll
                for (int r = 0; r < RG; ++r)
#pragma unroll
                    for (int q = 0; q < CPT; ++q) {
                        yv[r][q] = 0.0f;
                        if (g0 + r < nb && c0 + q < n_out)
                            yv[r][q] = __bfloat162float(base[static_cast<size_t>(s_rows[b0 + g0 + r]) * n_out + c0 + q]);
                    }
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    if (g0 + r >= nb) break;
                    float d[CPT];
#pragma unroll
                    for (int q = 0; q < CPT; ++q) d[q] = 0.0f;
#pragma unroll
                    for (int j = 0; j < RCAP; ++j) {
                        const float xv = s_acc[g0 + r][j];
#pragma unroll
                        for (int q = 0; q < CPT; ++q) d[q] = fmaf(xv, bw[q][j], d[q]);
                    }
                    const size_t s = static_cast<size_t>(s_rows[b0 + g0 + r]);
#pragma unroll
                    for (int q = 0; q < CPT; ++q) {
                        if (c0 + q >= n_out) continue;
                        const float dl = __bfloat162float(__float2bfloat16_rn(d[q]));  // bf16 delta
                        base[s * n_out + c0 + q] = __float2bfloat16_rn(__fadd_rn(yv[r][q], __fmul_rn(sc, dl)));
                    }
                }
            }
            __syncthreads();  // s_acc and s_rows are reused by the next batch or segment
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
    // resident blocks per SM of each kernel, from its registers and shared memory (queried once per device)
    static int configured_for = -1;
    static int occ_shrink = 0, occ_expand[3] = {0, 0, 0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        const void* ek[3] = {reinterpret_cast<const void*>(moe::lora_expand_fold_kernel<16>),
                             reinterpret_cast<const void*>(moe::lora_expand_fold_kernel<32>),
                             reinterpret_cast<const void*>(moe::lora_expand_fold_kernel<64>)};
        const size_t es[3] = {moe::lora_expand_smem<16>(), moe::lora_expand_smem<32>(), moe::lora_expand_smem<64>()};
        const size_t ss = moe::lora_shrink_smem(MOE_MAX_LORA_RANK);
        int rc = moe::set_smem_limit(reinterpret_cast<const void*>(moe::lora_shrink_kernel), static_cast<int>(ss));
        for (int i = 0; i < 3 && rc == MOE_OK; ++i) rc = moe::set_smem_limit(ek[i], static_cast<int>(es[i]));
        if (rc != MOE_OK) return rc;
        // the shrink at rank 16, the common case; larger ranks take more shared memory per block
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_shrink, moe::lora_shrink_kernel, 32 * moe::kShrinkWarps,
                                                          moe::lora_shrink_smem(16)) != cudaSuccess)
            return moe::fail(MOE_ERR_CUDA, "%s: occupancy query failed", who);
        for (int i = 0; i < 3; ++i)
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_expand[i], ek[i], moe::kExThreads, es[i]) !=
                cudaSuccess)
                return moe::fail(MOE_ERR_CUDA, "%s: occupancy query failed", who);
        configured_for = dev;
    }
    const int rslot = route->max_rank <= 16 ? 0 : (route->max_rank <= 32 ? 1 : 2);
    // upper bounds of the tile counts the kernels find on the device: every expert
    // adds at most one partial tile to the window's full ones
    const long s_tiles = (window + moe::kShrinkRows - 1) / moe::kShrinkRows + static_cast<long>(route->n_experts);
    const size_t shrink_smem = moe::lora_shrink_smem(static_cast<int>(route->max_rank));
    const long s_cap = static_cast<long>(route->max_rank <= 16 ? (occ_shrink > 0 ? occ_shrink : 1) : 1) * sms;
    const int s_grid = static_cast<int>(s_tiles < s_cap ? s_tiles : s_cap);
    const int n_chunks = (static_cast<int>(route->n_out) + moe::kExCols - 1) / moe::kExCols;
    const long units = ((window + moe::kExRows - 1) / moe::kExRows + static_cast<long>(route->n_experts)) * n_chunks;
    const long e_cap = static_cast<long>(occ_expand[rslot] > 0 ? occ_expand[rslot] : 1) * sms;
    const int grid = static_cast<int>(units < e_cap ? units : e_cap);
    const uint32_t vec16 = (route->n_out % 8 == 0 && moe::aligned16(base_out)) ? 1u : 0u;
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
        moe::launch_pdl(moe::lora_expand_fold_kernel<16>, grid, moe::kExThreads, moe::lora_expand_smem<16>(), st,
            xa_p, expert_offsets, sorted_token_ids, row_adapter, route->b_table, route->scale_table, base_p,
            route->n_experts, route->n_out, route->max_rank, row_offset, row_end, P, top_k, route->a_table, vec16);
    else if (route->max_rank <= 32)
        moe::launch_pdl(moe::lora_expand_fold_kernel<32>, grid, moe::kExThreads, moe::lora_expand_smem<32>(), st,
            xa_p, expert_offsets, sorted_token_ids, row_adapter, route->b_table, route->scale_table, base_p,
            route->n_experts, route->n_out, route->max_rank, row_offset, row_end, P, top_k, route->a_table, vec16);
    else
        moe::launch_pdl(moe::lora_expand_fold_kernel<64>, grid, moe::kExThreads, moe::lora_expand_smem<64>(), st,
            xa_p, expert_offsets, sorted_token_ids, row_adapter, route->b_table, route->scale_table, base_p,
            route->n_experts, route->n_out, route->max_rank, row_offset, row_end, P, top_k, route->a_table, vec16);
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
    if (n_slots >= moe::kGMinSlots && n_slots <= moe::kGMaxSlots) {
        // rows grouped by expert: a block per (expert, column chunk)
        const uint32_t ne = route->n_experts;
        auto grouped = [&](auto kernel, int cols) {
            const unsigned g = ne * static_cast<unsigned>((n_out + cols - 1) / cols);
            moe::launch_pdl(kernel, dim3(g), dim3(moe::kGThreads), 0, st, xp, indices, row_adapter, route->a_table,
                            route->b_table, route->scale_table, xa_p, base_p, ne, k_in, n_out, rank, n_slots, top_k,
                            x_gather);
        };
        if (rank <= 16) grouped(moe::lora_gather_grouped_kernel<16>, moe::GatherGroup<16>::COLS);
        else if (rank <= 32) grouped(moe::lora_gather_grouped_kernel<32>, moe::GatherGroup<32>::COLS);
        else grouped(moe::lora_gather_grouped_kernel<64>, moe::GatherGroup<64>::COLS);
        moe::count_launch();
        return moe::check_launch("moe_lora_gather_bgmv");
    }
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
