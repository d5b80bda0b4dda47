// Shared pieces of the grouped expert GEMMs (steps a3 and a4): launch
// parameters, the shared-memory tail, the device-built tile lists, the
// decode form's stream-K partition, and epilogue helpers. The kernel forms
// live in gemm_pair.cu (bf16 prefill, CTA pairs), gemm_decode.cu (bf16
// decode), gemm_ts.cu (GPTQ / NVFP4 / FP8 weights dequantised into TMEM) and
// gemm_tspair.cu (quantised prefill, dequantised into the TMEM of CTA pairs);
// gemm.cu holds the entry points.
#pragma once

#include "common.cuh"

namespace moe {
namespace gemm {

constexpr int BK = 64;
constexpr int W_ROWS = 256;             // weight rows per tile
constexpr int W_STAGE = W_ROWS * BK * 2;  // 32 KB
constexpr int NUM_EPI_WARPS = 4;
constexpr int NUM_DQ_WARPS = 8;  // two per SM sub-partition: dequantisation is latency-bound
constexpr int MAX_STAGES = 16;
constexpr int MAX_RSTAGES = 16;
constexpr int SMEM_LIMIT = 232448;      // dynamic shared memory per block (227 KB)

enum { MODE_GATE_UP = 0, MODE_DOWN = 1 };

struct GemmParams {
    const int32_t* offsets;     // [E + 1]
    const int32_t* sorted_ids;  // [max_padded]: pair ids, sentinel P
    int P;
    int E;
    int K;          // contraction length
    int n_out;      // output columns: I (gate/up) or H (down)
    int n_w;        // weight rows per expert: 2I or H
    int max_padded;
    void* out;      // [max_padded, n_out]
    const float* scale2;
    int group_size;
    int32_t* err;
    uint64_t wait_ns;  // how long a pipeline wait may last before the kernel gives up
    int block_size;  // align block size: spans are multiples of it, padding is a span's last < block_size rows
    int pad_free;    // the kernel's tile height is a multiple of block_size: no tile holds padding only
    const float* row_scale;  // FP8: fp32 scale per weight row [E, n_w]
    float* sk_part;  // split-K partial sums: one slice of SK_SLICE_FLOATS per CTA (decode form)
    int* sk_flag;    // split-K flags: 4 per CTA (one per epilogue warp)
    int sk_gen;      // this call's split-K generation (nonzero): the value a finished piece's flags hold
};

struct SmemTail {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t raw_full[MAX_RSTAGES];
    uint64_t raw_empty[MAX_RSTAGES];
    uint64_t afull[8];   // TMEM weight stages (TS forms)
    uint64_t aempty[8];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
    int n_tiles;
    int nt;  // column tiles per expert
    int off[MOE_MAX_EXPERTS + 1];
    int tstart[MOE_MAX_EXPERTS + 1];
};

constexpr int TAIL_BYTES = (static_cast<int>(sizeof(SmemTail)) + 127) / 128 * 128;

// split accumulators per half for a swapped tile of ntok tokens (see load_swapped)
__host__ __device__ constexpr int swapped_nacc(int ntok) { return ntok <= 32 ? 4 : (ntok <= 64 ? 2 : 1); }

__host__ __device__ constexpr int pow2_at_least(int v) {
    int p = 32;
    while (p < v) p <<= 1;
    return p;
}

// Compile-time shape of the bf16 decode form: NTOK activation rows (tokens)
// per tile are the MMA's N operand, the 256 weight rows of the tile two M=128
// A operands (gate | up halves, or two 128-column halves of the output).
template <int MODE, int NTOK>
struct DecodeShape {
    static constexpr int X_STAGE = NTOK * BK * 2;
    static constexpr int OUT_COLS = MODE == MODE_GATE_UP ? 128 : 256;  // output columns per tile
    // epilogue staging: per epilogue warp 2 halves x 16 tokens x 32 columns
    static constexpr int STG_BYTES = NUM_EPI_WARPS * 2 * 16 * 32 * 2;
    static constexpr int AVAIL = SMEM_LIMIT - 1024 - TAIL_BYTES - STG_BYTES;
    static constexpr int STAGES_FIT = AVAIL / (X_STAGE + W_STAGE);
    static constexpr int STAGES = STAGES_FIT < MAX_STAGES ? STAGES_FIT : MAX_STAGES;
    // two accumulator buffers (the epilogue drains one while the MMA fills the
    // other), each two halves x NACC split accumulators x NTOK columns
    static constexpr int NACC = swapped_nacc(NTOK);
    static constexpr int ACC = 2 * NTOK * NACC;
    static constexpr int TMEM_COLS = pow2_at_least(2 * ACC);
    // MMA issuers: one thread issues a tcgen05.mma about every 100 cycles
    // whatever its N, so from 64 tokens on each weight half has its own
    // issuing warp (with its own accumulators)
    static constexpr int NH = NTOK >= 64 ? 2 : 1;
    static constexpr int EPI0 = 1 + NH;  // first epilogue warp
    static constexpr int THREADS = 32 * (EPI0 + NUM_EPI_WARPS);
    static constexpr int SMEM = 1024 + STAGES * (X_STAGE + W_STAGE) + STG_BYTES + TAIL_BYTES;
    static_assert(STAGES >= 2, "not enough shared memory for two stages");
    static_assert(TMEM_COLS <= 512, "accumulators exceed TMEM");
    static_assert(SMEM <= SMEM_LIMIT, "shared memory over the limit");
};

struct TileInfo {
    int e, m0, n0, rows;
};

// ---- work partition of the decode form ----------------------------------------
// With whole tiles per CTA, a launch of n_tiles = w * G + rem tiles on G CTAs
// takes w + 1 tile-times however small rem is (153 tiles on 152 SMs take two).
// So the work is split as a hybrid of data-parallel waves and stream-K:
//   - n_tiles >= G: whole tiles are dealt round-robin (tile c + i * G), so
//     the CTAs of a wave work on neighbouring tiles at once and share the
//     weight rows of an expert's row blocks in L2. When the last wave is thin
//     (rem < G / 4: far too few SMs to keep HBM busy, one SM streams at most
//     about 1/90 of it), the last G + rem tiles are instead cut into G
//     contiguous ranges of k-blocks of nearly equal length (with a thicker
//     last wave, cutting measured no faster);
//   - n_tiles <= G / 2: each tile is cut into min(G / n_tiles, KB /
//     SK_MIN_PIECE) equal pieces.
// A tile cut by a range boundary is finished by the CTA whose range holds its
// k-block 0 (its owner: that piece ends the owner's range). Every other piece
// starts a range, so a CTA holds at most one; it leaves fp32 partial sums in
// the CTA's slice of the split-K area and raises the CTA's flags; the owner
// waits for the flags of the CTAs after it that hold the tile's other pieces,
// adds their slices and runs the epilogue. Waits only point to higher CTA
// indices, and a CTA's first item never waits, so with all CTAs resident (one
// per SM, grid <= SMs) the waits end.
constexpr int SK_MAX_CTAS = MOE_SPLITK_CTAS;
constexpr int SK_SLICE_FLOATS = 256 * 128;  // 2 halves x 128 weight rows x up to 128 tokens
constexpr int SK_MIN_PIECE = 4;
static_assert(static_cast<size_t>(SK_MAX_CTAS) * (SK_SLICE_FLOATS * 4 + 16) <= MOE_SPLITK_BYTES,
              "split-K area too small");

// One CTA's share: the whole tiles blockIdx.x + i * G below `base`, then the
// k-block units [lo, hi) of the stream-K region, which holds the tiles from
// `base` on (unit u = (tile - base) * KB + kb). The region holds fewer than 2 G tiles,
// so its unit counts stay far inside 32 bits (the launcher checks
// 2 G * KB * G < 2^31).
struct SkPlan {
    int base, geff;
    uint32_t U, lo, hi;
};

__device__ __forceinline__ SkPlan sk_plan(int n_tiles, int KB, int G, int c) {
    SkPlan pl;
    int region;
    if (n_tiles < G) {
        const int split_max = KB / SK_MIN_PIECE > 1 ? KB / SK_MIN_PIECE : 1;
        const int split = G / n_tiles < split_max ? G / n_tiles : split_max;
        region = split > 1 ? n_tiles : 0;
        pl.geff = split > 1 ? n_tiles * split : G;
    } else {
        const int w = n_tiles / G, rem = n_tiles - w * G;
        const bool cut = rem > 0 && 4 * rem < G;
        region = cut ? G + rem : 0;
        pl.geff = G;
    }
    pl.base = n_tiles - region;
    pl.U = static_cast<uint32_t>(region) * static_cast<uint32_t>(KB);
    pl.lo = c < pl.geff ? pl.U * static_cast<uint32_t>(c) / static_cast<uint32_t>(pl.geff) : 0u;
    pl.hi = c < pl.geff ? pl.U * static_cast<uint32_t>(c + 1) / static_cast<uint32_t>(pl.geff) : 0u;
    return pl;
}

// the CTA whose range holds unit u of the stream-K region
__device__ __forceinline__ int sk_cta_of(const SkPlan& pl, uint32_t u) {
    return static_cast<int>(((u + 1) * static_cast<uint32_t>(pl.geff) - 1) / pl.U);
}

// One piece of a tile: k-blocks [kb0, kb1) of `tile`.
struct SkItem {
    int tile, kb0, kb1;
};

// Walks a CTA's share in order (the same sequence in every role): the
// stream-K range first, then the round-robin whole tiles. A range is shorter
// than two tiles, so the owner's piece of a cut tile comes within its first
// three items, and the peer pieces it needs are the first items of the
// following CTAs: they are published by the time the owner's epilogue needs
// them, and that epilogue (which reads their slices from L2) overlaps the MMAs
// of the whole tiles that follow instead of ending the kernel.
struct SkWalk {
    int tile;
    uint32_t u;
    __device__ __forceinline__ explicit SkWalk(const SkPlan& pl) : tile(blockIdx.x), u(pl.lo) {}
    __device__ __forceinline__ bool next(const SkPlan& pl, int KB, SkItem& it) {
        if (u < pl.hi) {
            const uint32_t rt = u / static_cast<uint32_t>(KB);
            const uint32_t t0 = rt * static_cast<uint32_t>(KB);
            const uint32_t end = pl.hi < t0 + KB ? pl.hi : t0 + KB;
            it.tile = pl.base + static_cast<int>(rt);
            it.kb0 = static_cast<int>(u - t0);
            it.kb1 = static_cast<int>(end - t0);
            u = end;
            return true;
        }
        if (tile < pl.base) {  // whole tiles of the round-robin waves
            it.tile = tile;
            it.kb0 = 0;
            it.kb1 = KB;
            tile += gridDim.x;
            return true;
        }
        return false;
    }
    // the last CTA holding a piece of the owner's cut tile
    __device__ __forceinline__ static int last_peer(const SkPlan& pl, int KB, const SkItem& it) {
        if (it.kb0 > 0 || it.kb1 == KB) return blockIdx.x;
        return sk_cta_of(pl, static_cast<uint32_t>(it.tile - pl.base) * KB + KB - 1);
    }
};

template <int XROWS>
__device__ __forceinline__ TileInfo decode_tile(const SmemTail& s, int E, int tile, int out_cols) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.tstart[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    TileInfo t;
    t.e = lo;
    const int span = s.off[lo + 1] - s.off[lo];
    const int mt = (span + XROWS - 1) / XROWS;
    const int local = tile - s.tstart[lo];
    const int n_tile = local / mt;
    const int m_tile = local - n_tile * mt;
    t.m0 = s.off[lo] + m_tile * XROWS;
    t.n0 = n_tile * out_cols;
    t.rows = min(XROWS, s.off[lo + 1] - t.m0);
    return t;
}

// A tile whose first row is a padding row holds padding only. That cannot
// happen when the tile height is a multiple of the block size: a span is
// whole blocks and its padding is less than one block, so every tile of a
// span starts on a real row.
__device__ __forceinline__ bool tile_is_padding(const GemmParams& p, const TileInfo& t) {
    return !p.pad_free && __ldg(p.sorted_ids + t.m0) == p.P;
}

// first global weight row of each 128-row half of a tile (expert offset added by the caller)
template <int MODE>
__device__ __forceinline__ void half_bases(const GemmParams& p, int n0, int& c0, int& c1) {
    c0 = n0;
    c1 = (MODE == MODE_GATE_UP) ? p.n_out + n0 : n0 + 128;
}

// Every CTA builds the tile list from expert_offsets in shared memory: the
// offsets, and per expert the index of its first tile (row tiles of XROWS
// fastest, then column tiles of out_cols). Offsets that are negative,
// decreasing or beyond max_padded yield an empty list. Returns nonzero for
// bad offsets (the caller records the error once).
template <int XROWS>
__device__ __forceinline__ int build_tile_list(SmemTail& s, const GemmParams& p, int out_cols) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.E;
    for (int i = tid; i <= E; i += blockDim.x) s.off[i] = p.offsets[i];
    if (tid == 0) {
        s.abort_flag = 0;
        s.nt = (p.n_out + out_cols - 1) / out_cols;
    }
    __syncthreads();
    int bad = 0;
    for (int i = tid; i < E; i += blockDim.x) bad |= (s.off[i + 1] < s.off[i]);
    if (tid == 0) bad |= (s.off[0] < 0) | (s.off[E] > p.max_padded);
    bad = __syncthreads_or(bad);
    if (warp == 0) {
        // lane l owns experts [l * per, (l + 1) * per): local sums, warp scan, exclusive prefix
        const int per = (E + 31) / 32;
        int loc = 0;
        for (int j = 0; j < per; ++j) {
            const int e = lane * per + j;
            if (e < E) loc += ((s.off[e + 1] - s.off[e] + XROWS - 1) / XROWS) * s.nt;
        }
        int inc = loc;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, inc, d);
            if (lane >= d) inc += o;
        }
        int run = inc - loc;
        for (int j = 0; j < per; ++j) {
            const int e = lane * per + j;
            if (e < E) {
                s.tstart[e] = run;
                run += ((s.off[e + 1] - s.off[e] + XROWS - 1) / XROWS) * s.nt;
            }
        }
        if (lane == 31) s.n_tiles = bad ? 0 : inc;
    }
    return bad;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// ---- epilogue helpers ----------------------------------------------------------

template <int ACT>
__device__ __forceinline__ void store8(void* out, size_t elem_off, const float* f) {
    uint4 v;
    v.x = Act<ACT>::pack2(f[0], f[1]);
    v.y = Act<ACT>::pack2(f[2], f[3]);
    v.z = Act<ACT>::pack2(f[4], f[5]);
    v.w = Act<ACT>::pack2(f[6], f[7]);
    *reinterpret_cast<uint4*>(static_cast<typename Act<ACT>::T*>(out) + elem_off) = v;
}

// silu(g) * u = g / (1 + exp(-g)) * u with the fast exponential and the
// fast division (a few ulp of f32, far below the bf16 / fp16 rounding of the
// result). For very negative g, exp(-g) is inf or above 2^126 and the fast
// division returns 0 (the exact value is below 1e-36), so no NaN appears.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Rows of the tile that hold a pair: padding rows only sit at the end of an
// expert's span, fewer than block_size of them, so they are a suffix of the
// span's last tile within its last block_size - 1 rows. Each calling warp
// finds the first padding row with ballots over those sorted_token_ids.
__device__ __forceinline__ int valid_rows(const GemmParams& p, const SmemTail& s, const TileInfo& t, int lane) {
    if (t.m0 + t.rows != s.off[t.e + 1]) return t.rows;  // not the span's last tile
    for (int base = max(0, t.rows - (p.block_size - 1)); base < t.rows; base += 32) {
        const int r = base + lane;
        const bool pad = r < t.rows && __ldg(p.sorted_ids + t.m0 + r) == p.P;
        const unsigned m = __ballot_sync(0xffffffffu, pad);
        if (m) return base + __ffs(m) - 1;
    }
    return t.rows;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Swapped forms (D = weight row x token): each half's accumulator is split
// into NACC accumulators of NTOK columns, each filled by its own MMA issuer
// (or K step), so that several threads can issue. Half 0 owns columns
// [0, NACC*NTOK), half 1 the next NACC*NTOK. This loads tokens [c, c+16) of
// both halves and sums, in f32, the nsets accumulators s0, s0+1, ... (mod
// NACC) the tile used.
template <int NTOK, int NACC>
__device__ __forceinline__ void load_swapped(uint32_t taddr, int c, float (&fa)[16], float (&fb)[16],
                                             int nsets = NACC, int s0 = 0) {
    uint32_t a[16], b[16];
    tmem_ld16(taddr + s0 * NTOK + c, a);
    tmem_ld16(taddr + (NACC + s0) * NTOK + c, b);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        fa[j] = __uint_as_float(a[j]);
        fb[j] = __uint_as_float(b[j]);
    }
#pragma unroll
    for (int q = 1; q < NACC; ++q) {
        if (q >= nsets) break;
        const int sq = (s0 + q) % NACC;
        tmem_ld16(taddr + sq * NTOK + c, a);
        tmem_ld16(taddr + (NACC + sq) * NTOK + c, b);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            fa[j] += __uint_as_float(a[j]);
            fb[j] += __uint_as_float(b[j]);
        }
    }
}

// ---- tile list of the CTA-pair forms ------------------------------------------
//
// Row tiles of a pair form are cut from each expert's valid rows (its span
// minus the padding suffix) into ceil(rows / (16 MAXU)) tiles of nearly equal
// height, in steps of 16 rows; the MMA's N is the tile's height, so padding
// rows are not computed.

// Shared-memory tail of the pair kernel: the generic one plus each expert's
// count of valid (non-padding) rows.
struct PairTail : SmemTail {
    int vcnt[MOE_MAX_EXPERTS];
};

struct PairTile {
    int e, m0, n0;
    int rows;  // valid rows of the tile (the epilogue stores these)
    int n16;   // the MMA's N: rows rounded up to 16
};

// row tiles of an expert with v valid rows: units of 16 rows, at most MAXU units a tile
template <int MAXU>
__device__ __forceinline__ int pair_row_tiles(int v) {
    const int u = (v + 15) / 16;
    return (u + MAXU - 1) / MAXU;
}

// The pair kernel's tile list: like build_tile_list, with each expert's row
// tiles cut from its valid rows. Padding rows are a suffix of the span shorter
// than block_size, so one thread per expert finds the first one by a binary
// search over the span's last block_size - 1 rows.
template <int MAXU>
__device__ __forceinline__ int build_pair_tiles(PairTail& s, const GemmParams& p, int out_cols) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.E;
    for (int i = tid; i <= E; i += blockDim.x) s.off[i] = p.offsets[i];
    if (tid == 0) {
        s.abort_flag = 0;
        s.nt = (p.n_out + out_cols - 1) / out_cols;
    }
    __syncthreads();
    int bad = 0;
    for (int i = tid; i < E; i += blockDim.x) bad |= (s.off[i + 1] < s.off[i]);
    if (tid == 0) bad |= (s.off[0] < 0) | (s.off[E] > p.max_padded);
    bad = __syncthreads_or(bad);
    for (int e = tid; e < E; e += blockDim.x) {
        int v = 0;
        if (!bad) {
            const int r0 = s.off[e], r1 = s.off[e + 1];
            int lo = max(r0, r1 - (p.block_size - 1)), hi = r1;  // rows < lo hold pairs, rows >= hi padding
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (__ldg(p.sorted_ids + mid) == p.P) hi = mid; else lo = mid + 1;
            }
            v = lo - r0;
        }
        s.vcnt[e] = v;
    }
    __syncthreads();
    if (warp == 0) {
        const int per = (E + 31) / 32;
        int loc = 0;
        for (int j = 0; j < per; ++j) {
            const int e = lane * per + j;
            if (e < E) loc += pair_row_tiles<MAXU>(s.vcnt[e]) * s.nt;
        }
        int inc = loc;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, inc, d);
            if (lane >= d) inc += o;
        }
        int run = inc - loc;
        for (int j = 0; j < per; ++j) {
            const int e = lane * per + j;
            if (e < E) {
                s.tstart[e] = run;
                run += pair_row_tiles<MAXU>(s.vcnt[e]) * s.nt;
            }
        }
        if (lane == 31) s.n_tiles = bad ? 0 : inc;
    }
    return bad;
}

// Tile `tile` of a pair kernel's list: expert-major, then column tiles,
// row tiles fastest. Row tile i of mt covers units [U i / mt, U (i + 1) / mt)
// of the expert's U = ceil(valid / 16) units of 16 rows.
template <int MAXU>
__device__ __forceinline__ PairTile pair_tile(const PairTail& s, int E, int tile, int out_cols) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.tstart[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    PairTile t;
    t.e = lo;
    const int v = s.vcnt[lo];
    const int U = (v + 15) / 16;
    const int mt = (U + MAXU - 1) / MAXU;
    const int local = tile - s.tstart[lo];
    const int n_tile = local / mt;
    const int m_tile = local - n_tile * mt;
    const int u0 = U * m_tile / mt, u1 = U * (m_tile + 1) / mt;
    t.m0 = s.off[lo] + 16 * u0;
    t.rows = min(v, 16 * u1) - 16 * u0;
    t.n16 = 16 * (u1 - u0);
    t.n0 = n_tile * out_cols;
    return t;
}

struct Maps {
    CUtensorMap x, w, w5, r0, r1, r2;  // w5: gate/up rows interleaved by 8 (bf16 pair form)
    CUtensorMap q0, q1, q2;            // the quantised tensors in 128-row boxes per CTA (TS pair form)
};

// Launchers of the three forms (each in its own translation unit). mode is
// MODE_GATE_UP or MODE_DOWN; ntok the decode / TS tile height (0 selects the
// prefill form); wfmt / act the weight format and activation type.
int launch_pair_form(int mode, const Maps& m, const GemmParams& p, cudaStream_t st, const char* who);
int launch_decode_form(int mode, int ntok, const Maps& m, const GemmParams& p, cudaStream_t st, const char* who);
int launch_ts_form(int mode, int wfmt, int act, int ntok, const Maps& m, const GemmParams& p, cudaStream_t st,
                   const char* who);
// wide: the TS pair form's 256-row tiles (one accumulator buffer) instead of 192-row ones (two)
int launch_tspair_form(int mode, int wfmt, int act, int wide, const Maps& m, const GemmParams& p, cudaStream_t st,
                       const char* who);

}  // namespace gemm
}  // namespace moe
