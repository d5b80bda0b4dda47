// Steps a3 and a4: the grouped expert GEMMs on the 5th-generation tensor cores.
//
// What they compute restates metrale_gpu_runtime/cutlass/grouped.rs
// (nvfp4_grouped_gate_up_fused: group row i reads token sorted_token_ids[i],
// c_gate / c_up in group order; nvfp4_grouped_down: the intermediate is already
// in expert order) and ferrum-kernels src/backend/cuda/triton_fused_moe.rs
// (one launch covers all (token, expert) pairs; sentinel rows masked; raw
// GPTQ layout). The silu(gate) * up product is fused into the gate/up
// epilogue (spark_model moe_lora_grouped.rs: post-SiLU activations are stored
// in the activation type).
//
// Design (sm_103a):
//   * Persistent CTAs walk a static tile list built on the device from
//     expert_offsets, so nothing on the host depends on the routing and the
//     launch shape only depends on host-known sizes. A tile is 256 weight rows
//     (gate/up: 128 gate + 128 up rows of the same output columns, so the
//     epilogue fuses silu(gate) * up; down: 256 output columns) against a
//     block of activation rows, K in steps of 64 elements.
//   * Three kernels, chosen on the host from the average rows per touched
//     expert and the weight format:
//       - bf16 prefill (>= 128 rows per expert): grouped_gemm_pair_kernel, a
//         cluster of two CTAs issuing tcgen05.mma.cta_group::2 M=256 (128
//         activation rows per CTA) x N=256 (half the weight tile per CTA);
//       - bf16 decode: grouped_gemm_decode_kernel, operands swapped: each
//         weight half is an M=128 operand and NTOK tokens (16..128, one align
//         block) the N operand;
//       - GPTQ / NVFP4 / FP8, any size: grouped_gemm_ts_kernel, weights
//         dequantised by eight or sixteen warps into TMEM and used as the
//         M=128 A operand, NTOK tokens (128 for prefill) the N operand from
//         shared memory.
//   * Roles: TMA producer warps feed multi-stage rings; MMA issues go to
//     double-buffered TMEM accumulators where TMEM allows; four epilogue warps
//     drain them (tcgen05.ld -> activation -> global).
//   * Every mbarrier wait is bounded; on a timeout the CTA records
//     MOE_DEV_ERR_TIMEOUT, lets in-flight copies and MMAs land, frees TMEM and
//     returns.
#include "common.cuh"

namespace moe {
namespace {

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
    int* sk_flag;    // split-K flags: 4 per CTA (one per epilogue warp), zero between launches
};

struct SmemTail {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t raw_full[MAX_RSTAGES];
    uint64_t raw_empty[MAX_RSTAGES];
    uint64_t afull[4];   // TMEM weight stages (TS form)
    uint64_t aempty[4];
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

// ---- number conversions for the quantised formats ---------------------------------

__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(byte));
    return r;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    float v;
    if (e == 0) v = static_cast<float>(m) * 0.001953125f;  // m * 2^-9
    else if (e == 15 && m == 7) v = __uint_as_float(0x7fc00000u);
    else v = __uint_as_float(((e + 120u) << 23) | (m << 20));
    return (b & 0x80u) ? -v : v;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Four E2M1 codes (nibbles 0..3 of w) -> two bf16x2 words, with no
// conversion instructions: a byte permute looks up the high and low byte of
// each magnitude's bf16 value (0, .5, 1, 1.5, 2, 3, 4, 6 -> 0x0000, 0x3F00,
// 0x3F80, 0x3FC0, 0x4000, 0x4040, 0x4080, 0x40C0), a second permute
// interleaves them, and a sign-replicating permute carries each code's sign
// bit (bit 3) to bit 15 of its half.
__device__ __forceinline__ void e2m1x4_to_bf16x4(uint32_t w, uint32_t& p01, uint32_t& p23) {
    const uint32_t sel = w & 0x7777u;
    const uint32_t hi = prmt(0x3F3F3F00u, 0x40404040u, sel);
    const uint32_t lo = prmt(0xC0800000u, 0xC0804000u, sel);
    const uint32_t t = w << 4;  // byte 0 / 1 of t carry the signs of codes 0 / 2 in their top bit
    p01 = prmt(lo, hi, 0x5140u) | (prmt(t, w, 0xC888u) & 0x80008000u);
    p23 = prmt(lo, hi, 0x7362u) | (prmt(t, w, 0xD999u) & 0x80008000u);
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

// ---- bf16 decode form -------------------------------------------------------------

// One 16-token chunk of a decode tile to global memory: lane = weight row of
// each half, a / b = tokens [c, c+16) of half 0 / 1 (gate / up: one column's
// silu(gate) * up). The chunk goes through the warp's staging area
// ([half][token][32 columns]) so that it leaves as 16-byte stores of 8
// columns.
template <int MODE>
__device__ __forceinline__ void decode_store_chunk(const float (&a)[16], const float (&b)[16], __nv_bfloat16* stg,
                                                   __nv_bfloat16* out, int lane, int c, int nvalid, int m0,
                                                   int colw, int n_out) {
    using A = Act<MOE_ACT_BF16>;
    constexpr int HALVES = MODE == MODE_GATE_UP ? 1 : 2;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if (MODE == MODE_GATE_UP) {
            stg[j * 32 + lane] = A::from_f(silu_mul(a[j], b[j]));
        } else {
            stg[j * 32 + lane] = A::from_f(a[j]);
            stg[512 + j * 32 + lane] = A::from_f(b[j]);
        }
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 2 * HALVES; ++i) {
        const int pc = i * 32 + lane;  // [half][16 tokens][4 pieces of 8 columns]
        const int hh = pc >> 6, row = (pc >> 2) & 15, pq = pc & 3;
        const int col = colw + hh * 128 + pq * 8;
        if (c + row < nvalid && col < n_out)
            *reinterpret_cast<uint4*>(out + static_cast<size_t>(m0 + c + row) * n_out + col) =
                *reinterpret_cast<const uint4*>(stg + hh * 512 + row * 32 + pq * 8);
    }
    __syncwarp();
}

// Epilogue of one piece of a tile cut by the stream-K partition, for the
// calling epilogue warp (TMEM lane quarter q). A later piece (to_owner)
// leaves its fp32 sums in this CTA's slice of the split-K area and raises the
// CTA's flag for q; the owner waits for the flags of CTAs blockIdx.x + 1 ..
// last_peer, adds their slices to its own sums and stores the chunk. Returns
// false when a wait gave up.
template <int MODE, int NTOK, int NACC>
__device__ __forceinline__ bool decode_split_epilogue(const GemmParams& p, uint64_t* tfull, uint32_t aph,
                                                   const WaitCtx& wc, bool to_owner, int last_peer,
                                                   uint32_t tacc, int q, int lane, int nvalid,
                                                   __nv_bfloat16* stg, int m0, int colw) {
    const uint32_t taddr = tacc + (static_cast<uint32_t>(q * 32) << 16);
    // this lane's place in a slice: [quarter q][16-token chunk][half][4 floats of 16][lane], float4 units
    const size_t lane_off = static_cast<size_t>(q) * (NTOK / 16) * 256 + lane;
    constexpr size_t SLICE4 = SK_SLICE_FLOATS / 4;
    if (to_owner) {
        if (!mbar_wait(tfull, aph, wc)) return false;
        tc_fence_after();
        float4* d = reinterpret_cast<float4*>(p.sk_part) + blockIdx.x * SLICE4 + lane_off;
#pragma unroll 1
        for (int c = 0; c < NTOK && c < nvalid; c += 16) {
            float a[16], b[16];
            load_swapped<NTOK, NACC>(taddr, c, a, b);
            float4* dc = d + (c / 16) * 256;
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
                dc[j4 * 32] = make_float4(a[4 * j4], a[4 * j4 + 1], a[4 * j4 + 2], a[4 * j4 + 3]);
                dc[128 + j4 * 32] = make_float4(b[4 * j4], b[4 * j4 + 1], b[4 * j4 + 2], b[4 * j4 + 3]);
            }
        }
        // the slice is complete: publish it to the owner
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(p.sk_flag + blockIdx.x * 4 + q, 1);
        return true;
    }
    // owner: wait for the peers, fetch the first peer's first chunk while this
    // CTA's own MMAs may still run
    const int first_peer = blockIdx.x + 1;
    for (int pc = first_peer; pc <= last_peer; ++pc)
        if (!flag_wait(p.sk_flag + pc * 4 + q, wc)) return false;
    const float4* peer0 = reinterpret_cast<const float4*>(p.sk_part) + first_peer * SLICE4 + lane_off;
    float4 nx[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) nx[j] = __ldcg(peer0 + (j & 3) * 32 + (j >> 2) * 128);
    if (!mbar_wait(tfull, aph, wc)) return false;
    tc_fence_after();
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll 1
    for (int c = 0; c < NTOK && c < nvalid; c += 16) {
        float a[16], b[16];
        load_swapped<NTOK, NACC>(taddr, c, a, b);
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
            const float4 x = nx[j4], y = nx[4 + j4];
            a[4 * j4] += x.x; a[4 * j4 + 1] += x.y; a[4 * j4 + 2] += x.z; a[4 * j4 + 3] += x.w;
            b[4 * j4] += y.x; b[4 * j4 + 1] += y.y; b[4 * j4 + 2] += y.z; b[4 * j4 + 3] += y.w;
        }
        if (c + 16 < NTOK && c + 16 < nvalid) {  // the first peer's next chunk
            const float4* d = peer0 + (c / 16 + 1) * 256;
#pragma unroll
            for (int j = 0; j < 8; ++j) nx[j] = __ldcg(d + (j & 3) * 32 + (j >> 2) * 128);
        }
        for (int pc = first_peer + 1; pc <= last_peer; ++pc) {
            const float4* d = reinterpret_cast<const float4*>(p.sk_part) + pc * SLICE4 + lane_off + (c / 16) * 256;
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
                const float4 x = __ldcg(d + j4 * 32), y = __ldcg(d + 128 + j4 * 32);
                a[4 * j4] += x.x; a[4 * j4 + 1] += x.y; a[4 * j4 + 2] += x.z; a[4 * j4 + 3] += x.w;
                b[4 * j4] += y.x; b[4 * j4 + 1] += y.y; b[4 * j4 + 2] += y.z; b[4 * j4 + 3] += y.w;
            }
        }
        decode_store_chunk<MODE>(a, b, stg, out, lane, c, nvalid, m0, colw, p.n_out);
    }
    // every lane has read the peers' slices: clear their flags for the next launch
    __syncwarp();
    if (lane == 0)
        for (int pc = first_peer; pc <= last_peer; ++pc) p.sk_flag[pc * 4 + q] = 0;
    return true;
}

template <int MODE, int NTOK>
__global__ void __launch_bounds__(DecodeShape<MODE, NTOK>::THREADS, 1)
grouped_gemm_decode_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                           const GemmParams p) {
    pdl_wait();
    using S = DecodeShape<MODE, NTOK>;
    constexpr int ACT = MOE_ACT_BF16;
    constexpr int XROWS = NTOK, STAGES = S::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024_shared(smem_raw);
    uint8_t* sX = smem;
    uint8_t* sW = smem + STAGES * S::X_STAGE;
    uint8_t* sStg = sW + STAGES * W_STAGE;
    SmemTail& s = *reinterpret_cast<SmemTail*>(sStg + S::STG_BYTES);
    const WaitCtx wc{&s.abort_flag, p.err, p.wait_ns};

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int E = p.E;

    const int bad = build_tile_list<XROWS>(s, p, S::OUT_COLS);
    if (tid == 0) {
        if (bad) set_err(p.err, MOE_DEV_ERR_OFFSETS);
#pragma unroll
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], S::NH);  // every issuer releases the stage
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.tfull[i], S::NH);
            mbar_init(&s.tempty[i], NUM_EPI_WARPS);
        }
        mbar_init(&s.mma_done, S::NH);
        fence_mbar_init();
    }
    __syncthreads();
    const int n_tiles = s.n_tiles;
    if (n_tiles == 0) return;  // block-uniform: nothing allocated yet
    const int KB = (p.K + BK - 1) / BK;  // a ragged last block is zero-filled
    const SkPlan plan = sk_plan(n_tiles, KB, gridDim.x, blockIdx.x);
    if (static_cast<int>(blockIdx.x) >= plan.base && plan.lo >= plan.hi) return;

    if (warp == 1) {
        tmem_alloc(&s.tmem_base, S::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: activations and weights ----------------
            uint32_t stage = 0, phase = 0;
            long issued = 0;
            bool ok = true;
            SkItem it;
            for (SkWalk wk(plan); ok && wk.next(plan, KB, it);) {
                const TileInfo t = decode_tile<XROWS>(s, E, it.tile, S::OUT_COLS);
                if (tile_is_padding(p, t)) continue;
                int c0, c1;
                half_bases<MODE>(p, t.n0, c0, c1);
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1, wc)) { ok = false; break; }
                    mbar_arrive_expect_tx(&s.full[stage], S::X_STAGE + W_STAGE);
                    tma_load_2d(sX + stage * S::X_STAGE, &tmX, kb * BK, t.m0, &s.full[stage]);
                    uint8_t* w = sW + stage * W_STAGE;
                    tma_load_2d(w, &tmW, kb * BK, t.e * p.n_w + c0, &s.full[stage]);
                    tma_load_2d(w + W_STAGE / 2, &tmW, kb * BK, t.e * p.n_w + c1, &s.full[stage]);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            // let the copies still in flight land before the CTA may exit
            const long first = issued > STAGES ? issued - STAGES : 0;
            for (long j = first; j < issued; ++j)
                mbar_drain(&s.full[j % STAGES], static_cast<uint32_t>((j / STAGES) & 1), kWaitLimitNs / 8);
        }
    } else if (warp < S::EPI0) {
        if (lane == 0) {
            // ---------------- MMA issuers: A = weight halves, B = tokens ----------------
            const int hsel = S::NH == 2 ? warp - 1 : -1;  // the half this issuer owns (-1: both)
            constexpr uint32_t idesc = f16_idesc(ACT, 128, NTOK);
            uint32_t stage = 0, phase = 0;
            int local = 0;
            bool ok = true;
            SkItem it;
            for (SkWalk wk(plan); ok && wk.next(plan, KB, it);) {
                const TileInfo t = decode_tile<XROWS>(s, E, it.tile, S::OUT_COLS);
                if (tile_is_padding(p, t)) continue;
                const int acc = local & 1;
                const uint32_t aph = (local >> 1) & 1;
                ++local;
                if (!mbar_wait(&s.tempty[acc], aph ^ 1, wc)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + acc * S::ACC;
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!mbar_wait(&s.full[stage], phase, wc)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t xd = sw128_desc(smem_u32(sX + stage * S::X_STAGE));
                    const uint64_t wd = sw128_desc(smem_u32(sW + stage * W_STAGE));
                    const uint64_t wd1 = sw128_desc(smem_u32(sW + stage * W_STAGE + W_STAGE / 2));
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const int a = k % S::NACC;
                        const uint32_t en = kb > it.kb0 || k >= S::NACC;
                        if (hsel != 1) tc_mma(d + a * NTOK, wd + 2 * k, xd + 2 * k, idesc, en);
                        if (hsel != 0) tc_mma(d + (S::NACC + a) * NTOK, wd1 + 2 * k, xd + 2 * k, idesc, en);
                    }
                    tc_commit(&s.empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit(&s.tfull[acc]);
            }
            tc_commit(&s.mma_done);
            mbar_drain(&s.mma_done, 0, kWaitLimitNs / 8);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: lane = weight row of a half, columns = tokens ----------------
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        using T = typename Act<ACT>::T;
        T* out = static_cast<T*>(p.out);
        T* stg = reinterpret_cast<T*>(sStg) + (warp - S::EPI0) * (2 * 16 * 32);
        int local = 0;
        bool ok = true;
        SkItem it;
        for (SkWalk wk(plan); ok && wk.next(plan, KB, it);) {
            const TileInfo t = decode_tile<XROWS>(s, E, it.tile, S::OUT_COLS);
            if (tile_is_padding(p, t)) continue;
            const int acc = local & 1;
            const uint32_t aph = (local >> 1) & 1;
            ++local;
            const int nvalid = valid_rows(p, s, t, lane);  // its loads overlap the wait
            const int colw = t.n0 + q * 32;  // this warp's first column (half 0)
            const int last_peer = SkWalk::last_peer(plan, KB, it);
            if (it.kb0 > 0 || last_peer > static_cast<int>(blockIdx.x)) {
                // a piece of a cut tile (stream-K)
                if (!decode_split_epilogue<MODE, NTOK, S::NACC>(p, &s.tfull[acc], aph, wc, it.kb0 > 0,
                                                                 last_peer, tmem_base + acc * S::ACC, q, lane,
                                                                 nvalid, stg, t.m0, colw)) {
                    ok = false;
                    break;
                }
            } else {
                if (!mbar_wait(&s.tfull[acc], aph, wc)) break;
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * S::ACC;
#pragma unroll 1
                for (int c = 0; c < NTOK && c < nvalid; c += 16) {
                    float a[16], b[16];
                    load_swapped<NTOK, S::NACC>(taddr, c, a, b);
                    decode_store_chunk<MODE>(a, b, stg, out, lane, c, nvalid, t.m0, colw, p.n_out);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.tempty[acc]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, S::TMEM_COLS);
}

// ---- CTA-pair prefill kernel (bf16 weights) -------------------------------------
//
// The prefill form on a pair of SMs: tcgen05.mma.cta_group::2 with M=256
// weight rows (128 per CTA) and N = up to 256 activation rows of one expert
// (N/2 per CTA). Every SM then moves 32 KB through shared memory per 64-deep
// k block (a weight half and its rows), and holds six stages. One thread of
// the even CTA (the leader) issues the MMAs; both CTAs' TMA loads complete on
// the leader's full barrier; the leader's commits arrive on both CTAs'
// barriers; the follower's epilogue warps release the accumulator through the
// leader's barrier.
//
// Row tiles. An expert's valid rows (its span minus the padding suffix) are
// cut into ceil(rows / 256) tiles of nearly equal height, in steps of 16
// rows, and the MMA's N is the tile's height: 1040 rows run as five tiles of
// 208 rows instead of four full tiles and a 16-row tail. A thread issues a
// tcgen05.mma in about the same time whatever its N up to about 200
// (measured), so a short tail tile costs nearly a full tile's time, while
// equal tiles of 200 rows or more keep the tensor pipe busy throughout.
// Padding rows are not computed.
//
// Gate/up: each CTA takes 64 gate and the 64 up rows of the same output
// columns, interleaved in groups of 8 by one 5-D TMA copy, so the SiLU pairs
// TMEM lane j with lane j + 8.

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

// row tiles of an expert with v valid rows: units of 16 rows, at most 16 units a tile
__device__ __forceinline__ int pair_row_tiles(int v) {
    const int u = (v + 15) / 16;
    return (u + 15) / 16;
}

// The pair kernel's tile list: like build_tile_list, with each expert's row
// tiles cut from its valid rows. Padding rows are a suffix of the span shorter
// than block_size, so one thread per expert finds the first one by a binary
// search over the span's last block_size - 1 rows.
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
            if (e < E) loc += pair_row_tiles(s.vcnt[e]) * s.nt;
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
                run += pair_row_tiles(s.vcnt[e]) * s.nt;
            }
        }
        if (lane == 31) s.n_tiles = bad ? 0 : inc;
    }
    return bad;
}

// Tile `tile` of the pair kernel's list: expert-major, then column tiles,
// row tiles fastest. Row tile i of mt covers units [U i / mt, U (i + 1) / mt)
// of the expert's U = ceil(valid / 16) units of 16 rows.
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
    const int mt = (U + 15) / 16;
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

// Epilogue of a pair tile for the calling warp: TMEM lanes 32q..32q+31 of
// this CTA are weight rows, columns 0..N-1 the tile's rows (tokens).
//   gate/up: lane j holds, for output column n0 + 64 rank + 16 q + 8 (j >> 4) +
//   (j & 7), the gate sums if (j & 8) == 0 and the up sums otherwise;
//   down: lane j is output column n0 + 128 rank + 32 q + j.
// Each 16-row chunk goes through the warp's staging area and leaves as 16-byte
// stores of 8 columns.
template <int MODE>
__device__ __forceinline__ void pair_swapped_epilogue(const GemmParams& p, uint32_t ta, __nv_bfloat16* stg,
                                                      const PairTile& t, int nvalid, int rank, int q, int lane) {
    using A = Act<MOE_ACT_BF16>;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    // 32 rows per step; the next step's TMEM load is in flight while this one is converted
    uint32_t u[32], nx[32];
    tmem_ld32(ta, nx);
#pragma unroll 1
    for (int c = 0; c < nvalid; c += 32) {
        tmem_ld_wait_regs(nx);
#pragma unroll
        for (int j = 0; j < 32; ++j) u[j] = nx[j];
        if (c + 32 < nvalid) tmem_ld32(ta + c + 32, nx);
        if (MODE == MODE_GATE_UP) {
            // lane j and its partner j ^ 8 hold the gate and the up sums of one output
            // column; the gate lane finishes rows 0..15 of the step, the up lane rows 16..31
            const bool gate = (lane & 8) == 0;
            const int cl = 8 * (lane >> 4) + (lane & 7);  // column within the warp's 16
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float lo = __uint_as_float(u[j]), hi = __uint_as_float(u[16 + j]);
                const float other = __shfl_xor_sync(0xffffffffu, gate ? hi : lo, 8);
                const float g = gate ? lo : other;
                const float up = gate ? other : hi;
                stg[(gate ? j : 16 + j) * 16 + cl] = A::from_f(silu_mul(g, up));
            }
            __syncwarp();
            // [32 rows][16 columns]: 64 pieces of 8 columns, two per lane
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int pc = i * 32 + lane, r = pc >> 1, pq = pc & 1;
                const int col = t.n0 + 64 * rank + 16 * q + 8 * pq;
                if (c + r < nvalid && col < p.n_out)
                    *reinterpret_cast<uint4*>(out + static_cast<size_t>(t.m0 + c + r) * p.n_out + col) =
                        *reinterpret_cast<const uint4*>(stg + r * 16 + pq * 8);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) stg[j * 32 + lane] = A::from_f(__uint_as_float(u[j]));
            __syncwarp();
            // [32 rows][32 columns]: 128 pieces of 8 columns, four per lane
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int pc = i * 32 + lane, r = pc >> 2, pq = pc & 3;
                const int col = t.n0 + 128 * rank + 32 * q + 8 * pq;
                if (c + r < nvalid && col < p.n_out)
                    *reinterpret_cast<uint4*>(out + static_cast<size_t>(t.m0 + c + r) * p.n_out + col) =
                        *reinterpret_cast<const uint4*>(stg + r * 32 + pq * 8);
            }
        }
        __syncwarp();
    }
}

constexpr int PAIR_STAGES = 6;
constexpr int PAIR_A = 128 * BK * 2;  // this CTA's activation rows (a 128-row box, N/2 of them used)
constexpr int PAIR_B = 128 * BK * 2;  // this CTA's half of the weight tile
constexpr int PAIR_STG = NUM_EPI_WARPS * 32 * 32 * 2;  // epilogue staging: per warp 32 rows x 32 columns
constexpr int PAIR_TAIL_BYTES = (static_cast<int>(sizeof(PairTail)) + 127) / 128 * 128;
constexpr int PAIR_SMEM = 1024 + PAIR_STAGES * (PAIR_A + PAIR_B) + PAIR_STG + PAIR_TAIL_BYTES;
static_assert(PAIR_SMEM <= SMEM_LIMIT, "pair kernel shared memory over the limit");

template <int MODE>
__global__ void __launch_bounds__(192, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                         const __grid_constant__ CUtensorMap tmW5, const GemmParams p) {
    pdl_wait();
    constexpr int ACT = MOE_ACT_BF16;
    constexpr int OUT_COLS = MODE == MODE_GATE_UP ? 128 : 256;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024_shared(smem_raw);
    uint8_t* sA = smem;
    uint8_t* sB = smem + PAIR_STAGES * PAIR_A;
    uint8_t* sStg = sB + PAIR_STAGES * PAIR_B;
    PairTail& s = *reinterpret_cast<PairTail*>(sStg + PAIR_STG);
    const WaitCtx wc{&s.abort_flag, p.err, p.wait_ns};

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();  // 0: leader, 1: follower
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int E = p.E;

    const int bad = build_pair_tiles(s, p, OUT_COLS);  // identical in both CTAs
    if (tid == 0) {
        if (bad && rank == 0) set_err(p.err, MOE_DEV_ERR_OFFSETS);
        for (int i = 0; i < PAIR_STAGES; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.tfull[i], 1);
            mbar_init(&s.tempty[i], 2 * NUM_EPI_WARPS);
        }
        mbar_init(&s.mma_done, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const int n_tiles = s.n_tiles;
    if (pair >= n_tiles) return;  // the same in both CTAs of the pair: nothing allocated yet

    if (warp == 1) {
        tmem_alloc_pair(&s.tmem_base, 512);
        tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
        if (MODE == MODE_GATE_UP) tma_prefetch_desc(&tmW5);
    }
    tc_fence_before();
    cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = s.tmem_base;
    const uint32_t leader_full0 = mapa_shared(smem_u32(&s.full[0]), 0);
    const uint32_t leader_tempty0 = mapa_shared(smem_u32(&s.tempty[0]), 0);
    const int KB = (p.K + BK - 1) / BK;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            uint32_t stage = 0, phase = 0;
            long issued = 0;
            bool ok = true;
            for (int tile = pair; tile < n_tiles && ok; tile += npairs) {
                const PairTile t = pair_tile(s, E, tile, OUT_COLS);
                int c0, c1;
                half_bases<MODE>(p, t.n0, c0, c1);
                const int wrow = t.e * p.n_w + (rank == 0 ? c0 : c1);
                // this CTA holds the tile's rows [m0 + rank N/2, +N/2) (the 128-row box
                // may over-fetch; the MMA reads N/2 of them)
                const int arow = t.m0 + static_cast<int>(rank) * (t.n16 / 2);
                // gate/up: 8-row groups of gate and up rows for output columns
                // [n0 + 64 rank, +64): group coordinate (n0 + 64 rank) / 8
                const int g5 = t.n0 / 8 + 8 * static_cast<int>(rank);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1, wc)) { ok = false; break; }
                    if (rank == 0) mbar_arrive_expect_tx(&s.full[stage], 2 * (PAIR_A + PAIR_B));
                    const uint32_t bar = leader_full0 + stage * 8;
                    tma_load_2d_pair(sA + stage * PAIR_A, &tmX, kb * BK, arow, bar);
                    if (MODE == MODE_GATE_UP) tma_load_5d_pair(sB + stage * PAIR_B, &tmW5, kb * BK, 0, 0, g5, t.e, bar);
                    else tma_load_2d_pair(sB + stage * PAIR_B, &tmW, kb * BK, wrow, bar);
                    ++issued;
                    if (++stage == PAIR_STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (rank == 0) {  // let every copy of the pair land before either CTA may exit
                const long first = issued > PAIR_STAGES ? issued - PAIR_STAGES : 0;
                for (long j = first; j < issued; ++j)
                    mbar_drain(&s.full[j % PAIR_STAGES], static_cast<uint32_t>((j / PAIR_STAGES) & 1),
                               kWaitLimitNs / 8);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer (leader): D = weight rows x tile rows ----------------
            uint32_t stage = 0, phase = 0;
            int local = 0;
            bool ok = true;
            for (int tile = pair; tile < n_tiles && ok; tile += npairs) {
                const PairTile t = pair_tile(s, E, tile, OUT_COLS);
                const int acc = local & 1;
                const uint32_t aph = (local >> 1) & 1;
                ++local;
                if (!mbar_wait(&s.tempty[acc], aph ^ 1, wc)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + acc * 256;
                const uint32_t idesc = f16_idesc(ACT, 256, t.n16);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&s.full[stage], phase, wc)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(smem_u32(sA + stage * PAIR_A));
                    const uint64_t bd = sw128_desc(smem_u32(sB + stage * PAIR_B));
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) tc_mma_pair(d, bd + 2 * k, ad + 2 * k, idesc, (kb | k) != 0);
                    tc_commit_pair(&s.empty[stage], 0x3);
                    if (++stage == PAIR_STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit_pair(&s.tfull[acc], 0x3);
            }
            tc_commit_pair(&s.mma_done, 0x1);
            mbar_drain(&s.mma_done, 0, kWaitLimitNs / 8);
        }
        __syncwarp();
    } else if (warp < 2 + NUM_EPI_WARPS) {
        // ---------------- epilogue (both CTAs): lane = weight row, columns = tile rows ----------------
        const int q = warp & 3;
        __nv_bfloat16* stg = reinterpret_cast<__nv_bfloat16*>(sStg) + (warp - 2) * (32 * 32);
        int local = 0;
        for (int tile = pair; tile < n_tiles; tile += npairs) {
            const PairTile t = pair_tile(s, E, tile, OUT_COLS);
            const int acc = local & 1;
            const uint32_t aph = (local >> 1) & 1;
            ++local;
            if (!mbar_wait(&s.tfull[acc], aph, wc)) break;
            tc_fence_after();
            const uint32_t ta = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * 256;
            pair_swapped_epilogue<MODE>(p, ta, stg, t, t.rows, static_cast<int>(rank), q, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0) mbar_arrive(&s.tempty[acc]);
                else mbar_arrive_cluster(leader_tempty0 + acc * 8);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the leader's MMAs read this CTA's shared memory and write its TMEM
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, 512);
}

// ---- TS form: quantised weights dequantised into TMEM ----------------------------
//
// For GPTQ, NVFP4 and FP8 weights the weight tile is the MMA's A operand and
// lives in TMEM: each set of eight dequantising warps owns 32 weight rows
// (TMEM lanes) of one 128-row half per warp and writes a row's 64 k values of
// a k block as 32 columns with tcgen05.st. The activations (NTOK token rows) are the B operand in
// shared memory, fed by TMA. D is (weight row x token), two halves (gate |
// up, or two 128-column halves of the output) of NTOK columns each. Shared
// memory then carries only the raw quantised bytes and the activations; the
// 16-bit weights never touch it.
constexpr int TS_STAGES = 4;   // weight stages in TMEM (one 64-deep k block each)
constexpr int TS_A_COL = 256;  // first TMEM column of the weight stages (64 columns each)
constexpr int RAW2 = 18432;    // bytes of one raw stage: two k blocks (GPTQ, NVFP4) or one (FP8)

template <int MODE, int WFMT, int ACT, int NTOK>
struct TsShape {
    static constexpr int X_STAGE = NTOK * BK * 2;
    static constexpr int OUT_COLS = MODE == MODE_GATE_UP ? 128 : 256;
    // MMA issuers. One thread issues a tcgen05.mma about every 100 cycles
    // whatever its N, so several issuing warps share the work, each with its
    // own accumulators: NR issuers take the k blocks in turn (issuer set r
    // owns the CTA's k blocks g = r mod NR, counted over all its tiles, and
    // accumulator set r), and with NH = 2 each half (gate | up, or the two
    // output halves) has its own issuer. Per 64-deep k block an issuer then
    // issues 8 / NH MMAs and 2 commits for one k block in NR. Owning by the
    // CTA-wide index, with stage counts that are multiples of NR, gives every
    // ring stage a single issuer, which then sees its barrier phases in order
    // (owning by index within a tile breaks that when KB mod NR != 0: an
    // issuer could come back to a stage two phases ahead of its producer and
    // take a stale phase for the current one).
    static constexpr int NH = NTOK >= 64 ? 2 : 1;
    static constexpr int NR = NTOK >= 128 ? 1 : (NTOK >= 64 ? 2 : 4);
    static constexpr int NI = NH * NR;
    static constexpr int ACC = 2 * NR * NTOK;  // TMEM columns per accumulator buffer: [half][set][token]
    static constexpr int NBUF = 2 * ACC <= TS_A_COL ? 2 : 1;
    // Dequantising warps: NSET sets of eight (one warp per TMEM lane quarter
    // and weight half) take the k blocks in turn, so that one set converts
    // while the other waits on its loads. Two sets measured 11-13% faster on
    // GPTQ and NVFP4 decode layers and 2% on NVFP4 prefill; one set stays for
    // FP8 (its conversion is short: two sets measured 4% slower) and GPTQ
    // prefill (2% slower).
    static constexpr int NSET =
        WFMT == MOE_W_FP8_E4M3 || (WFMT == MOE_W_GPTQ_INT4 && NTOK >= 128) ? 1 : 2;
    static constexpr int NDQ = NSET * NUM_DQ_WARPS;
    static constexpr int EPI0 = 1 + NI;                 // first epilogue warp
    static constexpr int DQ0 = EPI0 + NUM_EPI_WARPS;    // first dequantising warp
    static constexpr int RAWW = DQ0 + NDQ;              // raw producer warp
    static constexpr int THREADS = 32 * (RAWW + 1);
    // epilogue staging: per epilogue warp 2 halves x 16 tokens x 32 columns
    static constexpr int STG_BYTES = NUM_EPI_WARPS * 2 * 16 * 32 * 2;
    static constexpr int AVAIL = SMEM_LIMIT - 1024 - TAIL_BYTES - STG_BYTES;
    // The activation ring is its own, deeper than the TMEM weight ring: its
    // loads queue behind the raw weight stream. At least 4 raw stages (8 k
    // blocks) are kept.
    static constexpr int X_FIT = (AVAIL - 4 * RAW2) / X_STAGE;
    static constexpr int XSTAGES = (X_FIT < 12 ? X_FIT : 12) / NR * NR;
    static constexpr int RAW_FIT = (AVAIL - XSTAGES * X_STAGE) / RAW2;
    static constexpr int RSTAGES = RAW_FIT < MAX_RSTAGES ? RAW_FIT : MAX_RSTAGES;
    static constexpr int SMEM = 1024 + XSTAGES * X_STAGE + RSTAGES * RAW2 + STG_BYTES + TAIL_BYTES;
    // GPTQ gate/up writes each group of 8 k values in the order 0,4,1,5,2,6,3,7
    // (the order the int4 -> fp16 conversion produces them in); the gather
    // kernel stores the activations in the same order, so the products match
    static constexpr bool PERM = WFMT == MOE_W_GPTQ_INT4 && MODE == MODE_GATE_UP;
    static_assert(NBUF * ACC <= TS_A_COL, "accumulators overlap the weight stages");
    static_assert(TS_A_COL + TS_STAGES * 64 <= 512, "weight stages exceed TMEM");
    static_assert(XSTAGES >= 4 && XSTAGES <= MAX_STAGES, "activation ring size");
    static_assert(XSTAGES % NR == 0 && TS_STAGES % NR == 0, "every ring stage must have one issuer");
    static_assert(TS_STAGES % NSET == 0, "every weight stage must have one dequantising set");
    static_assert(RSTAGES >= 4, "not enough shared memory for the raw ring");
    static_assert(SMEM <= SMEM_LIMIT, "shared memory over the limit");
};

__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t bits) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(bits));  // (a & mask) | bits
    return r;
}

// One GPTQ weight row for NW words of a k block (8 k values each): word i
// holds the codes of k = 8i .. 8i+7 (4 bits each, k order from the low bits),
// z the zero point and sh the fp16 scale of the row's group. Writes
// (q - z) * s as 4 NW columns of two 16-bit values. fp16: 1024 + q and 1024 + 16q come from the code bits
// by one mask-or each (exact), subtracting the zero point is exact, and the
// product with s is the only rounding.
template <int ACT, bool PERM, int NW = 8>
__device__ __forceinline__ void gptq_row(const uint32_t (&w)[NW], int z, __half sh, uint32_t (&o)[4 * NW]) {
    if (ACT == MOE_ACT_F16) {
        const __half2 s2 = __half2half2(sh);
        const __half2 z1 = __half2half2(__ushort_as_half(static_cast<unsigned short>(0x6400 | z)));      // 1024 + z
        const __half2 c16 = __half2half2(__ushort_as_half(static_cast<unsigned short>(0x2C00)));         // 1/16
        const __half2 nz16 = __half2half2(__ushort_as_half(static_cast<unsigned short>(0xD400 | (z << 4))));  // -(64 + z)
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            const uint32_t w8 = w[i] >> 8;
            uint32_t q[4] = {and_or(w[i], 0x000F000Fu, 0x64006400u),   // (k0, k4): 1024 + q
                             and_or(w[i], 0x00F000F0u, 0x64006400u),   // (k1, k5): 1024 + 16 q
                             and_or(w8, 0x000F000Fu, 0x64006400u),     // (k2, k6)
                             and_or(w8, 0x00F000F0u, 0x64006400u)};    // (k3, k7)
            uint32_t d[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __half2 h = *reinterpret_cast<__half2*>(&q[j]);
                const __half2 qz = (j & 1) ? __hfma2(h, c16, nz16) : __hsub2(h, z1);  // q - z, exact
                __half2 v = __hmul2(qz, s2);
                d[j] = *reinterpret_cast<uint32_t*>(&v);
            }
            if (PERM) {
                o[4 * i + 0] = d[0];
                o[4 * i + 1] = d[1];
                o[4 * i + 2] = d[2];
                o[4 * i + 3] = d[3];
            } else {
                o[4 * i + 0] = prmt(d[0], d[1], 0x5410);  // (k0, k1)
                o[4 * i + 1] = prmt(d[2], d[3], 0x5410);  // (k2, k3)
                o[4 * i + 2] = prmt(d[0], d[1], 0x7632);  // (k4, k5)
                o[4 * i + 3] = prmt(d[2], d[3], 0x7632);  // (k6, k7)
            }
        }
    } else {
        // bf16 activations: (q - z) * s is exact in f32 (a 5-bit integer times
        // an fp16 value) and rounds once to bf16
        const float s = __half2float(sh);
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = static_cast<float>(static_cast<int>((w[i] >> (4 * j)) & 15u) - z) * s;
            if (PERM) {
                o[4 * i + 0] = Act<ACT>::pack2(f[0], f[4]);
                o[4 * i + 1] = Act<ACT>::pack2(f[1], f[5]);
                o[4 * i + 2] = Act<ACT>::pack2(f[2], f[6]);
                o[4 * i + 3] = Act<ACT>::pack2(f[3], f[7]);
            } else {
                o[4 * i + 0] = Act<ACT>::pack2(f[0], f[1]);
                o[4 * i + 1] = Act<ACT>::pack2(f[2], f[3]);
                o[4 * i + 2] = Act<ACT>::pack2(f[4], f[5]);
                o[4 * i + 3] = Act<ACT>::pack2(f[6], f[7]);
            }
        }
    }
}

// One NVFP4 weight row for NW words of a k block: word i holds the E2M1 codes
// of k = 8i .. 8i+7 (low nibble first), sc[g] the E4M3 scale of k = 16g ..
// 16g+15. E2M1 x E4M3 products are exact in bf16 and fp16.
template <int ACT, int NW = 8>
__device__ __forceinline__ void nvfp4_row(const uint32_t (&w)[NW], const uint32_t (&sc)[NW / 2],
                                          uint32_t (&o)[4 * NW]) {
#pragma unroll
    for (int g = 0; g < NW / 2; ++g) {
        if (ACT == MOE_ACT_BF16) {
            const __nv_bfloat162 s2 = __float2bfloat162_rn(e4m3_to_f32(sc[g]));
#pragma unroll
            for (int ii = 0; ii < 2; ++ii) {
                const int i = 2 * g + ii;
                uint32_t a[4];
                e2m1x4_to_bf16x4(w[i], a[0], a[1]);
                e2m1x4_to_bf16x4(w[i] >> 16, a[2], a[3]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    __nv_bfloat162 v = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&a[j]), s2);
                    o[4 * i + j] = *reinterpret_cast<uint32_t*>(&v);
                }
            }
        } else {
            const __half2 s2 = __float2half2_rn(e4m3_to_f32(sc[g]));
#pragma unroll
            for (int ii = 0; ii < 2; ++ii) {
                const int i = 2 * g + ii;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t e2 = e2m1x2_to_f16x2((w[i] >> (8 * j)) & 0xffu);
                    __half2 v = __hmul2(*reinterpret_cast<__half2*>(&e2), s2);
                    o[4 * i + j] = *reinterpret_cast<uint32_t*>(&v);
                }
            }
        }
    }
}

// One FP8 weight row for a k block: word i holds the E4M3 codes of k = 4i ..
// 4i+3 (lowest byte first). Writes the codes' values unscaled (the row scale
// multiplies the f32 accumulator in the epilogue) as 32 columns of two 16-bit
// values: E4M3 -> f16 is one exact conversion per pair, and every E4M3 value
// is also exact in bf16 (4 significant bits, exponents 2^-9 .. 2^8).
template <int ACT>
__device__ __forceinline__ void fp8_row(const uint32_t (&w)[16], uint32_t (&o)[32]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        uint32_t lo, hi;  // (k 4i, 4i+1), (k 4i+2, 4i+3) as f16x2
        asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
            "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
            : "=r"(lo), "=r"(hi) : "r"(w[i]));
        if (ACT == MOE_ACT_F16) {
            o[2 * i] = lo;
            o[2 * i + 1] = hi;
        } else {
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
            o[2 * i] = Act<ACT>::pack2(a.x, a.y);
            o[2 * i + 1] = Act<ACT>::pack2(b.x, b.y);
        }
    }
}

// One weight row's raw bytes for a 64-deep k block, in registers: GPTQ 8
// words, the fp16 scale bits and the packed zero-point word; NVFP4 8 words and
// 4 scale bytes.
struct RawRow {
    uint32_t w[16];  // GPTQ / NVFP4: 8 words; FP8: 16 (one code byte per k)
    uint32_t s, z;
    uint32_t sc[4];
};

// A raw stage holds two k blocks (kp = 0, 1) of both 128-row halves:
//   GPTQ:  codes [16 packed k rows][2 halves][128 cols] int32 at 0, scales
//          [sg][2][128] fp16 at 16384, zeros [sg][2][16] int32 at 17408, where
//          sg = 2 group rows for group_size 64 and 1 otherwise;
//   NVFP4: codes [2 halves][128 rows][64 bytes] at 0, scales [8 k16 groups]
//          [2 halves][128 rows] E4M3 at 16384.
// An FP8 raw stage holds one k block: codes [2 halves][128 rows][64 bytes].
template <int WFMT>
__device__ __forceinline__ void load_raw_row(const uint8_t* raw, int h, int r, int kp, int g64, RawRow& x) {
    if (WFMT == MOE_W_FP8_E4M3) {
        const uint4* row = reinterpret_cast<const uint4*>(raw + h * 8192 + r * 64);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = row[i];
            x.w[4 * i] = v.x; x.w[4 * i + 1] = v.y; x.w[4 * i + 2] = v.z; x.w[4 * i + 3] = v.w;
        }
    } else if (WFMT == MOE_W_GPTQ_INT4) {
        const uint32_t* qw = reinterpret_cast<const uint32_t*>(raw);
#pragma unroll
        for (int i = 0; i < 8; ++i) x.w[i] = qw[((8 * kp + i) * 2 + h) * 128 + r];
        const int sg = g64 ? kp : 0;
        x.s = reinterpret_cast<const unsigned short*>(raw + 16384)[(sg * 2 + h) * 128 + r];
        x.z = reinterpret_cast<const uint32_t*>(raw + 17408)[(sg * 2 + h) * 16 + (r >> 3)];
    } else {
        const uint4* row = reinterpret_cast<const uint4*>(raw + h * 8192 + r * 64 + kp * 32);
        const uint4 v0 = row[0], v1 = row[1];
        x.w[0] = v0.x; x.w[1] = v0.y; x.w[2] = v0.z; x.w[3] = v0.w;
        x.w[4] = v1.x; x.w[5] = v1.y; x.w[6] = v1.z; x.w[7] = v1.w;
#pragma unroll
        for (int g = 0; g < 4; ++g) x.sc[g] = raw[16384 + ((4 * kp + g) * 2 + h) * 128 + r];
    }
}

template <int MODE, int WFMT, int ACT, int NTOK>
__global__ void __launch_bounds__(TsShape<MODE, WFMT, ACT, NTOK>::THREADS, 1)
grouped_gemm_ts_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmR0,
                       const __grid_constant__ CUtensorMap tmR1, const __grid_constant__ CUtensorMap tmR2,
                       const GemmParams p) {
    pdl_wait();
    using S = TsShape<MODE, WFMT, ACT, NTOK>;
    constexpr int XROWS = NTOK, XSTAGES = S::XSTAGES, ASTAGES = TS_STAGES, RSTAGES = S::RSTAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024_shared(smem_raw);
    uint8_t* sX = smem;
    uint8_t* sR = sX + XSTAGES * S::X_STAGE;
    uint8_t* sStg = sR + RSTAGES * RAW2;
    SmemTail& s = *reinterpret_cast<SmemTail*>(sStg + S::STG_BYTES);
    const WaitCtx wc{&s.abort_flag, p.err, p.wait_ns};

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int E = p.E;
    const int KB = (p.K + BK - 1) / BK;  // 64-deep k blocks (weight and activation stages)
    constexpr int KPR = WFMT == MOE_W_FP8_E4M3 ? 1 : 2;  // k blocks per raw stage
    const int KR = (KB + KPR - 1) / KPR;                   // raw stages per tile
    const int NSETS = KB < S::NR ? KB : S::NR;  // accumulator sets a tile uses
    // GPTQ group rows per raw stage: two for group_size 64, else one
    const int g64 = WFMT == MOE_W_GPTQ_INT4 && p.group_size == 64;

    const int bad = build_tile_list<XROWS>(s, p, S::OUT_COLS);
    if (tid == 0) {
        if (bad) set_err(p.err, MOE_DEV_ERR_OFFSETS);
#pragma unroll
        for (int i = 0; i < XSTAGES; ++i) {
            mbar_init(&s.full[i], 1);        // activation bytes
            mbar_init(&s.empty[i], S::NH);   // the issuers of the k block (one per half with NH = 2)
        }
#pragma unroll
        for (int i = 0; i < ASTAGES; ++i) {
            mbar_init(&s.afull[i], NUM_DQ_WARPS);  // every dequantising warp has written its rows
            mbar_init(&s.aempty[i], S::NH);
        }
#pragma unroll
        for (int i = 0; i < RSTAGES; ++i) {
            mbar_init(&s.raw_full[i], 1);
            mbar_init(&s.raw_empty[i], NUM_DQ_WARPS);  // the set that converts the stage
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.tfull[i], S::NH * NSETS);  // every issuer that had a k block of the tile
            mbar_init(&s.tempty[i], NUM_EPI_WARPS);
        }
        mbar_init(&s.mma_done, S::NI);
        fence_mbar_init();
    }
    __syncthreads();
    const int n_tiles = s.n_tiles;
    if (static_cast<int>(blockIdx.x) >= n_tiles) return;  // block-uniform: nothing allocated yet

    if (warp == 1) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&tmX);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: activations ----------------
            uint32_t stage = 0, phase = 0;
            long issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                const TileInfo t = decode_tile<XROWS>(s, E, tile, S::OUT_COLS);
                if (tile_is_padding(p, t)) continue;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1, wc)) { ok = false; break; }
                    mbar_arrive_expect_tx(&s.full[stage], S::X_STAGE);
                    tma_load_2d(sX + stage * S::X_STAGE, &tmX, kb * BK, t.m0, &s.full[stage]);
                    ++issued;
                    if (++stage == XSTAGES) { stage = 0; phase ^= 1; }
                }
            }
            const long first = issued > XSTAGES ? issued - XSTAGES : 0;
            for (long j = first; j < issued; ++j)
                mbar_drain(&s.full[j % XSTAGES], static_cast<uint32_t>((j / XSTAGES) & 1), kWaitLimitNs / 8);
        }
    } else if (warp < S::EPI0) {
        if (lane == 0) {
            // ---------------- MMA issuers: A = weights (TMEM), B = activations ----------------
            const int mi = warp - 1;
            const int hsel = S::NH == 2 ? (mi & 1) : -1;  // the half this issuer owns (-1: both)
            const int rset = mi / S::NH;                  // its k blocks: g = rset mod NR
            constexpr uint32_t idesc = f16_idesc(ACT, 128, NTOK);
            int g0 = 0;  // k blocks of this CTA's earlier tiles
            int local = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                const TileInfo t = decode_tile<XROWS>(s, E, tile, S::OUT_COLS);
                if (tile_is_padding(p, t)) continue;
                const int acc = S::NBUF == 2 ? (local & 1) : 0;
                const uint32_t aph = S::NBUF == 2 ? ((local >> 1) & 1) : (local & 1);
                ++local;
                const int first = (rset - g0 % S::NR + S::NR) % S::NR;  // its first kb in this tile
                if (first < KB) {
                    if (!mbar_wait(&s.tempty[acc], aph ^ 1, wc)) break;
                    tc_fence_after();
                    const uint32_t d = tmem_base + acc * S::ACC;
                    for (int kb = first; kb < KB; kb += S::NR) {
                        const int g = g0 + kb;
                        const int xs = g % XSTAGES, as = g % ASTAGES;
                        if (!mbar_wait(&s.full[xs], static_cast<uint32_t>((g / XSTAGES) & 1), wc) ||
                            !mbar_wait(&s.afull[as], static_cast<uint32_t>((g / ASTAGES) & 1), wc)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t xd = sw128_desc(smem_u32(sX + xs * S::X_STAGE));
                        const uint32_t a0 = tmem_base + TS_A_COL + as * 64;
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) {
                            const uint32_t en = kb > first || k > 0;
#pragma unroll
                            for (int h = 0; h < 2; ++h)
                                if (hsel < 0 || hsel == h)
                                    tc_mma_ts(d + (h * S::NR + rset) * NTOK, a0 + 32 * h + 8 * k, xd + 2 * k, idesc,
                                              en);
                        }
                        tc_commit(&s.empty[xs]);
                        tc_commit(&s.aempty[as]);
                    }
                    if (!ok) break;
                    tc_commit(&s.tfull[acc]);
                }
                g0 += KB;
            }
            tc_commit(&s.mma_done);
            mbar_drain(&s.mma_done, 0, kWaitLimitNs / 8);
        }
        __syncwarp();
    } else if (warp < S::DQ0) {
        // ---------------- epilogue: lane = weight row of a half, columns = tokens ----------------
        const int q = warp & 3;
        using T = typename Act<ACT>::T;
        T* out = static_cast<T*>(p.out);
        T* stg = reinterpret_cast<T*>(sStg) + (warp - S::EPI0) * (2 * 16 * 32);
        constexpr int HALVES = MODE == MODE_GATE_UP ? 1 : 2;
        int local = 0;
        int g0 = 0;  // k blocks of this CTA's earlier tiles: the tile's sets start at g0 mod NR
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
            const TileInfo t = decode_tile<XROWS>(s, E, tile, S::OUT_COLS);
            if (tile_is_padding(p, t)) continue;
            const int acc = S::NBUF == 2 ? (local & 1) : 0;
            const uint32_t aph = S::NBUF == 2 ? ((local >> 1) & 1) : (local & 1);
            ++local;
            // tile metadata first: its loads overlap the wait for the accumulator
            const int nvalid = valid_rows(p, s, t, lane);
            float s2a = 1.0f, s2b = 1.0f;
            if (WFMT == MOE_W_NVFP4) {
                s2a = __ldg(p.scale2 + t.e);
                s2b = (MODE == MODE_GATE_UP) ? __ldg(p.scale2 + p.E + t.e) : s2a;
            } else if (WFMT == MOE_W_FP8_E4M3) {
                // this lane's weight rows: half 0 row n, half 1 the up row I + n (gate/up)
                // or n + 128 (down); rows past the output are never stored
                const int n = t.n0 + q * 32 + lane;
                const float* rs = p.row_scale + static_cast<size_t>(t.e) * p.n_w;
                if (n < p.n_out) s2a = __ldg(rs + n);
                const int n1 = MODE == MODE_GATE_UP ? p.n_out + n : n + 128;
                if ((MODE == MODE_GATE_UP ? n : n + 128) < p.n_out) s2b = __ldg(rs + n1);
            }
            if (!mbar_wait(&s.tfull[acc], aph, wc)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * S::ACC;
            const int colw = t.n0 + q * 32;  // this warp's first column (half 0)
#pragma unroll 1
            for (int c = 0; c < NTOK && c < nvalid; c += 16) {
                float a[16], b[16];
                load_swapped<NTOK, S::NR>(taddr, c, a, b, NSETS, g0 % S::NR);
                // Through this warp's staging area ([half][token][32 columns]),
                // so that the chunk leaves as 16-byte stores of 8 columns.
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    if (MODE == MODE_GATE_UP) {
                        stg[j * 32 + lane] = Act<ACT>::from_f(silu_mul(a[j] * s2a, b[j] * s2b));
                    } else {
                        stg[j * 32 + lane] = Act<ACT>::from_f(a[j] * s2a);
                        stg[512 + j * 32 + lane] = Act<ACT>::from_f(b[j] * s2b);
                    }
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 2 * HALVES; ++i) {
                    const int pc = i * 32 + lane;  // [half][16 tokens][4 pieces of 8 columns]
                    const int hh = pc >> 6, row = (pc >> 2) & 15, pq = pc & 3;
                    const int col = colw + hh * 128 + pq * 8;
                    if (c + row < nvalid && col < p.n_out)
                        *reinterpret_cast<uint4*>(out + static_cast<size_t>(t.m0 + c + row) * p.n_out + col) =
                            *reinterpret_cast<const uint4*>(stg + hh * 512 + row * 32 + pq * 8);
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.tempty[acc]);
            g0 += KB;
        }
    } else if (warp < S::RAWW) {
        // ---------------- dequantising warps: raw shared bytes -> TMEM ----------------
        // The CTA's raw stages, counted j = 0, 1, ... over its tiles, go to the
        // sets in turn (set j mod NSET); a set converts all k blocks of a stage
        // (two for GPTQ and NVFP4, one for FP8), k block g into weight stage
        // g mod TS_STAGES. Each warp of the set owns 32 rows of one half: it
        // loads their raw bytes into registers, converts and stores each k
        // block, hands the raw stage back to TMA, then publishes the weight
        // stages. Ring positions are running counters (no division).
        static_assert(TS_STAGES == 4, "weight stage index is g & 3");
        const int dq = warp - S::DQ0;
        const int set = dq / NUM_DQ_WARPS;
        const int h = (dq >> 2) & 1;   // weight half
        const int sp = warp & 3;       // TMEM lane quarter this warp may access
        const int r = sp * 32 + lane;  // weight row within the half
        const uint32_t trow = tmem_base + (static_cast<uint32_t>(sp * 32) << 16) + TS_A_COL + h * 32;
        auto convert = [&](const RawRow& x, uint32_t (&o)[32]) {
            if (WFMT == MOE_W_GPTQ_INT4) {
                uint32_t w8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) w8[i] = x.w[i];
                gptq_row<ACT, S::PERM>(w8, (x.z >> (4 * (r & 7))) & 15,
                                       __ushort_as_half(static_cast<unsigned short>(x.s)), o);
            } else if (WFMT == MOE_W_NVFP4) {
                uint32_t w8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) w8[i] = x.w[i];
                nvfp4_row<ACT>(w8, x.sc, o);
            } else {
                fp8_row<ACT>(x.w, o);
            }
        };
        int rpos = set, rpar = 0;  // ring position and phase of this set's next raw stage
        int jmod = 0;              // (the CTA's next raw stage) mod NSET
        int g0 = 0;                // k blocks of this CTA's earlier tiles
        bool ok = true;
        for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
            if (tile_is_padding(p, decode_tile<XROWS>(s, E, tile, S::OUT_COLS))) continue;
            for (int kr = 0; kr < KR; ++kr) {
                const bool mine = jmod == set;
                if (++jmod == S::NSET) jmod = 0;
                if (!mine) continue;
                const int g = g0 + kr * KPR;
                const bool two = KPR == 2 && kr * KPR + 1 < KB;  // the stage's second k block is used
                if (!mbar_wait(&s.raw_full[rpos], static_cast<uint32_t>(rpar), wc)) { ok = false; break; }
                const uint8_t* raw = sR + rpos * RAW2;
                RawRow a, b;
                load_raw_row<WFMT>(raw, h, r, 0, g64, a);
                if (two) load_raw_row<WFMT>(raw, h, r, 1, g64, b);
                uint32_t o[32];
                convert(a, o);
                if (!mbar_wait(&s.aempty[g & 3], static_cast<uint32_t>(((g >> 2) & 1) ^ 1), wc)) { ok = false; break; }
                tc_fence_after();  // the MMAs that read this weight stage have completed
                tmem_st32(trow + (g & 3) * 64, o);
                if (two) {
                    convert(b, o);
                    const int g1 = g + 1;
                    if (!mbar_wait(&s.aempty[g1 & 3], static_cast<uint32_t>(((g1 >> 2) & 1) ^ 1), wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    tmem_st32(trow + (g1 & 3) * 64, o);
                }
                // the raw bytes were read through the generic proxy and the stage
                // is refilled by TMA (the async proxy): order the reads before
                // the release, or the next copy may land under them
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.raw_empty[rpos]);
                rpos += S::NSET;
                if (rpos >= RSTAGES) {
                    rpos -= RSTAGES;
                    rpar ^= 1;
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&s.afull[g & 3]);
                    if (two) mbar_arrive(&s.afull[(g + 1) & 3]);
                }
            }
            g0 += KB;
        }
        tmem_st_wait();  // nothing in flight into TMEM when it is freed
    } else {
        // ---------------- raw quantised-weight producer (last warp) ----------------
        // A TMA copy costs its issuing thread a roughly fixed time however
        // small it is, so a stage is fetched with as few copies as the layouts
        // allow: GPTQ codes + scales + zero points and NVFP4 codes + scales
        // for a 128-deep stage (two k blocks; for an odd number of k blocks
        // the second half of a tile's last stage is fetched but not used),
        // FP8 codes for a 64-deep one.
        if (lane == 0) {
            const uint32_t bytes = WFMT == MOE_W_GPTQ_INT4 ? 16384u + (g64 ? 2u : 1u) * 640u
                                   : WFMT == MOE_W_NVFP4   ? 18432u
                                                           : 16384u;
            uint32_t rstage = 0, rphase = 0;
            long issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                const TileInfo t = decode_tile<XROWS>(s, E, tile, S::OUT_COLS);
                if (tile_is_padding(p, t)) continue;
                for (int kr = 0; kr < KR; ++kr) {
                    if (!mbar_wait(&s.raw_empty[rstage], rphase ^ 1, wc)) { ok = false; break; }
                    uint64_t* bar = &s.raw_full[rstage];
                    uint8_t* rw = sR + rstage * RAW2;
                    mbar_arrive_expect_tx(bar, bytes);
                    if (WFMT == MOE_W_GPTQ_INT4) {
                        const int kq = t.e * (p.K / 8) + kr * 16;
                        const int g = t.e * (p.K / p.group_size) + (kr * 2 * BK) / p.group_size;
                        if (MODE == MODE_GATE_UP) {
                            tma_load_3d(rw, &tmR0, t.n0, 0, kq, bar);
                            tma_load_3d(rw + 16384, &tmR1, t.n0, 0, g, bar);
                            tma_load_3d(rw + 17408, &tmR2, t.n0 / 8, 0, g, bar);
                        } else {
                            tma_load_2d(rw, &tmR0, t.n0, kq, bar);
                            tma_load_2d(rw + 16384, &tmR1, t.n0, g, bar);
                            tma_load_2d(rw + 17408, &tmR2, t.n0 / 8, g, bar);
                        }
                    } else if (WFMT == MOE_W_FP8_E4M3) {
                        // one 64-deep k block of both halves: [2][128 rows][64 bytes]
                        if (MODE == MODE_GATE_UP)
                            tma_load_3d(rw, &tmR0, kr * BK, t.n0, 2 * t.e, bar);
                        else
                            tma_load_2d(rw, &tmR0, kr * BK, t.e * p.n_w + t.n0, bar);
                    } else {
                        const int sg = t.e * (p.K / 16) + kr * 8;
                        if (MODE == MODE_GATE_UP) {
                            tma_load_3d(rw, &tmR0, kr * BK, t.n0, 2 * t.e, bar);
                            tma_load_3d(rw + 16384, &tmR1, t.n0, 0, sg, bar);
                        } else {
                            tma_load_2d(rw, &tmR0, kr * BK, t.e * p.n_w + t.n0, bar);
                            tma_load_2d(rw + 16384, &tmR1, t.n0, sg, bar);
                        }
                    }
                    ++issued;
                    if (++rstage == RSTAGES) { rstage = 0; rphase ^= 1; }
                }
            }
            const long first = issued > RSTAGES ? issued - RSTAGES : 0;
            for (long j = first; j < issued; ++j)
                mbar_drain(&s.raw_full[j % RSTAGES], static_cast<uint32_t>((j / RSTAGES) & 1), kWaitLimitNs / 8);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// ---- gather of the activations into sorted-row order ---------------------------

// xs[r] = x[sorted_token_ids[r] / top_k] for r < expert_offsets[E]. Padding
// rows are left as they are: the GEMM epilogues never store a padding row,
// and a row of the MMA only feeds its own output row (or column). One warp
// per row, 16-byte vectors. With perm set, each group of 8 elements is stored
// in the order 0,4,1,5,2,6,3,7 (the k order of the GPTQ gate/up weights).
__device__ __forceinline__ uint4 perm8(uint4 v) {
    return make_uint4(prmt(v.x, v.z, 0x5410), prmt(v.x, v.z, 0x7632), prmt(v.y, v.w, 0x5410),
                      prmt(v.y, v.w, 0x7632));
}

__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ sorted_ids,
                   const int32_t* __restrict__ offsets, int E, int T, int top_k, int vec_per_row, int max_padded,
                   int perm, uint4* __restrict__ xs, int32_t* err) {
    pdl_wait();
    pdl_launch_next();
    const int total = min(__ldg(offsets + E), max_padded);
    const int P = T * top_k;
    for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < total; r += gridDim.x * 8) {
        const int pid = __ldg(sorted_ids + r);
        int tok = -1;
        if (pid >= 0 && pid < P) tok = pid / top_k;
        else if (pid != P && (threadIdx.x & 31) == 0) set_err(err, MOE_DEV_ERR_PAIR_ID);
        if (tok < 0) continue;
        uint4* dst = xs + static_cast<size_t>(r) * vec_per_row;
        const uint4* src = x + static_cast<size_t>(tok) * vec_per_row;
        if (perm)
            for (int v = threadIdx.x & 31; v < vec_per_row; v += 32) dst[v] = perm8(__ldg(src + v));
        else
            for (int v = threadIdx.x & 31; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
    }
}

// ---- host side -------------------------------------------------------------------

struct Maps {
    CUtensorMap x, w, w5, r0, r1, r2;  // w5: gate/up rows interleaved by 8 (bf16 pair form)
};

// Activation rows per tile. 0 selects the prefill form (128 rows as the MMA's
// M operand), used when experts average 128 or more rows. Otherwise the decode
// form takes one align block per tile (rounded up to a power of two, at least
// 16): spans are whole blocks and only a span's last block holds padding, so
// no tile is padding only and the tiles spread evenly over the CTAs.
int pick_ntok(long P, int E, int block_size) {
    const long touched = P < E ? P : E;
    const long avg = touched > 0 ? P / touched : 0;
    if (avg >= 128) return 0;
    int nt = 16;
    while (nt < block_size) nt <<= 1;
    return nt <= 128 ? nt : 0;
}

template <int MODE, int NTOK>
int launch_decode(const Maps& m, const GemmParams& p, cudaStream_t st, const char* who) {
    using S = DecodeShape<MODE, NTOK>;
    auto kernel = grouped_gemm_decode_kernel<MODE, NTOK>;
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        int rc = set_smem_limit(reinterpret_cast<const void*>(kernel), S::SMEM);
        if (rc != MOE_OK) return rc;
        configured_for = dev;
    }
    // tiles at most, times the pieces a tile may be cut into when tiles are fewer than SMs
    const int KB = (p.K + BK - 1) / BK;
    const long bound = static_cast<long>((p.max_padded + NTOK - 1) / NTOK + p.E) *
                       ((p.n_out + S::OUT_COLS - 1) / S::OUT_COLS) * (KB / SK_MIN_PIECE > 1 ? KB / SK_MIN_PIECE : 1);
    int sms = sm_count();
    if (sms <= 0) return fail(MOE_ERR_CUDA, "%s: cannot query the SM count", who);
    if (sms > SK_MAX_CTAS) sms = SK_MAX_CTAS;  // one split-K slice per CTA
    const int grid = static_cast<int>(bound < sms ? bound : sms);
    if (grid <= 0) return MOE_OK;
    if (!p.sk_part || !p.sk_flag) return fail(MOE_ERR_INVALID, "%s: no split-K area", who);
    // the stream-K unit arithmetic is 32-bit: region (< 2 grid tiles) x KB x grid
    if (2L * grid * KB * grid >= (1L << 31)) return fail(MOE_ERR_UNSUPPORTED, "%s: contraction too long", who);
    GemmParams q = p;
    q.pad_free = NTOK % p.block_size == 0;
    moe::launch_pdl(kernel, grid, S::THREADS, S::SMEM, st, m.x, m.w, q);
    count_launch();
    return check_launch(who);
}

// bf16 weights, fewer than 128 rows per touched expert: the decode form
template <int MODE>
int decode_by_ntok(int ntok, const Maps& m, const GemmParams& p, cudaStream_t st, const char* who) {
    switch (ntok) {
        case 16: return launch_decode<MODE, 16>(m, p, st, who);
        case 32: return launch_decode<MODE, 32>(m, p, st, who);
        case 64: return launch_decode<MODE, 64>(m, p, st, who);
        default: return launch_decode<MODE, 128>(m, p, st, who);
    }
}

template <int MODE, int WFMT, int ACT, int NTOK>
int launch_ts(const Maps& m, const GemmParams& p, cudaStream_t st, const char* who) {
    using S = TsShape<MODE, WFMT, ACT, NTOK>;
    auto kernel = grouped_gemm_ts_kernel<MODE, WFMT, ACT, NTOK>;
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        int rc = set_smem_limit(reinterpret_cast<const void*>(kernel), S::SMEM);
        if (rc != MOE_OK) return rc;
        configured_for = dev;
    }
    const long bound = static_cast<long>((p.max_padded + NTOK - 1) / NTOK + p.E) *
                       ((p.n_out + S::OUT_COLS - 1) / S::OUT_COLS);
    const int sms = sm_count();
    if (sms <= 0) return fail(MOE_ERR_CUDA, "%s: cannot query the SM count", who);
    const int grid = static_cast<int>(bound < sms ? bound : sms);
    if (grid <= 0) return MOE_OK;
    GemmParams q = p;
    q.pad_free = NTOK % p.block_size == 0;
    moe::launch_pdl(kernel, grid, S::THREADS, S::SMEM, st, m.x, m.r0, m.r1, m.r2, q);
    count_launch();
    return check_launch(who);
}

// quantised weights: the TS form, NTOK tokens per tile (128 for the prefill form)
template <int MODE, int WFMT, int ACT>
int ts_by_ntok(int ntok, const Maps& m, const GemmParams& p, cudaStream_t st, const char* who) {
    switch (ntok) {
        case 16: return launch_ts<MODE, WFMT, ACT, 16>(m, p, st, who);
        case 32: return launch_ts<MODE, WFMT, ACT, 32>(m, p, st, who);
        case 64: return launch_ts<MODE, WFMT, ACT, 64>(m, p, st, who);
        default: return launch_ts<MODE, WFMT, ACT, 128>(m, p, st, who);
    }
}

template <int MODE>
int launch_pair(const Maps& m, const GemmParams& p, cudaStream_t st, const char* who) {
    auto kernel = grouped_gemm_pair_kernel<MODE>;
    static int configured_for = -1;
    static int max_pairs = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = PAIR_SMEM;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (configured_for != dev) {
        int rc = set_smem_limit(reinterpret_cast<const void*>(kernel), PAIR_SMEM);
        if (rc != MOE_OK) return rc;
        const int sms = sm_count();
        cfg.gridDim = dim3(sms > 0 ? (sms / 2) * 2 : 2, 1, 1);
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
        if (e != cudaSuccess || n <= 0)
            return fail(MOE_ERR_CUDA, "%s: cannot place pairs of CTAs: %s", who, cudaGetErrorString(e));
        max_pairs = n;
        configured_for = dev;
    }
    constexpr int OUT_COLS = MODE == MODE_GATE_UP ? 128 : 256;
    // row tiles at most: ceil(valid / 256) per expert, so max_padded / 256 + E in all
    const long bound = static_cast<long>((p.max_padded + 255) / 256 + p.E) * ((p.n_out + OUT_COLS - 1) / OUT_COLS);
    const long pairs = bound < max_pairs ? bound : max_pairs;
    if (pairs <= 0) return MOE_OK;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    // programmatic dependent launch, as for every kernel of the library (launch_pdl)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, m.x, m.w, m.w5, p);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
    count_launch();
    return check_launch(who);
}

template <int MODE>
int dispatch(int wfmt, int act, int ntok, const Maps& m, const GemmParams& p, cudaStream_t st, const char* who) {
    if (wfmt == MOE_W_BF16) {
        if (ntok == 0) return launch_pair<MODE>(m, p, st, who);
        return decode_by_ntok<MODE>(ntok, m, p, st, who);
    }
    const int nt = ntok ? ntok : 128;  // prefill: 128-token tiles
    if (wfmt == MOE_W_GPTQ_INT4)
        return act == MOE_ACT_F16 ? ts_by_ntok<MODE, MOE_W_GPTQ_INT4, MOE_ACT_F16>(nt, m, p, st, who)
                                  : ts_by_ntok<MODE, MOE_W_GPTQ_INT4, MOE_ACT_BF16>(nt, m, p, st, who);
    if (wfmt == MOE_W_NVFP4)
        return act == MOE_ACT_F16 ? ts_by_ntok<MODE, MOE_W_NVFP4, MOE_ACT_F16>(nt, m, p, st, who)
                                  : ts_by_ntok<MODE, MOE_W_NVFP4, MOE_ACT_BF16>(nt, m, p, st, who);
    return act == MOE_ACT_F16 ? ts_by_ntok<MODE, MOE_W_FP8_E4M3, MOE_ACT_F16>(nt, m, p, st, who)
                              : ts_by_ntok<MODE, MOE_W_FP8_E4M3, MOE_ACT_BF16>(nt, m, p, st, who);
}

// Checks the weight descriptor and encodes its tensor maps. N = weight rows
// per expert, K = contraction, n_out = output columns (I for gate/up).
int weight_maps(const MoeWeight* w, int act, int E, int N, int K, int n_out, Maps& m, const char* who) {
    // TS form: tiles of 128 gate + 128 up (or 256 down) weight rows
    const uint32_t hc = 128, dc = 2 * hc;
    MOE_REQUIRE(w != nullptr, "%s: NULL weight descriptor", who);
    MOE_REQUIRE(act == MOE_ACT_BF16 || act == MOE_ACT_F16, "%s: unknown activation type %d", who, act);
    switch (w->format) {
        case MOE_W_BF16: {
            MOE_REQUIRE(act == MOE_ACT_BF16, "%s: a bf16 weight needs bf16 activations (the tensor cores take "
                                             "one 16-bit type for both operands)", who);
            MOE_REQUIRE(w->w != nullptr, "%s: NULL bf16 weight", who);
            int rc = make_tmap_2d(&m.w, w->w, static_cast<uint64_t>(E) * N, K, 128, act);
            if (rc != MOE_OK) return rc;
            m.w5 = m.w;
            if (N == 2 * n_out) {
                // gate/up rows as (k, 8 rows, gate | up, 8-row group, expert): one copy
                // brings 64 gate rows and the 64 up rows of the same columns, by 8
                const uint64_t I = static_cast<uint64_t>(n_out), row = static_cast<uint64_t>(K) * 2;
                const uint64_t d[5] = {static_cast<uint64_t>(K), 8, 2, I / 8, static_cast<uint64_t>(E)};
                const uint64_t st[4] = {row, I * row, 8 * row, 2 * I * row};
                const uint32_t b[5] = {64, 8, 2, 8, 1};
                rc = make_tmap_5d(&m.w5, w->w, act, d, st, b);
                if (rc != MOE_OK) return rc;
            }
            m.r0 = m.r1 = m.r2 = m.w;
            return MOE_OK;
        }
        case MOE_W_GPTQ_INT4: {
            MOE_REQUIRE(w->w && w->scales && w->zeros, "%s: GPTQ qweight / scales / qzeros must be non-NULL", who);
            const int G = w->group_size;
            MOE_REQUIRE(G >= 64 && G % 64 == 0 && K % G == 0,
                        "%s: GPTQ group_size=%d must be a multiple of 64 dividing K=%d", who, G, K);
            MOE_REQUIRE(n_out % 32 == 0, "%s: GPTQ needs %d output columns divisible by 32", who, n_out);
            // One copy per 128-deep raw stage fetches both 128-column halves of a
            // tile: for gate/up a 3-D map whose middle dimension steps from the
            // gate to the up columns (n_out apart), for down a 256-column box.
            // A stage spans one group row, or two for group_size 64.
            const uint64_t kq = static_cast<uint64_t>(E) * (K / 8), kg = static_cast<uint64_t>(E) * (K / G);
            const uint32_t sg = G == 64 ? 2 : 1;
            int rc;
            if (N == 2 * n_out) {
                const uint64_t I = n_out;
                rc = make_tmap_3d_raw(&m.r0, w->w, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, I, 2, kq, I * 4, 2 * I * 4, hc, 2,
                                      16);
                if (rc == MOE_OK)
                    rc = make_tmap_3d_raw(&m.r1, w->scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, I, 2, kg, I * 2,
                                          2 * I * 2, hc, 2, sg);
                if (rc == MOE_OK)
                    rc = make_tmap_3d_raw(&m.r2, w->zeros, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, I / 8, 2, kg, I / 8 * 4,
                                          2 * I / 8 * 4, hc / 8, 2, sg);
            } else {
                rc = make_tmap_2d_raw(&m.r0, w->w, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, kq, N, dc, 16);
                if (rc == MOE_OK)
                    rc = make_tmap_2d_raw(&m.r1, w->scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, kg, N, dc, sg);
                if (rc == MOE_OK)
                    rc = make_tmap_2d_raw(&m.r2, w->zeros, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, kg, N / 8, dc / 8, sg);
            }
            m.w = m.r0;
            return rc;
        }
        case MOE_W_NVFP4: {
            MOE_REQUIRE(w->w && w->scales && w->scale2, "%s: NVFP4 packed / scales / scale2 must be non-NULL", who);
            MOE_REQUIRE(K % 32 == 0, "%s: NVFP4 needs K=%d divisible by 32", who, K);
            MOE_REQUIRE(n_out % 16 == 0, "%s: NVFP4 needs %d output columns divisible by 16", who, n_out);
            // one copy per 128-deep raw stage for the packed codes and one for
            // the scales (3-D maps over the gate and up halves for gate/up,
            // 256-wide boxes for down)
            const uint64_t kg = static_cast<uint64_t>(E) * (K / 16);
            int rc;
            if (N == 2 * n_out) {
                const uint64_t I = n_out;
                rc = make_tmap_3d_raw(&m.r0, w->w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, I,
                                      2 * static_cast<uint64_t>(E), K / 2, I * (K / 2), 64, hc, 2);
                if (rc == MOE_OK)
                    rc = make_tmap_3d_raw(&m.r1, w->scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, I, 2, kg, I, 2 * I, hc,
                                          2, 8);
            } else {
                rc = make_tmap_2d_raw(&m.r0, w->w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, static_cast<uint64_t>(E) * N,
                                      K / 2, 64, dc);
                if (rc == MOE_OK) rc = make_tmap_2d_raw(&m.r1, w->scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kg, N, dc, 8);
            }
            m.r2 = m.r1;
            m.w = m.r0;
            return rc;
        }
        case MOE_W_FP8_E4M3: {
            MOE_REQUIRE(w->w && w->scales, "%s: FP8 codes / scales must be non-NULL", who);
            MOE_REQUIRE(K % 16 == 0, "%s: FP8 needs K=%d divisible by 16", who, K);
            // one copy per 64-deep raw stage: a 3-D map over the gate and up
            // halves for gate/up, a 256-row box for down
            int rc;
            if (N == 2 * n_out) {
                const uint64_t I = n_out;
                rc = make_tmap_3d_raw(&m.r0, w->w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, I, 2 * static_cast<uint64_t>(E),
                                      K, I * K, 64, hc, 2);
            } else {
                rc = make_tmap_2d_raw(&m.r0, w->w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, static_cast<uint64_t>(E) * N, K,
                                      64, dc);
            }
            m.r1 = m.r2 = m.r0;
            m.w = m.r0;
            return rc;
        }
        default:
            return fail(MOE_ERR_INVALID, "%s: unknown weight format %d", who, w->format);
    }
}

}  // namespace
}  // namespace moe

namespace moe {
namespace {
// the gathered activations, then the split-K area
size_t gather_bytes(int32_t max_padded, int32_t H) {
    return (static_cast<size_t>(max_padded) * H * 2 + 255) / 256 * 256;
}
void set_splitk(GemmParams& p, void* area) {
    p.sk_part = static_cast<float*>(area);
    p.sk_flag = reinterpret_cast<int*>(static_cast<uint8_t*>(area) + static_cast<size_t>(SK_MAX_CTAS) * SK_SLICE_FLOATS * 4);
}
}  // namespace
}  // namespace moe

extern "C" size_t moe_gate_up_workspace_size(int32_t max_padded, int32_t H) {
    if (max_padded < 0 || H < 0) return 0;
    return moe::gather_bytes(max_padded, H) + MOE_SPLITK_BYTES;
}

extern "C" size_t moe_down_workspace_size(void) { return MOE_SPLITK_BYTES; }

extern "C" int moe_grouped_gate_up(const void* x, int32_t act, const MoeWeight* w_gate_up,
                                   const int32_t* sorted_token_ids, const int32_t* expert_offsets, int32_t T,
                                   int32_t top_k, int32_t H, int32_t I, int32_t E, int32_t block_size,
                                   int32_t max_padded, void* h_out, int32_t* err_word, void* workspace,
                                   size_t workspace_bytes, void* stream) {
    const char* who = "moe_grouped_gate_up";
    MOE_REQUIRE(E >= 1 && E <= MOE_MAX_EXPERTS, "%s: E=%d outside [1, %d]", who, E, MOE_MAX_EXPERTS);
    MOE_REQUIRE(block_size >= 1, "%s: block_size=%d must be positive", who, block_size);
    MOE_REQUIRE(T >= 0 && top_k >= 1 && max_padded >= 0, "%s: bad T=%d / top_k=%d / max_padded=%d", who, T, top_k,
                max_padded);
    MOE_REQUIRE(H > 0 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", who, H);
    MOE_REQUIRE(I > 0 && I % 8 == 0, "%s: I=%d must be a positive multiple of 8", who, I);
    const long P = static_cast<long>(T) * top_k;
    const int ntok = moe::pick_ntok(P, E, block_size);
    moe::Maps m;
    int rc = moe::weight_maps(w_gate_up, act, E, 2 * I, H, I, m, who);
    if (rc != MOE_OK) return rc;
    if (max_padded == 0) return MOE_OK;
    MOE_REQUIRE(x && sorted_token_ids && expert_offsets && h_out, "%s: NULL pointer", who);
    MOE_REQUIRE(moe::aligned16(x) && moe::aligned16(h_out), "%s: x / h_out must be 16-byte aligned", who);
    const size_t need = moe_gate_up_workspace_size(max_padded, H);
    MOE_REQUIRE(workspace && workspace_bytes >= need && (reinterpret_cast<uintptr_t>(workspace) & 127) == 0,
                "%s: workspace of %zu bytes (128-byte aligned) required, got %zu", who, need, workspace_bytes);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // 1. gather activations into sorted-row order
    {
        const int sms = moe::sm_count();
        int blocks = (max_padded + 7) / 8;
        const int cap = sms > 0 ? sms * 8 : 1024;
        if (blocks > cap) blocks = cap;
        moe::launch_pdl(moe::gather_rows_kernel, blocks, 256, 0, st, static_cast<const uint4*>(x), sorted_token_ids,
                                                        expert_offsets, E, T, top_k, H / 8, max_padded,
                                                        w_gate_up->format == MOE_W_GPTQ_INT4 ? 1 : 0,
                                                        static_cast<uint4*>(workspace), err_word);
        moe::count_launch();
        rc = moe::check_launch("moe_grouped_gate_up (gather)");
        if (rc != MOE_OK) return rc;
    }
    // 2. the grouped GEMM
    rc = moe::make_tmap_2d(&m.x, workspace, max_padded, H, ntok ? ntok : 128, act);
    if (rc != MOE_OK) return rc;
    moe::GemmParams p{};
    p.offsets = expert_offsets;
    p.sorted_ids = sorted_token_ids;
    p.P = static_cast<int>(P);
    p.E = E;
    p.K = H;
    p.n_out = I;
    p.n_w = 2 * I;
    p.max_padded = max_padded;
    p.out = h_out;
    p.scale2 = w_gate_up->scale2;
    p.row_scale = static_cast<const float*>(w_gate_up->scales);
    p.group_size = w_gate_up->group_size;
    p.err = err_word;
    p.wait_ns = moe::wait_limit_ns();
    p.block_size = block_size;
    moe::set_splitk(p, static_cast<uint8_t*>(workspace) + moe::gather_bytes(max_padded, H));
    return moe::dispatch<moe::MODE_GATE_UP>(w_gate_up->format, act, ntok, m, p, st, who);
}

extern "C" int moe_grouped_down(const void* h, int32_t act, const MoeWeight* w_down, const int32_t* sorted_token_ids,
                                const int32_t* expert_offsets, int32_t T, int32_t top_k, int32_t H, int32_t I,
                                int32_t E, int32_t block_size, int32_t max_padded, void* y, int32_t* err_word,
                                void* workspace, size_t workspace_bytes, void* stream) {
    const char* who = "moe_grouped_down";
    MOE_REQUIRE(E >= 1 && E <= MOE_MAX_EXPERTS, "%s: E=%d outside [1, %d]", who, E, MOE_MAX_EXPERTS);
    MOE_REQUIRE(block_size >= 1, "%s: block_size=%d must be positive", who, block_size);
    MOE_REQUIRE(T >= 0 && top_k >= 1 && max_padded >= 0, "%s: bad T=%d / top_k=%d / max_padded=%d", who, T, top_k,
                max_padded);
    MOE_REQUIRE(I > 0 && I % 8 == 0, "%s: I=%d must be a positive multiple of 8", who, I);
    MOE_REQUIRE(H > 0 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", who, H);
    const long P = static_cast<long>(T) * top_k;
    const int ntok = moe::pick_ntok(P, E, block_size);
    moe::Maps m;
    int rc = moe::weight_maps(w_down, act, E, H, I, H, m, who);
    if (rc != MOE_OK) return rc;
    if (max_padded == 0) return MOE_OK;
    MOE_REQUIRE(h && sorted_token_ids && expert_offsets && y, "%s: NULL pointer", who);
    MOE_REQUIRE(moe::aligned16(h) && moe::aligned16(y), "%s: h / y must be 16-byte aligned", who);
    MOE_REQUIRE(workspace && workspace_bytes >= MOE_SPLITK_BYTES && (reinterpret_cast<uintptr_t>(workspace) & 127) == 0,
                "%s: workspace of %zu bytes (128-byte aligned) required, got %zu", who,
                static_cast<size_t>(MOE_SPLITK_BYTES), workspace_bytes);
    rc = moe::make_tmap_2d(&m.x, h, max_padded, I, ntok ? ntok : 128, act);
    if (rc != MOE_OK) return rc;
    moe::GemmParams p{};
    p.offsets = expert_offsets;
    p.sorted_ids = sorted_token_ids;
    p.P = static_cast<int>(P);
    p.E = E;
    p.K = I;
    p.n_out = H;
    p.n_w = H;
    p.max_padded = max_padded;
    p.out = y;
    p.scale2 = w_down->scale2;
    p.row_scale = static_cast<const float*>(w_down->scales);
    p.group_size = w_down->group_size;
    p.err = err_word;
    p.wait_ns = moe::wait_limit_ns();
    p.block_size = block_size;
    moe::set_splitk(p, workspace);
    return moe::dispatch<moe::MODE_DOWN>(w_down->format, act, ntok, m, p, static_cast<cudaStream_t>(stream), who);
}
