// Step a3 / a4, quantised-weight prefill form on CTA pairs: GPTQ int4, NVFP4
// or FP8 weights dequantised into TMEM by warps of both CTAs,
// tcgen05.mma.cta_group::2 with A from TMEM.
#include "gemm_common.cuh"
#include "gemm_dequant.cuh"

namespace moe {
namespace gemm {
namespace {

// ---- TS pair form ------------------------------------------------------------------
//
// The single-CTA TS form converts a 256-row weight tile per k block for at
// most 128 tokens, and at prefill that conversion (integer and permute
// instructions) sets its pace. Here a pair of SMs shares a tile of 256 weight
// rows and up to 192 (or 256) tokens of one expert: each CTA converts its own
// 128 rows into its own TMEM, and one thread of the leader issues M = 256 MMAs
// whose N is the tile's row count. Per token, each SM converts a quarter of
// what the single-CTA form converts for a 128-token tile and issues half as
// many MMAs; an expert's valid rows (up to the tile cap) are one tile instead
// of a 128-row tile and a mostly empty one.
//
// Rows of a CTA: gate/up takes 64 gate and the 64 up rows of the same output
// columns (n0 + 64 rank .. + 63), placed so that TMEM lane j of quarter q
// holds output column n0 + 64 rank + 16 q + 8 (j >> 4) + (j & 7), gate if
// (j & 8) == 0 else up (the bf16 pair form's layout); down takes output rows
// n0 + 128 rank + 32 q + j.
//
// TMEM of each CTA (512 columns), in one of two geometries (TspGeom): two
// accumulator buffers of up to 192 token columns (the epilogue drains one
// while the MMAs fill the other) and four weight stages of one 64-deep k block
// (32 columns: 64 16-bit values per lane), or one buffer of up to 256 columns
// and eight weight stages. The host takes the second when experts average
// 176 rows or more, so that experts of up to 256 rows stay one tile (measured:
// GPTQ T=2048, about 192 rows per expert, gate/up 231 -> 176 us; at 128-150
// rows the double buffer is 6-7% faster).
//
// Barriers: the activation ring is the pair kernel's (both CTAs' halves of a
// stage complete on the leader's barrier, the leader's commit frees it in
// both); each CTA has its own raw-weight ring; a weight stage is ready when
// the converting warps of both CTAs have arrived on the leader's barrier, and
// the leader's commit frees it in both.
template <int ACC_>
struct TspGeom {
    static constexpr int ACC = ACC_;                  // token columns of a buffer: the row-tile cap
    static constexpr int NBUF = ACC <= 192 ? 2 : 1;
    static constexpr int ASTAGES = ACC <= 192 ? 4 : 8;  // weight stages
    static constexpr int A_COL = NBUF * ACC;          // first TMEM column of the weight stages
    static constexpr int MAXU = ACC / 16;             // 16-row units per row tile
    static_assert(A_COL + ASTAGES * 32 <= 512, "weight stages exceed TMEM");
    static_assert(ASTAGES <= 8, "weight stage barriers");
};
constexpr int TSP_X_STAGE = 128 * BK * 2;  // this CTA's token rows of a k block (a 128-row box)
constexpr int TSP_NSET = 2;     // sets of four converting warps, taking the raw stages in turn
constexpr int TSP_STG = NUM_EPI_WARPS * 32 * 32 * 2;
constexpr int TSP_TAIL_BYTES = (static_cast<int>(sizeof(PairTail)) + 127) / 128 * 128;
constexpr int TSP_AVAIL = SMEM_LIMIT - 1024 - TSP_STG - TSP_TAIL_BYTES;
constexpr int TSP_XSTAGES = 8;
// warps: 0 activation TMA, 1 TMEM + MMA issuer, 2..5 epilogue, 6 raw TMA, 8..15 converting
constexpr int TSP_EPI0 = 2, TSP_RAWW = 6, TSP_DQ0 = 8;
constexpr int TSP_THREADS = 32 * (TSP_DQ0 + 4 * TSP_NSET);
static_assert(TSP_XSTAGES <= MAX_STAGES, "ring size");

// The raw-weight ring of a format. A raw stage holds this CTA's 128 rows of
//   GPTQ:  two k blocks, codes [16 packed k rows][128 columns] int32, fp16
//          scales [sg][128] at 8192 and zero points [sg][16] int32 at 8704
//          (sg = 2 group rows for group_size 64, else 1);
//   NVFP4: two k blocks, codes [128 rows][64 bytes] then scales [8 groups][128 rows];
//   FP8:   one k block, codes [128 rows][64 bytes] (row scales go to the epilogue).
// For gate/up the 128 are [gate | up][64] (one 3-D copy over both halves).
template <int WFMT>
struct TspRaw {
    static constexpr int KPR = WFMT == MOE_W_FP8_E4M3 ? 1 : 2;  // k blocks per raw stage
    static constexpr int BYTES = WFMT == MOE_W_FP8_E4M3 ? 8192 : (WFMT == MOE_W_GPTQ_INT4 ? 8832 : 9216);
    static constexpr int FIT = (TSP_AVAIL - TSP_XSTAGES * TSP_X_STAGE) / BYTES;
    static constexpr int STAGES = (FIT < MAX_RSTAGES ? FIT : MAX_RSTAGES) / TSP_NSET * TSP_NSET;
    static constexpr int SMEM = 1024 + TSP_XSTAGES * TSP_X_STAGE + STAGES * BYTES + TSP_STG + TSP_TAIL_BYTES;
    static_assert(STAGES >= 2 * TSP_NSET && STAGES <= MAX_RSTAGES, "raw ring size");
    static_assert(SMEM <= SMEM_LIMIT, "TS pair kernel shared memory over the limit");
};

// Epilogue of a TS pair tile for the calling warp (lanes 32q..32q+31 of this
// CTA's TMEM are its weight rows, columns the tile's tokens): the lane's
// weight scale (NVFP4: the per-tensor scale of the gate or up half; FP8: the
// row's scale; GPTQ: none, its scales are applied in the conversion) applied to
// every sum, then as the bf16 pair form: gate/up
// lanes j and j ^ 8 pair for SiLU(gate) * up; every 32-token step goes
// through the warp's staging area and leaves as 16-byte stores of 8 columns.
template <int MODE, int WFMT, int ACT>
__device__ __forceinline__ void tspair_epilogue(const GemmParams& p, uint32_t ta, typename Act<ACT>::T* stg,
                                                const PairTile& t, int rank, int q, int lane) {
    using A = Act<ACT>;
    using T = typename A::T;
    T* out = static_cast<T*>(p.out);
    const int nvalid = t.rows;
    float sc;
    if (WFMT == MOE_W_FP8_E4M3) {
        // this lane's weight row: gate/up column oc (gate row oc, up row n_out + oc), down row n
        const float* rs = p.row_scale + static_cast<size_t>(t.e) * p.n_w;
        if (MODE == MODE_GATE_UP) {
            const int oc = t.n0 + 64 * rank + 16 * q + 8 * (lane >> 4) + (lane & 7);
            sc = oc < p.n_out ? __ldg(rs + ((lane & 8) ? p.n_out + oc : oc)) : 0.0f;
        } else {
            const int n = t.n0 + 128 * rank + 32 * q + lane;
            sc = n < p.n_out ? __ldg(rs + n) : 0.0f;
        }
    } else if (WFMT == MOE_W_NVFP4) {
        sc = (MODE == MODE_GATE_UP && (lane & 8)) ? __ldg(p.scale2 + p.E + t.e) : __ldg(p.scale2 + t.e);
    } else {
        sc = 1.0f;
    }
    uint32_t u[32], nx[32];
    tmem_ld32(ta, nx);
#pragma unroll 1
    for (int c = 0; c < nvalid; c += 32) {
        tmem_ld_wait_regs(nx);
#pragma unroll
        for (int j = 0; j < 32; ++j) u[j] = nx[j];
        if (c + 32 < nvalid) tmem_ld32(ta + c + 32, nx);
        if (MODE == MODE_GATE_UP) {
            const bool gate = (lane & 8) == 0;
            const int cl = 8 * (lane >> 4) + (lane & 7);  // column within the warp's 16
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float lo = __uint_as_float(u[j]) * sc, hi = __uint_as_float(u[16 + j]) * sc;
                const float other = __shfl_xor_sync(0xffffffffu, gate ? hi : lo, 8);
                const float g = gate ? lo : other;
                const float up = gate ? other : hi;
                stg[(gate ? j : 16 + j) * 16 + cl] = A::from_f(silu_mul(g, up));
            }
            __syncwarp();
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
            for (int j = 0; j < 32; ++j) stg[j * 32 + lane] = A::from_f(__uint_as_float(u[j]) * sc);
            __syncwarp();
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

template <int MODE, int WFMT, int ACT, int ACCW>
__global__ void __launch_bounds__(TSP_THREADS, 1)
grouped_gemm_tspair_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmQ0,
                           const __grid_constant__ CUtensorMap tmQ1, const __grid_constant__ CUtensorMap tmQ2,
                           const GemmParams p) {
    pdl_wait();
    constexpr int OUT_COLS = MODE == MODE_GATE_UP ? 128 : 256;
    using R = TspRaw<WFMT>;
    using G = TspGeom<ACCW>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024_shared(smem_raw);
    uint8_t* sX = smem;
    uint8_t* sR = sX + TSP_XSTAGES * TSP_X_STAGE;
    uint8_t* sStg = sR + R::STAGES * R::BYTES;
    PairTail& s = *reinterpret_cast<PairTail*>(sStg + TSP_STG);
    const WaitCtx wc{&s.abort_flag, p.err, p.wait_ns};

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();  // 0: leader, 1: follower
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int E = p.E;
    const int KB = (p.K + BK - 1) / BK;  // 64-deep k blocks
    const int KR = (KB + R::KPR - 1) / R::KPR;  // raw stages per tile
    // GPTQ group rows per raw stage: two for group_size 64, else one
    const int g64 = WFMT == MOE_W_GPTQ_INT4 && p.group_size == 64;

    const int bad = build_pair_tiles<G::MAXU>(s, p, OUT_COLS);  // identical in both CTAs
    if (tid == 0) {
        if (bad && rank == 0) set_err(p.err, MOE_DEV_ERR_OFFSETS);
        for (int i = 0; i < TSP_XSTAGES; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < R::STAGES; ++i) {
            mbar_init(&s.raw_full[i], 1);
            mbar_init(&s.raw_empty[i], 4);  // the four warps of the set that converts the stage
        }
        for (int i = 0; i < G::ASTAGES; ++i) {
            mbar_init(&s.afull[i], 2 * 4);  // the converting warps of both CTAs (used in the leader)
            mbar_init(&s.aempty[i], 1);
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
        tma_prefetch_desc(&tmQ0);
        tma_prefetch_desc(&tmQ1);
        if (WFMT == MOE_W_GPTQ_INT4) tma_prefetch_desc(&tmQ2);
    }
    tc_fence_before();
    cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = s.tmem_base;
    const uint32_t leader_full0 = mapa_shared(smem_u32(&s.full[0]), 0);
    const uint32_t leader_afull0 = mapa_shared(smem_u32(&s.afull[0]), 0);
    const uint32_t leader_tempty0 = mapa_shared(smem_u32(&s.tempty[0]), 0);

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- activation TMA (both CTAs): this CTA's half of the tile's rows ----------------
            uint32_t stage = 0, phase = 0;
            long issued = 0;
            bool ok = true;
            for (int tile = pair; tile < n_tiles && ok; tile += npairs) {
                const PairTile t = pair_tile<G::MAXU>(s, E, tile, OUT_COLS);
                const int arow = t.m0 + static_cast<int>(rank) * (t.n16 / 2);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1, wc)) { ok = false; break; }
                    if (rank == 0) mbar_arrive_expect_tx(&s.full[stage], 2 * TSP_X_STAGE);
                    tma_load_2d_pair(sX + stage * TSP_X_STAGE, &tmX, kb * BK, arow, leader_full0 + stage * 8);
                    ++issued;
                    if (++stage == TSP_XSTAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (rank == 0) {  // let every copy of the pair land before either CTA may exit
                const long first = issued > TSP_XSTAGES ? issued - TSP_XSTAGES : 0;
                for (long j = first; j < issued; ++j)
                    mbar_drain(&s.full[j % TSP_XSTAGES], static_cast<uint32_t>((j / TSP_XSTAGES) & 1),
                               kWaitLimitNs / 8);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer (leader): D = weight rows x tile rows ----------------
            int g = 0;  // the CTA's k blocks so far (activation ring index and weight stage index)
            int local = 0;
            bool ok = true;
            for (int tile = pair; tile < n_tiles && ok; tile += npairs) {
                const PairTile t = pair_tile<G::MAXU>(s, E, tile, OUT_COLS);
                const int acc = G::NBUF == 2 ? (local & 1) : 0;
                const uint32_t aph = G::NBUF == 2 ? ((local >> 1) & 1) : (local & 1);
                ++local;
                if (!mbar_wait(&s.tempty[acc], aph ^ 1, wc)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + acc * G::ACC;
                const uint32_t idesc = f16_idesc(ACT, 256, t.n16);
                for (int kb = 0; kb < KB; ++kb, ++g) {
                    const int xs = g % TSP_XSTAGES, as = g % G::ASTAGES;
                    if (!mbar_wait(&s.full[xs], static_cast<uint32_t>((g / TSP_XSTAGES) & 1), wc) ||
                        !mbar_wait(&s.afull[as], static_cast<uint32_t>((g / G::ASTAGES) & 1), wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t xd = sw128_desc(smem_u32(sX + xs * TSP_X_STAGE));
                    const uint32_t a0 = tmem_base + G::A_COL + 32 * as;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) tc_mma_pair_ts(d, a0 + 8 * k, xd + 2 * k, idesc, (kb | k) != 0);
                    tc_commit_pair(&s.empty[xs], 0x3);
                    tc_commit_pair(&s.aempty[as], 0x3);
                }
                if (!ok) break;
                tc_commit_pair(&s.tfull[acc], 0x3);
            }
            tc_commit_pair(&s.mma_done, 0x1);
            mbar_drain(&s.mma_done, 0, kWaitLimitNs / 8);
        }
        __syncwarp();
    } else if (warp < TSP_EPI0 + NUM_EPI_WARPS) {
        // ---------------- epilogue (both CTAs): lane = weight row, columns = tile rows ----------------
        const int q = warp & 3;
        using T = typename Act<ACT>::T;
        T* stg = reinterpret_cast<T*>(sStg) + (warp - TSP_EPI0) * (32 * 32);
        int local = 0;
        for (int tile = pair; tile < n_tiles; tile += npairs) {
            const PairTile t = pair_tile<G::MAXU>(s, E, tile, OUT_COLS);
            const int acc = G::NBUF == 2 ? (local & 1) : 0;
            const uint32_t aph = G::NBUF == 2 ? ((local >> 1) & 1) : (local & 1);
            ++local;
            if (!mbar_wait(&s.tfull[acc], aph, wc)) break;
            tc_fence_after();
            const uint32_t ta = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * G::ACC;
            tspair_epilogue<MODE, WFMT, ACT>(p, ta, stg, t, static_cast<int>(rank), q, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0) mbar_arrive(&s.tempty[acc]);
                else mbar_arrive_cluster(leader_tempty0 + acc * 8);
            }
        }
    } else if (warp == TSP_RAWW) {
        // ---------------- raw-weight TMA (each CTA its own 128 rows) ----------------
        if (lane == 0) {
            uint32_t rstage = 0, rphase = 0;
            long issued = 0;
            bool ok = true;
            for (int tile = pair; tile < n_tiles && ok; tile += npairs) {
                const PairTile t = pair_tile<G::MAXU>(s, E, tile, OUT_COLS);
                for (int kr = 0; kr < KR; ++kr) {
                    if (!mbar_wait(&s.raw_empty[rstage], rphase ^ 1, wc)) { ok = false; break; }
                    uint64_t* bar = &s.raw_full[rstage];
                    uint8_t* rw = sR + rstage * R::BYTES;
                    const int sg = t.e * (p.K / 16) + kr * 8;  // NVFP4: the stage's first 16-deep scale group
                    if (WFMT == MOE_W_GPTQ_INT4) {
                        // codes: the stage's 16 packed k rows; scales / zero points: its group rows
                        mbar_arrive_expect_tx(bar, 8192u + (g64 ? 2u : 1u) * 320u);
                        const int kq = t.e * (p.K / 8) + kr * 16;
                        const int gr = t.e * (p.K / p.group_size) + (kr * 2 * BK) / p.group_size;
                        if (MODE == MODE_GATE_UP) {
                            const int c0 = t.n0 + 64 * static_cast<int>(rank);
                            tma_load_3d(rw, &tmQ0, c0, 0, kq, bar);
                            tma_load_3d(rw + 8192, &tmQ1, c0, 0, gr, bar);
                            tma_load_3d(rw + 8704, &tmQ2, c0 / 8, 0, gr, bar);
                        } else {
                            const int c0 = t.n0 + 128 * static_cast<int>(rank);
                            tma_load_2d(rw, &tmQ0, c0, kq, bar);
                            tma_load_2d(rw + 8192, &tmQ1, c0, gr, bar);
                            tma_load_2d(rw + 8704, &tmQ2, c0 / 8, gr, bar);
                        }
                    } else if (WFMT == MOE_W_FP8_E4M3) {
                        mbar_arrive_expect_tx(bar, R::BYTES);
                        // codes [gate | up][64 rows][64 bytes] or [128 rows][64 bytes]
                        if (MODE == MODE_GATE_UP)
                            tma_load_3d(rw, &tmQ0, kr * BK, t.n0 + 64 * static_cast<int>(rank), 2 * t.e, bar);
                        else
                            tma_load_2d(rw, &tmQ0, kr * BK, t.e * p.n_w + t.n0 + 128 * static_cast<int>(rank), bar);
                    } else if (MODE == MODE_GATE_UP) {
                        mbar_arrive_expect_tx(bar, R::BYTES);
                        // codes [gate | up][64 rows][64 bytes], scales [8 groups][gate | up][64 rows]
                        const int r0 = t.n0 + 64 * static_cast<int>(rank);
                        tma_load_3d(rw, &tmQ0, kr * BK, r0, 2 * t.e, bar);
                        tma_load_3d(rw + 8192, &tmQ1, r0, 0, sg, bar);
                    } else {
                        mbar_arrive_expect_tx(bar, R::BYTES);
                        // codes [128 rows][64 bytes], scales [8 groups][128 rows]
                        const int r0 = t.n0 + 128 * static_cast<int>(rank);
                        tma_load_2d(rw, &tmQ0, kr * BK, t.e * p.n_w + r0, bar);
                        tma_load_2d(rw + 8192, &tmQ1, r0, sg, bar);
                    }
                    ++issued;
                    if (++rstage == R::STAGES) { rstage = 0; rphase ^= 1; }
                }
            }
            const long first = issued > R::STAGES ? issued - R::STAGES : 0;
            for (long j = first; j < issued; ++j)
                mbar_drain(&s.raw_full[j % R::STAGES], static_cast<uint32_t>((j / R::STAGES) & 1),
                           kWaitLimitNs / 8);
        }
    } else if (warp >= TSP_DQ0) {
        // ---------------- converting warps: raw shared bytes -> this CTA's TMEM ----------------
        // The CTA's raw stages, counted j = 0, 1, ... over its tiles, go to the
        // sets in turn; a set converts both k blocks of a stage (k block g into
        // weight stage g mod G::ASTAGES). Warp sp of a set owns TMEM lanes 32 sp .. + 31.
        const int set = (warp - TSP_DQ0) >> 2;
        const int sp = warp & 3;
        // this lane's row of the raw stage: gate/up [gate | up][64], down [128]
        const int ri = MODE == MODE_GATE_UP ? 64 * ((lane >> 3) & 1) + 16 * sp + 8 * (lane >> 4) + (lane & 7)
                                            : 32 * sp + lane;
        const uint32_t trow = tmem_base + (static_cast<uint32_t>(sp * 32) << 16) + G::A_COL;
        auto convert = [&](const uint8_t* raw, int kp, uint32_t (&o)[32]) {
            if (WFMT == MOE_W_GPTQ_INT4) {
                // this lane's column (weight row) ri: 8 words of the k block's 8 packed
                // k rows, its group row's fp16 scale and packed zero point
                const uint32_t* qw = reinterpret_cast<const uint32_t*>(raw);
                uint32_t w8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) w8[i] = qw[(8 * kp + i) * 128 + ri];
                const int gs = g64 ? kp : 0;
                const unsigned short sh = reinterpret_cast<const unsigned short*>(raw + 8192)[gs * 128 + ri];
                const uint32_t zw = reinterpret_cast<const uint32_t*>(raw + 8704)[gs * 16 + (ri >> 3)];
                gptq_row<ACT, MODE == MODE_GATE_UP>(w8, (zw >> (4 * (ri & 7))) & 15, __ushort_as_half(sh), o);
            } else if (WFMT == MOE_W_FP8_E4M3) {
                uint32_t w16[16];
                const uint4* row = reinterpret_cast<const uint4*>(raw + ri * 64);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 v = row[i];
                    w16[4 * i] = v.x; w16[4 * i + 1] = v.y; w16[4 * i + 2] = v.z; w16[4 * i + 3] = v.w;
                }
                fp8_row<ACT>(w16, o);
            } else {
                uint32_t w8[8], sc[4];
                const uint4* row = reinterpret_cast<const uint4*>(raw + ri * 64 + kp * 32);
                const uint4 v0 = row[0], v1 = row[1];
                w8[0] = v0.x; w8[1] = v0.y; w8[2] = v0.z; w8[3] = v0.w;
                w8[4] = v1.x; w8[5] = v1.y; w8[6] = v1.z; w8[7] = v1.w;
#pragma unroll
                for (int g4 = 0; g4 < 4; ++g4) sc[g4] = raw[8192 + (4 * kp + g4) * 128 + ri];
                nvfp4_row<ACT>(w8, sc, o);
            }
        };
        int rpos = set, rpar = 0;  // ring position and phase of this set's next raw stage
        int jmod = 0;              // (the CTA's next raw stage) mod TSP_NSET
        int g0 = 0;                // k blocks of this CTA's earlier tiles
        bool ok = true;
        for (int tile = pair; tile < n_tiles && ok; tile += npairs) {
            for (int kr = 0; kr < KR; ++kr) {
                const bool mine = jmod == set;
                if (++jmod == TSP_NSET) jmod = 0;
                if (!mine) continue;
                const int g = g0 + R::KPR * kr;
                const bool two = R::KPR == 2 && 2 * kr + 1 < KB;  // the stage's second k block is used
                if (!mbar_wait(&s.raw_full[rpos], static_cast<uint32_t>(rpar), wc)) { ok = false; break; }
                const uint8_t* raw = sR + rpos * R::BYTES;
                // each k block is published as soon as it is in TMEM, before the next one
                // is converted: the MMA of k block g waits on it, and the conversion of
                // g + G::ASTAGES waits on that MMA
                // (the follower's arrival on the leader's barrier is relaxed: the TMEM
                // writes are complete once tcgen05.wait::st returns, and the leader's MMA
                // cannot issue before it sees the arrival)
                auto publish = [&](int gb) {
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (rank == 0) mbar_arrive(&s.afull[gb % G::ASTAGES]);
                        else mbar_arrive_cluster_relaxed(leader_afull0 + (gb % G::ASTAGES) * 8);
                    }
                };
                uint32_t o[32];
                convert(raw, 0, o);
                if (!mbar_wait(&s.aempty[g % G::ASTAGES], static_cast<uint32_t>(((g / G::ASTAGES) & 1) ^ 1), wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();  // the MMAs that read this weight stage have completed
                tmem_st32(trow + (g % G::ASTAGES) * 32, o);
                publish(g);
                if (two) {
                    convert(raw, 1, o);
                    const int g1 = g + 1;
                    if (!mbar_wait(&s.aempty[g1 % G::ASTAGES], static_cast<uint32_t>(((g1 / G::ASTAGES) & 1) ^ 1),
                                   wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    tmem_st32(trow + (g1 % G::ASTAGES) * 32, o);
                }
                // the raw bytes were read through the generic proxy and the stage is
                // refilled by TMA (the async proxy): order the reads before the release
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.raw_empty[rpos]);
                rpos += TSP_NSET;
                if (rpos >= R::STAGES) {
                    rpos -= R::STAGES;
                    rpar ^= 1;
                }
                if (two) publish(g + 1);
            }
            g0 += KB;
        }
        tmem_st_wait();  // nothing in flight into TMEM when it is freed
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the leader's MMAs read this CTA's shared memory and TMEM and write its TMEM
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, 512);
}

template <int MODE, int WFMT, int ACT, int ACCW>
int launch_tspair(const Maps& m, const GemmParams& p, cudaStream_t st, const char* who) {
    using R = TspRaw<WFMT>;
    using G = TspGeom<ACCW>;
    auto kernel = grouped_gemm_tspair_kernel<MODE, WFMT, ACT, ACCW>;
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
    cfg.blockDim = dim3(TSP_THREADS, 1, 1);
    cfg.dynamicSmemBytes = R::SMEM;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (configured_for != dev) {
        int rc = set_smem_limit(reinterpret_cast<const void*>(kernel), R::SMEM);
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
    // row tiles at most: ceil(valid / ACC) per expert, so max_padded / ACC + E in all
    const long bound = static_cast<long>((p.max_padded + G::ACC - 1) / G::ACC + p.E) *
                       ((p.n_out + OUT_COLS - 1) / OUT_COLS);
    const long pairs = bound < max_pairs ? bound : max_pairs;
    if (pairs <= 0) return MOE_OK;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, m.x, m.q0, m.q1, m.q2, p);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: launch failed: %s", who, cudaGetErrorString(e));
    count_launch();
    return check_launch(who);
}

}  // namespace

int launch_tspair_form(int mode, int wfmt, int act, int wide, const Maps& m, const GemmParams& p, cudaStream_t st,
                       const char* who) {
#define MOE_TSP_ACT(MODE, WFMT)                                                                              \
    do {                                                                                                     \
        if (wide)                                                                                            \
            return act == MOE_ACT_F16 ? launch_tspair<MODE, WFMT, MOE_ACT_F16, 256>(m, p, st, who)           \
                                      : launch_tspair<MODE, WFMT, MOE_ACT_BF16, 256>(m, p, st, who);         \
        return act == MOE_ACT_F16 ? launch_tspair<MODE, WFMT, MOE_ACT_F16, 192>(m, p, st, who)               \
                                  : launch_tspair<MODE, WFMT, MOE_ACT_BF16, 192>(m, p, st, who);             \
    } while (0)
    if (mode == MODE_GATE_UP) {
        if (wfmt == MOE_W_GPTQ_INT4) MOE_TSP_ACT(MODE_GATE_UP, MOE_W_GPTQ_INT4);
        if (wfmt == MOE_W_FP8_E4M3) MOE_TSP_ACT(MODE_GATE_UP, MOE_W_FP8_E4M3);
        MOE_TSP_ACT(MODE_GATE_UP, MOE_W_NVFP4);
    }
    if (wfmt == MOE_W_GPTQ_INT4) MOE_TSP_ACT(MODE_DOWN, MOE_W_GPTQ_INT4);
    if (wfmt == MOE_W_FP8_E4M3) MOE_TSP_ACT(MODE_DOWN, MOE_W_FP8_E4M3);
    MOE_TSP_ACT(MODE_DOWN, MOE_W_NVFP4);
#undef MOE_TSP_ACT
}

}  // namespace gemm
}  // namespace moe
