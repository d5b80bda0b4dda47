// Step a3 / a4 for quantised weights (GPTQ int4, NVFP4, FP8) at decode sizes:
// the TS form, weights dequantised by warps of the CTA into TMEM as the MMA's
// A operand (prefill runs the CTA-pair form of gemm_tspair.cu).
#include "gemm_common.cuh"
#include "gemm_dequant.cuh"

namespace moe {
namespace gemm {
namespace {

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
    // GPTQ and NVFP4 decode layers; one set stays for FP8 (its conversion is
    // short: two sets measured 4% slower) and for GPTQ at 128 tokens per tile
    // (2% slower when this form also ran GPTQ prefill).
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

// quantised weights at decode: the TS form, NTOK tokens (one align block) per tile
template <int MODE, int WFMT, int ACT>
int ts_by_ntok(int ntok, const Maps& m, const GemmParams& p, cudaStream_t st, const char* who) {
    switch (ntok) {
        case 16: return launch_ts<MODE, WFMT, ACT, 16>(m, p, st, who);
        case 32: return launch_ts<MODE, WFMT, ACT, 32>(m, p, st, who);
        case 64: return launch_ts<MODE, WFMT, ACT, 64>(m, p, st, who);
        default: return launch_ts<MODE, WFMT, ACT, 128>(m, p, st, who);
    }
}

}  // namespace

int launch_ts_form(int mode, int wfmt, int act, int ntok, const Maps& m, const GemmParams& p, cudaStream_t st,
                   const char* who) {
    const int nt = ntok ? ntok : 128;  // (prefill, ntok 0, takes the TS pair form instead)
#define MOE_TS_FMT(MODE)                                                                                     \
    do {                                                                                                     \
        if (wfmt == MOE_W_GPTQ_INT4)                                                                         \
            return act == MOE_ACT_F16 ? ts_by_ntok<MODE, MOE_W_GPTQ_INT4, MOE_ACT_F16>(nt, m, p, st, who)     \
                                      : ts_by_ntok<MODE, MOE_W_GPTQ_INT4, MOE_ACT_BF16>(nt, m, p, st, who);   \
        if (wfmt == MOE_W_NVFP4)                                                                             \
            return act == MOE_ACT_F16 ? ts_by_ntok<MODE, MOE_W_NVFP4, MOE_ACT_F16>(nt, m, p, st, who)         \
                                      : ts_by_ntok<MODE, MOE_W_NVFP4, MOE_ACT_BF16>(nt, m, p, st, who);       \
        return act == MOE_ACT_F16 ? ts_by_ntok<MODE, MOE_W_FP8_E4M3, MOE_ACT_F16>(nt, m, p, st, who)          \
                                  : ts_by_ntok<MODE, MOE_W_FP8_E4M3, MOE_ACT_BF16>(nt, m, p, st, who);        \
    } while (0)
    if (mode == MODE_GATE_UP) MOE_TS_FMT(MODE_GATE_UP);
    MOE_TS_FMT(MODE_DOWN);
#undef MOE_TS_FMT
}

}  // namespace gemm
}  // namespace moe
