// Step a3 / a4, bf16 prefill form: grouped expert GEMMs on CTA pairs
// (tcgen05.mma.cta_group::2).
#include "gemm_common.cuh"

namespace moe {
namespace gemm {
namespace {

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

    const int bad = build_pair_tiles<16>(s, p, OUT_COLS);  // identical in both CTAs
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
                const PairTile t = pair_tile<16>(s, E, tile, OUT_COLS);
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
                const PairTile t = pair_tile<16>(s, E, tile, OUT_COLS);
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
            const PairTile t = pair_tile<16>(s, E, tile, OUT_COLS);
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

}  // namespace

int launch_pair_form(int mode, const Maps& m, const GemmParams& p, cudaStream_t st, const char* who) {
    return mode == MODE_GATE_UP ? launch_pair<MODE_GATE_UP>(m, p, st, who) : launch_pair<MODE_DOWN>(m, p, st, who);
}

}  // namespace gemm
}  // namespace moe
