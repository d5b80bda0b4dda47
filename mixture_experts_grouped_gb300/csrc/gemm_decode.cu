// Step a3 / a4, bf16 decode form: grouped expert GEMMs with the operands
// swapped (weights are the MMA's M operand, one align block of tokens its N)
// and a stream-K cut of thin last waves.
#include "gemm_common.cuh"

namespace moe {
namespace gemm {
namespace {

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
// leaves its fp32 sums in this CTA's slice of the split-K area and sets the
// CTA's flag for q to the call's generation (p.sk_gen, nonzero, new for every
// call); the owner waits until the flags of CTAs blockIdx.x + 1 .. last_peer
// hold that generation, adds their slices to its own sums, stores the chunk
// and sets the flags back to 0. A flag or slice left by an earlier call (one
// that gave up, say) is never taken for this call's piece. Returns false
// when a wait gave up.
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
        if (lane == 0) st_release_gpu(p.sk_flag + blockIdx.x * 4 + q, p.sk_gen);
        return true;
    }
    // owner: wait for the peers, fetch the first peer's first chunk while this
    // CTA's own MMAs may still run
    const int first_peer = blockIdx.x + 1;
    for (int pc = first_peer; pc <= last_peer; ++pc)
        if (!flag_wait(p.sk_flag + pc * 4 + q, p.sk_gen, wc)) return false;
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

}  // namespace

int launch_decode_form(int mode, int ntok, const Maps& m, const GemmParams& p, cudaStream_t st, const char* who) {
    return mode == MODE_GATE_UP ? decode_by_ntok<MODE_GATE_UP>(ntok, m, p, st, who)
                                : decode_by_ntok<MODE_DOWN>(ntok, m, p, st, who);
}

}  // namespace gemm
}  // namespace moe
