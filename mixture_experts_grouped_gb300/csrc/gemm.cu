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
//   * one persistent CTA per SM walks a static tile list; the list is built on
//     the device from expert_offsets (per expert ceil(span / 128) row tiles x
//     the column tiles), so there is no host synchronisation and the launch
//     shape only depends on host-known sizes;
//   * tile = 128 rows x 256 accumulator columns, K in steps of 64 (one
//     128-byte swizzle span). Gate/up puts 128 gate and 128 up weight rows in
//     one 256-row B tile, so each tcgen05.mma (M=128, N=256, K=16) produces
//     both halves of 128 output columns and the epilogue can fuse silu*up;
//   * warp 0 issues TMA loads into a 4-stage ring, one thread of warp 1 issues
//     tcgen05.mma into one of two TMEM accumulators (2 x 256 columns), warps
//     2-5 drain the other accumulator (tcgen05.ld -> activation -> global);
//   * quantised weights (GPTQ int4, NVFP4) are dequantised by warps 6-9
//     straight into the swizzled shared-memory B tile; activations still come
//     by TMA. The NVFP4 global scale2 is applied to the f32 accumulator;
//   * every mbarrier wait is bounded; on a timeout the CTA records
//     MOE_DEV_ERR_TIMEOUT, lets in-flight copies and MMAs land, frees TMEM and
//     returns.
#include "common.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN = 256;  // MMA N
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;  // 16 KB
constexpr int B_STAGE = BN * BK * 2;  // 32 KB
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 512;
constexpr int NUM_EPI_WARPS = 4;
constexpr int NUM_DQ_WARPS = 4;

enum { MODE_GATE_UP = 0, MODE_DOWN = 1 };

struct GemmParams {
    const int32_t* offsets;  // [E + 1]
    int E;
    int K;          // contraction length
    int n_out;      // output columns: I (gate/up) or H (down)
    int n_w;        // weight rows per expert: 2I or H
    int max_padded;
    void* out;      // [max_padded, n_out]
    const void* qw; // quantised weight payload
    const void* qs; // scales
    const void* qz; // GPTQ zeros
    const float* scale2;
    int group_size;
    int32_t* err;
};

struct SmemTail {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
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

constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) + static_cast<int>(sizeof(SmemTail)) + 1024;

template <int MODE>
__host__ __device__ constexpr int out_cols_per_tile() {
    return MODE == MODE_GATE_UP ? 128 : 256;
}

struct TileInfo {
    int e, m0, n0, rows;
};

__device__ __forceinline__ TileInfo decode_tile(const SmemTail& s, int E, int tile, int cols_per_tile) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.tstart[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    TileInfo t;
    t.e = lo;
    const int span = s.off[lo + 1] - s.off[lo];
    const int mt = (span + BM - 1) / BM;
    const int local = tile - s.tstart[lo];
    const int n_tile = local / mt;
    const int m_tile = local - n_tile * mt;
    t.m0 = s.off[lo] + m_tile * BM;
    t.n0 = n_tile * cols_per_tile;
    t.rows = min(BM, s.off[lo + 1] - t.m0);
    return t;
}

// ---- dequantisation of one B stage (256 weight rows x 64 k) ----------------

// weight row of B-tile row n (gate/up: rows [0,128) gate, [128,256) up)
template <int MODE>
__device__ __forceinline__ int b_row(int n, int n0, int n_out, int n_w, bool& valid) {
    if (MODE == MODE_GATE_UP) {
        const int c = n0 + (n & 127);
        valid = c < n_out;
        return (n < 128) ? c : n_out + c;
    } else {
        const int c = n0 + n;
        valid = c < n_w;
        return c;
    }
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    float v;
    if (e == 0) v = static_cast<float>(m) * 0.001953125f;  // m * 2^-9
    else if (e == 15 && m == 7) v = __uint_as_float(0x7fc00000u);
    else v = __uint_as_float(((e + 120u) << 23) | (m << 20));
    return (b & 0x80u) ? -v : v;
}

// two E2M1 codes (low nibble first) -> f16x2, low half = low nibble
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(byte));
    return r;
}

template <int ACT>
__device__ __forceinline__ uint32_t f16x2_to_act2(uint32_t h2) {
    if (ACT == MOE_ACT_F16) return h2;
    const float2 f = __half22float2(*reinterpret_cast<__half2*>(&h2));
    return Act<MOE_ACT_BF16>::pack2(f.x, f.y);
}

template <int MODE, int WFMT, int ACT>
__device__ __forceinline__ void dequant_stage(uint8_t* bstage, const GemmParams& p, const TileInfo& t, int kb,
                                              int dq_tid) {
    if (WFMT == MOE_W_GPTQ_INT4) {
        // item = (packed k-row i in 0..7, tile row n in 0..255); consecutive
        // threads take consecutive n: coalesced along the contiguous N axis
        const int g = (kb * BK) / p.group_size;
        const size_t kq_rows = static_cast<size_t>(p.K / 8);
        const int32_t* qw = static_cast<const int32_t*>(p.qw) + static_cast<size_t>(t.e) * kq_rows * p.n_w;
        const __half* qs = static_cast<const __half*>(p.qs) +
                           (static_cast<size_t>(t.e) * (p.K / p.group_size) + g) * p.n_w;
        const int32_t* qz = static_cast<const int32_t*>(p.qz) +
                            (static_cast<size_t>(t.e) * (p.K / p.group_size) + g) * (p.n_w / 8);
#pragma unroll 4
        for (int it = 0; it < (BN * 8) / (NUM_DQ_WARPS * 32); ++it) {
            const int idx = it * NUM_DQ_WARPS * 32 + dq_tid;
            const int i = idx >> 8, n = idx & 255;
            bool valid;
            const int wr = b_row<MODE>(n, t.n0, p.n_out, p.n_w, valid);
            uint4 v = make_uint4(0, 0, 0, 0);
            if (valid) {
                const uint32_t word = static_cast<uint32_t>(__ldg(qw + (static_cast<size_t>(kb) * 8 + i) * p.n_w + wr));
                const float s = __half2float(qs[wr]);
                const int z = (static_cast<uint32_t>(__ldg(qz + wr / 8)) >> (4 * (wr & 7))) & 15;
                float f[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) f[j] = static_cast<float>(static_cast<int>((word >> (4 * j)) & 15u) - z) * s;
                v.x = Act<ACT>::pack2(f[0], f[1]);
                v.y = Act<ACT>::pack2(f[2], f[3]);
                v.z = Act<ACT>::pack2(f[4], f[5]);
                v.w = Act<ACT>::pack2(f[6], f[7]);
            }
            *reinterpret_cast<uint4*>(bstage + n * 128 + ((i ^ (n & 7)) << 4)) = v;
        }
    } else {  // NVFP4: item = (tile row n, 8-element chunk c); 8 lanes per row
        const uint8_t* pk = static_cast<const uint8_t*>(p.qw) + static_cast<size_t>(t.e) * p.n_w * (p.K / 2);
        const uint8_t* sc = static_cast<const uint8_t*>(p.qs) + static_cast<size_t>(t.e) * (p.K / 16) * p.n_w;
#pragma unroll 4
        for (int it = 0; it < (BN * 8) / (NUM_DQ_WARPS * 32); ++it) {
            const int idx = it * NUM_DQ_WARPS * 32 + dq_tid;
            const int n = idx >> 3, c = idx & 7;
            bool valid;
            const int wr = b_row<MODE>(n, t.n0, p.n_out, p.n_w, valid);
            uint4 v = make_uint4(0, 0, 0, 0);
            const int k0 = kb * BK + c * 8;
            if (valid && k0 < p.K) {
                const uint32_t bytes = __ldg(reinterpret_cast<const uint32_t*>(pk + static_cast<size_t>(wr) * (p.K / 2) + k0 / 2));
                const float s = e4m3_to_f32(__ldg(sc + static_cast<size_t>(k0 / 16) * p.n_w + wr));
                const __half2 s2 = __float2half2_rn(s);  // exact: an E4M3 value is an fp16 value
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t h = e2m1x2_to_f16x2((bytes >> (8 * j)) & 0xffu);
                    __half2 prod = __hmul2(*reinterpret_cast<__half2*>(&h), s2);  // exact in fp16
                    o[j] = f16x2_to_act2<ACT>(*reinterpret_cast<uint32_t*>(&prod));
                }
                v = make_uint4(o[0], o[1], o[2], o[3]);
            }
            *reinterpret_cast<uint4*>(bstage + n * 128 + ((c ^ (n & 7)) << 4)) = v;
        }
    }
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

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// ---- the kernel ------------------------------------------------------------------

template <int MODE, int WFMT, int ACT>
__global__ void __launch_bounds__(WFMT == MOE_W_BF16 ? 192 : 192 + 32 * NUM_DQ_WARPS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_STAGE;
    SmemTail& s = *reinterpret_cast<SmemTail*>(smem + STAGES * (A_STAGE + B_STAGE));
    volatile int* abort_flag = &s.abort_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int E = p.E;
    constexpr int CPT = out_cols_per_tile<MODE>();

    // ---- tile list from expert_offsets ----
    for (int i = tid; i <= E; i += blockDim.x) s.off[i] = p.offsets[i];
    if (tid == 0) {
        s.abort_flag = 0;
        s.nt = (p.n_out + CPT - 1) / CPT;
    }
    __syncthreads();
    int bad = 0;
    for (int i = tid; i < E; i += blockDim.x) bad |= (s.off[i + 1] < s.off[i]);
    if (tid == 0) bad |= (s.off[0] < 0) | (s.off[E] > p.max_padded);
    bad = __syncthreads_or(bad);
    if (warp == 0) {
        // lane l owns experts [l * per, (l + 1) * per): local sums, warp scan, write exclusive prefix
        const int per = (E + 31) / 32;
        int loc = 0;
        for (int j = 0; j < per; ++j) {
            const int e = lane * per + j;
            if (e < E) loc += ((s.off[e + 1] - s.off[e] + BM - 1) / BM) * s.nt;
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
                run += ((s.off[e + 1] - s.off[e] + BM - 1) / BM) * s.nt;
            }
        }
        if (lane == 31) s.n_tiles = bad ? 0 : inc;
    }
    if (tid == 0) {
        if (bad) set_err(p.err, MOE_DEV_ERR_OFFSETS);
#pragma unroll
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&s.full[i], 1 + (WFMT == MOE_W_BF16 ? 0 : NUM_DQ_WARPS));
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.tfull[i], 1);
            mbar_init(&s.tempty[i], NUM_EPI_WARPS);
        }
        mbar_init(&s.mma_done, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const int n_tiles = s.n_tiles;
    if (static_cast<int>(blockIdx.x) >= n_tiles) return;  // block-uniform: nothing allocated yet

    if (warp == 1) {
        tmem_alloc(&s.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        if (WFMT == MOE_W_BF16) tma_prefetch_desc(&tmB);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s.tmem_base;
    const int KB = (p.K + BK - 1) / BK;  // a ragged last block is zero-filled

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            uint32_t stage = 0, phase = 0;
            long issued = 0;
            const uint32_t tx = (WFMT == MOE_W_BF16) ? (A_STAGE + B_STAGE) : A_STAGE;
            for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x) {
                const TileInfo t = decode_tile(s, E, tile, CPT);
                bool ok = true;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1, abort_flag, p.err)) { ok = false; break; }
                    mbar_arrive_expect_tx(&s.full[stage], tx);
                    tma_load_2d(sA + stage * A_STAGE, &tmA, kb * BK, t.m0, &s.full[stage]);
                    if (WFMT == MOE_W_BF16) {
                        uint8_t* b = sB + stage * B_STAGE;
                        const int r0 = t.e * p.n_w + t.n0;
                        const int r1 = (MODE == MODE_GATE_UP) ? r0 + p.n_out : r0 + 128;
                        tma_load_2d(b, &tmB, kb * BK, r0, &s.full[stage]);
                        tma_load_2d(b + B_STAGE / 2, &tmB, kb * BK, r1, &s.full[stage]);
                    }
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
            }
            // let every copy still in flight land before the CTA may exit
            const long first = issued > STAGES ? issued - STAGES : 0;
            for (long j = first; j < issued; ++j)
                mbar_drain(&s.full[j % STAGES], static_cast<uint32_t>((j / STAGES) & 1), kWaitLimitNs);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t idesc = f16_idesc(ACT, BM, BN);
            uint32_t stage = 0, phase = 0;
            int local = 0;
            for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++local) {
                const int acc = local & 1;
                const uint32_t aph = (local >> 1) & 1;
                if (!mbar_wait(&s.tempty[acc], aph ^ 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + acc * ACC_COLS;
                bool ok = true;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&s.full[stage], phase, abort_flag, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(smem_u32(sA + stage * A_STAGE));
                    const uint64_t bd = sw128_desc(smem_u32(sB + stage * B_STAGE));
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        tc_mma(d, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0);
                    tc_commit(&s.empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit(&s.tfull[acc]);
            }
            tc_commit(&s.mma_done);
            mbar_drain(&s.mma_done, 0, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp < 2 + NUM_EPI_WARPS) {
        // ---------------- epilogue ----------------
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        float s2a = 1.0f, s2b = 1.0f;
        int local = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t aph = (local >> 1) & 1;
            if (!mbar_wait(&s.tfull[acc], aph, abort_flag, p.err)) break;
            tc_fence_after();
            const TileInfo t = decode_tile(s, E, tile, CPT);
            if (WFMT == MOE_W_NVFP4) {
                if (MODE == MODE_GATE_UP) {
                    s2a = __ldg(p.scale2 + t.e);
                    s2b = __ldg(p.scale2 + p.E + t.e);
                } else {
                    s2a = __ldg(p.scale2 + t.e);
                }
            }
            const bool row_ok = row < t.rows;
            const size_t orow = static_cast<size_t>(t.m0 + row) * p.n_out;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * ACC_COLS;
            if (MODE == MODE_GATE_UP) {
#pragma unroll 1
                for (int c = 0; c < 128; c += 32) {
                    uint32_t g[32], u[32];
                    tmem_ld32(taddr + c, g);
                    tmem_ld32(taddr + 128 + c, u);
                    tmem_ld_wait();
                    if (row_ok) {
#pragma unroll
                        for (int j = 0; j < 32; j += 8) {
                            const int col = t.n0 + c + j;
                            if (col < p.n_out) {
                                float f[8];
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    f[i] = silu_mul(__uint_as_float(g[j + i]) * s2a, __uint_as_float(u[j + i]) * s2b);
                                store8<ACT>(p.out, orow + col, f);
                            }
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < 256; c += 32) {
                    uint32_t g[32];
                    tmem_ld32(taddr + c, g);
                    tmem_ld_wait();
                    if (row_ok) {
#pragma unroll
                        for (int j = 0; j < 32; j += 8) {
                            const int col = t.n0 + c + j;
                            if (col < p.n_out) {
                                float f[8];
#pragma unroll
                                for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(g[j + i]) * s2a;
                                store8<ACT>(p.out, orow + col, f);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.tempty[acc]);
        }
    } else {
        // ---------------- dequantising producers (quantised weights only) ----------------
        if (WFMT != MOE_W_BF16) {
            const int dq_tid = tid - 32 * (2 + NUM_EPI_WARPS);
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                const TileInfo t = decode_tile(s, E, tile, CPT);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1, abort_flag, p.err)) { ok = false; break; }
                    dequant_stage<MODE, WFMT, ACT>(sB + stage * B_STAGE, p, t, kb, dq_tid);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s.full[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ---- gather of the activations into sorted-row order ---------------------------

// xs[r] = x[sorted_token_ids[r] / top_k] for r < expert_offsets[E]; padding
// rows (sentinel) are zero-filled. One warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ sorted_ids,
                   const int32_t* __restrict__ offsets, int E, int T, int top_k, int vec_per_row, int max_padded,
                   uint4* __restrict__ xs, int32_t* err) {
    const int total = min(__ldg(offsets + E), max_padded);
    const int P = T * top_k;
    for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < total; r += gridDim.x * 8) {
        const int pid = __ldg(sorted_ids + r);
        int tok = -1;
        if (pid >= 0 && pid < P) tok = pid / top_k;
        else if (pid != P && (threadIdx.x & 31) == 0) set_err(err, MOE_DEV_ERR_PAIR_ID);
        uint4* dst = xs + static_cast<size_t>(r) * vec_per_row;
        if (tok >= 0) {
            const uint4* src = x + static_cast<size_t>(tok) * vec_per_row;
            for (int v = threadIdx.x & 31; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
        } else {
            for (int v = threadIdx.x & 31; v < vec_per_row; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
        }
    }
}

// ---- host launchers ----------------------------------------------------------------

template <int MODE, int WFMT, int ACT>
int launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, cudaStream_t st,
                const char* who) {
    auto kernel = grouped_gemm_kernel<MODE, WFMT, ACT>;
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        int rc = set_smem_limit(reinterpret_cast<const void*>(kernel), SMEM_BYTES);
        if (rc != MOE_OK) return rc;
        configured_for = dev;
    }
    constexpr int CPT = out_cols_per_tile<MODE>();
    const long bound = static_cast<long>((p.max_padded + BM - 1) / BM + p.E) * ((p.n_out + CPT - 1) / CPT);
    const int sms = sm_count();
    if (sms <= 0) return fail(MOE_ERR_CUDA, "%s: cannot query the SM count", who);
    const int grid = static_cast<int>(bound < sms ? bound : sms);
    if (grid <= 0) return MOE_OK;
    const int threads = (WFMT == MOE_W_BF16) ? 192 : 192 + 32 * NUM_DQ_WARPS;
    kernel<<<grid, threads, SMEM_BYTES, st>>>(tmA, tmB, p);
    count_launch();
    return check_launch(who);
}

template <int MODE>
int dispatch(int wfmt, int act, const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p,
             cudaStream_t st, const char* who) {
    if (wfmt == MOE_W_BF16) return launch_gemm<MODE, MOE_W_BF16, MOE_ACT_BF16>(tmA, tmB, p, st, who);
    if (wfmt == MOE_W_GPTQ_INT4)
        return act == MOE_ACT_F16 ? launch_gemm<MODE, MOE_W_GPTQ_INT4, MOE_ACT_F16>(tmA, tmB, p, st, who)
                                  : launch_gemm<MODE, MOE_W_GPTQ_INT4, MOE_ACT_BF16>(tmA, tmB, p, st, who);
    return act == MOE_ACT_F16 ? launch_gemm<MODE, MOE_W_NVFP4, MOE_ACT_F16>(tmA, tmB, p, st, who)
                              : launch_gemm<MODE, MOE_W_NVFP4, MOE_ACT_BF16>(tmA, tmB, p, st, who);
}

int check_weight(const MoeWeight* w, int act, int N, int K, const char* who) {
    MOE_REQUIRE(w != nullptr, "%s: NULL weight descriptor", who);
    MOE_REQUIRE(act == MOE_ACT_BF16 || act == MOE_ACT_F16, "%s: unknown activation type %d", who, act);
    switch (w->format) {
        case MOE_W_BF16:
            MOE_REQUIRE(act == MOE_ACT_BF16, "%s: a bf16 weight needs bf16 activations (the tensor cores take "
                                             "one 16-bit type for both operands)", who);
            MOE_REQUIRE(w->w && aligned16(w->w), "%s: bf16 weight pointer NULL or not 16-byte aligned", who);
            return MOE_OK;
        case MOE_W_GPTQ_INT4:
            MOE_REQUIRE(w->w && w->scales && w->zeros, "%s: GPTQ qweight / scales / qzeros must be non-NULL", who);
            MOE_REQUIRE(w->group_size >= 64 && w->group_size % 64 == 0 && K % w->group_size == 0,
                        "%s: GPTQ group_size=%d must be a multiple of 64 dividing K=%d", who, w->group_size, K);
            MOE_REQUIRE(N % 8 == 0, "%s: GPTQ needs N=%d divisible by 8", who, N);
            return MOE_OK;
        case MOE_W_NVFP4:
            MOE_REQUIRE(w->w && w->scales && w->scale2, "%s: NVFP4 packed / scales / scale2 must be non-NULL", who);
            MOE_REQUIRE(K % 16 == 0, "%s: NVFP4 needs K=%d divisible by 16 (one E4M3 scale per 16)", who, K);
            MOE_REQUIRE((reinterpret_cast<uintptr_t>(w->w) & 3) == 0, "%s: NVFP4 packed weight not 4-byte aligned",
                        who);
            return MOE_OK;
        default:
            return fail(MOE_ERR_INVALID, "%s: unknown weight format %d", who, w->format);
    }
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_gate_up_workspace_size(int32_t max_padded, int32_t H) {
    if (max_padded < 0 || H < 0) return 0;
    return static_cast<size_t>(max_padded) * H * 2;
}

extern "C" int moe_grouped_gate_up(const void* x, int32_t act, const MoeWeight* w_gate_up,
                                   const int32_t* sorted_token_ids, const int32_t* expert_offsets, int32_t T,
                                   int32_t top_k, int32_t H, int32_t I, int32_t E, int32_t max_padded, void* h_out,
                                   int32_t* err_word, void* workspace, size_t workspace_bytes, void* stream) {
    const char* who = "moe_grouped_gate_up";
    MOE_REQUIRE(E >= 1 && E <= MOE_MAX_EXPERTS, "%s: E=%d outside [1, %d]", who, E, MOE_MAX_EXPERTS);
    MOE_REQUIRE(T >= 0 && top_k >= 1 && max_padded >= 0, "%s: bad T=%d / top_k=%d / max_padded=%d", who, T, top_k,
                max_padded);
    MOE_REQUIRE(H > 0 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", who, H);
    MOE_REQUIRE(I > 0 && I % 8 == 0, "%s: I=%d must be a positive multiple of 8", who, I);
    int rc = moe::check_weight(w_gate_up, act, 2 * I, H, who);
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
        const int rows_per_block = 8;
        int blocks = (max_padded + rows_per_block - 1) / rows_per_block;
        const int cap = sms > 0 ? sms * 8 : 1024;
        if (blocks > cap) blocks = cap;
        moe::gather_rows_kernel<<<blocks, 256, 0, st>>>(static_cast<const uint4*>(x), sorted_token_ids,
                                                        expert_offsets, E, T, top_k, H / 8, max_padded,
                                                        static_cast<uint4*>(workspace), err_word);
        moe::count_launch();
        rc = moe::check_launch("moe_grouped_gate_up (gather)");
        if (rc != MOE_OK) return rc;
    }
    // 2. the grouped GEMM
    CUtensorMap tmA, tmB;
    rc = moe::make_tmap_2d(&tmA, workspace, max_padded, H, 128, act);
    if (rc != MOE_OK) return rc;
    if (w_gate_up->format == MOE_W_BF16) {
        rc = moe::make_tmap_2d(&tmB, w_gate_up->w, static_cast<uint64_t>(E) * 2 * I, H, 128, act);
        if (rc != MOE_OK) return rc;
    } else {
        tmB = tmA;
    }
    moe::GemmParams p{};
    p.offsets = expert_offsets;
    p.E = E;
    p.K = H;
    p.n_out = I;
    p.n_w = 2 * I;
    p.max_padded = max_padded;
    p.out = h_out;
    p.qw = w_gate_up->w;
    p.qs = w_gate_up->scales;
    p.qz = w_gate_up->zeros;
    p.scale2 = w_gate_up->scale2;
    p.group_size = w_gate_up->group_size;
    p.err = err_word;
    return moe::dispatch<moe::MODE_GATE_UP>(w_gate_up->format, act, tmA, tmB, p, st, who);
}

extern "C" int moe_grouped_down(const void* h, int32_t act, const MoeWeight* w_down, const int32_t* expert_offsets,
                                int32_t H, int32_t I, int32_t E, int32_t max_padded, void* y, int32_t* err_word,
                                void* stream) {
    const char* who = "moe_grouped_down";
    MOE_REQUIRE(E >= 1 && E <= MOE_MAX_EXPERTS, "%s: E=%d outside [1, %d]", who, E, MOE_MAX_EXPERTS);
    MOE_REQUIRE(I > 0 && I % 8 == 0, "%s: I=%d must be a positive multiple of 8", who, I);
    MOE_REQUIRE(H > 0 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", who, H);
    MOE_REQUIRE(max_padded >= 0, "%s: max_padded=%d is negative", who, max_padded);
    int rc = moe::check_weight(w_down, act, H, I, who);
    if (rc != MOE_OK) return rc;
    if (max_padded == 0) return MOE_OK;
    MOE_REQUIRE(h && expert_offsets && y, "%s: NULL pointer", who);
    MOE_REQUIRE(moe::aligned16(h) && moe::aligned16(y), "%s: h / y must be 16-byte aligned", who);
    CUtensorMap tmA, tmB;
    rc = moe::make_tmap_2d(&tmA, h, max_padded, I, 128, act);
    if (rc != MOE_OK) return rc;
    if (w_down->format == MOE_W_BF16) {
        rc = moe::make_tmap_2d(&tmB, w_down->w, static_cast<uint64_t>(E) * H, I, 128, act);
        if (rc != MOE_OK) return rc;
    } else {
        tmB = tmA;
    }
    moe::GemmParams p{};
    p.offsets = expert_offsets;
    p.E = E;
    p.K = I;
    p.n_out = H;
    p.n_w = H;
    p.max_padded = max_padded;
    p.out = y;
    p.qw = w_down->w;
    p.qs = w_down->scales;
    p.qz = w_down->zeros;
    p.scale2 = w_down->scale2;
    p.group_size = w_down->group_size;
    p.err = err_word;
    return moe::dispatch<moe::MODE_DOWN>(w_down->format, act, tmA, tmB, p, static_cast<cudaStream_t>(stream), who);
}
