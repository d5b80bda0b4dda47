// Step a1: top-k softmax routing, one warp per token row.
//
// Restates ferrum-kernels 0.7.7 src/backend/cuda/moe.rs, route_topk_softmax
// (one warp per row, a per-row f32 probability vector, norm_topk_prob). The
// row's logits stay in registers (E <= 256: at most 8 per lane), so no shared
// memory is needed. Selection compares logits (softmax is monotone), larger
// first and, on equal logits, the lower expert index first.
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kPerLane = MOE_MAX_EXPERTS / 32;  // 8
constexpr int kRowsPerBlock = 1;  // one warp per block: rows spread over every SM (the fp64
                                   // exponential runs on few units per SM)

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

// Top-k softmax of one row whose logits sit in registers: lane l holds
// v[j] = logit of expert l + 32 j (E <= 256). Writes the row's top_k ids and
// weights (lanes < top_k). Shared by the routing kernel and the fused router
// kernel, so both take the same decisions in the same arithmetic.
__device__ __forceinline__ void route_row(const float (&v)[kPerLane], int lane, int E, int k, int renorm,
                                          int32_t* __restrict__ ids_row, float* __restrict__ w_row) {
    uint32_t taken = 0;  // bit j: element lane + 32 j already selected (or absent)
#pragma unroll
    for (int j = 0; j < kPerLane; ++j)
        if (lane + 32 * j >= E) taken |= 1u << j;

    int sel_i[MOE_MAX_TOPK];
    float sel_v[MOE_MAX_TOPK];
#pragma unroll
    for (int r = 0; r < MOE_MAX_TOPK; ++r) {
        sel_i[r] = 0;
        sel_v[r] = 0.0f;
        if (r >= k) continue;
        float bv = 0.0f;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < kPerLane; ++j) {
            const int i = lane + 32 * j;
            if (!(taken >> j & 1u) && (bi == 0x7fffffff || better(v[j], i, bv, bi))) {
                bv = v[j];
                bi = i;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (oi != 0x7fffffff && (bi == 0x7fffffff || better(ov, oi, bv, bi))) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        sel_i[r] = bi;
        sel_v[r] = bv;
    }

    const float m = sel_v[0];
    // lane r < k holds the exponential of its selected expert: the fp64 exp is
    // evaluated once per selected expert, in parallel across the lanes
    float sv = 0.0f;
    int si = 0;
#pragma unroll
    for (int q = 0; q < MOE_MAX_TOPK; ++q)
        if (q == lane) {
            sv = sel_v[q];
            si = sel_i[q];
        }
    const float e_mine = (lane < k) ? __double2float_rn(exp(static_cast<double>(__fsub_rn(sv, m)))) : 0.0f;
    float denom;
    if (renorm) {
        denom = 0.0f;  // e_0 + e_1 + ... in rank order
#pragma unroll
        for (int r = 0; r < MOE_MAX_TOPK; ++r) {
            const float er = __shfl_sync(0xffffffffu, e_mine, r);
            if (r < k) denom = __fadd_rn(denom, er);
        }
    } else {
        float part = 0.0f;
#pragma unroll
        for (int j = 0; j < kPerLane; ++j) {
            if (lane + 32 * j < E)
                part = __fadd_rn(part, __double2float_rn(exp(static_cast<double>(__fsub_rn(v[j], m)))));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, off));
        denom = part;
    }
    if (lane < k) {
        ids_row[lane] = si;
        w_row[lane] = __fdiv_rn(e_mine, denom);
    }
}

__global__ void __launch_bounds__(32 * kRowsPerBlock)
route_topk_softmax_kernel(const float* __restrict__ logits, int32_t* __restrict__ ids, float* __restrict__ w, int T,
                          int E, int k, int renorm) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (row >= T) return;
    const float* lrow = logits + static_cast<size_t>(row) * E;
    float v[kPerLane];
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
        const int i = lane + 32 * j;
        v[j] = (i < E) ? __ldg(lrow + i) : 0.0f;
    }
    route_row(v, lane, E, k, renorm, ids + static_cast<size_t>(row) * k, w + static_cast<size_t>(row) * k);
}

// ---- router GEMM fused with routing ----------------------------------------------
//
// The workloads define the router the pages leave out: logits[t, e] =
// sum_h x[t, h] * Wr[h, e] with Wr f32 [H, E] (E <= 256). At E = 8 it is a
// few FLOPs per activation byte, so the kernel is built to stream x at HBM
// rate with every CTA of the grid resident at once; at E >= 128 it is bound
// by the fp32 fused multiply-adds.
//   * A cluster of CS CTAs (CS = 1, 2, 4 or 8) takes TT = 32 TPL tokens
//     (lane l holds tokens l, l + 32, ...: TPL = 2 for E <= 16, else 1); CTA
//     c of the cluster takes the contraction range [c HR, (c + 1) HR). Its
//     eight warps are G expert groups (EG = 8, 16 or 32 experts, one
//     accumulator register each per token) times S = 8 / G contraction
//     slices.
//   * The CTA's router-weight rows are staged in shared memory in chunks of
//     HC rows (two buffers, cp.async); each lane reads its tokens'
//     activations straight from global memory as 16-byte vectors, the next
//     chunk's in flight while the current one is used.
//   * Sums: a lane accumulates its slice of each chunk in ascending h by
//     fused multiply-adds; the S slice sums of a CTA are added in slice
//     order, then the CS CTA sums in rank order, read through distributed
//     shared memory, so the result does not depend on timing.
//   * CTA c then finishes tokens [c TT / CS, (c + 1) TT / CS) of the
//     cluster: it writes their logits and routes them, one warp per token,
//     with the same route_row as moe_route_topk_softmax.
constexpr int kRtThreads = 256, kRtWarps = kRtThreads / 32;
constexpr int kRtChunkFloats = 8192;  // router-weight floats per staged chunk at most (32 KB)
constexpr int kRtMaxSmem = 100 * 1024;  // shared memory of the largest plan (E = 256: 96 KB)

// 16-byte activation vectors per lane and token per chunk at most
__host__ __device__ constexpr int rt_max_vec(int tpl) { return tpl == 2 ? 2 : 4; }

struct RtPlan {
    int eg, g, s;  // experts per group, groups, contraction slices
    int tpl, tt;   // tokens per lane, tokens per cluster
    int ep;        // E rounded up to 4: row stride of the staged weights
    int hc;        // weight rows per chunk (a multiple of 8 S)
    int cs;        // CTAs per cluster
    int hr;        // contraction rows per CTA (a multiple of 8 S)
};

inline RtPlan rt_plan(int H, int E) {
    RtPlan r;
    r.eg = E <= 8 ? 8 : (E <= 16 ? 16 : 32);
    r.g = (E + r.eg - 1) / r.eg;  // <= 8
    r.s = kRtWarps / r.g;         // >= 1
    r.tpl = r.eg <= 16 ? 2 : 1;
    r.tt = 32 * r.tpl;
    r.ep = (E + 3) / 4 * 4;
    const int step = 8 * r.s;
    int hc = kRtChunkFloats / r.ep / step * step;
    if (hc > rt_max_vec(r.tpl) * step) hc = rt_max_vec(r.tpl) * step;
    r.hc = hc < step ? step : hc;
    // as many CTAs per token block as leave each warp slice at least one
    // 16-byte vector (8 h) of the contraction
    r.cs = 8;
    while (r.cs > 1 && H < r.cs * step) r.cs >>= 1;
    const int per = (H + r.cs - 1) / r.cs;
    r.hr = (per + step - 1) / step * step;
    return r;
}

// weight chunks (two) or, afterwards, the finished logits; then the slice sums
__host__ __device__ inline int rt_wbuf_floats(const RtPlan& r) { return (2 * r.hc > r.tt ? 2 * r.hc : r.tt) * r.ep; }
inline size_t rt_smem_bytes(const RtPlan& r) {
    return (static_cast<size_t>(rt_wbuf_floats(r)) + static_cast<size_t>(r.s) * r.tt * r.ep) * sizeof(float);
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t cluster_addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
    return v;
}

template <int ACT, int EG, int TPL>
__global__ void __launch_bounds__(kRtThreads, EG == 8 ? 4 : (EG == 16 ? 3 : 2))  // E <= 8: one wave at T = 4096
router_topk_kernel(const typename Act<ACT>::T* __restrict__ x, const float* __restrict__ wr,
                   float* __restrict__ logits, int32_t* __restrict__ ids, float* __restrict__ wout, int T, int H,
                   int E, int k, int renorm, const RtPlan pl) {
    constexpr int V = rt_max_vec(TPL);
    constexpr int TT = 32 * TPL;
    pdl_wait();
    extern __shared__ float rt_smem[];
    float* wbuf = rt_smem;                     // two weight chunks [hc][ep]; afterwards the finals [tpc][ep]
    float* red = rt_smem + rt_wbuf_floats(pl);  // slice sums [s][TT tokens][ep]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = static_cast<int>(cluster_ctarank());
    const int t0 = (blockIdx.x / pl.cs) * TT;
    const int g = warp / pl.s, sl = warp % pl.s;
    const bool active = g < pl.g;
    const int e0 = g * EG;
    const int hs = pl.hc / pl.s;  // contraction rows per warp per chunk (a multiple of 8)
    const int h_begin = c * pl.hr;
    const int h_end = min(H, h_begin + pl.hr);
    const int nchunks = h_end > h_begin ? (h_end - h_begin + pl.hc - 1) / pl.hc : 0;

    // stage weight chunk j (rows h_begin + j hc ...) into buffer j & 1
    auto stage_w = [&](int j) {
        const int h0 = h_begin + j * pl.hc;
        const int rows = min(pl.hc, h_end - h0);
        float* dst = wbuf + (j & 1) * pl.hc * pl.ep;
        const float* src = wr + static_cast<size_t>(h0) * E;
        if ((E & 3) == 0) {
            const int n4 = rows * E / 4;
            for (int i = tid; i < n4; i += kRtThreads) cp_async16(dst + 4 * i, src + 4 * i);
        } else {
            for (int rr = warp; rr < rows; rr += kRtWarps)
                for (int e = lane; e < E; e += 32) cp_async4(dst + rr * pl.ep + e, src + rr * E + e);
        }
        cp_async_commit();
    };
    // this lane's activation vectors of chunk j (zeros past the token count or H)
    auto load_x = [&](int j, uint4 (&v)[TPL][V]) {
        const int hb = h_begin + j * pl.hc + sl * hs;
#pragma unroll
        for (int q = 0; q < TPL; ++q) {
            const int t = t0 + lane + 32 * q;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const int h = hb + 8 * i;
                v[q][i] = make_uint4(0u, 0u, 0u, 0u);
                if (active && 8 * i < hs && t < T && h < h_end)
                    v[q][i] = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H + h));
            }
        }
    };

    float acc[TPL][EG];
#pragma unroll
    for (int q = 0; q < TPL; ++q)
#pragma unroll
        for (int j = 0; j < EG; ++j) acc[q][j] = 0.0f;
    uint4 cur[TPL][V], nxt[TPL][V];
    if (nchunks > 0) {
        stage_w(0);
        load_x(0, cur);
    }
    for (int j = 0; j < nchunks; ++j) {
        cp_async_wait_all();
        __syncthreads();  // chunk j staged; everyone is done with chunk j - 1's buffer
        if (j + 1 < nchunks) {
            stage_w(j + 1);
            load_x(j + 1, nxt);
        }
        if (active) {
            const float* wc = wbuf + (j & 1) * pl.hc * pl.ep;
            const int hb = h_begin + j * pl.hc + sl * hs;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                if (8 * i >= hs || hb + 8 * i >= h_end) break;
                float xf[TPL][8];
#pragma unroll
                for (int q = 0; q < TPL; ++q) {
                    const float2 p0 = Act<ACT>::unpack2(cur[q][i].x), p1 = Act<ACT>::unpack2(cur[q][i].y);
                    const float2 p2 = Act<ACT>::unpack2(cur[q][i].z), p3 = Act<ACT>::unpack2(cur[q][i].w);
                    xf[q][0] = p0.x; xf[q][1] = p0.y; xf[q][2] = p1.x; xf[q][3] = p1.y;
                    xf[q][4] = p2.x; xf[q][5] = p2.y; xf[q][6] = p3.x; xf[q][7] = p3.y;
                }
#pragma unroll
                for (int hh = 0; hh < 8; ++hh) {
                    const float4* w4 = reinterpret_cast<const float4*>(wc + (sl * hs + 8 * i + hh) * pl.ep + e0);
#pragma unroll
                    for (int j4 = 0; j4 < EG / 4; ++j4) {
                        const float4 wv = w4[j4];  // the same address in every lane: a broadcast
#pragma unroll
                        for (int q = 0; q < TPL; ++q) {
                            acc[q][4 * j4] = fmaf(xf[q][hh], wv.x, acc[q][4 * j4]);
                            acc[q][4 * j4 + 1] = fmaf(xf[q][hh], wv.y, acc[q][4 * j4 + 1]);
                            acc[q][4 * j4 + 2] = fmaf(xf[q][hh], wv.z, acc[q][4 * j4 + 2]);
                            acc[q][4 * j4 + 3] = fmaf(xf[q][hh], wv.w, acc[q][4 * j4 + 3]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < TPL; ++q)
#pragma unroll
            for (int i = 0; i < V; ++i) cur[q][i] = nxt[q][i];
    }
    // slice sums of this CTA, added in slice order into red[0]
    if (active)
#pragma unroll
        for (int q = 0; q < TPL; ++q)
#pragma unroll
            for (int j = 0; j < EG; ++j)
                if (e0 + j < E) red[(sl * TT + lane + 32 * q) * pl.ep + e0 + j] = acc[q][j];
    __syncthreads();
    if (pl.s > 1)
        for (int tok = warp; tok < TT; tok += kRtWarps)
            for (int e = lane; e < E; e += 32) {
                float v = red[tok * pl.ep + e];
                for (int s = 1; s < pl.s; ++s) v = __fadd_rn(v, red[(s * TT + tok) * pl.ep + e]);
                red[tok * pl.ep + e] = v;
            }
    cluster_sync_all();  // every CTA's sums are in its red[0]
    // finish tokens [c tpc, (c + 1) tpc): add the CTA sums in rank order
    // (every rank's value is loaded first, then they are added in order)
    const int tpc = TT / pl.cs;
    float* fin = wbuf;  // [tpc][ep]
    for (int tl = warp; tl < tpc; tl += kRtWarps)
        for (int e = lane; e < E; e += 32) {
            const uint32_t a = smem_u32(red + (c * tpc + tl) * pl.ep + e);
            float part[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) part[r] = r < pl.cs ? ld_dsmem_f32(mapa_shared(a, r)) : 0.0f;
            float v = part[0];
#pragma unroll
            for (int r = 1; r < 8; ++r)
                if (r < pl.cs) v = __fadd_rn(v, part[r]);
            fin[tl * pl.ep + e] = v;
            const int tt = t0 + c * tpc + tl;
            if (tt < T) logits[static_cast<size_t>(tt) * E + e] = v;
        }
    cluster_arrive();  // this CTA has read its peers' sums
    __syncthreads();
    for (int tl = warp; tl < tpc; tl += kRtWarps) {
        const int tt = t0 + c * tpc + tl;
        if (tt >= T) break;
        float v[kPerLane];
#pragma unroll
        for (int j = 0; j < kPerLane; ++j) {
            const int e = lane + 32 * j;
            v[j] = e < E ? fin[tl * pl.ep + e] : 0.0f;
        }
        route_row(v, lane, E, k, renorm, ids + static_cast<size_t>(tt) * k, wout + static_cast<size_t>(tt) * k);
    }
    cluster_wait();  // no CTA leaves while a peer may still read its shared memory
}

template <int ACT>
int launch_router(const void* x, const float* w_router, float* logits, int32_t* ids, float* w, int T, int H, int E,
                  int k, int renorm, cudaStream_t st) {
    const RtPlan pl = rt_plan(H, E);
    const size_t smem = rt_smem_bytes(pl);
    if (smem > static_cast<size_t>(kRtMaxSmem)) return fail(MOE_ERR_UNSUPPORTED, "moe_router_topk_softmax: plan too large");
    cudaError_t e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = pl.cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>((T + pl.tt - 1) / pl.tt * pl.cs), 1, 1);
    cfg.blockDim = dim3(kRtThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    using T_ = typename Act<ACT>::T;
    const T_* xp = static_cast<const T_*>(x);
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {  // every plan fits in kRtMaxSmem bytes
        for (const void* f : {reinterpret_cast<const void*>(router_topk_kernel<ACT, 8, 2>),
                              reinterpret_cast<const void*>(router_topk_kernel<ACT, 16, 2>),
                              reinterpret_cast<const void*>(router_topk_kernel<ACT, 32, 1>)}) {
            const int rc = set_smem_limit(f, kRtMaxSmem);
            if (rc != MOE_OK) return rc;
        }
        configured_for = dev;
    }
    if (pl.eg == 8)
        e = cudaLaunchKernelEx(&cfg, router_topk_kernel<ACT, 8, 2>, xp, w_router, logits, ids, w, T, H, E, k, renorm,
                               pl);
    else if (pl.eg == 16)
        e = cudaLaunchKernelEx(&cfg, router_topk_kernel<ACT, 16, 2>, xp, w_router, logits, ids, w, T, H, E, k, renorm,
                               pl);
    else
        e = cudaLaunchKernelEx(&cfg, router_topk_kernel<ACT, 32, 1>, xp, w_router, logits, ids, w, T, H, E, k, renorm,
                               pl);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "moe_router_topk_softmax: launch failed: %s", cudaGetErrorString(e));
    count_launch();
    return check_launch("moe_router_topk_softmax");
}

}  // namespace
}  // namespace moe

extern "C" int moe_route_topk_softmax(const float* logits, int32_t* topk_ids, float* topk_weights, int32_t T,
                                      int32_t E, int32_t top_k, int32_t renormalize, void* stream) {
    MOE_REQUIRE(E >= 1 && E <= MOE_MAX_EXPERTS, "moe_route_topk_softmax: E=%d outside [1, %d]", E,
                MOE_MAX_EXPERTS);
    MOE_REQUIRE(top_k >= 1 && top_k <= E && top_k <= MOE_MAX_TOPK,
                "moe_route_topk_softmax: top_k=%d outside [1, min(E=%d, %d)]", top_k, E, MOE_MAX_TOPK);
    MOE_REQUIRE(T >= 0, "moe_route_topk_softmax: T=%d is negative", T);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(logits && topk_ids && topk_weights, "moe_route_topk_softmax: NULL pointer");
    const int blocks = (T + moe::kRowsPerBlock - 1) / moe::kRowsPerBlock;
    moe::launch_pdl(moe::route_topk_softmax_kernel, blocks, 32 * moe::kRowsPerBlock, 0, static_cast<cudaStream_t>(stream),
        logits, topk_ids, topk_weights, T, E, top_k, renormalize ? 1 : 0);
    moe::count_launch();
    return moe::check_launch("moe_route_topk_softmax");
}

extern "C" int moe_router_topk_softmax(const void* x, int32_t act, const float* w_router, int32_t T, int32_t H,
                                       int32_t E, int32_t top_k, int32_t renormalize, float* logits,
                                       int32_t* topk_ids, float* topk_weights, void* stream) {
    const char* who = "moe_router_topk_softmax";
    MOE_REQUIRE(E >= 1 && E <= MOE_MAX_EXPERTS, "%s: E=%d outside [1, %d]", who, E, MOE_MAX_EXPERTS);
    MOE_REQUIRE(top_k >= 1 && top_k <= E && top_k <= MOE_MAX_TOPK, "%s: top_k=%d outside [1, min(E=%d, %d)]", who,
                top_k, E, MOE_MAX_TOPK);
    MOE_REQUIRE(act == MOE_ACT_BF16 || act == MOE_ACT_F16, "%s: act=%d is neither bf16 nor fp16", who, act);
    MOE_REQUIRE(T >= 0, "%s: T=%d is negative", who, T);
    MOE_REQUIRE(H > 0 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", who, H);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(x && w_router && logits && topk_ids && topk_weights, "%s: NULL pointer", who);
    MOE_REQUIRE(moe::aligned16(x), "%s: x must be 16-byte aligned", who);
    MOE_REQUIRE((E % 4 != 0) || moe::aligned16(w_router), "%s: w_router must be 16-byte aligned", who);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int renorm = renormalize ? 1 : 0;
    if (act == MOE_ACT_BF16)
        return moe::launch_router<MOE_ACT_BF16>(x, w_router, logits, topk_ids, topk_weights, T, H, E, top_k, renorm,
                                                st);
    return moe::launch_router<MOE_ACT_F16>(x, w_router, logits, topk_ids, topk_weights, T, H, E, top_k, renorm, st);
}
