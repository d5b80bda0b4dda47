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
        ids[static_cast<size_t>(row) * k + lane] = si;
        w[static_cast<size_t>(row) * k + lane] = __fdiv_rn(e_mine, denom);
    }
}

// ---- router GEMM: logits = x . Wr ----------------------------------------------
//
// The workloads define the router the pages leave out: logits[t, e] =
// sum_h x[t, h] * Wr[h, e] with Wr f32 [H, E] (E <= 256, a few hundred FLOPs
// per token: the work is small and latency-bound). A block computes 32 tokens
// (lane = token) x E logits in fp32 fused multiply-adds. Its eight warps split
// the experts into NG groups of up to 32 and the contraction into S = 8 / NG
// slices; each D-deep chunk of activations (as f32, rows padded against bank
// conflicts) and of Wr is staged in shared memory while the next chunk's
// loads are in flight in registers. Slice s of a chunk is h = h0 + s * D / S
// ... h0 + (s + 1) * D / S - 1 in ascending order; the S slice sums are added
// in order 0, 1, ... at the end, so the result does not depend on timing.
constexpr int kRtTok = 32, kRtThreads = 256, kRtWarps = kRtThreads / 32;
constexpr int kRtMaxD = 512;                            // chunk depth at most
constexpr int kRtXPer = kRtTok * kRtMaxD / 4 / kRtThreads;  // 4-feature activation loads per thread: 16
constexpr int kRtWPer = 8192 / kRtThreads;               // weight words per thread at most: 32 (D * E <= 8192)

struct RtShape {
    int eg, ng, s, d;  // experts per group, groups, slices, chunk depth
};

__host__ __device__ inline RtShape rt_shape(int E) {
    RtShape r;
    r.eg = E < 32 ? E : 32;
    r.ng = (E + r.eg - 1) / r.eg;                        // <= 8
    r.s = kRtWarps / r.ng;                               // >= 1
    // as deep as D * E <= 8192 weight words allows, at most 512: few chunks,
    // so few load latencies in a row
    const int m = 256 / E;                               // 8192 / (32 E)
    r.d = 32 * (m < 1 ? 1 : (m > 16 ? 16 : m));          // 32 .. 512
    return r;
}

template <int ACT>
__global__ void __launch_bounds__(kRtThreads)
router_logits_kernel(const typename Act<ACT>::T* __restrict__ x, const float* __restrict__ wr,
                     float* __restrict__ logits, int T, int H, int E) {
    pdl_wait();
    extern __shared__ float rt_smem[];
    const RtShape sh = rt_shape(E);
    const int D = sh.d, XP = D + 1;
    float* xs = rt_smem;                  // [32 tokens][D + 1]
    float* ws = rt_smem + kRtTok * XP;    // [D][E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * kRtTok;
    const int g = warp / sh.s, sl = warp % sh.s;       // expert group, contraction slice
    const bool active = g < sh.ng;
    const int e0 = g * sh.eg;
    const int hs = D / sh.s;                           // h per slice per chunk
    // staging map: activation loads of 4 features, thread -> (token, feature)
    const int xq = D / 4;                              // 4-feature groups per token row
    uint2 xr[kRtXPer];
    float wv[kRtWPer];
    auto load_chunk = [&](int h0) {
#pragma unroll
        for (int i = 0; i < kRtXPer; ++i) {
            const int idx = tid + i * kRtThreads;      // < 32 * xq when i < 32 * xq / 256
            const int tok = idx / xq, h = h0 + (idx % xq) * 4;
            const int t = t0 + tok;
            xr[i] = make_uint2(0u, 0u);
            if (idx < kRtTok * xq && t < T && h < H)   // H % 8 == 0: the 4 features are in range
                xr[i] = *reinterpret_cast<const uint2*>(x + static_cast<size_t>(t) * H + h);
        }
        const int n = (H - h0 < D ? H - h0 : D) * E;
#pragma unroll
        for (int i = 0; i < kRtWPer; ++i) {
            const int idx = tid + i * kRtThreads;
            wv[i] = idx < n ? __ldg(wr + static_cast<size_t>(h0) * E + idx) : 0.0f;
        }
    };
    auto store_chunk = [&]() {
#pragma unroll
        for (int i = 0; i < kRtXPer; ++i) {
            const int idx = tid + i * kRtThreads;
            if (idx < kRtTok * xq) {
                const int tok = idx / xq, hq = (idx % xq) * 4;
                const float2 a = Act<ACT>::unpack2(xr[i].x), b = Act<ACT>::unpack2(xr[i].y);
                float* d = xs + tok * XP + hq;
                d[0] = a.x; d[1] = a.y; d[2] = b.x; d[3] = b.y;
            }
        }
#pragma unroll
        for (int i = 0; i < kRtWPer; ++i) {
            const int idx = tid + i * kRtThreads;
            if (idx < D * E) ws[idx] = wv[i];          // past the contraction: zeros
        }
    };
    float acc[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.0f;
    load_chunk(0);
    for (int h0 = 0; h0 < H; h0 += D) {
        store_chunk();
        __syncthreads();
        if (h0 + D < H) load_chunk(h0 + D);            // in flight during the FMAs below
        if (active) {
            const int hb = sl * hs;
            if ((E & 3) == 0) {  // rows and groups 16-byte aligned: 4 experts per read
                for (int hh = hb; hh < hb + hs; ++hh) {  // rows past H were staged as zeros
                    const float xv = xs[lane * XP + hh];
                    const float4* wrow = reinterpret_cast<const float4*>(ws + hh * E + e0);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4)
                        if (4 * j4 < sh.eg && e0 + 4 * j4 < E) {
                            const float4 wq = wrow[j4];
                            acc[4 * j4] = fmaf(xv, wq.x, acc[4 * j4]);
                            acc[4 * j4 + 1] = fmaf(xv, wq.y, acc[4 * j4 + 1]);
                            acc[4 * j4 + 2] = fmaf(xv, wq.z, acc[4 * j4 + 2]);
                            acc[4 * j4 + 3] = fmaf(xv, wq.w, acc[4 * j4 + 3]);
                        }
                }
            } else {
                for (int hh = hb; hh < hb + hs; ++hh) {
                    const float xv = xs[lane * XP + hh];
                    const float* wrow = ws + hh * E + e0;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < sh.eg && e0 + j < E) acc[j] = fmaf(xv, wrow[j], acc[j]);
                }
            }
        }
        __syncthreads();
    }
    // add the slices in order: slice s writes its sums, slice 0 adds them up
    float* red = rt_smem;  // [slices 1..S-1][32 tokens][E]
    for (int s = 1; s < sh.s; ++s) {
        if (active && sl == s)
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < sh.eg && e0 + j < E) red[((s - 1) * kRtTok + lane) * E + e0 + j] = acc[j];
    }
    __syncthreads();
    const int t = t0 + lane;
    if (active && sl == 0 && t < T) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int e = e0 + j;
            if (j < sh.eg && e < E) {
                float v = acc[j];
                for (int s = 1; s < sh.s; ++s) v = __fadd_rn(v, red[((s - 1) * kRtTok + lane) * E + e]);
                logits[static_cast<size_t>(t) * E + e] = v;
            }
        }
    }
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
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const moe::RtShape sh = moe::rt_shape(E);
    const size_t stage = static_cast<size_t>(moe::kRtTok) * (sh.d + 1) + static_cast<size_t>(sh.d) * E;
    const size_t red = static_cast<size_t>(sh.s - 1) * moe::kRtTok * E;
    const size_t smem = (stage > red ? stage : red) * sizeof(float);
    static int configured_for = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {  // up to 32 x 513 + 8192 words: 98 KB
        const int max_smem = static_cast<int>((moe::kRtTok * (moe::kRtMaxD + 1) + 8192) * sizeof(float));
        int rc = moe::set_smem_limit(reinterpret_cast<const void*>(moe::router_logits_kernel<MOE_ACT_BF16>), max_smem);
        if (rc == MOE_OK)
            rc = moe::set_smem_limit(reinterpret_cast<const void*>(moe::router_logits_kernel<MOE_ACT_F16>), max_smem);
        if (rc != MOE_OK) return rc;
        configured_for = dev;
    }
    const dim3 grid((T + moe::kRtTok - 1) / moe::kRtTok);
    if (act == MOE_ACT_BF16)
        moe::launch_pdl(moe::router_logits_kernel<MOE_ACT_BF16>, grid, moe::kRtThreads, smem, st,
                        static_cast<const __nv_bfloat16*>(x), w_router, logits, T, H, E);
    else
        moe::launch_pdl(moe::router_logits_kernel<MOE_ACT_F16>, grid, moe::kRtThreads, smem, st,
                        static_cast<const __half*>(x), w_router, logits, T, H, E);
    moe::count_launch();
    int rc = moe::check_launch("moe_router_topk_softmax (router GEMM)");
    if (rc != MOE_OK) return rc;
    return moe_route_topk_softmax(logits, topk_ids, topk_weights, T, E, top_k, renormalize, stream);
}
