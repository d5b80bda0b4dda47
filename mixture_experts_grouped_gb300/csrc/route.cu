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
