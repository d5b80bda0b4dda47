// Step a6: the weighted top-k combine.
//
// Restates ferrum-kernels 0.7.7 src/backend/cuda/moe.rs, moe_combine:
// out[t, :] = sum_j w[t, j] * y[pairs_by_token[t * k + j], :], with the pair ->
// row map written by the align step. HBM-bound: every thread moves 16-byte
// vectors (8 activations), a block covers 2048 columns of one token, and the
// k expert rows of a token are read once each.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

template <int ACT>
__global__ void __launch_bounds__(kThreads)
combine_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ pair_to_row, const float* __restrict__ w,
               uint4* __restrict__ out, int H, int top_k, int max_padded, int32_t* err) {
    pdl_wait();
    const int t = blockIdx.y;
    const int v = blockIdx.x * kThreads + threadIdx.x;  // 16-byte vector index in the row
    const int vpr = H / 8;
    if (v >= vpr) return;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j = 0; j < top_k; ++j) {
        const int r = __ldg(pair_to_row + static_cast<size_t>(t) * top_k + j);
        if (r < 0) continue;
        if (r >= max_padded) {
            if (v == 0) set_err(err, MOE_DEV_ERR_PAIR_ID);
            continue;
        }
        const float wt = __ldg(w + static_cast<size_t>(t) * top_k + j);
        const uint4 yv = __ldg(y + static_cast<size_t>(r) * vpr + v);
        const uint32_t yw[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = Act<ACT>::unpack2(yw[q]);
            acc[2 * q] = fmaf(wt, f.x, acc[2 * q]);
            acc[2 * q + 1] = fmaf(wt, f.y, acc[2 * q + 1]);
        }
    }
    uint4 o;
    o.x = Act<ACT>::pack2(acc[0], acc[1]);
    o.y = Act<ACT>::pack2(acc[2], acc[3]);
    o.z = Act<ACT>::pack2(acc[4], acc[5]);
    o.w = Act<ACT>::pack2(acc[6], acc[7]);
    out[static_cast<size_t>(t) * vpr + v] = o;
}

}  // namespace
}  // namespace moe

extern "C" int moe_combine(const void* y, int32_t act, const int32_t* pair_to_row, const float* topk_weights,
                           void* out, int32_t T, int32_t H, int32_t top_k, int32_t max_padded, int32_t* err_word,
                           void* stream) {
    const char* who = "moe_combine";
    MOE_REQUIRE(act == MOE_ACT_BF16 || act == MOE_ACT_F16, "%s: unknown activation type %d", who, act);
    MOE_REQUIRE(T >= 0 && top_k >= 1 && max_padded >= 0, "%s: bad T=%d / top_k=%d / max_padded=%d", who, T, top_k,
                max_padded);
    MOE_REQUIRE(H > 0 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", who, H);
    MOE_REQUIRE(T <= 65535 * 16, "%s: T=%d too large", who, T);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(y && pair_to_row && topk_weights && out, "%s: NULL pointer", who);
    MOE_REQUIRE(moe::aligned16(y) && moe::aligned16(out), "%s: y / out must be 16-byte aligned", who);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int launches = 0;
    // grid.y is limited to 65535: split very long token ranges
    for (int t0 = 0; t0 < T; t0 += 65535) {
        const int nt = (T - t0) < 65535 ? (T - t0) : 65535;
        dim3 grid((H / 8 + moe::kThreads - 1) / moe::kThreads, nt);
        const size_t vrow = static_cast<size_t>(H) / 8;
        const uint4* yv = static_cast<const uint4*>(y);
        uint4* ov = static_cast<uint4*>(out) + static_cast<size_t>(t0) * vrow;
        const int32_t* pr = pair_to_row + static_cast<size_t>(t0) * top_k;
        const float* wt = topk_weights + static_cast<size_t>(t0) * top_k;
        if (act == MOE_ACT_BF16)
            moe::launch_pdl(moe::combine_kernel<MOE_ACT_BF16>, grid, moe::kThreads, 0, st, yv, pr, wt, ov, H, top_k, max_padded,
                                                                             err_word);
        else
            moe::launch_pdl(moe::combine_kernel<MOE_ACT_F16>, grid, moe::kThreads, 0, st, yv, pr, wt, ov, H, top_k, max_padded,
                                                                            err_word);
        ++launches;
    }
    moe::count_launch(launches);
    return moe::check_launch(who);
}
