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
//   * Four kernel forms, chosen on the host from the average rows per touched
//     expert and the weight format:
//       - bf16 prefill (>= 128 rows per expert): grouped_gemm_pair_kernel, a
//         cluster of two CTAs issuing tcgen05.mma.cta_group::2 with M=256
//         weight rows (128 per CTA) and N = up to 256 activation rows of one
//         expert (N/2 per CTA);
//       - bf16 decode: grouped_gemm_decode_kernel, operands swapped: each
//         weight half is an M=128 operand and NTOK tokens (16..128, one align
//         block) the N operand;
//       - NVFP4 / FP8 prefill: grouped_gemm_tspair_kernel, CTA pairs again,
//         each CTA dequantising its 128 weight rows into its own TMEM as the
//         A operand of M=256 MMAs, N = up to 192 activation rows;
//       - GPTQ (any size) and NVFP4 / FP8 decode: grouped_gemm_ts_kernel,
//         weights dequantised by eight or sixteen warps into TMEM and used as
//         the M=128 A operand, NTOK tokens (128 for GPTQ prefill) the N operand
//         from shared memory.
//   * Roles: TMA producer warps feed multi-stage rings; MMA issues go to
//     double-buffered TMEM accumulators where TMEM allows; four epilogue warps
//     drain them (tcgen05.ld -> activation -> global).
//   * Every mbarrier wait is bounded; on a timeout the CTA records
//     MOE_DEV_ERR_TIMEOUT, lets in-flight copies and MMAs land, frees TMEM and
//     returns.
#include "gemm_common.cuh"

namespace moe {
namespace gemm {
namespace {

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

// Activation rows per tile. 0 selects the prefill forms (CTA pairs, each
// expert's valid rows as the MMA's N operand), used when experts average 128
// or more rows. Otherwise the decode form takes one align block per tile
// (rounded up to a power of two, at least 16): spans are whole blocks and
// only a span's last block holds padding, so no tile is padding only and the
// tiles spread evenly over the CTAs.
int pick_ntok(long P, int E, int block_size) {
    const long touched = P < E ? P : E;
    const long avg = touched > 0 ? P / touched : 0;
    if (avg >= 128) return 0;
    int nt = 16;
    while (nt < block_size) nt <<= 1;
    return nt <= 128 ? nt : 0;
}

template <int MODE>
int dispatch(int wfmt, int act, int ntok, const Maps& m, const GemmParams& p, cudaStream_t st, const char* who) {
    if (wfmt == MOE_W_BF16) {
        if (ntok == 0) return launch_pair_form(MODE, m, p, st, who);
        return launch_decode_form(MODE, ntok, m, p, st, who);
    }
    if (ntok == 0) {
        // quantised prefill on CTA pairs; 256-row tiles once experts average 176
        // rows or more (beyond 192 a 192-row cap would cut most experts in two)
        const long touched = p.P < p.E ? p.P : p.E;
        const int wide = touched > 0 && p.P / touched >= 176;
        return launch_tspair_form(MODE, wfmt, act, wide, m, p, st, who);
    }
    return launch_ts_form(MODE, wfmt, act, ntok, m, p, st, who);
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
            int rc = MOE_OK;
            // (q0 / q1 / q2: the same tensors in the TS pair form's 128-column boxes per
            // CTA, 64 gate and 64 up columns for gate/up)
            for (int pass = 0; pass < 2 && rc == MOE_OK; ++pass) {
                const uint32_t b = pass == 0 ? hc : hc / 2;  // columns per half (gate/up) in the box
                CUtensorMap* t0 = pass == 0 ? &m.r0 : &m.q0;
                CUtensorMap* t1 = pass == 0 ? &m.r1 : &m.q1;
                CUtensorMap* t2 = pass == 0 ? &m.r2 : &m.q2;
                if (N == 2 * n_out) {
                    const uint64_t I = n_out;
                    rc = make_tmap_3d_raw(t0, w->w, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, I, 2, kq, I * 4, 2 * I * 4, b, 2,
                                          16);
                    if (rc == MOE_OK)
                        rc = make_tmap_3d_raw(t1, w->scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, I, 2, kg, I * 2,
                                              2 * I * 2, b, 2, sg);
                    if (rc == MOE_OK)
                        rc = make_tmap_3d_raw(t2, w->zeros, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, I / 8, 2, kg, I / 8 * 4,
                                              2 * I / 8 * 4, b / 8, 2, sg);
                } else {
                    rc = make_tmap_2d_raw(t0, w->w, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, kq, N, 2 * b, 16);
                    if (rc == MOE_OK)
                        rc = make_tmap_2d_raw(t1, w->scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, kg, N, 2 * b, sg);
                    if (rc == MOE_OK)
                        rc = make_tmap_2d_raw(t2, w->zeros, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, kg, N / 8, 2 * b / 8, sg);
                }
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
            // The TS pair form takes 128 rows per CTA: 64 gate and 64 up rows, or
            // 128 down rows (q0 / q1: the same tensors in those boxes).
            if (N == 2 * n_out) {
                const uint64_t I = n_out;
                rc = make_tmap_3d_raw(&m.r0, w->w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, I,
                                      2 * static_cast<uint64_t>(E), K / 2, I * (K / 2), 64, hc, 2);
                if (rc == MOE_OK)
                    rc = make_tmap_3d_raw(&m.r1, w->scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, I, 2, kg, I, 2 * I, hc,
                                          2, 8);
                if (rc == MOE_OK)
                    rc = make_tmap_3d_raw(&m.q0, w->w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, I,
                                          2 * static_cast<uint64_t>(E), K / 2, I * (K / 2), 64, hc / 2, 2);
                if (rc == MOE_OK)
                    rc = make_tmap_3d_raw(&m.q1, w->scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, I, 2, kg, I, 2 * I,
                                          hc / 2, 2, 8);
            } else {
                rc = make_tmap_2d_raw(&m.r0, w->w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, static_cast<uint64_t>(E) * N,
                                      K / 2, 64, dc);
                if (rc == MOE_OK) rc = make_tmap_2d_raw(&m.r1, w->scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kg, N, dc, 8);
                if (rc == MOE_OK)
                    rc = make_tmap_2d_raw(&m.q0, w->w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, static_cast<uint64_t>(E) * N,
                                          K / 2, 64, hc);
                if (rc == MOE_OK) rc = make_tmap_2d_raw(&m.q1, w->scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kg, N, hc, 8);
            }
            m.r2 = m.r1;
            m.q2 = m.q1;
            m.w = m.r0;
            return rc;
        }
        case MOE_W_FP8_E4M3: {
            MOE_REQUIRE(w->w && w->scales, "%s: FP8 codes / scales must be non-NULL", who);
            MOE_REQUIRE(K % 16 == 0, "%s: FP8 needs K=%d divisible by 16", who, K);
            // one copy per 64-deep raw stage: a 3-D map over the gate and up
            // halves for gate/up, a 256-row box for down
            int rc;
            // (q0: the same codes in the TS pair form's 128-row boxes per CTA)
            if (N == 2 * n_out) {
                const uint64_t I = n_out;
                rc = make_tmap_3d_raw(&m.r0, w->w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, I, 2 * static_cast<uint64_t>(E),
                                      K, I * K, 64, hc, 2);
                if (rc == MOE_OK)
                    rc = make_tmap_3d_raw(&m.q0, w->w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, I,
                                          2 * static_cast<uint64_t>(E), K, I * K, 64, hc / 2, 2);
            } else {
                rc = make_tmap_2d_raw(&m.r0, w->w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, static_cast<uint64_t>(E) * N, K,
                                      64, dc);
                if (rc == MOE_OK)
                    rc = make_tmap_2d_raw(&m.q0, w->w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, static_cast<uint64_t>(E) * N,
                                          K, 64, hc);
            }
            m.r1 = m.r2 = m.r0;
            m.q1 = m.q2 = m.q0;
            m.w = m.r0;
            return rc;
        }
        default:
            return fail(MOE_ERR_INVALID, "%s: unknown weight format %d", who, w->format);
    }
}
}  // namespace
}  // namespace gemm
}  // namespace moe

namespace moe {
namespace gemm {
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
}  // namespace gemm
}  // namespace moe

extern "C" size_t moe_gate_up_workspace_size(int32_t max_padded, int32_t H) {
    if (max_padded < 0 || H < 0) return 0;
    return moe::gemm::gather_bytes(max_padded, H) + MOE_SPLITK_BYTES;
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
    const int ntok = moe::gemm::pick_ntok(P, E, block_size);
    moe::gemm::Maps m;
    int rc = moe::gemm::weight_maps(w_gate_up, act, E, 2 * I, H, I, m, who);
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
        moe::launch_pdl(moe::gemm::gather_rows_kernel, blocks, 256, 0, st, static_cast<const uint4*>(x), sorted_token_ids,
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
    moe::gemm::GemmParams p{};
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
    p.sk_gen = static_cast<int>(moe::next_splitk_gen());
    p.block_size = block_size;
    moe::gemm::set_splitk(p, static_cast<uint8_t*>(workspace) + moe::gemm::gather_bytes(max_padded, H));
    return moe::gemm::dispatch<moe::gemm::MODE_GATE_UP>(w_gate_up->format, act, ntok, m, p, st, who);
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
    const int ntok = moe::gemm::pick_ntok(P, E, block_size);
    moe::gemm::Maps m;
    int rc = moe::gemm::weight_maps(w_down, act, E, H, I, H, m, who);
    if (rc != MOE_OK) return rc;
    if (max_padded == 0) return MOE_OK;
    MOE_REQUIRE(h && sorted_token_ids && expert_offsets && y, "%s: NULL pointer", who);
    MOE_REQUIRE(moe::aligned16(h) && moe::aligned16(y), "%s: h / y must be 16-byte aligned", who);
    MOE_REQUIRE(workspace && workspace_bytes >= MOE_SPLITK_BYTES && (reinterpret_cast<uintptr_t>(workspace) & 127) == 0,
                "%s: workspace of %zu bytes (128-byte aligned) required, got %zu", who,
                static_cast<size_t>(MOE_SPLITK_BYTES), workspace_bytes);
    rc = moe::make_tmap_2d(&m.x, h, max_padded, I, ntok ? ntok : 128, act);
    if (rc != MOE_OK) return rc;
    moe::gemm::GemmParams p{};
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
    p.sk_gen = static_cast<int>(moe::next_splitk_gen());
    p.block_size = block_size;
    moe::gemm::set_splitk(p, workspace);
    return moe::gemm::dispatch<moe::gemm::MODE_DOWN>(w_down->format, act, ntok, m, p, static_cast<cudaStream_t>(stream), who);
}
