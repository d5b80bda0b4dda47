// Host-side services of libmoe.so: error messages, launch accounting, device
// properties, TMA descriptor encoding and the grouped-array validation rules.
#include <cudaTypedefs.h>
#include <stdarg.h>
#include <stdio.h>

#include <mutex>
#include <vector>

#include "common.cuh"

namespace moe {

namespace {
thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}
}  // namespace

int fail(int status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

int check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    return MOE_OK;
}

void count_launch(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

// Split-K generation: a nonzero number per GEMM call, process-wide. The
// decode form's piece holders store it in their flags and owners accept only
// their own call's number.
static std::atomic<uint32_t> g_splitk_gen{0};
uint32_t next_splitk_gen() {
    uint32_t v = g_splitk_gen.fetch_add(1, std::memory_order_relaxed) + 1;
    while (v == 0) v = g_splitk_gen.fetch_add(1, std::memory_order_relaxed) + 1;
    return v;
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

int set_smem_limit(const void* kernel, int bytes) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess)
        return fail(MOE_ERR_CUDA, "cudaFuncSetAttribute(%d bytes of shared memory): %s", bytes,
                    cudaGetErrorString(e));
    return MOE_OK;
}

int make_tmap_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 int act) {
    auto fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    if (!aligned16(base)) return fail(MOE_ERR_INVALID, "tensor base address %p is not 16-byte aligned", base);
    if ((cols * 2) % 16 != 0) return fail(MOE_ERR_INVALID, "row pitch of %llu elements is not a 16-byte multiple",
                                          (unsigned long long)cols);
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, act == MOE_ACT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MOE_ERR_INVALID, "cuTensorMapEncodeTiled failed (%d) for a %llux%llu tensor", (int)r,
                    (unsigned long long)rows, (unsigned long long)cols);
    return MOE_OK;
}

int make_tmap_2d_raw(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t rows,
                     uint64_t cols, uint32_t box_cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    if (!aligned16(base)) return fail(MOE_ERR_INVALID, "tensor base address %p is not 16-byte aligned", base);
    if ((cols * elem_bytes) % 16 != 0)
        return fail(MOE_ERR_INVALID, "row pitch of %llu x %d bytes is not a 16-byte multiple",
                    (unsigned long long)cols, elem_bytes);
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * static_cast<uint64_t>(elem_bytes)};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MOE_ERR_INVALID, "cuTensorMapEncodeTiled failed (%d) for a %llux%llu tensor", (int)r,
                    (unsigned long long)rows, (unsigned long long)cols);
    return MOE_OK;
}

int make_tmap_5d(CUtensorMap* map, const void* base, int act, const uint64_t (&d)[5], const uint64_t (&st)[4],
                 const uint32_t (&b)[5]) {
    auto fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    if (!aligned16(base)) return fail(MOE_ERR_INVALID, "tensor base address %p is not 16-byte aligned", base);
    for (int i = 0; i < 4; ++i)
        if (st[i] % 16 != 0)
            return fail(MOE_ERR_INVALID, "tensor stride %llu is not a 16-byte multiple", (unsigned long long)st[i]);
    cuuint64_t dims[5] = {d[0], d[1], d[2], d[3], d[4]};
    cuuint64_t strides[4] = {st[0], st[1], st[2], st[3]};
    cuuint32_t box[5] = {b[0], b[1], b[2], b[3], b[4]};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(map, act == MOE_ACT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MOE_ERR_INVALID, "cuTensorMapEncodeTiled failed (%d) for a 5-D map", (int)r);
    return MOE_OK;
}

int make_tmap_3d_raw(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t d0,
                     uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
    auto fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    if (!aligned16(base)) return fail(MOE_ERR_INVALID, "tensor base address %p is not 16-byte aligned", base);
    if (s1 % 16 != 0 || s2 % 16 != 0)
        return fail(MOE_ERR_INVALID, "tensor strides %llu / %llu bytes are not 16-byte multiples",
                    (unsigned long long)s1, (unsigned long long)s2);
    (void)elem_bytes;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MOE_ERR_INVALID, "cuTensorMapEncodeTiled failed (%d) for a %llux%llux%llu tensor", (int)r,
                    (unsigned long long)d0, (unsigned long long)d1, (unsigned long long)d2);
    return MOE_OK;
}

}  // namespace moe

extern "C" {

const char* moe_last_error(void) { return moe::g_last_error.c_str(); }

uint64_t moe_launch_count(void) { return moe::g_launches.load(std::memory_order_relaxed); }

uint64_t moe_set_wait_limit_ns(uint64_t ns) {
    return moe::g_wait_limit_ns.exchange(ns ? ns : moe::kWaitLimitNs, std::memory_order_relaxed);
}

int64_t moe_align_capacity(int64_t P, int32_t E, int32_t block_size) {
    if (P < 0 || E < 1 || block_size < 1) return -1;
    const int64_t nonempty = P < E ? P : E;
    const int64_t raw = P + nonempty * (block_size - 1);
    return (raw + block_size - 1) / block_size * block_size;
}

int moe_validate_group_arrays(const char* who, int32_t num_experts, const int32_t* offsets, int32_t offsets_len,
                              const char* const* names, const int32_t* lens, int32_t n_arrays) {
    if (!who) who = "grouped launch";
    if (num_experts < 0) return moe::fail(MOE_ERR_INVALID, "%s: num_experts %d is negative", who, num_experts);
    if (offsets_len != num_experts + 1)
        return moe::fail(MOE_ERR_INVALID, "%s: expert_offsets len %d != num_experts+1 %d", who, offsets_len,
                         num_experts + 1);
    if (n_arrays > 0 && (!names || !lens)) return moe::fail(MOE_ERR_INVALID, "%s: NULL per-expert arrays", who);
    for (int32_t i = 0; i < n_arrays; ++i) {
        if (lens[i] != num_experts)
            return moe::fail(MOE_ERR_INVALID, "%s: %s len %d != num_experts %d", who, names[i] ? names[i] : "?",
                             lens[i], num_experts);
    }
    if (!offsets) return moe::fail(MOE_ERR_INVALID, "%s: expert_offsets is NULL", who);
    if (offsets[0] < 0) return moe::fail(MOE_ERR_INVALID, "%s: expert_offsets[0] = %d is negative", who, offsets[0]);
    for (int32_t i = 0; i + 1 < offsets_len; ++i) {
        if (offsets[i + 1] < offsets[i])
            return moe::fail(MOE_ERR_INVALID,
                             "%s: expert_offsets is not non-decreasing (%d then %d): a group would have a "
                             "negative row count",
                             who, offsets[i], offsets[i + 1]);
    }
    return MOE_OK;
}

}  // extern "C"
