// Dequantisation of the quantised weight formats (GPTQ int4, NVFP4, FP8
// E4M3) into 16-bit MMA operands, shared by the TS forms (weights
// dequantised into TMEM by warps of the CTA): one weight row's 64-deep k block
// at a time, from registers to the 32 TMEM columns it occupies.
#pragma once

#include "gemm_common.cuh"

namespace moe {
namespace gemm {

// ---- number conversions for the quantised formats ---------------------------------

__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(byte));
    return r;
}

// Four E2M1 codes (nibbles 0..3 of w) -> two bf16x2 words, with no
// conversion instructions: a byte permute looks up the high and low byte of
// each magnitude's bf16 value (0, .5, 1, 1.5, 2, 3, 4, 6 -> 0x0000, 0x3F00,
// 0x3F80, 0x3FC0, 0x4000, 0x4040, 0x4080, 0x40C0), a second permute
// interleaves them, and a sign-replicating permute carries each code's sign
// bit (bit 3) to bit 15 of its half.
__device__ __forceinline__ void e2m1x4_to_bf16x4(uint32_t w, uint32_t& p01, uint32_t& p23) {
    const uint32_t sel = w & 0x7777u;
    const uint32_t hi = prmt(0x3F3F3F00u, 0x40404040u, sel);
    const uint32_t lo = prmt(0xC0800000u, 0xC0804000u, sel);
    const uint32_t t = w << 4;  // byte 0 / 1 of t carry the signs of codes 0 / 2 in their top bit
    p01 = prmt(lo, hi, 0x5140u) | (prmt(t, w, 0xC888u) & 0x80008000u);
    p23 = prmt(lo, hi, 0x7362u) | (prmt(t, w, 0xD999u) & 0x80008000u);
}

__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t bits) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(bits));  // (a & mask) | bits
    return r;
}

// One GPTQ weight row for NW words of a k block (8 k values each): word i
// holds the codes of k = 8i .. 8i+7 (4 bits each, k order from the low bits),
// z the zero point and sh the fp16 scale of the row's group. Writes
// (q - z) * s as 4 NW columns of two 16-bit values. fp16: 1024 + q and 1024 + 16q come from the code bits
// by one mask-or each (exact), subtracting the zero point is exact, and the
// product with s is the only rounding.
template <int ACT, bool PERM, int NW = 8>
__device__ __forceinline__ void gptq_row(const uint32_t (&w)[NW], int z, __half sh, uint32_t (&o)[4 * NW]) {
    if (ACT == MOE_ACT_F16) {
        const __half2 s2 = __half2half2(sh);
        const __half2 z1 = __half2half2(__ushort_as_half(static_cast<unsigned short>(0x6400 | z)));      // 1024 + z
        const __half2 c16 = __half2half2(__ushort_as_half(static_cast<unsigned short>(0x2C00)));         // 1/16
        const __half2 nz16 = __half2half2(__ushort_as_half(static_cast<unsigned short>(0xD400 | (z << 4))));  // -(64 + z)
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            const uint32_t w8 = w[i] >> 8;
            uint32_t q[4] = {and_or(w[i], 0x000F000Fu, 0x64006400u),   // (k0, k4): 1024 + q
                             and_or(w[i], 0x00F000F0u, 0x64006400u),   // (k1, k5): 1024 + 16 q
                             and_or(w8, 0x000F000Fu, 0x64006400u),     // (k2, k6)
                             and_or(w8, 0x00F000F0u, 0x64006400u)};    // (k3, k7)
            uint32_t d[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __half2 h = *reinterpret_cast<__half2*>(&q[j]);
                const __half2 qz = (j & 1) ? __hfma2(h, c16, nz16) : __hsub2(h, z1);  // q - z, exact
                __half2 v = __hmul2(qz, s2);
                d[j] = *reinterpret_cast<uint32_t*>(&v);
            }
            if (PERM) {
                o[4 * i + 0] = d[0];
                o[4 * i + 1] = d[1];
                o[4 * i + 2] = d[2];
                o[4 * i + 3] = d[3];
            } else {
                o[4 * i + 0] = prmt(d[0], d[1], 0x5410);  // (k0, k1)
                o[4 * i + 1] = prmt(d[2], d[3], 0x5410);  // (k2, k3)
                o[4 * i + 2] = prmt(d[0], d[1], 0x7632);  // (k4, k5)
                o[4 * i + 3] = prmt(d[2], d[3], 0x7632);  // (k6, k7)
            }
        }
    } else {
        // bf16 activations: (q - z) * s is exact in f32 (a 5-bit integer times
        // an fp16 value) and rounds once to bf16
        const float s = __half2float(sh);
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = static_cast<float>(static_cast<int>((w[i] >> (4 * j)) & 15u) - z) * s;
            if (PERM) {
                o[4 * i + 0] = Act<ACT>::pack2(f[0], f[4]);
                o[4 * i + 1] = Act<ACT>::pack2(f[1], f[5]);
                o[4 * i + 2] = Act<ACT>::pack2(f[2], f[6]);
                o[4 * i + 3] = Act<ACT>::pack2(f[3], f[7]);
            } else {
                o[4 * i + 0] = Act<ACT>::pack2(f[0], f[1]);
                o[4 * i + 1] = Act<ACT>::pack2(f[2], f[3]);
                o[4 * i + 2] = Act<ACT>::pack2(f[4], f[5]);
                o[4 * i + 3] = Act<ACT>::pack2(f[6], f[7]);
            }
        }
    }
}

// The E4M3 block scales sc[0..NS) (one byte each) as scale pairs of the
// activation type, s2[g] = (sc[g], sc[g]): two scales per hardware E4M3 ->
// f16x2 conversion (low byte to the low half), then to bf16 through f32. Every
// E4M3 value is exact in f16 and in bf16 (4 significant bits, exponents 2^-9
// .. 2^8), so both paths are exact.
template <int ACT, int NS>
__device__ __forceinline__ void e4m3_scale_pairs(const uint32_t (&sc)[NS], uint32_t (&s2)[NS]) {
    static_assert(NS % 2 == 0, "scales come in pairs");
#pragma unroll
    for (int g = 0; g < NS; g += 2) {
        uint32_t h;
        asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
            : "=r"(h)
            : "r"(sc[g] | (sc[g + 1] << 8)));
        if (ACT == MOE_ACT_F16) {
            s2[g] = prmt(h, h, 0x1010u);      // low half twice
            s2[g + 1] = prmt(h, h, 0x3232u);  // high half twice
        } else {
            const float lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xffffu)));
            const float hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
            s2[g] = Act<MOE_ACT_BF16>::pack2(lo, lo);
            s2[g + 1] = Act<MOE_ACT_BF16>::pack2(hi, hi);
        }
    }
}

// One NVFP4 weight row for NW words of a k block: word i holds the E2M1 codes
// of k = 8i .. 8i+7 (low nibble first), sc[g] the E4M3 scale of k = 16g ..
// 16g+15. E2M1 x E4M3 products are exact in bf16 and fp16.
template <int ACT, int NW = 8>
__device__ __forceinline__ void nvfp4_row(const uint32_t (&w)[NW], const uint32_t (&sc)[NW / 2],
                                          uint32_t (&o)[4 * NW]) {
    uint32_t s2w[NW / 2];
    e4m3_scale_pairs<ACT, NW / 2>(sc, s2w);
#pragma unroll
    for (int g = 0; g < NW / 2; ++g) {
        if (ACT == MOE_ACT_BF16) {
            const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162*>(&s2w[g]);
#pragma unroll
            for (int ii = 0; ii < 2; ++ii) {
                const int i = 2 * g + ii;
                uint32_t a[4];
                e2m1x4_to_bf16x4(w[i], a[0], a[1]);
                e2m1x4_to_bf16x4(w[i] >> 16, a[2], a[3]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    __nv_bfloat162 v = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&a[j]), s2);
                    o[4 * i + j] = *reinterpret_cast<uint32_t*>(&v);
                }
            }
        } else {
            const __half2 s2 = *reinterpret_cast<const __half2*>(&s2w[g]);
#pragma unroll
            for (int ii = 0; ii < 2; ++ii) {
                const int i = 2 * g + ii;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t e2 = e2m1x2_to_f16x2((w[i] >> (8 * j)) & 0xffu);
                    __half2 v = __hmul2(*reinterpret_cast<__half2*>(&e2), s2);
                    o[4 * i + j] = *reinterpret_cast<uint32_t*>(&v);
                }
            }
        }
    }
}

// One FP8 weight row for a k block: word i holds the E4M3 codes of k = 4i ..
// 4i+3 (lowest byte first). Writes the codes' values unscaled (the row scale
// multiplies the f32 accumulator in the epilogue) as 32 columns of two 16-bit
// values: E4M3 -> f16 is one exact conversion per pair, and every E4M3 value
// is also exact in bf16 (4 significant bits, exponents 2^-9 .. 2^8).
template <int ACT>
__device__ __forceinline__ void fp8_row(const uint32_t (&w)[16], uint32_t (&o)[32]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        uint32_t lo, hi;  // (k 4i, 4i+1), (k 4i+2, 4i+3) as f16x2
        asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
            "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
            : "=r"(lo), "=r"(hi) : "r"(w[i]));
        if (ACT == MOE_ACT_F16) {
            o[2 * i] = lo;
            o[2 * i + 1] = hi;
        } else {
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
            o[2 * i] = Act<ACT>::pack2(a.x, a.y);
            o[2 * i + 1] = Act<ACT>::pack2(b.x, b.y);
        }
    }
}

}  // namespace gemm
}  // namespace moe
