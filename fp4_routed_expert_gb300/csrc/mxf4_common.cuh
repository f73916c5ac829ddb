// mxf4_common.cuh -- pieces shared by the tensor-core expert FFN kernels (sm_103a): tcgen05 /
// TMEM wrappers, the MXFP4 multi-term quantisers of activations and the prefill activation
// block layout.
#pragma once

#include <cuda_fp16.h>

#include "moe_internal.cuh"

namespace fp4moe {

constexpr int kTerms = 4;
constexpr int kBM = 128;              // weight rows per tile
constexpr int kKB = 256;              // K elements per K block
constexpr int kKBytes = 128;          // code bytes per row per stage
constexpr int kMaxEpiWarps = 8;                    // epilogue warps at most: two per TMEM lane quarter
constexpr int kTmemCols = 512;
constexpr int kSfRing = 2;                // scale buffers in TMEM (tcgen05.cp and MMAs run in issue order)
constexpr int kDecodeNT = 16;             // decode tile rows at most: the tokens of x; a key's pairs of h
constexpr int kMaxDecodePairs = kTcDecodeMaxKeys;   // decode calls on the tensor cores: T*k <= 128


// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major operand tile, 128-byte rows, SWIZZLE_128B, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t a) {
    return (uint64_t)((a & 0x3FFFF) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// Scale atom: 32 rows of 16 bytes, no swizzle, core matrices (8 rows) 128 bytes apart.
__device__ __forceinline__ uint64_t desc_sf(uint32_t a) {
    return (uint64_t)((a & 0x3FFFF) >> 4) | ((uint64_t)(128 >> 4) << 32) | (1ull << 46);
}
// Instruction descriptor of kind::mxf4 (e2m1 x e2m1, UE8M0 scales, K-major A and B).
// sf_id selects the first of the two scale bytes used by one K=64 MMA: 0 or 2.
__device__ __forceinline__ uint32_t idesc_mxf4(int n, int sf_id) {
    return ((uint32_t)(sf_id & 3) << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
           ((uint32_t)(kBM >> 4) << 24) | ((uint32_t)(sf_id & 3) << 29);
}
__device__ __forceinline__ void mma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// Asynchronous 32x32b.x16 / .x8 loads: the registers are valid only after tc_wait_ld on them
// (the wait takes them as operands, so no use can be scheduled before it).
__device__ __forceinline__ void tc_ld_issue(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}
// 16x256b.x4 (16 TMEM lanes, 32 columns): thread i receives, for column group g = 0..3,
// r[4g], r[4g+1] = lane i/4, columns 8g + 2(i%4) + {0, 1}, and r[4g+2], r[4g+3] = lane 8 + i/4,
// the same columns (checked on GB300 against 32x32b stores).
__device__ __forceinline__ void tc_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_ld_issue(uint32_t taddr, uint32_t (&r)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld(uint32_t (&r)[4]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]) : : "memory");
}
__device__ __forceinline__ void tc_ld_issue(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld(uint32_t (&r)[8]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
                 :
                 : "memory");
}

// ------------------------------------------------------------------ MXFP4 multi-term quantiser

// Term t of a 32-element block takes the residual r left by terms 0..t-1: scale 2^e with e the
// smallest integer such that max|r| <= 6 * 2^e (clamped to the UE8M0 range; a block whose
// residual maximum is subnormal or zero gets e = -127 and all-zero codes), codes = r / 2^e
// rounded to the nearest e2m1 value (ties to even: the hardware conversion), and the next
// residual is r minus the coded value (exact).  From the block maximum's bit pattern: the
// scale byte, 2^-e (0 when e = -127) and 2^e.
__device__ __forceinline__ void term_scale(uint32_t amax_bits, uint32_t& sc, float& inv, float& scl) {
    int e = -127;
    if ((amax_bits >> 23) != 0u) {                                   // normal amax
        const int e0 = (int)((amax_bits >> 23) & 0xFF) - 127;        // floor(log2 amax)
        const float m = __uint_as_float((amax_bits & 0x007FFFFFu) | 0x3F800000u);   // amax / 2^e0 in [1, 2)
        e = (m <= 1.5f) ? e0 - 2 : e0 - 1;                           // amax <= 6 * 2^e, minimal e
    }
    e = max(-127, min(127, e));
    sc = (uint32_t)(e + 127);
    inv = (e >= -126 && e <= 126) ? __uint_as_float((uint32_t)(127 - e) << 23) : 0.f;   // 2^-e
    scl = (e >= -126) ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// Two values (|q| <= 6) -> one byte of e2m1 codes (lo in the low nibble), nearest with ties to
// even, and the two coded values.
__device__ __forceinline__ uint32_t e2m1x2_code(float lo, float hi, float& vlo, float& vhi) {
    uint32_t byte, h2;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %2, %3;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, t;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(byte), "=r"(h2)
        : "f"(hi), "f"(lo));
    float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
    vlo = f.x;
    vhi = f.y;
    return byte;
}

// One warp quantises one 32-element block (lane i holds element i) into kTerms MXFP4 terms.
// Every lane receives the 16 code bytes of every term in codes[t] and the scale bytes.
__device__ __forceinline__ void warp_quantize32(float v, int lane, uint4* codes /*[kTerms]*/,
                                                uint32_t* scales /*[kTerms]*/) {
#pragma unroll
    for (int t = 0; t < kTerms; ++t) {
        // max |v| over the warp: magnitudes order like their bit patterns as unsigned integers
        const uint32_t u = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
        float inv, scl;
        term_scale(u, scales[t], inv, scl);
        // lanes 2i and 2i+1 code their pair together; the even lane holds the byte
        const float q = v * inv, qn = __shfl_xor_sync(0xffffffffu, q, 1);
        float vlo, vhi;
        const uint32_t byte = e2m1x2_code((lane & 1) ? qn : q, (lane & 1) ? q : qn, vlo, vhi);
        v -= ((lane & 1) ? vhi : vlo) * scl;
        uint32_t w = (lane & 1) ? 0u : byte << (8 * ((lane >> 1) & 3));
        w |= __shfl_xor_sync(0xffffffffu, w, 1);
        w |= __shfl_xor_sync(0xffffffffu, w, 2);
        w |= __shfl_xor_sync(0xffffffffu, w, 4);                     // lanes 8w..8w+7 hold word w
        const uint32_t w1 = __shfl_sync(0xffffffffu, w, 8), w2 = __shfl_sync(0xffffffffu, w, 16),
                       w3 = __shfl_sync(0xffffffffu, w, 24);
        codes[t] = make_uint4(w, w1, w2, w3);
    }
}

// The same quantisation by one thread for the 32 values v (registers): the code words of term
// t in w[t][0..3] (element i in word i/8, nibble i%8), its scale byte in sc[t].
__device__ __forceinline__ void thread_quantize32(float (&v)[32], uint32_t (&w)[kTerms][4], uint32_t (&sc)[kTerms]) {
#pragma unroll
    for (int t = 0; t < kTerms; ++t) {
        // max |v| as a tree (five dependent steps rather than 32)
        float m[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) m[i] = fmaxf(fabsf(v[i]), fabsf(v[i + 16]));
#pragma unroll
        for (int w2 = 8; w2 > 0; w2 >>= 1)
#pragma unroll
            for (int i = 0; i < w2; ++i) m[i] = fmaxf(m[i], m[i + w2]);
        float inv, scl;
        term_scale(__float_as_uint(m[0]), sc[t], inv, scl);
#pragma unroll
        for (int k = 0; k < 4; ++k) w[t][k] = 0u;
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            float vlo, vhi;
            const uint32_t byte = e2m1x2_code(v[i] * inv, v[i + 1] * inv, vlo, vhi);
            v[i] -= vlo * scl;
            v[i + 1] -= vhi * scl;
            w[t][i >> 3] |= byte << (4 * (i & 7));
        }
    }
}

// The same quantisation by the 8 lanes of an octet (lanes 8o..8o+7 of a warp; lane s = lane & 7
// holds elements 4s..4s+3 in v): the 32-bit code word w = s/2 of term t (elements 8w..8w+7)
// lands in word[t] of the even lane s = 2w, every lane of the octet gets the scale bytes.  The
// whole warp calls it (the shuffles stay inside each octet).
__device__ __forceinline__ void octet_quantize32(float (&v)[4], int lane, uint32_t (&word)[kTerms],
                                                 uint32_t (&sc)[kTerms]) {
#pragma unroll
    for (int t = 0; t < kTerms; ++t) {
        uint32_t u = __float_as_uint(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
        u = max(u, __shfl_xor_sync(0xffffffffu, u, 1));
        u = max(u, __shfl_xor_sync(0xffffffffu, u, 2));
        u = max(u, __shfl_xor_sync(0xffffffffu, u, 4));
        float inv, scl;
        term_scale(u, sc[t], inv, scl);
        float a0, a1, b0, b1;
        const uint32_t lo = e2m1x2_code(v[0] * inv, v[1] * inv, a0, a1);
        const uint32_t hi = e2m1x2_code(v[2] * inv, v[3] * inv, b0, b1);
        v[0] -= a0 * scl;
        v[1] -= a1 * scl;
        v[2] -= b0 * scl;
        v[3] -= b1 * scl;
        // elements 4s..4s+3 are nibbles 4(s&1).. of word s/2
        const uint32_t half = lo | (hi << 8);
        const uint32_t other = __shfl_xor_sync(0xffffffffu, half, 1);
        word[t] = (lane & 1) ? 0u : (half | (other << 16));
    }
}

// Padded index of h value i (0..63) of column c in the gate/up epilogue's shared tile: the
// 32-value blocks start 33 words apart, so threads reading one block each hit distinct banks.
__device__ __forceinline__ int hidx(int c, int i) { return c * 66 + (i >> 5) * 33 + (i & 31); }

// Activation operands are kept in blocks: block (tile t, K block kb) holds the kTerms x NT
// rows of B (row r' = term*NT + row, codes pre-swizzled, 128 bytes per row) followed by their
// scale atoms, 1 KB per 128 rows of r'; the KB blocks of a tile are consecutive.
__host__ __device__ constexpr int act_block_bytes(int NT) { return kTerms * NT * 128 + (kTerms * NT + 127) / 128 * 1024; }
__device__ __forceinline__ int64_t act_code_off(int tile, int kb, int term, int row, int chunk, int NT, int KB) {
    return ((int64_t)tile * KB + kb) * act_block_bytes(NT) + (term * NT + row) * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}
__device__ __forceinline__ int64_t act_scale_off(int tile, int kb, int term, int row, int j /*0..7*/, int NT, int KB) {
    const int rr = term * NT + row;
    const int r = rr & 127;
    return ((int64_t)tile * KB + kb) * act_block_bytes(NT) + kTerms * NT * 128 + (rr >> 7) * 1024 + (j >> 2) * 512 +
           (r & 31) * 16 + (r >> 5) * 4 + (j & 3);
}

}  // namespace fp4moe
