// mxf4_gemm.cu -- expert FFN on the 5th-generation tensor cores (sm_103a): grouped
// block-scaled MXFP4 GEMMs with tcgen05.mma (kind::mxf4), TMEM accumulators, TMA operand
// loads and fused epilogues.
//
// Operands.  A = expert weight rows straight from the slot arena: e2m1 codes and UE8M0
// scales per 32 K elements, exactly the checkpoint's format ("DeepSeek-V4.1-Flash on a
// single NVIDIA DGX Spark", "Why it is built this way": FP4 + UE8M0/32, never requantised).
// B = activations, written by this library as a sum of kTerms MXFP4 tensors
// (x ~ q_1 + q_2 + ..., each q_i e2m1 codes with its own UE8M0 scale per 32 elements, q_i
// quantising the residual left by q_1..q_(i-1)); the MMA accumulates every term into the same
// fp32 accumulator, so D = W . x up to the residual after kTerms terms.
//
// One persistent kernel, one CTA per SM, 7 warps:
//   warp 0  TMA producer: weight tile (128 rows x 128 bytes) and kTerms activation tiles
//           (NT rows x 128 bytes) per 256-element K block, SWIZZLE_128B
//   warp 1  scale stager: gathers the 8 scale bytes per row of both operands and writes
//           them in the 512-byte tensor-memory scale atom layout
//   warp 2  MMA issuer (one lane): tcgen05.cp of the scale atoms, 4 x kTerms MMAs per
//           K block, tcgen05.commit to release smem stages and publish accumulators
//   warps 3-6  epilogue: tcgen05.ld of the accumulator (double-buffered in TMEM), then
//           gate/up: SwiGLU + requantisation of h into kTerms MXFP4 terms for the down GEMM
//           down:    fp32 rows for the fixed-order combine
// Every wait is bounded; a timeout sets MOE_STATUS_TIMEOUT and the CTA drains and exits.
#include <cuda.h>

#include "moe_internal.cuh"

namespace fp4moe {

constexpr int kTerms = 4;
constexpr int kBM = 128;              // weight rows per tile
constexpr int kKB = 256;              // K elements per stage
constexpr int kKBytes = 128;          // code bytes per row per stage
constexpr int kThreadsGemm = 7 * 32;
constexpr unsigned kSpinLimit = 1u << 25;
constexpr int kTmemCols = 512;
constexpr int kSfCols = 8 + 8 * kTerms;   // scale columns per stage in TMEM (A: 2 atoms, B: 2 per term)
constexpr int kSfRing = 2;

enum { kModeGateUp = 0, kModeDown = 1 };
enum { kRegimeDecode = 0, kRegimePrefill = 1 };

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(done)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return done != 0;
}
// Bounded wait: false after kSpinLimit polls or once another warp has aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    for (unsigned i = 0; i < kSpinLimit; ++i) {
        if (mbar_try(bar, parity)) return true;
        if ((i & 1023u) == 1023u && *abort_flag) return false;
    }
    return false;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
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
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------ MXFP4 multi-term quantiser

// Nearest e2m1 magnitude code of |v| <= 6 (0, .5, 1, 1.5, 2, 3, 4, 6).
__device__ __forceinline__ uint32_t e2m1_mag_code(float a) {
    return (a >= 0.25f) + (a >= 0.75f) + (a >= 1.25f) + (a >= 1.75f) + (a >= 2.5f) + (a >= 3.5f) + (a >= 5.0f);
}
__device__ __forceinline__ float e2m1_mag_value(uint32_t c) {
    return c < 4 ? 0.5f * (float)c : (float)(1u << ((c >> 1) - 1)) * (1.0f + 0.5f * (float)(c & 1u));
}

// Quantise 32 values into kTerms MXFP4 terms (codes: 16 bytes per term, scale byte per term).
// Term i takes the residual r left by terms 0..i-1: scale 2^e with e the smallest integer
// such that max|r| <= 6 * 2^e (clamped to the UE8M0 range), codes = nearest e2m1 of r/2^e.
__device__ void quantize_block32(float* v /*[32], destroyed*/, uint4* codes /*[kTerms]*/, uint8_t* scales /*[kTerms]*/) {
#pragma unroll 1
    for (int t = 0; t < kTerms; ++t) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
        int e = -127;
        const uint32_t u = __float_as_uint(amax);
        if (amax > 0.f && (u >> 23) != 0u) {                    // normal amax; subnormal residuals are dropped
            const int e0 = (int)((u >> 23) & 0xFF) - 127;       // floor(log2 amax)
            const float m = __uint_as_float((u & 0x007FFFFFu) | 0x3F800000u);   // amax / 2^e0 in [1, 2)
            e = (m <= 1.5f) ? e0 - 2 : e0 - 1;                  // amax <= 6 * 2^e, minimal e
        }
        if (e < -127) e = -127;
        if (e > 127) e = 127;
        scales[t] = (uint8_t)(e + 127);
        const float inv = (e >= -126 && e <= 126) ? __uint_as_float((uint32_t)(127 - e) << 23) : 0.f;   // 2^-e
        const float sc = (e >= -126) ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
        uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float q = v[i] * inv;
            const uint32_t c = e2m1_mag_code(fminf(fabsf(q), 6.0f));
            float val = e2m1_mag_value(c) * sc;
            const uint32_t sgn = (q < 0.f && c) ? 8u : 0u;
            if (sgn) val = -val;
            v[i] -= val;
            w[i >> 3] |= (c | sgn) << (4 * (i & 7));
        }
        codes[t] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Activation rows -> kTerms MXFP4 terms.  Output row r (r < nrows) takes token row_src[r]/k,
// or token r when row_src is NULL (rows r >= T are zero).  Codes [kTerms][nrows][d/2],
// scales [kTerms][nrows][d/32].  One thread per 32-element block.
__global__ void quantize_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ row_src, int k, int T,
                                     int nrows, int d, uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
    const int nblk = d / 32;
    const long total = (long)nrows * nblk;
    for (long idx = blockIdx.x * (long)blockDim.x + threadIdx.x; idx < total; idx += (long)gridDim.x * blockDim.x) {
        const int r = (int)(idx / nblk), b = (int)(idx % nblk);
        int tok = (r < T) ? r : -1;
        if (row_src) {
            const int s = row_src[r];
            tok = (s >= 0 && s < T * k) ? s / k : -1;
        }
        float v[32];
        if (tok >= 0) {
            const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)tok * d + 32 * b);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 u = src[i];
                v[8 * i + 0] = bf16_lo(u.x); v[8 * i + 1] = bf16_hi(u.x);
                v[8 * i + 2] = bf16_lo(u.y); v[8 * i + 3] = bf16_hi(u.y);
                v[8 * i + 4] = bf16_lo(u.z); v[8 * i + 5] = bf16_hi(u.z);
                v[8 * i + 6] = bf16_lo(u.w); v[8 * i + 7] = bf16_hi(u.w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        uint4 codes[kTerms];
        uint8_t scales[kTerms];
        quantize_block32(v, codes, scales);
#pragma unroll
        for (int t = 0; t < kTerms; ++t) {
            reinterpret_cast<uint4*>(q + ((size_t)t * nrows + r) * (d / 2))[b] = codes[t];
            sf[((size_t)t * nrows + r) * nblk + b] = scales[t];
        }
    }
}

// ------------------------------------------------------------------ the GEMM kernel

struct GemmParams {
    int mode, regime;
    int K, kblocks, mtiles;          // reduction length, K / 256, weight rows / 128
    int T, k, E, num_slots;
    const int32_t* slot;             // [T*k]
    int brows;                       // rows of the B operand buffers
    int decode_cols;                 // decode: B rows [0, decode_cols) in every unit
    const int32_t* plan;             // prefill: [n_active, tiles, e_0.., tile_start_0..] (NT-row tiles)
    const int32_t* offsets;
    const int32_t* row_src;
    const uint8_t* arena;
    int64_t slot_bytes, a_sf_off;    // scales of the A matrix inside a slot (row-major [rows][K/32])
    const uint8_t* b_sf;             // activations' scales, row-major [kTerms][brows][K/32]
    uint8_t* hq;                     // gate/up: h codes [kTerms][hrows][f/2]
    uint8_t* hsf;                    // gate/up: h scales [kTerms][hrows][f/32]
    int hrows;
    int f;
    float* rows_out;                 // down: [rows][d]
    int d;
    int32_t* status;
};

template <int NT>
struct GemmSmem {
    static constexpr int kA = kBM * kKBytes;                 // 16 KB
    static constexpr int kB = kTerms * NT * kKBytes;
    static constexpr int kSFA = 1024;
    static constexpr int kSFB = kTerms * 1024;
    static constexpr int kStage = kA + kB + kSFA + kSFB;     // a multiple of 1024
    static constexpr int kH = NT * 64 * 4;                   // gate/up epilogue h tile
    static constexpr int kBudget = 224 * 1024;               // dynamic smem (static use stays below 3 KB)
    static constexpr int kFit = (kBudget - kH - 2048) / kStage;
    static constexpr int kStages = kFit > 8 ? 8 : kFit;
    static constexpr int kBytes = kStages * kStage + kH + 1024 /*barriers*/ + 1024 /*alignment*/;
    static_assert(kStages >= 2, "operand tile too large for a two-stage pipeline");
};

struct UnitInfo {
    int slot;       // arena slot of the weights
    int m;          // weight row tile
    int brow0;      // first B row
    int ncols;      // valid B rows (columns of D)
};

template <int NT>
__device__ __forceinline__ bool unit_info(const GemmParams& p, int unit, const int* uslots, UnitInfo& u) {
    if (p.regime == kRegimeDecode) {
        u.m = unit % p.mtiles;
        u.slot = uslots[unit / p.mtiles];
        u.brow0 = 0;
        u.ncols = p.decode_cols;
        return true;
    }
    // prefill: unit = tile_start[g]*mtiles + m*ntiles_g + ntile (tiles sharing weights adjacent)
    const int E = p.E, na = p.plan[0];
    int lo = 0, hi = na - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.plan[2 + E + mid] * p.mtiles <= unit) lo = mid; else hi = mid - 1;
    }
    const int g = lo, e = p.plan[2 + g];
    const int o0 = p.offsets[e], o1 = p.offsets[e + 1];
    const int ntiles = (o1 - o0 + NT - 1) / NT;
    const int local = unit - p.plan[2 + E + g] * p.mtiles;
    u.m = local / ntiles;
    u.brow0 = o0 + (local % ntiles) * NT;
    u.ncols = min(NT, o1 - u.brow0);
    const int src = p.row_src[o0];
    u.slot = (src >= 0 && src < p.T * p.k) ? p.slot[src] : -1;
    return u.slot >= 0 && u.slot < p.num_slots;
}

template <int NT, int MODE>
__global__ void __launch_bounds__(kThreadsGemm, 1)
    mxf4_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB, GemmParams p) {
    using S = GemmSmem<NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stage_base = smem;
    float* hbuf = reinterpret_cast<float*>(smem + S::kStages * S::kStage);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kStages * S::kStage + S::kH);
    uint64_t* full = bars;                       // TMA bytes of a stage landed
    uint64_t* sf_full = bars + S::kStages;       // scales of a stage staged
    uint64_t* empty = bars + 2 * S::kStages;     // MMAs of a stage finished
    uint64_t* tfull = bars + 3 * S::kStages;     // [2] accumulator ready
    uint64_t* tempty = tfull + 2;                // [2] accumulator drained
    uint64_t* epibar = tempty + 2;               // [2] epilogue warps' h-tile hand-offs
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    __shared__ int n_units_sh;
    __shared__ int wcount[8];
    __shared__ int uslots[128];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < S::kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&sf_full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), 4);
            mbar_init(smem_u32(&epibar[a]), 4);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_sh)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // decode: the unique valid slots, in order of first appearance, give the units
    if (p.regime == kRegimeDecode) {
        const int n = p.T * p.k;   // <= 128, checked on the host
        int s = -1;
        bool first = false;
        if (tid < n) {
            s = p.slot[tid];
            const bool ok = s >= 0 && s < p.num_slots;
            if (s >= p.num_slots && blockIdx.x == 0) atomicOr(p.status, MOE_STATUS_BAD_SLOT);
            first = ok;
            for (int j = 0; j < tid && first; ++j)
                if (p.slot[j] == s) first = false;
        }
        const unsigned bal = __ballot_sync(0xffffffffu, first);
        if (lane == 0) wcount[warp] = __popc(bal);
        __syncthreads();
        int off = 0;
        for (int w = 0; w < warp; ++w) off += wcount[w];
        if (first) uslots[off + __popc(bal & ((1u << lane) - 1u))] = s;
        if (tid == 0) {
            int tot = 0;
            for (int w = 0; w < kThreadsGemm / 32; ++w) tot += wcount[w];
            n_units_sh = tot * p.mtiles;
        }
    } else if (tid == 0) {
        n_units_sh = p.plan[1] * p.mtiles;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    const int n_units = n_units_sh;
    volatile int* abortp = &abort_flag;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;   // per-stage bit masks
            for (int unit = blockIdx.x; unit < n_units && !*abortp; unit += gridDim.x) {
                UnitInfo u;
                const bool ok = unit_info<NT>(p, unit, uslots, u);
                const int slot = ok ? u.slot : 0;
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abortp)) {
                        atomicOr(p.status, MOE_STATUS_TIMEOUT);
                        *abortp = 1;
                        break;
                    }
                    uint8_t* st = stage_base + stage * S::kStage;
                    const uint32_t bar = smem_u32(&full[stage]);
                    mbar_expect_tx(bar, S::kA + S::kB);
                    tma_load_3d(smem_u32(st), &mapA, kb * kKBytes, u.m * kBM, slot, bar);
#pragma unroll
                    for (int t = 0; t < kTerms; ++t)
                        tma_load_3d(smem_u32(st + S::kA + t * NT * kKBytes), &mapB, kb * kKBytes, u.brow0, t, bar);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == S::kStages) { stage = 0; phase ^= 1u; }
                }
            }
            // every issued load lands before the CTA may exit (bounded)
            for (int s2 = 0; s2 < S::kStages; ++s2) {
                if (!((issued >> s2) & 1u)) continue;
                const uint32_t ph = (issued_parity >> s2) & 1u;
                for (unsigned i = 0; i < kSpinLimit; ++i)
                    if (mbar_try(smem_u32(&full[s2]), ph)) break;
            }
        }
    } else if (warp == 1) {
        // ---------------- scale stager: 8 bytes per row and 256-element K block
        int stage = 0;
        uint32_t phase = 0;
        const int rowbytes = p.K / 32;
        for (int unit = blockIdx.x; unit < n_units && !*abortp; unit += gridDim.x) {
            UnitInfo u;
            const bool ok = unit_info<NT>(p, unit, uslots, u);
            const uint8_t* asf = p.arena + (int64_t)(ok ? u.slot : 0) * p.slot_bytes + p.a_sf_off;
            bool failed = false;
            for (int kb = 0; kb < p.kblocks; ++kb) {
                if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abortp)) {
                    if (lane == 0) { atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
                    failed = true;
                    break;
                }
                uint8_t* st = stage_base + stage * S::kStage;
                uint8_t* sfa = st + S::kA + S::kB;
                uint8_t* sfb = sfa + S::kSFA;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = lane + 32 * i;
                    const uint2 v = *reinterpret_cast<const uint2*>(asf + (int64_t)(u.m * kBM + r) * rowbytes + kb * 8);
                    const int o = (r & 31) * 16 + (r >> 5) * 4;
                    *reinterpret_cast<uint32_t*>(sfa + o) = v.x;
                    *reinterpret_cast<uint32_t*>(sfa + 512 + o) = v.y;
                }
#pragma unroll
                for (int t = 0; t < kTerms; ++t) {
                    for (int r = lane; r < NT; r += 32) {
                        const int row = u.brow0 + r;
                        uint2 v = make_uint2(0, 0);
                        if (row < p.brows)
                            v = *reinterpret_cast<const uint2*>(p.b_sf + ((int64_t)t * p.brows + row) * rowbytes + kb * 8);
                        const int o = (r & 31) * 16 + (r >> 5) * 4;
                        *reinterpret_cast<uint32_t*>(sfb + t * 1024 + o) = v.x;
                        *reinterpret_cast<uint32_t*>(sfb + t * 1024 + 512 + o) = v.y;
                    }
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sf_full[stage]));
                if (++stage == S::kStages) { stage = 0; phase ^= 1u; }
            }
            if (failed) break;
        }
    } else if (warp == 2) {
        // ---------------- MMA issuer
        if (lane == 0) {
            int stage = 0, sfring = 0, acc = 0;
            uint32_t phase = 0, aphase = 0;
            for (int unit = blockIdx.x; unit < n_units && !*abortp; unit += gridDim.x) {
                if (!mbar_wait(smem_u32(&tempty[acc]), aphase ^ 1u, abortp)) {
                    atomicOr(p.status, MOE_STATUS_TIMEOUT);
                    *abortp = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t dcol = tmem + acc * NT;
                bool failed = false;
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abortp) ||
                        !mbar_wait(smem_u32(&sf_full[stage]), phase, abortp)) {
                        atomicOr(p.status, MOE_STATUS_TIMEOUT);
                        *abortp = 1;
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    uint8_t* st = stage_base + stage * S::kStage;
                    const uint32_t sa = smem_u32(st), sb = smem_u32(st + S::kA);
                    const uint32_t ssfa = smem_u32(st + S::kA + S::kB), ssfb = ssfa + S::kSFA;
                    const uint32_t sfcol = tmem + 256 + sfring * kSfCols;
                    tc_cp_sf(sfcol + 0, desc_sf(ssfa));
                    tc_cp_sf(sfcol + 4, desc_sf(ssfa + 512));
#pragma unroll
                    for (int t = 0; t < kTerms; ++t) {
                        tc_cp_sf(sfcol + 8 + 8 * t, desc_sf(ssfb + t * 1024));
                        tc_cp_sf(sfcol + 8 + 8 * t + 4, desc_sf(ssfb + t * 1024 + 512));
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t id = idesc_mxf4(NT, 2 * (j & 1));
                        const uint64_t ad = desc_sw128(sa + 32 * j);
#pragma unroll
                        for (int t = 0; t < kTerms; ++t) {
                            const uint64_t bd = desc_sw128(sb + t * NT * kKBytes + 32 * j);
                            mma_mxf4(dcol, ad, bd, id, sfcol + 4 * (j >> 1), sfcol + 8 + 8 * t + 4 * (j >> 1),
                                     (kb | j | t) ? 1u : 0u);
                        }
                    }
                    tc_commit(smem_u32(&empty[stage]));
                    if (++stage == S::kStages) { stage = 0; phase ^= 1u; }
                    sfring = (sfring + 1) % kSfRing;
                }
                if (failed) break;
                tc_commit(smem_u32(&tfull[acc]));
                if (++acc == 2) { acc = 0; aphase ^= 1u; }
            }
        }
    } else {
        // ---------------- epilogue (warps 3..6 -> TMEM lane quarters 3, 0, 1, 2)
        const int q = warp & 3;
        const int ew = warp - 3;
        int acc = 0;
        uint32_t aphase = 0, ephase = 0;
        for (int unit = blockIdx.x; unit < n_units && !*abortp; unit += gridDim.x) {
            UnitInfo u;
            const bool ok = unit_info<NT>(p, unit, uslots, u);
            if (!mbar_wait(smem_u32(&tfull[acc]), aphase, abortp)) {
                if (lane == 0) { atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
                break;
            }
            tc_fence_after();
            const int row = q * 32 + lane;       // accumulator row = weight row within the tile
            float vals[NT];
#pragma unroll
            for (int c0 = 0; c0 < NT; c0 += 16) tc_ld16(tmem + ((uint32_t)(q * 32) << 16) + acc * NT + c0, vals + c0);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
            if (++acc == 2) { acc = 0; aphase ^= 1u; }
            if (!ok) continue;
            if (MODE == kModeDown) {
                const int r = u.m * kBM + row;    // output feature
#pragma unroll
                for (int c = 0; c < NT; ++c) {
                    const bool valid = (p.regime == kRegimeDecode) ? (c < u.ncols && p.slot[c] == u.slot) : (c < u.ncols);
                    if (valid) p.rows_out[(size_t)(u.brow0 + c) * p.d + r] = vals[c];
                }
            } else {
                // rows 2i' = gate, 2i'+1 = up of output i' = row/2 within the tile (i = 64m + i')
#pragma unroll
                for (int c = 0; c < NT; ++c) {
                    const float partner = __shfl_xor_sync(0xffffffffu, vals[c], 1);
                    if ((lane & 1) == 0) {
                        const float g = vals[c];
                        hbuf[c * 64 + (row >> 1)] = g / (1.0f + expf(-g)) * partner;
                    }
                }
                // hand-off 1: every warp's h values are in hbuf
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&epibar[0]));
                if (!mbar_wait(smem_u32(&epibar[0]), ephase, abortp)) {
                    if (lane == 0) { atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
                    break;
                }
                // quantise: job = (column c, block b of 32 outputs)
                const int fblk = p.f / 32;
                for (int job = ew * 32 + lane; job < NT * 2; job += 128) {
                    const int c = job >> 1, b = job & 1;
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = hbuf[c * 64 + 32 * b + i];
                    uint4 codes[kTerms];
                    uint8_t scales[kTerms];
                    quantize_block32(v, codes, scales);
                    auto write_row = [&](int hrow) {
#pragma unroll
                        for (int t = 0; t < kTerms; ++t) {
                            reinterpret_cast<uint4*>(p.hq + ((size_t)t * p.hrows + hrow) * (p.f / 2))[u.m * 2 + b] = codes[t];
                            p.hsf[((size_t)t * p.hrows + hrow) * fblk + u.m * 2 + b] = scales[t];
                        }
                    };
                    if (p.regime == kRegimeDecode) {
                        // column c = token; h for every pair (c, j) routed to this slot
                        if (c < p.T)
                            for (int j = 0; j < p.k; ++j)
                                if (p.slot[c * p.k + j] == u.slot) write_row(c * p.k + j);
                    } else if (c < u.ncols) {
                        write_row(u.brow0 + c);
                    }
                }
                // hand-off 2: hbuf may be overwritten by the next unit
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&epibar[1]));
                if (!mbar_wait(smem_u32(&epibar[1]), ephase, abortp)) {
                    if (lane == 0) { atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
                    break;
                }
                ephase ^= 1u;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// y[t] = bf16( sum_j w[t,j] rows[t*k + j] ) in ascending j, skipping pairs without a valid slot.
__global__ void decode_combine_kernel(int T, int d, int k, int num_slots, const float* __restrict__ rows,
                                      const int32_t* __restrict__ slot, const float* __restrict__ w, uint16_t* y) {
    const int vec = d / 4;
    for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < T * vec; idx += gridDim.x * blockDim.x) {
        const int t = idx / vec, c4 = idx % vec;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const int pr = t * k + j, s = slot[pr];
            if (s < 0 || s >= num_slots) continue;
            const float wj = w[pr];
            const float4 z = reinterpret_cast<const float4*>(rows + (size_t)pr * d)[c4];
            acc.x = fmaf(wj, z.x, acc.x);
            acc.y = fmaf(wj, z.y, acc.y);
            acc.z = fmaf(wj, z.z, acc.z);
            acc.w = fmaf(wj, z.w, acc.w);
        }
        const uint32_t lo = (uint32_t)f32_to_bf16(acc.x) | ((uint32_t)f32_to_bf16(acc.y) << 16);
        const uint32_t hi = (uint32_t)f32_to_bf16(acc.z) | ((uint32_t)f32_to_bf16(acc.w) << 16);
        reinterpret_cast<uint2*>(y + (size_t)t * d)[c4] = make_uint2(lo, hi);
    }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)ptr;
    }
    return fn;
}

// 3-D uint8 tensor [planes][rows][xbytes] with the given row and plane strides;
// box {128 bytes, box_rows, 1}, SWIZZLE_128B; out-of-range rows read as zero.
static bool make_map(CUtensorMap* m, const void* base, uint64_t xbytes, uint64_t rows, uint64_t planes,
                     uint64_t row_stride, uint64_t plane_stride, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {xbytes, rows, planes};
    cuuint64_t strides[2] = {row_stride, plane_stride};
    cuuint32_t box[3] = {128, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NT, int MODE>
static int launch_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const GemmParams& p, int grid, cudaStream_t st) {
    using S = GemmSmem<NT>;
    if (cudaFuncSetAttribute(mxf4_gemm_kernel<NT, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes) !=
        cudaSuccess)
        return MOE_ERR_LAUNCH;
    mxf4_gemm_kernel<NT, MODE><<<grid, kThreadsGemm, S::kBytes, st>>>(ma, mb, p);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

template <int MODE>
static int launch_gemm_nt(int NT, const CUtensorMap& ma, const CUtensorMap& mb, const GemmParams& p, int grid,
                          cudaStream_t st) {
    switch (NT) {
        case 16: return launch_gemm<16, MODE>(ma, mb, p, grid, st);
        case 32: return launch_gemm<32, MODE>(ma, mb, p, grid, st);
        case 64: return launch_gemm<64, MODE>(ma, mb, p, grid, st);
        case 128: return launch_gemm<128, MODE>(ma, mb, p, grid, st);
        default: return MOE_ERR_LAUNCH;
    }
}

// Tensor-core buffers inside the workspace (WsLayout.tc), sized for R = T*k rows.
struct TcBuffers {
    uint8_t *xq, *xsf, *hq, *hsf;
    float* rows;
    int32_t* plan;
};

static TcBuffers tc_buffers(const moe_dims* m, int T, char* ws, const WsLayout& L) {
    TcBuffers b;
    const size_t R = (size_t)(T > 0 ? T : 1) * m->top_k;
    char* o = ws + L.tc;
    b.xq = reinterpret_cast<uint8_t*>(o);  o += align256((size_t)kTerms * R * m->d / 2);
    b.xsf = reinterpret_cast<uint8_t*>(o); o += align256((size_t)kTerms * R * m->d / 32);
    b.hq = reinterpret_cast<uint8_t*>(o);  o += align256((size_t)kTerms * R * m->f / 2);
    b.hsf = reinterpret_cast<uint8_t*>(o); o += align256((size_t)kTerms * R * m->f / 32);
    b.rows = reinterpret_cast<float*>(o);
    b.plan = reinterpret_cast<int32_t*>(ws + L.active);
    return b;
}

size_t tc_workspace_bytes(const moe_dims* m, int T) {
    const size_t R = (size_t)(T > 0 ? T : 1) * m->top_k;
    return align256((size_t)kTerms * R * m->d / 2) + align256((size_t)kTerms * R * m->d / 32) +
           align256((size_t)kTerms * R * m->f / 2) + align256((size_t)kTerms * R * m->f / 32) + align256(R * m->d * 4);
}

static int nt_for(int cols) { return cols <= 16 ? 16 : cols <= 32 ? 32 : cols <= 64 ? 64 : 128; }

bool tc_supported(const moe_dims* m) { return m->d % kKB == 0 && m->f % kKB == 0; }
bool tc_decode_supported(const moe_dims* m, int T) { return tc_supported(m) && T >= 1 && T * m->top_k <= 128; }

// Decode regime: quantise x, gate/up GEMM (SwiGLU, h quantised per (token, j) pair), down
// GEMM (one fp32 row per pair), fixed-order combine into y.
int launch_tc_decode(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                     const float* w, uint16_t* y, int32_t* status, char* ws, const WsLayout& L, cudaStream_t st,
                     int num_sms) {
    if (T == 0) return MOE_OK;
    TcBuffers b = tc_buffers(m, T, ws, L);
    const int d = m->d, f = m->f, k = m->top_k;
    const int R = T * k;
    const SlotLayout SL = slot_layout(d, f);
    quantize_rows_kernel<<<(T * (d / 32) + 255) / 256, 256, 0, st>>>(x, nullptr, k, T, T, d, b.xq, b.xsf);
    const uint8_t* base = reinterpret_cast<const uint8_t*>(ar->base);
    CUtensorMap mA, mB, mA2, mB2;
    const int nt1 = nt_for(T);
    if (!make_map(&mA, base + SL.gu_q, d / 2, 2 * f, ar->num_slots, d / 2, ar->slot_bytes, kBM)) return MOE_ERR_LAUNCH;
    if (!make_map(&mB, b.xq, d / 2, T, kTerms, d / 2, (uint64_t)T * d / 2, nt1)) return MOE_ERR_LAUNCH;
    GemmParams p{};
    p.mode = kModeGateUp; p.regime = kRegimeDecode;
    p.K = d; p.kblocks = d / kKB; p.mtiles = 2 * f / kBM;
    p.T = T; p.k = k; p.E = m->num_experts; p.num_slots = ar->num_slots;
    p.slot = slot; p.brows = T; p.hrows = R; p.decode_cols = T;
    p.arena = base; p.slot_bytes = ar->slot_bytes; p.a_sf_off = SL.gu_s;
    p.b_sf = b.xsf; p.hq = b.hq; p.hsf = b.hsf; p.f = f; p.rows_out = b.rows; p.d = d; p.status = status;
    int rc = launch_gemm_nt<kModeGateUp>(nt1, mA, mB, p, num_sms, st);
    if (rc) return rc;
    const int nt2 = nt_for(R);
    if (!make_map(&mA2, base + SL.dn_q, f / 2, d, ar->num_slots, f / 2, ar->slot_bytes, kBM)) return MOE_ERR_LAUNCH;
    if (!make_map(&mB2, b.hq, f / 2, R, kTerms, f / 2, (uint64_t)R * f / 2, nt2)) return MOE_ERR_LAUNCH;
    GemmParams q = p;
    q.mode = kModeDown; q.K = f; q.kblocks = f / kKB; q.mtiles = d / kBM;
    q.brows = R; q.decode_cols = R; q.a_sf_off = SL.dn_s; q.b_sf = b.hsf;
    rc = launch_gemm_nt<kModeDown>(nt2, mA2, mB2, q, num_sms, st);
    if (rc) return rc;
    decode_combine_kernel<<<(T * (d / 4) + 255) / 256, 256, 0, st>>>(T, d, k, ar->num_slots, b.rows, slot, w, y);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

__global__ void plan_kernel(int E, int n, const int32_t* offsets, int32_t* plan, int32_t* status, int tile_rows);

constexpr int kPrefillNT = 64;

// Prefill regime: x rows quantised in permuted (grouped) order, gate/up GEMM per (group,
// weight tile, 64-row tile) with SwiGLU + h quantisation, down GEMM to per-row fp32 outputs;
// the caller's combine sums them in fixed order.
int launch_tc_prefill(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                      const int32_t* offsets, const int32_t* row_src, float* rows_out, int32_t* status, char* ws,
                      const WsLayout& L, cudaStream_t st, int num_sms) {
    if (T == 0) return MOE_OK;
    TcBuffers b = tc_buffers(m, T, ws, L);
    const int d = m->d, f = m->f, k = m->top_k, n = T * k;
    const SlotLayout SL = slot_layout(d, f);
    plan_kernel<<<1, 32, 0, st>>>(m->num_experts, n, offsets, b.plan, status, kPrefillNT);
    const long qblocks = ((long)n * (d / 32) + 255) / 256;
    quantize_rows_kernel<<<(int)(qblocks > 8L * num_sms ? 8L * num_sms : qblocks), 256, 0, st>>>(x, row_src, k, T, n, d,
                                                                                                 b.xq, b.xsf);
    const uint8_t* base = reinterpret_cast<const uint8_t*>(ar->base);
    CUtensorMap mA, mB, mA2, mB2;
    if (!make_map(&mA, base + SL.gu_q, d / 2, 2 * f, ar->num_slots, d / 2, ar->slot_bytes, kBM)) return MOE_ERR_LAUNCH;
    if (!make_map(&mB, b.xq, d / 2, n, kTerms, d / 2, (uint64_t)n * d / 2, kPrefillNT)) return MOE_ERR_LAUNCH;
    GemmParams p{};
    p.mode = kModeGateUp; p.regime = kRegimePrefill;
    p.K = d; p.kblocks = d / kKB; p.mtiles = 2 * f / kBM;
    p.T = T; p.k = k; p.E = m->num_experts; p.num_slots = ar->num_slots;
    p.slot = slot; p.brows = n; p.hrows = n; p.decode_cols = 0;
    p.plan = b.plan; p.offsets = offsets; p.row_src = row_src;
    p.arena = base; p.slot_bytes = ar->slot_bytes; p.a_sf_off = SL.gu_s;
    p.b_sf = b.xsf; p.hq = b.hq; p.hsf = b.hsf; p.f = f; p.rows_out = rows_out; p.d = d; p.status = status;
    int rc = launch_gemm_nt<kModeGateUp>(kPrefillNT, mA, mB, p, num_sms, st);
    if (rc) return rc;
    if (!make_map(&mA2, base + SL.dn_q, f / 2, d, ar->num_slots, f / 2, ar->slot_bytes, kBM)) return MOE_ERR_LAUNCH;
    if (!make_map(&mB2, b.hq, f / 2, n, kTerms, f / 2, (uint64_t)n * f / 2, kPrefillNT)) return MOE_ERR_LAUNCH;
    GemmParams q = p;
    q.mode = kModeDown; q.K = f; q.kblocks = f / kKB; q.mtiles = d / kBM; q.a_sf_off = SL.dn_s; q.b_sf = b.hsf;
    return launch_gemm_nt<kModeDown>(kPrefillNT, mA2, mB2, q, num_sms, st);
}

}  // namespace fp4moe
