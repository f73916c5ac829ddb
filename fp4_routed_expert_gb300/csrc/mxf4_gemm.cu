// mxf4_gemm.cu -- the prefill expert FFN on the 5th-generation tensor cores (sm_103a): grouped
// block-scaled MXFP4 GEMMs with tcgen05.mma (kind::mxf4), TMEM accumulators, bulk-copy operand
// loads and fused epilogues.  (The decode regime's kernel is in mxf4_decode.cu.)
//
// Operands.  A = expert weight rows straight from the slot arena: e2m1 codes and UE8M0
// scales per 32 K elements, exactly the checkpoint's format ("DeepSeek-V4.1-Flash on a
// single NVIDIA DGX Spark", "Why it is built this way": FP4 + UE8M0/32, never requantised).
// B = activations, written by this library as a sum of kTerms MXFP4 tensors
// (x ~ q_1 + q_2 + ..., each q_i e2m1 codes with its own UE8M0 scale per 32 elements, q_i
// quantising the residual left by q_1..q_(i-1)); the MMA accumulates every term into the same
// fp32 accumulator, so D = W . x up to the residual after kTerms terms.  B's rows are the
// expert-grouped permutation of the tokens in tiles of kPrefillNT rows (N = kTerms x 64 = 256).
//
// Every operand sits in global memory in blocks of 256 K elements that carry their codes
// (128-byte rows pre-swizzled for SWIZZLE_128B) followed by their scale atoms, and the blocks
// of one row tile are consecutive along K.  A pipeline stage spans kKPS such K blocks and is
// two contiguous bulk copies (cp.async.bulk), weights and activations: a bulk copy costs the
// SM's copy engine a fixed time on top of its bytes, so few large copies stream fastest.
//
// One persistent kernel, one CTA per SM, 10 warps:
//   warp 0  producer: per stage one bulk copy of the weight tiles (codes + scale atoms) and
//           one of the activation blocks (kTerms x NT rows + scale atoms)
//   warp 1  MMA issuer (one lane): tcgen05.cp of the scale atoms, 4 MMAs per K block,
//           tcgen05.commit to release smem stages and publish accumulators
//   warps 2..9  epilogue (two per TMEM lane quarter over column halves): tcgen05.ld of the
//           accumulator, then gate/up: SwiGLU + requantisation of h into kTerms MXFP4 tiles for
//           the down GEMM; down: fp32 rows for the fixed-order combine
// Every wait is bounded; a timeout sets MOE_STATUS_TIMEOUT and the CTA drains and exits.
#include <cuda.h>

#include "mxf4_common.cuh"

namespace fp4moe {

// Prefill activations -> kTerms MXFP4 terms in tile layout, one thread per (token t, 32-element
// block b): the block is quantised once and written into the tile row of each of the token's k
// pairs (pair_row, from the plan).  Rows of a tile past its group's end are never written: they
// feed only accumulator columns that the epilogues discard.  Also clears `nzero` counters for
// the FFN kernel that follows.
__global__ void __launch_bounds__(256) quantize_tiles_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ pair_row,
                                                             int k, int T, int d, uint8_t* __restrict__ q,
                                                             int32_t* __restrict__ zero, int nzero) {
    constexpr int NT = kPrefillNT;
    // launched early behind the previous kernel: nothing it wrote is read before it completes;
    // the FFN kernel may launch at once (it waits for this kernel in turn)
    pdl_trigger();
    pdl_wait();
    // the FFN kernel's counters start at zero
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nzero; i += gridDim.x * blockDim.x) zero[i] = 0;
    const int nblk = d / 32, KB = d / kKB;
    const long total = (long)T * nblk;
    for (long idx = blockIdx.x * (long)blockDim.x + threadIdx.x; idx < total; idx += (long)gridDim.x * blockDim.x) {
        const int b = (int)(idx % nblk);
        const int t = (int)(idx / nblk);
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d + 32 * b);
        float v[32];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint4 w4 = __ldg(src + u);
            const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                v[8 * u + 2 * h] = bf16_lo(ww[h]);
                v[8 * u + 2 * h + 1] = bf16_hi(ww[h]);
            }
        }
        uint32_t wds[kTerms][4], scl[kTerms];
        thread_quantize32(v, wds, scl);
        const int kb = b / 8, j = b % 8;
        for (int jj = 0; jj < k; ++jj) {
            const int lin = __ldg(pair_row + (size_t)t * k + jj);
            if (lin < 0) continue;
            const int tile = lin / NT, r = lin % NT;
#pragma unroll
            for (int tt = 0; tt < kTerms; ++tt) {
                *reinterpret_cast<uint4*>(q + act_code_off(tile, kb, tt, r, j, NT, KB)) =
                    make_uint4(wds[tt][0], wds[tt][1], wds[tt][2], wds[tt][3]);
                q[act_scale_off(tile, kb, tt, r, j, NT, KB)] = (uint8_t)scl[tt];
            }
        }
    }
}

// ------------------------------------------------------------------ the expert FFN kernel

// One GEMM of the FFN: gate/up (phase 0, K = d, weight rows 2f interleaved gate/up) or down
// (phase 1, K = f, weight rows d).
struct PhaseParams {
    int kblocks, mtiles;             // K / 256, weight rows / 128
    int64_t a_off;                   // the weight matrix inside a slot
    const uint8_t* b;                // activation blocks
};

struct FfnParams {
    int T, k, E, num_slots;
    const int32_t* slot;             // [T*k]
    const int32_t* plan;             // prefill: the plan (see plan_grec_off / plan_tile_group_off)
    const int32_t* tile_group;       // prefill: group of each tile
    const int4* grec;                // prefill: {first row, end row, slot, first tile} per group
    const int32_t* offsets;
    const int32_t* row_src;
    const uint8_t* arena;
    int64_t slot_bytes;
    PhaseParams ph[2];
    uint8_t* h;                      // h blocks written by phase 0, read by phase 1
    int f, d;
    float* rows_out;                 // phase 1 output rows [rows][d] (fp32)
    int32_t* status;
    int32_t* work;                   // next unit to hand out (zero at launch)
    int32_t* ready;                  // phase 0 units finished, per activation tile
    // polls after which a wait on another CTA's progress gives up (0: kSpinLimit); read after
    // the wait on the kernel ahead
    const int32_t* wait_limit;
};

// Work list: units [0, n0) are gate/up units, [n0, n0 + n1) down units, n_i = tiles x weight
// tiles of phase i; a unit is one (weight tile, activation tile) pair over the whole K, units
// sharing weights adjacent.  CTAs take units in that order from a global counter, so every
// gate/up unit is handed out before any down unit.
constexpr int kUQ = 8;   // unit ids in flight from the producer to the MMA and epilogue warps

// Per-NT shape of the pipeline (one CTA per SM, the whole shared memory and 512 TMEM columns).
// B rows per tile = kTerms*NT (N of one MMA, <= 256).  ACC independent accumulators (K slices
// alternate between them so the tensor core can overlap their dependency chains; the count
// depends only on the row count) and DBUF accumulator sets (epilogue of one unit overlapping
// the next unit's MMAs) fill TMEM columns [0, kAccCols); the scale ring follows.
template <int NT>
struct GemmCfg {
    static constexpr int kTmem = kTmemCols;                  // TMEM columns of the CTA
    static constexpr int kRows = kTerms * NT;                // B rows = N of one MMA (<= 256)
    static_assert(kRows <= 256 && kRows % 16 == 0, "one MMA covers every B row");
    static constexpr int kN = kRows;
    // B scales: one 32x128b copy per 128 B rows (group g) and half of a K block's eight
    // 32-element blocks (jq); the MMA of K slice j reads from column base + kBsfQ * (j / 2) and,
    // for B rows 128.., four columns further (the layout of one MMA with N > 128, checked on
    // GB300 against a host product).  Wide tiles keep every base a multiple of 16 columns.
    static constexpr int kSg = (kRows + 127) / 128;
    static constexpr int kBsfQ = kSg == 1 ? 4 : 16;
    static constexpr int kSfB = kSg == 1 ? 8 : 16;           // B scales' offset in a ring slot
    static constexpr int kSfCols = kSfB + 2 * kBsfQ;         // scale columns per K block (A + B)
    static constexpr int kAcc = kRows <= 64 ? 2 : 1;         // short chains only at small N
    static constexpr int kDbuf = (2 * kAcc * kRows + kSfRing * kSfCols <= kTmem) ? 2 : 1;
    static constexpr int kAccCols = (kDbuf * kAcc * kRows + 31) / 32 * 32;
    static_assert(kAccCols + kSfRing * kSfCols <= kTmem, "accumulators and scales exceed the TMEM columns");
    static constexpr int kBCodes = kRows * kKBytes;          // activation codes per K block
    static constexpr int kBBlk = act_block_bytes(NT);        // activation block (codes + atoms)
    static constexpr int kH = NT * 66 * 4;                   // gate/up epilogue h tile (padded rows)
    static constexpr int kBudget = 226 * 1024;               // dynamic smem (static stays below 2 KB)
    // K blocks per stage: two (fewer, larger copies) unless that leaves fewer than three stages
    static constexpr int kKPS = (kBudget - kH - 2048) / (2 * (kTileBytes + kBBlk)) >= 3 ? 2 : 1;
    // stage: kKPS weight tiles (kTileBytes each), then kKPS activation blocks; every operand
    // start is a multiple of 1024 bytes
    static constexpr int kStage = kKPS * (kTileBytes + kBBlk);
    // Epilogue warps: eight, two per TMEM lane quarter, each taking half of the columns (the
    // wide tiles' SwiGLU and quantisation need the issue slots).
    static constexpr int kEpi = 8;
    static constexpr int kThreads = (2 + kEpi) * 32;
    static constexpr int kNH = NT / (kEpi / 4);              // columns of one epilogue warp
    static constexpr int kLdW = kNH < 16 ? kNH : 16;         // accumulator columns per tcgen05.ld
    static constexpr int kFit = (kBudget - kH - 2048) / kStage;
    static constexpr int kStages = kFit > 8 ? 8 : kFit;
    static constexpr int kBytes = kStages * kStage + kH + 1024 /*barriers*/ + 1024 /*alignment*/;
    static_assert(kStages >= 2, "operand tile too large for a two-stage pipeline");
};

struct UnitInfo {
    int slot;       // arena slot of the weights
    int m;          // weight row tile
    int key;        // activation tile (its h readiness counter)
    int btile;      // activation tile
    int brow0;      // first B row (row index of the activation rows / outputs)
    int ncols;      // valid columns of D
};

template <int NT>
__device__ __forceinline__ bool unit_info(const FfnParams& p, const PhaseParams& P, int unit, UnitInfo& u) {
    // unit = first_tile_g*mtiles + m*ntiles_g + ntile (tiles sharing weights adjacent), so
    // unit / mtiles is a tile of group g
    const int4 gr = p.grec[p.tile_group[unit / P.mtiles]];   // first row, end row, slot, first tile
    const int ntiles = (gr.y - gr.x + NT - 1) / NT;
    const int local = unit - gr.w * P.mtiles;
    u.m = local / ntiles;
    const int nt = local % ntiles;
    u.btile = gr.w + nt;
    u.key = u.btile;
    u.brow0 = gr.x + nt * NT;
    u.ncols = min(NT, gr.y - u.brow0);
    u.slot = gr.z;
    return u.slot >= 0 && u.slot < p.num_slots;
}


// The whole expert FFN of a prefill call in one persistent launch (one CTA per SM, every CTA
// resident).  The producer takes units from the work list; a down unit needs the h rows of its
// activation tile from every gate/up unit of that tile, so the producer issues the unit's
// weight copies, then waits (bounded) for the tile's count of finished gate/up units before
// issuing the h copies.
template <int NT>
__global__ void __launch_bounds__(10 * 32, 1) mxf4_ffn_kernel(FfnParams p) {
    using C = GemmCfg<NT>;
    static_assert(C::kThreads == 10 * 32 && C::kNH * (C::kEpi / 4) == NT, "epilogue warp layout");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stage_base = smem;
    float* hbuf = reinterpret_cast<float*>(smem + C::kStages * C::kStage);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage + C::kH);
    uint64_t* full = bars;                       // bytes of a stage landed
    uint64_t* empty = bars + C::kStages;         // MMAs of a stage finished
    uint64_t* tfull = bars + 2 * C::kStages;     // [2] accumulator set ready
    uint64_t* tempty = tfull + 2;                // [2] accumulator set drained
    uint64_t* epibar = tempty + 2;               // [2] epilogue warps' h-tile hand-offs
    uint64_t* uqfull = epibar + 2;               // [kUQ] unit id written
    uint64_t* uqempty = uqfull + kUQ;            // [kUQ] unit id read by the MMA and epilogue warps
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    __shared__ int n_keys_sh;
    __shared__ int uq[kUQ];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), C::kEpi);
            mbar_init(smem_u32(&epibar[a]), C::kEpi);
        }
        for (int i = 0; i < kUQ; ++i) {
            mbar_init(smem_u32(&uqfull[i]), 1);
            mbar_init(smem_u32(&uqempty[i]), 1 + C::kEpi);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_sh)),
                     "r"(C::kTmem)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();   // barriers initialised, TMEM address published
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    volatile int* abortp = &abort_flag;
    // everything above overlaps the previous kernel; its outputs are read from here on
    pdl_wait();
    unsigned dep_limit = kSpinLimit;
    if (p.wait_limit && *p.wait_limit > 0) dep_limit = (unsigned)*p.wait_limit;
    if (tid == 0) n_keys_sh = p.plan[1];   // activation tiles of the plan
    // every role reads the tile count here, before any of them can abort on a later wait
    __syncthreads();
    const int n_keys = n_keys_sh;
    const int n0 = n_keys * p.ph[0].mtiles, n_all = n0 + n_keys * p.ph[1].mtiles;
    // position in the unit-id ring (same sequence for every role)
    int qi = 0;
    uint32_t qphase = 0;

    if (warp == 0) {
        // ---------------- producer: takes units, two contiguous bulk copies per stage
        if (lane == 0) {
            int stage = 0, ready_key = -1;
            uint32_t phase = 0, issued = 0, issued_parity = 0;   // per-stage bit masks
            while (true) {
                int unit = *abortp ? -1 : atomicAdd(p.work, 1);
                if (unit >= n_all) unit = -1;
                if (!mbar_wait(smem_u32(&uqempty[qi]), qphase ^ 1u, abortp)) {
                    atomicOr(p.status, MOE_STATUS_TIMEOUT);
                    *abortp = 1;
                    unit = -1;
                }
                uq[qi] = unit;
                mbar_arrive(smem_u32(&uqfull[qi]));
                if (++qi == kUQ) { qi = 0; qphase ^= 1u; }
                if (unit < 0) break;
                const int ph = unit < n0 ? 0 : 1;
                const PhaseParams& P = p.ph[ph];
                UnitInfo u;
                const bool ok = unit_info<NT>(p, P, ph ? unit - n0 : unit, u);
                const uint8_t* sbase = p.arena + (int64_t)(ok ? u.slot : 0) * p.slot_bytes;
                // A down unit whose h is not ready yet gets its weight copies issued into every
                // free stage; the h copies of those stages follow once it is ready.
                bool have_b = (ph == 0) || !(ok && u.key != ready_key);
                const int nst = (P.kblocks + C::kKPS - 1) / C::kKPS;   // stages of this unit
                int pend_n = 0, pend_s0 = 0, pend_stage0 = 0;
                // activation blocks of stage s of the unit (K blocks kKPS*s ..) into smem stage stg
                auto issue_b = [&](int s, int stg) {
                    const int kb = s * C::kKPS, nkb = min(C::kKPS, P.kblocks - kb);
                    const int64_t blk = (int64_t)u.btile * P.kblocks + kb;
                    bulk_g2s(smem_u32(stage_base + stg * C::kStage + C::kKPS * kTileBytes), P.b + blk * C::kBBlk,
                             nkb * C::kBBlk, smem_u32(&full[stg]));
                };
                auto flush = [&]() {
                    for (int i = 0; i < pend_n; ++i) issue_b(pend_s0 + i, (pend_stage0 + i) % C::kStages);
                    pend_n = 0;
                };
                auto key_ready = [&](bool block) -> bool {
                    // every gate/up unit of the activation tile has written its h rows
                    const int32_t* flag = p.ready + u.key;
                    const int target = p.ph[0].mtiles;
                    unsigned spins = 0;
                    while (ld_acquire(flag) < target) {
                        if (!block) return false;
                        if (++spins > dep_limit || *abortp) {
                            atomicOr(p.status, MOE_STATUS_TIMEOUT);
                            *abortp = 1;
                            break;   // the copies still go out, so that every stage's barrier completes
                        }
                        __nanosleep(64);
                    }
                    fence_proxy_async();
                    ready_key = u.key;
                    have_b = true;
                    return true;
                };
                for (int s = 0; s < nst; ++s) {
                    if (pend_n == C::kStages) {   // the next stage still waits for its h copy
                        key_ready(true);
                        flush();
                    }
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abortp)) {
                        atomicOr(p.status, MOE_STATUS_TIMEOUT);
                        *abortp = 1;
                        break;
                    }
                    const uint32_t st = smem_u32(stage_base + stage * C::kStage);
                    const uint32_t bar = smem_u32(&full[stage]);
                    const int kb = s * C::kKPS, nkb = min(C::kKPS, P.kblocks - kb);
                    const int64_t atile = (int64_t)u.m * P.kblocks + kb;
                    mbar_expect_tx(bar, nkb * (kTileBytes + C::kBBlk));
                    bulk_g2s(st, sbase + P.a_off + atile * kTileBytes, nkb * kTileBytes, bar);
                    if (!have_b && key_ready(false)) flush();
                    if (have_b) {
                        issue_b(s, stage);
                    } else {
                        if (pend_n == 0) { pend_s0 = s; pend_stage0 = stage; }
                        ++pend_n;
                    }
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                }
                if (pend_n) {
                    key_ready(true);
                    flush();
                }
            }
            // every issued copy lands before the CTA may exit (bounded)
            for (int s2 = 0; s2 < C::kStages; ++s2) {
                if (!((issued >> s2) & 1u)) continue;
                const uint32_t ph = (issued_parity >> s2) & 1u;
                for (unsigned i = 0; i < kSpinLimit; ++i)
                    if (mbar_try(smem_u32(&full[s2]), ph)) break;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            int stage = 0, sfring = 0, acc = 0;
            uint32_t phase = 0, aphase = 0;
            const uint32_t idesc_lo = idesc_mxf4(C::kN, 0), idesc_hi = idesc_mxf4(C::kN, 2);
            while (true) {
                int unit = -1;
                if (mbar_wait(smem_u32(&uqfull[qi]), qphase, abortp)) unit = uq[qi];
                mbar_arrive(smem_u32(&uqempty[qi]));
                if (++qi == kUQ) { qi = 0; qphase ^= 1u; }
                if (unit < 0) break;
                const int KB = p.ph[unit < n0 ? 0 : 1].kblocks;
                if (!mbar_wait(smem_u32(&tempty[acc]), aphase ^ 1u, abortp)) {
                    atomicOr(p.status, MOE_STATUS_TIMEOUT);
                    *abortp = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t dset = tmem + acc * C::kAcc * C::kRows;
                bool failed = false;
                const int nst = (KB + C::kKPS - 1) / C::kKPS;
                for (int s = 0; s < nst; ++s) {
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abortp)) {
                        atomicOr(p.status, MOE_STATUS_TIMEOUT);
                        *abortp = 1;
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    uint8_t* st = stage_base + stage * C::kStage;
                    const int nkb = min(C::kKPS, KB - s * C::kKPS);
#pragma unroll
                    for (int i = 0; i < C::kKPS; ++i) {
                        if (i >= nkb) break;
                        const uint32_t sa = smem_u32(st + i * kTileBytes);
                        const uint32_t sb = smem_u32(st + C::kKPS * kTileBytes + i * C::kBBlk);
                        const uint32_t ssfa = sa + kTileCodeBytes, ssfb = sb + C::kBCodes;
                        const uint32_t sfcol = tmem + C::kAccCols + sfring * C::kSfCols;
                        const uint32_t sfb = sfcol + C::kSfB;
                        tc_cp_sf(sfcol + 0, desc_sf(ssfa));
                        tc_cp_sf(sfcol + 4, desc_sf(ssfa + 512));
#pragma unroll
                        for (int g = 0; g < C::kSg; ++g) {
                            tc_cp_sf(sfb + 4 * g, desc_sf(ssfb + g * 1024));
                            tc_cp_sf(sfb + C::kBsfQ + 4 * g, desc_sf(ssfb + g * 1024 + 512));
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int a = j % C::kAcc;
                            const uint32_t accumulate = (s > 0 || i > 0 || j >= C::kAcc) ? 1u : 0u;
                            mma_mxf4(dset + a * C::kRows, desc_sw128(sa + 32 * j), desc_sw128(sb + 32 * j),
                                     (j & 1) ? idesc_hi : idesc_lo, sfcol + 4 * (j >> 1), sfb + C::kBsfQ * (j >> 1),
                                     accumulate);
                        }
                        sfring = (sfring + 1) % kSfRing;
                    }
                    tc_commit(smem_u32(&empty[stage]));
                    if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                }
                if (failed) break;
                tc_commit(smem_u32(&tfull[acc]));
                if (++acc == C::kDbuf) { acc = 0; aphase ^= 1u; }
            }
        }
    } else {
        // ---------------- epilogue (warps 2..9 -> TMEM lane quarters 2, 3, 0, 1, 2, 3, 0, 1; the
        // first four take columns [0, NT/2), the other four [NT/2, NT))
        const int q = warp & 3;
        const int ew = warp - 2;
        const int c_lo = (ew >> 2) * C::kNH;  // this warp's first column (two warps per quarter)
        const int row = q * 32 + lane;       // accumulator row = weight row within the tile
        int acc = 0;
        uint32_t aphase = 0, ephase = 0;
        const int KBf = p.f / kKB;
        // Two warm-up passes first (a gate/up unit, then a down unit of tile 0) with every global
        // write, atomic and hand-off disabled: they run the epilogue's instructions once while
        // the warps would idle anyway, so the first real units do not fetch them cold.  They
        // read TMEM (allocated, contents unused) and write only this warp's rows of hbuf.
        int warm = (n_keys > 0) ? 2 : 0;
        while (true) {
            const bool dry = warm > 0;
            int unit = -1;
            if (dry) {
                unit = (warm == 2) ? 0 : n0;
                --warm;
            } else {
                if (mbar_wait(smem_u32(&uqfull[qi]), qphase, abortp)) unit = uq[qi];
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&uqempty[qi]));
                if (++qi == kUQ) { qi = 0; qphase ^= 1u; }
            }
            if (unit < 0) break;
            const int ph = unit < n0 ? 0 : 1;
            const PhaseParams& P = p.ph[ph];
            UnitInfo u;
            const bool ok = unit_info<NT>(p, P, ph ? unit - n0 : unit, u);
            if (!dry && !mbar_wait(smem_u32(&tfull[acc]), aphase, abortp)) {
                if (lane == 0) { atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
                break;
            }
            __syncwarp();
            tc_fence_after();
            // D[row][n] = sum over accumulators and terms of column (a*kRows + t*NT + n); this
            // warp's columns n = c_lo + cl
            float vals[C::kNH];
#pragma unroll
            for (int c = 0; c < C::kNH; ++c) vals[c] = 0.f;
            const uint32_t lanebase = tmem + ((uint32_t)(q * 32) << 16) + acc * C::kAcc * C::kRows;
#pragma unroll
            for (int a = 0; a < C::kAcc; ++a)
#pragma unroll
                for (int c0 = 0; c0 < C::kNH; c0 += C::kLdW) {
                    if (c_lo + c0 >= u.ncols) break;   // warp-uniform: columns past ncols are padding
                    uint32_t tmp[kTerms][C::kLdW];
#pragma unroll
                    for (int t = 0; t < kTerms; ++t)
                        tc_ld_issue(lanebase + a * C::kRows + t * NT + c_lo + c0, tmp[t]);
#pragma unroll
                    for (int t = 0; t < kTerms; ++t) {
                        tc_wait_ld(tmp[t]);
#pragma unroll
                        for (int i = 0; i < C::kLdW; ++i) vals[c0 + i] += __uint_as_float(tmp[t][i]);
                    }
                }
            tc_fence_before();
            __syncwarp();
            if (!dry) {
                if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
                if (++acc == C::kDbuf) { acc = 0; aphase ^= 1u; }
            }
            if (!ok) continue;
            if (ph == 1) {
                const int r = u.m * kBM + row;    // output feature
#pragma unroll
                for (int cl = 0; cl < C::kNH; ++cl) {
                    const int c = c_lo + cl;
                    if (c >= u.ncols || dry) continue;
                    p.rows_out[(size_t)(u.brow0 + c) * p.d + r] = vals[cl];
                }
            } else {
                // rows 2i' = gate, 2i'+1 = up of output i' = row/2 within the tile (i = 64m + i')
#pragma unroll
                for (int cl = 0; cl < C::kNH; ++cl) {
                    const int c = c_lo + cl;
                    if (c >= u.ncols) break;
                    const float partner = __shfl_xor_sync(0xffffffffu, vals[cl], 1);
                    if ((lane & 1) == 0) {
                        const float g = vals[cl];
                        hbuf[hidx(c, row >> 1)] = g / (1.0f + expf(-g)) * partner;
                    }
                }
                // hand-off 1: every warp's h values are in hbuf
                __syncwarp();
                if (!dry) {
                    if (lane == 0) mbar_arrive(smem_u32(&epibar[0]));
                    if (!mbar_wait(smem_u32(&epibar[0]), ephase, abortp)) {
                        if (lane == 0) { atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
                        break;
                    }
                    __syncwarp();
                }
                // quantise; a job is (column c, block b of 32 outputs i0 = 64m + 32b): few jobs
                // (a tile of at most 4 rows) one warp each, else one octet of lanes each (32
                // octets over the eight warps); both compute the same terms, written to row c of
                // the tile's h block
                auto h_rows = [&](int c, auto&& write_row) { write_row(u.btile, c); };
                if (u.ncols * 2 <= 8) {
                    for (int job = ew; job < u.ncols * 2; job += C::kEpi) {
                        const int c = job >> 1, b = job & 1;
                        uint4 codes[kTerms];
                        uint32_t scales[kTerms];
                        warp_quantize32(hbuf[hidx(c, 32 * b + lane)], lane, codes, scales);
                        if (dry) continue;
                        const int i0 = u.m * 64 + 32 * b, kb = i0 / kKB, j = (i0 % kKB) / 32;
                        h_rows(c, [&](int htile, int hrow) {
                            if (lane < kTerms) {
                                // lane t writes term t (the codes of every term sit in lane 0)
                                uint4 cv = codes[0];
                                uint32_t sv = scales[0];
#pragma unroll
                                for (int t = 1; t < kTerms; ++t)
                                    if (lane == t) { cv = codes[t]; sv = scales[t]; }
                                *reinterpret_cast<uint4*>(p.h + act_code_off(htile, kb, lane, hrow, j, NT, KBf)) = cv;
                                p.h[act_scale_off(htile, kb, lane, hrow, j, NT, KBf)] = (uint8_t)sv;
                            }
                        });
                    }
                } else {
                    for (int base = 0; base < u.ncols * 2; base += 4 * C::kEpi) {
                        const int job = base + ew * 4 + (lane >> 3), sl = lane & 7;
                        const bool act = job < u.ncols * 2;
                        const int c = act ? job >> 1 : 0, b = job & 1;
                        float v[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) v[i] = act ? hbuf[hidx(c, 32 * b + 4 * sl + i)] : 0.f;
                        uint32_t wd[kTerms], scl[kTerms];
                        octet_quantize32(v, lane, wd, scl);
                        if (!act || dry) continue;
                        const int i0 = u.m * 64 + 32 * b, kb = i0 / kKB, j = (i0 % kKB) / 32;
                        h_rows(c, [&](int htile, int hrow) {
#pragma unroll
                            for (int t = 0; t < kTerms; ++t) {
                                if ((sl & 1) == 0)
                                    *reinterpret_cast<uint32_t*>(p.h + act_code_off(htile, kb, t, hrow, j, NT, KBf) +
                                                                 2 * sl) = wd[t];
                                if (sl == 0) p.h[act_scale_off(htile, kb, t, hrow, j, NT, KBf)] = (uint8_t)scl[t];
                            }
                        });
                    }
                }
                // the h rows are read by the async proxy (bulk copies) of other CTAs
                fence_proxy_async();
                // hand-off 2: hbuf may be overwritten by the next unit; h of this unit is written
                __syncwarp();
                if (dry) continue;
                if (lane == 0) mbar_arrive(smem_u32(&epibar[1]));
                if (!mbar_wait(smem_u32(&epibar[1]), ephase, abortp)) {
                    if (lane == 0) { atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
                    break;
                }
                ephase ^= 1u;
                if (ew == 0 && lane == 0) red_add_release(p.ready + u.key, 1);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmem) : "memory");
}

// ------------------------------------------------------------------ host side

constexpr int kMaxGemmCtas = 160;

// Decode keys for T tokens: at most one per pair (a slot's pairs in chunks of kDecodeNT).
static size_t decode_keys(const moe_dims* m, int T) {
    const size_t n = (size_t)(T > 0 ? T : 1) * m->top_k;
    return n < (size_t)kMaxDecodePairs ? n : (size_t)kMaxDecodePairs;
}
// Capacity of an activation buffer (reduction length K) for T tokens, in tiles of K/256 blocks:
// decode x is one tile of kDecodeNT rows and decode h one such tile per key; the prefill plan
// needs at most act_tiles(m, T) tiles of kPrefillNT rows.
static size_t act_bytes(const moe_dims* m, int T, int K, size_t decode_tiles) {
    const size_t dec = decode_tiles * act_block_bytes(kDecodeNT), pre = act_tiles(m, T) * (size_t)act_block_bytes(kPrefillNT);
    return (size_t)(K / kKB) * (dec > pre ? dec : pre);
}
static size_t act_bytes_x(const moe_dims* m, int T) { return act_bytes(m, T, m->d, 1); }
static size_t act_bytes_h(const moe_dims* m, int T) { return act_bytes(m, T, m->f, decode_keys(m, T)); }
// keys (decode: slot chunks; prefill: tiles) and units of either phase
static size_t max_keys(const moe_dims* m, int T) {
    return act_tiles(m, T) > decode_keys(m, T) ? act_tiles(m, T) : decode_keys(m, T);
}

struct TcBuffers {
    uint8_t *x, *h;        // activation blocks of x (K = d) and h (K = f)
    int32_t* zero;         // counters cleared by the quantiser: work, ready[nkeys]
    size_t nkeys, nzero;
    float* rows;
    int32_t* plan;
};

static size_t counters_of(const moe_dims* m, int T) { return 1 + max_keys(m, T); }

static TcBuffers tc_buffers(const moe_dims* m, int T, char* ws, const WsLayout& L) {
    TcBuffers b;
    char* o = ws + L.tc;
    b.x = reinterpret_cast<uint8_t*>(o); o += align256(act_bytes_x(m, T));
    b.h = reinterpret_cast<uint8_t*>(o); o += align256(act_bytes_h(m, T));
    b.nkeys = max_keys(m, T);
    b.nzero = counters_of(m, T);
    b.zero = reinterpret_cast<int32_t*>(o); o += align256(b.nzero * 4);
    b.rows = reinterpret_cast<float*>(o);
    b.plan = reinterpret_cast<int32_t*>(ws + L.active);
    return b;
}

size_t tc_workspace_bytes(const moe_dims* m, int T) {
    const size_t R = (size_t)(T > 0 ? T : 1) * m->top_k;
    return align256(act_bytes_x(m, T)) + align256(act_bytes_h(m, T)) + align256(counters_of(m, T) * 4) +
           align256(R * m->d * 4);
}

template <int NT>
static int launch_ffn(const FfnParams& p, int grid, cudaStream_t st) {
    using C = GemmCfg<NT>;
    if (cudaFuncSetAttribute(mxf4_ffn_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kBytes) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    if (launch_pdl(mxf4_ffn_kernel<NT>, dim3(grid), dim3(C::kThreads), (size_t)C::kBytes, st, p) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    note_launch(1);
    return MOE_OK;
}

bool tc_supported(const moe_dims* m) { return m->d % kKB == 0 && m->f % kKB == 0; }
bool tc_decode_supported(const moe_dims* m, int T) {
    return tc_supported(m) && T >= 1 && T <= kDecodeNT && T * m->top_k <= kMaxDecodePairs && m->top_k <= 8;
}

static FfnParams ffn_params(const moe_dims* m, const moe_arena* ar, int T, const int32_t* slot, int32_t* status,
                            const TcBuffers& b) {
    FfnParams p{};
    const SlotLayout SL = slot_layout(m->d, m->f);
    p.T = T; p.k = m->top_k; p.E = m->num_experts; p.num_slots = ar->num_slots;
    p.slot = slot; p.arena = reinterpret_cast<const uint8_t*>(ar->base); p.slot_bytes = ar->slot_bytes;
    p.f = m->f; p.d = m->d; p.status = status;
    PhaseParams& g = p.ph[0];
    g.kblocks = m->d / kKB; g.mtiles = 2 * m->f / kBM;
    g.a_off = SL.gu;
    g.b = b.x;
    PhaseParams& dn = p.ph[1];
    dn.kblocks = m->f / kKB; dn.mtiles = m->d / kBM;
    dn.a_off = SL.dn;
    dn.b = b.h;
    p.h = b.h;
    p.work = b.zero;
    p.ready = b.zero + 1;
    return p;
}

// Decode regime (mxf4_decode.cu): one FFN launch with the weights as the MMAs' wide operand,
// on this workspace's x and h tiles, per-pair rows and persistent counters.
int launch_decode_wide(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                       const float* w, uint16_t* y, int32_t* status, uint8_t* xq, uint8_t* hq, float* rows,
                       int32_t* ctr, cudaStream_t st, int num_sms, const RouteArgs* ra, int route_blocks);

int launch_tc_decode(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                     const float* w, uint16_t* y, int32_t* status, char* ws, const WsLayout& L, cudaStream_t st,
                     int num_sms, const RouteArgs* ra, int route_blocks) {
    if (T == 0) return MOE_OK;
    TcBuffers b = tc_buffers(m, T, ws, L);
    return launch_decode_wide(m, ar, T, x, slot, w, y, status, b.x, b.h, b.rows,
                              reinterpret_cast<int32_t*>(ws + L.counter), st, num_sms, ra, route_blocks);
}

__global__ void plan_kernel(int E, int n, const int32_t* offsets, const int32_t* row_src, const int32_t* slot,
                            int nrows, int32_t* plan, int32_t* status, int tile_rows, int max_tiles);

// Prefill regime: x rows quantised into the plan's tiles (grouped by expert), then one FFN
// launch (gate/up per (group, weight tile, row tile) with SwiGLU + h quantisation into the same
// tiles, down to per-row fp32 outputs); the caller's combine sums them in fixed order.
int launch_tc_prefill(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                      const int32_t* offsets, const int32_t* row_src, float* rows_out, int32_t* status, char* ws,
                      const WsLayout& L, cudaStream_t st, int num_sms) {
    if (T == 0) return MOE_OK;
    TcBuffers b = tc_buffers(m, T, ws, L);
    const int d = m->d, k = m->top_k, n = T * k;
    const int max_tiles = (int)act_tiles(m, T);
    plan_kernel<<<1, 1024, 0, st>>>(m->num_experts, n, offsets, row_src, slot, n, b.plan, status, kPrefillNT, max_tiles);
    const long qjobs = (long)T * (d / 32);
    const long qblocks = (qjobs + 255) / 256;
    quantize_tiles_kernel<<<(int)(qblocks > 8L * num_sms ? 8L * num_sms : qblocks), 256, 0, st>>>(
        x, b.plan + plan_pair_off(m->num_experts, max_tiles), k, T, d, b.x, b.zero, (int)b.nzero);
    note_launch(2);
    FfnParams p = ffn_params(m, ar, T, slot, status, b);
    p.plan = b.plan; p.offsets = offsets; p.row_src = row_src;
    p.tile_group = b.plan + plan_tile_group_off(m->num_experts);
    p.grec = reinterpret_cast<const int4*>(b.plan + plan_grec_off(m->num_experts));
    p.rows_out = rows_out;
    p.wait_limit = reinterpret_cast<int32_t*>(ws + L.counter) + kCtrWaitLimit;
    const int grid = num_sms < kMaxGemmCtas ? num_sms : kMaxGemmCtas;
    return launch_ffn<kPrefillNT>(p, grid, st);
}

}  // namespace fp4moe
