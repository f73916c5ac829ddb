// ffn_decode_tc.cu -- the expert FFN of a decode call (T <= 16 tokens) on the 5th-generation
// tensor cores (sm_103a), scheduled as a split-K dataflow so that every SM streams weights for
// the whole call.
//
// What is computed is the layer of "DeepSeek-V4.1-Flash on a single NVIDIA DGX Spark" ("Why it
// is built this way": FP4 experts with UE8M0 scales per 32 elements, used as stored): for each
// (token t, choice j) pair with slot s = slot[t*k + j],
//   h = silu(W_gate[s] x_t) * (W_up[s] x_t),   z_(t,j) = W_down[s] h,
//   y_t = sum over j in ascending order of w_(t,j) z_(t,j)   (fp32, then bf16).
// The weights are the slot's e2m1 codes with their UE8M0 scales, multiplied by tcgen05.mma
// kind::mxf4 against activations written as kTerms MXFP4 terms (x ~ q_1 + q_2 + ..., each term
// quantising the residual of the ones before it), accumulated in fp32 in TMEM.
//
// Work.  A key is a slot's pairs (in chunks of at most NT); each key's FFN is cut into units:
//   gate/up unit (key, m, s): weight row tile m (64 gate rows interleaved with 64 up rows) over
//     K split s of d (KCg K blocks of 256); splits 0..SG-2 write their fp32 partial sums to the
//     workspace and count themselves; split SG-1 (the tile's reducer) waits for that count,
//     adds the SG partials in split order, applies SwiGLU and writes h[64m, 64m+64) of the
//     key's pairs as kTerms MXFP4 terms, then counts that h K block (4 tiles per block of 256);
//   down unit (key, m, s): output row tile m over K split s of f (KCd K blocks of h), once the
//     h blocks of that split are complete; writes fp32 partials per pair and counts itself; the
//     last key's split SD-1 (the tile's reducer) waits for the other n_keys * SD - 1 units and
//     combines y[t][128m, +128) for every token: per pair the SD partials in split order, then
//     the pairs in ascending j.
// Every token's arithmetic is the same whatever the other tokens of the call: an MMA column is
// its own dot product, and the splits, the summation orders and the quantisation depend only
// on d and f.
//
// The work list puts a key's down units one key after its gate/up units (gate/up of key 0,
// gate/up of key 1, down of key 0, gate/up of key 2, down of key 1, ...), so that by the time
// a CTA takes a down unit its h blocks are usually complete; CTAs take units from a counter.
//
// One persistent kernel, one CTA per SM, 6 warps: warp 0 producer (bulk copies of weight tiles
// and activation blocks into a ring of stages), warp 1 MMA issuer, warps 2-5 epilogue.  Every
// wait is bounded; a timeout sets MOE_STATUS_TIMEOUT and the CTA drains its copies and exits.
#include "mxf4_common.cuh"

namespace fp4moe {

namespace {

struct DecParams {
    int T, k, d, f, num_slots;
    const int32_t* slot;         // [T*k]
    const float* w;              // [T*k]
    const uint16_t* x;           // [T][d] bf16
    uint16_t* y;                 // [T][d] bf16
    const uint8_t* arena;
    int64_t slot_bytes, gu_off, dn_off;   // slot stride; gate/up and down matrices inside a slot
    int KBd, KBf, MTg, MTd;      // K blocks of d and f; weight row tiles of gate/up (2f/128) and down (d/128)
    int SG, KCg, SD, KCd;        // K splits and K blocks per split: gate/up, down
    uint8_t* xq;                 // x as kTerms MXFP4 terms: one activation tile of NT rows, KBd blocks
    uint8_t* hq;                 // h as kTerms MXFP4 terms: one tile per key, KBf blocks
    float* pgu;                  // gate/up partials [T*k][MTg][SG][128]
    float* pdn;                  // down partials   [T*k][MTd][SD][128]
    int32_t* status;
    int32_t* ctr;                // work, x jobs, x ready, exit ticket (see kDc*), then the tile counters
    const int32_t* wait_limit;   // 0: kSpinLimit polls
};

enum { kDcWork = 0, kDcXJob = 1, kDcXReady = 2, kDcExit = 3, kDcHead = 16 };
constexpr int kDecMaxSplits = 8;   // K splits of either phase at most
constexpr int kMaxTopKDec = 8;     // top-k of a tensor-core decode call at most
constexpr int kDecUQ = 8;   // unit ids in flight from the producer to the MMA and epilogue warps

// counters after the head: gate/up tickets [key][MTg], h blocks [key][KBf], down tickets [MTd]
__host__ __device__ inline int dc_gu_off() { return kDcHead; }
__host__ __device__ inline int dc_h_off(int MTg) { return kDcHead + kTcDecodeMaxKeys * MTg; }
__host__ __device__ inline int dc_dn_off(int MTg, int KBf) { return dc_h_off(MTg) + kTcDecodeMaxKeys * KBf; }

template <int NT>
struct DecCfg {
    static constexpr int kRows = kTerms * NT;                  // B rows: kTerms x NT
    static constexpr int kN = kRows;                           // <= 64: one MMA group
    static constexpr int kAcc = 2;                             // K slices alternate between two chains
    static constexpr int kDbuf = 256 / (kAcc * kRows) > 4 ? 4 : 256 / (kAcc * kRows);
    static_assert(kRows <= 128 && kDbuf >= 2, "decode tile too wide");
    static constexpr int kSfCols = 16;                         // A scales (8) + B scales (8) per K block
    static constexpr int kBBlk = act_block_bytes(NT);
    static constexpr int kKPS = 2;                             // K blocks per stage
    static constexpr int kStage = kKPS * (kTileBytes + kBBlk);
    static constexpr int kH = NT * 66 * 4;                     // h tile of the completing gate/up unit
    static constexpr int kLdW = NT < 16 ? NT : 16;
    static constexpr int kBudget = 226 * 1024;
    static constexpr int kFit = (kBudget - kH - 2048) / kStage;
    static constexpr int kStages = kFit > 8 ? 8 : kFit;
    static constexpr int kBytes = kStages * kStage + kH + 1024 + 1024;
    static_assert(kStages >= 2, "operand tile too large for a two-stage pipeline");
};

// Unit u of the work list -> kind (0 gate/up, 1 down), key, row tile m, split s.
struct DUnit {
    int kind, key, m, s;
};
__device__ __forceinline__ DUnit decode_unit(const DecParams& p, int n_keys, int u) {
    const int nG = p.MTg * p.SG, nD = p.MTd * p.SD;
    DUnit r;
    int seg_kind, key, i;
    if (u < nG) {
        seg_kind = 0; key = 0; i = u;
    } else {
        const int v = u - nG, pairs = n_keys - 1, per = nG + nD;
        if (v < pairs * per) {
            const int q = v / per, rr = v % per;
            if (rr < nG) { seg_kind = 0; key = q + 1; i = rr; }
            else { seg_kind = 1; key = q; i = rr - nG; }
        } else {
            seg_kind = 1; key = n_keys - 1; i = v - pairs * per;
        }
    }
    r.kind = seg_kind;
    r.key = key;
    if (seg_kind == 0) { r.m = i / p.SG; r.s = i % p.SG; }
    else { r.s = i / p.MTd; r.m = i % p.MTd; }
    return r;
}

__device__ __forceinline__ unsigned dec_limit(const DecParams& p) {
    const int v = *p.wait_limit;
    return v > 0 ? (unsigned)v : kSpinLimit;
}

template <int NT>
__global__ void __launch_bounds__(kThreadsGemm, 1) mxf4_decode_kernel(DecParams p) {
    using C = DecCfg<NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stage_base = smem;
    float* hbuf = reinterpret_cast<float*>(smem + C::kStages * C::kStage);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage + C::kH);
    uint64_t* full = bars;                          // [kStages] bytes of a stage landed
    uint64_t* empty = bars + C::kStages;            // [kStages] MMAs of a stage finished
    uint64_t* tfull = bars + 2 * C::kStages;        // [kDbuf] accumulator set ready
    uint64_t* tempty = tfull + C::kDbuf;            // [kDbuf] accumulator set drained
    uint64_t* uqfull = tempty + C::kDbuf;           // [kDecUQ]
    uint64_t* uqempty = uqfull + kDecUQ;            // [kDecUQ]
    uint64_t* setupbar = uqempty + kDecUQ;
    uint64_t* epibar = setupbar + 1;                // the four epilogue warps' rendezvous
    uint64_t* drainbar = setupbar + 2;              // every MMA of the CTA complete
    uint64_t* warmbar = setupbar + 3;               // the warm-up MMAs complete
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    __shared__ int n_keys_sh, pairs_total_sh;
    __shared__ int tick_sh;
    __shared__ int pinfo[kMaxDecodePairs];          // pair -> key << 5 | row in the key's tile, -1: none
    __shared__ int kslot[kMaxDecodePairs];          // key -> slot
    __shared__ int kinfo[kMaxDecodePairs];          // key -> first kplist index << 16 | pairs
    __shared__ short kplist[kMaxDecodePairs];       // the pairs of each key in row order
    __shared__ int uq[kDecUQ];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < C::kDbuf; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1);
            mbar_init(smem_u32(&tempty[a]), 4);
        }
        for (int i = 0; i < kDecUQ; ++i) {
            mbar_init(smem_u32(&uqfull[i]), 1);
            mbar_init(smem_u32(&uqempty[i]), 5);
        }
        mbar_init(smem_u32(setupbar), 1);
        mbar_init(smem_u32(epibar), 4);
        mbar_init(smem_u32(drainbar), 1);
        mbar_init(smem_u32(warmbar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_sh)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    volatile int* abortp = &abort_flag;
    // The producer claims its first unit before the wait below: the work counter was left at
    // zero by the previous call, which completed before the kernel ahead of this one started.
    int pre_unit = -2;
    if (warp == 0 && lane == 0) pre_unit = atomicAdd(p.ctr + kDcWork, 1);
    // x -> kTerms MXFP4 terms, one warp per (token, 32-element block), jobs from a counter; x is
    // an input of this call that the kernel ahead (the router) does not write.
    if (warp >= 2) {
        const int nblk = p.d / 32, total = p.T * nblk;
        while (true) {
            int job = 0;
            if (lane == 0) job = atomicAdd(p.ctr + kDcXJob, 1);
            job = __shfl_sync(0xffffffffu, job, 0);
            if (job >= total) break;
            const int r = job / nblk, b = job % nblk, kb = b / 8, j = b % 8;
            uint4 codes[kTerms];
            uint32_t scales[kTerms];
            warp_quantize32(bf16_to_f32(p.x[(size_t)r * p.d + 32 * b + lane]), lane, codes, scales);
            if (lane < kTerms) {
                uint4 cv = codes[0];
                uint32_t sv = scales[0];
#pragma unroll
                for (int t = 1; t < kTerms; ++t)
                    if (lane == t) { cv = codes[t]; sv = scales[t]; }
                *reinterpret_cast<uint4*>(p.xq + act_code_off(0, kb, lane, r, j, NT, p.KBd)) = cv;
                p.xq[act_scale_off(0, kb, lane, r, j, NT, p.KBd)] = (uint8_t)sv;
            }
            fence_proxy_async();   // read by the bulk copies of every CTA
            __syncwarp();
            if (lane == 0) red_add_release(p.ctr + kDcXReady, 1);
        }
    }
    if (warp == 1 && lane == 0) {
        // Warm-up while the router still runs: one K block of scale copies and MMAs on whatever
        // stage 0 holds, into accumulator set 0 (the first unit overwrites it), so that the
        // first real stage does not pay for a cold issue path.
        const uint32_t sa = smem_u32(stage_base), sb = sa + C::kKPS * kTileBytes;
        const uint32_t sfcol = tmem + 256;
        tc_cp_sf(sfcol + 0, desc_sf(sa + kTileCodeBytes));
        tc_cp_sf(sfcol + 4, desc_sf(sa + kTileCodeBytes + 512));
        tc_cp_sf(sfcol + 8, desc_sf(sb + C::kRows * kKBytes));
        tc_cp_sf(sfcol + 12, desc_sf(sb + C::kRows * kKBytes + 512));
        const uint32_t idesc_lo = idesc_mxf4(C::kN, 0), idesc_hi = idesc_mxf4(C::kN, 2);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            mma_mxf4(tmem + (j % C::kAcc) * C::kRows, desc_sw128(sa + 32 * j), desc_sw128(sb + 32 * j),
                     (j & 1) ? idesc_hi : idesc_lo, sfcol + 4 * (j >> 1), sfcol + 8 + 4 * (j >> 1), j >= C::kAcc ? 1u : 0u);
        tc_commit(smem_u32(warmbar));
        for (unsigned i = 0; i < kSpinLimit; ++i)
            if (mbar_try(smem_u32(warmbar), 0)) break;
    }
    pdl_wait();   // the router's outputs (slots, weights) are read from here on
    const unsigned limit = dec_limit(p);
    if (warp == 0) {
        // keys in order of their first pair: a slot's pairs in chunks of at most NT (pair i on
        // lane i mod 32)
        const int n = p.T * p.k;   // <= kMaxDecodePairs, checked on the host
        if (n <= 32) {
            // one pair per lane, in registers: a slot's pairs are found by one match, a pair's
            // occurrence is the count of its slot's lanes below it
            const unsigned below = (1u << lane) - 1u;
            const int s = lane < n ? p.slot[lane] : -1;
            const bool ok = lane < n && s >= 0 && s < p.num_slots;
            if (lane < n && s >= p.num_slots && blockIdx.x == 0) atomicOr(p.status, MOE_STATUS_BAD_SLOT);
            const unsigned peers = __match_any_sync(0xffffffffu, ok ? s : -1 - lane);
            const int occ = __popc(peers & below), tot = __popc(peers);
            const bool start = ok && (occ % NT) == 0;
            const unsigned bal = __ballot_sync(0xffffffffu, start);
            const int mykey = start ? __popc(bal & below) : 0;
            // the lane that starts this pair's key: the (occ0 + 1)-th lane of its slot
            const int src = (ok && !start) ? (int)__fns(peers, 0, occ - occ % NT + 1) : lane;
            const int key = __shfl_sync(0xffffffffu, mykey, src);
            const int csize = start ? min(NT, tot - occ) : 0;
            int inc = csize;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int yv = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += yv;
            }
            const int base = __shfl_sync(0xffffffffu, inc - csize, src);
            if (lane < n) pinfo[lane] = ok ? ((key << 5) | (occ % NT)) : -1;
            if (start) {
                kslot[mykey] = s;
                kinfo[mykey] = (base << 16) | csize;
            }
            if (ok) kplist[base + occ % NT] = (short)lane;
            const unsigned okbal = __ballot_sync(0xffffffffu, ok);
            __syncwarp();
            if (lane == 0) {
                n_keys_sh = __popc(bal);
                pairs_total_sh = __popc(okbal);
                mbar_arrive(smem_u32(setupbar));
            }
            __syncwarp();
        } else {
        int* sslot = reinterpret_cast<int*>(hbuf);   // the slots, during the setup only
        for (int i = lane; i < n; i += 32) sslot[i] = p.slot[i];
        __syncwarp();
        int ord = 0, pairs = 0;
        for (int i0 = 0; i0 < n; i0 += 32) {
            const int i = i0 + lane;
            int s = -1, occ = 0, tot = 0;
            bool ok = false;
            if (i < n) {
                s = sslot[i];
                ok = s >= 0 && s < p.num_slots;
                if (s >= p.num_slots && blockIdx.x == 0) atomicOr(p.status, MOE_STATUS_BAD_SLOT);
                if (ok)
                    for (int j = 0; j < n; ++j) {
                        const bool same = sslot[j] == s;
                        occ += (same && j < i);
                        tot += same;
                    }
                kplist[i] = (short)occ;
                pinfo[i] = -1;
            }
            pairs += ok;
            const bool start = ok && (occ % NT) == 0;
            const unsigned bal = __ballot_sync(0xffffffffu, start);
            if (start) {
                const int key = ord + __popc(bal & ((1u << lane) - 1u));
                pinfo[i] = key << 5;
                kslot[key] = s;
                kinfo[key] = min(NT, tot - occ);
            }
            ord += __popc(bal);
        }
        __syncwarp();
        for (int i = lane; i < n; i += 32) {
            const int s = sslot[i], occ = kplist[i];
            if (s < 0 || s >= p.num_slots || (occ % NT) == 0) continue;
            const int occ0 = occ - occ % NT;
            for (int j = 0; j < i; ++j)
                if (sslot[j] == s && kplist[j] == occ0) {
                    pinfo[i] = (pinfo[j] & ~31) | (occ % NT);
                    break;
                }
        }
        __syncwarp();
        int carry = 0;
        for (int k0 = 0; k0 < ord; k0 += 32) {
            const int kk = k0 + lane;
            const int cnt = kk < ord ? kinfo[kk] : 0;
            int inc = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int yv = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += yv;
            }
            if (kk < ord) kinfo[kk] = ((carry + inc - cnt) << 16) | cnt;
            carry += __shfl_sync(0xffffffffu, inc, 31);
        }
        __syncwarp();
        for (int i = lane; i < n; i += 32) {
            const int pi = pinfo[i];
            if (pi >= 0) kplist[(kinfo[pi >> 5] >> 16) + (pi & 31)] = (short)i;
        }
        pairs = __reduce_add_sync(0xffffffffu, (uint32_t)pairs);
        if (lane == 0) {
            n_keys_sh = ord;
            pairs_total_sh = pairs;
            mbar_arrive(smem_u32(setupbar));
        }
        __syncwarp();
        }
    }
    if (!mbar_wait(smem_u32(setupbar), 0, abortp)) {
        if (lane == 0) { atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
    }
    const int n_keys = *abortp ? 0 : n_keys_sh;
    const int n_all = n_keys * (p.MTg * p.SG + p.MTd * p.SD);
    // no valid pair: y is zero
    if (n_keys == 0 && blockIdx.x == 0)
        for (int i = tid; i < p.T * p.d; i += blockDim.x) p.y[i] = 0;
    int32_t* gu_cnt = p.ctr + dc_gu_off();
    int32_t* h_cnt = p.ctr + dc_h_off(p.MTg);
    int32_t* dn_cnt = p.ctr + dc_dn_off(p.MTg, p.KBf);
    int qi = 0;
    uint32_t qphase = 0;

    if (warp == 0) {
        // ---------------- producer
        if (lane == 0) {
            int stage = 0;
            bool x_ok = false;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            while (true) {
                int unit;
                if (pre_unit != -2) {
                    unit = *abortp ? -1 : pre_unit;
                    pre_unit = -2;
                } else {
                    unit = *abortp ? -1 : atomicAdd(p.ctr + kDcWork, 1);
                }
                if (unit >= n_all) unit = -1;
                if (!mbar_wait(smem_u32(&uqempty[qi]), qphase ^ 1u, abortp)) {
                    atomicOr(p.status, MOE_STATUS_TIMEOUT);
                    *abortp = 1;
                    unit = -1;
                }
                uq[qi] = unit;
                mbar_arrive(smem_u32(&uqfull[qi]));
                if (++qi == kDecUQ) { qi = 0; qphase ^= 1u; }
                if (unit < 0) break;
                const DUnit u = decode_unit(p, n_keys, unit);
                const uint8_t* sbase = p.arena + (int64_t)kslot[u.key] * p.slot_bytes;
                const int KB = u.kind ? p.KBf : p.KBd, KC = u.kind ? p.KCd : p.KCg;
                const int kb0 = u.s * KC, kb1 = min(KB, kb0 + KC);
                const int64_t a_off = u.kind ? p.dn_off : p.gu_off;
                const uint8_t* bsrc = u.kind ? p.hq + (int64_t)u.key * p.KBf * C::kBBlk : p.xq;
                bool have_b = u.kind ? false : x_ok;
                // activations ready: gate/up -- every x job done; down -- every h block of the split
                auto ready_now = [&]() -> bool {
                    if (u.kind == 0) return ld_acquire(p.ctr + kDcXReady) >= p.T * (p.d / 32);
                    for (int kb = kb0; kb < kb1; ++kb)
                        if (ld_acquire(h_cnt + u.key * p.KBf + kb) < kKB / 64) return false;
                    return true;
                };
                auto wait_ready = [&]() {
                    unsigned spins = 0;
                    while (!ready_now()) {
                        if (++spins > limit || *abortp) {
                            atomicOr(p.status, MOE_STATUS_TIMEOUT);
                            *abortp = 1;
                            break;   // the copies still go out, so that every stage's barrier completes
                        }
                        __nanosleep(64);
                    }
                    fence_proxy_async();
                    if (u.kind == 0) x_ok = true;
                    have_b = true;
                };
                const int nst = (kb1 - kb0 + C::kKPS - 1) / C::kKPS;
                int pend_n = 0, pend_s0 = 0, pend_stage0 = 0;
                auto issue_b = [&](int s, int stg) {
                    const int kb = kb0 + s * C::kKPS, nkb = min(C::kKPS, kb1 - kb);
                    bulk_g2s(smem_u32(stage_base + stg * C::kStage + C::kKPS * kTileBytes), bsrc + (int64_t)kb * C::kBBlk,
                             nkb * C::kBBlk, smem_u32(&full[stg]));
                };
                auto flush = [&]() {
                    for (int i = 0; i < pend_n; ++i) issue_b(pend_s0 + i, (pend_stage0 + i) % C::kStages);
                    pend_n = 0;
                };
                for (int s = 0; s < nst; ++s) {
                    if (pend_n == C::kStages) {   // every stage waits for its activations
                        wait_ready();
                        flush();
                    }
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abortp)) {
                        atomicOr(p.status, MOE_STATUS_TIMEOUT);
                        *abortp = 1;
                        break;
                    }
                    const uint32_t st = smem_u32(stage_base + stage * C::kStage);
                    const uint32_t bar = smem_u32(&full[stage]);
                    const int kb = kb0 + s * C::kKPS, nkb = min(C::kKPS, kb1 - kb);
                    const int64_t atile = (int64_t)u.m * KB + kb;
                    mbar_expect_tx(bar, nkb * (kTileBytes + C::kBBlk));
                    bulk_g2s(st, sbase + a_off + atile * kTileBytes, nkb * kTileBytes, bar);
                    if (!have_b && ready_now()) {
                        fence_proxy_async();
                        if (u.kind == 0) x_ok = true;
                        have_b = true;
                        flush();
                    }
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
                    wait_ready();
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
            // x is the same B operand for every gate/up unit: its scale atoms are copied into TMEM
            // once per K block (after the scale ring) when they fit
            const uint32_t xsf = tmem + 256 + kSfRing * C::kSfCols;
            const bool xsf_fits = 256 + kSfRing * C::kSfCols + p.KBd * 8 <= kTmemCols;
            uint32_t xsf_have[2] = {0u, 0u};   // K blocks (< 64) whose x scales are in TMEM
            while (true) {
                int unit = -1;
                if (mbar_wait(smem_u32(&uqfull[qi]), qphase, abortp)) unit = uq[qi];
                mbar_arrive(smem_u32(&uqempty[qi]));
                if (++qi == kDecUQ) { qi = 0; qphase ^= 1u; }
                if (unit < 0) break;
                const DUnit u = decode_unit(p, n_keys, unit);
                const int KB = u.kind ? p.KBf : p.KBd, KC = u.kind ? p.KCd : p.KCg;
                const int kb0 = u.s * KC, kb1 = min(KB, kb0 + KC);
                const bool use_xsf = xsf_fits && u.kind == 0;
                if (!mbar_wait(smem_u32(&tempty[acc]), aphase ^ 1u, abortp)) {
                    atomicOr(p.status, MOE_STATUS_TIMEOUT);
                    *abortp = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t dset = tmem + acc * C::kAcc * C::kRows;
                bool failed = false;
                const int nst = (kb1 - kb0 + C::kKPS - 1) / C::kKPS;
                for (int s = 0; s < nst; ++s) {
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abortp)) {
                        atomicOr(p.status, MOE_STATUS_TIMEOUT);
                        *abortp = 1;
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    uint8_t* st = stage_base + stage * C::kStage;
                    const int nkb = min(C::kKPS, kb1 - (kb0 + s * C::kKPS));
#pragma unroll
                    for (int i = 0; i < C::kKPS; ++i) {
                        if (i >= nkb) break;
                        const int kb = kb0 + s * C::kKPS + i;
                        const uint32_t sa = smem_u32(st + i * kTileBytes);
                        const uint32_t sb = smem_u32(st + C::kKPS * kTileBytes + i * C::kBBlk);
                        const uint32_t ssfa = sa + kTileCodeBytes, ssfb = sb + C::kRows * kKBytes;
                        const uint32_t sfcol = tmem + 256 + sfring * C::kSfCols;
                        const uint32_t sfb = use_xsf ? xsf + kb * 8 : sfcol + 8;
                        tc_cp_sf(sfcol + 0, desc_sf(ssfa));
                        tc_cp_sf(sfcol + 4, desc_sf(ssfa + 512));
                        const bool have = use_xsf && ((xsf_have[kb >> 5] >> (kb & 31)) & 1u);
                        if (!have) {
                            tc_cp_sf(sfb, desc_sf(ssfb));
                            tc_cp_sf(sfb + 4, desc_sf(ssfb + 512));
                            if (use_xsf) xsf_have[kb >> 5] |= 1u << (kb & 31);
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int a = j % C::kAcc;
                            const uint32_t accumulate = (s > 0 || i > 0 || j >= C::kAcc) ? 1u : 0u;
                            mma_mxf4(dset + a * C::kRows, desc_sw128(sa + 32 * j), desc_sw128(sb + 32 * j),
                                     (j & 1) ? idesc_hi : idesc_lo, sfcol + 4 * (j >> 1), sfb + 4 * (j >> 1), accumulate);
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
            // every MMA issued by this thread has completed before TMEM is released (bounded)
            tc_commit(smem_u32(drainbar));
            for (unsigned i = 0; i < kSpinLimit; ++i)
                if (mbar_try(smem_u32(drainbar), 0)) break;
        }
    } else {
        // ---------------- epilogue (warps 2..5 -> TMEM lane quarters 2, 3, 0, 1)
        const int q = warp & 3;
        const int ew = warp - 2;
        const int row = q * 32 + lane;       // accumulator row = weight row within the tile
        int acc = 0;
        uint32_t aphase = 0, ephase = 0;
        // rendezvous of the four epilogue warps (an mbarrier, so that the wait is bounded)
        auto epi_sync = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(epibar));
            if (!mbar_wait(smem_u32(epibar), ephase, abortp)) {
                if (lane == 0) { atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
            }
            ephase ^= 1u;
        };
        // Ticket: after every epilogue thread's stores, one thread adds one to *counter (a
        // gpu-scope fence first: the rendezvous orders the other threads' stores before it);
        // true, for all four warps, for the unit whose addition completed `target`.  The next
        // ticket's first rendezvous keeps tick_sh until every warp has read it.
        auto ticket = [&](int32_t* counter, int target) -> bool {
            epi_sync();
            if (ew == 0 && lane == 0) {
                __threadfence();
                tick_sh = (atom_add_acq_rel(counter, 1) + 1 == target);
            }
            epi_sync();
            const bool last = tick_sh != 0;
            if (last) __threadfence();
            return last;
        };
        while (true) {
            int unit = -1;
            if (mbar_wait(smem_u32(&uqfull[qi]), qphase, abortp)) unit = uq[qi];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&uqempty[qi]));
            if (++qi == kDecUQ) { qi = 0; qphase ^= 1u; }
            if (unit < 0) break;
            const DUnit u = decode_unit(p, n_keys, unit);
            const int kbase = kinfo[u.key] >> 16, kcnt = kinfo[u.key] & 0xFFFF;
            const int ncols = u.kind ? kcnt : p.T;
            if (!mbar_wait(smem_u32(&tfull[acc]), aphase, abortp)) {
                if (lane == 0) { atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
                break;
            }
            tc_fence_after();
            // D[row][n] = sum over accumulators and terms of column (a*kRows + t*NT + n)
            float vals[NT];
#pragma unroll
            for (int c = 0; c < NT; ++c) vals[c] = 0.f;
            const uint32_t lanebase = tmem + ((uint32_t)(q * 32) << 16) + acc * C::kAcc * C::kRows;
#pragma unroll
            for (int a = 0; a < C::kAcc; ++a)
#pragma unroll
                for (int c0 = 0; c0 < NT; c0 += C::kLdW) {
                    if (c0 >= ncols) break;          // warp-uniform: columns past ncols are padding
                    uint32_t tmp[kTerms][C::kLdW];
#pragma unroll
                    for (int t = 0; t < kTerms; ++t) tc_ld_issue(lanebase + a * C::kRows + t * NT + c0, tmp[t]);
#pragma unroll
                    for (int t = 0; t < kTerms; ++t) {
                        tc_wait_ld(tmp[t]);
#pragma unroll
                        for (int i = 0; i < C::kLdW; ++i) vals[c0 + i] += __uint_as_float(tmp[t][i]);
                    }
                }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
            if (++acc == C::kDbuf) { acc = 0; aphase ^= 1u; }
            if (u.kind == 0) {
                // gate/up split: this unit's partial per pair of the key (column = the pair's
                // token); the unit whose ticket completes the tile adds the SG partials in split
                // order, applies SwiGLU and writes h as MXFP4 terms
                if (p.SG > 1) {
#pragma unroll
                    for (int c = 0; c < NT; ++c) {
                        if (c >= p.T) break;
                        for (int jj = 0; jj < p.k; ++jj) {
                            const int pr = c * p.k + jj, pi = pinfo[pr];
                            if (pi >= 0 && (pi >> 5) == u.key)
                                p.pgu[(((size_t)pr * p.MTg + u.m) * p.SG + u.s) * kBM + row] = vals[c];
                        }
                    }
                    if (!ticket(gu_cnt + u.key * p.MTg + u.m, p.SG)) continue;
                }
#pragma unroll
                for (int c = 0; c < NT; ++c) {
                    if (c >= p.T) break;
                    int pr0 = -1;
                    for (int jj = 0; jj < p.k; ++jj) {
                        const int pi = pinfo[c * p.k + jj];
                        if (pr0 < 0 && pi >= 0 && (pi >> 5) == u.key) pr0 = c * p.k + jj;
                    }
                    float v = vals[c];
                    if (pr0 >= 0 && p.SG > 1) {
                        const float* src = p.pgu + ((size_t)pr0 * p.MTg + u.m) * p.SG * kBM + row;
                        float pv[kDecMaxSplits];
#pragma unroll
                        for (int s2 = 0; s2 < kDecMaxSplits; ++s2)
                            if (s2 < p.SG) pv[s2] = (s2 == u.s) ? vals[c] : __ldcg(src + s2 * kBM);
                        v = pv[0];
#pragma unroll
                        for (int s2 = 1; s2 < kDecMaxSplits; ++s2)
                            if (s2 < p.SG) v = v + pv[s2];
                    }
                    // rows 2i' = gate, 2i'+1 = up of output i' = row/2 within the tile
                    const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
                    if ((lane & 1) == 0) hbuf[hidx(c, row >> 1)] = v / (1.0f + expf(-v)) * partner;
                }
                epi_sync();   // every h value of the tile is in hbuf
                const int KBf = p.KBf;
                for (int base = 0; base < p.T * 2; base += 16) {
                    const int job = base + ew * 4 + (lane >> 3), sl = lane & 7;
                    const bool act = job < p.T * 2;
                    const int c = act ? job >> 1 : 0, b = job & 1;
                    float v[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[i] = act ? hbuf[hidx(c, 32 * b + 4 * sl + i)] : 0.f;
                    uint32_t wd[kTerms], scl[kTerms];
                    octet_quantize32(v, lane, wd, scl);
                    if (!act) continue;
                    const int i0 = u.m * 64 + 32 * b, kb = i0 / kKB, j = (i0 % kKB) / 32;
                    for (int jj = 0; jj < p.k; ++jj) {
                        const int pi = pinfo[c * p.k + jj];
                        if (pi < 0 || (pi >> 5) != u.key) continue;
                        const int hrow = pi & 31;
#pragma unroll
                        for (int t = 0; t < kTerms; ++t) {
                            if ((sl & 1) == 0)
                                *reinterpret_cast<uint32_t*>(p.hq + act_code_off(u.key, kb, t, hrow, j, NT, KBf) + 2 * sl) =
                                    wd[t];
                            if (sl == 0) p.hq[act_scale_off(u.key, kb, t, hrow, j, NT, KBf)] = (uint8_t)scl[t];
                        }
                    }
                }
                fence_proxy_async();   // the h rows are read by the bulk copies of other CTAs
                epi_sync();            // every h write of the tile issued; hbuf free again
                if (ew == 0 && lane == 0) red_add_release(h_cnt + u.key * p.KBf + (u.m * 64) / kKB, 1);
            } else {
                // down split: this unit's partial per pair (column c = row c of the key's tile)
                const int r = u.m * kBM + row;   // output feature
#pragma unroll
                for (int c = 0; c < NT; ++c) {
                    if (c >= ncols) break;
                    const int pr = kplist[kbase + c];
                    p.pdn[(((size_t)pr * p.MTd + u.m) * p.SD + u.s) * kBM + row] = vals[c];
                }
                // the unit whose ticket completes tile m: y rows [128m, 128m + 128) of every
                // token, per pair the splits in order, then the pairs in ascending j
                if (!ticket(dn_cnt + u.m, n_keys * p.SD)) continue;
                for (int t = 0; t < p.T; ++t) {
                    float z[kMaxTopKDec];
#pragma unroll
                    for (int j = 0; j < kMaxTopKDec; ++j) {
                        z[j] = 0.f;
                        if (j < p.k && pinfo[t * p.k + j] >= 0) {
                            const float* src = p.pdn + ((size_t)(t * p.k + j) * p.MTd + u.m) * p.SD * kBM + row;
                            float pv[kDecMaxSplits];
#pragma unroll
                            for (int s2 = 0; s2 < kDecMaxSplits; ++s2)
                                if (s2 < p.SD) pv[s2] = __ldcg(src + s2 * kBM);
                            z[j] = pv[0];
#pragma unroll
                            for (int s2 = 1; s2 < kDecMaxSplits; ++s2)
                                if (s2 < p.SD) z[j] = z[j] + pv[s2];
                        }
                    }
                    float yv = 0.f;
#pragma unroll
                    for (int j = 0; j < kMaxTopKDec; ++j)
                        if (j < p.k && pinfo[t * p.k + j] >= 0) yv = __fadd_rn(yv, __fmul_rn(__ldg(p.w + t * p.k + j), z[j]));
                    p.y[(size_t)t * p.d + r] = f32_to_bf16(yv);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    pdl_trigger();
    // the last CTA to leave clears the counters for the next call
    __shared__ int last_cta;
    if (tid == 0) last_cta = (atom_add_acq_rel(p.ctr + kDcExit, 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (last_cta) {
        for (int i = tid; i < n_keys * p.MTg; i += blockDim.x) gu_cnt[i] = 0;
        for (int i = tid; i < n_keys * p.KBf; i += blockDim.x) h_cnt[i] = 0;
        for (int i = tid; i < p.MTd; i += blockDim.x) dn_cnt[i] = 0;
        if (tid == 0) {
            p.ctr[kDcWork] = 0;
            p.ctr[kDcXJob] = 0;
            p.ctr[kDcXReady] = 0;
            p.ctr[kDcExit] = 0;
        }
    }
}

// K split of a K-block count: about `target` blocks per split, at most kDecMaxSplits splits.
void k_split(int KB, int target, int* S, int* KC) {
    int s = (KB + target - 1) / target;
    s = s < 1 ? 1 : (s > kDecMaxSplits ? kDecMaxSplits : s);
    *KC = (KB + s - 1) / s;
    *S = (KB + *KC - 1) / *KC;
}

template <int NT>
int launch_dec(const DecParams& p, int grid, cudaStream_t st) {
    using C = DecCfg<NT>;
    if (cudaFuncSetAttribute(mxf4_decode_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kBytes) !=
        cudaSuccess)
        return MOE_ERR_LAUNCH;
    if (launch_pdl(mxf4_decode_kernel<NT>, dim3(grid), dim3(kThreadsGemm), (size_t)C::kBytes, st, p) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    note_launch(1);
    return MOE_OK;
}

}  // namespace

size_t dec_counter_words(const moe_dims* m) {
    return (size_t)dc_dn_off(2 * m->f / kBM, m->f / kKB) + m->d / kBM;
}

// Partial sums of the decode kernel for T tokens (T <= kDecodeMaxT).
size_t dec_partial_bytes(const moe_dims* m, int T) {
    const int Tc = T < 1 ? 1 : (T > kDecodeMaxT ? kDecodeMaxT : T);
    int SG, KCg, SD, KCd;
    k_split(m->d / kKB, kDecGuSplitBlocks, &SG, &KCg);
    k_split(m->f / kKB, kDecDnSplitBlocks, &SD, &KCd);
    const size_t pairs = (size_t)Tc * m->top_k;
    return pairs * ((size_t)(2 * m->f / kBM) * SG + (size_t)(m->d / kBM) * SD) * kBM * sizeof(float);
}

int launch_dec_tc(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                  const float* w, uint16_t* y, int32_t* status, uint8_t* xq, uint8_t* hq, float* partials,
                  int32_t* ctr, const int32_t* wait_limit, cudaStream_t st, int num_sms) {
    if (T == 0) return MOE_OK;
    DecParams p{};
    const SlotLayout SL = slot_layout(m->d, m->f);
    p.T = T; p.k = m->top_k; p.d = m->d; p.f = m->f; p.num_slots = ar->num_slots;
    p.slot = slot; p.w = w; p.x = x; p.y = y;
    p.arena = reinterpret_cast<const uint8_t*>(ar->base);
    p.slot_bytes = ar->slot_bytes; p.gu_off = SL.gu; p.dn_off = SL.dn;
    p.KBd = m->d / kKB; p.KBf = m->f / kKB; p.MTg = 2 * m->f / kBM; p.MTd = m->d / kBM;
    k_split(p.KBd, kDecGuSplitBlocks, &p.SG, &p.KCg);
    k_split(p.KBf, kDecDnSplitBlocks, &p.SD, &p.KCd);
    p.xq = xq; p.hq = hq;
    p.pgu = partials;
    p.pdn = partials + (size_t)T * m->top_k * p.MTg * p.SG * kBM;
    p.status = status; p.ctr = ctr; p.wait_limit = wait_limit;
    const int grid = num_sms < 160 ? num_sms : 160;
    return T <= 8 ? launch_dec<8>(p, grid, st) : launch_dec<16>(p, grid, st);
}

}  // namespace fp4moe
