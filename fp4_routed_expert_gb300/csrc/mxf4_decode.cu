// mxf4_decode.cu -- the decode-regime expert FFN on the tensor cores (sm_103a), weights as the
// wide operand.
//
// A decode call multiplies a few tokens by the k routed experts' FP4 weights (e2m1 codes with
// a UE8M0 scale per 32 K elements: "DeepSeek-V4.1-Flash on a single NVIDIA DGX Spark", "Why
// it is built this way"), so its cost is the expert weight bytes it streams (same page, "The
// numbers": the bytes of expert weights per generated token set the decode rate).  The
// block-scaled MMA (tcgen05.mma kind::mxf4, M = 128, K = 64) takes the same time per
// instruction for N = 32 and N = 256, so this kernel puts 256 weight rows on the N side of
// every MMA and the activations (kTerms MXFP4 terms of at most 16 tokens: <= 64 of the 128
// rows of M) on the other: one instruction moves twice the weight bytes of a 128-row weight
// tile.  D[m][n] is then activation row m times weight row n, the rows of tokens 8q..8q+7
// in TMEM lane quarter q, term-major inside it (row = 32 (token / 8) + 8 term + token % 8), so
// that one 16x256b load pair hands each thread all kTerms rows of one token.
//
// A unit is one (key, 256 weight rows) pair over the whole K: gate/up (rows 2f interleaved
// gate/up, K = d) and down (rows d, K = f).  The weights' two 128-row tiles of one K block are
// fetched by one tensor-map copy into consecutive 16 KB, their scale atoms by a second one.
#include <cuda.h>

#include "mxf4_common.cuh"
#include "route_select.cuh"

namespace fp4moe {

constexpr int kWRows = 256;                       // weight rows per unit (N of every MMA)
constexpr int kWCodes = kWRows * kKBytes;         // 32 KB of codes per K block
constexpr int kWScales = 2 * kTileScaleBytes;     // the two tiles' scale atoms
constexpr int kDecEpi = 16;                       // epilogue warps: four per TMEM lane quarter
constexpr int kDecThreads = (2 + kDecEpi) * 32;   // producer, MMA issuer, epilogue warps
constexpr int kDecUQ = 8;                         // unit ids in flight from the producer to the other warps
constexpr int kDecMaxK = 8;                       // top-k of a decode call on the tensor cores at most

// Activation blocks of this kernel: block (tile t, K block kb) holds kTerms * NT rows of 128
// code bytes, row r = 32 (token / 8) + 8 term + token % 8 (codes pre-swizzled for SWIZZLE_128B
// by r mod 8), then two 512-byte scale atoms (32-element blocks 0-3 and 4-7 of the K block).
__device__ __forceinline__ int dact_row(int term, int row) { return 32 * (row >> 3) + 8 * term + (row & 7); }
__device__ __forceinline__ int64_t dact_code_off(int tile, int kb, int term, int row, int chunk, int NT, int KB) {
    const int r = dact_row(term, row);
    return ((int64_t)tile * KB + kb) * act_block_bytes(NT) + r * 128 + (((chunk & 7) ^ (r & 7)) << 4);
}
__device__ __forceinline__ int64_t dact_scale_off(int tile, int kb, int term, int row, int j /*0..7*/, int NT, int KB) {
    const int r = dact_row(term, row);
    return ((int64_t)tile * KB + kb) * act_block_bytes(NT) + kTerms * NT * 128 + (j >> 2) * 512 + (r & 31) * 16 +
           (r >> 5) * 4 + (j & 3);
}

struct DecParams {
    // per matrix (0 gate/up, 1 down): 5-D byte maps over the arena, dims {128 bytes of a row,
    // 136 rows of a tile (128 code rows, then 8 rows = the 1 KB of scale atoms), K block, row
    // tile, slot}; codes: box {128, 128, 1, 2, 1}, scales: box {128, 8, 1, 2, 1}
    CUtensorMap wcodes[2];
    CUtensorMap wscales[2];
    int T, k, num_slots, d, f;
    int kblocks[2];                  // d / 256, f / 256
    int units[2];                    // units per key: 2f / 256, d / 256
    const int32_t* slot;             // [T*k]
    const float* w;                  // [T*k] routing weights
    const uint16_t* x_src;           // [T][d] bf16
    uint8_t* x;                      // the x tile (activation blocks, K = d)
    uint8_t* h;                      // one h tile per key (K = f)
    float* rows_out;                 // [T*k][d] per-pair down outputs
    uint16_t* y;                     // [T][d] bf16
    int32_t* status;
    int32_t* work;                   // next unit (zero at launch)
    int32_t* ready;                  // gate/up units finished per key
    int32_t* ycnt;                   // pair rows written per 32 features of y
    int32_t* xready;
    int32_t* exit_ctr;
    const int32_t* wait_limit;       // polls of a wait on another CTA (0: kSpinLimit)
    // Selection handed over by the routing call (sel_epl 4 or 12, the experts per lane of a
    // selecting warp; 0: slot and w are the routing call's outputs): its key records, one
    // release per router block on ra.counter (route_blocks in all); this kernel selects and
    // CTA 0 writes ra.ids, ra.w and ra.slots.
    RouteArgs ra;
    int route_blocks;
    int sel_epl;
};

// Selecting warps' arrays in the stage buffers (free until the producer starts): one
// select_smem_per_warp(kHandoffMaxExperts) region per token, then the chosen slots and ids.
constexpr int kSelWarpBytes = (int)select_smem_per_warp(kHandoffMaxExperts);
constexpr int kSelSlotOff = kDecodeMaxT * kSelWarpBytes;
constexpr int kSelIdOff = kSelSlotOff + kMaxDecodePairs * 4;

template <int EPL>
__device__ __forceinline__ void dec_select(const RouteArgs& a, int t, int lane, float4* rec, float* exk, int* out, SelOut o) {
    select_row<EPL>(a, t, lane, rec, exk, out, o);
}

// Decode keys of one call (one warp, pair i = t*k + j on lane i mod 32): a key is a slot's pairs,
// in order of their appearance, in chunks of at most NT (the rows of one activation tile).
//   pinfo[i]  = key << 5 | row of pair i in its key's tile, -1 for a pair without a valid slot
//   kslot[key] = slot; kinfo[key] = first kplist index << 16 | pairs; kplist = pairs per key in row order
// n_keys and pairs_total (valid pairs) are set on lane 0.  A slot outside [0, num_slots) sets
// MOE_STATUS_BAD_SLOT (when report) and its pair is dropped.  scratch: n ints of shared memory.
template <int NT>
__device__ void decode_key_setup(const int32_t* __restrict__ slot, int n, int num_slots, int32_t* status, bool report,
                                 int lane, int* pinfo, int* kslot, int* kinfo, short* kplist, int* scratch,
                                 int& n_keys, int& pairs_total) {
    if (n <= 32) {
        // one pair per lane, in registers: a slot's pairs are found by one match, a
        // pair's occurrence is the count of its slot's lanes below it
        const unsigned below = (1u << lane) - 1u;
        const int s = lane < n ? slot[lane] : -1;
        const bool ok = lane < n && s >= 0 && s < num_slots;
        if (lane < n && s >= num_slots && report) atomicOr(status, MOE_STATUS_BAD_SLOT);
        const unsigned peers = __match_any_sync(0xffffffffu, ok ? s : -1 - lane);
        const int occ = __popc(peers & below), tot = __popc(peers);
        const bool start = ok && (occ % NT) == 0;
        const unsigned bal = __ballot_sync(0xffffffffu, start);
        const int mykey = start ? __popc(bal & below) : 0;
        // the lane that starts this pair's key: the (occ0 + 1)-th lane of its slot
        const int src = (ok && !start) ? (int)__fns(peers, 0, occ - occ % NT + 1) : lane;
        const int key = __shfl_sync(0xffffffffu, mykey, src);
        // first kplist index of each key: exclusive scan of the key sizes, key order =
        // lane order of the starting pairs
        const int csize = start ? min(NT, tot - occ) : 0;
        int inc = csize;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        const int base = __shfl_sync(0xffffffffu, inc - csize, src);
        if (lane < n) pinfo[lane] = ok ? ((key << 5) | (occ % NT)) : -1;
        if (start) {
            kslot[mykey] = s;
            kinfo[mykey] = (base << 16) | csize;
        }
        if (ok) kplist[base + occ % NT] = (short)lane;
        const unsigned okbal = __ballot_sync(0xffffffffu, ok);
        if (lane == 0) {
            n_keys = __popc(bal);
            pairs_total = __popc(okbal);
        }
    } else {
        int* sslot = scratch;   // the slots, during the setup only
        for (int i = lane; i < n; i += 32) sslot[i] = slot[i];
        __syncwarp();
        // occurrence of each pair's slot among the pairs before it (kept in kplist for
        // now); a pair whose occurrence is a multiple of NT starts a key
        int ord = 0, pairs = 0;
        for (int i0 = 0; i0 < n; i0 += 32) {
            const int i = i0 + lane;
            int s = -1, occ = 0, tot = 0;
            bool ok = false;
            if (i < n) {
                s = sslot[i];
                ok = s >= 0 && s < num_slots;
                if (s >= num_slots && report) atomicOr(status, MOE_STATUS_BAD_SLOT);
                if (ok) {
                    for (int j = 0; j < n; ++j) {
                        const bool same = sslot[j] == s;
                        occ += (same && j < i);
                        tot += same;
                    }
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
                kinfo[key] = min(NT, tot - occ);   // pairs of the key (first index later)
            }
            ord += __popc(bal);
        }
        __syncwarp();
        // the other pairs join the key started by their chunk's first pair
        for (int i = lane; i < n; i += 32) {
            const int s = sslot[i], occ = kplist[i];
            if (s < 0 || s >= num_slots || (occ % NT) == 0) continue;
            const int occ0 = occ - occ % NT;
            for (int j = 0; j < i; ++j)
                if (sslot[j] == s && kplist[j] == occ0) {
                    pinfo[i] = (pinfo[j] & ~31) | (occ % NT);
                    break;
                }
        }
        __syncwarp();
        // each key's first index in kplist: exclusive prefix sum of the key sizes
        int carry = 0;
        for (int k0 = 0; k0 < ord; k0 += 32) {
            const int kk = k0 + lane;
            const int cnt = kk < ord ? kinfo[kk] : 0;
            int inc = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
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
            n_keys = ord;
            pairs_total = pairs;
        }
    }
}

// Shape for NT token rows (8 or 16): a stage is one K block: the activation block first (the
// MMA reads A rows 0..127 from its start; rows past kTerms * NT fall on the weights and feed
// only accumulator lanes that nobody reads), then the weights' codes and scale atoms.
template <int NT>
struct DecCfg {
    static constexpr int kRows = kTerms * NT;                // activation rows (<= 64)
    static constexpr int kQuarters = kRows / 32;             // TMEM lane quarters holding them
    static constexpr int kABlk = act_block_bytes(NT);        // 5 KB (NT = 8) or 9 KB
    static constexpr int kStage = kABlk + kWCodes + kWScales;
    static_assert(kABlk % 1024 == 0 && kStage % 1024 == 0, "operands start on 1024-byte boundaries");
    static_assert(kStage >= 16384, "the A operand's 128 rows stay inside the stage");
    static constexpr int kH = NT * 128 * 4;                  // h values of a gate/up unit (fp32)
    static constexpr int kBudget = 226 * 1024;
    static constexpr int kFit = (kBudget - kH - 2048) / kStage;
    static constexpr int kStages = kFit > 8 ? 8 : kFit;
    static_assert(kStages >= 3, "pipeline depth");
    static constexpr int kBytes = kStages * kStage + kH + 1024 /*barriers*/ + 1024 /*alignment*/;
    // TMEM: accumulator [0, 256); scale ring slots of 48 columns at 256 (A scales +0, +4; B
    // scales +16 + 16 q + 4 g for 32-element-block quarter q and weight tile g: every B base a
    // multiple of 16); the x scales of every K block at 352 (8 columns each) when they fit
    static constexpr int kAcc = 0;
    static constexpr int kRing = 256;
    static constexpr int kSlot = 48;
    static constexpr int kXsf = kRing + kSfRing * kSlot;
};

// 5-D tensor-map load into shared memory with an L2 cache policy.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3, int c4,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar), "l"(policy)
        : "memory");
}

// One launch per decode call, one CTA per SM, every CTA resident:
//   warp 0  producer: takes units from the work list; per K block one tensor-map copy of the
//           weights' codes (two 128-row tiles, 32 KB), one of their scale atoms (2 KB) and one
//           bulk copy of the activation block (x, or the key's h once every gate/up unit of
//           the key has written it)
//   warp 1  MMA issuer (one lane): scale atoms into TMEM, 4 MMAs of N = 256 per K block
//   warps 2..17 epilogue, four per TMEM lane quarter: the warps on the quarters that hold
//           activation rows read the accumulator (each warp 64 of the 256 columns, by
//           16x256b loads that hand a thread every term of one token), add the terms, then
//           gate/up: SwiGLU into shared memory, and one thread per (token, 32-element block)
//           encodes h into kTerms MXFP4 terms in each pair's row of its key's h tile;
//           down: fp32 rows per pair, and the fixed-order combine of every 32 features of y
//           by the warp that completes them
// x is encoded by the CTAs before the wait on the router.  Every wait is bounded; a timeout
// sets MOE_STATUS_TIMEOUT and the CTA drains its own copies and MMAs and exits.  The last CTA
// to exit clears the counters for the next call.
template <int NT>
__global__ void __launch_bounds__(kDecThreads, 1) mxf4_decode_kernel(const __grid_constant__ DecParams p) {
    using C = DecCfg<NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stage_base = smem;
    float* hbuf = reinterpret_cast<float*>(smem + C::kStages * C::kStage);   // [NT][128] h of a gate/up unit
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage + C::kH);
    uint64_t* full = bars;                       // a stage's bytes landed
    uint64_t* empty = bars + C::kStages;         // a stage's MMAs finished
    uint64_t* tfull = bars + 2 * C::kStages;     // accumulator ready
    uint64_t* tempty = tfull + 1;                // accumulator read
    uint64_t* epibar = tempty + 1;               // [2] h hand-offs between the epilogue warps
    uint64_t* uqfull = epibar + 2;               // [kDecUQ] unit id written
    uint64_t* uqempty = uqfull + kDecUQ;         // [kDecUQ] unit id read by the MMA and epilogue warps
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    __shared__ int n_keys_sh, pairs_total_sh;
    __shared__ int pinfo[kMaxDecodePairs];
    __shared__ int kslot[kMaxDecodePairs];
    __shared__ int kinfo[kMaxDecodePairs];
    __shared__ short kplist[kMaxDecodePairs];
    __shared__ int uq[kDecUQ];
    __shared__ int sel_ok_sh, wait_limit_sh;
    static_assert(2 * C::kStages + 4 + 2 * kDecUQ <= 64, "the barriers fit below the routing weights");
    float* selw = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 512);   // [T*k] routing weights

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int kEpi = kDecEpi;
    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(tfull), 1);
        mbar_init(smem_u32(tempty), kEpi);
        mbar_init(smem_u32(&epibar[0]), kEpi);
        mbar_init(smem_u32(&epibar[1]), kEpi);
        for (int i = 0; i < kDecUQ; ++i) {
            mbar_init(smem_u32(&uqfull[i]), 1);
            mbar_init(smem_u32(&uqempty[i]), 1 + kEpi);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_sh)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.wcodes[0])) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.wscales[0])) : "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    volatile int* abortp = &abort_flag;
    const int KBd = p.kblocks[0], KBf = p.kblocks[1];

    // x -> kTerms MXFP4 terms, one epilogue thread per (token, 32-element block), the jobs
    // dealt out by block (a few CTAs hold them all), each warp counting its finished jobs on
    // xready.  This runs before the wait below: x is an input of this call, the kernel ahead
    // (the router) does not write it, and the expert kernel of the previous call has completed
    // before this one launched (the router lets it launch only after its own wait).
    if (warp >= 2) {
        const int nblk = p.d / 32, total = p.T * nblk;
        for (int j0 = blockIdx.x * (kEpi * 32) + (warp - 2) * 32; j0 < total; j0 += gridDim.x * (kEpi * 32)) {
            const int job = j0 + lane;
            if (job < total) {
                const int r = job / nblk, b = job % nblk, kb = b / 8, jb = b % 8;
                const uint4* src = reinterpret_cast<const uint4*>(p.x_src + (size_t)r * p.d + 32 * b);
                float v[32];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint4 w4 = src[u];
                    const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        v[8 * u + 2 * h] = bf16_lo(ww[h]);
                        v[8 * u + 2 * h + 1] = bf16_hi(ww[h]);
                    }
                }
                uint32_t wd[kTerms][4], sc[kTerms];
                thread_quantize32(v, wd, sc);
#pragma unroll
                for (int t = 0; t < kTerms; ++t) {
                    *reinterpret_cast<uint4*>(p.x + dact_code_off(0, kb, t, r, jb, NT, KBd)) =
                        make_uint4(wd[t][0], wd[t][1], wd[t][2], wd[t][3]);
                    p.x[dact_scale_off(0, kb, t, r, jb, NT, KBd)] = (uint8_t)sc[t];
                }
                fence_proxy_async();   // read by the async proxy (bulk copies) of every CTA
            }
            __syncwarp();
            if (lane == 0) red_add_release(p.xready, min(32, total - j0));
        }
    }
    // The setup below runs once per call right after the wait, on cold instructions: run it
    // first on a dummy slot list (one slot per pair) so that its code is fetched while the
    // router still runs.  It writes only shared memory that the real setup overwrites.
    if (warp == 0) {
        int* dummy = reinterpret_cast<int*>(hbuf);
        const int n = p.T * p.k;
        for (int i = lane; i < n; i += 32) dummy[i] = 0;
        __syncwarp();
        int nk = 0, np = 0;
        decode_key_setup<NT>(dummy, n, 1, p.status, false, lane, pinfo, kslot, kinfo, kplist, dummy + kMaxDecodePairs,
                             nk, np);
        __syncwarp();
        // a call that selects here sets up its keys in warp 2: it waits for this warm-up (barrier 2)
        if (p.sel_epl) asm volatile("bar.arrive 2, 64;" ::: "memory");
    }
    unsigned dep_limit = kSpinLimit;
    const int npairs = p.T * p.k;
    if (p.sel_epl) {
        // The routing call handed its key records over.  The next kernel may launch now (it
        // waits for this one before it writes anything this kernel reads); warps 2 .. T + 1
        // select one token each once every router block has released its records (CTA 0 also
        // writes the routing outputs), then warp 2 sets up the keys.
        pdl_trigger();
        int32_t* sel_slot = reinterpret_cast<int32_t*>(stage_base + kSelSlotOff);
        int32_t* sel_id = reinterpret_cast<int32_t*>(stage_base + kSelIdOff);
        const int t = warp - 2;
        if (t >= 0 && t < p.T) {
            if (t == 0 && lane == 0) {
                // the wait limit and the first poll in flight together
                const int wl = ld_relaxed(p.wait_limit);
                int ok = ld_acquire(reinterpret_cast<const int32_t*>(p.ra.counter)) >= p.route_blocks;
                const unsigned lim = wl > 0 ? (unsigned)wl : kSpinLimit;
                for (unsigned i = 1; !ok && i < lim; ++i)
                    ok = ld_acquire(reinterpret_cast<const int32_t*>(p.ra.counter)) >= p.route_blocks;
                if (!ok) {
                    atomicOr(p.status, MOE_STATUS_TIMEOUT);
                    *abortp = 1;
                }
                sel_ok_sh = ok;
                wait_limit_sh = wl;
            }
            __syncwarp();
            asm volatile("bar.sync 1, %0;" ::"r"(32 * p.T) : "memory");   // the selecting warps
            const SelOut o{sel_id + t * p.k, selw + t * p.k, sel_slot + t * p.k, blockIdx.x == 0 ? p.status : nullptr};
            if (sel_ok_sh) {
                uint8_t* wsm = stage_base + (size_t)t * kSelWarpBytes;
                float4* rec = reinterpret_cast<float4*>(wsm);
                float* exk = reinterpret_cast<float*>(wsm + (size_t)p.ra.E * 16);
                int* out = reinterpret_cast<int*>(wsm + (size_t)p.ra.E * 20);
                if (p.sel_epl == 4) dec_select<4>(p.ra, t, lane, rec, exk, out, o);
                else dec_select<12>(p.ra, t, lane, rec, exk, out, o);
            } else {
                for (int j = lane; j < p.k; j += 32) {
                    o.ids[j] = -1;
                    o.w[j] = 0.0f;
                    o.slots[j] = -1;
                }
            }
            __syncwarp();
            if (blockIdx.x == 0)
                for (int j = lane; j < p.k; j += 32) {
                    p.ra.ids[t * p.k + j] = o.ids[j];
                    p.ra.w[t * p.k + j] = o.w[j];
                    p.ra.slots[t * p.k + j] = o.slots[j];
                }
            // the keys, by the first selecting warp once every token is selected
            if (p.T > 1) asm volatile("bar.sync 1, %0;" ::"r"(32 * p.T) : "memory");
            if (t == 0) asm volatile("bar.sync 2, 64;" ::: "memory");   // warp 0's warm-up is done
            if (t == 0)
                decode_key_setup<NT>(sel_slot, npairs, p.num_slots, p.status, blockIdx.x == 0, lane, pinfo, kslot,
                                     kinfo, kplist, reinterpret_cast<int*>(hbuf), n_keys_sh, pairs_total_sh);
        }
    } else {
        // the router's outputs are read from here on; the next kernel (the next call's router)
        // may launch now: before it waits for this kernel in turn it only stages its own weights
        pdl_wait();
        pdl_trigger();
        if (p.wait_limit && *p.wait_limit > 0) dep_limit = (unsigned)*p.wait_limit;
        if (warp == 1)
            for (int i = lane; i < npairs; i += 32) selw[i] = p.w[i];
        if (warp == 0)
            decode_key_setup<NT>(p.slot, npairs, p.num_slots, p.status, blockIdx.x == 0, lane, pinfo, kslot, kinfo,
                                 kplist, reinterpret_cast<int*>(hbuf), n_keys_sh, pairs_total_sh);
    }
    // the keys are known; every role reads their count here, before any of them can abort
    // on a later wait (a selecting CTA whose poll gave up set every slot to -1: no keys)
    __syncthreads();
    if (p.sel_epl && wait_limit_sh > 0) dep_limit = (unsigned)wait_limit_sh;
    const int n_keys = n_keys_sh;
    const int n0 = n_keys * p.units[0], n_all = n0 + n_keys * p.units[1];
    if (n_keys == 0 && blockIdx.x == 0)   // no valid pair: y is zero
        for (int i = tid; i < p.T * p.d; i += blockDim.x) p.y[i] = 0;
    int qi = 0;
    uint32_t qphase = 0;

    if (warp == 0) {
        // ---------------- producer
        if (lane == 0) {
            int stage = 0, ready_key = -1;
            bool x_ok = false;
            // expert weights are read once per call: first out of L2, so that what every call
            // reads (the router rows, x, the counters) stays there
            const uint64_t wpol = l2_evict_first();
            uint32_t phase = 0, issued = 0, issued_parity = 0;   // per-stage bit masks
            bool first = true;
            while (true) {
                // the first unit of CTA b is unit b; the rest come from the counter in order
                int unit = first ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(p.work, 1);
                first = false;
                if (*abortp || unit >= n_all) unit = -1;
                if (!mbar_wait(smem_u32(&uqempty[qi]), qphase ^ 1u, abortp)) {
                    atomicOr(p.status, MOE_STATUS_TIMEOUT);
                    *abortp = 1;
                    unit = -1;
                }
                uq[qi] = unit;
                mbar_arrive(smem_u32(&uqfull[qi]));
                if (++qi == kDecUQ) { qi = 0; qphase ^= 1u; }
                if (unit < 0) break;
                const int ph = unit < n0 ? 0 : 1;
                const int local = ph ? unit - n0 : unit;
                const int key = local / p.units[ph], um = local % p.units[ph];
                const int slot = kslot[key];
                const int KB = p.kblocks[ph];
                const uint8_t* act = ph ? p.h + (int64_t)key * KB * C::kABlk : p.x;
                // A unit whose activations are not ready yet (gate/up: x still being encoded;
                // down: h of its key) gets its weight copies issued into every free stage; the
                // activation copies of those stages follow once they are ready.
                bool have_b = (ph == 0) ? x_ok : (key == ready_key);
                int pend_n = 0, pend_s0 = 0, pend_stage0 = 0;
                auto issue_b = [&](int s, int stg) {
                    bulk_g2s(smem_u32(stage_base + stg * C::kStage), act + (int64_t)s * C::kABlk, C::kABlk,
                             smem_u32(&full[stg]));
                };
                auto flush = [&]() {
                    for (int i = 0; i < pend_n; ++i) issue_b(pend_s0 + i, (pend_stage0 + i) % C::kStages);
                    pend_n = 0;
                };
                auto key_ready = [&](bool block) -> bool {
                    const int32_t* flag = (ph == 0) ? p.xready : p.ready + key;
                    const int target = (ph == 0) ? p.T * (p.d / 32) : p.units[0];
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
                    if (ph == 0) x_ok = true;
                    else ready_key = key;
                    have_b = true;
                    return true;
                };
                for (int s = 0; s < KB; ++s) {
                    if (pend_n == C::kStages) {   // the next stage still waits for its activations
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
                    mbar_expect_tx(bar, C::kStage);
                    tma_load_5d(st + C::kABlk, &p.wcodes[ph], 0, 0, s, 2 * um, slot, bar, wpol);
                    tma_load_5d(st + C::kABlk + kWCodes, &p.wscales[ph], 0, kBM, s, 2 * um, slot, bar, wpol);
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
            int stage = 0, sfring = 0;
            uint32_t phase = 0, aphase = 0;
            const uint32_t idesc_lo = idesc_mxf4(kWRows, 0), idesc_hi = idesc_mxf4(kWRows, 2);
            // every gate/up unit multiplies the same x tile: its scale atoms go into TMEM once
            // (by the CTA's first gate/up unit) when they fit after the scale ring
            const uint32_t xsf = tmem + C::kXsf;
            const bool xsf_fits = C::kXsf + 8 * KBd <= kTmemCols;
            bool xsf_done = false;
            while (true) {
                int unit = -1;
                if (mbar_wait(smem_u32(&uqfull[qi]), qphase, abortp)) unit = uq[qi];
                mbar_arrive(smem_u32(&uqempty[qi]));
                if (++qi == kDecUQ) { qi = 0; qphase ^= 1u; }
                if (unit < 0) break;
                const int ph = unit < n0 ? 0 : 1;
                const int KB = p.kblocks[ph];
                const bool use_xsf = xsf_fits && ph == 0;
                if (!mbar_wait(smem_u32(tempty), aphase ^ 1u, abortp)) {
                    atomicOr(p.status, MOE_STATUS_TIMEOUT);
                    *abortp = 1;
                    break;
                }
                tc_fence_after();
                bool failed = false;
                for (int s = 0; s < KB; ++s) {
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abortp)) {
                        atomicOr(p.status, MOE_STATUS_TIMEOUT);
                        *abortp = 1;
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(stage_base + stage * C::kStage);   // activations (A)
                    const uint32_t sb = sa + C::kABlk;                               // weights (B)
                    const uint32_t ssfa = sa + C::kRows * kKBytes, ssfb = sb + kWCodes;
                    const uint32_t ring = tmem + C::kRing + sfring * C::kSlot;
                    const uint32_t sfa = use_xsf ? xsf + 8 * s : ring, sfb = ring + 16;
                    if (!(use_xsf && xsf_done)) {
                        tc_cp_sf(sfa, desc_sf(ssfa));
                        tc_cp_sf(sfa + 4, desc_sf(ssfa + 512));
                    }
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        tc_cp_sf(sfb + 4 * g, desc_sf(ssfb + g * kTileScaleBytes));
                        tc_cp_sf(sfb + 16 + 4 * g, desc_sf(ssfb + g * kTileScaleBytes + 512));
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        mma_mxf4(tmem + C::kAcc, desc_sw128(sa + 32 * j), desc_sw128(sb + 32 * j),
                                 (j & 1) ? idesc_hi : idesc_lo, sfa + 4 * (j >> 1), sfb + 16 * (j >> 1),
                                 (s > 0 || j > 0) ? 1u : 0u);
                    sfring ^= 1;
                    tc_commit(smem_u32(&empty[stage]));
                    if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                }
                if (failed) break;
                if (use_xsf) xsf_done = true;
                tc_commit(smem_u32(tfull));
                aphase ^= 1u;
            }
        }
    } else {
        // ---------------- epilogue: warp w reads TMEM lane quarter w mod 4 (activation rows
        // 32q.., tokens or key rows 8q..8q+7) and columns [64 sl, +64), sl = (w - 2) / 4
        const int q = warp & 3, ew = warp - 2, sl = ew >> 2;
        const int arow = q * 8 + (lane >> 2);   // token (gate/up) or key row (down) of this lane
        const int cp = lane & 3;                 // its column pair within each group of 8
        uint32_t aphase = 0, ephase = 0;
        // Two warm-up passes first (gate/up unit 0, then down unit n0) with every global write,
        // atomic and hand-off skipped: the epilogue runs once per unit, and instructions fetched
        // cold while every SM streams weights cost microseconds.  They read TMEM (allocated,
        // contents unused) and write only this warp's own part of hbuf, which its real passes
        // write again before any other warp reads it.
        int warm = n_keys > 0 ? 2 : 0;
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
                if (++qi == kDecUQ) { qi = 0; qphase ^= 1u; }
            }
            if (unit < 0) break;
            const int ph = unit < n0 ? 0 : 1;
            const int local = ph ? unit - n0 : unit;
            const int key = local / p.units[ph], um = local % p.units[ph];
            const int ncols = ph ? (kinfo[key] & 0xFFFF) : p.T;   // valid activation rows
            if (!dry && !mbar_wait(smem_u32(tfull), aphase, abortp)) {
                if (lane == 0) { atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
                break;
            }
            __syncwarp();
            tc_fence_after();
            if (q < C::kQuarters) {
                const uint32_t lanebase = tmem + ((uint32_t)(q * 32) << 16) + C::kAcc;
                const int r0u = 256 * um + 64 * sl;   // down: first output feature of this warp
                const int pair = (ph == 1 && arow < ncols) ? kplist[(kinfo[key] >> 16) + arow] : 0;
                // The warp's two 32-column chunks, each as two 16x256b loads (lanes 0-15: terms 0
                // and 1, lanes 16-31: terms 2 and 3 of the quarter's eight rows), all in flight
                // together: thread i gets all four terms of row 8q + i/4 for columns
                // 8g + 2(i%4) + {0, 1}, g = 0..3, and sums them as (t0 + t1) + (t2 + t3).
                {
                    constexpr int cc = 0;
                    uint32_t ra[2][16], rb[2][16];
                    if (!dry) {
#pragma unroll
                        for (int c2 = 0; c2 < 2; ++c2) {
                            tc_ld16_issue(lanebase + 64 * sl + 32 * c2, ra[c2]);
                            tc_ld16_issue(lanebase + (16u << 16) + 64 * sl + 32 * c2, rb[c2]);
                        }
#pragma unroll
                        for (int c2 = 0; c2 < 2; ++c2) {
                            tc_wait_ld(ra[c2]);
                            tc_wait_ld(rb[c2]);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) ra[0][i] = ra[1][i] = rb[0][i] = rb[1][i] = 0u;
                    }
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const int c = cc + c2;
                        float v[4][2];   // [column group g][column 2(i%4) + e]
#pragma unroll
                        for (int g = 0; g < 4; ++g)
#pragma unroll
                            for (int e = 0; e < 2; ++e)
                                v[g][e] = (__uint_as_float(ra[c2][4 * g + e]) + __uint_as_float(ra[c2][4 * g + 2 + e])) +
                                          (__uint_as_float(rb[c2][4 * g + e]) + __uint_as_float(rb[c2][4 * g + 2 + e]));
                        if (ph == 0) {
                            // columns 8g + 2cp (gate) and + 1 (up): h of output 128 um + 32 sl + 16 c + 4 g + cp
                            if (arow < p.T) {
                                float* dst = hbuf + arow * 128 + 32 * sl + 16 * c + cp;
#pragma unroll
                                for (int g = 0; g < 4; ++g) {
                                    const float gt = v[g][0];
                                    dst[4 * g] = gt * __frcp_rn(1.0f + __expf(-gt)) * v[g][1];
                                }
                            }
                        } else if (arow < ncols && !dry) {
                            // column n = output feature 256 um + n of this key row's pair
                            float* dst = p.rows_out + (size_t)pair * p.d + r0u + 32 * c + 2 * cp;
#pragma unroll
                            for (int g = 0; g < 4; ++g)
                                *reinterpret_cast<float2*>(dst + 8 * g) = make_float2(v[g][0], v[g][1]);
                        }
                    }
                }
                if (ph == 1) {
                    // Features [r0u + 32c, +32) of y are complete once every valid pair's rows
                    // there are written: one counter per 32 features, one arrival per warp with
                    // its row count (lane c arrives for chunk c, both in flight at once); the
                    // warp that completes a chunk sums it in fixed order.
                    const int mine = max(0, min(8, ncols - 8 * q));
                    if (mine > 0) {
                        __syncwarp();
                        int l = dry;
                        if (lane < 2 && !dry)
                            l = (atom_add_acq_rel(p.ycnt + r0u / 32 + lane, mine) + mine == pairs_total_sh);
                        const unsigned lastm = __ballot_sync(0xffffffffu, l) & 0x3u;
                        if (lastm) {
                            for (int t = 0; t < p.T; ++t) {
                                // every load of the token first, then the sums in ascending j
                                float rv[2][kDecMaxK], wv[kDecMaxK];
#pragma unroll
                                for (int jj = 0; jj < kDecMaxK; ++jj) {
                                    const int pr = t * p.k + jj;
                                    const bool ok = jj < p.k && pinfo[pr] >= 0;
                                    wv[jj] = ok ? selw[pr] : 0.f;
#pragma unroll
                                    for (int c = 0; c < 2; ++c)
                                        rv[c][jj] = (ok && ((lastm >> c) & 1u))
                                                        ? __ldcg(p.rows_out + (size_t)pr * p.d + r0u + 32 * c + lane)
                                                        : 0.f;
                                }
#pragma unroll
                                for (int c = 0; c < 2; ++c) {
                                    if (!((lastm >> c) & 1u)) continue;
                                    float yv = 0.f;
#pragma unroll
                                    for (int jj = 0; jj < kDecMaxK; ++jj)
                                        if (jj < p.k && pinfo[t * p.k + jj] >= 0) yv = fmaf(wv[jj], rv[c][jj], yv);
                                    if (!dry) p.y[(size_t)t * p.d + r0u + 32 * c + lane] = f32_to_bf16(yv);
                                }
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (!dry) {
                if (lane == 0) mbar_arrive(smem_u32(tempty));
                aphase ^= 1u;
            }
            if (ph == 1) continue;
            // gate/up: every h value of the unit is in hbuf
            if (!dry) {
                if (lane == 0) mbar_arrive(smem_u32(&epibar[0]));
                if (!mbar_wait(smem_u32(&epibar[0]), ephase, abortp)) {
                    if (lane == 0) { atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
                    break;
                }
                __syncwarp();
            }
            // encode: a job is (token n, block b of 32 outputs i0 = 128 um + 32 b), one thread
            // each (no cross-lane steps on the path); the terms go into the row of each of the
            // token's pairs in this key
            {
                const int e = ew * 32 + lane;
                if (e < p.T * 4) {
                    const int n = e >> 2, b = e & 3;
                    float v[32];
                    const float4* src = reinterpret_cast<const float4*>(hbuf + n * 128 + 32 * b);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 t4 = src[i];
                        v[4 * i] = t4.x;
                        v[4 * i + 1] = t4.y;
                        v[4 * i + 2] = t4.z;
                        v[4 * i + 3] = t4.w;
                    }
                    uint32_t wd[kTerms][4], sc[kTerms];
                    thread_quantize32(v, wd, sc);
                    const int i0 = 128 * um + 32 * b, kb = i0 / kKB, j = (i0 % kKB) / 32;
                    if (!dry)
                        for (int jj = 0; jj < p.k; ++jj) {
                            const int pi = pinfo[n * p.k + jj];
                            if (pi < 0 || (pi >> 5) != key) continue;
                            const int hrow = pi & 31;
#pragma unroll
                            for (int t = 0; t < kTerms; ++t) {
                                *reinterpret_cast<uint4*>(p.h + dact_code_off(key, kb, t, hrow, j, NT, KBf)) =
                                    make_uint4(wd[t][0], wd[t][1], wd[t][2], wd[t][3]);
                                p.h[dact_scale_off(key, kb, t, hrow, j, NT, KBf)] = (uint8_t)sc[t];
                            }
                        }
                }
            }
            // the h rows are read by the async proxy (bulk copies) of other CTAs
            fence_proxy_async();
            __syncwarp();
            if (dry) continue;
            if (lane == 0) mbar_arrive(smem_u32(&epibar[1]));
            if (!mbar_wait(smem_u32(&epibar[1]), ephase, abortp)) {
                if (lane == 0) { atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
                break;
            }
            __syncwarp();
            ephase ^= 1u;
            if (ew == 0 && lane == 0) red_add_release(p.ready + key, 1);
        }
    }
    if (p.sel_epl) pdl_wait();   // a call that selects completes after its routing call
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    // the last CTA to leave clears the counters for the next call
    __shared__ int last_cta;
    if (tid == 0) last_cta = (atom_add_acq_rel(p.exit_ctr, 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (last_cta) {
        for (int i = tid; i < n_keys; i += blockDim.x) p.ready[i] = 0;
        for (int i = tid; i < p.d / 32; i += blockDim.x) p.ycnt[i] = 0;
        if (tid == 0) {
            *p.work = 0;
            *p.xready = 0;
            *p.exit_ctr = 0;
            if (p.sel_epl) *reinterpret_cast<int32_t*>(p.ra.counter) = 0;
        }
    }
}

// ------------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, through the runtime (no link against the driver library).
static EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// Maps of one weight matrix (KB K blocks, mtiles row tiles) in every slot of the arena.
static bool weight_maps(CUtensorMap* codes, CUtensorMap* scales, const moe_arena* ar, int64_t matrix_off, int KB,
                        int mtiles) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    void* base = static_cast<uint8_t*>(ar->base) + matrix_off;
    const cuuint64_t dims[5] = {(cuuint64_t)kKBytes, (cuuint64_t)(kTileBytes / kKBytes), (cuuint64_t)KB,
                                (cuuint64_t)mtiles, (cuuint64_t)ar->num_slots};
    const cuuint64_t strides[4] = {(cuuint64_t)kKBytes, (cuuint64_t)kTileBytes, (cuuint64_t)KB * kTileBytes,
                                   (cuuint64_t)ar->slot_bytes};
    const cuuint32_t box_c[5] = {(cuuint32_t)kKBytes, (cuuint32_t)kBM, 1, 2, 1};
    const cuuint32_t box_s[5] = {(cuuint32_t)kKBytes, (cuuint32_t)(kTileScaleBytes / kKBytes), 1, 2, 1};
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (enc(codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, base, dims, strides, box_c, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    return enc(scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, base, dims, strides, box_s, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NT>
static int launch_dec(const DecParams& p, int grid, cudaStream_t st) {
    using C = DecCfg<NT>;
    if (cudaFuncSetAttribute(mxf4_decode_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kBytes) !=
        cudaSuccess)
        return MOE_ERR_LAUNCH;
    if (launch_pdl(mxf4_decode_kernel<NT>, dim3(grid), dim3(kDecThreads), (size_t)C::kBytes, st, p) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    note_launch(1);
    return MOE_OK;
}

// Decode FFN for T <= 16 tokens (x, slot, w from the router; y bf16 [T][d]).  xq, hq: the
// activation tiles (one of 16 rows for x; one per key for h), rows: [T*k][d] fp32, ctr: the
// workspace's persistent counters.  Token tiles of 8 rows up to T = 8, 16 beyond: the lanes of
// one token never mix with another's, so a token's results are the same with either.
int launch_decode_wide(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                       const float* w, uint16_t* y, int32_t* status, uint8_t* xq, uint8_t* hq, float* rows,
                       int32_t* ctr, cudaStream_t st, int num_sms, const RouteArgs* ra, int route_blocks) {
    if (T == 0) return MOE_OK;
    if (m->top_k > kDecMaxK || T > kDecodeNT) return MOE_ERR_DIMS;
    if (ra && (ra->E > kHandoffMaxExperts || ra->T != T || ra->k != m->top_k || route_blocks < 1)) return MOE_ERR_DIMS;
    DecParams p{};
    const SlotLayout SL = slot_layout(m->d, m->f);
    if (!weight_maps(&p.wcodes[0], &p.wscales[0], ar, SL.gu, m->d / kKB, 2 * m->f / kBM) ||
        !weight_maps(&p.wcodes[1], &p.wscales[1], ar, SL.dn, m->f / kKB, m->d / kBM))
        return MOE_ERR_LAUNCH;
    p.T = T; p.k = m->top_k; p.num_slots = ar->num_slots; p.d = m->d; p.f = m->f;
    p.kblocks[0] = m->d / kKB; p.kblocks[1] = m->f / kKB;
    p.units[0] = 2 * m->f / kWRows; p.units[1] = m->d / kWRows;
    p.slot = slot; p.w = w; p.x_src = x; p.x = xq; p.h = hq; p.rows_out = rows; p.y = y; p.status = status;
    p.work = ctr + kCtrFfnWork;
    p.xready = ctr + kCtrFfnXReady;
    p.exit_ctr = ctr + kCtrFfnExit;
    p.ready = ctr + kCtrFfnReady;
    p.ycnt = ctr + kCtrFfnY;
    p.wait_limit = ctr + kCtrWaitLimit;
    if (ra) {
        p.ra = *ra;
        p.route_blocks = route_blocks;
        p.sel_epl = ra->E <= 128 ? 4 : 12;
    }
    const int grid = num_sms < 256 ? num_sms : 256;
    return T <= 8 ? launch_dec<8>(p, grid, st) : launch_dec<kDecodeNT>(p, grid, st);
}

}  // namespace fp4moe
