// ffn_stream.cu -- decode-regime expert FFN (T <= 16 tokens) on the CUDA cores: one persistent
// kernel that streams every selected expert's FP4 weights from HBM exactly once, dequantises
// them in registers and reduces with warp shuffles.
//
// Single-token decode is a byte-movement problem ("Fast single-box DeepSeek v4.1 Flash
// runtime": decode byte model, fused matvec geometries; "Start the expert reads before the GPU
// is done", 28 September follow-up: the decode kernels run at 69-100% of the memory roofline),
// so the design goal is that every SM streams the same number of bytes, from its first
// microsecond to its last, with as little cross-SM synchronisation as possible:
//
//  - Keys and stages.  A key is an arena slot with its pairs (token, j) of this call, at most
//    P of them (a slot chosen by more pairs gets several keys).  A stage is one contiguous
//    bulk copy of two 256-element K tiles of a 128-row weight tile (codes and scale atoms,
//    34 KB) plus the activation records of the key's pairs.
//  - Gate/up.  A CTA takes whole 128-row gate/up tiles (all of K, d/512 stages each), the
//    tiles dealt round-robin over the CTAs; its warps keep each row's sum in registers across
//    the stages, and at the tile's end form its 64 SwiGLU values h and write them as an
//    activation record.  No partial sum leaves the SM.
//  - Down.  Split along K into single-stage units that fill every CTA up to the same total:
//    a CTA's next down unit is the next one in key order among all CTAs reaching that point in
//    time, so the CTAs that finish their gate/up tiles first take the keys whose h is complete
//    first.  Units write partial sums.
//  - Combine.  A second, small kernel (launched to start as soon as this one ends) sums each
//    pair's partials in K order and combines y = sum_j w_j z_j in ascending j (ascending expert
//    id) into bf16 -- the fixed-order slot sum of "Start the expert reads before the GPU is
//    done", 30 September follow-up -- with every SM taking part.
//  - Arithmetic.  x (and h) reach the kernel as records of f16 values with one power-of-two
//    fp32 scale per 32 elements (exact for bf16 x); e2m1 pairs become f16 pairs with one
//    conversion instruction, and every product code * activation is exact in the fp32
//    accumulator of a mixed-precision FMA.  Each 32-element block sum is multiplied by its
//    weight scale times its activation scale and added to the row's fp32 total.
//  - Determinism.  Every sum order is fixed by the shapes alone, and a token's arithmetic
//    never involves another token, so row t of a T-token call equals the one-token call on
//    token t bit for bit (multi-row verification reproduces decoding).
//
// Warp 0 produces (one lane issues the bulk copies; a stage's weights go out before its
// activations are ready, so the weight stream never waits on a dependency; it also publishes the
// h tiles its consumers finish), warps 1..8 consume (warp w works on rows 16*(w-1) .. +15 of
// each stage, both K tiles).  Every wait is bounded: a wait that gives up sets
// MOE_STATUS_TIMEOUT, the CTA stops taking work, still lands every copy it issued and exits.
#include <cuda_fp16.h>

#include "moe_internal.cuh"

namespace fp4moe {

namespace {

constexpr int kRunTilesConst = 2;
constexpr int kKW = 2;                               // K tiles of a stage per consumer warp (1 or 2)
constexpr int kCW = 8 * kRunTilesConst / kKW;        // consumer warps: 8 row groups x (2 / kKW) K slices
constexpr int kThreads = 32 * (kCW + 1);             // + producer warp
constexpr int kHQ = 16;                              // finished gate/up tiles queued for publication
constexpr int kRunTiles = 2;                         // K tiles per stage
constexpr int kRunK = kRunTiles * kTileK;            // K elements per stage
constexpr int kWBytes = kRunTiles * kTileBytes;      // weight bytes of a full stage
// Activation record of one token (x) or one pair (h) over one run of 512 K elements: 16
// chunks of 32 f16 at an 80-byte stride (the 16-byte pad spreads the 8 chunks that 8 lanes
// read at once over distinct banks), then 16 fp32 power-of-two scales.
constexpr int kRecStride = 80;
constexpr int kRecScale = 16 * kRecStride;
constexpr int kRecBytes = kRecScale + 64;
constexpr int kMaxKeyPairs = 4;                      // pairs of one key at most (kernel instances: 1, 2, 4)
constexpr int kSmemBudget = 227 * 1024;
constexpr int kHBuf = kMaxKeyPairs * (kRunTilesConst / kKW) * 128 * 4;   // per-tile row sums of the consumer warps


struct StreamParams {
    int T, k, d, f, num_slots;
    int P;                      // pairs per key at most (the host's choice: min(T, kMaxKeyPairs))
    int nstages, stage_bytes;
    int mt_gu, mt_dn;           // 128-row tiles of the gate/up (2f rows) and down (d rows) matrices
    int kt_gu, kt_dn;           // 256-element K tiles: d/256, f/256
    int nr_gu, nr_dn;           // stages per row tile along K: ceil(kt / 2)
    const uint16_t* x;          // bf16 [T, d]
    const int32_t* slot;        // [T*k]
    const float* w;             // [T*k]
    const uint8_t* arena;
    int64_t slot_bytes;
    int64_t off_gu, off_dn;     // matrix offsets inside a slot
    uint16_t* y;                // bf16 [T, d]
    int32_t* status;
    uint8_t* xrec;              // [T][nr_gu] records
    uint8_t* hrec;              // [nr_dn][T*k] records (pair positions of the key table)
    float* part_dn;             // [T*k][mt_dn][nr_dn][2 / kKW][128] down partial sums (per K slice)
    int32_t* ctr;               // counter section
    int32_t* hcnt;              // [keys] gate/up tiles whose h is written
    int32_t* pos_of_pair;       // [T*k] position of each pair in the key table (-1: no slot), for the combine
};

__device__ __forceinline__ int ld_acquire(const int32_t* a) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ int atom_add_acq_rel(int32_t* a, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ void red_add_release(int32_t* a, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// Bulk copy global -> shared with an L2 eviction-priority policy (the weights are read once:
// evict them first so the small records and partials stay in L2).
__device__ __forceinline__ void bulk_g2s_policy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// acc += the 8 codes of word w (element 2i in the low nibble of byte i) times 8 f16
// activations in x0..x3 (element pairs, low half first): one fp32 chain of exact products.
__device__ __forceinline__ float dot8(float acc, uint32_t w, uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .b32 h0, h1, h2, h3;\n\t"
        ".reg .f16 a0, a1, a2, a3, a4, a5, a6, a7, y0, y1, y2, y3, y4, y5, y6, y7;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 h0, b0;\n\tcvt.rn.f16x2.e2m1x2 h1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 h2, b2;\n\tcvt.rn.f16x2.e2m1x2 h3, b3;\n\t"
        "mov.b32 {a0, a1}, h0;\n\tmov.b32 {a2, a3}, h1;\n\tmov.b32 {a4, a5}, h2;\n\tmov.b32 {a6, a7}, h3;\n\t"
        "mov.b32 {y0, y1}, %2;\n\tmov.b32 {y2, y3}, %3;\n\tmov.b32 {y4, y5}, %4;\n\tmov.b32 {y6, y7}, %5;\n\t"
        "fma.rn.f32.f16 %0, a0, y0, %0;\n\tfma.rn.f32.f16 %0, a1, y1, %0;\n\t"
        "fma.rn.f32.f16 %0, a2, y2, %0;\n\tfma.rn.f32.f16 %0, a3, y3, %0;\n\t"
        "fma.rn.f32.f16 %0, a4, y4, %0;\n\tfma.rn.f32.f16 %0, a5, y5, %0;\n\t"
        "fma.rn.f32.f16 %0, a6, y6, %0;\n\tfma.rn.f32.f16 %0, a7, y7, %0;\n\t}"
        : "+f"(acc)
        : "r"(w), "r"(x0), "r"(x1), "r"(x2), "r"(x3));
    return acc;
}

// Power-of-two record scale for a block whose largest magnitude is amax: 2^e with the block
// scaled by 2^-e into [2^14, 2^15) (f16 normal range, no overflow), e clamped to [-100, 100].
__device__ __forceinline__ int rec_exponent(float amax) {
    const uint32_t b = __float_as_uint(amax);
    if (b == 0u) return 0;
    int e = (int)((b >> 23) & 0xFF) - 127 - 14;
    return max(-100, min(100, e));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Dynamic shared memory: stages, then barriers, stage infos, ring entries, the row-sum buffer
// of the gate/up tiles, then the key tables (n = T*k pairs).
struct Smem {
    uint8_t* stage;
    uint64_t* full;      // [nstages] a stage's bytes landed (or the end of work was posted)
    uint64_t* empty;     // [nstages] every consumer warp is done with a stage
    uint64_t* hsync;     // [2] consumer-warp hand-offs at the end of a gate/up tile
    int4* sinfo;         // [nstages] the unit of each stage
    float* hbuf;         // [kMaxKeyPairs][slices][128] row sums of the tile that ends
    int* misc;           // [0] n_keys, [1] valid pairs, [2] abort flag, [3] h tiles finished,
                         // [4 .. 4+kHQ) their keys (a ring; the producer publishes them)
    int* sslot;          // [n] the pairs' slots
    int* pinfo;          // [n] pair -> key << 8 | position within the key, -1: no valid slot
    int* kslot;          // [n] key -> slot
    int* kinfo;          // [n] key -> first position << 16 | pairs
    short* kplist;       // [n] positions -> pair (t*k + j), by key
};

__host__ __device__ inline size_t smem_bytes(int nstages, int stage_bytes, int n) {
    return 1024 + (size_t)nstages * stage_bytes + (size_t)nstages * 16 + 16 + (size_t)nstages * 16 + kHBuf +
           4 * (4 + kHQ + 12) + (size_t)n * 18 + 64;
}

__device__ inline Smem carve(uint8_t* raw, const StreamParams& p) {
    Smem s;
    uint8_t* b = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.stage = b;
    b += (size_t)p.nstages * p.stage_bytes;                 // a multiple of 16
    s.full = reinterpret_cast<uint64_t*>(b);
    s.empty = s.full + p.nstages;
    s.hsync = s.empty + p.nstages;
    s.sinfo = reinterpret_cast<int4*>(s.hsync + 2);
    s.hbuf = reinterpret_cast<float*>(s.sinfo + p.nstages);
    s.misc = reinterpret_cast<int*>(s.hbuf + kHBuf / 4);
    const int n = p.T * p.k;
    s.sslot = s.misc + 4 + kHQ + 12;
    s.pinfo = s.sslot + n;
    s.kslot = s.pinfo + n;
    s.kinfo = s.kslot + n;
    s.kplist = reinterpret_cast<short*>(s.kinfo + n);
    return s;
}

// Keys of this call, by one warp: a slot's pairs in order of appearance, cut into chunks of at
// most P; keys in order of their first pair.  Every CTA builds the same tables.
__device__ void build_keys(const StreamParams& p, Smem& s, int lane) {
    const int n = p.T * p.k, P = p.P;
    for (int i = lane; i < n; i += 32) {
        const int sl = p.slot[i];
        s.sslot[i] = sl;
        if (sl >= p.num_slots && blockIdx.x == 0) atomicOr(p.status, MOE_STATUS_BAD_SLOT);
    }
    __syncwarp();
    int nkeys = 0, npairs = 0;
    for (int i0 = 0; i0 < n; i0 += 32) {
        const int i = i0 + lane;
        int sl = -1, occ = 0, tot = 0;
        bool ok = false;
        if (i < n) {
            sl = s.sslot[i];
            ok = sl >= 0 && sl < p.num_slots;
            if (ok)
                for (int j = 0; j < n; ++j) {
                    const bool same = s.sslot[j] == sl;
                    occ += (same && j < i);
                    tot += same;
                }
            s.pinfo[i] = -1;
            s.kplist[i] = (short)occ;   // the pair's occurrence among its slot's pairs, for now
        }
        const bool start = ok && (occ % P) == 0;
        const unsigned bal = __ballot_sync(0xffffffffu, start);
        if (start) {
            const int key = nkeys + __popc(bal & ((1u << lane) - 1u));
            s.pinfo[i] = key << 8;
            s.kslot[key] = sl;
            s.kinfo[key] = min(P, tot - occ);
        }
        nkeys += __popc(bal);
        npairs += __popc(__ballot_sync(0xffffffffu, ok));
    }
    __syncwarp();
    // every other pair joins the key started by the first pair of its chunk
    for (int i = lane; i < n; i += 32) {
        const int sl = s.sslot[i];
        const int occ = s.kplist[i];
        if (sl < 0 || sl >= p.num_slots || (occ % P) == 0) continue;
        const int occ0 = occ - occ % P;
        for (int j = 0; j < i; ++j)
            if (s.sslot[j] == sl && s.kplist[j] == occ0) {
                s.pinfo[i] = (s.pinfo[j] & ~0xFF) | (occ % P);
                break;
            }
    }
    __syncwarp();
    // first position of each key: exclusive prefix sum of the key sizes
    int carry = 0;
    for (int k0 = 0; k0 < nkeys; k0 += 32) {
        const int kk = k0 + lane;
        const int cnt = kk < nkeys ? s.kinfo[kk] : 0;
        int inc = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        if (kk < nkeys) s.kinfo[kk] = ((carry + inc - cnt) << 16) | cnt;
        carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    __syncwarp();
    for (int i = lane; i < n; i += 32) {
        const int pi = s.pinfo[i];
        if (pi >= 0) s.kplist[(s.kinfo[pi >> 8] >> 16) + (pi & 0xFF)] = (short)i;
    }
    if (lane == 0) {
        s.misc[0] = nkeys;
        s.misc[1] = npairs;
    }
}

// Stage info: x = ph | key << 1 | end << 30, y = m, z = q | nt << 8 | last-of-tile << 12,
// w = first position << 16 | pairs.
__device__ __forceinline__ int4 stage_info(const Smem& s, int ph, int key, int m, int q, int nt, bool last) {
    return make_int4(ph | (key << 1), m, q | (nt << 8) | ((last ? 1 : 0) << 12), s.kinfo[key]);
}

// The down units of CTA b: its l-th one is number v of the list in key order, dealt by time
// slot: a CTA with w gate/up stages processes its l-th down unit at slot w + l, and each slot
// deals the next units of the list to the CTAs present there, in CTA order.  CTAs b < R hold
// one gate/up tile more than the others (R = tiles mod CTAs).
struct DownDeal {
    int G, R, lo, hi, wb;
    __device__ int unit(int b, int l) const {
        const int tau = wb + l;
        long before;
        int rank;
        if (R == 0) {
            before = (long)(tau - lo) * G;
            rank = b;
        } else if (tau < hi) {
            before = (long)(tau - lo) * (G - R);
            rank = b - R;
        } else {
            before = (long)(hi - lo) * (G - R) + (long)(tau - hi) * G;
            rank = b;
        }
        const long v = before + rank;
        return v > 0x3fffffff ? 0x3fffffff : (int)v;
    }
};

// One poll of another CTA's progress: *flag >= target, read with acquire.
__device__ __forceinline__ bool poll_count(const int32_t* flag, int target) { return ld_acquire(flag) >= target; }

template <int KP>
__global__ void __launch_bounds__(kThreads, 1) stream_ffn_kernel(StreamParams p) {
    extern __shared__ uint8_t smem_raw[];
    Smem s = carve(smem_raw, p);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abortp = &s.misc[2];
    if (tid == 0) {
        s.misc[2] = 0;
        s.misc[3] = 0;
        s.misc[4 + kHQ] = 0;
        for (int i = 0; i < p.nstages; ++i) {
            mbar_init(smem_u32(&s.full[i]), 1);
            mbar_init(smem_u32(&s.empty[i]), kCW);
        }
        mbar_init(smem_u32(&s.hsync[0]), kCW);
        mbar_init(smem_u32(&s.hsync[1]), kCW);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // x -> records, one warp per (token, 32-element block), jobs from a global counter (left at
    // zero by the previous call on this workspace) so that the CTAs resident first do them all.
    // x is an input of this call and the kernel that may still be running (the router's) does
    // not write it, so this runs before the wait below.
    if (warp >= 1 && warp <= kCW) {
        const int nblk = p.d / 32, total = p.T * nblk;
        while (true) {
            int job = 0;
            if (lane == 0) job = atomicAdd(p.ctr + kCtrStrXJob, 1);
            job = __shfl_sync(0xffffffffu, job, 0);
            if (job >= total) break;
            const int t = job / nblk, b = job % nblk;
            const float v = bf16_to_f32(p.x[(size_t)t * p.d + 32 * b + lane]);
            const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v))));
            const int e = rec_exponent(amax);
            uint8_t* rec = p.xrec + ((size_t)t * p.nr_gu + b / 16) * kRecBytes;
            const __half hv = __float2half_rn(v * exp2i(-e));
            reinterpret_cast<__half*>(rec + (b % 16) * kRecStride)[lane] = hv;
            if (lane == 0) reinterpret_cast<float*>(rec + kRecScale)[b % 16] = exp2i(e);
            fence_proxy_async();   // read by the bulk copies of every CTA
            __syncwarp();
            if (lane == 0) red_add_release(p.ctr + kCtrStrXReady, 1);
        }
    }
    // everything above overlaps the previous kernel; its outputs are read from here on
    pdl_wait();
    const int32_t wl = p.ctr[kCtrWaitLimit];
    const unsigned wait_limit = wl > 0 ? (unsigned)wl : kSpinLimit;
    if (warp == 0) build_keys(p, s, lane);
    __syncthreads();
    const int nkeys = s.misc[0];
    // the combine kernel finds each pair's partial sums through its position in the key table
    if (blockIdx.x == 0)
        for (int i = tid; i < p.T * p.k; i += blockDim.x) {
            const int pi = s.pinfo[i];
            p.pos_of_pair[i] = pi >= 0 ? (s.kinfo[pi >> 8] >> 16) + (pi & 0xFF) : -1;
        }

    if (warp == 0) {
        // ---------------- producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const int G = gridDim.x, b = blockIdx.x;
            const int n_gut = nkeys * p.mt_gu;
            const int A = n_gut / G, R = n_gut % G;
            const int my_tiles = A + (b < R ? 1 : 0);
            DownDeal deal{G, R, A * p.nr_gu, (A + 1) * p.nr_gu, my_tiles * p.nr_gu};
            const int per_key_dn = p.mt_dn * p.nr_dn, n_dn = nkeys * per_key_dn;
            // item iterator: my gate/up tiles' stages, then my down units
            int it_tile = 0, it_q = 0, it_l = 0;
            bool have = true;
            // pending activations: the npend stages before `stage` in ring order have their weights
            // out and wait for their activation copies (oldest first)
            int npend = 0;
            // dependencies seen complete (each seen once through an acquire and a proxy fence): x,
            // and the keys up to ready_key (a CTA's down units come in increasing key order)
            bool x_ok = false, stop = false;
            int ready_key = -1;
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            unsigned idle = 0, dep_polls = 0;
            int published = 0;   // h tiles of this CTA published so far
            bool have_info = false;   // `info` holds the next item (computed once per item)
            int4 info = make_int4(0, 0, 0, 0);
            while (true) {
                bool progress = false;
                // publish the gate/up tiles whose h the consumers have written (gpu scope: the
                // consumers' writes were handed over through shared memory)
                {
                    const int done = *reinterpret_cast<volatile int*>(&s.misc[3]);
                    if (done != published) {
                        __threadfence_block();
                        for (; published < done; ++published) red_add_release(p.hcnt + s.misc[4 + published % kHQ], 1);
                        *reinterpret_cast<volatile int*>(&s.misc[4 + kHQ]) = published;
                        progress = true;
                    }
                }
                // next item
                if (have && !stop && !have_info) {
                    have_info = true;
                    if (it_tile < my_tiles) {
                        const int g = b + it_tile * G;
                        const int key = g / p.mt_gu, m = g % p.mt_gu;
                        const int nt = min(kRunTiles, p.kt_gu - kRunTiles * it_q);
                        info = stage_info(s, 0, key, m, it_q, nt, it_q == p.nr_gu - 1);
                    } else {
                        const int v = deal.unit(b, it_l);
                        if (v >= n_dn) {
                            have = false;
                        } else {
                            const int key = v / per_key_dn, rem = v % per_key_dn;
                            const int m = rem / p.nr_dn, q = rem % p.nr_dn;
                            info = stage_info(s, 1, key, m, q, min(kRunTiles, p.kt_dn - kRunTiles * q), false);
                        }
                    }
                }
                // 1) its weights into the next free stage
                if (have && !stop && npend < p.nstages && mbar_test(smem_u32(&s.empty[stage]), phase ^ 1u)) {
                    have_info = false;
                    issued &= ~(1u << stage);   // the stage's previous copies have landed and been consumed
                    s.sinfo[stage] = info;
                    const int ph = info.x & 1, key = (info.x >> 1) & 0x3FFF, m = info.y, q = info.z & 0xFF,
                              nt = (info.z >> 8) & 0xF, np = info.w & 0xFFFF;
                    const uint32_t fb = smem_u32(&s.full[stage]);
                    mbar_expect_tx(fb, (uint32_t)nt * kTileBytes + (uint32_t)np * kRecBytes);
                    const uint8_t* wsrc = p.arena + (int64_t)s.kslot[key] * p.slot_bytes + (ph ? p.off_dn : p.off_gu) +
                                          ((int64_t)m * (ph ? p.kt_dn : p.kt_gu) + kRunTiles * q) * kTileBytes;
                    bulk_g2s_policy(smem_u32(s.stage + (size_t)stage * p.stage_bytes), wsrc, (uint32_t)nt * kTileBytes,
                                    fb, pol);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    ++npend;
                    if (++stage == p.nstages) { stage = 0; phase ^= 1u; }
                    if (ph == 0) {
                        if (++it_q == p.nr_gu) { it_q = 0; ++it_tile; }
                    } else {
                        ++it_l;
                    }
                    progress = true;
                }
                // 2) the activations of the oldest pending stage, once its inputs exist
                if (npend > 0) {
                    const int hs = (stage + p.nstages - npend) % p.nstages;
                    const int4 pi = s.sinfo[hs];
                    const int ph = pi.x & 1, key = (pi.x >> 1) & 0x3FFF, q = pi.z & 0xFF;
                    const int first = pi.w >> 16, np = pi.w & 0xFFFF;
                    const bool known = ph == 0 ? x_ok : key <= ready_key;
                    bool ready = known || (ph == 0 ? poll_count(p.ctr + kCtrStrXReady, p.T * (p.d / 32))
                                                   : poll_count(p.hcnt + key, p.mt_gu));
                    if (!ready && (*abortp || ++dep_polls > wait_limit)) {
                        // give up: the copies still go out so that the stage's barrier completes
                        if (!*abortp) atomicOr(p.status, MOE_STATUS_TIMEOUT);
                        *abortp = 1;
                        stop = true;
                        ready = true;
                    }
                    if (ready) {
                        if (!known) {
                            // first sight of this dependency: order the bulk copies after it
                            fence_proxy_async();
                            if (ph == 0) x_ok = true;
                            else ready_key = key;
                        }
                        dep_polls = 0;
                        const uint32_t sdst = smem_u32(s.stage + (size_t)hs * p.stage_bytes) + kWBytes;
                        const uint32_t fb = smem_u32(&s.full[hs]);
                        if (ph == 0) {
                            for (int i = 0; i < np; ++i) {
                                const int t = s.kplist[first + i] / p.k;
                                bulk_g2s(sdst + i * kRecBytes, p.xrec + ((size_t)t * p.nr_gu + q) * kRecBytes, kRecBytes, fb);
                            }
                        } else {
                            bulk_g2s(sdst, p.hrec + ((size_t)q * (p.T * p.k) + first) * kRecBytes, (uint32_t)np * kRecBytes,
                                     fb);
                        }
                        --npend;
                        progress = true;
                    }
                }
                if (npend == 0 && (!have || stop)) break;
                if (*abortp) stop = true;
                if (progress) {
                    idle = 0;
                } else {
                    if (++idle > kSpinLimit) {   // no stage freed for a very long time
                        if (!*abortp) atomicOr(p.status, MOE_STATUS_TIMEOUT);
                        *abortp = 1;
                        stop = true;
                    }
                    // stages complete about a microsecond apart: poll sparingly, so that the two
                    // consumer warps sharing this warp's scheduler keep their issue slots
                    __nanosleep(400);
                }
            }
            // the consumers may still be finishing this CTA's last gate/up tiles: publish them all
            for (unsigned i = 0; published < my_tiles && !*abortp; ++i) {
                const int done = *reinterpret_cast<volatile int*>(&s.misc[3]);
                if (done != published) {
                    __threadfence_block();
                    for (; published < done; ++published) red_add_release(p.hcnt + s.misc[4 + published % kHQ], 1);
                    *reinterpret_cast<volatile int*>(&s.misc[4 + kHQ]) = published;
                } else if (i > kSpinLimit) {
                    atomicOr(p.status, MOE_STATUS_TIMEOUT);
                    *abortp = 1;
                } else {
                    __nanosleep(100);
                }
            }
            // end of work: the consumers see it in the next stage (after its previous use)
            if (!*abortp && mbar_wait(smem_u32(&s.empty[stage]), phase ^ 1u, abortp)) {
                issued &= ~(1u << stage);
                s.sinfo[stage] = make_int4(1 << 30, 0, 0, 0);
                mbar_arrive(smem_u32(&s.full[stage]));
            } else {
                *abortp = 1;   // the consumers stop on the flag
            }
            // every issued copy lands before the CTA may exit (bounded)
            for (int st = 0; st < p.nstages; ++st) {
                if (!((issued >> st) & 1u)) continue;
                const uint32_t ph = (issued_parity >> st) & 1u;
                for (unsigned i = 0; i < kSpinLimit; ++i)
                    if (mbar_try(smem_u32(&s.full[st]), ph)) break;
            }
        }
    } else if (warp <= kCW) {
        // ---------------- consumers
        const int cw = warp - 1, rg = cw & 7, ks = cw >> 3, c = lane & 7, rsub = lane >> 3;
        constexpr int NS = kRunTiles / kKW;          // K slices per stage
        int stage = 0, tiles_done = 0;
        uint32_t phase = 0;
        float tot[KP][4];
#pragma unroll
        for (int a = 0; a < KP; ++a)
#pragma unroll
            for (int i = 0; i < 4; ++i) tot[a][i] = 0.f;
        while (true) {
            if (!mbar_wait(smem_u32(&s.full[stage]), phase, abortp)) {
                if (lane == 0) { if (!*abortp) atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
                break;
            }
            const int4 info = s.sinfo[stage];
            if (info.x & (1 << 30)) break;   // end of work
            const int ph = info.x & 1, m = info.y, q = info.z & 0xFF, nt = (info.z >> 8) & 0xF;
            const bool last = (info.z >> 12) & 1;
            const int first = info.w >> 16, np = info.w & 0xFFFF;
            const uint32_t sb = smem_u32(s.stage + (size_t)stage * p.stage_bytes);
            // this warp's rows r_i = 16 rg + 4 i + rsub, chunk c of the K tiles kt = ks*kKW + u
            uint4 code[kKW][4];
            float wsc[kKW][4];
#pragma unroll
            for (int u = 0; u < kKW; ++u)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int kt = ks * kKW + u;
                    code[u][i] = make_uint4(0, 0, 0, 0);
                    wsc[u][i] = 0.f;
                    if (kt < nt) {
                        const int r = 16 * rg + 4 * i + rsub;
                        const uint32_t tb = sb + kt * kTileBytes;
                        code[u][i] = lds128(tb + r * 128 + ((c ^ (r & 7)) << 4));
                        const uint32_t sw = lds32(tb + kTileCodeBytes + (c >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4);
                        wsc[u][i] = ue8m0_to_f32((sw >> (8 * (c & 3))) & 0xFFu);
                    }
                }
            // dot products of the pairs: per K tile, 4 rows x 32 codes against the pair's 32
            // activations (one record chunk); the block sums times their scales make the stage's
            // row sums (one copy of this loop serves both phases)
            const int nu = min(kKW, nt - ks * kKW);   // K tiles of this warp in this stage (may be <= 0)
            float acc[KP][4];
#pragma unroll
            for (int pi = 0; pi < KP; ++pi) {
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[pi][i] = 0.f;
                if (pi < np) {
#pragma unroll
                    for (int u = 0; u < kKW; ++u) {
                        if (u < nu) {
                            const int kt = ks * kKW + u;
                            const uint32_t ab = sb + kWBytes + pi * kRecBytes + (kt * 8 + c) * kRecStride;
                            const uint4 x0 = lds128(ab), x1 = lds128(ab + 16), x2 = lds128(ab + 32), x3 = lds128(ab + 48);
                            const float xs =
                                __uint_as_float(lds32(sb + kWBytes + pi * kRecBytes + kRecScale + (kt * 8 + c) * 4));
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                float a0 = dot8(0.f, code[u][i].x, x0.x, x0.y, x0.z, x0.w);
                                float a1 = dot8(0.f, code[u][i].y, x1.x, x1.y, x1.z, x1.w);
                                a0 = dot8(a0, code[u][i].z, x2.x, x2.y, x2.z, x2.w);
                                a1 = dot8(a1, code[u][i].w, x3.x, x3.y, x3.z, x3.w);
                                acc[pi][i] = fmaf(a0 + a1, wsc[u][i] * xs, acc[pi][i]);
                            }
                        }
                    }
                }
            }
            if (ph == 0) {
#pragma unroll
                for (int pi = 0; pi < KP; ++pi)
#pragma unroll
                    for (int i = 0; i < 4; ++i) tot[pi][i] += acc[pi][i];
            } else if (nu > 0) {
                // down: rows r_i's partial sums of this unit (K slice ks), the 8 lanes of a row
                // added in a fixed tree, written by lane c == 0
#pragma unroll
                for (int pi = 0; pi < KP; ++pi) {
                    if (pi >= np) break;
                    float* dst = p.part_dn + ((((size_t)(first + pi) * p.mt_dn + m) * p.nr_dn + q) * NS + ks) * 128 +
                                 16 * rg + rsub;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float v = acc[pi][i];
                        v += __shfl_xor_sync(0xffffffffu, v, 1);
                        v += __shfl_xor_sync(0xffffffffu, v, 2);
                        v += __shfl_xor_sync(0xffffffffu, v, 4);
                        if (c == 0) dst[4 * i] = v;
                    }
                }
            }
            // the stage may be refilled: this warp has read all it needs from it
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&s.empty[stage]));
            if (++stage == p.nstages) { stage = 0; phase ^= 1u; }
            if (ph == 0 && last) {
                // gate/up tile complete: row sums into shared memory; warp 0 forms h (rows 2i'
                // gate, 2i'+1 up of h index 64 m + i') and writes its record
                const float* hb = s.hbuf;
#pragma unroll
                for (int pi = 0; pi < KP; ++pi) {
                    if (pi >= np) break;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float v = tot[pi][i];
                        v += __shfl_xor_sync(0xffffffffu, v, 1);
                        v += __shfl_xor_sync(0xffffffffu, v, 2);
                        v += __shfl_xor_sync(0xffffffffu, v, 4);
                        if (c == 0) s.hbuf[(pi * NS + ks) * 128 + 16 * rg + 4 * i + rsub] = v;
                        tot[pi][i] = 0.f;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&s.hsync[0]));
                const uint32_t hpar = tiles_done & 1;
                if (!mbar_wait(smem_u32(&s.hsync[0]), hpar, abortp)) {
                    if (lane == 0) { if (!*abortp) atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
                    break;
                }
                // rows 4l, 4l+2 are the gate rows of h values 2l, 2l+1; rows 4l+1, 4l+3 their up rows
                float hv[KP][2];
                if (cw == 0)
#pragma unroll
                    for (int pi = 0; pi < KP; ++pi) {
                        hv[pi][0] = hv[pi][1] = 0.f;
                        if (pi >= np) break;
                        float4 a = *reinterpret_cast<const float4*>(hb + (pi * NS) * 128 + 4 * lane);
#pragma unroll
                        for (int k2 = 1; k2 < NS; ++k2) {   // the K slices in order
                            const float4 b2 = *reinterpret_cast<const float4*>(hb + (pi * NS + k2) * 128 + 4 * lane);
                            a.x += b2.x; a.y += b2.y; a.z += b2.z; a.w += b2.w;
                        }
                        hv[pi][0] = a.x / (1.0f + expf(-a.x)) * a.y;
                        hv[pi][1] = a.z / (1.0f + expf(-a.z)) * a.w;
                    }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&s.hsync[1]));
                if (!mbar_wait(smem_u32(&s.hsync[1]), hpar, abortp)) {
                    if (lane == 0) { if (!*abortp) atomicOr(p.status, MOE_STATUS_TIMEOUT); *abortp = 1; }
                    break;
                }
                ++tiles_done;
                if (cw == 0) {
#pragma unroll
                    for (int pi = 0; pi < KP; ++pi) {
                        if (pi >= np) break;
                        const float h0 = hv[pi][0], h1 = hv[pi][1];
                        float amax = fmaxf(fabsf(h0), fabsf(h1));
#pragma unroll
                        for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                        const int e = rec_exponent(amax);
                        const float inv = exp2i(-e);
                        const int I = 64 * m + 2 * lane;        // h index of this lane's first value
                        const int run = I / kRunK, P = I % kRunK;
                        uint8_t* rec = p.hrec + ((size_t)run * (p.T * p.k) + first + pi) * kRecBytes;
                        *reinterpret_cast<uint32_t*>(rec + (P / 32) * kRecStride + (P % 32) * 2) = pack_f16x2(h0 * inv, h1 * inv);
                        if ((lane & 15) == 0) reinterpret_cast<float*>(rec + kRecScale)[P / 32] = exp2i(e);
                    }
                    fence_proxy_async();   // read by the bulk copies of other CTAs
                    __syncwarp();
                    // hand the tile to the producer, which publishes it (a queue of kHQ keys)
                    if (lane == 0) {
                        const int mine = s.misc[3];
                        bool room = false;
                        for (unsigned i = 0; i < kSpinLimit; ++i) {
                            if (mine - *reinterpret_cast<volatile int*>(&s.misc[4 + kHQ]) < kHQ) { room = true; break; }
                            if (*abortp) break;
                        }
                        if (room) {
                            s.misc[4 + mine % kHQ] = (info.x >> 1) & 0x3FFF;
                            __threadfence_block();
                            *reinterpret_cast<volatile int*>(&s.misc[3]) = mine + 1;
                        } else {
                            if (!*abortp) atomicOr(p.status, MOE_STATUS_TIMEOUT);
                            *abortp = 1;
                        }
                    }
                    __syncwarp();
                }
            }
        }
    }
    // the combine kernel may become resident now; it waits for this grid's completion
    pdl_trigger();
    __syncthreads();
    // the last CTA to leave clears this call's counters for the next call
    __shared__ int last_cta;
    if (tid == 0) last_cta = (atom_add_acq_rel(p.ctr + kCtrStrExit, 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (last_cta) {
        for (int i = tid; i < nkeys; i += blockDim.x) p.hcnt[i] = 0;
        if (tid == 0) {
            p.ctr[kCtrStrXJob] = 0;
            p.ctr[kCtrStrXReady] = 0;
            p.ctr[kCtrStrExit] = 0;
        }
    }
}

// The weighted combine of a decode call, after the expert kernel (programmatic dependent
// launch: it becomes resident early and waits for that kernel's completion).  A block owns
// one token's 128-feature output tile: thread (quad, jj) sums pair jj's partial sums for its
// 4 features in K order (the loads of a pair issued together), and the threads of jj = 0 fold
// the pairs in ascending j, y = bf16(sum_j w_j z_j) -- the fixed-order slot sum.
struct CombineParams {
    int T, k, d, mt_dn, nparts, kt_dn;
    const float* part;          // [T*k][mt_dn][nparts][128]
    const int32_t* pos_of_pair; // [T*k]
    const float* w;             // [T*k]
    uint16_t* y;                // [T, d]
};

__global__ void __launch_bounds__(256) stream_combine_kernel(CombineParams c) {
    __shared__ float4 zs[8][32];
    pdl_wait();
    const int t = blockIdx.y, m = blockIdx.x;
    const int quad = threadIdx.x & 31, jj = threadIdx.x >> 5;
    constexpr int NS = kRunTiles / kKW;
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < c.k; j0 += 8) {
        const int j = j0 + jj;
        float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        const int pos = j < c.k ? c.pos_of_pair[t * c.k + j] : -1;
        if (pos >= 0) {
            const float* src = c.part + (((size_t)pos * c.mt_dn + m) * c.nparts) * 128 + 4 * quad;
            for (int b0 = 0; b0 < c.nparts; b0 += 8) {
                float4 v8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int idx = b0 + u, q = idx / NS, k2 = idx % NS;
                    const bool have = idx < c.nparts && k2 * kKW < min(kRunTiles, c.kt_dn - kRunTiles * q);
                    v8[u] = have ? __ldcg(reinterpret_cast<const float4*>(src + (size_t)idx * 128)) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int idx = b0 + u, q = idx / NS, k2 = idx % NS;
                    if (idx < c.nparts && k2 * kKW < min(kRunTiles, c.kt_dn - kRunTiles * q)) {
                        z.x += v8[u].x; z.y += v8[u].y; z.z += v8[u].z; z.w += v8[u].w;
                    }
                }
            }
        }
        zs[jj][quad] = z;
        __syncthreads();
        if (jj == 0)
            for (int u = 0; u < 8 && j0 + u < c.k; ++u) {
                if (c.pos_of_pair[t * c.k + j0 + u] < 0) continue;   // no slot: contributes nothing
                const float wj = c.w[t * c.k + j0 + u];
                const float4 zz = zs[u][quad];
                y.x = __fadd_rn(y.x, __fmul_rn(wj, zz.x));
                y.y = __fadd_rn(y.y, __fmul_rn(wj, zz.y));
                y.z = __fadd_rn(y.z, __fmul_rn(wj, zz.z));
                y.w = __fadd_rn(y.w, __fmul_rn(wj, zz.w));
            }
        __syncthreads();
    }
    if (jj == 0) {
        const uint32_t lo = (uint32_t)f32_to_bf16(y.x) | ((uint32_t)f32_to_bf16(y.y) << 16);
        const uint32_t hi = (uint32_t)f32_to_bf16(y.z) | ((uint32_t)f32_to_bf16(y.w) << 16);
        *reinterpret_cast<uint2*>(c.y + (size_t)t * c.d + 128 * m + 4 * quad) = make_uint2(lo, hi);
    }
}

// Workspace pieces for T tokens (T <= 16).
struct StreamWs {
    size_t xrec, hrec, part_dn, pos, total;
};
StreamWs stream_ws(const moe_dims* m, int T) {
    const size_t Tc = (size_t)(T < 1 ? 1 : (T > kDecodeMaxT ? kDecodeMaxT : T));
    const size_t n = Tc * m->top_k;
    const size_t kt_gu = m->d / kTileK, kt_dn = m->f / kTileK;
    const size_t nr_gu = (kt_gu + 1) / 2, nr_dn = (kt_dn + 1) / 2;
    const size_t mt_gu = 2 * (size_t)m->f / kTileRows, mt_dn = (size_t)m->d / kTileRows;
    StreamWs w;
    size_t o = 0;
    w.xrec = o;    o = align256(o + Tc * nr_gu * kRecBytes);
    w.hrec = o;    o = align256(o + nr_dn * n * kRecBytes);
    w.part_dn = o; o = align256(o + n * mt_dn * nr_dn * (kRunTilesConst / kKW) * 128 * 4);
    w.pos = o;     o = align256(o + n * 4);
    (void)mt_gu;
    w.total = o;
    return w;
}

}  // namespace

size_t stream_workspace_bytes(const moe_dims* m, int T) { return stream_ws(m, T).total; }

int launch_stream_ffn(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                      const float* w, uint16_t* y, int32_t* status, char* ws, const WsLayout& L, cudaStream_t st,
                      int num_sms) {
    if (T == 0) return MOE_OK;
    if (T > kDecodeMaxT) return MOE_ERR_TOKENS;
    StreamParams p{};
    p.T = T; p.k = m->top_k; p.d = m->d; p.f = m->f; p.num_slots = ar->num_slots;
    p.P = T == 1 ? 1 : (T == 2 ? 2 : kMaxKeyPairs);
    p.stage_bytes = kWBytes + p.P * kRecBytes;
    const int n = T * m->top_k;
    int ns = 8;
    while (ns > 2 && smem_bytes(ns, p.stage_bytes, n) > (size_t)kSmemBudget) --ns;
    p.nstages = ns;
    p.mt_gu = 2 * m->f / kTileRows; p.mt_dn = m->d / kTileRows;
    p.kt_gu = m->d / kTileK; p.kt_dn = m->f / kTileK;
    p.nr_gu = (p.kt_gu + 1) / 2; p.nr_dn = (p.kt_dn + 1) / 2;
    p.x = x; p.slot = slot; p.w = w;
    p.arena = reinterpret_cast<const uint8_t*>(ar->base);
    p.slot_bytes = ar->slot_bytes;
    const SlotLayout SL = slot_layout(m->d, m->f);
    p.off_gu = SL.gu; p.off_dn = SL.dn;
    p.y = y; p.status = status;
    const StreamWs W = stream_ws(m, T);
    char* base = ws + L.stream;
    p.xrec = reinterpret_cast<uint8_t*>(base + W.xrec);
    p.hrec = reinterpret_cast<uint8_t*>(base + W.hrec);
    p.part_dn = reinterpret_cast<float*>(base + W.part_dn);
    p.ctr = reinterpret_cast<int32_t*>(ws + L.counter);
    p.hcnt = p.ctr + stream_hcnt_off(m);
    p.pos_of_pair = reinterpret_cast<int32_t*>(base + W.pos);
    const size_t smem = smem_bytes(ns, p.stage_bytes, n);
    void (*kern)(StreamParams) = p.P == 1 ? stream_ffn_kernel<1> : (p.P == 2 ? stream_ffn_kernel<2> : stream_ffn_kernel<4>);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    if (launch_pdl(kern, dim3(num_sms), dim3(kThreads), smem, st, p) != cudaSuccess) return MOE_ERR_LAUNCH;
    CombineParams c{};
    c.T = T; c.k = m->top_k; c.d = m->d; c.mt_dn = p.mt_dn; c.nparts = p.nr_dn * (kRunTiles / kKW); c.kt_dn = p.kt_dn;
    c.part = p.part_dn; c.pos_of_pair = p.pos_of_pair; c.w = w; c.y = y;
    if (launch_pdl(stream_combine_kernel, dim3(p.mt_dn, T), dim3(256), 0, st, c) != cudaSuccess) return MOE_ERR_LAUNCH;
    note_launch(1);
    note_launch(1);
    return MOE_OK;
}

}  // namespace fp4moe
