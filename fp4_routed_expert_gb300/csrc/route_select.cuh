// route_select.cuh -- the router's key records and their certified top-k selection, shared
// by the router kernels and by the decode expert kernel, which selects its experts itself
// when a routing call hands it the key records (moe_layer_decode_fp4).
//
// Each (token, expert) pair has a 16-byte key record {point key, klo, khi, score}: the key
// interval [klo, khi] holds the exact key sigma(l32) + bias (l32 the exact logit rounded once
// to fp32), score < 0 marks an expert that is not resident.  A warp selects one token's top-k
// from its records; whatever the records' widths, the chosen set and weights are those of the
// exact keys (ties to the lower expert id).
#pragma once

#include "moe_internal.cuh"

namespace fp4moe {

struct RouteArgs {
    int T, d, E, k;
    const uint16_t* x;
    const uint16_t* wr;
    const float* bias;
    const int32_t* table;
    int32_t* ids;
    float* w;
    int32_t* slots;
    int32_t* status;
    float4* keys;      // [T, E] key records
    float* xnorm;      // [T]   (prefill bound)
    float* wnorm;      // [E]   (prefill bound)
    unsigned* counter;
    float bound_coef;  // prefill: gamma_L * (1 + 2^-10); decode: gamma_(c-1) + gamma_m^2 + 2^-34
    float refine_coef; // the decode bound for chunks of one product (selection's refinement)
    int dec_epb;       // decode: experts per block and round (1 .. kDecodeWarps)
    int handoff;       // decode: publish the records on counter, select nothing (the expert kernel selects)
};

// Where a selecting warp writes token t's k outputs (ascending expert id, -1 / 0 / -1 past
// the chosen ones), and the status word it reports to (null: report nothing).
struct SelOut {
    int32_t* ids;
    float* w;
    int32_t* slots;
    int32_t* status;
};
// Experts of a call whose expert kernel selects (12 per lane of its selecting warps).
constexpr int kHandoffMaxExperts = 384;

// Decode router for a call whose expert kernel selects: key records only, one release per
// block on a.counter.  *ra receives the arguments of the selection, *blocks the router's
// grid size.  Returns 1, launching nothing, when the call takes another router path or has
// more than kHandoffMaxExperts experts.
int launch_route_handoff(const moe_dims* m, int T, const uint16_t* x, const uint16_t* wr, const float* bias,
                         const int32_t* table, int32_t* ids, float* w, int32_t* slots, int32_t* status, char* ws,
                         const WsLayout& L, cudaStream_t st, int num_sms, RouteArgs* ra, int* blocks);

// The routing call's own outputs for token t.
__device__ __forceinline__ SelOut route_out(const RouteArgs& a, int t) {
    return SelOut{a.ids + (size_t)t * a.k, a.w + (size_t)t * a.k, a.slots + (size_t)t * a.k, a.status};
}

// ------------------------------------------------------------------ exact logit (Kulisch)

constexpr int kLimbs = 18;   // 18 x 32 bits hold any sum of up to 2^30 bf16*bf16 products
constexpr int kUnit = 266;   // fixed point unit 2^-266 (smallest product quantum)

__device__ __forceinline__ uint32_t limb_window(const uint32_t* dig, int bit) {
    // 32 bits of the big number starting at bit index `bit` (bit >= 0)
    int li = bit >> 5, sh = bit & 31;
    uint64_t lo = dig[li];
    uint64_t hi = (li + 1 < kLimbs) ? dig[li + 1] : 0u;
    return (uint32_t)(((hi << 32) | lo) >> sh);
}

// Exact x.w rounded once to fp32, computed by the whole warp (every lane returns it).
inline __device__ __noinline__ float exact_dot_bf16_warp(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w,
                                     int d, int lane) {
    long long acc[kLimbs];
#pragma unroll
    for (int i = 0; i < kLimbs; ++i) acc[i] = 0;
    // lane reads 8 consecutive bf16 of each vector per step (d is a multiple of 256)
    for (int base = lane * 8; base < d; base += 256) {
        const uint4 xv = *reinterpret_cast<const uint4*>(x + base);
        const uint4 wv = *reinterpret_cast<const uint4*>(w + base);
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int h = 0; h < 8; ++h) {
            const uint32_t bx = (xw[h >> 1] >> (16 * (h & 1))) & 0xFFFFu;
            const uint32_t bw = (ww[h >> 1] >> (16 * (h & 1))) & 0xFFFFu;
            const uint32_t ex = (bx >> 7) & 0xFFu, ew = (bw >> 7) & 0xFFu;
            const uint32_t mx = (bx & 0x7Fu) | (ex ? 0x80u : 0u);
            const uint32_t mw = (bw & 0x7Fu) | (ew ? 0x80u : 0u);
            const uint32_t P = mx * mw;
            if (P == 0) continue;
            const int pos = (int)(ex ? ex : 1u) + (int)(ew ? ew : 1u) - 268 + kUnit;   // (e-134) twice
            const uint64_t v = (uint64_t)P << (pos & 31);
            long long lo = (long long)(v & 0xFFFFFFFFull), hi = (long long)(v >> 32);
            if ((bx ^ bw) & 0x8000u) { lo = -lo; hi = -hi; }
            acc[pos >> 5] += lo;
            acc[(pos >> 5) + 1] += hi;
        }
    }
#pragma unroll
    for (int i = 0; i < kLimbs; ++i) acc[i] = warp_sum(acc[i]);
    // carry-normalise; a final carry of -1 means a negative total (two's complement digits)
    uint32_t dig[kLimbs];
    long long carry = 0;
#pragma unroll
    for (int i = 0; i < kLimbs; ++i) {
        long long v = acc[i] + carry;
        long long dgt = v & 0xFFFFFFFFll;
        dig[i] = (uint32_t)dgt;
        carry = (v - dgt) >> 32;   // exact: v - dgt is a multiple of 2^32
    }
    bool neg = carry < 0;
    if (neg) {
        unsigned long long c = 1;
#pragma unroll
        for (int i = 0; i < kLimbs; ++i) {
            unsigned long long v = (unsigned long long)(uint32_t)(~dig[i]) + c;
            dig[i] = (uint32_t)v;
            c = v >> 32;
        }
    }
    int msb = -1;
    for (int i = kLimbs - 1; i >= 0 && msb < 0; --i)
        if (dig[i]) msb = i * 32 + 31 - __clz(dig[i]);
    if (msb < 0) return 0.0f;
    int q = msb - 23;                       // 24 significant bits ...
    if (q < kUnit - 149) q = kUnit - 149;   // ... but no quantum below 2^-149
    uint32_t r = (msb >= q) ? (limb_window(dig, q) & ((msb - q + 1 >= 32) ? 0xFFFFFFFFu : ((1u << (msb - q + 1)) - 1u))) : 0u;
    bool half = (limb_window(dig, q - 1) & 1u) != 0;
    bool sticky = false;
    {
        int below = q - 1;                  // bits [0, below) are the sticky bits
        int full = below >> 5;
        for (int i = 0; i < full && !sticky; ++i) sticky = dig[i] != 0;
        int rem = below & 31;
        if (!sticky && rem) sticky = (dig[full] & ((1u << rem) - 1u)) != 0;
    }
    if (half && (sticky || (r & 1u))) r += 1;
    float mag = scalbnf((float)r, q - kUnit);   // exact, or +inf beyond the fp32 range
    return neg ? -mag : mag;
}

__device__ __forceinline__ float sigmoid_fast(float v) { return 1.0f / (1.0f + expf(-v)); }

__device__ __forceinline__ float sigmoid_exact32(float l32) {
    return __double2float_rn(1.0 / (1.0 + exp(-(double)l32)));
}

// Key record of expert e from a point logit and an fp32 interval [lo, hi] holding l32
// (table entry tb and bias b of the expert passed in).
__device__ __forceinline__ float4 make_key(int tb, float b, float lf, float lo, float hi) {
    const float NEG_INF = -__int_as_float(0x7f800000);
    if (tb < 0) return make_float4(NEG_INF, NEG_INF, NEG_INF, -1.0f);
    const float margin = 1.0f / 2097152.0f;   // 2^-21
    const float sv = sigmoid_fast(lf);
    return make_float4(sv + b, __fadd_rd(__fsub_rd(sigmoid_fast(lo), margin), b),
                       __fadd_ru(__fadd_ru(sigmoid_fast(hi), margin), b), sv);
}

// TwoSum (Knuth): s + err == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& err) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Key record of (token x, expert row w) by the decode kernel's compensated dot product with
// chunks of one product (lane l: vectors l, l+32, ..., eight TwoSum chains, then chains and
// lanes added as (sum, compensation) pairs), read from global memory by a whole warp; every
// lane returns the record.  coef is that kernel's bound for one-product chunks.
inline __device__ __noinline__ float4 refine_key_warp(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w, int d,
                                               int lane, float coef, int tb, float bias) {
    const uint4* xr = reinterpret_cast<const uint4*>(x);
    const uint4* wr = reinterpret_cast<const uint4*>(w);
    float s[8], c[8], A = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) s[q] = c[q] = 0.f;
    for (int cv = lane; cv < d / 8; cv += 32) {
        const uint4 wv = __ldg(wr + cv), xv = __ldg(xr + cv);
        const float w8[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                             bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
        const float x8[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                             bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float err;
            two_sum(s[q], __fmul_rn(x8[q], w8[q]), s[q], err);   // bf16 x bf16 products are exact in fp32
            c[q] = __fadd_rn(c[q], err);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) A = __fmaf_rn(fabsf(x8[i]), fabsf(w8[i]), A);
    }
    float S = s[0], C = c[0];
#pragma unroll
    for (int q = 1; q < 8; ++q) {
        float err;
        two_sum(S, s[q], S, err);
        C = __fadd_rn(C, __fadd_rn(c[q], err));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float S2 = __shfl_xor_sync(0xffffffffu, S, o), C2 = __shfl_xor_sync(0xffffffffu, C, o);
        float err;
        two_sum(S, S2, S, err);
        C = __fadd_rn(__fadd_rn(C, C2), err);
        A = __fadd_ru(A, __shfl_xor_sync(0xffffffffu, A, o));
    }
    // |S + C - exact| <= coef * sum|x w| * (1 + 2^-9) + d * 2^-147
    float delta = __fmul_ru(__fmul_ru(coef, A), 1.001953125f);
    delta = __fadd_ru(delta, (float)d * 5.605193857299268e-45f);
    return make_key(tb, bias, __fadd_rn(S, C), __fadd_rd(S, __fsub_rd(C, delta)), __fadd_ru(S, __fadd_ru(C, delta)));
}

// ------------------------------------------------------------------ certified selection

// Shared-memory bytes of one selecting warp: E key records, E exact keys and 96 words for
// the chosen experts (scores, ids, slots).
__host__ __device__ constexpr size_t select_smem_per_warp(int E) { return ((size_t)E * 20 + 384 + 15) / 16 * 16; }

// Order-preserving map of a float key to uint32 (every non-NaN key maps above 0, so 0 means
// "no candidate"), and its inverse.
__device__ __forceinline__ uint32_t key_order(float k) {
    const uint32_t u = __float_as_uint(k);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// One warp selects the experts of token t.  rec (E records), exk (E floats) and out (64
// words) are this warp's shared memory; lane l owns experts e = l + 32 m (m < ceil(E/32) <=
// 32), bit m of its masks.  A top-k round is two warp reductions (largest key, then lowest
// id among equal keys); only the winning lane rescans its experts.
inline __device__ __noinline__ void select_token(const RouteArgs& a, int t, int lane, float4* rec, float* exk, int* out,
                                                 SelOut o) {
    const float NEG_INF = -__int_as_float(0x7f800000);
    const int E = a.E, EPL = (E + 31) >> 5;
    const float4* krow = a.keys + (size_t)t * E;
    uint32_t valid = 0, picked = 0, best_u = 0;
    int best_m = -1;
    for (int m0 = 0; m0 < EPL; m0 += 4) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = lane + 32 * (m0 + u);
            v[u] = (m0 + u < EPL && e < E) ? __ldcg(krow + e) : make_float4(NEG_INF, NEG_INF, NEG_INF, -1.0f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int m = m0 + u, e = lane + 32 * m;
            if (m < EPL && e < E) {
                rec[e] = v[u];
                if (v[u].w >= 0.0f) {
                    valid |= 1u << m;
                    const uint32_t ku = key_order(v[u].x);
                    if (ku > best_u) { best_u = ku; best_m = m; }
                }
            }
        }
    }
    __syncwarp();
    // S = top-k by point estimate (key desc, id asc)
    int nsel = 0;
    for (int j = 0; j < a.k; ++j) {
        const uint32_t M = __reduce_max_sync(0xffffffffu, best_u);
        if (M == 0) break;
        const uint32_t win = __reduce_min_sync(0xffffffffu, best_u == M ? (uint32_t)(lane + 32 * best_m) : 0xFFFFFFFFu);
        if ((int)(win & 31) == lane) {
            picked |= 1u << (win >> 5);
            best_u = 0;
            best_m = -1;
            for (uint32_t r = valid & ~picked; r; r &= r - 1) {
                const int m = __ffs(r) - 1;
                const uint32_t ku = key_order(rec[lane + 32 * m].x);
                if (ku > best_u) { best_u = ku; best_m = m; }
            }
        }
        ++nsel;
    }
    if (nsel < a.k && lane == 0 && o.status) atomicOr(o.status, MOE_STATUS_FEW_RESIDENT);
    // interval thresholds
    float min_lo_in = __int_as_float(0x7f800000), max_hi_out = NEG_INF;
    for (uint32_t r = valid; r; r &= r - 1) {
        const int m = __ffs(r) - 1, e = lane + 32 * m;
        if ((picked >> m) & 1u) min_lo_in = fminf(min_lo_in, rec[e].y);
        else max_hi_out = fmaxf(max_hi_out, rec[e].z);
    }
    min_lo_in = key_value(__reduce_min_sync(0xffffffffu, key_order(min_lo_in)));
    max_hi_out = key_value(__reduce_max_sync(0xffffffffu, key_order(max_hi_out)));
    uint32_t certain = 0, uncertain = 0;
    for (uint32_t r = valid; r; r &= r - 1) {
        const int m = __ffs(r) - 1, e = lane + 32 * m;
        const bool pk = (picked >> m) & 1u;
        if (pk && rec[e].y > max_hi_out) certain |= 1u << m;
        else if (pk || rec[e].z >= min_lo_in) uncertain |= 1u << m;
    }
    uint32_t final_mask = certain;
    const uint16_t* xt = a.x + (size_t)t * a.d;
    // exact scores (and keys) of the experts in `mask`, one expert at a time by the whole warp
    auto exact_scores = [&](uint32_t mask) {
        for (int m = 0; m < EPL; ++m) {
            uint32_t bal = __ballot_sync(0xffffffffu, (mask >> m) & 1u);
            while (bal) {
                const int src = __ffs(bal) - 1;
                bal &= bal - 1;
                const int e = src + 32 * m;
                const float s32 = sigmoid_exact32(exact_dot_bf16_warp(xt, a.wr + (size_t)e * a.d, a.d, lane));
                if (lane == src) {
                    exk[e] = __fadd_rn(s32, a.bias ? a.bias[e] : 0.0f);
                    rec[e].w = s32;
                }
            }
        }
        __syncwarp();
    };
    if (__any_sync(0xffffffffu, uncertain != 0)) {
        const int need = nsel - __reduce_add_sync(0xffffffffu, (uint32_t)__popc(certain));
        exact_scores(uncertain);
        uint32_t chosen = 0;
        for (int j = 0; j < need; ++j) {
            float bk = NEG_INF;
            int be = -1;
            for (uint32_t r = uncertain & ~chosen; r; r &= r - 1) {
                const int e = lane + 32 * (__ffs(r) - 1);
                if (be < 0 || exk[e] > bk) { bk = exk[e]; be = e; }
            }
            // key desc, id asc over the warp (candidates without a key carry id 0x7FFFFFFF)
            const uint32_t M = __reduce_max_sync(0xffffffffu, be < 0 ? 0u : key_order(bk));
            if (M == 0) break;
            const uint32_t win =
                __reduce_min_sync(0xffffffffu, (be >= 0 && key_order(bk) == M) ? (uint32_t)be : 0xFFFFFFFFu);
            if ((int)(win & 31) == lane) chosen |= 1u << (win >> 5);
        }
        final_mask |= chosen;
    }
    // weights: a chosen expert whose key interval is wider than 1e-5 of its score gets its
    // record recomputed with the compensated dot product (the refinement of select_row), and
    // if that interval is still wide, its score from the exact logit, so every score has
    // relative error below 1e-5
    uint32_t wide = 0;
    for (uint32_t r = final_mask & ~uncertain; r; r &= r - 1) {
        const int m = __ffs(r) - 1, e = lane + 32 * m;
        if (rec[e].z - rec[e].y > 1e-5f * rec[e].w) wide |= 1u << m;
    }
    if (a.refine_coef > 0.0f && __any_sync(0xffffffffu, wide != 0)) {
        for (int m = 0; m < EPL; ++m) {
            uint32_t bal = __ballot_sync(0xffffffffu, (wide >> m) & 1u);
            while (bal) {
                const int src = __ffs(bal) - 1;
                bal &= bal - 1;
                const int e = src + 32 * m;
                const float be = a.bias ? a.bias[e] : 0.0f;
                const float4 nr = refine_key_warp(xt, a.wr + (size_t)e * a.d, a.d, lane, a.refine_coef, a.table[e], be);
                if (lane == src && !(nr.z - nr.y > 1e-5f * nr.w)) {
                    rec[e] = nr;
                    wide &= ~(1u << m);
                }
            }
        }
        __syncwarp();
    }
    if (__any_sync(0xffffffffu, wide != 0)) exact_scores(wide);
    // chosen experts in ascending id (m outer, lane inner) into out[0..n); weight sum in that order
    int n = 0;
    const uint32_t below = (1u << lane) - 1u;
    for (int m = 0; m < EPL; ++m) {
        const uint32_t bal = __ballot_sync(0xffffffffu, (final_mask >> m) & 1u);
        if ((final_mask >> m) & 1u) out[n + __popc(bal & below)] = lane + 32 * m;
        n += __popc(bal);
    }
    __syncwarp();
    float sum = 0.0f;
    if (lane == 0)
        for (int i = 0; i < n; ++i) sum += rec[out[i]].w;
    sum = __shfl_sync(0xffffffffu, sum, 0);
    int32_t* ids = o.ids;
    float* wo = o.w;
    int32_t* so = o.slots;
    for (int j = lane; j < a.k; j += 32) {
        if (j < n) {
            const int e = out[j];
            ids[j] = e;
            wo[j] = (sum > 0.0f) ? __fdiv_rn(rec[e].w, sum) : 0.0f;
            so[j] = a.table[e];
        } else {
            ids[j] = -1;
            wo[j] = 0.0f;
            so[j] = -1;
        }
    }
    __syncwarp();
}

// The selection of token t by one warp (lane l holds the key records of experts l + 32 m,
// m < EPL, in registers): a top-k round is a warp reduction (largest key) and a ballot of
// the lanes holding it (a second reduction, lowest id, only when several do); the winning
// lane promotes its second candidate and rescans its registers.  The chosen set is final when
// every chosen expert's key interval lies above every other expert's and every chosen score
// is narrow; otherwise the token goes whole to select_token (same warp).  E <= 32 * EPL.
// rec, exk and out are this warp's select_token arrays in shared memory.
// Largest key order among this lane's experts m with bit m of `mask` set (0 when none), ties
// to the lower m (the lower expert id): a pairwise tree, a few dependent steps instead of EPL.
template <int EPL>
__device__ __forceinline__ void lane_best(const uint32_t (&ko)[EPL], uint32_t mask, uint32_t& bu, int& bm) {
    uint32_t v[EPL];
    int ix[EPL];
#pragma unroll
    for (int m = 0; m < EPL; ++m) {
        v[m] = ((mask >> m) & 1u) ? ko[m] : 0u;
        ix[m] = m;
    }
#pragma unroll
    for (int w = 1; w < EPL; w *= 2)
#pragma unroll
        for (int m = 0; m + w < EPL; m += 2 * w)
            if (v[m + w] > v[m]) {   // strict: on equal keys the lower index stays
                v[m] = v[m + w];
                ix[m] = ix[m + w];
            }
    bu = v[0];
    bm = ix[0];
}

template <int EPL>
__device__ __forceinline__ void select_row(const RouteArgs& a, int t, int lane, float4* rec, float* exk, int* out,
                                           SelOut o) {
    const float NEG_INF = -__int_as_float(0x7f800000);
    const int E = a.E, k = a.k;
    const float4* krow = a.keys + (size_t)t * E;
    // key records and slot-table entries of experts lane + 32 m, loaded together
    float4 r[EPL];
    int tb[EPL];
#pragma unroll
    for (int m = 0; m < EPL; ++m) {
        const int e = lane + 32 * m;
        r[m] = (e < E) ? __ldcg(krow + e) : make_float4(NEG_INF, NEG_INF, NEG_INF, -1.0f);
        tb[m] = (e < E) ? __ldg(a.table + e) : -1;
    }
    uint32_t valid = 0, picked = 0, bu = 0;
    uint32_t ko[EPL];
    int bm = 0;
#pragma unroll
    for (int m = 0; m < EPL; ++m) {
        if (r[m].w >= 0.0f) valid |= 1u << m;
        ko[m] = key_order(r[m].x);
    }
    lane_best<EPL>(ko, valid, bu, bm);
    // Each lane also keeps its second candidate: a winning lane promotes it at once and
    // rescans for the next one just after the following round's reduction is issued, so that
    // the rescan overlaps the reduction instead of preceding it.
    uint32_t bu2;
    int bm2;
    lane_best<EPL>(ko, valid & ~(1u << bm), bu2, bm2);
    bool refill = false;
    int n = 0;
    for (int j = 0; j < k; ++j) {
        const uint32_t M = __reduce_max_sync(0xffffffffu, bu);
        if (refill) {
            lane_best<EPL>(ko, valid & ~picked & ~(1u << bm), bu2, bm2);
            refill = false;
        }
        if (M == 0) break;
        // the winner: the one lane holding M, else the lowest expert id among those that do
        const uint32_t hold = __ballot_sync(0xffffffffu, bu == M);
        int wl = __ffs(hold) - 1;
        if (hold & (hold - 1u))
            wl = (int)(__reduce_min_sync(0xffffffffu, bu == M ? (uint32_t)(lane + 32 * bm) : 0xFFFFFFFFu) & 31u);
        if (lane == wl) {
            picked |= 1u << bm;
            bu = bu2;
            bm = bm2;
            refill = true;
        }
        ++n;
    }
    if (n < k && lane == 0 && o.status) atomicOr(o.status, MOE_STATUS_FEW_RESIDENT);
    // certification thresholds: min klo over the chosen, max khi over the rest (pairwise trees)
    float lov[EPL], hiv[EPL];
#pragma unroll
    for (int m = 0; m < EPL; ++m) {
        const bool pk = (picked >> m) & 1u;
        lov[m] = pk ? r[m].y : __int_as_float(0x7f800000);
        hiv[m] = (!pk && ((valid >> m) & 1u)) ? r[m].z : NEG_INF;
    }
#pragma unroll
    for (int w = 1; w < EPL; w *= 2)
#pragma unroll
        for (int m = 0; m + w < EPL; m += 2 * w) {
            lov[m] = fminf(lov[m], lov[m + w]);
            hiv[m] = fmaxf(hiv[m], hiv[m + w]);
        }
    const float lo_in = lov[0], hi_out = hiv[0];
    const float min_lo_in = key_value(__reduce_min_sync(0xffffffffu, key_order(lo_in)));
    const float max_hi_out = key_value(__reduce_max_sync(0xffffffffu, key_order(hi_out)));
    bool doubt = false, order_doubt = false;
#pragma unroll
    for (int m = 0; m < EPL; ++m) {
        if ((picked >> m) & 1u) {
            if (!(r[m].y > max_hi_out)) order_doubt = true;
            else if (r[m].z - r[m].y > 1e-5f * r[m].w) doubt = true;
        } else if (((valid >> m) & 1u) && r[m].z >= min_lo_in) {
            order_doubt = true;
        }
    }
    if (__any_sync(0xffffffffu, doubt || order_doubt)) {
        // Refinement: when the chosen set is certain and only some chosen scores are wide
        // (the tiled logits' bound), the chosen experts' records are recomputed with the
        // compensated dot product; if every chosen interval is then narrow and still above
        // every other expert's, the token is done without exact logits.
        bool resolved = false;
        if (!__any_sync(0xffffffffu, order_doubt) && a.refine_coef > 0.0f) {
            const uint16_t* xt = a.x + (size_t)t * a.d;
            bool still = false;
#pragma unroll
            for (int m = 0; m < EPL; ++m) {
                uint32_t bal = __ballot_sync(0xffffffffu, (picked >> m) & 1u);
                while (bal) {
                    const int src = __ffs(bal) - 1;
                    bal &= bal - 1;
                    const int e = src + 32 * m;
                    const float be = a.bias ? a.bias[e] : 0.0f;
                    const int tbe = __shfl_sync(0xffffffffu, tb[m], src);
                    const float4 nr = refine_key_warp(xt, a.wr + (size_t)e * a.d, a.d, lane, a.refine_coef, tbe, be);
                    if (lane == src) {
                        r[m] = nr;
                        if (!(nr.y > max_hi_out) || nr.z - nr.y > 1e-5f * nr.w) still = true;
                    }
                }
            }
            resolved = !__any_sync(0xffffffffu, still);
        }
        if (!resolved) {
            select_token(a, t, lane, rec, exk, out, o);
            return;
        }
    }
    // outputs in ascending id (m outer, lane inner); weight sum in that order
    float* osc = reinterpret_cast<float*>(out);
    int* oid = out + 32;
    int* osl = out + 64;
    const uint32_t below = (1u << lane) - 1u;
    int base = 0;
#pragma unroll
    for (int m = 0; m < EPL; ++m) {
        const uint32_t bal = __ballot_sync(0xffffffffu, (picked >> m) & 1u);
        if ((picked >> m) & 1u) {
            const int rank = base + __popc(bal & below);
            osc[rank] = r[m].w;
            oid[rank] = lane + 32 * m;
            osl[rank] = tb[m];
        }
        base += __popc(bal);
    }
    __syncwarp();
    float sum = 0.0f;
    if (lane == 0)
        for (int i0 = 0; i0 < n; i0 += 8) {   // the loads of 8 scores together, then their sum in order
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = (i0 + i < n) ? osc[i0 + i] : 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i0 + i < n) sum += v[i];
        }
    sum = __shfl_sync(0xffffffffu, sum, 0);
    int32_t* ids = o.ids;
    float* wo = o.w;
    int32_t* so = o.slots;
    for (int j = lane; j < k; j += 32) {
        if (j < n) {
            ids[j] = oid[j];
            wo[j] = (sum > 0.0f) ? __fdiv_rn(osc[j], sum) : 0.0f;
            so[j] = osl[j];
        } else {
            ids[j] = -1;
            wo[j] = 0.0f;
            so[j] = -1;
        }
    }
    __syncwarp();
}

#define FP4MOE_EPL_DISPATCH(E, ...)                                   \
    do {                                                              \
        const int epl_ = ((E) + 31) / 32;                             \
        if (epl_ <= 2) { constexpr int EPL = 2; __VA_ARGS__; }        \
        else if (epl_ <= 4) { constexpr int EPL = 4; __VA_ARGS__; }   \
        else if (epl_ <= 8) { constexpr int EPL = 8; __VA_ARGS__; }   \
        else if (epl_ <= 12) { constexpr int EPL = 12; __VA_ARGS__; } \
        else if (epl_ <= 16) { constexpr int EPL = 16; __VA_ARGS__; } \
        else if (epl_ <= 24) { constexpr int EPL = 24; __VA_ARGS__; } \
        else { constexpr int EPL = 32; __VA_ARGS__; }                 \
    } while (0)

}  // namespace fp4moe
