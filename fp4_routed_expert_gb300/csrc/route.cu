// route.cu -- router logits, certified top-k selection and slot lookup (sm_103a).
//
// What is computed (per token t, expert e):
//   logit l32 = the exact dot product x[t] . W_r[e] rounded once to fp32
//   score s32 = fp32(1 / (1 + exp(-(double)l32)))
//   key       = fp32(s32 + bias[e])            (-inf when expert_to_slot[e] < 0)
//   top-k keys, ties to the lower expert id; weights w_j = s_j / sum s (fp32, ascending id)
// The pages ("Start the expert reads before the GPU is done", 28 September follow-up) name
// the router and its top-k but no formula; the exact-then-round logit makes the chosen set
// independent of summation order.
//
// How the device reaches the exact set without computing every exact logit:
//  1. a fast logit D with an error bound delta, |D - exact| <= delta:
//     decode (T <= 16): each lane sums its bf16 products (exact in fp32) in chunks of c = 1
//       product (the kernel takes any c; one keeps a token's arithmetic independent of T),
//       the chunks with TwoSum compensation (Ogita, Rump, Oishi, "Accurate sum and
//       dot product", SIAM J. Sci. Comput. 26(6), 2005, Sum2) along 8/c independent chains of
//       m = d/256 chunks; chains and lanes are then added as (sum, compensation) pairs with
//       TwoSum in fp32:
//       delta = (gamma_(c-1) + gamma_m^2 + 2^-34) * sum|x_k w_k| * (1 + 2^-9) + d 2^-147,
//       the 2^-34 term covering the pair additions (a few 1e-9 at d = 5120);
//     prefill: fp32 FMA chains with at most L roundings on any path,
//       delta = gamma_L * ||x|| ||w|| (Cauchy-Schwarz), inflated by 2^-10 for the norms;
//  2. [D - delta, D + delta] rounded outward to fp32 holds l32; through the monotone
//     sigmoid (fp32 with a 2^-21 absolute margin that covers its error, at most 3 ulp, and
//     the final fp32 rounding) and the bias add (directed rounding) it gives a key interval [klo, khi];
//  3. S = top-k by the point estimate; an expert of S whose klo exceeds every outside khi is
//     certainly chosen, an outside expert whose khi is below every klo of S certainly not;
//  4. the rest are recomputed exactly (integer Kulisch accumulation of the bf16 products,
//     one rounding to fp32, double sigmoid) and ranked by exact key;
//  5. a chosen expert whose key interval is wider than 1e-5 of its score also gets its
//     exact score, so every weight is within 2e-5 (relative) of the exact one.
// Each (token, expert) gets one 16-byte key record {point key, klo, khi, score}; score < 0
// marks an expert that is not resident.
#include <algorithm>

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
};

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
__device__ __noinline__ float exact_dot_bf16_warp(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w,
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
__device__ __noinline__ float4 refine_key_warp(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w, int d,
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

// (key desc, id asc): is a better than b?
__device__ __forceinline__ bool better(float ka, int ea, float kb, int eb) {
    if (eb < 0) return ea >= 0;
    if (ea < 0) return false;
    return ka > kb || (ka == kb && ea < eb);
}

__device__ __forceinline__ void warp_best(float& k, int& e) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float ko = __shfl_xor_sync(0xffffffffu, k, o);
        int eo = __shfl_xor_sync(0xffffffffu, e, o);
        if (better(ko, eo, k, e)) { k = ko; e = eo; }
    }
}

// Shared-memory bytes of one selecting warp: E key records, E exact keys and 96 words for
// the chosen experts (scores, ids, slots).
__host__ __device__ inline size_t select_smem_per_warp(int E) { return ((size_t)E * 20 + 384 + 15) / 16 * 16; }

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
__device__ __noinline__ void select_token(const RouteArgs& a, int t, int lane, float4* rec, float* exk, int* out) {
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
    if (nsel < a.k && lane == 0) atomicOr(a.status, MOE_STATUS_FEW_RESIDENT);
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
    // score from the exact logit, so every score has relative error below 1e-5
    uint32_t wide = 0;
    for (uint32_t r = final_mask & ~uncertain; r; r &= r - 1) {
        const int m = __ffs(r) - 1, e = lane + 32 * m;
        if (rec[e].z - rec[e].y > 1e-5f * rec[e].w) wide |= 1u << m;
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
    int32_t* ids = a.ids + (size_t)t * a.k;
    float* wo = a.w + (size_t)t * a.k;
    int32_t* so = a.slots + (size_t)t * a.k;
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

constexpr int kSelWarps = 4;

// The selection of token t by one warp (lane l holds the key records of experts l + 32 m,
// m < EPL, in registers): a top-k round is two warp reductions (largest key, then lowest id
// among equal keys) and a register rescan by the winning lane.  The chosen set is final when
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
__device__ __forceinline__ void select_row(const RouteArgs& a, int t, int lane, float4* rec, float* exk, int* out) {
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
    int n = 0;
    for (int j = 0; j < k; ++j) {
        const uint32_t M = __reduce_max_sync(0xffffffffu, bu);
        if (M == 0) break;
        const uint32_t win = __reduce_min_sync(0xffffffffu, bu == M ? (uint32_t)(lane + 32 * bm) : 0xFFFFFFFFu);
        if ((int)(win & 31) == lane) {
            picked |= 1u << (win >> 5);
            lane_best<EPL>(ko, valid & ~picked, bu, bm);
        }
        ++n;
    }
    if (n < k && lane == 0) atomicOr(a.status, MOE_STATUS_FEW_RESIDENT);
    // certification thresholds: min klo over the chosen, max khi over the rest
    float lo_in = __int_as_float(0x7f800000), hi_out = NEG_INF;
#pragma unroll
    for (int m = 0; m < EPL; ++m) {
        if ((picked >> m) & 1u) lo_in = fminf(lo_in, r[m].y);
        else if ((valid >> m) & 1u) hi_out = fmaxf(hi_out, r[m].z);
    }
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
            select_token(a, t, lane, rec, exk, out);
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
        for (int i = 0; i < n; ++i) sum += osc[i];
    sum = __shfl_sync(0xffffffffu, sum, 0);
    int32_t* ids = a.ids + (size_t)t * k;
    float* wo = a.w + (size_t)t * k;
    int32_t* so = a.slots + (size_t)t * k;
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

// One warp per token, launched behind the key-record kernel of the tiled (large T) router.
template <int EPL>
__global__ void __launch_bounds__(kSelWarps * 32) route_select_kernel(RouteArgs a) {
    extern __shared__ unsigned char sel_smem[];   // per warp: select_token's arrays
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned char* wsm = sel_smem + (size_t)warp * select_smem_per_warp(a.E);
    float4* rec = reinterpret_cast<float4*>(wsm);
    float* exk = reinterpret_cast<float*>(wsm + (size_t)a.E * 16);
    int* out = reinterpret_cast<int*>(wsm + (size_t)a.E * 20);   // 96 words: ranks' scores, ids, slots
    pdl_trigger();
    pdl_wait();   // the key records of the logit kernel
    for (int t = blockIdx.x * kSelWarps + warp; t < a.T; t += gridDim.x * kSelWarps)
        select_row<EPL>(a, t, lane, rec, exk, out);
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

// ------------------------------------------------------------------ decode: one warp per expert

constexpr int kDecodeWarps = 4;                 // experts per block and round at most
constexpr int kDecodeKS = 4;                    // warps per (expert, token group): K in four parts
constexpr int kDecodeThreads = 512;             // threads per block at most
constexpr size_t kDecodeSmemMax = 226 * 1024;

__host__ __device__ inline size_t decode_smem_bytes(int T, int d, int epb) {
    return (size_t)(epb + T) * d * 2 + 16;   // W rows, x rows, one mbarrier
}

// Number of token groups of a decode router launch: kDecodeKS warps per (expert, group).
inline int decode_groups(int T, int epb) {
    const int g = kDecodeThreads / (32 * epb * kDecodeKS);
    return T < g ? T : (g > 1 ? g : 1);
}

// Key records for T <= 16 tokens.  A block takes EPB = a.dec_epb experts per round (the
// fewest that spread the experts over the SMs): their router rows (kept in L2 between calls)
// and (once) the tokens' rows arrive in shared memory by bulk copies, then warp w works on
// expert e0 + w % EPB, quarter (w / EPB) % kDecodeKS of the K range, for the tokens of group
// w / (EPB kDecodeKS), one token at a time; a token's arithmetic does not depend on its group
// nor on EPB.  Lane l owns vectors l, l+32, ... of its quarter; per token it keeps 8/CH
// compensated sums (s, c) -- one per plain FMA chunk of CH products of a vector, so the chains
// are independent -- and sum|x w|; the quarters' (sum, compensation) pairs are then added in
// quarter order like the lanes'.  The loops are kept short: this code runs once
// per call and is seldom in the instruction cache.  The last block to finish (a ticket on
// a.counter, left at zero again) then selects every token's experts, one warp per token, in
// its own shared memory.
template <int CH, int EPL>
__global__ void __launch_bounds__(kDecodeThreads) route_decode_kernel(RouteArgs a) {
    constexpr int NCH = 8 / CH;
    extern __shared__ __align__(16) unsigned char dsm[];
    __shared__ float4 part[kDecodeWarps * kDecodeMaxT * kDecodeKS];   // (S, C, A) per expert, token, quarter
    const int EPB = a.dec_epb;
    const int tid = threadIdx.x, lane = tid & 31, wq = tid >> 5;
    const int warp = wq % EPB, ks = (wq / EPB) % kDecodeKS, grp = wq / (EPB * kDecodeKS);
    const int ngrp = blockDim.x / (32 * EPB * kDecodeKS);
    const int tpg = (a.T + ngrp - 1) / ngrp, t_lo = grp * tpg, t_hi = min(a.T, t_lo + tpg);
    const int T = a.T, d = a.d, E = a.E, nvec = d / 8;
    uint16_t* ws = reinterpret_cast<uint16_t*>(dsm);
    const uint16_t* xs = ws + (size_t)EPB * d;
    uint64_t* bar = reinterpret_cast<uint64_t*>(dsm + (size_t)(EPB + T) * d * 2);
    __shared__ int abort_flag;
    if (tid == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    uint32_t phase = 0;
    for (int e0 = blockIdx.x * EPB; e0 < E; e0 += gridDim.x * EPB) {
        const int nw = min(EPB, E - e0);
        const bool first = (e0 == (int)blockIdx.x * EPB);
        const uint32_t rowb = (uint32_t)d * 2;
        if (tid == 0) {
            mbar_expect_tx(smem_u32(bar), rowb * nw + (first ? rowb * T : 0u));
            // Launched behind the previous kernel (programmatic dependent launch), the logit
            // phase reads only the router rows (one copy: a bulk copy costs a fixed time on top
            // of its bytes) and x, which the kernel ahead does not write (the header's
            // contract); so it overlaps the end of that kernel.  The bias, the table, the
            // ticket and every output are touched only after the wait below.
            if (first) bulk_g2s(smem_u32(xs), a.x, rowb * T, smem_u32(bar));
            bulk_g2s_hint(smem_u32(ws), a.wr + (size_t)e0 * d, rowb * nw, smem_u32(bar), l2_evict_last());
        }
        const int e = e0 + warp;
        // bounded wait; the copies are waited for (again bounded) even after a timeout
        if (!mbar_wait(smem_u32(bar), phase, &abort_flag)) {
            if (tid == 0) atomicOr(a.status, MOE_STATUS_TIMEOUT);
            for (unsigned i = 0; i < kSpinLimit && !mbar_try(smem_u32(bar), phase); ++i) {
            }
        }
        phase ^= 1u;
        if (e < E) {
            const uint4* wrow = reinterpret_cast<const uint4*>(ws + (size_t)warp * d);
            const int qv = nvec / kDecodeKS, cv_lo = ks * qv, cv_hi = cv_lo + qv;
            for (int t = t_lo; t < t_hi; ++t) {
                const uint4* xrow = reinterpret_cast<const uint4*>(xs + (size_t)t * d);
                float s[NCH], c[NCH], A = 0.f;
#pragma unroll
                for (int q = 0; q < NCH; ++q) s[q] = c[q] = 0.f;
#pragma unroll 2
                for (int cv = cv_lo + lane; cv < cv_hi; cv += 32) {
                    const uint4 wv = wrow[cv], xv = xrow[cv];
                    const float w8[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                                         bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
                    const float x8[8] = {bf16_lo(xv.x), bf16_hi(xv.x), bf16_lo(xv.y), bf16_hi(xv.y),
                                         bf16_lo(xv.z), bf16_hi(xv.z), bf16_lo(xv.w), bf16_hi(xv.w)};
#pragma unroll
                    for (int q = 0; q < NCH; ++q) {
                        const int i0 = q * CH;
                        float qs = __fmul_rn(x8[i0], w8[i0]);
#pragma unroll
                        for (int i = i0 + 1; i < i0 + CH; ++i) qs = __fmaf_rn(x8[i], w8[i], qs);
                        float err;
                        two_sum(s[q], qs, s[q], err);
                        c[q] = __fadd_rn(c[q], err);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) A = __fmaf_rn(fabsf(x8[i]), fabsf(w8[i]), A);
                }
                // (S, C) = sum over chains and lanes of (s + c) as TwoSum pairs, A = sum|x w|
                // rounded up across lanes; every lane ends with the same values
                float S = s[0], Cc = c[0];
#pragma unroll
                for (int q = 1; q < NCH; ++q) {
                    float err;
                    two_sum(S, s[q], S, err);
                    Cc = __fadd_rn(Cc, __fadd_rn(c[q], err));
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float S2 = __shfl_xor_sync(0xffffffffu, S, o), C2 = __shfl_xor_sync(0xffffffffu, Cc, o);
                    float err;
                    two_sum(S, S2, S, err);
                    Cc = __fadd_rn(__fadd_rn(Cc, C2), err);
                    A = __fadd_ru(A, __shfl_xor_sync(0xffffffffu, A, o));
                }
                if (lane == 0) part[(warp * T + t) * kDecodeKS + ks] = make_float4(S, Cc, A, 0.f);
            }
        }
        __syncthreads();   // every quarter's pair is in part
        if (first) {
            // the kernel ahead has completed from here on; the next kernel (the expert kernel,
            // which waits for this one before reading anything but x) may launch
            pdl_wait();
            pdl_trigger();
        }
        const int tb = (e < E) ? a.table[e] : -1;
        const float bias_e = (e < E && a.bias) ? a.bias[e] : 0.0f;
        if (e < E && ks == 0 && lane < t_hi - t_lo) {
            {
                const float4* pp = part + (warp * T + t_lo + lane) * kDecodeKS;
                float myS = pp[0].x, myC = pp[0].y, myA = pp[0].z;
#pragma unroll
                for (int k2 = 1; k2 < kDecodeKS; ++k2) {
                    float err;
                    two_sum(myS, pp[k2].x, myS, err);
                    myC = __fadd_rn(__fadd_rn(myC, pp[k2].y), err);
                    myA = __fadd_ru(myA, pp[k2].z);
                }
                // |S + C - exact| <= coef * sum|x w| * (1 + 2^-9) + d * 2^-147
                float delta = __fmul_ru(__fmul_ru(a.bound_coef, myA), 1.001953125f);
                delta = __fadd_ru(delta, (float)d * 5.605193857299268e-45f);
                const float lo = __fadd_rd(myS, __fsub_rd(myC, delta));
                const float hi = __fadd_ru(myS, __fadd_ru(myC, delta));
                a.keys[(size_t)(t_lo + lane) * E + e] = make_key(tb, bias_e, __fadd_rn(myS, myC), lo, hi);
            }
        }
        __syncthreads();   // the next iteration's copies overwrite the router rows
    }
    __shared__ int last_block;
    __syncthreads();   // every key record of this block is written
    // the ticket releases this block's records and acquires every earlier block's
    if (tid == 0)
        last_block = (atom_add_acq_rel(reinterpret_cast<int32_t*>(a.counter), 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (!last_block) return;
    const int nsel = blockDim.x >> 5, wsel = tid >> 5;
    unsigned char* wsm = dsm + (size_t)wsel * select_smem_per_warp(E);
    float4* rec = reinterpret_cast<float4*>(wsm);
    float* exk = reinterpret_cast<float*>(wsm + (size_t)E * 16);
    int* out = reinterpret_cast<int*>(wsm + (size_t)E * 20);
    for (int t = wsel; t < T; t += nsel) select_row<EPL>(a, t, lane, rec, exk, out);
    if (tid == 0) *a.counter = 0u;
}

// ------------------------------------------------------------------ large T: tiled logits

// ||x_t|| and ||W_r[e]|| (one warp per row).
__global__ void route_norms_kernel(RouteArgs a) {
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int rows = a.T + a.E;
    for (int r = gw; r < rows; r += (gridDim.x * blockDim.x) >> 5) {
        const uint16_t* p = (r < a.T) ? a.x + (size_t)r * a.d : a.wr + (size_t)(r - a.T) * a.d;
        float s = 0.f;
        for (int i = lane; i < a.d; i += 32) {
            const float v = bf16_to_f32(p[i]);
            s = fmaf(v, v, s);
        }
        s = warp_sum(s);
        if (lane == 0) {
            if (r < a.T) a.xnorm[r] = sqrtf(s);
            else a.wnorm[r - a.T] = sqrtf(s);
        }
    }
}

// 64 tokens x 64 experts per block of 128 threads (four resident per SM, so that a grid of a
// few hundred tiles spreads evenly over the SMs), 8 tokens x 4 experts per thread, K staged 32
// at a time (the next step's operands are loaded into registers while the current one is
// multiplied).
// Each output is accumulated in chunks of 256 products (fresh partial sums, products in
// ascending K) added into a running total, so every rounding path has at most 256 + ceil(d/256)
// roundings.  The epilogue turns each logit into its key record with the Cauchy-Schwarz bound
// (norms computed beforehand).
constexpr int kTileT = 64, kTileE = 64, kRouteTileK = 32, kChunkK = 256, kTiledThreads = 128;

__global__ void __launch_bounds__(kTiledThreads, 4) route_tiled_kernel(RouteArgs a) {
    __shared__ __align__(16) float xs[kRouteTileK][kTileT + 4];
    __shared__ __align__(16) float ws[kRouteTileK][kTileE + 4];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.y * kTileT, e0 = blockIdx.x * kTileE;
    // loads: a warp takes 32 consecutive rows at one K offset, so its transposed stores hit
    // distinct banks.  x and W alike: row 32 (w % 2) + lane, K offset 16 (w / 2), 16 values.
    const int xr = 32 * (warp & 1) + lane, xc = 16 * (warp >> 1);
    const bool xok = t0 + xr < a.T, wok = e0 + xr < a.E;
    const uint16_t* xp = a.x + (size_t)(t0 + xr) * a.d + xc;
    const uint16_t* wp = a.wr + (size_t)(e0 + xr) * a.d + xc;
    uint4 xv0, xv1, wv0, wv1;
    auto load = [&](int k0) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        xv0 = xok ? __ldg(reinterpret_cast<const uint4*>(xp + k0)) : z;
        xv1 = xok ? __ldg(reinterpret_cast<const uint4*>(xp + k0 + 8)) : z;
        wv0 = wok ? __ldg(reinterpret_cast<const uint4*>(wp + k0)) : z;
        wv1 = wok ? __ldg(reinterpret_cast<const uint4*>(wp + k0 + 8)) : z;
    };
    auto store = [&]() {
        const uint32_t xw[8] = {xv0.x, xv0.y, xv0.z, xv0.w, xv1.x, xv1.y, xv1.z, xv1.w};
        const uint32_t ww[8] = {wv0.x, wv0.y, wv0.z, wv0.w, wv1.x, wv1.y, wv1.z, wv1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            xs[xc + 2 * i][xr] = bf16_lo(xw[i]);
            xs[xc + 2 * i + 1][xr] = bf16_hi(xw[i]);
            ws[xc + 2 * i][xr] = bf16_lo(ww[i]);
            ws[xc + 2 * i + 1][xr] = bf16_hi(ww[i]);
        }
    };
    float tot[8][4], part[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) tot[i][j] = part[i][j] = 0.f;
    load(0);
    store();
    __syncthreads();
    for (int k0 = 0; k0 < a.d; k0 += kRouteTileK) {
        const bool more = k0 + kRouteTileK < a.d;
        if (more) load(k0 + kRouteTileK);
#pragma unroll 8
        for (int kk = 0; kk < kRouteTileK; ++kk) {
            const float4 xa = *reinterpret_cast<const float4*>(&xs[kk][ty * 8]);
            const float4 xb = *reinterpret_cast<const float4*>(&xs[kk][ty * 8 + 4]);
            const float4 wb = *reinterpret_cast<const float4*>(&ws[kk][tx * 4]);
            const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w}, wvv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) part[i][j] = fmaf(xv[i], wvv[j], part[i][j]);
        }
        if (((k0 + kRouteTileK) % kChunkK) == 0 || !more) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) { tot[i][j] += part[i][j]; part[i][j] = 0.f; }
        }
        __syncthreads();   // every thread is done with this step's tiles
        if (more) {
            store();
            __syncthreads();
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int t = t0 + ty * 8 + i;
        if (t >= a.T) continue;
        const float xn = __ldg(a.xnorm + t);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e >= a.E) continue;
            const float l = tot[i][j];
            float delta = fmaf(a.bound_coef * xn, __ldg(a.wnorm + e), 7.5e-37f);
            delta = __fmul_ru(delta, 1.0f + 1.0f / 1048576.0f);
            a.keys[(size_t)t * a.E + e] =
                make_key(a.table[e], a.bias ? a.bias[e] : 0.0f, l, __fsub_rd(l, delta), __fadd_ru(l, delta));
        }
    }
}

// ------------------------------------------------------------------ host side

// gamma_n = n u / (1 - n u), u = 2^-24
static double gamma32(int n) {
    const double u = 1.0 / 16777216.0;
    return n * u / (1.0 - n * u);
}

static float gamma_coef(int L) { return (float)(gamma32(L) * (1.0 + 1.0 / 1024.0)); }

// Selection: one warp per token, launched behind the key-record kernel.
template <int EPL>
static int launch_select_epl(const RouteArgs& a, cudaStream_t st) {
    const size_t sel = kSelWarps * select_smem_per_warp(a.E);
    if (sel > 48 * 1024 &&
        cudaFuncSetAttribute(route_select_kernel<EPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sel) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    int grid = (a.T + kSelWarps - 1) / kSelWarps;
    if (grid > 4096) grid = 4096;
    if (launch_pdl(route_select_kernel<EPL>, dim3(grid), dim3(kSelWarps * 32), sel, st, a) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    note_launch(1);
    return MOE_OK;
}
static int launch_select(const RouteArgs& a, cudaStream_t st) {
    FP4MOE_EPL_DISPATCH(a.E, return launch_select_epl<EPL>(a, st));
    return MOE_ERR_LAUNCH;
}

// Dynamic shared memory of the decode router: the router rows and token rows of the logit
// phase, or the selecting warps' arrays, whichever is larger.
static size_t decode_route_smem(int T, int d, int E, int epb) {
    const int sel_warps = std::min(epb * kDecodeKS * decode_groups(T, epb), T);
    return std::max(decode_smem_bytes(T, d, epb), (size_t)sel_warps * select_smem_per_warp(E));
}
// Experts per decode-router block: the fewest (at most kDecodeWarps) that cover E with one
// block per SM.
static int decode_epb(int E, int num_sms) {
    const int sms = num_sms > 0 ? num_sms : 1;
    const int e = (E + sms - 1) / sms;
    return e < 1 ? 1 : (e > kDecodeWarps ? kDecodeWarps : e);
}

template <int CH, int EPL>
static int launch_decode_ch(RouteArgs a, cudaStream_t st, int num_sms) {
    a.dec_epb = decode_epb(a.E, num_sms);
    const int threads = a.dec_epb * kDecodeKS * 32 * decode_groups(a.T, a.dec_epb);
    const size_t smem = decode_route_smem(a.T, a.d, a.E, a.dec_epb);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(route_decode_kernel<CH, EPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
        return MOE_ERR_LAUNCH;
    const int m = a.d / 256;    // compensated steps per chain and lane
    const double coef = gamma32(CH - 1) + gamma32(m) * gamma32(m) + 1.0 / 17179869184.0;   // + 2^-34
    a.bound_coef = (float)(coef * (1.0 + 1.0 / 4096.0));                                   // rounded up
    int blocks = (a.E + a.dec_epb - 1) / a.dec_epb;
    if (num_sms > 0 && blocks > num_sms) blocks = num_sms;
    if (launch_pdl(route_decode_kernel<CH, EPL>, dim3(blocks), dim3(threads), smem, st, a) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    note_launch(1);
    return MOE_OK;
}

// Router launches for RouteArgs with every pointer set: the decode kernel when the tokens'
// rows fit in shared memory, else norms -> tiled logits -> selection.
static int launch_route_args(RouteArgs& a, cudaStream_t st, int num_sms) {
    if (a.T == 0) return MOE_OK;
    {
        const int m = a.d / 256;   // the decode bound for one-product chunks (selection's refinement)
        const double coef = gamma32(0) + gamma32(m) * gamma32(m) + 1.0 / 17179869184.0;
        a.refine_coef = (float)(coef * (1.0 + 1.0 / 4096.0));
    }
    if (a.T <= kDecodeMaxT && decode_route_smem(a.T, a.d, a.E, decode_epb(a.E, num_sms)) <= kDecodeSmemMax) {
        // chunks of one product for every T: a token's logits are then the same arithmetic
        // whatever the other tokens of the call (verify rows equal their decode calls)
        FP4MOE_EPL_DISPATCH(a.E, return launch_decode_ch<1, EPL>(a, st, num_sms));
        return MOE_ERR_LAUNCH;
    }
    a.bound_coef = gamma_coef(kChunkK + (a.d + kChunkK - 1) / kChunkK + 1);
    const int rows = a.T + a.E;
    route_norms_kernel<<<(rows + 7) / 8, 256, 0, st>>>(a);
    dim3 grid((a.E + kTileE - 1) / kTileE, (a.T + kTileT - 1) / kTileT);
    route_tiled_kernel<<<grid, kTiledThreads, 0, st>>>(a);
    note_launch(2);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_LAUNCH;
    return launch_select(a, st);
}

int launch_route(const moe_dims* m, int T, const uint16_t* x, const uint16_t* wr, const float* bias,
                 const int32_t* table, int32_t* ids, float* w, int32_t* slots, int32_t* status,
                 char* ws, const WsLayout& L, cudaStream_t st, int num_sms) {
    RouteArgs a{};
    a.T = T; a.d = m->d; a.E = m->num_experts; a.k = m->top_k;
    a.x = x; a.wr = wr; a.bias = bias; a.table = table;
    a.ids = ids; a.w = w; a.slots = slots; a.status = status;
    a.keys = reinterpret_cast<float4*>(ws + L.keys);
    a.xnorm = reinterpret_cast<float*>(ws + L.xnorm);
    a.wnorm = reinterpret_cast<float*>(ws + L.wnorm);
    a.counter = reinterpret_cast<unsigned*>(ws + L.counter) + kCtrRoute;
    return launch_route_args(a, st, num_sms);
}

}  // namespace fp4moe

// ------------------------------------------------------------------ router with static scratch
//
// A variant of the decode-regime router for callers that cannot allocate device memory: an
// op hosted by an engine that owns the whole device pool and hands its ops no workspace, or
// a serving loop that must not allocate between steps.  Its scratch (fast logits, norms and
// the completion ticket) lives in the file-scope array below instead of a caller workspace.
// Every GPU that loads this library holds the array until the process exits.

namespace fp4moe {

constexpr int kStaticMaxT = kDecodeMaxT;   // tokens per call
constexpr size_t kStaticCounterBytes = 256;
constexpr size_t kStaticKeyBytes = sizeof(float4) * kStaticMaxT * kMaxExperts;
constexpr size_t kStaticXnormBytes = 256;
constexpr size_t kStaticWnormBytes = sizeof(float) * kMaxExperts;
constexpr size_t kStaticScratchBytes = kStaticCounterBytes + kStaticKeyBytes + kStaticXnormBytes + kStaticWnormBytes;

static __device__ __align__(256) unsigned char g_route_scratch[kStaticScratchBytes];

}  // namespace fp4moe

#include <mutex>

namespace {
std::mutex g_route_scratch_mu;
void* g_route_scratch_addr[64] = {nullptr};
}  // namespace

extern "C" int moe_route_topk_noalloc(const moe_dims* dims, int32_t T, const uint16_t* x, const uint16_t* w_router,
                                      const float* score_bias, const int32_t* expert_to_slot, int32_t* topk_ids,
                                      float* topk_w, int32_t* topk_slot, int32_t* dev_status, void* stream) {
    using namespace fp4moe;
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    if (T < 0 || T > kStaticMaxT) return MOE_ERR_TOKENS;
    if (!x || !w_router || !expert_to_slot || !topk_ids || !topk_w || !topk_slot || !dev_status) return MOE_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(w_router) & 15u)) return MOE_ERR_ALIGN;
    if (T == 0) return MOE_OK;
    // Host code may not use g_route_scratch as an address: look up its device address once
    // per device, with that device current.
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_LAUNCH;
    unsigned char* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_route_scratch_mu);
        if (!g_route_scratch_addr[dev]) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_LAUNCH;
            g_route_scratch_addr[dev] = p;
        }
        base = static_cast<unsigned char*>(g_route_scratch_addr[dev]);
    }
    cudaStream_t st = (cudaStream_t)stream;
    RouteArgs a{};
    a.T = T; a.d = dims->d; a.E = dims->num_experts; a.k = dims->top_k;
    a.x = x; a.wr = w_router; a.bias = score_bias; a.table = expert_to_slot;
    a.ids = topk_ids; a.w = topk_w; a.slots = topk_slot; a.status = dev_status;
    a.counter = reinterpret_cast<unsigned*>(base);
    a.keys = reinterpret_cast<float4*>(base + kStaticCounterBytes);
    a.xnorm = reinterpret_cast<float*>(base + kStaticCounterBytes + kStaticKeyBytes);
    a.wnorm = reinterpret_cast<float*>(base + kStaticCounterBytes + kStaticKeyBytes + kStaticXnormBytes);
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_LAUNCH;
    return launch_route_args(a, st, sms);
}
