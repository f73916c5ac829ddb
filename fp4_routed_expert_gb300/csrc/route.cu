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

#include "route_select.cuh"

namespace fp4moe {

constexpr int kSelWarps = 4;

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
        select_row<EPL>(a, t, lane, rec, exk, out, route_out(a, t));
}


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
// its own shared memory -- unless a.handoff is set (moe_layer_decode_fp4): then every block
// only releases its records on a.counter and the expert kernel launched next selects.
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
    if (a.handoff) {
        // the expert kernel of this call selects: it waits for one release per block, and
        // the last of its CTAs to exit puts the counter back to zero
        if (tid == 0) red_add_release(reinterpret_cast<int32_t*>(a.counter), 1);
        return;
    }
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
    for (int t = wsel; t < T; t += nsel) select_row<EPL>(a, t, lane, rec, exk, out, route_out(a, t));
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
static int launch_decode_ch(RouteArgs a, cudaStream_t st, int num_sms, int* blocks_out = nullptr) {
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
    if (blocks_out) *blocks_out = blocks;
    return MOE_OK;
}

// The decode bound for chunks of one product (the selection's refinement).
static float refine_coef_of(int d) {
    const int m = d / 256;
    const double coef = gamma32(0) + gamma32(m) * gamma32(m) + 1.0 / 17179869184.0;
    return (float)(coef * (1.0 + 1.0 / 4096.0));
}

// Router launches for RouteArgs with every pointer set: the decode kernel when the tokens'
// rows fit in shared memory, else norms -> tiled logits -> selection.
static int launch_route_args(RouteArgs& a, cudaStream_t st, int num_sms) {
    if (a.T == 0) return MOE_OK;
    a.refine_coef = refine_coef_of(a.d);
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

static RouteArgs route_args(const moe_dims* m, int T, const uint16_t* x, const uint16_t* wr, const float* bias,
                            const int32_t* table, int32_t* ids, float* w, int32_t* slots, int32_t* status, char* ws,
                            const WsLayout& L) {
    RouteArgs a{};
    a.T = T; a.d = m->d; a.E = m->num_experts; a.k = m->top_k;
    a.x = x; a.wr = wr; a.bias = bias; a.table = table;
    a.ids = ids; a.w = w; a.slots = slots; a.status = status;
    a.keys = reinterpret_cast<float4*>(ws + L.keys);
    a.xnorm = reinterpret_cast<float*>(ws + L.xnorm);
    a.wnorm = reinterpret_cast<float*>(ws + L.wnorm);
    a.counter = reinterpret_cast<unsigned*>(ws + L.counter) + kCtrRoute;
    return a;
}

int launch_route(const moe_dims* m, int T, const uint16_t* x, const uint16_t* wr, const float* bias,
                 const int32_t* table, int32_t* ids, float* w, int32_t* slots, int32_t* status,
                 char* ws, const WsLayout& L, cudaStream_t st, int num_sms) {
    RouteArgs a = route_args(m, T, x, wr, bias, table, ids, w, slots, status, ws, L);
    return launch_route_args(a, st, num_sms);
}

int launch_route_handoff(const moe_dims* m, int T, const uint16_t* x, const uint16_t* wr, const float* bias,
                         const int32_t* table, int32_t* ids, float* w, int32_t* slots, int32_t* status, char* ws,
                         const WsLayout& L, cudaStream_t st, int num_sms, RouteArgs* ra, int* blocks) {
    RouteArgs a = route_args(m, T, x, wr, bias, table, ids, w, slots, status, ws, L);
    if (T < 1 || T > kDecodeMaxT || a.E > kHandoffMaxExperts ||
        decode_route_smem(a.T, a.d, a.E, decode_epb(a.E, num_sms)) > kDecodeSmemMax)
        return 1;
    a.refine_coef = refine_coef_of(a.d);
    a.handoff = 1;
    int rc = MOE_ERR_LAUNCH;
    FP4MOE_EPL_DISPATCH(a.E, rc = launch_decode_ch<1, EPL>(a, st, num_sms, blocks));
    *ra = a;
    return rc;
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
