// ffn_prefill.cu -- prefill-regime permutation, grouped expert FFN and combine (sm_103a).
//
//   permute   stable grouping of the T*k (token, j) rows by expert id
//   gate/up   per group: H[r, i] = silu(Wg[i] . x_r) * (Wu[i] . x_r)
//   down      per group: Z[r, c] = Wd[c] . H[r]
//   combine   y[t, c] = bf16( sum_j w[t, j] * Z[row_dst[t*k + j], c] ),  j ascending
// Every (token, j) row is written once and the slot sum is a separate fixed-order step
// ("Start the expert reads before the GPU is done", 30 September follow-up).
//
// The GEMMs here run on CUDA cores: a 64-row x 64-token tile per block, each 32-wide K step
// is one UE8M0 block, whose FP4 codes are decoded into shared memory as exact fp32 values
// code * 2^(b-127); products with the bf16 / fp32 activations are then exact and summed by
// fp32 FMA chains.
#include "moe_internal.cuh"

namespace fp4moe {

// ---------------------------------------------------------------------------- permute

// One block of 1024 threads.  Counts per expert, exclusive scan, then a stable scatter in
// flat (t*k + j) order: entries are taken 1024 at a time; inside a tile, warp w assigns its
// ranks after warps 0..w-1 (a per-expert cursor in shared memory), lanes of one warp rank by
// their position among lanes with the same id.
__global__ void __launch_bounds__(1024) permute_kernel(int n, int E, const int32_t* __restrict__ ids,
                                                       int32_t* offsets, int32_t* row_src, int32_t* row_dst) {
    __shared__ int cnt[kMaxExperts + 1];
    __shared__ int cursor[kMaxExperts];
    __shared__ int wsum[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e <= E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += blockDim.x) {
        int e = ids[i];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    // exclusive scan of cnt[0..E) (E <= 1024: one element per thread)
    int v = (tid < E) ? cnt[tid] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int s = wsum[lane];
        int is = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int u = __shfl_up_sync(0xffffffffu, is, o);
            if (lane >= o) is += u;
        }
        wsum[lane] = is - s;
    }
    __syncthreads();
    int excl = incl - v + wsum[warp];
    if (tid < E) { offsets[tid] = excl; cursor[tid] = excl; }
    if (tid == E - 1) offsets[E] = excl + v;
    __syncthreads();
    for (int base = 0; base < n; base += blockDim.x) {
        int i = base + tid;
        int e = (i < n) ? ids[i] : -1;
        bool ok = e >= 0 && e < E;
        unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
        for (int w = 0; w < 32; ++w) {
            if (warp == w) {
                int pos = ok ? cursor[e] + __popc(peers & ((1u << lane) - 1u)) : 0;
                __syncwarp();   // every lane has read the cursor before any lane advances it
                if (ok) {
                    row_src[pos] = i;
                    row_dst[i] = pos;
                    if ((peers >> lane) == 1u) cursor[e] += __popc(peers);   // highest lane of the id
                }
            }
            __syncthreads();
        }
        if (i < n && !ok) row_dst[i] = -1;
    }
}

__global__ void permute_tail_kernel(int n, int E, const int32_t* offsets, int32_t* row_src) {
    int total = offsets[E];
    for (int i = total + blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) row_src[i] = -1;
}

// ---------------------------------------------------------------------------- plan

// Validates group_offsets (monotone in [0, n]) and lists the non-empty groups with the
// prefix of their tile counts (tile_rows rows per tile), and the tile row of every pair.
// plan = [n_active, total_tiles, e_0.., tile_start_0..] (layout: see plan_pair_off)
// One block of 1024 threads, thread e = expert e (E <= 1024): block-wide exclusive scans of
// "has rows" and "tiles of tile_rows rows" give each non-empty expert its group index and first
// tile; every group writes its record and its tiles' entries of tile_group.  Offsets that are
// not a valid group partition of n rows (or more tiles than max_tiles) give an empty plan and
// MOE_STATUS_BAD_SLOT.
__global__ void __launch_bounds__(1024) plan_kernel(int E, int n, const int32_t* __restrict__ offsets,
                                                    const int32_t* __restrict__ row_src, const int32_t* __restrict__ slot,
                                                    int nrows, int32_t* plan, int32_t* status, int tile_rows, int max_tiles) {
    __shared__ int wa[32], wt[32];
    __shared__ int bad_sh;
    const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
    if (e == 0) bad_sh = (offsets[0] != 0);
    __syncthreads();
    int o0 = 0, o1 = 0, act = 0, nt = 0;
    if (e < E) {
        o0 = offsets[e];
        o1 = offsets[e + 1];
        if (o1 < o0 || o1 > n) bad_sh = 1;
        act = o1 > o0;
        nt = act ? (o1 - o0 + tile_rows - 1) / tile_rows : 0;
    }
    // inclusive warp scans, then the warp totals
    int sa = act, st = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int ya = __shfl_up_sync(0xffffffffu, sa, o), yt = __shfl_up_sync(0xffffffffu, st, o);
        if (lane >= o) { sa += ya; st += yt; }
    }
    if (lane == 31) { wa[warp] = sa; wt[warp] = st; }
    __syncthreads();
    if (warp == 0) {
        int a = wa[lane], t = wt[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ya = __shfl_up_sync(0xffffffffu, a, o), yt = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) { a += ya; t += yt; }
        }
        wa[lane] = a;   // inclusive over warps
        wt[lane] = t;
    }
    __syncthreads();
    const int g = sa - act + (warp > 0 ? wa[warp - 1] : 0);       // exclusive
    const int ts = st - nt + (warp > 0 ? wt[warp - 1] : 0);
    const int na = wa[31], tiles = wt[31];
    const bool bad = bad_sh || tiles > max_tiles;
    if (!bad && act) {
        plan[2 + g] = e;
        plan[2 + E + g] = ts;
        const int src = row_src[o0];
        const int sl = (src >= 0 && src < nrows) ? slot[src] : -1;
        reinterpret_cast<int4*>(plan + plan_grec_off(E))[g] = make_int4(o0, o1, sl, ts);
        int32_t* tg = plan + plan_tile_group_off(E);
        for (int t = ts; t < ts + nt; ++t) tg[t] = g;
    }
    if (e == 0) {
        plan[0] = bad ? 0 : na;
        plan[1] = bad ? 0 : tiles;
        if (bad) atomicOr(status, MOE_STATUS_BAD_SLOT);
    }
    // pair s -> tile row: permuted row i of expert e (offsets[e] <= i < offsets[e + 1]) sits in
    // row i - offsets[e] of the expert's tiles, which start at tile_start: the linear tile row
    // is tile_start * tile_rows + i - offsets[e]
    __shared__ int so0[kMaxExperts], sts[kMaxExperts];
    int32_t* prow = plan + plan_pair_off(E, max_tiles);
    if (e < E) {
        so0[e] = o0;
        sts[e] = ts;
    }
    for (int i = e; i < nrows; i += blockDim.x) prow[i] = -1;
    __syncthreads();
    if (bad || E < 1) return;
    const int rows_end = offsets[E];
    for (int i = e; i < rows_end && i < nrows; i += blockDim.x) {
        int lo = 0, hi = E - 1;   // the last expert whose rows start at or before i
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (so0[mid] <= i) lo = mid; else hi = mid - 1;
        }
        const int src = row_src[i];
        if (src >= 0 && src < nrows) prow[src] = sts[lo] * tile_rows + (i - so0[lo]);
    }
}

// ---------------------------------------------------------------------------- grouped GEMM

struct GroupedArgs {
    int T, d, f, k, E, num_slots, n;
    const uint16_t* x;          // [T, d]
    const int32_t* offsets;     // [E+1]
    const int32_t* row_src;     // [n]
    const int32_t* slot;        // [T*k]
    const int32_t* plan;
    const uint8_t* arena;
    int64_t slot_bytes;
    SlotLayout L;
    float* h;                   // [n, f] by permuted row
    float* rows;                // [n, d] by permuted row
    int32_t* status;
};

constexpr int kBR = 64, kBT = 64, kBK = 32;

// Decode one 16-byte chunk (32 codes) with its scale byte into exact fp32 values.
__device__ __forceinline__ void decode_chunk(const uint4 q, uint32_t sbyte, float* out /*stride*/, int stride) {
    // code * 2^-126 (bit moves), then * 2^(b-1): exact unless the product leaves the fp32 range
    float sc;
    {
        int e = (int)sbyte - 1;
        sc = (e >= -126) ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(1u << (e + 149));
    }
    uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        uint32_t w = wv[wi];
        out[(8 * wi + 0) * stride] = e2m1_scaled<0>(w) * sc;
        out[(8 * wi + 1) * stride] = e2m1_scaled<1>(w) * sc;
        out[(8 * wi + 2) * stride] = e2m1_scaled<2>(w) * sc;
        out[(8 * wi + 3) * stride] = e2m1_scaled<3>(w) * sc;
        out[(8 * wi + 4) * stride] = e2m1_scaled<4>(w) * sc;
        out[(8 * wi + 5) * stride] = e2m1_scaled<5>(w) * sc;
        out[(8 * wi + 6) * stride] = e2m1_scaled<6>(w) * sc;
        out[(8 * wi + 7) * stride] = e2m1_scaled<7>(w) * sc;
    }
}

// Locate tile `tile` of the flattened (group, token tile) list.
__device__ __forceinline__ int find_group(const int32_t* plan, int E, int na, int ttile) {
    int lo = 0, hi = na - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (plan[2 + E + mid] <= ttile) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// DOWN = false: gate/up + SwiGLU, weight rows = the 2f interleaved gate/up rows, K = d,
//               activations = x rows gathered through row_src; writes h.
// DOWN = true:  down, weight rows = d, K = f, activations = h rows; writes rows.
template <bool DOWN>
__global__ void __launch_bounds__(256) grouped_gemm_kernel(GroupedArgs a) {
    __shared__ float Ws[kBK][kBR + 4];
    __shared__ float Xs[kBK][kBT + 4];
    __shared__ int tok_row[kBT];   // activation row (token for gate/up, permuted row for down), -1 = none
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int E = a.E;
    const int na = a.plan[0], ttiles = a.plan[1];
    const int wrows = DOWN ? a.d : 2 * a.f;
    const int K = DOWN ? a.f : a.d;
    const int nrt = wrows / kBR;
    const long total = (long)ttiles * nrt;
    for (long tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const int ttile = (int)(tile / nrt), rt = (int)(tile % nrt);
        const int g = find_group(a.plan, E, na, ttile);
        const int e = a.plan[2 + g];
        const int r0 = a.offsets[e] + (ttile - a.plan[2 + E + g]) * kBT;
        const int r1 = a.offsets[e + 1];
        __syncthreads();
        if (tid < kBT) {
            int r = r0 + tid;
            int v = -1;
            if (r < r1) {
                int src = a.row_src[r];
                if (src >= 0 && src < a.T * a.k) v = DOWN ? r : src / a.k;
            }
            tok_row[tid] = v;
        }
        // the group's slot (all rows of one group share the expert)
        int s = -1;
        {
            int src = a.row_src[r0];
            if (src >= 0 && src < a.T * a.k) s = a.slot[src];
        }
        const bool slot_ok = s >= 0 && s < a.num_slots;
        if (!slot_ok && tid == 0 && rt == 0) atomicOr(a.status, MOE_STATUS_BAD_SLOT);
        const uint8_t* base = a.arena + (slot_ok ? (int64_t)s * a.slot_bytes : 0);
        const uint8_t* wq = base + (DOWN ? a.L.dn : a.L.gu);
        const uint8_t* wsb = base + (DOWN ? a.L.dn : a.L.gu);
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
        __syncthreads();
        for (int k0 = 0; k0 < K; k0 += kBK) {
            // weights: 64 rows x one 16-byte chunk + scale byte
            if (tid < kBR) {
                int wr = rt * kBR + tid;
                uint4 q = make_uint4(0, 0, 0, 0);
                uint32_t sb = 127;
                if (slot_ok) {
                    q = __ldg(reinterpret_cast<const uint4*>(wq + code_chunk_off(wr, k0 / 32, K)));
                    sb = __ldg(wsb + scale_off(wr, k0 / 32, K));
                }
                decode_chunk(q, sb, &Ws[0][tid], kBR + 4);
            }
            // activations: 64 rows x 32 values
            {
                int rr = tid >> 2, c = (tid & 3) * 8;
                int ar = tok_row[rr];
                float v8[8];
                if (ar >= 0) {
                    if (DOWN) {
                        const float4* hp = reinterpret_cast<const float4*>(a.h + (size_t)ar * a.f + k0 + c);
                        float4 p0 = hp[0], p1 = hp[1];
                        v8[0] = p0.x; v8[1] = p0.y; v8[2] = p0.z; v8[3] = p0.w;
                        v8[4] = p1.x; v8[5] = p1.y; v8[6] = p1.z; v8[7] = p1.w;
                    } else {
                        uint4 u = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)ar * a.d + k0 + c));
                        v8[0] = bf16_lo(u.x); v8[1] = bf16_hi(u.x); v8[2] = bf16_lo(u.y); v8[3] = bf16_hi(u.y);
                        v8[4] = bf16_lo(u.z); v8[5] = bf16_hi(u.z); v8[6] = bf16_lo(u.w); v8[7] = bf16_hi(u.w);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v8[i] = 0.f;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) Xs[c + i][rr] = v8[i];
            }
            __syncthreads();
#pragma unroll 8
            for (int kk = 0; kk < kBK; ++kk) {
                float4 wv = *reinterpret_cast<const float4*>(&Ws[kk][ty * 4]);
                float4 xv = *reinterpret_cast<const float4*>(&Xs[kk][tx * 4]);
                float w4[4] = {wv.x, wv.y, wv.z, wv.w}, x4[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(w4[i], x4[j], acc[i][j]);
            }
            __syncthreads();
        }
        // epilogue
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int rr = tx * 4 + j;
            int r = r0 + rr;
            if (r >= r1 || tok_row[rr] < 0) continue;
            if (DOWN) {
                float4 o = make_float4(acc[0][j], acc[1][j], acc[2][j], acc[3][j]);
                *reinterpret_cast<float4*>(a.rows + (size_t)r * a.d + rt * kBR + ty * 4) = o;
            } else {
                // rows 4ty..4ty+3 are (gate i, up i, gate i+1, up i+1)
                int i0 = (rt * kBR + ty * 4) / 2;
                float g0 = acc[0][j], u0 = acc[1][j], g1 = acc[2][j], u1 = acc[3][j];
                float h0 = g0 / (1.0f + expf(-g0)) * u0;
                float h1 = g1 / (1.0f + expf(-g1)) * u1;
                *reinterpret_cast<float2*>(a.h + (size_t)r * a.f + i0) = make_float2(h0, h1);
            }
        }
    }
}

// ---------------------------------------------------------------------------- combine

__global__ void combine_kernel(int T, int d, int k, const float* __restrict__ rows, const int32_t* __restrict__ row_dst,
                               const float* __restrict__ w, int n, uint16_t* y) {
    const int vec = d / 4;
    for (long idx = blockIdx.x * (long)blockDim.x + threadIdx.x; idx < (long)T * vec; idx += (long)gridDim.x * blockDim.x) {
        int t = (int)(idx / vec), c4 = (int)(idx % vec);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            int r = row_dst[t * k + j];
            if (r < 0 || r >= n) continue;
            float wj = w[t * k + j];
            float4 z = reinterpret_cast<const float4*>(rows + (size_t)r * d)[c4];
            acc.x = fmaf(wj, z.x, acc.x);
            acc.y = fmaf(wj, z.y, acc.y);
            acc.z = fmaf(wj, z.z, acc.z);
            acc.w = fmaf(wj, z.w, acc.w);
        }
        uint32_t lo = (uint32_t)f32_to_bf16(acc.x) | ((uint32_t)f32_to_bf16(acc.y) << 16);
        uint32_t hi = (uint32_t)f32_to_bf16(acc.z) | ((uint32_t)f32_to_bf16(acc.w) << 16);
        reinterpret_cast<uint2*>(y + (size_t)t * d)[c4] = make_uint2(lo, hi);
    }
}

// ---------------------------------------------------------------------------- host side

int launch_permute(const moe_dims* m, int T, const int32_t* ids, int32_t* offsets, int32_t* row_src,
                   int32_t* row_dst, cudaStream_t st) {
    int n = T * m->top_k;
    if (n == 0) {
        return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (m->num_experts + 1), st) == cudaSuccess ? MOE_OK
                                                                                                       : MOE_ERR_LAUNCH;
    }
    permute_kernel<<<1, 1024, 0, st>>>(n, m->num_experts, ids, offsets, row_src, row_dst);
    permute_tail_kernel<<<(n + 255) / 256, 256, 0, st>>>(n, m->num_experts, offsets, row_src);
    note_launch(2);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

int launch_prefill_ffn(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                       const int32_t* offsets, const int32_t* row_src, float* rows_out, int32_t* status, char* ws,
                       const WsLayout& L, cudaStream_t st, int num_sms) {
    GroupedArgs a;
    a.T = T; a.d = m->d; a.f = m->f; a.k = m->top_k; a.E = m->num_experts;
    a.num_slots = ar->num_slots; a.n = T * m->top_k;
    a.x = x; a.offsets = offsets; a.row_src = row_src; a.slot = slot;
    a.plan = reinterpret_cast<const int32_t*>(ws + L.active);
    a.arena = reinterpret_cast<const uint8_t*>(ar->base);
    a.slot_bytes = ar->slot_bytes;
    a.L = slot_layout(m->d, m->f);
    a.h = reinterpret_cast<float*>(ws + L.h);
    a.rows = rows_out;
    a.status = status;
    if (T == 0) return MOE_OK;
    plan_kernel<<<1, 1024, 0, st>>>(a.E, a.n, offsets, row_src, slot, a.n, reinterpret_cast<int32_t*>(ws + L.active),
                                    status, kBT, (int)act_tiles(m, T));
    int blocks = 4 * num_sms;
    grouped_gemm_kernel<false><<<blocks, 256, 0, st>>>(a);
    grouped_gemm_kernel<true><<<blocks, 256, 0, st>>>(a);
    note_launch(3);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

int launch_combine(const moe_dims* m, int T, const float* rows, const int32_t* row_dst, const float* w,
                   uint16_t* y, cudaStream_t st, int num_sms) {
    if (T == 0) return MOE_OK;
    long work = (long)T * (m->d / 4);
    int blocks = (int)((work + 255) / 256);
    if (blocks > 8 * num_sms) blocks = 8 * num_sms;
    combine_kernel<<<blocks, 256, 0, st>>>(T, m->d, m->top_k, rows, row_dst, w, T * m->top_k, y);
    note_launch(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

}  // namespace fp4moe
