// cb3.cu -- the cb3 expert format: a 3-bit per-row codebook packed from the FP4 experts, its
// packer and its decode-regime expert FFN.
//
// "DeepSeek-V4.1-Flash on a single NVIDIA DGX Spark", section "The numbers": resident experts
// held in a 3-bit per-row codebook packed from the checkpoint's own FP4 experts (an
// approximation of the model, traded for capacity: 13.4 MB per expert instead of 18.8 MB at
// d=5120, f=2304).  Every matrix row gets 8 bf16 levels; every weight a 3-bit index.  The
// levels are the optimal 1-D 8-means of the row's FP4 values: clusters are contiguous runs of
// the sorted distinct values, found exactly by dynamic programming over split points (ties to
// the smaller split), and a level is its cluster's mean rounded once to bf16.  The packer
// keeps every fp64 step in one fixed order (explicit _rn intrinsics, no contraction), so its
// output is a function of the row alone.
//
// Slot layout (rows rho: gate 0..f-1, up f..2f-1, down 2f..2f+d-1; K = d for gate/up rows,
// K = f for down rows):
//   levels   16 bytes per row at 16*rho: 8 bf16, ascending; unused levels are 0.
//   indices  from 16*(2f+d): gate rows (3d/8 bytes each), up rows, down rows (3f/8 bytes
//            each).  A row is three arrays of K/32 uint32 words A[c], B[c], Z[c] for the
//            32-element groups c.  Element j of group c with index v has
//              A[c]: (v & 3) at bit 4(j%8) + 2(j/8)           for j < 16
//              B[c]: (v & 3) at bit 4(j%8) + 2((j-16)/8)      for j >= 16
//              Z[c]: (v >> 2) at bit 4(j%8) + {2, 3, 0, 1}[j/8]
//            so two masks and two shifts turn (A or B, Z) into 8 nibbles that are the indices
//            of 8 consecutive elements -- byte-permute selectors into the row's level bytes.
#include "moe_internal.cuh"

namespace fp4moe {

constexpr int kCb3Bins = 1037;          // sortable FP4 value bins (see cb3_bin)
constexpr int kCb3MaxDistinct = 256;    // distinct values a row may hold
constexpr int kCb3ZeroBin = 518;

struct Cb3Layout {
    int64_t gate, up, down, bytes;      // index regions; levels start at 0
};

__host__ __device__ inline Cb3Layout cb3_layout(int d, int f) {
    Cb3Layout L;
    const int64_t R = 2 * (int64_t)f + d;
    L.gate = 16 * R;
    L.up = L.gate + (int64_t)f * (3 * d / 8);
    L.down = L.up + (int64_t)f * (3 * d / 8);
    const int64_t end = L.down + (int64_t)d * (3 * f / 8);
    L.bytes = (end + 1023) / 1024 * 1024;
    return L;
}

int64_t cb3_slot_bytes(int d, int f) { return cb3_layout(d, f).bytes; }

// ---------------------------------------------------------------------------- packer

// Bin of the FP4 value (code, UE8M0 byte sb < 255), ascending in value.  A nonzero magnitude
// is o * 2^E with o in {1, 3}; q = 2E (o = 1) or 2E + 3 (o = 3) orders the magnitudes
// (2^E < 3*2^(E-1) < 2^(E+1) < 3*2^E ...), and E = sb - 127 + k lies in [-128, 129].
__device__ __forceinline__ int cb3_bin(uint32_t code, uint32_t sb) {
    const uint32_t m = code & 7u;
    if (m == 0) return kCb3ZeroBin;
    // magnitude m (0.5, 1, 1.5, 2, 3, 4, 6) = o * 2^k: m=1 (1,-1), 2 (1,0), 3 (3,-1), 4 (1,1),
    // 5 (3,0), 6 (1,2), 7 (3,1)
    const int k = (m == 1 || m == 3) ? -1 : (m == 2 || m == 5) ? 0 : (m == 4 || m == 7) ? 1 : 2;
    const int odd3 = (m == 3 || m == 5 || m == 7) ? 3 : 0;
    const int q = 2 * ((int)sb - 127 + k) + odd3 + 256;      // 0 .. 515
    return (code & 8u) ? 517 - q : 519 + q;
}

__device__ __forceinline__ double pow2d(int e) {            // 2^e, -1022 <= e <= 1023
    return __longlong_as_double((long long)(e + 1023) << 52);
}

__device__ __forceinline__ double cb3_bin_value(int bin) {
    if (bin == kCb3ZeroBin) return 0.0;
    const int q = (bin > kCb3ZeroBin ? bin - 519 : 517 - bin) - 256;
    const double mag = (q & 1) ? 3.0 * pow2d((q - 3) / 2) : pow2d(q / 2);
    return bin > kCb3ZeroBin ? mag : -mag;
}

// bf16 nearest to a double, ties to even, one rounding; overflow gives infinity.
__device__ __forceinline__ uint16_t bf16_from_f64(double v) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(v);
    const uint16_t sign = (uint16_t)((u >> 48) & 0x8000u);
    const unsigned long long a = u & 0x7FFFFFFFFFFFFFFFull;
    if (a == 0) return sign;
    const int e = (int)(a >> 52) - 1023;                      // |v| in [2^e, 2^(e+1)); v is normal
    const unsigned long long M = (a & 0x000FFFFFFFFFFFFFull) | (1ull << 52);
    const int q = (e - 7 > -133) ? e - 7 : -133;              // quantum 2^q (subnormal floor)
    const int s = q - e + 52;                                  // M >> s counts quanta
    unsigned long long r;
    if (s >= 64) {
        r = 0;
    } else {
        r = M >> s;
        const unsigned long long rem = M & ((1ull << s) - 1), half = 1ull << (s - 1);
        if (rem > half || (rem == half && (r & 1))) ++r;
    }
    uint32_t bits = (q == -133) ? (uint32_t)r : (uint32_t)((e + 127) << 7) + (uint32_t)(r - 128);
    if (bits >= 0x7F80u) bits = 0x7F80u;
    return (uint16_t)(sign | bits);
}

struct Cb3Row {
    const uint8_t* mat;   // FP4 matrix of the row (tiled arena layout)
    int row, K;           // row within that matrix
    uint8_t* idx;         // the row's index arrays
};

__device__ __forceinline__ Cb3Row cb3_row(const uint8_t* src, const SlotLayout& L, uint8_t* dst, const Cb3Layout& C,
                                          int rho, int d, int f) {
    Cb3Row r;
    if (rho < f) {
        r.mat = src + L.gu; r.row = 2 * rho; r.K = d; r.idx = dst + C.gate + (int64_t)rho * (3 * d / 8);
    } else if (rho < 2 * f) {
        r.mat = src + L.gu; r.row = 2 * (rho - f) + 1; r.K = d; r.idx = dst + C.up + (int64_t)(rho - f) * (3 * d / 8);
    } else {
        r.mat = src + L.dn; r.row = rho - 2 * f; r.K = f; r.idx = dst + C.down + (int64_t)(rho - 2 * f) * (3 * f / 8);
    }
    return r;
}

// One block per row.  Histogram of the row's values over the sortable bins, the distinct
// values ascending, prefix sums, the 8-means dynamic program, levels, then the 3-bit indices.
__global__ void __launch_bounds__(256) cb3_pack_kernel(const uint8_t* __restrict__ src, SlotLayout L,
                                                       uint8_t* __restrict__ dst, Cb3Layout C, int d, int f,
                                                       int32_t* status) {
    __shared__ int hist[kCb3Bins];
    __shared__ short pos_of[kCb3Bins];
    __shared__ double uval[kCb3MaxDistinct];
    __shared__ double ucnt[kCb3MaxDistinct];
    __shared__ double Np[kCb3MaxDistinct + 1], Sp[kCb3MaxDistinct + 1], Qp[kCb3MaxDistinct + 1];
    __shared__ double Dp[2][kCb3MaxDistinct + 1];
    __shared__ short split[9][kCb3MaxDistinct + 1];
    __shared__ unsigned char grp[kCb3MaxDistinct];
    __shared__ int n_s, bad_s;
    const int tid = threadIdx.x, lane = tid & 31;
    const int rho = blockIdx.x;
    const Cb3Row R = cb3_row(src, L, dst, C, rho, d, f);
    const int K = R.K, nc = K / 32;
    for (int i = tid; i < kCb3Bins; i += blockDim.x) hist[i] = 0;
    if (tid == 0) bad_s = 0;
    __syncthreads();
    for (int c = tid; c < nc; c += blockDim.x) {
        const uint4 q = *reinterpret_cast<const uint4*>(R.mat + code_chunk_off(R.row, c, K));
        const uint32_t sb = R.mat[scale_off(R.row, c, K)];
        if (sb == 255u) { bad_s = 1; continue; }
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 32; ++e) atomicAdd(&hist[cb3_bin((w[e >> 3] >> (4 * (e & 7))) & 15u, sb)], 1);
    }
    __syncthreads();
    // distinct values, ascending (warp 0)
    if (tid < 32) {
        int n = 0;
        for (int base = 0; base < kCb3Bins; base += 32) {
            const int bin = base + lane;
            const bool has = bin < kCb3Bins && hist[bin] > 0;
            const unsigned m = __ballot_sync(0xffffffffu, has);
            const int p = n + __popc(m & ((1u << lane) - 1u));
            if (has) {
                pos_of[bin] = (short)p;
                if (p < kCb3MaxDistinct) { uval[p] = cb3_bin_value(bin); ucnt[p] = (double)hist[bin]; }
            }
            n += __popc(m);
        }
        if (lane == 0) n_s = n;
    }
    __syncthreads();
    const int n = n_s;
    uint4* lv_out = reinterpret_cast<uint4*>(dst + 16 * (int64_t)rho);
    if (bad_s || n > kCb3MaxDistinct) {
        // not representable: zero levels and indices, flagged
        if (tid == 0) { atomicOr(status, MOE_STATUS_CB3_ROW); *lv_out = make_uint4(0, 0, 0, 0); }
        for (int i = tid; i < 3 * nc; i += blockDim.x) reinterpret_cast<uint32_t*>(R.idx)[i] = 0u;
        return;
    }
    if (tid == 0) {
        Np[0] = Sp[0] = Qp[0] = 0.0;
        for (int i = 0; i < n; ++i) {
            const double cu = __dmul_rn(ucnt[i], uval[i]);
            Np[i + 1] = __dadd_rn(Np[i], ucnt[i]);
            Sp[i + 1] = __dadd_rn(Sp[i], cu);
            Qp[i + 1] = __dadd_rn(Qp[i], __dmul_rn(cu, uval[i]));
        }
    }
    __syncthreads();
    // squared error of distinct values [a, b)
    auto cost = [&](int a, int b) -> double {
        const double s1 = __dsub_rn(Sp[b], Sp[a]);
        const double s2 = __dsub_rn(Qp[b], Qp[a]);
        const double nn = __dsub_rn(Np[b], Np[a]);
        return __dsub_rn(s2, __ddiv_rn(__dmul_rn(s1, s1), nn));
    };
    const int G = n < 8 ? n : 8;
    for (int i = 1 + tid; i <= n; i += blockDim.x) { Dp[1][i] = cost(0, i); split[1][i] = 0; }
    for (int g = 2; g <= G; ++g) {
        __syncthreads();
        const double* prev = Dp[(g - 1) & 1];
        double* cur = Dp[g & 1];
        for (int i = g + tid; i <= n; i += blockDim.x) {
            int best = -1;
            double bv = 0.0;
            for (int m = g - 1; m < i; ++m) {
                const double c = __dadd_rn(prev[m], cost(m, i));
                if (best < 0 || c < bv) { best = m; bv = c; }
            }
            cur[i] = bv;
            split[g][i] = (short)best;
        }
    }
    __syncthreads();
    if (tid == 0) {
        uint16_t lv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        int b = n;
        for (int g = G; g >= 1; --g) {
            const int a = split[g][b];
            lv[g - 1] = bf16_from_f64(__ddiv_rn(__dsub_rn(Sp[b], Sp[a]), __dsub_rn(Np[b], Np[a])));
            for (int p = a; p < b; ++p) grp[p] = (unsigned char)(g - 1);
            b = a;
        }
        *lv_out = make_uint4(lv[0] | (uint32_t)lv[1] << 16, lv[2] | (uint32_t)lv[3] << 16, lv[4] | (uint32_t)lv[5] << 16,
                             lv[6] | (uint32_t)lv[7] << 16);
    }
    __syncthreads();
    uint32_t* Aw = reinterpret_cast<uint32_t*>(R.idx);
    for (int c = tid; c < nc; c += blockDim.x) {
        const uint4 q = *reinterpret_cast<const uint4*>(R.mat + code_chunk_off(R.row, c, K));
        const uint32_t sb = R.mat[scale_off(R.row, c, K)];
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        uint32_t A = 0, B = 0, Z = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const uint32_t v = grp[pos_of[cb3_bin((w[j >> 3] >> (4 * (j & 7))) & 15u, sb)]];
            const int nib = 4 * (j & 7);
            if (j < 16) A |= (v & 3u) << (nib + 2 * (j >> 3));
            else B |= (v & 3u) << (nib + 2 * ((j - 16) >> 3));
            Z |= (v >> 2) << (nib + ((j >> 3) == 0 ? 2 : (j >> 3) == 1 ? 3 : (j >> 3) == 2 ? 0 : 1));
        }
        Aw[c] = A;
        Aw[nc + c] = B;
        Aw[2 * nc + c] = Z;
    }
}

// ---------------------------------------------------------------------------- FFN

// Row decoding.  The 8 levels of a row as byte tables for prmt: lo[0..1] hold the low bytes
// of levels 0-3 and 4-7, hi[0..1] the high bytes.
struct Cb3Levels {
    uint32_t lo0, lo1, hi0, hi1;
};

__device__ __forceinline__ Cb3Levels cb3_levels(const uint8_t* p) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    Cb3Levels l;
    l.lo0 = __byte_perm(v.x, v.y, 0x6420);
    l.hi0 = __byte_perm(v.x, v.y, 0x7531);
    l.lo1 = __byte_perm(v.z, v.w, 0x6420);
    l.hi1 = __byte_perm(v.z, v.w, 0x7531);
    return l;
}

// Nibble selectors of quarter Q (elements 8Q..8Q+7) of a group from its A, B, Z words.
template <int Q>
__device__ __forceinline__ uint32_t cb3_nibbles(uint32_t A, uint32_t B, uint32_t Z) {
    if (Q == 0) return (A & 0x33333333u) | (Z & 0x44444444u);
    if (Q == 1) return ((A >> 2) & 0x33333333u) | ((Z >> 1) & 0x44444444u);
    if (Q == 2) return (B & 0x33333333u) | ((Z << 2) & 0x44444444u);
    return ((B >> 2) & 0x33333333u) | ((Z << 1) & 0x44444444u);
}

// The 8 weights (fp32) selected by the 8 nibbles of N.
__device__ __forceinline__ void cb3_weights8(const Cb3Levels& l, uint32_t N, float* w) {
    const uint32_t la = __byte_perm(l.lo0, l.lo1, N), ha = __byte_perm(l.hi0, l.hi1, N);
    const uint32_t lb = __byte_perm(l.lo0, l.lo1, N >> 16), hb = __byte_perm(l.hi0, l.hi1, N >> 16);
    const uint32_t e01 = __byte_perm(la, ha, 0x5140), e23 = __byte_perm(la, ha, 0x7362);
    const uint32_t e45 = __byte_perm(lb, hb, 0x5140), e67 = __byte_perm(lb, hb, 0x7362);
    w[0] = bf16_lo(e01); w[1] = bf16_hi(e01); w[2] = bf16_lo(e23); w[3] = bf16_hi(e23);
    w[4] = bf16_lo(e45); w[5] = bf16_hi(e45); w[6] = bf16_lo(e67); w[7] = bf16_hi(e67);
}

__device__ __forceinline__ uint32_t ldg_nc_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

constexpr int kCb3XT = 8;   // tokens per pass of the gate/up kernel

__host__ __device__ constexpr int cb3_padded(int n) { return n + n / 8; }

struct Cb3Args {
    int T, d, f, k, num_slots;
    int t0, tn;
    const uint16_t* x;
    const int32_t* slot;        // [T, k]
    const float* w;             // [T, k]
    const uint8_t* arena;
    int64_t slot_bytes;
    Cb3Layout C;
    float* h;                   // [T*k, f]
    uint16_t* y;                // [T, d]
    int32_t* status;
};

// Dot of one 32-element group of a row with staged activations a (36-float stride per group:
// 32 values then 4 pad), accumulated into acc[0..nq) for the nq tokens at a + tok_off[q].
template <int XT>
__device__ __forceinline__ void cb3_group_dot(const Cb3Levels& l, uint32_t A, uint32_t B, uint32_t Z, const float* a,
                                              const int* tok_off, int nq, float* acc) {
    float wv[8];
#pragma unroll
    for (int Q = 0; Q < 4; ++Q) {
        const uint32_t N = Q == 0 ? cb3_nibbles<0>(A, B, Z) : Q == 1 ? cb3_nibbles<1>(A, B, Z)
                         : Q == 2 ? cb3_nibbles<2>(A, B, Z) : cb3_nibbles<3>(A, B, Z);
        cb3_weights8(l, N, wv);
#pragma unroll
        for (int q = 0; q < XT; ++q) {
            if (q >= nq) break;
            const float4* a4 = reinterpret_cast<const float4*>(a + tok_off[q] + 8 * Q);
            const float4 p = a4[0], r = a4[1];
            float s = acc[q];
            s = fmaf(wv[0], p.x, s); s = fmaf(wv[1], p.y, s); s = fmaf(wv[2], p.z, s); s = fmaf(wv[3], p.w, s);
            s = fmaf(wv[4], r.x, s); s = fmaf(wv[5], r.y, s); s = fmaf(wv[6], r.z, s); s = fmaf(wv[7], r.w, s);
            acc[q] = s;
        }
    }
}

// Gate/up + SwiGLU.  Items are (unique slot u, output i); a warp reads gate row i and up row
// i of slot u (lane owns groups lane, lane+32, ...) and reduces for every token of this pass
// routed to u.  Shared memory: the pass's tokens as fp32 [tn][cb3_padded(d)].
template <int XT>
__global__ void __launch_bounds__(256) cb3_gateup_kernel(Cb3Args a) {
    extern __shared__ float xs[];
    __shared__ int uniq_slot[kCb3XT * kMaxTopK];
    __shared__ int mem_cnt[kCb3XT * kMaxTopK];
    __shared__ int mem_pair[kCb3XT * kMaxTopK][kCb3XT];
    __shared__ int n_uniq;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, f = a.f, k = a.k, tn = a.tn;
    if (tid == 0) {
        int nu = 0;
        for (int q = 0; q < tn * k; ++q) {
            const int p = a.t0 * k + q;
            const int s = a.slot[p];
            if (s < 0) continue;
            if (s >= a.num_slots) { if (blockIdx.x == 0) atomicOr(a.status, MOE_STATUS_BAD_SLOT); continue; }
            int u = 0;
            while (u < nu && !(uniq_slot[u] == s && mem_cnt[u] < XT)) ++u;
            if (u == nu) { uniq_slot[nu] = s; mem_cnt[nu] = 0; ++nu; }
            mem_pair[u][mem_cnt[u]++] = p;
        }
        n_uniq = nu;
    }
    for (int t = 0; t < tn; ++t) {
        const uint16_t* xt = a.x + (size_t)(a.t0 + t) * d;
        for (int i = tid; i < d; i += blockDim.x) xs[(size_t)t * cb3_padded(d) + i + 4 * (i >> 5)] = bf16_to_f32(xt[i]);
    }
    __syncthreads();
    const int nu = n_uniq, nc = d / 32;
    const int gw = blockIdx.x * (blockDim.x >> 5) + warp, nw = gridDim.x * (blockDim.x >> 5);
    for (int it = gw; it < nu * f; it += nw) {
        const int u = it / f, i = it % f;
        const uint8_t* base = a.arena + (int64_t)uniq_slot[u] * a.slot_bytes;
        const Cb3Levels lg = cb3_levels(base + 16 * (int64_t)i), lu = cb3_levels(base + 16 * (int64_t)(f + i));
        const uint32_t* ig = reinterpret_cast<const uint32_t*>(base + a.C.gate + (int64_t)i * (3 * d / 8));
        const uint32_t* iu = reinterpret_cast<const uint32_t*>(base + a.C.up + (int64_t)i * (3 * d / 8));
        const int nmem = mem_cnt[u];
        int tok_off[XT];
#pragma unroll
        for (int q = 0; q < XT; ++q) tok_off[q] = q < nmem ? (mem_pair[u][q] / k - a.t0) * cb3_padded(d) : 0;
        float accg[XT], accu[XT];
#pragma unroll
        for (int q = 0; q < XT; ++q) accg[q] = accu[q] = 0.f;
        for (int c0 = lane; c0 < nc; c0 += 32 * 4) {
            uint32_t g3[4][3], u3[4][3];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int c = c0 + 32 * b;
                if (c < nc) {
#pragma unroll
                    for (int r = 0; r < 3; ++r) { g3[b][r] = ldg_nc_u32(ig + r * nc + c); u3[b][r] = ldg_nc_u32(iu + r * nc + c); }
                }
            }
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int c = c0 + 32 * b;
                if (c >= nc) break;
                const float* xa = xs + 36 * c;
                cb3_group_dot<XT>(lg, g3[b][0], g3[b][1], g3[b][2], xa, tok_off, nmem, accg);
                cb3_group_dot<XT>(lu, u3[b][0], u3[b][1], u3[b][2], xa, tok_off, nmem, accu);
            }
        }
#pragma unroll
        for (int q = 0; q < XT; ++q) {
            if (q >= nmem) break;
            const float g = warp_sum(accg[q]), uu = warp_sum(accu[q]);
            if (lane == 0) a.h[(size_t)mem_pair[u][q] * f + i] = g / (1.0f + expf(-g)) * uu;
        }
    }
}

// Down + fixed-order combine.  Each warp owns 4 output rows (8 lanes per row; lane owns
// groups l8, l8+8, ...); for each token the k pairs are visited in ascending j.  Shared
// memory: the token's k vectors h [k][cb3_padded(f)].
__global__ void __launch_bounds__(256) cb3_down_kernel(Cb3Args a) {
    extern __shared__ float hs[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, f = a.f, k = a.k;
    const int l8 = lane & 7, grp = lane >> 3;
    const int nc = f / 32;
    const int r = blockIdx.x * ((blockDim.x >> 5) * 4) + warp * 4 + grp;
    for (int t = 0; t < a.T; ++t) {
        __syncthreads();
        for (int j = 0; j < k; ++j) {
            const int pair = t * k + j;
            const int s = a.slot[pair];
            const bool ok = s >= 0 && s < a.num_slots;
            const float* hp = a.h + (size_t)pair * f;
            for (int i = tid; i < f; i += blockDim.x) hs[(size_t)j * cb3_padded(f) + i + 4 * (i >> 5)] = ok ? __ldcg(hp + i) : 0.f;
        }
        __syncthreads();
        if (r >= d) continue;
        float y = 0.f;
        for (int j = 0; j < k; ++j) {
            const int pair = t * k + j;
            const int s = a.slot[pair];
            if (s < 0 || s >= a.num_slots) continue;      // the same pair for the whole warp
            const uint8_t* base = a.arena + (int64_t)s * a.slot_bytes;
            const Cb3Levels l = cb3_levels(base + 16 * (int64_t)(2 * f + r));
            const uint32_t* ix = reinterpret_cast<const uint32_t*>(base + a.C.down + (int64_t)r * (3 * f / 8));
            const float* hj = hs + (size_t)j * cb3_padded(f);
            const int tok0[1] = {0};
            float acc = 0.f;
            for (int c0 = l8; c0 < nc; c0 += 8 * 3) {
                uint32_t w3[3][3];
#pragma unroll
                for (int b = 0; b < 3; ++b) {
                    const int c = c0 + 8 * b;
                    if (c < nc) {
#pragma unroll
                        for (int q = 0; q < 3; ++q) w3[b][q] = ldg_nc_u32(ix + q * nc + c);
                    }
                }
#pragma unroll
                for (int b = 0; b < 3; ++b) {
                    const int c = c0 + 8 * b;
                    if (c >= nc) break;
                    cb3_group_dot<1>(l, w3[b][0], w3[b][1], w3[b][2], hj + 36 * c, tok0, 1, &acc);
                }
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 4);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            y = fmaf(a.w[pair], acc, y);
        }
        if (l8 == 0) a.y[(size_t)t * d + r] = f32_to_bf16(y);
    }
}

// ---------------------------------------------------------------------------- host side

int launch_pack_cb3(const moe_dims* m, const uint8_t* src_slot, uint8_t* dst_slot, int32_t* status, cudaStream_t st) {
    const int rows = 2 * m->f + m->d;
    cb3_pack_kernel<<<rows, 256, 0, st>>>(src_slot, slot_layout(m->d, m->f), dst_slot, cb3_layout(m->d, m->f), m->d,
                                          m->f, status);
    note_launch(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

template <int XT>
static int launch_cb3_gateup(const Cb3Args& a, size_t smem, int blocks, cudaStream_t st) {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(cb3_gateup_kernel<XT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    cb3_gateup_kernel<XT><<<blocks, 256, smem, st>>>(a);
    note_launch(1);
    return MOE_OK;
}

int launch_cb3_ffn(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                   const float* w, uint16_t* y, int32_t* status, char* ws, const WsLayout& L, cudaStream_t st,
                   int num_sms) {
    if (T == 0) return MOE_OK;
    Cb3Args a;
    a.T = T; a.d = m->d; a.f = m->f; a.k = m->top_k; a.num_slots = ar->num_slots;
    a.x = x; a.slot = slot; a.w = w;
    a.arena = reinterpret_cast<const uint8_t*>(ar->base);
    a.slot_bytes = ar->slot_bytes;
    a.C = cb3_layout(m->d, m->f);
    a.h = reinterpret_cast<float*>(ws + L.h);
    a.y = y; a.status = status;
    for (int t0 = 0; t0 < T; t0 += kCb3XT) {
        a.t0 = t0;
        a.tn = (T - t0 < kCb3XT) ? T - t0 : kCb3XT;
        const size_t smem = (size_t)a.tn * cb3_padded(m->d) * 4;
        const int blocks = 2 * num_sms;
        int rc;
        if (a.tn == 1) rc = launch_cb3_gateup<1>(a, smem, blocks, st);
        else if (a.tn == 2) rc = launch_cb3_gateup<2>(a, smem, blocks, st);
        else if (a.tn <= 4) rc = launch_cb3_gateup<4>(a, smem, blocks, st);
        else rc = launch_cb3_gateup<8>(a, smem, blocks, st);
        if (rc) return rc;
    }
    const size_t smem2 = (size_t)m->top_k * cb3_padded(m->f) * 4;
    if (smem2 > 48 * 1024 &&
        cudaFuncSetAttribute(cb3_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    cb3_down_kernel<<<(m->d + 31) / 32, 256, smem2, st>>>(a);
    note_launch(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

}  // namespace fp4moe
