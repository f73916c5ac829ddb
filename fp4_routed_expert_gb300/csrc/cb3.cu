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

// Work split.  A warp owns a whole output (gate/up: one h element of one pair; down: 2 rows of
// one pair's z) and adds its lanes' sums by a butterfly.  Gate/up: lane l owns the 32-element
// groups l, l+32, ... of the row, in that order; the token is staged in shared memory as bf16
// and bf16 levels multiply bf16 activations with fma.rn.f32.bf16 (exact products, fp32 sums).
// Down: lane l owns the 8-element quarters l, l+32, ... (f/8 is a multiple of 32, so every
// lane has the same count, and the quarter's position in its group is l % 4 for all of them);
// h is rounded once to bf16 when the gate/up kernel writes it, staged in shared memory, and
// multiplied the same way.  The order of every sum is fixed by the shapes alone,
// so a token's results do not depend on the other tokens of the call.  z rows go to the
// workspace and a last kernel forms y = sum_j w_j z_j in ascending j.

constexpr int kCb3MaxGL = 8;       // gate/up: groups per lane (d <= 8192)
constexpr int kCb3MaxQL = 9;       // down: quarters per lane (f <= 2304)
constexpr int kCb3DnRows = 2;      // output rows per down item

// Levels of a row as byte tables for prmt: lo0/lo1 hold the low bytes of levels 0-3 / 4-7,
// hi0/hi1 their high bytes.
struct Cb3Levels {
    uint32_t lo0, lo1, hi0, hi1;
};

// The levels of row r of a batch whose 16-byte level records lanes 0.. hold (lane r has row r).
__device__ __forceinline__ Cb3Levels cb3_levels_from(const uint4& mine, int r) {
    uint4 v;
    v.x = __shfl_sync(0xffffffffu, mine.x, r);
    v.y = __shfl_sync(0xffffffffu, mine.y, r);
    v.z = __shfl_sync(0xffffffffu, mine.z, r);
    v.w = __shfl_sync(0xffffffffu, mine.w, r);
    Cb3Levels l;
    l.lo0 = __byte_perm(v.x, v.y, 0x6420);
    l.hi0 = __byte_perm(v.x, v.y, 0x7531);
    l.lo1 = __byte_perm(v.z, v.w, 0x6420);
    l.hi1 = __byte_perm(v.z, v.w, 0x7531);
    return l;
}

// Nibble selectors of quarter Q (elements 8Q..8Q+7) of a group from its A, B, Z words.
template <int Q>
__device__ __forceinline__ uint32_t cb3_nibbles(const uint32_t* g) {
    const uint32_t A = g[0], B = g[1], Z = g[2];
    if (Q == 0) return (A & 0x33333333u) | (Z & 0x44444444u);
    if (Q == 1) return ((A >> 2) & 0x33333333u) | ((Z >> 1) & 0x44444444u);
    if (Q == 2) return (B & 0x33333333u) | ((Z << 2) & 0x44444444u);
    return ((B >> 2) & 0x33333333u) | ((Z << 1) & 0x44444444u);
}

// The 8 weights selected by the 8 nibbles of N, as four bf16 pairs (elements 2i, 2i+1).
__device__ __forceinline__ void cb3_pairs8(const Cb3Levels& l, uint32_t N, uint32_t* e) {
    const uint32_t la = __byte_perm(l.lo0, l.lo1, N), ha = __byte_perm(l.hi0, l.hi1, N);
    const uint32_t lb = __byte_perm(l.lo0, l.lo1, N >> 16), hb = __byte_perm(l.hi0, l.hi1, N >> 16);
    e[0] = __byte_perm(la, ha, 0x5140);
    e[1] = __byte_perm(la, ha, 0x7362);
    e[2] = __byte_perm(lb, hb, 0x5140);
    e[3] = __byte_perm(lb, hb, 0x7362);
}

// s + w.lo * x.lo, then + w.hi * x.hi: bf16 operands, exact products, fp32 accumulation.
__device__ __forceinline__ float fma2_bf16(uint32_t w, uint32_t x, float s) {
    asm("{ .reg .b16 wl, wh, xl, xh;\n"
        "  mov.b32 {wl, wh}, %1;\n"
        "  mov.b32 {xl, xh}, %2;\n"
        "  fma.rn.f32.bf16 %0, wl, xl, %0;\n"
        "  fma.rn.f32.bf16 %0, wh, xh, %0;\n}"
        : "+f"(s)
        : "r"(w), "r"(x));
    return s;
}

template <int Q>
__device__ __forceinline__ float cb3_quarter_bf16(const Cb3Levels& l, const uint32_t* g, const uint32_t* x, float s) {
    uint32_t e[4];
    cb3_pairs8(l, cb3_nibbles<Q>(g), e);
#pragma unroll
    for (int i = 0; i < 4; ++i) s = fma2_bf16(e[i], x[4 * Q + i], s);
    return s;
}

// One group (index words g[3]) against 32 bf16 activations (16 pairs x[]), elements in order.
__device__ __forceinline__ float cb3_dot_bf16(const Cb3Levels& l, const uint32_t* g, const uint32_t* x, float s) {
    s = cb3_quarter_bf16<0>(l, g, x, s);
    s = cb3_quarter_bf16<1>(l, g, x, s);
    s = cb3_quarter_bf16<2>(l, g, x, s);
    return cb3_quarter_bf16<3>(l, g, x, s);
}

__device__ __forceinline__ uint32_t ldg_nc_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

struct Cb3Args {
    int T, d, f, k, num_slots;
    int t;                      // token of the gate/up launch
    const uint16_t* x;
    const int32_t* slot;        // [T, k]
    const float* w;             // [T, k]
    const uint8_t* arena;
    int64_t slot_bytes;
    Cb3Layout C;
    uint16_t* h;                // [T*k, f] bf16
    float* z;                   // [T*k, d]: row t*k + j is pair (t, j)
    const int32_t* row_dst;     // rows output instead (null: z, then the combine into y):
    float* rows_out;            // pair (t, j) into row row_dst[t*k + j], skipped when < 0
    uint16_t* y;                // [T, d]
    int32_t* status;
};

// Gate/up + SwiGLU for token a.t: items are (j, i) -- output i of the token's pair j; the warp
// decodes gate row i and up row i of the pair's slot.  The token sits in shared memory as bf16,
// 32-element groups 80 bytes apart (64 bytes + 16 of padding: conflict-free 16-byte reads
// when consecutive lanes read consecutive groups).
template <int GL>
__global__ void __launch_bounds__(128) cb3_gateup_kernel(Cb3Args a) {
    extern __shared__ uint4 xs4[];                        // [nc][5]: 4 data + 1 pad
    const int tid = threadIdx.x, lane = tid & 31;
    const int d = a.d, f = a.f, k = a.k, nc = d / 32;
    const uint4* xg = reinterpret_cast<const uint4*>(a.x + (size_t)a.t * d);
    for (int v = tid; v < nc * 4; v += blockDim.x) xs4[(v >> 2) * 5 + (v & 3)] = __ldg(xg + v);
    __syncthreads();
    const int gw = (blockIdx.x * blockDim.x + tid) >> 5, nw = (gridDim.x * blockDim.x) >> 5;
    for (int it = gw; it < k * f; it += nw) {
        const int j = it / f, i = it % f, pair = a.t * k + j;
        const int s = a.slot[pair];
        if (s < 0 || s >= a.num_slots) {
            if (s >= a.num_slots && i == 0 && lane == 0) atomicOr(a.status, MOE_STATUS_BAD_SLOT);
            continue;
        }
        const uint8_t* base = a.arena + (int64_t)s * a.slot_bytes;
        const uint4 lvmine = lane < 2 ? __ldg(reinterpret_cast<const uint4*>(base + 16 * (int64_t)(lane ? f + i : i)))
                                      : make_uint4(0, 0, 0, 0);
        const uint32_t* pg = reinterpret_cast<const uint32_t*>(base + a.C.gate + (int64_t)i * (3 * d / 8));
        const uint32_t* pu = reinterpret_cast<const uint32_t*>(base + a.C.up + (int64_t)i * (3 * d / 8));
        uint32_t wg[GL][3], wu[GL][3];
#pragma unroll
        for (int g = 0; g < GL; ++g) {
            const int c = lane + 32 * g;
            if (c < nc) {
#pragma unroll
                for (int q = 0; q < 3; ++q) { wg[g][q] = ldg_nc_u32(pg + q * nc + c); wu[g][q] = ldg_nc_u32(pu + q * nc + c); }
            }
        }
        const Cb3Levels lg = cb3_levels_from(lvmine, 0), lu = cb3_levels_from(lvmine, 1);
        float accg = 0.f, accu = 0.f;
#pragma unroll
        for (int g = 0; g < GL; ++g) {
            const int c = lane + 32 * g;
            if (c < nc) {
                uint32_t xr[16];
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint4 q = xs4[c * 5 + v];
                    xr[4 * v] = q.x; xr[4 * v + 1] = q.y; xr[4 * v + 2] = q.z; xr[4 * v + 3] = q.w;
                }
                accg = cb3_dot_bf16(lg, wg[g], xr, accg);
                accu = cb3_dot_bf16(lu, wu[g], xr, accu);
            }
        }
        const float gs = warp_sum(accg), us = warp_sum(accu);
        if (lane == 0) a.h[(size_t)pair * f + i] = f32_to_bf16(gs / (1.0f + expf(-gs)) * us);
    }
}

// Down: for each token the block stages the token's k vectors h [k][f] (bf16); items are
// (j, 2 output rows) and write z rows of the pair.  Lane l owns quarters l + 32m (m < QL,
// QL = f/256); its quarter position Q = l % 4 is the same in every group.
template <int QL>
__global__ void __launch_bounds__(256) cb3_down_kernel(Cb3Args a) {
    extern __shared__ uint4 hs4[];                        // [k][f/8]: 8 bf16 per entry
    const int tid = threadIdx.x, lane = tid & 31;
    const int d = a.d, f = a.f, k = a.k, nc = f / 32;
    const int gw = (blockIdx.x * blockDim.x + tid) >> 5, nw = (gridDim.x * blockDim.x) >> 5;
    const int nb = d / kCb3DnRows;
    const int Q = lane & 3;
    const int wsel = (Q >> 1) * nc;                       // A (quarters 0, 1) or B (2, 3)
    const uint32_t ash = 2u * (Q & 1), zrot = Q == 0 ? 0u : Q == 1 ? 31u : Q == 2 ? 2u : 1u;
    for (int t = 0; t < a.T; ++t) {
        __syncthreads();
        // stage the token's h rows with asynchronous 16-byte copies (all in flight at once)
        for (int e = tid; e < k * (f / 8); e += blockDim.x) {
            const int j = e / (f / 8), i = (e % (f / 8)) * 8, pair = t * k + j;
            const int s = a.slot[pair];
            uint4* dst = hs4 + e;
            if (s >= 0 && s < a.num_slots) {
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(a.h + (size_t)pair * f + i)
                             : "memory");
            } else {
                *dst = make_uint4(0, 0, 0, 0);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        // the first item's index words are requested before the wait for h, so the two
        // latencies overlap; every thread passes the barrier once per token
        bool staged = false;
        for (int it = gw;; it += nw) {
            const bool have = it < k * nb;
            const int j = have ? it / nb : 0, r0 = have ? (it % nb) * kCb3DnRows : 0, pair = t * k + j;
            const int s = have ? a.slot[pair] : -1;
            const bool valid = s >= 0 && s < a.num_slots;
            const uint8_t* base = a.arena + (int64_t)(valid ? s : 0) * a.slot_bytes;
            uint4 lvmine = make_uint4(0, 0, 0, 0);
            uint32_t wab[kCb3DnRows][QL], wz[kCb3DnRows][QL];
            if (valid) {
                if (lane < kCb3DnRows) lvmine = __ldg(reinterpret_cast<const uint4*>(base + 16 * (int64_t)(2 * f + r0 + lane)));
#pragma unroll
                for (int r = 0; r < kCb3DnRows; ++r) {
                    const uint32_t* p = reinterpret_cast<const uint32_t*>(base + a.C.down + (int64_t)(r0 + r) * (3 * f / 8));
#pragma unroll
                    for (int m = 0; m < QL; ++m) {
                        const int c = (lane + 32 * m) >> 2;
                        wab[r][m] = ldg_nc_u32(p + wsel + c);
                        wz[r][m] = ldg_nc_u32(p + 2 * nc + c);
                    }
                }
            }
            if (!staged) {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
                __syncthreads();
                staged = true;
            }
            if (!have) break;
            if (!valid) continue;
            const int zrow = a.row_dst ? a.row_dst[pair] : pair;
            if (zrow < 0) continue;
            float* zr = (a.row_dst ? a.rows_out : a.z) + (size_t)zrow * d;
            // quarter (c, Q) of h_j: 16 bytes at entry 4c + Q; 8 consecutive lanes read 128
            // consecutive bytes (no bank conflict)
            const uint4* hj = hs4 + (size_t)j * (f / 8) + Q;
            Cb3Levels l[kCb3DnRows];
            float acc[kCb3DnRows];
#pragma unroll
            for (int r = 0; r < kCb3DnRows; ++r) { l[r] = cb3_levels_from(lvmine, r); acc[r] = 0.f; }
#pragma unroll
            for (int m = 0; m < QL; ++m) {
                const int c = (lane + 32 * m) >> 2;
                const uint4 hq = hj[4 * c];
#pragma unroll
                for (int r = 0; r < kCb3DnRows; ++r) {
                    const uint32_t N =
                        ((wab[r][m] >> ash) & 0x33333333u) | (__funnelshift_l(wz[r][m], wz[r][m], zrot) & 0x44444444u);
                    uint32_t e[4];
                    cb3_pairs8(l[r], N, e);
                    float v = acc[r];
                    v = fma2_bf16(e[0], hq.x, v);
                    v = fma2_bf16(e[1], hq.y, v);
                    v = fma2_bf16(e[2], hq.z, v);
                    v = fma2_bf16(e[3], hq.w, v);
                    acc[r] = v;
                }
            }
#pragma unroll
            for (int r = 0; r < kCb3DnRows; ++r) {
                const float v = warp_sum(acc[r]);
                if (lane == 0) zr[r0 + r] = v;
            }
        }
    }
}

// y[t, r] = bf16(sum_j w_j z_j[r]) over the pairs with a valid slot, ascending j.
__global__ void __launch_bounds__(256) cb3_combine_kernel(Cb3Args a) {
    const int d = a.d, k = a.k;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < a.T * d; e += gridDim.x * blockDim.x) {
        const int t = e / d, r = e % d;
        float y = 0.f;
        for (int j = 0; j < k; ++j) {
            const int s = a.slot[t * k + j];
            if (s < 0 || s >= a.num_slots) continue;
            y = fmaf(a.w[t * k + j], __ldcg(a.z + (size_t)(t * k + j) * d + r), y);
        }
        a.y[e] = f32_to_bf16(y);
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

bool cb3_ffn_supported(const moe_dims* m) { return m->d <= 1024 * kCb3MaxGL && m->f <= 256 * kCb3MaxQL; }

template <int GL>
static void launch_gateup_gl(const Cb3Args& a, int blocks, cudaStream_t st) {
    cb3_gateup_kernel<GL><<<blocks, 128, (size_t)(a.d / 32) * 80, st>>>(a);
}

template <int GL>
static int launch_down_gl(const Cb3Args& a, size_t smem, int blocks, cudaStream_t st) {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(cb3_down_kernel<GL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    cb3_down_kernel<GL><<<blocks, 256, smem, st>>>(a);
    return MOE_OK;
}

int launch_cb3_ffn(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                   const float* w, uint16_t* y, int32_t* status, char* ws, const WsLayout& L, cudaStream_t st,
                   int num_sms, const int32_t* row_dst, float* rows_out) {
    if (T == 0) return MOE_OK;
    Cb3Args a;
    a.row_dst = rows_out ? row_dst : nullptr;
    a.rows_out = rows_out;
    a.T = T; a.d = m->d; a.f = m->f; a.k = m->top_k; a.num_slots = ar->num_slots;
    a.x = x; a.slot = slot; a.w = w;
    a.arena = reinterpret_cast<const uint8_t*>(ar->base);
    a.slot_bytes = ar->slot_bytes;
    a.C = cb3_layout(m->d, m->f);
    a.h = reinterpret_cast<uint16_t*>(ws + L.h);
    a.z = reinterpret_cast<float*>(ws + L.rows);
    a.y = y; a.status = status;
    const int glu = (m->d / 32 + 31) / 32, qld = m->f / 256;
    const int items = m->top_k * m->f;
    const int gblocks = (items / 4 < 8 * num_sms) ? (items + 3) / 4 : 8 * num_sms;
    for (int t = 0; t < T; ++t) {          // one launch per token: the T = 1 kernel, exactly
        a.t = t;
        switch (glu) {
            case 1: launch_gateup_gl<1>(a, gblocks, st); break;
            case 2: launch_gateup_gl<2>(a, gblocks, st); break;
            case 3: launch_gateup_gl<3>(a, gblocks, st); break;
            case 4: launch_gateup_gl<4>(a, gblocks, st); break;
            case 5: launch_gateup_gl<5>(a, gblocks, st); break;
            case 6: launch_gateup_gl<6>(a, gblocks, st); break;
            case 7: launch_gateup_gl<7>(a, gblocks, st); break;
            default: launch_gateup_gl<8>(a, gblocks, st); break;
        }
        note_launch(1);
    }
    const size_t smem = (size_t)m->top_k * m->f * 2;
    const int dn_items = m->top_k * (m->d / kCb3DnRows);
    const int dblocks = (dn_items / 8 < 2 * num_sms) ? (dn_items + 7) / 8 : 2 * num_sms;
    int rc;
    switch (qld) {
        case 1: rc = launch_down_gl<1>(a, smem, dblocks, st); break;
        case 2: rc = launch_down_gl<2>(a, smem, dblocks, st); break;
        case 3: rc = launch_down_gl<3>(a, smem, dblocks, st); break;
        case 4: rc = launch_down_gl<4>(a, smem, dblocks, st); break;
        case 5: rc = launch_down_gl<5>(a, smem, dblocks, st); break;
        case 6: rc = launch_down_gl<6>(a, smem, dblocks, st); break;
        case 7: rc = launch_down_gl<7>(a, smem, dblocks, st); break;
        case 8: rc = launch_down_gl<8>(a, smem, dblocks, st); break;
        case 9: rc = launch_down_gl<9>(a, smem, dblocks, st); break;
        default: return MOE_ERR_DIMS;
    }
    if (rc) return rc;
    note_launch(1);
    if (rows_out) return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;   // the caller combines
    cb3_combine_kernel<<<(T * m->d + 255) / 256 < 2 * num_sms ? (T * m->d + 255) / 256 : 2 * num_sms, 256, 0, st>>>(a);
    note_launch(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

}  // namespace fp4moe
