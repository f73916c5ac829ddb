// ffn_decode.cu -- decode-regime expert FFN (T <= 16 tokens): CUDA-core kernels that stream
// each selected expert's FP4 rows once and dequantise in registers.
//
//   kernel 1  h[t,j,i] = silu(g) * u,  g = W_gate[slot_tj, i] . x_t,  u = W_up[slot_tj, i] . x_t
//   kernel 2  y[t,r]   = bf16( sum_j w_tj * (W_down[slot_tj, r] . h[t,j]) ),  j ascending
// Single-token decode is a byte-movement problem: every weight byte is read once per call
// (shared by every token routed to the same slot), from HBM straight into registers with
// 16-byte non-coherent loads; the fixed-order combine is fused into kernel 2
// ("Start the expert reads before the GPU is done", 30 September follow-up: rows written
// once, fixed-order slot sum).
//
// Arithmetic: codes become code * 2^-126 fp32 patterns by bit moves (see e2m1_scaled); the
// activation operand is staged in shared memory scaled by an exact power of two 2^p, so
// every product code * act is exact in fp32 and the sum is an fp32 FMA chain; each
// 32-element block sum is multiplied by 2^(b - 1 - p) (the UE8M0 scale and the undoing of
// both power-of-two factors) before joining the running fp32 total.
#include "moe_internal.cuh"

namespace fp4moe {

constexpr int kXT = 8;   // tokens staged per pass of kernel 1

// Shared-memory rows are padded by 4 floats after every 32 (one 16-byte code chunk's worth
// of activations): a lane's 32-float chunk starts at 36c, so the 16-byte reads of 8
// consecutive chunks fall in 8 distinct groups of 4 banks.
__host__ __device__ constexpr int padded(int n) { return n + n / 8; }
__device__ __forceinline__ int pad_idx(int i) { return i + 4 * (i >> 5); }

struct DecodeArgs {
    int T, d, f, k, num_slots;
    int t0, tn;                 // token pass [t0, t0 + tn) of kernel 1
    const uint16_t* x;
    const int32_t* slot;        // [T, k]
    const float* w;             // [T, k]
    const uint8_t* arena;
    int64_t slot_bytes;
    SlotLayout L;
    float* h;                   // [T*k, f]
    uint16_t* y;                // [T, d]
    int32_t* status;
};

// 2^e as an fp32 for any integer e (exact from 2^-149 to 2^127; 0 below, +inf above).
__device__ __forceinline__ float pow2f(int e) {
    if (e > 127) return __int_as_float(0x7f800000);
    if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
    if (e >= -149) return __uint_as_float(1u << (e + 149));
    return 0.0f;
}

// Dot of 32 codes (one 16-byte chunk) with 32 staged activations: exact products,
// one FMA chain.
__device__ __forceinline__ float chunk_dot(const uint4 q, const float* __restrict__ a) {
    const float4* a4 = reinterpret_cast<const float4*>(a);
    float s = 0.f;
    uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        float4 p = a4[2 * wi], r = a4[2 * wi + 1];
        uint32_t w = wv[wi];
        s = fmaf(e2m1_scaled<0>(w), p.x, s);
        s = fmaf(e2m1_scaled<1>(w), p.y, s);
        s = fmaf(e2m1_scaled<2>(w), p.z, s);
        s = fmaf(e2m1_scaled<3>(w), p.w, s);
        s = fmaf(e2m1_scaled<4>(w), r.x, s);
        s = fmaf(e2m1_scaled<5>(w), r.y, s);
        s = fmaf(e2m1_scaled<6>(w), r.z, s);
        s = fmaf(e2m1_scaled<7>(w), r.w, s);
    }
    return s;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Block-wide max of |v| over a smem-staged row (all threads participate).
__device__ float block_absmax(float v, float* red) {
    v = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float m = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    return m;
}

// ---------------------------------------------------------------------------- kernel 1

// Items are (unique slot u, output i).  A warp loads gate row i and up row i of slot u
// (lane owns chunks lane, lane+32, ...), then reduces for every token of this pass routed
// to u.  Shared memory: staged activations [tn][d] fp32 and the slot/member lists.
template <int XT>
__global__ void __launch_bounds__(256) decode_gateup_kernel(DecodeArgs a) {
    extern __shared__ float xs[];                         // [tn][padded(d)]
    __shared__ int uniq_slot[kXT * kMaxTopK];
    __shared__ int mem_cnt[kXT * kMaxTopK];
    __shared__ int mem_pair[kXT * kMaxTopK][kXT];
    __shared__ int pexp[kXT];
    __shared__ float red[32];
    __shared__ int n_uniq;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, f = a.f, k = a.k, tn = a.tn;
    // unique slots among the pairs of this pass, each with at most kXT member pairs (a slot
    // shared by more pairs -- only possible with a degenerate table -- gets several entries)
    if (tid == 0) {
        int nu = 0;
        int npairs = tn * k;
        for (int q = 0; q < npairs; ++q) {
            int p = a.t0 * k + q;
            int s = a.slot[p];
            if (s < 0) continue;
            if (s >= a.num_slots) { if (blockIdx.x == 0) atomicOr(a.status, MOE_STATUS_BAD_SLOT); continue; }
            int u = 0;
            while (u < nu && !(uniq_slot[u] == s && mem_cnt[u] < XT)) ++u;
            if (u == nu) { uniq_slot[nu] = s; mem_cnt[nu] = 0; ++nu; }
            mem_pair[u][mem_cnt[u]++] = p;
        }
        n_uniq = nu;
    }
    // stage x_t * 2^p_t (exact) for the tokens of this pass
    for (int t = 0; t < tn; ++t) {
        const uint16_t* xt = a.x + (size_t)(a.t0 + t) * d;
        float m = 0.f;
        for (int i = tid; i < d; i += blockDim.x) m = fmaxf(m, fabsf(bf16_to_f32(xt[i])));
        m = block_absmax(m, red);
        int p = prescale_exponent(m);
        if (tid == 0) pexp[t] = p;
        float sc = exp2i(p > 127 ? 127 : p);
        for (int i = tid; i < d; i += blockDim.x) xs[(size_t)t * padded(d) + pad_idx(i)] = bf16_to_f32(xt[i]) * sc;
    }
    __syncthreads();
    const int nu = n_uniq;
    const int nchunk = d / kChunk;
    const int gw = blockIdx.x * (blockDim.x >> 5) + warp, nw = gridDim.x * (blockDim.x >> 5);
    const int items = nu * f;
    for (int it = gw; it < items; it += nw) {
        const int u = it / f, i = it % f;
        const uint8_t* base = a.arena + (int64_t)uniq_slot[u] * a.slot_bytes;
        const uint8_t* cq = base + a.L.gu;   // gate row 2i, up row 2i+1 of the tiled matrix
        const uint8_t* cs = base + a.L.gu;
        float accg[XT], accu[XT];
#pragma unroll
        for (int q = 0; q < XT; ++q) accg[q] = accu[q] = 0.f;
        const int nmem = mem_cnt[u];
        for (int c0 = lane; c0 < nchunk; c0 += 32 * 5) {
            uint4 qg[5], qu[5];
            uint32_t sg[5], su[5];
#pragma unroll
            for (int b = 0; b < 5; ++b) {
                int c = c0 + 32 * b;
                if (c < nchunk) {
                    qg[b] = ldg_stream(cq + code_chunk_off(2 * i, c, d));
                    qu[b] = ldg_stream(cq + code_chunk_off(2 * i + 1, c, d));
                    sg[b] = __ldg(cs + scale_off(2 * i, c, d));
                    su[b] = __ldg(cs + scale_off(2 * i + 1, c, d));
                }
            }
#pragma unroll
            for (int b = 0; b < 5; ++b) {
                int c = c0 + 32 * b;
                if (c >= nchunk) break;
#pragma unroll
                for (int q = 0; q < XT; ++q) {
                    if (q >= nmem) break;
                    int t = mem_pair[u][q] / k - a.t0;
                    const float* xa = xs + (size_t)t * padded(d) + 36 * c;
                    int p = pexp[t];
                    accg[q] = fmaf(chunk_dot(qg[b], xa), pow2f((int)sg[b] - 1 - p), accg[q]);
                    accu[q] = fmaf(chunk_dot(qu[b], xa), pow2f((int)su[b] - 1 - p), accu[q]);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < XT; ++q) {
            if (q >= nmem) break;
            float g = warp_sum(accg[q]), uu = warp_sum(accu[q]);
            if (lane == 0) a.h[(size_t)mem_pair[u][q] * f + i] = silu_mul(g, uu);
        }
    }
}

// ---------------------------------------------------------------------------- kernel 2

// Each warp owns 4 output rows (8 lanes per row; lane owns chunks l8, l8+8, ...).  For each
// token, the k pairs are visited in ascending j and combined in that order.  Shared memory:
// the token's k vectors h * 2^p (exact) [k][f].
__global__ void __launch_bounds__(256) decode_down_kernel(DecodeArgs a) {
    extern __shared__ float hs[];                         // [k][padded(f)]
    __shared__ int pexp[kMaxTopK];
    __shared__ float red[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, f = a.f, k = a.k;
    const int l8 = lane & 7, grp = lane >> 3;
    const int nchunk = f / kChunk;
    const int rows_per_block = (blockDim.x >> 5) * 4;
    const int r = blockIdx.x * rows_per_block + warp * 4 + grp;
    for (int t = 0; t < a.T; ++t) {
        __syncthreads();
        for (int j = 0; j < k; ++j) {
            const int pair = t * k + j;
            const float* hp = a.h + (size_t)pair * f;
            int s = a.slot[pair];
            bool ok = s >= 0 && s < a.num_slots;
            float m = 0.f;
            if (ok)
                for (int i = tid; i < f; i += blockDim.x) m = fmaxf(m, fabsf(__ldcg(hp + i)));
            m = block_absmax(m, red);
            int p = prescale_exponent(m);
            if (tid == 0) pexp[j] = p;
            float sc = exp2i(p > 127 ? 127 : p);
            for (int i = tid; i < f; i += blockDim.x) hs[(size_t)j * padded(f) + pad_idx(i)] = ok ? __ldcg(hp + i) * sc : 0.f;
        }
        __syncthreads();
        if (r < d) {
            float y = 0.f;
            for (int j = 0; j < k; ++j) {
                const int pair = t * k + j;
                int s = a.slot[pair];
                if (s < 0 || s >= a.num_slots) continue;   // group-uniform: same pair for the warp
                const uint8_t* base = a.arena + (int64_t)s * a.slot_bytes;
                const uint8_t* dq = base + a.L.dn;
                const uint8_t* ds = base + a.L.dn;
                const int p = pexp[j];
                float acc = 0.f;
                for (int c0 = l8; c0 < nchunk; c0 += 8 * 9) {
                    uint4 qv[9];
                    uint32_t sb[9];
#pragma unroll
                    for (int b = 0; b < 9; ++b) {
                        int c = c0 + 8 * b;
                        if (c < nchunk) { qv[b] = ldg_stream(dq + code_chunk_off(r, c, f)); sb[b] = __ldg(ds + scale_off(r, c, f)); }
                    }
#pragma unroll
                    for (int b = 0; b < 9; ++b) {
                        int c = c0 + 8 * b;
                        if (c >= nchunk) break;
                        acc = fmaf(chunk_dot(qv[b], hs + (size_t)j * padded(f) + 36 * c), pow2f((int)sb[b] - 1 - p), acc);
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
}

// ---------------------------------------------------------------------------- host side

template <int XT>
static int launch_gateup(const DecodeArgs& a, size_t smem, int blocks, cudaStream_t st) {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(decode_gateup_kernel<XT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    decode_gateup_kernel<XT><<<blocks, 256, smem, st>>>(a);
    note_launch(1);
    return MOE_OK;
}

int launch_decode_ffn(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x,
                      const int32_t* slot, const float* w, uint16_t* y, int32_t* status, char* ws,
                      const WsLayout& L, cudaStream_t st, int num_sms) {
    DecodeArgs a;
    a.T = T; a.d = m->d; a.f = m->f; a.k = m->top_k; a.num_slots = ar->num_slots;
    a.x = x; a.slot = slot; a.w = w;
    a.arena = reinterpret_cast<const uint8_t*>(ar->base);
    a.slot_bytes = ar->slot_bytes;
    a.L = slot_layout(m->d, m->f);
    a.h = reinterpret_cast<float*>(ws + L.h);
    a.y = y; a.status = status;
    if (T == 0) return MOE_OK;
    for (int t0 = 0; t0 < T; t0 += kXT) {
        a.t0 = t0;
        a.tn = (T - t0 < kXT) ? T - t0 : kXT;
        size_t smem = (size_t)a.tn * padded(m->d) * 4;
        int blocks = 2 * num_sms;
        int rc = MOE_OK;
        if (a.tn == 1) rc = launch_gateup<1>(a, smem, blocks, st);
        else if (a.tn == 2) rc = launch_gateup<2>(a, smem, blocks, st);
        else if (a.tn <= 4) rc = launch_gateup<4>(a, smem, blocks, st);
        else rc = launch_gateup<8>(a, smem, blocks, st);
        if (rc) return rc;
    }
    size_t smem2 = (size_t)m->top_k * padded(m->f) * 4;
    if (smem2 > 48 * 1024 &&
        cudaFuncSetAttribute(decode_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    int rows_per_block = 8 * 4;
    decode_down_kernel<<<(m->d + rows_per_block - 1) / rows_per_block, 256, smem2, st>>>(a);
    note_launch(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

}  // namespace fp4moe
