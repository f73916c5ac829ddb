// moe_internal.cuh -- shared definitions of the routed-expert FP4 MoE library (sm_103a).
//
// Arena slot layout (private to this library; moe_pack_expert is its only writer).  A slot
// holds two matrices:
//   gate/up: 2f rows, K = d; row 2i is gate row i and row 2i+1 is up row i
//   down:    d rows, K = f
// Each matrix is stored as tiles of 128 rows x 256 K elements, tile (rt, kb) at index
// rt * (K/256) + kb, codes and scales in separate regions:
//   codes  16,384 bytes per tile.  Byte c (0..127) of tile row r sits at
//          r*128 + ((c/16) ^ (r%8))*16 + c%16 -- the SWIZZLE_128B arrangement, so one
//          contiguous copy lands a tile in shared memory ready for the tensor cores.
//   scales 1,024 bytes per tile: two 512-byte tensor-memory scale atoms.  Scale block j
//          (0..7) of tile row r sits at (j/4)*512 + (r%32)*16 + (r/32)*4 + j%4.
// Codes keep the checkpoint's e2m1 nibble order (element 2i in the low nibble) and scales
// are UE8M0 bytes, one per 32 consecutive K elements; only their placement changes.
// Region order: gate/up codes [0, f*d), gate/up scales (f*d/16 bytes), down codes (d*f/2),
// down scales (d*f/32); 18,800,640 bytes in all at d=5120, f=2304.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/fp4moe.h"

namespace fp4moe {

constexpr int kDecodeMaxT = 16;     // tokens handled by the decode regime
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kChunk = 32;          // K elements per UE8M0 scale = 16 code bytes
constexpr int kTileRows = 128;      // rows per arena tile
constexpr int kTileK = 256;         // K elements per arena tile
constexpr int kTileCodeBytes = 16384;
constexpr int kTileScaleBytes = 1024;
constexpr int kTileBytes = kTileCodeBytes + kTileScaleBytes;   // a tile: its codes, then its scale atoms

// A slot holds two matrices, gate/up (2f rows interleaved gate/up, K = d) and then down
// (d rows, K = f), each as tiles of 128 rows x 256 K elements in (row tile, K tile) order.
// A tile is 16 KB of codes (pre-swizzled for SWIZZLE_128B) followed by its 1 KB of scale
// atoms, so one contiguous copy brings a tile, or a run of tiles along K, with its scales.
struct SlotLayout {
    int64_t gu, dn, bytes;   // matrix offsets inside the slot, slot size
};

__host__ __device__ inline SlotLayout slot_layout(int d, int f) {
    SlotLayout L;
    const int64_t fd = (int64_t)f * d;
    L.gu = 0;
    L.dn = (fd / 16384) * kTileBytes;                  // (2f/128) x (d/256) tiles
    const int64_t end = L.dn + (fd / 32768) * kTileBytes;   // (d/128) x (f/256) tiles
    L.bytes = (end + 1023) / 1024 * 1024;
    return L;
}

// Offset, from a matrix's start, of 16-byte code chunk `chunk` (K elements 32*chunk..+31) of
// matrix row `row`, for a matrix with reduction length K.
__host__ __device__ inline int64_t code_chunk_off(int row, int chunk, int K) {
    const int64_t tile = (int64_t)(row / kTileRows) * (K / kTileK) + chunk / 8;
    const int r = row % kTileRows;
    return tile * kTileBytes + r * 128 + (((chunk & 7) ^ (r & 7)) << 4);
}

// Offset, from a matrix's start, of the scale byte of K block `kb` (32 elements) of matrix
// row `row`: in the tile's scale atoms (32-row atoms of 16 bytes per row, two atoms per 128
// rows' 8 blocks, the layout tcgen05.cp 32x128b.warpx4 reads).
__host__ __device__ inline int64_t scale_off(int row, int kb, int K) {
    const int64_t tile = (int64_t)(row / kTileRows) * (K / kTileK) + kb / 8;
    const int r = row % kTileRows, j = kb & 7;
    return tile * kTileBytes + kTileCodeBytes + (j >> 2) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (j & 3);
}

inline bool dims_ok(const moe_dims* m) {
    return m && m->d >= 256 && m->f >= 256 && m->d % 256 == 0 && m->f % 256 == 0 &&
           m->num_experts >= 1 && m->num_experts <= kMaxExperts && m->top_k >= 1 &&
           m->top_k <= kMaxTopK && m->top_k <= m->num_experts && m->d <= 65536 && m->f <= 65536;
}

// Counters inside the counter section (zeroed by moe_workspace_init; every user leaves them
// zero again): the tensor-core FFN kernel's work list, x jobs and x-ready, exit ticket, per-key
// readiness (256 decode keys) and y counts per 32 output features (d/32 <= 2048); the streaming
// decode kernel's x jobs, x-ready and exit ticket; the wait limit (kCtrWaitLimit: 0 = the
// default kSpinLimit polls, else the number of polls after which a wait on another CTA's
// progress gives up -- set only by moe_workspace_set_wait_limit); then the streaming kernel's
// h readiness per key (gate/up tiles whose h is written).
enum { kCtrRoute = 0, kCtrFfnWork = 64, kCtrFfnXReady = 65, kCtrFfnExit = 66, kCtrFfnXJob = 67,
       kCtrStrXJob = 69, kCtrStrXReady = 70, kCtrStrExit = 71, kCtrWaitLimit = 72,
       kCtrFfnReady = 128, kCtrFfnY = 384, kCounterWords = 2432 };
constexpr int kStreamMaxKeys = kDecodeMaxT * kMaxTopK;   // keys of a decode call: at most one per pair
inline size_t stream_hcnt_off(const moe_dims*) { return kCounterWords; }
constexpr int kTcDecodeMaxKeys = 128;   // pairs (T*k) of a decode call on the tensor cores at most
inline size_t counter_words(const moe_dims* m) { return stream_hcnt_off(m) + kStreamMaxKeys; }

// Prefill activation tiles: kPrefillNT permuted rows each (tensor-core path).  The plan of a
// prefill call (written by plan_kernel) describes the expert groups and their tiles:
//   int32 [0] n_active, [1] tiles, [2, 2+E) expert of group g, [2+E, 2+2E) first tile of g,
//   int4  grec[E] at plan_grec_off(E): {first row, end row, arena slot, first tile} of g,
//   int32 tile_group[max_tiles] at plan_tile_group_off(E): the group of each tile,
//   int32 pair_row[n] at plan_pair_off(E, max_tiles): the tile row of pair t*k + j
//         (tile * tile_rows + row), -1 for a pair that has no row.
constexpr int kPrefillNT = 64;
inline size_t act_tiles(const moe_dims* m, int T) {
    const size_t n = (size_t)(T > 0 ? T : 1) * m->top_k;
    const size_t t = (n + kPrefillNT - 1) / kPrefillNT + (n < (size_t)m->num_experts ? n : (size_t)m->num_experts);
    return t > 1 ? t : 1;
}
__host__ __device__ inline int plan_grec_off(int E) { return (2 + 2 * E + 3) / 4 * 4; }
__host__ __device__ inline int plan_tile_group_off(int E) { return plan_grec_off(E) + 4 * E; }
__host__ __device__ inline int plan_pair_off(int E, int max_tiles) { return plan_tile_group_off(E) + max_tiles; }

// Workspace sections, each 256-byte aligned.  The persistent counters come first so that
// their offset is the same for every token count; the other sections are per call.
struct RouteArgs;   // router launch arguments (route_select.cuh)

struct WsLayout {
    size_t keys;        // float4 [T_max, E] router key records {key, key lo, key hi, score}
    size_t xnorm;       // fp32 [T_max]      ||x_t||_2
    size_t wnorm;       // fp32 [E]          ||W_r[e]||_2
    size_t counter;     // uint32 [64]       completion tickets (zeroed once, self-resetting)
    size_t active;      // prefill group plan (see plan_grec_off / plan_tile_group_off)
    size_t h;           // fp32 [T_max*k, f] SwiGLU output per (token, j) pair or permuted row
    size_t rows;        // fp32 [T_max*k, d] per-row expert outputs (prefill with fused combine; cb3 z rows)
    size_t tc;          // tensor-core path: quantised activations, quantised h, per-row outputs
    size_t stream;      // streaming decode path: x and h records, partial sums
    size_t total;
};

inline size_t align256(size_t v) { return (v + 255) / 256 * 256; }

size_t tc_workspace_bytes(const moe_dims* m, int T);   // mxf4_gemm.cu
size_t stream_workspace_bytes(const moe_dims* m, int T);   // ffn_stream.cu

// Adds n to the count of kernels this library has enqueued (abi.cu).
void note_launch(int n);

inline WsLayout ws_layout(const moe_dims* m, int T_max) {
    WsLayout w;
    size_t o = 0;
    size_t T = (size_t)(T_max > 0 ? T_max : 1), E = (size_t)m->num_experts, k = (size_t)m->top_k;
    w.counter = o; o = align256(o + 4 * counter_words(m));   // first: its offset must not depend on T
    w.keys = o;    o = align256(o + 16 * T * E);
    w.xnorm = o;   o = align256(o + 4 * T);
    w.wnorm = o;   o = align256(o + 4 * E);
    w.active = o;  o = align256(o + 4 * ((size_t)plan_tile_group_off((int)E) + act_tiles(m, (int)T) + T * k));
    w.h = o;       o = align256(o + 4 * T * k * (size_t)m->f);
    w.rows = o;    o = align256(o + 4 * T * k * (size_t)m->d);
    w.tc = o;      o = align256(o + tc_workspace_bytes(m, (int)T));
    w.stream = o;  o = align256(o + stream_workspace_bytes(m, T_max > 0 ? T_max : 1));
    w.total = o;
    return w;
}


// ---------------------------------------------------------------------------- device helpers

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// bf16 from fp32, round to nearest even (NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16(float v) {
    uint32_t u = __float_as_uint(v);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

// 2^(b-127) for a UE8M0 byte b < 255 (b = 0 gives the fp32 subnormal 2^-127).
__device__ __forceinline__ float ue8m0_to_f32(uint32_t b) {
    return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

// e2m1 code in nibble position i of w, as an fp32 bit pattern equal to code * 2^-126:
// the 3 magnitude bits (2 exponent, 1 mantissa) land in fp32 exponent bits 23-24 and
// mantissa bit 22, so exponent 0 codes become fp32 subnormals of the same relative value.
template <int I>
__device__ __forceinline__ float e2m1_scaled(uint32_t w) {
    uint32_t mag = (I <= 5) ? (w << (22 - 4 * I)) : (w >> (4 * I - 22));
    uint32_t sgn = (I <= 7) ? (w << (28 - 4 * I)) : 0u;
    return __uint_as_float((mag & 0x01C00000u) | (sgn & 0x80000000u));
}

// Programmatic dependent launch: a kernel launched with launch_pdl may start while the
// previous kernel in the stream runs; pdl_wait() returns once that kernel has completed and
// its memory is visible (immediately for a kernel launched the ordinary way), and
// pdl_trigger() lets the next such kernel start early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// mbarrier and bulk-copy wrappers (PTX).  Every wait is bounded by kSpinLimit polls.
constexpr unsigned kSpinLimit = 1u << 25;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(done)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return done != 0;
}
// Non-blocking probe (test_wait never suspends the thread; try_wait may, for a while).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(done)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return done != 0;
}
// Bounded wait: false after kSpinLimit polls or once another warp has aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    for (unsigned i = 0; i < kSpinLimit; ++i) {
        if (mbar_try(bar, parity)) return true;
        if ((i & 1023u) == 1023u && *abort_flag) return false;
    }
    return false;
}
// gpu-scope counter operations

__device__ __forceinline__ int ld_acquire(const int32_t* a) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ int ld_relaxed(const int32_t* a) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
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

// Contiguous global->shared bulk copy completing on an mbarrier (16-byte aligned, size a
// multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
// L2 policies for copies: evict_first for data streamed once per call (expert weights),
// evict_last for small data read by every call (router weights).
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t policy) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar), "l"(policy)
                 : "memory");
}
template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Power-of-two exponent p (as an integer) such that x * 2^p keeps every |x| below 2^64 and
// every code*x product within the fp32 normal range for |x| >= 2^-60 * max|x|.
__device__ __forceinline__ int prescale_exponent(float amax) {
    int e = 0;
    if (amax > 0.f) e = ((__float_as_uint(amax) >> 23) & 0xFF) - 127;   // floor(log2 amax)
    int p = 100 - (e > 0 ? e : 0);                                        // amax * 2^p < 2^101
    if (p > 100) p = 100;
    return p;
}

// 2^p as float for -126 <= p <= 127.
__device__ __forceinline__ float exp2i(int p) { return __uint_as_float((uint32_t)(p + 127) << 23); }

}  // namespace fp4moe
