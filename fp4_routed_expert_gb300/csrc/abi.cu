// abi.cu -- the extern "C" entry points declared in include/fp4moe.h: argument checks on the
// host, then kernel launches on the caller's stream.  Nothing here allocates, synchronises
// or reads device memory back.
#include <atomic>
#include <cstdio>

#include "route_select.cuh"

namespace fp4moe {

static std::atomic<unsigned long long> g_kernel_launches{0};
void note_launch(int n) { g_kernel_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

int launch_route(const moe_dims* m, int T, const uint16_t* x, const uint16_t* wr, const float* bias,
                 const int32_t* table, int32_t* ids, float* w, int32_t* slots, int32_t* status,
                 char* ws, const WsLayout& L, cudaStream_t st, int num_sms);
int launch_permute(const moe_dims* m, int T, const int32_t* ids, int32_t* offsets, int32_t* row_src,
                   int32_t* row_dst, cudaStream_t st);
int launch_stream_ffn(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                      const float* w, uint16_t* y, int32_t* status, char* ws, const WsLayout& L, cudaStream_t st,
                      int num_sms);
int launch_prefill_ffn(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                       const int32_t* offsets, const int32_t* row_src, float* rows_out, int32_t* status, char* ws,
                       const WsLayout& L, cudaStream_t st, int num_sms);
int launch_combine(const moe_dims* m, int T, const float* rows, const int32_t* row_dst, const float* w,
                   uint16_t* y, cudaStream_t st, int num_sms);
bool tc_supported(const moe_dims* m);
int64_t cb3_slot_bytes(int d, int f);
bool cb3_ffn_supported(const moe_dims* m);
int launch_pack_cb3(const moe_dims* m, const uint8_t* src_slot, uint8_t* dst_slot, int32_t* status, cudaStream_t st);
int launch_cb3_ffn(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                   const float* w, uint16_t* y, int32_t* status, char* ws, const WsLayout& L, cudaStream_t st,
                   int num_sms, const int32_t* row_dst = nullptr, float* rows_out = nullptr);
bool tc_decode_supported(const moe_dims* m, int T);
int launch_tc_decode(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                     const float* w, uint16_t* y, int32_t* status, char* ws, const WsLayout& L, cudaStream_t st,
                     int num_sms, const RouteArgs* ra = nullptr, int route_blocks = 0);
int launch_residency_bias(const moe_dims* m, const int32_t* expert_to_slot, const int32_t* resident_expert,
                          int num_slots, const float* bias, float lambda, float* bias_out, cudaStream_t st);
int launch_split_waves(const moe_dims* m, int T, const int32_t* ids, const int32_t* slot, const int32_t* resident_expert,
                       int num_slots, int32_t* wave1, int32_t* wave2, int32_t* missing, int32_t* n_missing,
                       cudaStream_t st);
int launch_gather_experts(const moe_arena* ar, const uint8_t* store, int n_store, const int32_t* missing,
                          const int32_t* n_missing, const int32_t* expert_to_slot, int32_t* resident_expert,
                          int32_t* status, cudaStream_t st, int num_sms);
int launch_residual_rmsnorm(int T, int d, const uint16_t* x, const uint16_t* y, float eps, uint16_t* out, cudaStream_t st);
int launch_tc_prefill(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                      const int32_t* offsets, const int32_t* row_src, float* rows_out, int32_t* status, char* ws,
                      const WsLayout& L, cudaStream_t st, int num_sms);

// Canonical rows -> arena tiles.  With `up` set, matrix row 2i takes row i of `gate` and
// row 2i+1 takes row i of `up` (the gate/up interleave); otherwise matrix row R is row R of
// `gate`.  One thread per 16-byte code chunk.
__global__ void pack_codes_kernel(const uint8_t* __restrict__ gate, const uint8_t* __restrict__ up,
                                  uint8_t* __restrict__ dst, int rows, int K) {
    const int chunks = K / 32;
    const long total = (long)rows * chunks;
    for (long idx = blockIdx.x * (long)blockDim.x + threadIdx.x; idx < total; idx += (long)gridDim.x * blockDim.x) {
        const int R = (int)(idx / chunks), c = (int)(idx % chunks);
        const uint8_t* src = up ? ((R & 1) ? up : gate) + (size_t)(R >> 1) * (K / 2) : gate + (size_t)R * (K / 2);
        *reinterpret_cast<uint4*>(dst + code_chunk_off(R, c, K)) = *reinterpret_cast<const uint4*>(src + 16 * c);
    }
}

// Canonical scale rows [rows][K/32] -> arena scale atoms (same row mapping as the codes).
__global__ void pack_scales_kernel(const uint8_t* __restrict__ gate, const uint8_t* __restrict__ up,
                                   uint8_t* __restrict__ dst, int rows, int K) {
    const int nb = K / 32;
    const long total = (long)rows * nb;
    for (long idx = blockIdx.x * (long)blockDim.x + threadIdx.x; idx < total; idx += (long)gridDim.x * blockDim.x) {
        const int R = (int)(idx / nb), kb = (int)(idx % nb);
        const uint8_t* src = up ? ((R & 1) ? up : gate) + (size_t)(R >> 1) * nb : gate + (size_t)R * nb;
        dst[scale_off(R, kb, K)] = src[kb];
    }
}

static int num_sms_of_current_device() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
    if (dev < 64 && cache[dev]) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    if (dev < 64) cache[dev] = n;
    return n;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int check_ws(const moe_dims* m, int T, void* ws, size_t ws_bytes, WsLayout* out) {
    if (!ws) return MOE_ERR_NULL;
    if (!aligned16(ws)) return MOE_ERR_ALIGN;
    WsLayout L = ws_layout(m, T);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    *out = L;
    return MOE_OK;
}

__global__ void set_word_kernel(int32_t* p, int32_t v) { *p = v; }

static int check_arena(const moe_dims* m, const moe_arena* ar, bool cb3 = false) {
    if (!ar || !ar->base) return MOE_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(ar->base) & 1023u) != 0) return MOE_ERR_ARENA;
    const int64_t want = cb3 ? cb3_slot_bytes(m->d, m->f) : slot_layout(m->d, m->f).bytes;
    if (ar->slot_bytes != want || ar->num_slots <= 0) return MOE_ERR_ARENA;
    return MOE_OK;
}

}  // namespace fp4moe

using namespace fp4moe;

extern "C" {

int64_t moe_slot_bytes(const moe_dims* dims) {
    if (!dims_ok(dims)) return -1;
    return slot_layout(dims->d, dims->f).bytes;
}

size_t moe_workspace_bytes(const moe_dims* dims, int32_t T_max) {
    if (!dims_ok(dims) || T_max < 0) return 0;
    return ws_layout(dims, T_max).total;
}

int moe_workspace_set_wait_limit(const moe_dims* dims, void* ws, size_t ws_bytes, int32_t polls, void* stream) {
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    if (polls < 0) return MOE_ERR_DIMS;
    WsLayout L;
    int rc = check_ws(dims, 0, ws, ws_bytes, &L);
    if (rc) return rc;
    set_word_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(reinterpret_cast<int32_t*>(static_cast<char*>(ws) + L.counter) +
                                                            kCtrWaitLimit, polls);
    note_launch(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

int moe_workspace_init(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream) {
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    WsLayout L;
    int rc = check_ws(dims, 0, ws, ws_bytes, &L);
    if (rc) return rc;
    cudaError_t e = cudaMemsetAsync(static_cast<char*>(ws) + L.counter, 0, 4 * counter_words(dims), (cudaStream_t)stream);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

int moe_pack_expert(const moe_dims* dims, const uint8_t* gate_q, const uint8_t* gate_s, const uint8_t* up_q,
                    const uint8_t* up_s, const uint8_t* down_q, const uint8_t* down_s, const moe_arena* arena,
                    int32_t slot, void* stream) {
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    if (!gate_q || !gate_s || !up_q || !up_s || !down_q || !down_s) return MOE_ERR_NULL;
    int rc = check_arena(dims, arena);
    if (rc) return rc;
    if (slot < 0 || slot >= arena->num_slots) return MOE_ERR_ARENA;
    if (!aligned16(gate_q) || !aligned16(up_q) || !aligned16(down_q)) return MOE_ERR_ALIGN;
    cudaStream_t st = (cudaStream_t)stream;
    const int d = dims->d, f = dims->f;
    SlotLayout L = slot_layout(d, f);
    uint8_t* base = static_cast<uint8_t*>(arena->base) + (int64_t)slot * arena->slot_bytes;
    int sms = num_sms_of_current_device();
    pack_codes_kernel<<<2 * sms, 256, 0, st>>>(gate_q, up_q, base + L.gu, 2 * f, d);
    pack_scales_kernel<<<sms, 256, 0, st>>>(gate_s, up_s, base + L.gu, 2 * f, d);
    pack_codes_kernel<<<2 * sms, 256, 0, st>>>(down_q, nullptr, base + L.dn, d, f);
    pack_scales_kernel<<<sms, 256, 0, st>>>(down_s, nullptr, base + L.dn, d, f);
    note_launch(4);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_LAUNCH;
    return MOE_OK;
}

int moe_route_topk(const moe_dims* dims, int32_t T, const uint16_t* x, const uint16_t* w_router,
                   const float* score_bias, const int32_t* expert_to_slot, int32_t* topk_ids, float* topk_w,
                   int32_t* topk_slot, int32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    if (T < 0) return MOE_ERR_TOKENS;
    if (!x || !w_router || !expert_to_slot || !topk_ids || !topk_w || !topk_slot || !dev_status) return MOE_ERR_NULL;
    if (!aligned16(x) || !aligned16(w_router)) return MOE_ERR_ALIGN;
    WsLayout L;
    int rc = check_ws(dims, T, ws, ws_bytes, &L);
    if (rc) return rc;
    return launch_route(dims, T, x, w_router, score_bias, expert_to_slot, topk_ids, topk_w, topk_slot, dev_status,
                        static_cast<char*>(ws), L, (cudaStream_t)stream, num_sms_of_current_device());
}

int moe_permute(const moe_dims* dims, int32_t T, const int32_t* topk_ids, int32_t* group_offsets, int32_t* row_src,
                int32_t* row_dst, void* ws, size_t ws_bytes, void* stream) {
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    if (T < 0) return MOE_ERR_TOKENS;
    if (!group_offsets || (T > 0 && (!topk_ids || !row_src || !row_dst))) return MOE_ERR_NULL;
    WsLayout L;
    int rc = check_ws(dims, T, ws, ws_bytes, &L);
    if (rc) return rc;
    return launch_permute(dims, T, topk_ids, group_offsets, row_src, row_dst, (cudaStream_t)stream);
}

int moe_expert_ffn_fp4(const moe_dims* dims, const moe_arena* arena, int32_t T, const uint16_t* x,
                       const int32_t* topk_ids, const int32_t* topk_slot, const float* topk_w,
                       const int32_t* group_offsets, const int32_t* row_src, const int32_t* row_dst, int32_t flags,
                       float* rows_out, uint16_t* y, int32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    if (T < 0) return MOE_ERR_TOKENS;
    if (flags & ~(MOE_FUSE_COMBINE | MOE_FFN_CUDA_CORES)) return MOE_ERR_FLAGS;
    int rc = check_arena(dims, arena);
    if (rc) return rc;
    if (!x || !topk_ids || !topk_slot || !topk_w || !dev_status) return MOE_ERR_NULL;
    if (!aligned16(x)) return MOE_ERR_ALIGN;
    const bool fused = (flags & MOE_FUSE_COMBINE) != 0;
    const bool cuda_cores = (flags & MOE_FFN_CUDA_CORES) != 0;
    if (fused && !y) return MOE_ERR_NULL;
    if (!fused && !rows_out) return MOE_ERR_NULL;
    WsLayout L;
    rc = check_ws(dims, T, ws, ws_bytes, &L);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    char* w = static_cast<char*>(ws);
    int sms = num_sms_of_current_device();
    if (T <= kDecodeMaxT && fused) {
        if (!cuda_cores && tc_decode_supported(dims, T))
            return launch_tc_decode(dims, arena, T, x, topk_slot, topk_w, y, dev_status, w, L, st, sms);
        return launch_stream_ffn(dims, arena, T, x, topk_slot, topk_w, y, dev_status, w, L, st, sms);
    }
    if (!group_offsets || !row_src || (fused && !row_dst)) return MOE_ERR_NULL;
    if (rows_out && !aligned16(rows_out)) return MOE_ERR_ALIGN;
    // fused requests reach this point only for T > kDecodeMaxT, where the workspace holds rows
    float* rows = fused ? reinterpret_cast<float*>(w + L.rows) : rows_out;
    if (!cuda_cores && tc_supported(dims))
        rc = launch_tc_prefill(dims, arena, T, x, topk_slot, group_offsets, row_src, rows, dev_status, w, L, st, sms);
    else
        rc = launch_prefill_ffn(dims, arena, T, x, topk_slot, group_offsets, row_src, rows, dev_status, w, L, st, sms);
    if (rc || !fused) return rc;
    return launch_combine(dims, T, rows, row_dst, topk_w, y, st, sms);
}

int moe_layer_decode_fp4(const moe_dims* dims, const moe_arena* arena, int32_t T, const uint16_t* x,
                         const uint16_t* w_router, const float* score_bias, const int32_t* expert_to_slot,
                         int32_t* topk_ids, float* topk_w, int32_t* topk_slot, uint16_t* y, int32_t* dev_status,
                         void* ws, size_t ws_bytes, void* stream) {
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    if (T < 0 || T > kDecodeMaxT) return MOE_ERR_TOKENS;
    int rc = check_arena(dims, arena);
    if (rc) return rc;
    if (!x || !w_router || !expert_to_slot || !topk_ids || !topk_w || !topk_slot || !y || !dev_status)
        return MOE_ERR_NULL;
    if (!aligned16(x) || !aligned16(w_router)) return MOE_ERR_ALIGN;
    WsLayout L;
    rc = check_ws(dims, T, ws, ws_bytes, &L);
    if (rc) return rc;
    if (T == 0) return MOE_OK;
    cudaStream_t st = (cudaStream_t)stream;
    char* w = static_cast<char*>(ws);
    const int sms = num_sms_of_current_device();
    const bool tc = tc_decode_supported(dims, T);
    if (tc) {
        // router kernel with its records handed to the expert kernel, which selects
        RouteArgs ra{};
        int blocks = 0;
        rc = launch_route_handoff(dims, T, x, w_router, score_bias, expert_to_slot, topk_ids, topk_w, topk_slot,
                                  dev_status, w, L, st, sms, &ra, &blocks);
        if (rc == MOE_OK)
            return launch_tc_decode(dims, arena, T, x, topk_slot, topk_w, y, dev_status, w, L, st, sms, &ra, blocks);
        if (rc != 1) return rc;
    }
    rc = launch_route(dims, T, x, w_router, score_bias, expert_to_slot, topk_ids, topk_w, topk_slot, dev_status, w,
                      L, st, sms);
    if (rc) return rc;
    if (tc) return launch_tc_decode(dims, arena, T, x, topk_slot, topk_w, y, dev_status, w, L, st, sms);
    return launch_stream_ffn(dims, arena, T, x, topk_slot, topk_w, y, dev_status, w, L, st, sms);
}

int moe_residency_bias(const moe_dims* dims, const float* score_bias, const int32_t* expert_to_slot,
                       const int32_t* resident_expert, int32_t num_slots, float lambda, float* bias_out, void* stream) {
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    if (num_slots <= 0) return MOE_ERR_ARENA;
    if (!(lambda >= 0.0f) || !(lambda < 3.0e38f)) return MOE_ERR_DIMS;   // finite, >= 0 (NaN fails both)
    if (!expert_to_slot || !resident_expert || !bias_out) return MOE_ERR_NULL;
    return launch_residency_bias(dims, expert_to_slot, resident_expert, num_slots, score_bias, lambda, bias_out,
                                 (cudaStream_t)stream);
}

int moe_split_waves(const moe_dims* dims, int32_t T, const int32_t* topk_ids, const int32_t* topk_slot,
                    const int32_t* resident_expert, int32_t num_slots, int32_t* slot_wave1, int32_t* slot_wave2,
                    int32_t* missing, int32_t* n_missing, void* stream) {
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    if (T < 0) return MOE_ERR_TOKENS;
    if (num_slots <= 0) return MOE_ERR_ARENA;
    if (!topk_ids || !topk_slot || !resident_expert || !slot_wave1 || !slot_wave2 || !missing || !n_missing)
        return MOE_ERR_NULL;
    return launch_split_waves(dims, T, topk_ids, topk_slot, resident_expert, num_slots, slot_wave1, slot_wave2, missing,
                              n_missing, (cudaStream_t)stream);
}

int moe_gather_experts(const moe_dims* dims, const moe_arena* arena, const void* store, int32_t n_store,
                       const int32_t* missing, const int32_t* n_missing, const int32_t* expert_to_slot,
                       int32_t* resident_expert, int32_t* dev_status, void* stream) {
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    int rc = check_arena(dims, arena);
    if (rc == MOE_ERR_ARENA) rc = check_arena(dims, arena, true);   // a cb3 arena: images of its format
    if (rc) return rc;
    if (!store || !missing || !n_missing || !expert_to_slot || !resident_expert || !dev_status) return MOE_ERR_NULL;
    if (n_store <= 0) return MOE_ERR_DIMS;
    if (!aligned16(store)) return MOE_ERR_ALIGN;
    return launch_gather_experts(arena, static_cast<const uint8_t*>(store), n_store, missing, n_missing, expert_to_slot,
                                 resident_expert, dev_status, (cudaStream_t)stream, num_sms_of_current_device());
}

int moe_combine(const moe_dims* dims, int32_t T, const float* rows, const int32_t* row_dst, const float* topk_w,
                uint16_t* y, void* stream) {
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    if (T < 0) return MOE_ERR_TOKENS;
    if (T > 0 && (!rows || !row_dst || !topk_w || !y)) return MOE_ERR_NULL;
    if (T > 0 && (!aligned16(rows) || !aligned16(y))) return MOE_ERR_ALIGN;
    return launch_combine(dims, T, rows, row_dst, topk_w, y, (cudaStream_t)stream, num_sms_of_current_device());
}

int64_t moe_cb3_slot_bytes(const moe_dims* dims) {
    if (!dims_ok(dims)) return -1;
    return cb3_slot_bytes(dims->d, dims->f);
}

int moe_pack_cb3(const moe_dims* dims, const moe_arena* fp4_arena, int32_t fp4_slot, const moe_arena* cb3_arena,
                 int32_t cb3_slot, int32_t* dev_status, void* stream) {
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    int rc = check_arena(dims, fp4_arena);
    if (rc) return rc;
    rc = check_arena(dims, cb3_arena, true);
    if (rc) return rc;
    if (!dev_status) return MOE_ERR_NULL;
    if (fp4_slot < 0 || fp4_slot >= fp4_arena->num_slots || cb3_slot < 0 || cb3_slot >= cb3_arena->num_slots)
        return MOE_ERR_ARENA;
    const uint8_t* src = static_cast<const uint8_t*>(fp4_arena->base) + (int64_t)fp4_slot * fp4_arena->slot_bytes;
    uint8_t* dst = static_cast<uint8_t*>(cb3_arena->base) + (int64_t)cb3_slot * cb3_arena->slot_bytes;
    return launch_pack_cb3(dims, src, dst, dev_status, (cudaStream_t)stream);
}

}  // extern "C"

namespace fp4moe {
// The cb3 expert calls in consecutive calls of at most kDecodeMaxT tokens (each the decode-size
// kernels, whose per-token arithmetic does not depend on the other tokens of the call).
static int cb3_in_chunks(const moe_dims* m, const moe_arena* ar, int T, const uint16_t* x, const int32_t* slot,
                         const float* w, uint16_t* y, const int32_t* row_dst, float* rows_out, int32_t* status,
                         char* ws, const WsLayout& L, cudaStream_t st) {
    const int sms = num_sms_of_current_device(), d = m->d, k = m->top_k;
    for (int c0 = 0; c0 < T; c0 += kDecodeMaxT) {
        const int tc = T - c0 < kDecodeMaxT ? T - c0 : kDecodeMaxT;
        const int rc = launch_cb3_ffn(m, ar, tc, x + (size_t)c0 * d, slot + (size_t)c0 * k,
                                      w ? w + (size_t)c0 * k : nullptr, y ? y + (size_t)c0 * d : nullptr, status, ws,
                                      L, st, sms, row_dst ? row_dst + (size_t)c0 * k : nullptr, rows_out);
        if (rc) return rc;
    }
    return MOE_OK;
}
}  // namespace fp4moe

extern "C" {

int moe_expert_ffn_cb3(const moe_dims* dims, const moe_arena* cb3_arena, int32_t T, const uint16_t* x,
                       const int32_t* topk_slot, const float* topk_w, uint16_t* y, int32_t* dev_status, void* ws,
                       size_t ws_bytes, void* stream) {
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    if (!cb3_ffn_supported(dims)) return MOE_ERR_DIMS;
    if (T < 0) return MOE_ERR_TOKENS;
    int rc = check_arena(dims, cb3_arena, true);
    if (rc) return rc;
    if (!x || !topk_slot || !topk_w || !y || !dev_status) return MOE_ERR_NULL;
    if (!aligned16(x)) return MOE_ERR_ALIGN;
    WsLayout L;
    rc = check_ws(dims, T, ws, ws_bytes, &L);
    if (rc) return rc;
    return cb3_in_chunks(dims, cb3_arena, T, x, topk_slot, topk_w, y, nullptr, nullptr, dev_status,
                         static_cast<char*>(ws), L, (cudaStream_t)stream);
}

int moe_expert_ffn_cb3_rows(const moe_dims* dims, const moe_arena* cb3_arena, int32_t T, const uint16_t* x,
                            const int32_t* topk_slot, const int32_t* row_dst, float* rows_out, int32_t* dev_status,
                            void* ws, size_t ws_bytes, void* stream) {
    if (!dims_ok(dims)) return MOE_ERR_DIMS;
    if (!cb3_ffn_supported(dims)) return MOE_ERR_DIMS;
    if (T < 0) return MOE_ERR_TOKENS;
    int rc = check_arena(dims, cb3_arena, true);
    if (rc) return rc;
    if (!x || !topk_slot || !row_dst || !rows_out || !dev_status) return MOE_ERR_NULL;
    if (!aligned16(x)) return MOE_ERR_ALIGN;
    WsLayout L;
    rc = check_ws(dims, T, ws, ws_bytes, &L);
    if (rc) return rc;
    return cb3_in_chunks(dims, cb3_arena, T, x, topk_slot, nullptr, nullptr, row_dst, rows_out, dev_status,
                         static_cast<char*>(ws), L, (cudaStream_t)stream);
}

int moe_residual_rmsnorm(int32_t T, int32_t d, const uint16_t* x, const uint16_t* y, float eps, uint16_t* x_next,
                         void* stream) {
    if (T < 0) return MOE_ERR_TOKENS;
    if (d <= 0 || d > 65536) return MOE_ERR_DIMS;
    if (!(eps >= 0.0f) || !(eps < 3.0e38f)) return MOE_ERR_DIMS;
    if (T > 0 && (!x || !y || !x_next)) return MOE_ERR_NULL;
    return launch_residual_rmsnorm(T, d, x, y, eps, x_next, (cudaStream_t)stream);
}

uint64_t moe_kernel_launches(void) { return fp4moe::g_kernel_launches.load(std::memory_order_relaxed); }

const char* moe_status_str(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_NULL: return "a required pointer is NULL";
        case MOE_ERR_DIMS: return "unsupported dims (d, f multiples of 256 up to 65536; 1 <= k <= E <= 1024; k <= 32)";
        case MOE_ERR_TOKENS: return "token count out of range";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_ARENA: return "arena misaligned, wrong slot_bytes or slot out of range";
        case MOE_ERR_FLAGS: return "unknown flags or missing output for the chosen flags";
        case MOE_ERR_LAUNCH: return "kernel launch failed";
        case MOE_ERR_ALIGN: return "pointer not sufficiently aligned";
        default: return "unknown status";
    }
}

}  // extern "C"
