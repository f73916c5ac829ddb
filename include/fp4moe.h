/*
 * fp4moe.h -- C ABI of the GB300 (sm_103a) routed-expert FP4 MoE layer.
 *
 * The layer (DeepSeek-V4.1-Flash routed experts) per token t:
 *   a1  l[t,e]   = x[t] . W_r[e]                                  router logits
 *   a2  s = sigmoid(l); key = s + bias[e] (-inf when expert e has no slot);
 *       top-k keys (ties to the lower expert id); w_j = s_j / sum(s)   selection
 *   a3  slot_j   = expert_to_slot[id_j]                           slot lookup
 *   a4  rows grouped by expert (prefill)                           permutation
 *   a5  h        = silu(W_gate x) * (W_up x)                       gate/up + SwiGLU
 *   a6  y[t]     = sum_j w_j * (W_down h_j), fixed ascending-id order, bf16 out
 * Experts are FP4: e2m1 codes, one UE8M0 scale per 32 consecutive K elements, three
 * f x d matrices per expert ("DeepSeek-V4.1-Flash on a single NVIDIA DGX Spark", section
 * "Why it is built this way": 15,360 x 3 x 2304 x 5120, 288.8 GB at FP4 + UE8M0/32).
 * Experts sit in a resident slot arena reached through an expert->slot table (same page,
 * headline list: a 73.8 GB arena of slots).  Rows are written once and summed by a
 * separate fixed-order step ("Start the expert reads before the GPU is done",
 * 30 September follow-up).
 *
 * Conventions for every call:
 *  - Pointers are DEVICE pointers unless stated.  The caller owns every buffer; no call
 *    allocates device memory, synchronises the device or reads results back.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*; NULL is the
 *    legacy default stream).
 *  - bf16 tensors are raw 16-bit bfloat16 bit patterns (uint16_t).  All tensors are dense
 *    row-major with the shapes given.
 *  - Return value: MOE_OK (0), or a negative MOE_ERR_* for an argument error detected on
 *    the host before anything is launched (nothing was enqueued).
 *  - Device-side conditions are OR-ed into *dev_status (an int32 the caller zeroes and reads
 *    after its own synchronisation): MOE_STATUS_* bits below.
 *  - Calls on different streams are independent when given different workspaces.
 *  - Some kernels are launched with programmatic dependent launch: they may become resident
 *    while the previous kernel on `stream` still runs.  Before that kernel has completed they
 *    read only these inputs, which the kernel enqueued immediately before the call must
 *    therefore not write: x and w_router of a decode-size routing call (T <= 16), whose
 *    logits are computed while the previous call's expert kernel finishes, and x of a decode
 *    call of moe_expert_ffn_fp4 or moe_layer_decode_fp4 (which also reads w_router early).  Every other input, every output and the workspace are
 *    touched only after it has completed.  (A kernel that never signals an early launch --
 *    a plain CUDA kernel, or this library's residual/RMSNorm step -- completes before the
 *    next one starts, so x written by such a kernel is safe.)
 *  - After a call that set MOE_STATUS_TIMEOUT the workspace must be re-initialised
 *    (moe_workspace_init) before its next use.
 */
#ifndef FP4MOE_H
#define FP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Per-layer shape.  d (hidden) and f (expert intermediate) must be multiples of 256;
 * 1 <= top_k <= num_experts <= 1024; top_k <= 32. */
typedef struct {
    int32_t d;
    int32_t f;
    int32_t num_experts;
    int32_t top_k;
} moe_dims;

/* Resident expert arena: num_slots slots of slot_bytes each, starting at base (device
 * memory, 1024-byte aligned).  slot_bytes must equal moe_slot_bytes(dims).  The layout
 * inside a slot is private to this library; moe_pack_expert is its only writer. */
typedef struct {
    void* base;
    int64_t slot_bytes;
    int32_t num_slots;
} moe_arena;

enum {
    MOE_OK = 0,
    MOE_ERR_NULL = -1,       /* a required pointer is NULL */
    MOE_ERR_DIMS = -2,       /* unsupported d, f, num_experts or top_k (see moe_dims) */
    MOE_ERR_TOKENS = -3,     /* T < 0 or T beyond what the workspace was sized for */
    MOE_ERR_WORKSPACE = -4,  /* ws_bytes smaller than moe_workspace_bytes(dims, T) */
    MOE_ERR_ARENA = -5,      /* arena base misaligned, slot_bytes mismatch or slot index out of range */
    MOE_ERR_FLAGS = -6,      /* unknown flag or inconsistent optional outputs */
    MOE_ERR_LAUNCH = -7,     /* a kernel launch was rejected by the CUDA runtime */
    MOE_ERR_ALIGN = -8       /* a pointer is not 16-byte aligned */
};

#define MOE_STATUS_FEW_RESIDENT 1  /* a token had fewer than top_k resident experts */
#define MOE_STATUS_BAD_SLOT 2      /* a slot id outside [0, num_slots): that term was skipped */
#define MOE_STATUS_TIMEOUT 4       /* a bounded device wait gave up */
#define MOE_STATUS_CB3_ROW 8       /* moe_pack_cb3: a row with more than 256 distinct values or a
                                      NaN scale; its levels and indices were written as zero */

/* Flags of moe_expert_ffn_fp4. */
#define MOE_FUSE_COMBINE 1         /* write y directly (fixed-order combine fused in) */
#define MOE_FFN_CUDA_CORES 2       /* use the CUDA-core kernels (exact fp4 x bf16 products, fp32
                                      accumulation) instead of the tensor-core kernels */

/* Bytes of one arena slot: 3*f*d/2 code bytes + 3*f*d/32 scale bytes, rounded up to
 * 1024 (18,800,640 at d=5120, f=2304).  Returns -1 for unsupported dims. */
int64_t moe_slot_bytes(const moe_dims* dims);

/* Workspace bytes needed by every call of this API for up to T_max tokens.  One workspace
 * may be shared by the calls of one layer issued in order on one stream.  Its contents
 * between calls are private; the first call on a new workspace needs no initialisation
 * beyond what moe_workspace_init performs.  Returns 0 for unsupported dims. */
size_t moe_workspace_bytes(const moe_dims* dims, int32_t T_max);

/* Zero the workspace's persistent counters (once, after allocating it).  This also restores
 * the default wait limit. */
int moe_workspace_init(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream);

/* Diagnostic knob for the bounded waits: after this call, every wait of an expert kernel on
 * another CTA's progress (decode: x encoded, a key's h complete; prefill on the tensor cores:
 * a token tile's h complete) through this workspace gives up after
 * `polls` polls instead of the default (about a second), sets MOE_STATUS_TIMEOUT and lets the
 * kernel drain its copies and return.  polls = 0 restores the default; so does
 * moe_workspace_init.  Waits on a CTA's own copies keep the default limit.  It exists so that
 * the timeout path can be exercised without a fault: a small limit makes a dependency wait run
 * out.  Enqueued on `stream` (one one-thread kernel); polls < 0 returns MOE_ERR_DIMS. */
int moe_workspace_set_wait_limit(const moe_dims* dims, void* ws, size_t ws_bytes, int32_t polls, void* stream);

/* Pack one expert from the canonical (checkpoint) layout into arena slot `slot`.
 * Canonical layout, device pointers, two e2m1 codes per byte (element 2i in the low
 * nibble), one UE8M0 byte per 32 consecutive K elements, row-major:
 *   gate_q, up_q : uint8 [f, d/2]     gate_s, up_s : uint8 [f, d/32]
 *   down_q       : uint8 [d, f/2]     down_s       : uint8 [d, f/32]
 * The source buffers may be reused once the stream has passed this call. */
int moe_pack_expert(const moe_dims* dims, const uint8_t* gate_q, const uint8_t* gate_s,
                    const uint8_t* up_q, const uint8_t* up_s, const uint8_t* down_q,
                    const uint8_t* down_s, const moe_arena* arena, int32_t slot, void* stream);

/* a1-a3: router scoring, top-k selection and slot lookup for T tokens ("Start the expert
 * reads before the GPU is done", 28 September follow-up: each layer's router runs on the GPU
 * and its chosen expert ids -- read back through the router mailbox there -- decide which
 * experts are read and computed; here they stay on the device as topk_slot).
 *   x              bf16 [T, d]
 *   w_router       bf16 [E, d]
 *   score_bias     fp32 [E] added to the score for selection only, or NULL
 *   expert_to_slot int32 [E]; -1 marks an expert without a slot (never selected)
 * Outputs, per token in ascending expert id:
 *   topk_ids int32 [T, k], topk_w fp32 [T, k] (sum to 1), topk_slot int32 [T, k];
 *   missing entries (fewer than k resident) are -1 / 0 / -1 with MOE_STATUS_FEW_RESIDENT.
 * The logit is the exact dot product rounded once to fp32 and the score is
 * fp32(1/(1+exp(-logit))) from a double evaluation; the chosen set is certified against
 * these exact values (fast fp32 logits with a rigorous error bound, exact recomputation of
 * any expert whose key interval straddles the k-th place). */
int moe_route_topk(const moe_dims* dims, int32_t T, const uint16_t* x, const uint16_t* w_router,
                   const float* score_bias, const int32_t* expert_to_slot, int32_t* topk_ids,
                   float* topk_w, int32_t* topk_slot, int32_t* dev_status, void* ws,
                   size_t ws_bytes, void* stream);

/* moe_route_topk without a workspace, for callers that cannot allocate device memory: an
 * op hosted by an engine that owns the whole device pool and gives its ops no workspace, or
 * a serving loop that must not allocate between steps.  The pages have no counterpart to
 * this entry point; it computes exactly what moe_route_topk computes.
 * Limits: 0 <= T <= 16 (larger T returns MOE_ERR_TOKENS before anything is enqueued) and the
 * dims limits above.  Its scratch (key records and norms, about 260 KB)
 * is a static device array inside this library, held by every GPU that loads the library
 * until the process exits.  It allocates nothing and calls no allocating routine.
 * The first call on each device looks up the array's device address with that device
 * current; make that first call before any stream capture.  That address is kept for the life
 * of the process, so this entry point must not be called on a device after cudaDeviceReset
 * there (the reset unloads the library's device code and its array with it).  Every call overwrites the
 * array: calls whose execution overlaps on the GPU -- on different streams, or from
 * different threads -- race on the shared array and must be serialised by the caller. */
int moe_route_topk_noalloc(const moe_dims* dims, int32_t T, const uint16_t* x, const uint16_t* w_router,
                           const float* score_bias, const int32_t* expert_to_slot, int32_t* topk_ids,
                           float* topk_w, int32_t* topk_slot, int32_t* dev_status, void* stream);

/* a4: stable grouping of the T*k (token, j) rows by expert id (tokens ascending inside a
 * group), so that every (token, slot) row has one place and is written once ("Start the
 * expert reads before the GPU is done", 30 September follow-up).
 *   group_offsets int32 [E+1]: group e = rows [off[e], off[e+1]); off[E] = rows with a valid id
 *   row_src int32 [T*k]: row r came from pair t*k + j; entries >= off[E] are -1
 *   row_dst int32 [T*k]: the inverse; -1 for id -1
 * The activations are not gathered here: the expert call reads x through row_src and encodes
 * its own tensor-core operand (so this call takes no x and writes no A operand). */
int moe_permute(const moe_dims* dims, int32_t T, const int32_t* topk_ids, int32_t* group_offsets,
                int32_t* row_src, int32_t* row_dst, void* ws, size_t ws_bytes, void* stream);

/* a5-a6: the experts.  Reads x bf16 [T, d], the routing outputs and the permutation
 * (group_offsets/row_src/row_dst from moe_permute of the same topk_ids).
 * flags = MOE_FUSE_COMBINE: writes y bf16 [T, d] (rows_out may be NULL).
 * flags = 0: writes rows_out fp32 [T*k, d] (row r = z for row_src[r], unweighted); y unused.
 * Slots outside [0, num_slots) set MOE_STATUS_BAD_SLOT and contribute zero.
 * Decode (T <= 16 with MOE_FUSE_COMBINE) needs only the routing outputs; the permutation
 * arguments may be NULL there.
 * Tensor cores (the default): tcgen05 block-scaled MMAs that feed x and h as a sum of four
 * MXFP4 terms each (e2m1 codes, UE8M0 scale per 32 elements, every term quantising the previous
 * terms' residual); expert outputs match exact fp4 x bf16 products to about 1e-4 relative
 * before the bf16 rounding of y.  They take decode calls with T*k <= 128.
 * CUDA cores (MOE_FFN_CUDA_CORES, and the other decode calls): decode streams every selected
 * expert once through one persistent kernel (then a small combine kernel); every product fp4 x
 * activation is exact in fp32 (x as f16 under a power-of-two scale per 32 elements, exact for
 * bf16; h rounded once to f16 under the same kind of scale), sums in fp32 in an order fixed by
 * the shapes.  Prefill runs grouped CUDA-core GEMMs with exact products.
 * In every decode kernel a call's row t is bit-identical to the T = 1 call on token t alone
 * (with the same routing), so multi-row verification reproduces single-token decoding. */
int moe_expert_ffn_fp4(const moe_dims* dims, const moe_arena* arena, int32_t T, const uint16_t* x,
                       const int32_t* topk_ids, const int32_t* topk_slot, const float* topk_w,
                       const int32_t* group_offsets, const int32_t* row_src, const int32_t* row_dst,
                       int32_t flags, float* rows_out, uint16_t* y, int32_t* dev_status, void* ws,
                       size_t ws_bytes, void* stream);

/* a1-a3 and a5-a6 of a decode call in one request: the outputs (topk_ids, topk_w, topk_slot,
 * y) are bit for bit those of moe_route_topk followed by moe_expert_ffn_fp4 with
 * MOE_FUSE_COMBINE on the same stream and workspace.  0 <= T <= 16 (larger T returns
 * MOE_ERR_TOKENS); arguments as in those two calls.  On the tensor-core path with at most 384
 * experts the router kernel writes only its key records and the expert kernel selects from
 * them itself (one warp per token in every CTA; CTA 0 writes the routing outputs), so the
 * expert reads start without waiting for a separate selection to complete: the boundary
 * between the router's result and the expert reads ("Start the expert reads before the GPU is
 * done", 28 September follow-up: the wait on the router mailbox and the boundaries between a
 * layer's command buffers) becomes a counter inside the GPU.  Other calls run the two steps as
 * separate launches.  The routing outputs are written while the expert kernel runs: read them
 * after this call completes. */
int moe_layer_decode_fp4(const moe_dims* dims, const moe_arena* arena, int32_t T, const uint16_t* x,
                         const uint16_t* w_router, const float* score_bias, const int32_t* expert_to_slot,
                         int32_t* topk_ids, float* topk_w, int32_t* topk_slot, uint16_t* y,
                         int32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/* a6 (unfused): y[t] = bf16( sum_j topk_w[t,j] * rows[row_dst[t*k+j]] ) in ascending j,
 * skipping row_dst = -1.  rows fp32 [T*k, d]. */
int moe_combine(const moe_dims* dims, int32_t T, const float* rows, const int32_t* row_dst,
                const float* topk_w, uint16_t* y, void* stream);

/* Partial residency (the two-wave routed MoE; "Start the expert reads before the GPU is
 * done", 30 September follow-up: compute the experts on hand before the top-up read and the
 * rest after it, bit-exact because every (token, slot) row is written once and the slot sum is
 * a separate fixed-order kernel; same page, 28 September follow-up: a GPU-driven expert gather
 * that removes the per-layer command buffers, proposed there as the next step).
 *
 * The routing is made with the table of destination slots (expert_to_slot: where each expert
 * lives when resident; missing experts must have distinct slots).  resident_expert int32
 * [num_slots] (device) says which expert each slot holds now (-1: none).
 *
 * moe_split_waves: for the T*k pairs, slot_wave1 = the pair's slot if that slot holds the
 * pair's expert now, else -1; slot_wave2 = the pair's slot otherwise, else -1 (pairs without a
 * valid slot are -1 in both).  missing int32 [T*k] receives the distinct experts of wave 2 in
 * ascending id and *n_missing (device int32) their count.  One kernel; all device memory.
 *
 * moe_gather_experts: copies, for each of the *n_missing experts e in missing, the slot image
 * at store + e * slot_bytes (n_store images in the arena's format: moe_pack_expert's layout
 * for an FP4 arena, moe_pack_cb3's for a cb3 arena, e.g. packed into a slot and copied out)
 * into slot expert_to_slot[e] of the arena, and sets resident_expert of that
 * slot to e.  store is any device-accessible address: device memory, or pinned host memory
 * mapped into the device (the kernel reads it directly; no copy is issued by the host).
 * 16-byte aligned.  An expert with no valid slot sets MOE_STATUS_BAD_SLOT and is skipped.
 *
 * Two waves: split; moe_expert_ffn_fp4 (flags 0) with slot_wave1 into rows; gather; the same
 * call with slot_wave2 into the same rows (each row is written by one of the two calls); then
 * moe_combine.  The result equals the one-wave call (all experts resident, same routing) bit
 * for bit.  On a cb3 arena the calls are moe_expert_ffn_cb3_rows (decode sizes). */
/* Cache-conditional routing ("DeepSeek-V4.1-Flash on a single NVIDIA DGX Spark", Conventions,
 * and the expert-cache notes list it as an approved approximation, after "Mixture of
 * Cache-Conditional Experts", arXiv 2412.00099; they give no formula, the reading here is an
 * additive bonus): instead of masking non-resident experts (expert_to_slot = -1),
 * route with every expert's destination slot and this bias:
 *   bias_out[e] = score_bias[e] (0 if score_bias is NULL) + lambda   if slot expert_to_slot[e]
 *                 holds e now (resident_expert), else score_bias[e].
 * Selection keys become s_e + bias_out[e]; weights stay s_j / sum s.  lambda = 0 is the exact
 * routing; a lambda above the spread of the keys gives the hard mask whenever k experts are
 * resident.  lambda must be finite and >= 0 (else MOE_ERR_DIMS).  One kernel, E entries. */
int moe_residency_bias(const moe_dims* dims, const float* score_bias, const int32_t* expert_to_slot,
                       const int32_t* resident_expert, int32_t num_slots, float lambda, float* bias_out,
                       void* stream);
int moe_split_waves(const moe_dims* dims, int32_t T, const int32_t* topk_ids, const int32_t* topk_slot,
                    const int32_t* resident_expert, int32_t num_slots, int32_t* slot_wave1, int32_t* slot_wave2,
                    int32_t* missing, int32_t* n_missing, void* stream);
int moe_gather_experts(const moe_dims* dims, const moe_arena* arena, const void* store, int32_t n_store,
                       const int32_t* missing, const int32_t* n_missing, const int32_t* expert_to_slot,
                       int32_t* resident_expert, int32_t* dev_status, void* stream);

/* cb3 expert format ("DeepSeek-V4.1-Flash on a single NVIDIA DGX Spark", section "The
 * numbers": resident experts in a 3-bit per-row codebook packed from the checkpoint's own FP4
 * experts).  An approximation of the model that trades accuracy for capacity: 13.4 MB per
 * expert instead of 18.8 MB at d=5120, f=2304.  Every matrix row (gate, up: K = d; down:
 * K = f) holds 8 bf16 levels and a 3-bit index per weight.  The pages give no packing rule;
 * the one used: the levels are the optimal 1-D 8-means of the row's FP4 values (clusters are
 * contiguous runs of the sorted distinct values, exact dynamic programming over the split
 * points in fp64, ties to the smaller split), each level its cluster's mean rounded once to
 * bf16, and a weight's index is its cluster.  A row with at most 8 distinct values is exact.
 * The slot layout is private to this library (moe_pack_cb3 is its only writer).
 *
 * moe_cb3_slot_bytes: bytes per cb3 slot (a multiple of 1024), or -1 for unsupported dims.
 *
 * moe_pack_cb3: packs the FP4 expert in slot fp4_slot of fp4_arena (moe_pack_expert's layout)
 * into slot cb3_slot of cb3_arena (slot_bytes = moe_cb3_slot_bytes).  One kernel, one block
 * per row.  A row with more than 256 distinct values or a NaN scale sets MOE_STATUS_CB3_ROW.
 *
 * moe_expert_ffn_cb3: a5-a6 on cb3 experts for T >= 0 tokens (decode and multi-token verify in
 * one call; more than 16 tokens, e.g. a prefill chunk, as consecutive calls of 16) and d <= 8192,
 * f <= 2304 (else MOE_ERR_DIMS):
 * h = silu(W_gate x) * (W_up x) rounded once to bf16, y[t] = bf16(sum_j w_j W_down h_j) in
 * ascending j; CUDA cores, bf16 x bf16 products (exact) summed in fp32.  Same routing inputs as the decode call of moe_expert_ffn_fp4 (topk_slot,
 * topk_w [T, k]); uses the workspace of moe_workspace_bytes(dims, T).  Row t equals the T = 1
 * call on token t bit for bit.  Slots outside [0, num_slots) set MOE_STATUS_BAD_SLOT.
 *
 * moe_expert_ffn_cb3_rows: the same expert work without the combine, for the two-wave flow
 * above (cb3 slots gathered like FP4 ones, since moe_gather_experts copies slot images): row
 * row_dst[t*k + j] of rows_out fp32 [T*k, d] receives z of pair (t, j) (W_down h_j,
 * unweighted) for every pair with a valid slot and row_dst >= 0 (row_dst < T*k, e.g. from
 * moe_permute); every other row is left untouched.  moe_combine of the rows then equals
 * moe_expert_ffn_cb3's y bit for bit (the same fma order). */
int64_t moe_cb3_slot_bytes(const moe_dims* dims);
int moe_pack_cb3(const moe_dims* dims, const moe_arena* fp4_arena, int32_t fp4_slot, const moe_arena* cb3_arena,
                 int32_t cb3_slot, int32_t* dev_status, void* stream);
int moe_expert_ffn_cb3(const moe_dims* dims, const moe_arena* cb3_arena, int32_t T, const uint16_t* x,
                       const int32_t* topk_slot, const float* topk_w, uint16_t* y, int32_t* dev_status, void* ws,
                       size_t ws_bytes, void* stream);
int moe_expert_ffn_cb3_rows(const moe_dims* dims, const moe_arena* cb3_arena, int32_t T, const uint16_t* x,
                            const int32_t* topk_slot, const int32_t* row_dst, float* rows_out, int32_t* dev_status,
                            void* ws, size_t ws_bytes, void* stream);

/* Layer chaining for multi-layer workloads (a harness step, not part of the routed-expert
 * layer): x_next[t] = bf16_RNE( v / sqrt(mean_i(v_i^2) + eps) ), v = x[t] + y[t] in fp32 (unit
 * RMSNorm weight).  x, y, x_next bf16 [T, d]; x_next may alias x.  One kernel, one block per
 * token.  eps must be finite and >= 0 (else MOE_ERR_DIMS); 1 <= d <= 65536. */
int moe_residual_rmsnorm(int32_t T, int32_t d, const uint16_t* x, const uint16_t* y, float eps, uint16_t* x_next,
                         void* stream);

/* Number of kernels this library has enqueued in this process so far (every entry point
 * above counts the kernels it launches).  A call captured into a CUDA graph counts once, at
 * capture, so the difference across a capture is the kernel count of one graph replay.
 * Thread-safe; never fails. */
uint64_t moe_kernel_launches(void);

/* Human-readable text of a return code. */
const char* moe_status_str(int code);

#ifdef __cplusplus
}
#endif

#endif /* FP4MOE_H */
