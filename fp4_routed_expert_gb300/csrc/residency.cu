// residency.cu -- partial residency: the two-wave routed MoE and the GPU-driven expert gather.
//
// "DeepSeek-V4.1-Flash on a single NVIDIA DGX Spark", 30 September follow-up (prefill): the
// two-wave routed MoE computes the experts already on hand before the top-up read and the rest
// after it; it is bit-exact because every (token, slot) row is written once and the slot sum
// is a separate fixed-order kernel.  28 September follow-up: the next step named there is a
// GPU-driven expert gather that removes the per-layer command buffers.
//
// Here the arena's slot table says where every expert lives when resident (expert_to_slot) and
// resident_expert[slot] says which expert a slot holds now.  moe_split_waves turns one routing
// into the slot arrays of the two waves and the list of missing experts, on the device;
// moe_gather_experts copies those experts' slot images from a store in (mapped, pinned) host
// memory into their slots, one kernel, no host step per expert.  The two waves are ordinary
// unfused expert calls (write-once fp32 rows) and moe_combine is the fixed-order sum, so the
// result equals the one-wave call on the same routing bit for bit.
#include "moe_internal.cuh"

namespace fp4moe {

// One block.  Pair i with slot s and expert e: wave 1 computes it when slot s holds e now,
// wave 2 otherwise (after the gather); pairs without a slot are in neither.  Missing experts
// are listed once each, ascending.
__global__ void __launch_bounds__(1024) split_waves_kernel(int n, int E, int num_slots, const int32_t* __restrict__ ids,
                                                           const int32_t* __restrict__ slot,
                                                           const int32_t* __restrict__ resident_expert, int32_t* wave1,
                                                           int32_t* wave2, int32_t* missing, int32_t* n_missing) {
    __shared__ unsigned miss[kMaxExperts / 32];
    __shared__ int base[kMaxExperts / 32 + 1];
    for (int i = threadIdx.x; i < kMaxExperts / 32; i += blockDim.x) miss[i] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int s = slot[i], e = ids[i];
        int w1 = -1, w2 = -1;
        if (s >= 0 && s < num_slots && e >= 0 && e < E) {
            if (resident_expert[s] == e) {
                w1 = s;
            } else {
                w2 = s;
                atomicOr(&miss[e >> 5], 1u << (e & 31));
            }
        }
        wave1[i] = w1;
        wave2[i] = w2;
    }
    __syncthreads();
    // ascending list: each 32-expert word's count, an exclusive scan (one thread: at most 32
    // words), then each word's experts in order
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int w = 0; w < (E + 31) / 32; ++w) {
            base[w] = acc;
            acc += __popc(miss[w]);
        }
        *n_missing = acc;
    }
    __syncthreads();
    for (int w = threadIdx.x; w < (E + 31) / 32; w += blockDim.x) {
        unsigned m = miss[w];
        int o = base[w];
        while (m) {
            const int b = __ffs(m) - 1;
            m &= m - 1;
            missing[o++] = w * 32 + b;
        }
    }
}

// Copies the slot image of missing expert e (store + e * slot_bytes) into slot
// expert_to_slot[e], then records the slot's new expert.  Work item = (list entry, 64 KB chunk);
// every thread moves 16-byte vectors; the store is read once, straight from host memory.
constexpr int64_t kGatherChunk = 65536;

__global__ void __launch_bounds__(256) gather_experts_kernel(const uint8_t* __restrict__ store, int n_store,
                                                             const int32_t* __restrict__ missing,
                                                             const int32_t* __restrict__ n_missing,
                                                             const int32_t* __restrict__ expert_to_slot, uint8_t* arena,
                                                             int64_t slot_bytes, int num_slots, int32_t* resident_expert,
                                                             int32_t* status) {
    const int nm = *n_missing;
    const int64_t chunks = (slot_bytes + kGatherChunk - 1) / kGatherChunk;
    for (int64_t item = blockIdx.x; item < (int64_t)nm * chunks; item += gridDim.x) {
        const int li = (int)(item / chunks);
        const int64_t c0 = (item % chunks) * kGatherChunk;
        const int e = missing[li];
        const int s = (e >= 0 && e < n_store) ? expert_to_slot[e] : -1;
        if (s < 0 || s >= num_slots) {
            if (threadIdx.x == 0 && c0 == 0) atomicOr(status, MOE_STATUS_BAD_SLOT);
            continue;
        }
        const int64_t len = (slot_bytes - c0 < kGatherChunk) ? slot_bytes - c0 : kGatherChunk;
        const uint4* src = reinterpret_cast<const uint4*>(store + (int64_t)e * slot_bytes + c0);
        uint4* dst = reinterpret_cast<uint4*>(arena + (int64_t)s * slot_bytes + c0);
        for (int64_t v = threadIdx.x; v < len / 16; v += blockDim.x) dst[v] = __ldcv(src + v);
        if (threadIdx.x == 0 && c0 == 0) resident_expert[s] = e;
    }
}

// Cache-conditional routing ("DeepSeek-V4.1-Flash on a single NVIDIA DGX Spark", Conventions
// and the expert-cache document list it as an approved approximation, after "Mixture of
// Cache-Conditional Experts", arXiv 2412.00099): instead of the hard mask of non-resident
// experts, a resident expert's selection key gets a bonus lambda.  bias_out[e] = bias[e] +
// lambda if expert e sits in its slot now, else bias[e].
__global__ void residency_bias_kernel(int E, const int32_t* __restrict__ expert_to_slot,
                                      const int32_t* __restrict__ resident_expert, int num_slots,
                                      const float* __restrict__ bias, float lambda, float* __restrict__ bias_out) {
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x) {
        const int s = expert_to_slot[e];
        const bool on_hand = s >= 0 && s < num_slots && resident_expert[s] == e;
        const float b = bias ? bias[e] : 0.0f;
        bias_out[e] = on_hand ? __fadd_rn(b, lambda) : b;
    }
}

int launch_residency_bias(const moe_dims* m, const int32_t* expert_to_slot, const int32_t* resident_expert,
                          int num_slots, const float* bias, float lambda, float* bias_out, cudaStream_t st) {
    residency_bias_kernel<<<(m->num_experts + 255) / 256, 256, 0, st>>>(m->num_experts, expert_to_slot, resident_expert,
                                                                        num_slots, bias, lambda, bias_out);
    note_launch(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

int launch_split_waves(const moe_dims* m, int T, const int32_t* ids, const int32_t* slot, const int32_t* resident_expert,
                       int num_slots, int32_t* wave1, int32_t* wave2, int32_t* missing, int32_t* n_missing,
                       cudaStream_t st) {
    split_waves_kernel<<<1, 1024, 0, st>>>(T * m->top_k, m->num_experts, num_slots, ids, slot, resident_expert, wave1,
                                           wave2, missing, n_missing);
    note_launch(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

int launch_gather_experts(const moe_arena* ar, const uint8_t* store, int n_store, const int32_t* missing,
                          const int32_t* n_missing, const int32_t* expert_to_slot, int32_t* resident_expert,
                          int32_t* status, cudaStream_t st, int num_sms) {
    gather_experts_kernel<<<4 * num_sms, 256, 0, st>>>(store, n_store, missing, n_missing, expert_to_slot,
                                                       static_cast<uint8_t*>(ar->base), ar->slot_bytes, ar->num_slots,
                                                       resident_expert, status);
    note_launch(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

}  // namespace fp4moe
