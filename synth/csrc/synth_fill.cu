// synth_fill.cu -- device-side Philox4x32-10 fill of the synthetic FP4 expert tensors.
// Produces exactly the bytes of synth/philox.py + synth/tensors.py (same key, counter and
// word/byte order), so large arenas can be generated on the device and regenerated on the
// host for any expert.  Input generation only: no MoE arithmetic.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        uint32_t hi0 = __umulhi(0xD2511F53u, c[0]), lo0 = 0xD2511F53u * c[0];
        uint32_t hi1 = __umulhi(0xCD9E8D57u, c[2]), lo1 = 0xCD9E8D57u * c[2];
        uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
}

// n bytes: byte i = byte (i % 4) of word (i / 4); a block gives 16 bytes.
__global__ void fill_bytes_kernel(uint8_t* dst, long long n, uint32_t seed, uint32_t tag) {
    long long nb = (n + 15) / 16;
    for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nb; b += (long long)gridDim.x * blockDim.x) {
        uint32_t c[4] = {(uint32_t)b, 0u, 0u, 0u};
        philox4x32_10(c, seed, tag);
        long long o = b * 16;
        if (o + 16 <= n) {
            reinterpret_cast<uint4*>(dst)[b] = make_uint4(c[0], c[1], c[2], c[3]);
        } else {
            for (int i = 0; o + i < n; ++i) dst[o + i] = (uint8_t)(c[i / 4] >> (8 * (i % 4)));
        }
    }
}

// n scale bytes: byte i = 127 + lo + (word i mod (hi - lo + 1)).
__global__ void fill_scales_kernel(uint8_t* dst, long long n, uint32_t seed, uint32_t tag, int lo, int hi) {
    long long nb = (n + 3) / 4;
    uint32_t span = (uint32_t)(hi - lo + 1);
    for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nb; b += (long long)gridDim.x * blockDim.x) {
        uint32_t c[4] = {(uint32_t)b, 0u, 0u, 0u};
        philox4x32_10(c, seed, tag);
        for (int i = 0; i < 4 && b * 4 + i < n; ++i) dst[b * 4 + i] = (uint8_t)(127 + lo + (int)(c[i] % span));
    }
}

}  // namespace

extern "C" {

int synth_fill_bytes(void* dst, long long n, uint32_t seed, uint32_t tag, void* stream) {
    if (!dst || n < 0 || ((uintptr_t)dst & 15u)) return -1;
    if (n == 0) return 0;
    fill_bytes_kernel<<<1024, 256, 0, (cudaStream_t)stream>>>((uint8_t*)dst, n, seed, tag);
    return cudaGetLastError() == cudaSuccess ? 0 : -7;
}

int synth_fill_scales(void* dst, long long n, uint32_t seed, uint32_t tag, int lo, int hi, void* stream) {
    if (!dst || n < 0 || hi < lo) return -1;
    if (n == 0) return 0;
    fill_scales_kernel<<<512, 256, 0, (cudaStream_t)stream>>>((uint8_t*)dst, n, seed, tag, lo, hi);
    return cudaGetLastError() == cudaSuccess ? 0 : -7;
}

}
